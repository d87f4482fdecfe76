"""The decode entry point for callers that cannot allocate device memory.

pa_decode_attention_static is for code that may not call cudaMalloc where it
runs the decode step (a fixed memory map, a serving thread that must not
trigger an allocation's device-wide synchronisation, a plugin that only gets
its tensors).  It keeps the split-context partials and the work counter in a
fixed array inside the library, and must give what pa_decode_attention gives
with a caller workspace, and what the oracle gives.

The cases run the split-context kernel (forced, and chosen automatically for
a batch too large for the per-head cluster kernel), which is the kernel that
reads and writes the array: every call leaves partials and a work counter
behind, so two calls in a row with different batches and grids check that
nothing carries over from one call to the next.  Calls go through the C ABI.
"""
import ctypes

import numpy as np
import pytest

import oracle
import pa_workloads as wl
from helpers import assert_attention_close, dev_bf16, dev_i32, host_f64, workspace_for

pytestmark = pytest.mark.gpu

N_Q, D = 32, 64


def _pk():
    import paged_kv_cache_205_gb300 as pk
    return pk


def _static_fn():
    fn = _pk().library().pa_decode_attention_static
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.argtypes = [P, P, P, I, P, I, I, P, I, I, F, P, P]
    fn.restype = I
    return fn


def _case(seed, ctx):
    rng = np.random.default_rng(seed)
    ctx = np.asarray(ctx, dtype=np.int32)
    nbk = int(((ctx + 15) // 16).sum()) + 8
    mb = int(max(1, ((ctx + 15) // 16).max())) + 1
    w = wl.make_workload("tiny", seed=seed, context_lens=ctx, num_blocks=nbk, max_blocks_per_seq=mb)
    pool = wl.make_pool_numpy(w, rng, poison=True)
    q = wl.normal_bf16(rng, (len(ctx), N_Q, D), scale=2.0)
    return w, pool, q


def _run_both(fn, w, pool, q):
    """The same call through pa_decode_attention (caller workspace) and
    pa_decode_attention_static; returns both outputs as fp64."""
    import torch
    pk = _pk()
    n = w.num_seqs
    qd, poold = dev_bf16(q), dev_bf16(pool)
    btd, ctxd = dev_i32(w.block_table), dev_i32(w.context_lens)
    ref = torch.full((n, N_Q, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    got = torch.full((n, N_Q, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    err_ref = torch.zeros(1, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pk.pa_decode_attention(ref, qd, poold, btd, ctxd, 0, 0.125,
                           workspace_for(n, w.max_blocks_per_seq), err_ref)
    rc = fn(got.data_ptr(), qd.data_ptr(), poold.data_ptr(), w.num_blocks, btd.data_ptr(),
            w.n_layers, w.max_blocks_per_seq, ctxd.data_ptr(), n, 0, 0.125, err.data_ptr(),
            torch.cuda.current_stream().cuda_stream)
    assert rc == 0, rc
    torch.cuda.synchronize()
    assert int(err.item()) == 0 and int(err_ref.item()) == 0
    return host_f64(got), host_f64(ref)


def test_static_scratch_split_kernel_twice_in_a_row_matches_oracle():
    """Two calls in a row on the split-context kernel, with different batch
    sizes and grids (so the partial slots and the work counter of the first
    call sit where the second one reads): each matches the oracle and the
    workspace entry point."""
    pk = _pk()
    fn = _static_fn()
    cases = [(_case(71, [1, 300, 17, 2048, 0, 95, 640, 16, 1500, 33]), 0),
             (_case(72, [5000, 3, 129, 64, 1, 777]), 7)]
    pk.pa_decode_set_path(pk.PA_DECODE_SPLIT)
    try:
        for i, ((w, pool, q), grid) in enumerate(cases):
            pk.pa_decode_set_grid_limit(grid)
            assert pk.pa_decode_kernel_for(w.num_seqs) == pk.PA_DECODE_SPLIT
            got, ref = _run_both(fn, w, pool, q)
            o, e = oracle.decode_attention(q, pool, w.block_table, w.context_lens, 0)
            assert e == 0
            assert_attention_close(got, o, f"call {i} vs oracle")
            assert_attention_close(got, ref, f"call {i} vs workspace entry point")
    finally:
        pk.pa_decode_set_path(pk.PA_DECODE_AUTO)
        pk.pa_decode_set_grid_limit(0)


def test_static_scratch_automatic_choice_on_a_large_batch():
    """A batch of 40 sequences takes the split-context kernel under the
    automatic choice (more (sequence, kv head) pairs than the GPU holds two
    CTAs for), followed by a smaller one that takes the per-head cluster
    kernel: both match the oracle."""
    pk = _pk()
    fn = _static_fn()
    pk.pa_decode_set_path(pk.PA_DECODE_AUTO)
    pk.pa_decode_set_grid_limit(0)
    rng = np.random.default_rng(73)
    for i, ctx in enumerate([rng.integers(0, 1200, size=40), [900, 4, 2100]]):
        w, pool, q = _case(74 + i, ctx)
        got, ref = _run_both(fn, w, pool, q)
        o, e = oracle.decode_attention(q, pool, w.block_table, w.context_lens, 0)
        assert e == 0
        assert_attention_close(got, o, f"call {i} ({w.num_seqs} sequences) vs oracle")
        assert_attention_close(got, ref, f"call {i} vs workspace entry point")
    assert pk.pa_decode_kernel_for(40) == pk.PA_DECODE_SPLIT


def test_static_scratch_refuses_more_sequences_than_it_holds():
    import torch
    fn = _static_fn()
    n = 513
    t = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = fn(t.data_ptr(), t.data_ptr(), t.data_ptr(), 1, t.data_ptr(), 1, 1, t.data_ptr(), n, 0,
            0.125, t.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == -4
