"""The decode entry point for callers that cannot allocate device memory.

pa_decode_attention_static is for code that may not call cudaMalloc where it
runs the decode step (a fixed memory map, a serving thread that must not
trigger an allocation's device-wide synchronisation, a plugin that only gets
its tensors).  It keeps its scratch in a fixed array inside the library and
must give what pa_decode_attention gives with a caller workspace.  Both are
called through the C ABI; two calls in a row, with different inputs, check
that the shared array carries nothing over from one call to the next.
"""
import ctypes

import numpy as np
import pytest

import pa_workloads as wl
from helpers import assert_attention_close, dev_bf16, dev_i32, host_f64, workspace_for

pytestmark = pytest.mark.gpu

N_Q, D = 32, 64


def _static_fn():
    import paged_kv_cache_205_gb300 as pk
    fn = pk.library().pa_decode_attention_static
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


def test_static_scratch_matches_workspace_entry_point_twice_in_a_row():
    import torch
    import paged_kv_cache_205_gb300 as pk
    fn = _static_fn()
    stream = torch.cuda.current_stream().cuda_stream
    cases = [_case(71, [1, 300, 17, 2048, 0, 95, 640, 16]),
             _case(72, [5000, 3, 129, 64, 1, 777])]
    for i, (w, pool, q) in enumerate(cases):
        n = w.num_seqs
        qd, poold = dev_bf16(q), dev_bf16(pool)
        btd, ctxd = dev_i32(w.block_table), dev_i32(w.context_lens)
        ref = torch.empty((n, N_Q, D), dtype=torch.bfloat16, device="cuda")
        got = torch.full((n, N_Q, D), float("nan"), dtype=torch.bfloat16, device="cuda")
        err_ref = torch.zeros(1, dtype=torch.int32, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        pk.pa_decode_attention(ref, qd, poold, btd, ctxd, 0, 0.125,
                               workspace_for(n, w.max_blocks_per_seq), err_ref)
        rc = fn(got.data_ptr(), qd.data_ptr(), poold.data_ptr(), w.num_blocks, btd.data_ptr(),
                w.n_layers, w.max_blocks_per_seq, ctxd.data_ptr(), n, 0, 0.125, err.data_ptr(),
                stream)
        assert rc == 0, rc
        torch.cuda.synchronize()
        assert int(err.item()) == 0 and int(err_ref.item()) == 0
        assert_attention_close(host_f64(got), host_f64(ref), f"call {i}")


def test_static_scratch_refuses_more_sequences_than_it_holds():
    import torch
    fn = _static_fn()
    n = 513
    t = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = fn(t.data_ptr(), t.data_ptr(), t.data_ptr(), 1, t.data_ptr(), 1, 1, t.data_ptr(), n, 0,
            0.125, t.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == -4
