"""Full-size parity against the fp64 CPU oracle, every output compared.

* The four large decode workloads (llama1b, pool2g, long32k, ragged without
  its append), device pools drawn by torch's seeded generator as the
  benchmark draws them: pa_decode_attention in the benchmark's launch
  configuration (automatic kernel choice) on every layer, every sequence;
  then each decode kernel forced on the first and last layer, every
  sequence.
* The ragged workload's whole step at its real size (256 sequences, 16
  layers, a 262,144-page pool, the shuffled free list): per layer
  pa_kv_append_rope with q (page allocation, Llama-3 RoPE, K/V stores), then
  pa_decode_attention over ctx + 1.  Tables, free list and free count are
  compared bit for bit, V stores bit for bit, K and q within the RoPE bound,
  and the attention against the oracle fed only with the workload's inputs
  and the oracle's own append results.

Tolerance (bf16 output vs the fp64 oracle): max abs error <= 1e-2, mean abs
error <= 1e-3.  Calls go through the C ABI.
"""
import numpy as np
import pytest

import oracle
import pa_workloads as wl
from helpers import (assert_attention_close, dev_bf16, dev_i32, gather_for_oracle, host_bits,
                     host_f64, oracle_attention_threads, ulp_diff, workspace_for)

pytestmark = pytest.mark.gpu

N_Q, N_KV, D, BS = 32, 8, 64, 16
# The kernels rotate in fp32 (angle reduced in fp64): an element a*c - b*s
# carries up to about 2^-22 (|a| + |b|) before its bf16 rounding, so where the
# two terms cancel it may sit more than one bf16 ulp from the fp64 oracle.
ROPE_ABS = 1.5e-5


def _pk():
    import paged_kv_cache_205_gb300 as pk
    return pk


def assert_rope_close(gpu_bits, ref_bits, what):
    d = ulp_diff(gpu_bits, ref_bits)
    absd = np.abs(oracle.bf16_to_f64(gpu_bits) - oracle.bf16_to_f64(ref_bits))
    bad = (d > 1) & ~(absd <= ROPE_ABS)
    assert not np.any(bad), f"{what}: {int(bad.sum())} elements off by up to {d.max()} ulp"
    assert np.mean(d > 0) < 1e-2, f"{what}: {np.mean(d > 0):.3%} elements differ"


def _layer_refs(pool, w, q, ctx, layers):
    refs = {}
    for layer in layers:
        sub, bt = gather_for_oracle(pool, w.block_table, range(w.num_seqs), ctx, layer)
        ref, e = oracle_attention_threads(q[layer], sub, bt, ctx, 0, scale=w.scale)
        assert e == 0
        refs[layer] = ref
    return refs


@pytest.mark.parametrize("name", ["llama1b", "pool2g", "long32k", "ragged"])
def test_full_size_every_sequence_every_layer(name):
    import torch
    pk = _pk()
    w = wl.make_workload(name)
    pool = wl.make_pool_torch(w, "cuda", seed=w.seed)
    ctx = w.context_lens            # ragged here without its append: attention over ctx
    rng = np.random.default_rng(w.seed + 1000)
    L, n = w.n_layers, w.num_seqs
    q = wl.normal_bf16(rng, (L, n, N_Q, D), scale=w.q_scale)
    qd, btd, ctxd = dev_bf16(q), dev_i32(w.block_table), dev_i32(ctx)
    out = torch.full((L, n, N_Q, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = workspace_for(n, w.max_blocks_per_seq)
    refs = _layer_refs(pool, w, q, ctx, range(L))
    try:
        pk.pa_decode_set_grid_limit(0)
        paths = [("auto", pk.PA_DECODE_AUTO, range(L)), ("split", pk.PA_DECODE_SPLIT, (0, L - 1)),
                 ("cluster", pk.PA_DECODE_CLUSTER, (0, L - 1)), ("seq", pk.PA_DECODE_SEQ, (0, L - 1))]
        for path, code, layers in paths:
            pk.pa_decode_set_path(code)
            out.fill_(float("nan"))
            for layer in layers:
                pk.pa_decode_attention(out[layer], qd[layer], pool, btd, ctxd, layer, w.scale, ws,
                                       err)
            torch.cuda.synchronize()
            assert int(err.item()) == 0, path
            got = host_f64(out)
            for layer in layers:
                assert_attention_close(got[layer], refs[layer], f"{name} {path} layer {layer}")
    finally:
        pk.pa_decode_set_path(pk.PA_DECODE_AUTO)
    del pool
    torch.cuda.empty_cache()


def _renaming(num_blocks, touched):
    """A permutation of the page ids that sends the pages in `touched` to
    0 .. len(touched)-1 (in that order) and the others after them, and its
    inverse; -1 stays -1."""
    touched = np.asarray(touched, dtype=np.int64)
    new = np.empty(num_blocks, dtype=np.int64)
    rest = np.setdiff1d(np.arange(num_blocks), touched)
    new[touched] = np.arange(len(touched))
    new[rest] = len(touched) + np.arange(len(rest))
    inv = np.empty(num_blocks, dtype=np.int64)
    inv[new] = np.arange(num_blocks)

    def fwd(a):
        return np.where(a >= 0, new[np.clip(a, 0, num_blocks - 1)], a).astype(np.int32)

    def back(a):
        return np.where(a >= 0, inv[np.clip(a, 0, num_blocks - 1)], a).astype(np.int32)

    return fwd, back


def test_ragged_step_at_full_size_append_then_attention():
    """The ragged workload's step, layer by layer, at its real size.

    The oracle's append works on a copy of the pool, so it is run over only
    the pages one call can touch: each sequence's page at position ctx when
    ctx is inside a page, and the last num_seqs entries of the free list (no
    call pops more).  Page ids are renamed so that those pages are 0 .. R-1
    of a compact pool and the oracle is told the pool has R pages: a touch of
    any other page would be reported as a bad page, not written.  The
    oracle's tables and free list are renamed back before they are compared.
    """
    import torch
    pk = _pk()
    w = wl.make_workload("ragged")
    L, n, NB = w.n_layers, w.num_seqs, w.num_blocks
    pool = wl.make_pool_torch(w, "cuda", seed=w.seed)
    rng = np.random.default_rng(w.seed + 2000)
    q_all, k_all, v_all = wl.make_step_inputs(w, rng)
    ctx = w.context_lens.astype(np.int32)
    btd, fld = dev_i32(w.block_table), dev_i32(w.free_list)
    fcd = dev_i32(np.array([w.free_count]))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ctxd, ctx1d = dev_i32(ctx), dev_i32(ctx + 1)
    out = torch.full((n, N_Q, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = workspace_for(n, w.max_blocks_per_seq)
    table, fl, fc = w.block_table.copy(), w.free_list.copy(), int(w.free_count)
    opened = 0
    pk.pa_decode_set_path(pk.PA_DECODE_AUTO)
    pk.pa_decode_set_grid_limit(0)
    for layer in range(L):
        inside = ctx % BS != 0
        existing = table[np.arange(n), layer, ctx // BS][inside]
        top = fl[max(0, fc - n):fc]
        touched = np.concatenate([existing, top]).astype(np.int64)
        assert len(np.unique(touched)) == len(touched) and np.all(touched >= 0)
        fwd, back = _renaming(NB, touched)
        tid = torch.from_numpy(touched).to("cuda")
        before = host_bits(pool.index_select(0, tid))

        qd = dev_bf16(q_all[layer])
        pk.pa_kv_append_rope(dev_bf16(k_all[layer]), dev_bf16(v_all[layer]), qd, pool, btd,
                             ctxd, layer, fld, fcd, err)
        pk.pa_decode_attention(out, qd, pool, btd, ctx1d, layer, w.scale, ws, err)

        q_rot, after, bt2, fl2, fc2, e = oracle.kv_append_rope(
            k_all[layer], v_all[layer], q_all[layer], before, fwd(table), ctx, layer, fwd(fl), fc,
            num_blocks=len(touched))
        assert e == 0, layer
        table_ref = back(bt2)
        fl_ref = back(fl2[:fc2])
        torch.cuda.synchronize()
        assert int(err.item()) == 0, layer
        # tables, free list and count: bit for bit
        assert np.array_equal(btd.cpu().numpy(), table_ref), layer
        assert int(fcd.item()) == fc2, layer
        assert np.array_equal(fld.cpu().numpy()[:fc2], fl_ref), layer
        opened += fc - fc2
        # the touched pages: V and untouched slots bit for bit, K within the RoPE bound
        got_pages = host_bits(pool.index_select(0, tid))
        same = (got_pages == after) | ((got_pages == wl.BF16_NAN) & (after == wl.BF16_NAN))
        assert np.all(same[:, 1]), f"layer {layer}: V stores differ"
        if not np.all(same[:, 0]):
            assert_rope_close(got_pages[:, 0], after[:, 0], f"layer {layer} K")
        assert_rope_close(host_bits(qd), q_rot, f"layer {layer} q")
        # attention over ctx + 1: the layer's pages as drawn, the touched ones
        # as the oracle wrote them, and the oracle's rotated q
        sub, sbt, ids = gather_for_oracle(pool, table_ref, range(n), ctx + 1, layer,
                                          return_ids=True)
        pos = {int(b): i for i, b in enumerate(touched.tolist())}
        for i, b in enumerate(ids.tolist()):
            if b in pos:
                sub[i] = after[pos[b]]
        ref, e = oracle_attention_threads(q_rot, sub, sbt, ctx + 1, 0, scale=w.scale)
        assert e == 0
        assert_attention_close(host_f64(out), ref, f"ragged layer {layer} attention over ctx+1")
        table, fl, fc = table_ref, np.concatenate([fl_ref, fl[fc2:]]), fc2
    # pages open at every layer where a context ends on a page boundary
    assert opened == L * int(np.sum(ctx % BS == 0))
    del pool
    torch.cuda.empty_cache()
