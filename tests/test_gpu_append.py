"""GPU parity of pa_kv_append_rope and pa_free against the CPU oracle.

Tables, free lists, free counts, V stores and untouched pool bytes must be
bit-exact; rotated K and q within 1 bf16 ulp of the fp64 oracle (almost
all exact).  Calls go through the C ABI.
"""
import json
import os

import numpy as np
import pytest

import oracle
import pa_workloads as wl
from helpers import (assert_attention_close, dev_bf16, dev_i32, host_bits, host_f64,
                     ulp_diff, workspace_for)

pytestmark = pytest.mark.gpu

N_Q, N_KV, D, BS = 32, 8, 64, 16
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "append_free_worked_example.json")


def _pk():
    import paged_kv_cache_205_gb300 as pk
    return pk


class DevState:
    def __init__(self, pool, bt, fl, fc):
        import torch
        self.pool = dev_bf16(pool)
        self.bt = dev_i32(bt)
        self.fl = dev_i32(fl)
        self.fc = dev_i32(np.array([fc]))
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")

    def host(self):
        import torch
        torch.cuda.synchronize()
        return (host_bits(self.pool), self.bt.cpu().numpy(), self.fl.cpu().numpy(),
                int(self.fc.item()), int(self.err.item()))


def _append(st, k, v, q, ctx, layer):
    qd = None if q is None else dev_bf16(q)
    _pk().pa_kv_append_rope(dev_bf16(k), dev_bf16(v), qd, st.pool, st.bt, dev_i32(ctx), layer,
                            st.fl, st.fc, st.err)
    return qd


# The kernels rotate in fp32: a rotated element a*c - b*s carries an absolute
# error up to about 2^-22 (|a| + |b|) before its bf16 rounding, so where the
# two terms cancel it may sit more than one bf16 ulp from the fp64 oracle.
# Inputs here are N(0,1) in bf16 (|a|, |b| < 6): allow one ulp, or 1.5e-5.
ROPE_ABS = 1.5e-5


def assert_rope_close(gpu_bits, ref_bits, what):
    d = ulp_diff(gpu_bits, ref_bits)
    absd = np.abs(oracle.bf16_to_f64(gpu_bits) - oracle.bf16_to_f64(ref_bits))
    bad = (d > 1) & ~(absd <= ROPE_ABS)
    assert not np.any(bad), f"{what}: {int(bad.sum())} elements off by up to {d.max()} ulp / {absd.max():.2e}"
    assert np.mean(d > 0) < 1e-2, f"{what}: {np.mean(d > 0):.3%} elements differ"


def _compare_pools(gpu_pool, ref_pool):
    """V and untouched bytes exact; K within the fp32 rotation bound."""
    same = gpu_pool == ref_pool
    nan_both = (gpu_pool == wl.BF16_NAN) & (ref_pool == wl.BF16_NAN)
    same |= nan_both
    assert np.all(same[:, 1]), "V stores differ"
    if not np.all(same[:, 0]):
        assert_rope_close(gpu_pool[:, 0], ref_pool[:, 0], "K")


def test_worked_example_append_then_free():
    g = json.load(open(GOLDEN))
    rng = np.random.default_rng(0)
    pool = wl.normal_bf16(rng, (g["num_blocks"], 2, BS, N_KV, D))
    st = DevState(pool, np.array(g["block_table"]), np.array(g["free_list"]), g["free_count"])
    ctx = np.array(g["append"]["context_lens"], dtype=np.int32)
    n = len(ctx)
    ref = (pool, np.array(g["block_table"], dtype=np.int32), np.array(g["free_list"], dtype=np.int32),
           g["free_count"])
    for layer in g["append"]["layers"]:
        k = wl.normal_bf16(rng, (n, N_KV, D))
        v = wl.normal_bf16(rng, (n, N_KV, D))
        _append(st, k, v, None, ctx, layer)
        _, p2, b2, f2, c2, e = oracle.kv_append_rope(k, v, None, ref[0], ref[1], ctx, layer, ref[2], ref[3])
        assert e == 0
        ref = (p2, b2, f2, c2)
    gp, gb, gf, gc, ge = st.host()
    assert ge == 0
    assert np.array_equal(gb, np.array(g["append"]["expect_block_table"]))
    assert np.array_equal(gb, ref[1]) and np.array_equal(gf, ref[2]) and gc == ref[3]
    assert gc == g["append"]["expect_free_count"]
    _compare_pools(gp, ref[0])

    f = g["free"]
    _pk().pa_free(dev_i32(f["seq_ids"]), st.bt, dev_i32(f["context_lens"]), st.fl, st.fc,
                  g["num_blocks"], st.err)
    _, gb, gf, gc, ge = st.host()
    assert ge == f["expect_err"]
    assert np.array_equal(gb, np.array(f["expect_block_table"]))
    assert gc == f["expect_free_count"]
    assert list(gf[:gc]) == f["expect_free_list_head"]


def test_worked_example_underflow():
    u = json.load(open(GOLDEN))["underflow"]
    rng = np.random.default_rng(1)
    pool = wl.normal_bf16(rng, (u["num_blocks"], 2, BS, N_KV, D))
    st = DevState(pool, np.array(u["block_table"]), np.array(u["free_list"]), u["free_count"])
    n = len(u["context_lens"])
    k = wl.normal_bf16(rng, (n, N_KV, D))
    v = wl.normal_bf16(rng, (n, N_KV, D))
    _append(st, k, v, None, np.array(u["context_lens"]), 0)
    gp, gb, gf, gc, ge = st.host()
    assert ge == u["expect_err"]
    assert np.array_equal(gb, np.array(u["expect_block_table"]))
    assert gc == u["expect_free_count"]
    _, p2, b2, _, c2, e2 = oracle.kv_append_rope(k, v, None, pool, np.array(u["block_table"]),
                                                 u["context_lens"], 0, u["free_list"], u["free_count"])
    assert e2 == ge and np.array_equal(b2, gb) and c2 == gc
    _compare_pools(gp, p2)


@pytest.mark.parametrize("seed,positions", [
    (1, [0, 1, 15, 16, 17, 31, 32, 100, 2047, 2048, 8191, 8192]),
    (2, list(range(0, 64))),
    (3, [32767, 32768 - 16, 5000, 0]),
])
def test_append_with_q_matches_oracle(seed, positions):
    rng = np.random.default_rng(seed)
    ctx = np.array(positions, dtype=np.int32)
    n = len(ctx)
    n_layers = 2
    mb = int(ctx.max()) // BS + 2
    nbk = int(((ctx + 15) // 16).sum()) * n_layers + 2 * n + 5
    w = wl.make_workload("tiny", seed=seed, context_lens=ctx, n_layers=n_layers, num_blocks=nbk,
                         max_blocks_per_seq=mb)
    pool = wl.make_pool_numpy(w, rng, poison=True)
    st = DevState(pool, w.block_table, w.free_list, w.free_count)
    ref = (pool, w.block_table, w.free_list, w.free_count)
    for layer in range(n_layers):
        k = wl.normal_bf16(rng, (n, N_KV, D))
        v = wl.normal_bf16(rng, (n, N_KV, D))
        q = wl.normal_bf16(rng, (n, N_Q, D))
        qd = _append(st, k, v, q, ctx, layer)
        q2, p2, b2, f2, c2, e = oracle.kv_append_rope(k, v, q, ref[0], ref[1], ctx, layer, ref[2], ref[3])
        assert e == 0
        ref = (p2, b2, f2, c2)
        assert_rope_close(host_bits(qd), q2, f"q layer {layer}")
    gp, gb, gf, gc, ge = st.host()
    assert ge == 0
    assert np.array_equal(gb, ref[1]) and np.array_equal(gf, ref[2]) and gc == ref[3]
    _compare_pools(gp, ref[0])


def test_capacity_and_bad_entry_errors_match_oracle():
    rng = np.random.default_rng(4)
    w = wl.make_workload("tiny", context_lens=[64, 3, 20], max_blocks_per_seq=4)
    pool = wl.make_pool_numpy(w, rng)
    bt = w.block_table.copy()
    bt[2, 0, 1] = -1                      # existing page of seq 2 is missing
    st = DevState(pool, bt, w.free_list, w.free_count)
    k = wl.normal_bf16(rng, (3, N_KV, D))
    v = wl.normal_bf16(rng, (3, N_KV, D))
    q = wl.normal_bf16(rng, (3, N_Q, D))
    qd = _append(st, k, v, q, w.context_lens, 0)
    gp, gb, gf, gc, ge = st.host()
    q2, p2, b2, f2, c2, e2 = oracle.kv_append_rope(k, v, q, pool, bt, w.context_lens, 0,
                                                   w.free_list, w.free_count)
    assert ge == e2 == (oracle.ERR_CTX_RANGE | oracle.ERR_BAD_BLOCK)
    assert np.array_equal(gb, b2) and gc == c2
    _compare_pools(gp, p2)
    assert_rope_close(host_bits(qd)[1:], q2[1:], "q")
    assert np.array_equal(host_bits(qd)[0], q[0])      # out-of-range position: q untouched


def test_free_matches_oracle_with_overflow_and_bad_entries():
    bt = np.array([[[0, 1, -1]], [[2, -1, -1]], [[5, 6, 7]]], dtype=np.int32)
    fl = np.array([3, 4, -1, -1, -1, -1, -1, -1], dtype=np.int32)
    ctx = np.array([20, 10, 48], dtype=np.int32)
    for ids, fc, nbk in (([0, 1], 2, 8), ([2, 0], 6, 8), ([1, 2, 0], 2, 8)):
        st = DevState(np.zeros((nbk, 2, BS, N_KV, D), np.uint16), bt, fl, fc)
        _pk().pa_free(dev_i32(ids), st.bt, dev_i32(ctx), st.fl, st.fc, nbk, st.err)
        _, gb, gf, gc, ge = st.host()
        b2, f2, c2, e2 = oracle.free(ids, bt, ctx, fl, fc, nbk)
        assert ge == e2 and gc == c2
        assert np.array_equal(gb, b2) and np.array_equal(gf, f2)


def test_decode_step_append_then_attention_over_new_token():
    """Ragged continuous-batching step at small scale: each layer appends the
    token at pos = ctx (RoPE on k and q), then attends over ctx + 1."""
    import torch
    pk = _pk()
    rng = np.random.default_rng(6)
    w = wl.make_workload("ragged", seed=6, num_seqs=24, max_ctx=300, n_layers=3, num_blocks=2000)
    pool = wl.make_pool_numpy(w, rng, poison=True)
    st = DevState(pool, w.block_table, w.free_list, w.free_count)
    ref = (pool, w.block_table, w.free_list, w.free_count)
    n = w.num_seqs
    out = torch.empty((n, N_Q, D), dtype=torch.bfloat16, device="cuda")
    ws = workspace_for(n, w.max_blocks_per_seq)
    ctx_attn = dev_i32(w.context_lens + 1)
    for layer in range(w.n_layers):
        k = wl.normal_bf16(rng, (n, N_KV, D))
        v = wl.normal_bf16(rng, (n, N_KV, D))
        q = wl.normal_bf16(rng, (n, N_Q, D))
        qd = _append(st, k, v, q, w.context_lens, layer)
        pk.pa_decode_attention(out, qd, st.pool, st.bt, ctx_attn, layer, w.scale, ws, st.err)
        q2, p2, b2, f2, c2, e = oracle.kv_append_rope(k, v, q, ref[0], ref[1], w.context_lens,
                                                      layer, ref[2], ref[3])
        assert e == 0
        ref = (p2, b2, f2, c2)
        torch.cuda.synchronize()
        o_ref, e = oracle.decode_attention(q2, p2, b2, w.context_lens + 1, layer)
        assert e == 0
        assert_attention_close(host_f64(out), o_ref, f"layer {layer}")
    gp, gb, gf, gc, ge = st.host()
    assert ge == 0
    assert np.array_equal(gb, ref[1]) and np.array_equal(gf, ref[2]) and gc == ref[3]
    _compare_pools(gp, ref[0])


def test_whole_decode_step_captured_in_one_graph():
    """A ragged decode step (append with RoPE, then attention over ctx + 1,
    for every layer) captured as one CUDA graph and replayed: each replay
    re-appends the same token and must match the oracle."""
    import torch
    pk = _pk()
    rng = np.random.default_rng(8)
    w = wl.make_workload("ragged", seed=8, num_seqs=20, max_ctx=200, n_layers=3, num_blocks=1200)
    pool = wl.make_pool_numpy(w, rng, poison=True)
    st = DevState(pool, w.block_table, w.free_list, w.free_count)
    n, L = w.num_seqs, w.n_layers
    k = wl.normal_bf16(rng, (L, n, N_KV, D))
    v = wl.normal_bf16(rng, (L, n, N_KV, D))
    q = wl.normal_bf16(rng, (L, n, N_Q, D))
    kd, vd = dev_bf16(k), dev_bf16(v)
    q_in = dev_bf16(q)
    qd = q_in.clone()
    fc0 = st.fc.clone()
    ctx, ctx1 = dev_i32(w.context_lens), dev_i32(w.context_lens + 1)
    out = torch.zeros((L, n, N_Q, D), dtype=torch.bfloat16, device="cuda")
    ws = workspace_for(n, w.max_blocks_per_seq)

    def step():
        qd.copy_(q_in)           # fresh q every replay (rotated in place)
        st.fc.copy_(fc0)         # the same pages are taken again
        for l in range(L):
            pk.pa_kv_append_rope(kd[l], vd[l], qd[l], st.pool, st.bt, ctx, l, st.fl, st.fc, st.err)
            pk.pa_decode_attention(out[l], qd[l], st.pool, st.bt, ctx1, l, w.scale, ws, st.err)

    step()                        # eager warm-up outside the capture
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            step()
    torch.cuda.current_stream().wait_stream(side)

    ref = (pool, w.block_table, w.free_list, w.free_count)
    outs = []
    for l in range(L):
        q2, p2, b2, f2, c2, e = oracle.kv_append_rope(k[l], v[l], q[l], ref[0], ref[1],
                                                      w.context_lens, l, ref[2], ref[3])
        assert e == 0
        ref = (p2, b2, f2, c2)
        o_ref, e = oracle.decode_attention(q2, p2, b2, w.context_lens + 1, l)
        assert e == 0
        outs.append(o_ref)
    for rep in range(2):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert int(st.err.item()) == 0
        for l in range(L):
            assert_attention_close(host_f64(out[l]), outs[l], f"replay {rep} layer {l}")
        gp, gb, gf, gc, ge = st.host()
        assert np.array_equal(gb, ref[1]) and gc == ref[3]
        _compare_pools(gp, ref[0])


@pytest.mark.parametrize("path", ["split", "cluster", "seq"])
def test_attention_right_after_appends_that_open_pages(path):
    """Every sequence's new token opens a page, and each replay starts from
    the table as it was before the appends.  The allocation kernel lets the
    kernels after it start before it writes the new entries, so the
    attention's reads before its dependency wait may see the old -1 entries
    (the cluster kernel then streams its range again from the current
    values).  Whatever those early reads saw, every replay matches the
    oracle on both decode kernels."""
    import torch
    pk = _pk()
    pk.pa_decode_set_path({"split": pk.PA_DECODE_SPLIT, "cluster": pk.PA_DECODE_CLUSTER,
                           "seq": pk.PA_DECODE_SEQ}[path])
    try:
        ctx = np.array([16, 32, 48, 64, 96, 128, 160, 192, 256, 320, 384, 512], dtype=np.int32)
        n, L = len(ctx), 2
        mb = int(ctx.max()) // 16 + 2
        nbk = int(((ctx + 16) // 16).sum()) * L + 16
        rng = np.random.default_rng(21)
        w = wl.make_workload("tiny", seed=21, context_lens=ctx, n_layers=L, num_blocks=nbk,
                             max_blocks_per_seq=mb)
        pool = wl.make_pool_numpy(w, rng, poison=True)
        st = DevState(pool, w.block_table, w.free_list, w.free_count)
        k = wl.normal_bf16(rng, (L, n, N_KV, D))
        v = wl.normal_bf16(rng, (L, n, N_KV, D))
        q = wl.normal_bf16(rng, (L, n, N_Q, D))
        kd, vd, q_in = dev_bf16(k), dev_bf16(v), dev_bf16(q)
        qd = q_in.clone()
        bt0, fc0 = st.bt.clone(), st.fc.clone()
        ctxd, ctx1 = dev_i32(ctx), dev_i32(ctx + 1)
        out = torch.zeros((L, n, N_Q, D), dtype=torch.bfloat16, device="cuda")
        ws = workspace_for(n, mb)

        def step():
            st.bt.copy_(bt0)          # the new pages' entries are -1 again
            st.fc.copy_(fc0)
            qd.copy_(q_in)
            for l in range(L):
                pk.pa_kv_append_rope(kd[l], vd[l], qd[l], st.pool, st.bt, ctxd, l, st.fl, st.fc,
                                     st.err)
                pk.pa_decode_attention(out[l], qd[l], st.pool, st.bt, ctx1, l, w.scale, ws, st.err)

        step()
        torch.cuda.synchronize()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                step()
        torch.cuda.current_stream().wait_stream(side)

        ref = (pool, w.block_table, w.free_list, w.free_count)
        outs = []
        for l in range(L):
            q2, p2, b2, f2, c2, e = oracle.kv_append_rope(k[l], v[l], q[l], ref[0], ref[1], ctx, l,
                                                          ref[2], ref[3])
            assert e == 0
            ref = (p2, b2, f2, c2)
            o_ref, e = oracle.decode_attention(q2, p2, b2, ctx + 1, l)
            assert e == 0
            outs.append(o_ref)
        assert np.all(ref[1][np.arange(n), :, ctx // 16] >= 0)   # every sequence opened a page
        for rep in range(8):
            out.zero_()
            g.replay()
            torch.cuda.synchronize()
            assert int(st.err.item()) == 0
            for l in range(L):
                assert_attention_close(host_f64(out[l]), outs[l], f"replay {rep} layer {l}")
            gp, gb, gf, gc, ge = st.host()
            assert np.array_equal(gb, ref[1]) and gc == ref[3]
    finally:
        pk.pa_decode_set_path(pk.PA_DECODE_AUTO)
