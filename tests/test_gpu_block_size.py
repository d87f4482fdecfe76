"""GPU parity of the page-size entry points (pa_kv_append_rope_bt,
pa_decode_attention_bt, pa_free_bt, pa_prefill_append_rope_bt,
pa_prefill_attention_bt with 8- and 32-token pages) against the oracle run
with the same page size, through the C ABI.

Page: "An Inference Engine in 1,500 Lines of CUDA: The Map", "What is in the
box" (16-token pages + block_table; the page size taken as a tunable).
Tolerances as for 16-token pages: attention max 1e-2 / mean 1e-3 against
fp64; tables, free lists and V stores bit-exact; K within the RoPE bound.
"""
import json
import os

import numpy as np
import pytest

import oracle
import pa_workloads as wl
from helpers import (assert_attention_close, dev_bf16, dev_i32, gather_for_oracle, host_bits,
                     host_f64)
from test_gpu_append import DevState, _compare_pools, assert_rope_close
import test_gpu_prefill as tp

pytestmark = pytest.mark.gpu

N_Q, N_KV, D = 32, 8, 64
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "block_size_append_example.json")
PAGES = [8, 32]


def _pk():
    import paged_kv_cache_205_gb300 as pk
    return pk


@pytest.fixture(autouse=True)
def _reset_grid():
    _pk().pa_decode_set_grid_limit(0)
    yield
    _pk().pa_decode_set_grid_limit(0)


def _case(seed, ctx, page, q_scale=1.0, extra=6):
    """Pages of `page` tokens scattered over a NaN-poisoned pool."""
    rng = np.random.default_rng(seed)
    ctx = np.asarray(ctx, dtype=np.int32)
    pages = (ctx + page - 1) // page
    nb = int(pages.sum()) + extra
    mb = int(max(1, pages.max())) + 1
    pool = np.full((nb, 2, page, N_KV, D), wl.BF16_NAN, dtype=np.uint16)
    table = np.full((len(ctx), 1, mb), -1, dtype=np.int32)
    ids = rng.permutation(nb).astype(np.int32)
    off = 0
    for s, c in enumerate(ctx):
        for j in range(pages[s]):
            blk = ids[off]
            off += 1
            table[s, 0, j] = blk
            n = min(page, int(c) - j * page)
            pool[blk, :, :n] = wl.normal_bf16(rng, (2, n, N_KV, D))
    q = wl.normal_bf16(rng, (len(ctx), N_Q, D), scale=q_scale)
    return pool, table, ctx, q


def _gpu_attention(pool, table, ctx, q, grid=0):
    import torch
    pk = _pk()
    pk.pa_decode_set_grid_limit(grid)
    page = pool.shape[2]
    n = len(ctx)
    out = torch.full((n, N_Q, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = pk.decode_workspace(n, table.shape[2], block_tokens=page)
    pk.pa_decode_attention(out, dev_bf16(q), dev_bf16(pool), dev_i32(table), dev_i32(ctx), 0,
                           0.125, ws, err)
    torch.cuda.synchronize()
    return host_f64(out), int(err.item())


EDGE = [0, 1, 7, 8, 9, 15, 16, 17, 23, 24, 25, 31, 32, 33, 47, 63, 64, 65, 100, 2047]


@pytest.mark.parametrize("page", PAGES)
@pytest.mark.parametrize("grid", [0, 1, 5])
def test_edge_contexts_and_splits(page, grid):
    pool, table, ctx, q = _case(40 + page, EDGE, page, q_scale=2.0)
    ref, e_ref = oracle.decode_attention(q, pool, table, ctx, 0, block_tokens=page)
    out, err = _gpu_attention(pool, table, ctx, q, grid)
    assert err == e_ref == 0
    assert_attention_close(out, ref, f"page {page} grid {grid}")


@pytest.mark.parametrize("page", PAGES)
@pytest.mark.parametrize("n", [4, 20])
def test_per_head_cluster_kernel_forced(page, n):
    """The per-head cluster kernel forced (clusters of 8 CTAs at 4
    sequences, of 1 at 20): with 32-token pages a tile is half a page, with
    8-token pages two pages (four 1 KiB copies).  A page id out of range in
    one sequence is reported and its tokens dropped."""
    pk = _pk()
    ctx_list = EDGE[-n:]
    pool, table, ctx, q = _case(90 + page + n, ctx_list, page, q_scale=2.0)
    s_bad = len(ctx) - 2                    # a sequence of 65 tokens or more
    table[s_bad, 0, 1] = pool.shape[0] + 3
    pk.pa_decode_set_path(pk.PA_DECODE_CLUSTER)
    try:
        assert pk.pa_decode_kernel_for(n, page) == pk.PA_DECODE_CLUSTER
        ref, e_ref = oracle.decode_attention(q, pool, table, ctx, 0, block_tokens=page)
        out, err = _gpu_attention(pool, table, ctx, q)
    finally:
        pk.pa_decode_set_path(pk.PA_DECODE_AUTO)
    assert e_ref == oracle.ERR_BAD_BLOCK and err == e_ref
    assert_attention_close(out, ref, f"page {page}, {n} sequences, cluster kernel forced")


@pytest.mark.parametrize("page", PAGES)
def test_page_size_does_not_change_attention(page):
    """The same tokens under 8-, 16- and 32-token pages give the same output
    (up to rounding order) on the GPU too."""
    rng = np.random.default_rng(3)
    ctx = np.array([5, 40, 300, 1000], dtype=np.int32)
    K = [wl.normal_bf16(rng, (c, N_KV, D)) for c in ctx]
    V = [wl.normal_bf16(rng, (c, N_KV, D)) for c in ctx]
    q = wl.normal_bf16(rng, (len(ctx), N_Q, D))
    outs = {}
    for p in (16, page):
        pages = (ctx + p - 1) // p
        nb = int(pages.sum())
        pool = np.zeros((nb, 2, p, N_KV, D), dtype=np.uint16)
        table = np.full((len(ctx), 1, int(pages.max()) + 1), -1, np.int32)
        ids = rng.permutation(nb)
        off = 0
        for s, c in enumerate(ctx):
            for j in range(pages[s]):
                n = min(p, int(c) - j * p)
                table[s, 0, j] = ids[off]
                pool[ids[off], 0, :n] = K[s][j * p:j * p + n]
                pool[ids[off], 1, :n] = V[s][j * p:j * p + n]
                off += 1
        outs[p], err = _gpu_attention(pool, table, ctx, q)
        assert err == 0
    assert np.abs(outs[16] - outs[page]).max() <= 2e-2


def test_eight_token_pages_with_one_bad_page_in_a_tile():
    """With 8-token pages a 16-token tile spans two pages; a bad id in one of
    them drops only that page's tokens and is reported, as the oracle does."""
    pool, table, ctx, q = _case(9, [40, 40, 13], 8, extra=2)
    table[0, 0, 1] = pool.shape[0] + 3          # second page of the first tile
    table[1, 0, 2] = -1                         # first page of the second tile
    ref, e_ref = oracle.decode_attention(q, pool, table, ctx, 0, block_tokens=8)
    out, err = _gpu_attention(pool, table, ctx, q)
    assert e_ref == oracle.ERR_BAD_BLOCK and err == e_ref
    assert_attention_close(out, ref, "bad page")


@pytest.mark.parametrize("case", range(2))
def test_hand_worked_append(case):
    c = json.load(open(GOLDEN))["cases"][case]
    page = c["block_tokens"]
    rng = np.random.default_rng(case)
    n = len(c["context_lens"])
    nb = len(c["free_list"])
    pool = wl.normal_bf16(rng, (nb, 2, page, N_KV, D))
    k = wl.normal_bf16(rng, (n, N_KV, D))
    v = wl.normal_bf16(rng, (n, N_KV, D))
    bt = np.array(c["block_table"], np.int32)
    fl = np.array(c["free_list"], np.int32)
    st = DevState(pool, bt, fl, c["free_count"])
    _pk().pa_kv_append_rope(dev_bf16(k), dev_bf16(v), None, st.pool, st.bt,
                            dev_i32(c["context_lens"]), 0, st.fl, st.fc, st.err)
    gpool, gbt, gfl, gfc, gerr = st.host()
    assert gerr == 0
    assert np.array_equal(gbt, np.array(c["expect_block_table"]))
    assert gfc == c["expect_free_count"]
    for s, (blk, slot) in enumerate(c["expect_slots"]):
        assert np.array_equal(gpool[blk, 1, slot], v[s])
    _, p2, b2, f2, c2, e2 = oracle.kv_append_rope(k, v, None, pool, bt, c["context_lens"], 0, fl,
                                                  c["free_count"], block_tokens=page)
    _compare_pools(gpool, p2)


@pytest.mark.parametrize("page", PAGES)
def test_appending_decode_steps_then_free(page):
    """40 sequences append 70 tokens each, one decode step at a time (q
    rotated, attention over ctx + 1 after every append), then all are freed:
    tables, free list and pool bit-exact or within the RoPE bound, outputs
    within tolerance at every step, everything returned at the end."""
    import torch
    pk = _pk()
    rng = np.random.default_rng(page)
    n, steps = 40, 70
    start = rng.integers(0, 3 * page, size=n).astype(np.int32)
    end = start + steps
    mb = int((end.max() + page - 1) // page) + 1
    nb = int(((end + page - 1) // page).sum()) + 5
    pool = wl.normal_bf16(rng, (nb, 2, page, N_KV, D))
    bt = np.full((n, 1, mb), -1, np.int32)
    perm = rng.permutation(nb).astype(np.int32)
    top = nb
    for s in range(n):                               # pages of the starting contexts
        k0 = (int(start[s]) + page - 1) // page
        bt[s, 0, :k0] = perm[top - k0:top][::-1]
        top -= k0
    fl = perm.copy()
    fc = top
    st = DevState(pool, bt, fl, fc)
    ref_pool, ref_bt, ref_fl, ref_fc = pool, bt, fl, fc
    ws = pk.decode_workspace(n, mb, block_tokens=page)
    out = torch.empty((n, N_Q, D), dtype=torch.bfloat16, device="cuda")
    for t in range(steps):
        ctx = start + t
        k = wl.normal_bf16(rng, (n, N_KV, D))
        v = wl.normal_bf16(rng, (n, N_KV, D))
        q = wl.normal_bf16(rng, (n, N_Q, D))
        qd = dev_bf16(q)
        pk.pa_kv_append_rope(dev_bf16(k), dev_bf16(v), qd, st.pool, st.bt, dev_i32(ctx), 0,
                             st.fl, st.fc, st.err)
        pk.pa_decode_attention(out, qd, st.pool, st.bt, dev_i32(ctx + 1), 0, 0.125, ws, st.err)
        q2, ref_pool, ref_bt, ref_fl, ref_fc, e = oracle.kv_append_rope(
            k, v, q, ref_pool, ref_bt, ctx, 0, ref_fl, ref_fc, block_tokens=page)
        assert e == 0
        if t % 23 == 0 or t == steps - 1:
            gpool, gbt, gfl, gfc, gerr = st.host()
            assert gerr == 0 and gfc == ref_fc and np.array_equal(gbt, ref_bt)
            assert np.array_equal(gfl[:gfc], ref_fl[:ref_fc])
            _compare_pools(gpool, ref_pool)
            assert_rope_close(host_bits(qd), q2, f"q page {page} step {t}")
            # attention from the GPU's own pool and rotated q
            ref, e = oracle.decode_attention(host_bits(qd), gpool, gbt, ctx + 1, 0,
                                             block_tokens=page)
            assert e == 0
            assert_attention_close(host_f64(out), ref, f"page {page} step {t}")
    ids = np.arange(n, dtype=np.int32)
    pk.pa_free(dev_i32(ids), st.bt, dev_i32(end), st.fl, st.fc, nb, st.err, block_tokens=page)
    b3, f3, c3, e3 = oracle.free(ids, ref_bt, end, ref_fl, ref_fc, nb, block_tokens=page)
    gpool, gbt, gfl, gfc, gerr = st.host()
    assert gerr == e3 == 0 and gfc == c3 == nb
    assert np.array_equal(gbt, b3) and np.array_equal(gfl, f3)


@pytest.mark.parametrize("page", PAGES)
@pytest.mark.parametrize("name", ["llama1b", "ragged"])
def test_full_size_workloads_sampled(name, page):
    """The bench's workloads laid out in 8- or 32-token pages, launched as the
    bench launches them, sampled sequences against the oracle."""
    import torch
    pk = _pk()
    w = wl.make_workload(name, block_tokens=page)
    pool = wl.make_pool_torch(w, "cuda", seed=w.seed)
    ctx = w.context_lens
    rng = np.random.default_rng(w.seed + 1000)
    q = wl.normal_bf16(rng, (w.num_seqs, N_Q, D), scale=w.q_scale)
    order = np.argsort(ctx)
    sample = sorted({int(order[0]), int(order[-1]), *rng.choice(w.num_seqs, 3, replace=False).tolist()})
    qd, btd, ctxd = dev_bf16(q), dev_i32(w.block_table), dev_i32(ctx)
    out = torch.empty((w.num_seqs, N_Q, D), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = pk.decode_workspace(w.num_seqs, w.max_blocks_per_seq, block_tokens=page)
    for layer in (0, w.n_layers - 1):
        pk.pa_decode_attention(out, qd, pool, btd, ctxd, layer, w.scale, ws, err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        got = host_f64(out)
        sub, bt = gather_for_oracle(pool, w.block_table, sample, ctx, layer)
        ref, e = oracle.decode_attention(q[sample], sub, bt, ctx[sample], 0, scale=w.scale,
                                         block_tokens=page)
        assert e == 0
        assert_attention_close(got[sample], ref, f"{name} page {page} layer {layer}")
    del pool
    torch.cuda.empty_cache()



# ---------------------------------------------------------------- prefill
# pa_prefill_append_rope_bt / pa_prefill_attention_bt (the binding picks them
# from the pool's page dimension) against the oracle at the same page size.


@pytest.mark.parametrize("page", PAGES)
@pytest.mark.parametrize("ctx,lens", [
    ([0, 0], [17, 14]),                                # the page's two prompts
    ([0, 7, 8, 31, 100, 5], [1, 3, 16, 33, 40, 0]),    # page starts at 8 and 32, empty chunk
    ([2047, 0, 4000], [300, 1000, 96]),                # long prompts, chunks after long contexts
])
def test_prefill_append_matches_oracle(page, ctx, lens):
    tp._run_append_case(tp._append_case(40 + page + len(ctx), ctx, lens, page=page))


@pytest.mark.parametrize("page", PAGES)
def test_prefill_append_underflow_refuses_the_last_pages(page):
    c = tp._append_case(44 + page, [0, 10, 0], [40, 30, 20], spare=0, free_short=3, page=page)
    _, ref = tp._run_append_case(c)
    assert ref[5] & oracle.ERR_FREE_UNDERFLOW


@pytest.mark.parametrize("page", PAGES)
@pytest.mark.parametrize("ctx,lens,q_scale", [
    ([0, 0], [17, 14], 1.0),
    ([0, 3, 8, 100, 31, 7], [16, 45, 1, 64, 33, 0], 2.0),    # tile edges, ragged tails, empty chunk
    ([250, 0, 1000], [7, 130, 48], 3.0),                      # chunks after a cached context
])
def test_prefill_attention_matches_oracle(page, ctx, lens, q_scale):
    pool, bt, ctx, cu, q = tp._attention_state(60 + page + len(lens), ctx, lens, q_scale=q_scale,
                                               page=page)
    out, err = tp._gpu_prefill_attention(pool, bt, ctx, cu, q)
    ref, e_ref = oracle.prefill_attention(q, cu, pool, bt, ctx, 0, tp.SCALE, block_tokens=page)
    assert err == e_ref == 0
    tp._close(host_f64(out), ref, f"page={page} ctx={ctx.tolist()} lens={lens}")


@pytest.mark.parametrize("page", PAGES)
def test_prefill_attention_bad_page_is_dropped_and_reported(page):
    pool, bt, ctx, cu, q = tp._attention_state(70 + page, [60, 0], [10, 20], extra_blocks=2,
                                               page=page)
    bt[0, 0, 1] = pool.shape[0] + 7         # page 1 of sequence 0 lies outside the pool
    out, err = tp._gpu_prefill_attention(pool, bt, ctx, cu, q)
    ref, e_ref = oracle.prefill_attention(q, cu, pool, bt, ctx, 0, tp.SCALE, block_tokens=page)
    assert e_ref == oracle.ERR_BAD_BLOCK and err == e_ref
    tp._close(host_f64(out), ref, f"bad page, page={page}")


@pytest.mark.parametrize("page", PAGES)
def test_prefill_append_then_attention_chain(page):
    """Append the chunks (RoPE on k and q), then causal attention over the
    cache, on both sides, with pages of `page` tokens."""
    import torch
    c = tp._append_case(80 + page, [0, 37, 0, 16], [17, 40, 14, 1], n_layers=2, layer=0,
                        page=page)
    st = DevState(c["pool"], c["bt"], c["fl"], c["fc"])
    qd = tp._prefill_append(st, c["k"], c["v"], c["q"], c["cu"], c["ctx"], 0)
    out = torch.empty((qd.shape[0], N_Q, D), dtype=torch.bfloat16, device="cuda")
    _pk().pa_prefill_attention(out, qd, dev_i32(c["cu"]), st.pool, st.bt, dev_i32(c["ctx"]), 0,
                               tp.SCALE, st.err)
    q_ref, p_ref, b_ref, _, _, e_ref = oracle.prefill_append_rope(
        c["k"], c["v"], c["q"], c["cu"], c["pool"], c["bt"], c["ctx"], 0, c["fl"], c["fc"],
        block_tokens=page)
    ref, e2 = oracle.prefill_attention(q_ref, c["cu"], p_ref, b_ref, c["ctx"], 0, tp.SCALE,
                                       block_tokens=page)
    torch.cuda.synchronize()
    assert int(st.err.item()) == e_ref == e2 == 0
    tp._close(host_f64(out), ref, f"append -> attention, page={page}")
