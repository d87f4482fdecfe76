"""GPU parity of the prefill path (pa_prefill_append_rope,
pa_prefill_attention) against the CPU oracle, through the C ABI.

Page: "An Inference Engine in 1,500 Lines of CUDA: The Map", "The path of one
inference": prefill pushes a whole prompt through at once (the page's two
example prompts are 17 and 14 tokens long).  Tables, free lists, free counts,
V stores and untouched pool bytes are bit-exact; rotated K and q within the
fp32 rotation bound of the decode append; attention outputs within the decode
tolerance (max 1e-2 beyond the output's own bf16 rounding, mean 1e-3,
absolute against fp64): the first rows of a prompt attend over a few keys,
so their outputs reach the size of single V entries, where half a bf16 ulp
alone is up to 0.0156.
"""
import json
import os

import numpy as np
import pytest

import oracle
import pa_workloads as wl
from helpers import assert_attention_close, dev_bf16, dev_i32, host_bits, host_f64
from test_gpu_append import DevState, _compare_pools, assert_rope_close

pytestmark = pytest.mark.gpu

N_Q, N_KV, D, BS = 32, 8, 64, 16
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "prefill_append_worked_example.json")
SCALE = 0.125


def _pk():
    import paged_kv_cache_205_gb300 as pk
    return pk


def _close(got, ref, what):
    assert_attention_close(got, ref, what, output_rounding=True)


def _cu(lens):
    return np.concatenate([[0], np.cumsum(np.asarray(lens, dtype=np.int64))]).astype(np.int32)


def _chunk(rng, rows, q_scale=1.0):
    return (wl.normal_bf16(rng, (rows, N_KV, D)), wl.normal_bf16(rng, (rows, N_KV, D)),
            wl.normal_bf16(rng, (rows, N_Q, D), scale=q_scale))


def _prefill_append(st, k, v, q, cu, ctx, layer):
    qd = None if q is None else dev_bf16(q)
    _pk().pa_prefill_append_rope(dev_bf16(k), dev_bf16(v), qd, dev_i32(cu), st.pool, st.bt,
                                 dev_i32(ctx), layer, st.fl, st.fc, st.err)
    return qd


def _check_append(st, qd, ref):
    q_ref, p_ref, b_ref, f_ref, c_ref, e_ref = ref
    pool, bt, fl, fc, err = st.host()
    assert err == e_ref, (err, e_ref)
    assert np.array_equal(bt, b_ref)
    assert fc == c_ref
    assert np.array_equal(fl[:fc], f_ref[:fc])
    _compare_pools(pool, p_ref)
    if q_ref is not None:
        assert_rope_close(host_bits(qd), q_ref, "q")


def test_worked_example_page_order():
    g = json.load(open(GOLDEN))
    rng = np.random.default_rng(0)
    cu = np.array(g["cu_tokens"], dtype=np.int32)
    k, v, q = _chunk(rng, int(cu[-1]))
    pool = wl.normal_bf16(rng, (g["num_blocks"], 2, BS, N_KV, D))
    bt = np.array(g["block_table"], dtype=np.int32)
    fl = np.array(g["free_list"], dtype=np.int32)
    st = DevState(pool, bt, fl, g["free_count"])
    qd = _prefill_append(st, k, v, q, cu, g["context_lens"], 0)
    gpool, gbt, _, gfc, gerr = st.host()
    assert gerr == g["expect_err"]
    assert np.array_equal(gbt, np.array(g["expect_block_table"]))
    assert gfc == g["expect_free_count"]
    for r, (blk, slot) in enumerate(g["expect_slots"]):
        assert np.array_equal(gpool[blk, 1, slot], v[r])
    ref = oracle.prefill_append_rope(k, v, q, cu, pool, bt, g["context_lens"], 0, fl,
                                     g["free_count"])
    _check_append(st, qd, ref)


def _append_case(seed, ctx, lens, n_layers=2, layer=1, spare=4, free_short=0, with_q=True,
                 page=BS):
    """Sequences with `ctx` tokens already paged in `layer`, appending chunks
    of `lens` tokens; the free list holds what they need plus `spare`, minus
    `free_short`."""
    rng = np.random.default_rng(seed)
    ctx = np.asarray(ctx, dtype=np.int32)
    lens = np.asarray(lens, dtype=np.int32)
    old_pages = (ctx + page - 1) // page
    new_pages = (ctx + lens + page - 1) // page - old_pages
    mb = int(max(1, ((ctx + lens + page - 1) // page).max())) + 1
    nb = int(old_pages.sum() + new_pages.sum()) + spare
    perm = rng.permutation(nb).astype(np.int32)
    bt = np.full((len(ctx), n_layers, mb), -1, dtype=np.int32)
    used = 0
    for s in range(len(ctx)):
        bt[s, layer, :old_pages[s]] = perm[used:used + old_pages[s]]
        used += int(old_pages[s])
    free = perm[used:]
    fc = max(len(free) - free_short, 0)
    fl = np.full(nb, -1, dtype=np.int32)
    fl[:fc] = free[:fc]
    pool = wl.normal_bf16(rng, (nb, 2, page, N_KV, D))
    k, v, q = _chunk(rng, int(lens.sum()))
    return dict(pool=pool, bt=bt, fl=fl, fc=fc, ctx=ctx, cu=_cu(lens), k=k, v=v,
                q=q if with_q else None, layer=layer, page=page)


def _run_append_case(c):
    st = DevState(c["pool"], c["bt"], c["fl"], c["fc"])
    qd = _prefill_append(st, c["k"], c["v"], c["q"], c["cu"], c["ctx"], c["layer"])
    ref = oracle.prefill_append_rope(c["k"], c["v"], c["q"], c["cu"], c["pool"], c["bt"],
                                     c["ctx"], c["layer"], c["fl"], c["fc"],
                                     block_tokens=c["page"])
    _check_append(st, qd, ref)
    return st, ref


@pytest.mark.parametrize("ctx,lens", [
    ([0, 0], [17, 14]),                                # the page's two prompts
    ([0, 14, 16, 31, 100, 5], [1, 3, 16, 33, 40, 0]),  # page starts, full pages, empty chunk
    ([0] * 40, list(range(1, 41))),                    # many sequences, every tail length
    ([2047, 0, 4000], [300, 1000, 96]),                # long prompts, chunks after long contexts
])
def test_prefill_append_matches_oracle(ctx, lens):
    _run_append_case(_append_case(11 + len(ctx), ctx, lens))


def test_prefill_append_without_q():
    _run_append_case(_append_case(5, [3, 0], [29, 16], with_q=False))


def test_prefill_append_underflow_refuses_the_last_pages():
    c = _append_case(6, [0, 10, 0], [40, 30, 20], spare=0, free_short=3)
    _, ref = _run_append_case(c)
    assert ref[5] & oracle.ERR_FREE_UNDERFLOW


def test_prefill_append_refuses_a_chunk_past_the_table():
    c = _append_case(7, [10, 0, 20], [20, 17, 5])
    c["ctx"] = c["ctx"].copy()
    mb = c["bt"].shape[2]
    c["ctx"][1] = mb * BS - 10          # 17 tokens do not fit: the whole chunk is refused
    _, ref = _run_append_case(c)
    assert ref[5] & oracle.ERR_CTX_RANGE


# ---------------------------------------------------------------- attention
def _attention_state(seed, ctx, lens, n_layers=1, layer=0, q_scale=1.0, extra_blocks=5, page=BS):
    """Pages (of `page` tokens) of ctx + len tokens per sequence scattered
    over a NaN-poisoned pool (slots past a sequence's last token stay NaN)."""
    rng = np.random.default_rng(seed)
    ctx = np.asarray(ctx, dtype=np.int32)
    lens = np.asarray(lens, dtype=np.int32)
    total = ctx + lens
    pages = (total + page - 1) // page
    mb = int(max(1, pages.max())) + 1
    nb = int(pages.sum()) + extra_blocks
    perm = rng.permutation(nb).astype(np.int32)
    pool = np.full((nb, 2, page, N_KV, D), wl.BF16_NAN, dtype=np.uint16)
    bt = np.full((len(ctx), n_layers, mb), -1, dtype=np.int32)
    used = 0
    for s in range(len(ctx)):
        ids = perm[used:used + pages[s]]
        used += int(pages[s])
        bt[s, layer, :pages[s]] = ids
        t = int(total[s])
        kv = wl.normal_bf16(rng, (2, t, N_KV, D))
        full = t // page
        if full:
            pool[ids[:full], 0] = kv[0, :full * page].reshape(full, page, N_KV, D)
            pool[ids[:full], 1] = kv[1, :full * page].reshape(full, page, N_KV, D)
        if t % page:
            pool[ids[full], 0, :t % page] = kv[0, full * page:]
            pool[ids[full], 1, :t % page] = kv[1, full * page:]
    q = wl.normal_bf16(rng, (int(lens.sum()), N_Q, D), scale=q_scale)
    return pool, bt, ctx, _cu(lens), q


def _gpu_prefill_attention(pool, bt, ctx, cu, q, layer=0):
    import torch
    out = torch.full((q.shape[0], N_Q, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    _pk().pa_prefill_attention(out, dev_bf16(q), dev_i32(cu), dev_bf16(pool), dev_i32(bt),
                               dev_i32(ctx), layer, SCALE, err)
    torch.cuda.synchronize()
    return out, int(err.item())


@pytest.mark.parametrize("ctx,lens,q_scale", [
    ([0, 0], [17, 14], 1.0),                                  # the page's two prompts
    ([0], [1], 1.0),
    ([0, 3, 16, 100, 31, 7], [16, 45, 1, 64, 33, 0], 2.0),    # tile edges, ragged tails, empty chunk
    ([250, 0, 1000], [7, 130, 48], 3.0),                      # chunks after a cached context
    ([0] * 24, list(range(1, 25)), 1.0),                      # every tail length
])
def test_prefill_attention_matches_oracle(ctx, lens, q_scale):
    pool, bt, ctx, cu, q = _attention_state(100 + len(lens), ctx, lens, q_scale=q_scale)
    out, err = _gpu_prefill_attention(pool, bt, ctx, cu, q)
    ref, e_ref = oracle.prefill_attention(q, cu, pool, bt, ctx, 0, SCALE)
    assert err == e_ref == 0
    _close(host_f64(out), ref, f"ctx={ctx.tolist()} lens={lens}")


def test_prefill_attention_many_short_two_half_tiles():
    """200 prompts of 33..64 tokens: every (tile, kv head) item has both
    halves and a single, partial chunk, so each CTA runs some 10 items in a
    row in which one MMA warp zeroes V rows and hands the stage to the
    other."""
    lens = [33 + (i * 7) % 32 for i in range(200)]
    pool, bt, ctx, cu, q = _attention_state(13, [0] * 200, lens, q_scale=2.0, extra_blocks=3)
    out, err = _gpu_prefill_attention(pool, bt, ctx, cu, q)
    ref, e_ref = oracle.prefill_attention(q, cu, pool, bt, ctx, 0, SCALE)
    assert err == e_ref == 0
    _close(host_f64(out), ref, "short two-half tiles")


def test_prefill_attention_second_layer():
    pool, bt, ctx, cu, q = _attention_state(9, [40, 5], [20, 30], n_layers=3, layer=2)
    out, err = _gpu_prefill_attention(pool, bt, ctx, cu, q, layer=2)
    ref, e_ref = oracle.prefill_attention(q, cu, pool, bt, ctx, 2, SCALE)
    assert err == e_ref == 0
    _close(host_f64(out), ref, "layer 2")


def test_prefill_attention_bad_block_is_dropped_and_reported():
    pool, bt, ctx, cu, q = _attention_state(10, [60, 0], [10, 20], extra_blocks=2)
    bt[0, 0, 1] = pool.shape[0] + 7         # tokens 16..31 of sequence 0 are out of the pool
    out, err = _gpu_prefill_attention(pool, bt, ctx, cu, q)
    ref, e_ref = oracle.prefill_attention(q, cu, pool, bt, ctx, 0, SCALE)
    assert e_ref == oracle.ERR_BAD_BLOCK and err == e_ref
    _close(host_f64(out), ref, "bad block")


def test_prefill_attention_refuses_chunks_that_do_not_fit():
    pool, bt, ctx, cu, q = _attention_state(12, [10, 0, 30], [20, 17, 5])
    mb = bt.shape[2]
    ctx = ctx.copy()
    ctx[1] = mb * BS - 10
    out, err = _gpu_prefill_attention(pool, bt, ctx, cu, q)
    ref, e_ref = oracle.prefill_attention(q, cu, pool, bt, ctx, 0, SCALE)
    assert e_ref == oracle.ERR_CTX_RANGE and err == e_ref
    got = host_f64(out)
    keep = np.ones(q.shape[0], dtype=bool)
    keep[cu[1]:cu[2]] = False
    assert np.all(np.isnan(got[~keep])), "a refused chunk's rows were written"
    _close(got[keep], ref[keep], "accepted chunks")


def test_prefill_attention_refuses_rows_past_total_tokens():
    import torch
    pool, bt, ctx, cu, q = _attention_state(13, [0, 0], [20, 12])
    cu_bad = cu.copy()
    cu_bad[2] = cu[2] + 5                  # claims rows the buffers do not hold
    out = torch.full((q.shape[0], N_Q, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    qd, cud, poold = dev_bf16(q), dev_i32(cu_bad), dev_bf16(pool)
    btd, ctxd = dev_i32(bt), dev_i32(ctx)
    rc = _pk().library().pa_prefill_attention(
        out.data_ptr(), qd.data_ptr(), q.shape[0], cud.data_ptr(), poold.data_ptr(),
        pool.shape[0], btd.data_ptr(), 1, bt.shape[2], ctxd.data_ptr(), 2, 0, SCALE,
        err.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(err.item()) == oracle.ERR_CTX_RANGE
    got = host_f64(out)
    assert np.all(np.isnan(got[20:]))
    ref, _ = oracle.prefill_attention(q[:20], cu[:2], pool, bt[:1], ctx[:1], 0, SCALE)
    _close(got[:20], ref, "first chunk")


def test_prefill_append_then_attention_matches_oracle_chain():
    """The whole prefill of one layer: the chunk's K/V appended (with RoPE on
    k and q), then causal attention over the cache, on both sides."""
    import torch
    c = _append_case(21, [0, 37, 0, 16], [17, 40, 14, 1], n_layers=2, layer=0)
    st = DevState(c["pool"], c["bt"], c["fl"], c["fc"])
    qd = _prefill_append(st, c["k"], c["v"], c["q"], c["cu"], c["ctx"], 0)
    out = torch.empty((qd.shape[0], N_Q, D), dtype=torch.bfloat16, device="cuda")
    _pk().pa_prefill_attention(out, qd, dev_i32(c["cu"]), st.pool, st.bt, dev_i32(c["ctx"]), 0,
                               SCALE, st.err)
    q_ref, p_ref, b_ref, _, _, e_ref = oracle.prefill_append_rope(
        c["k"], c["v"], c["q"], c["cu"], c["pool"], c["bt"], c["ctx"], 0, c["fl"], c["fc"])
    ref, e2 = oracle.prefill_attention(q_ref, c["cu"], p_ref, b_ref, c["ctx"], 0, SCALE)
    torch.cuda.synchronize()
    assert int(st.err.item()) == e_ref == e2 == 0
    _close(host_f64(out), ref, "append -> attention")


def test_prefill_attention_long_prompt_sampled_rows():
    """Long prompts (several hundred query tiles): sampled rows against the
    oracle's decode attention over positions 0..pos, which a prefill row at
    position pos equals by definition."""
    lens = [2048, 1, 777, 3000]
    ctxs = [0, 4095, 1500, 0]
    pool, bt, ctx, cu, q = _attention_state(31, ctxs, lens, q_scale=2.0)
    out, err = _gpu_prefill_attention(pool, bt, ctx, cu, q)
    assert err == 0
    got = host_f64(out)
    assert np.all(np.isfinite(got))
    rng = np.random.default_rng(3)
    rows, seqs, poss = [], [], []
    for s in range(len(lens)):
        pick = set(rng.choice(lens[s], size=min(lens[s], 12), replace=False).tolist())
        pick |= {0, lens[s] - 1}
        for i in sorted(pick):
            rows.append(int(cu[s]) + i)
            seqs.append(s)
            poss.append(int(ctx[s]) + i)
    ref, e_ref = oracle.decode_attention(q[np.array(rows)], pool, bt[np.array(seqs)],
                                         np.array(poss, dtype=np.int32) + 1, 0, SCALE)
    assert e_ref == 0
    _close(got[np.array(rows)], ref, "sampled rows")


@pytest.mark.parametrize("name", ["prefill8x2k", "chunked32x512"])
def test_bench_prefill_workload_sampled(name):
    """The benchmark's prefill step at full size, launched as the benchmark
    launches it (every layer: append then attention, one stream): the
    appended pages hold no error, the rotated q rows match the oracle's RoPE,
    and sampled output rows match the oracle's attention over the pages the
    GPU wrote."""
    import torch
    from helpers import gather_for_oracle
    w = wl.make_prefill_workload(name)
    dev = torch.device("cuda")
    L, T = w.n_layers, w.total_tokens
    pool = wl.make_prefill_pool_torch(w, dev, seed=w.seed)
    bt = torch.from_numpy(w.block_table).to(dev)
    fl = torch.from_numpy(w.free_list).to(dev)
    fc = torch.tensor([w.free_count], dtype=torch.int32, device=dev)
    cu = torch.from_numpy(w.cu_tokens).to(dev)
    ctx = torch.from_numpy(w.context_lens).to(dev)
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed + 1)
    q = torch.randn((L, T, N_Q, D), generator=g, device=dev).to(torch.bfloat16)
    k = torch.randn((L, T, N_KV, D), generator=g, device=dev).to(torch.bfloat16)
    v = torch.randn((L, T, N_KV, D), generator=g, device=dev).to(torch.bfloat16)
    q_in = q.clone()
    out = torch.empty_like(q)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    for l in range(L):
        _pk().pa_prefill_append_rope(k[l], v[l], q[l], cu, pool, bt, ctx, l, fl, fc, err)
        _pk().pa_prefill_attention(out[l], q[l], cu, pool, bt, ctx, l, w.scale, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    n_pages = ((w.context_lens + w.chunk_lens + BS - 1) // BS - (w.context_lens + BS - 1) // BS)
    assert int(fc.item()) == w.free_count - int(n_pages.sum()) * L
    table = bt.cpu().numpy()
    ctx_after = (w.context_lens + w.chunk_lens).astype(np.int32)
    rng = np.random.default_rng(5)
    cu_h = w.cu_tokens
    for layer in (0, L - 1):
        seqs = sorted({0, w.num_seqs - 1, int(rng.integers(w.num_seqs))})
        sub, sub_bt = gather_for_oracle(pool, table, seqs, ctx_after, layer)
        rows, pos, which = [], [], []
        for i, s in enumerate(seqs):
            n = int(w.chunk_lens[s])
            for t in sorted({0, n - 1, *rng.integers(n, size=6).tolist()}):
                rows.append(int(cu_h[s]) + t)
                pos.append(int(w.context_lens[s]) + t)
                which.append(i)
        rows = np.array(rows)
        q_rot = host_bits(q[layer][torch.from_numpy(rows).to(dev)])
        q_orig = host_bits(q_in[layer][torch.from_numpy(rows).to(dev)])
        ref_q = np.stack([
            np.stack([oracle.f64_to_bf16(oracle.rope_rotate(oracle.bf16_to_f64(q_orig[i, h]),
                                                            pos[i]))
                      for h in range(N_Q)]) for i in range(len(rows))])
        assert_rope_close(q_rot, ref_q, f"{name} layer {layer} q")
        ref, e_ref = oracle.decode_attention(q_rot, sub, sub_bt[np.array(which)],
                                             np.array(pos, dtype=np.int32) + 1, 0, w.scale)
        assert e_ref == 0
        got = host_f64(out[layer][torch.from_numpy(rows).to(dev)])
        _close(got, ref, f"{name} layer {layer}")


@pytest.mark.parametrize("tiles", [4096, 4097])
def test_prefill_attention_at_and_past_the_sorted_tile_count(tiles):
    """2048 prompts of 65..129 tokens: 4096 query tiles (the most the kernel
    orders by weight) and 4097 (past it, the items go in tile order).  Every
    output row is written (none stays NaN) and sampled rows of every length
    match the oracle's attention over the same pages."""
    import torch
    from helpers import gather_for_oracle
    n = 2048
    lens = np.full(n, 65, dtype=np.int32)
    lens[n // 2:] = 64 + (np.arange(n - n // 2) % 2)      # 1 or 2 tiles alternating in the tail
    lens[: n // 2] = 65
    extra = tiles - int(((lens + 63) // 64).sum())
    assert 0 <= extra <= n
    lens[:extra] = 129                                     # 3 tiles each
    assert int(((lens + 63) // 64).sum()) == tiles
    ctx = np.zeros(n, dtype=np.int32)
    cu = _cu(lens)
    T = int(cu[-1])
    pages = (lens + BS - 1) // BS
    mb = int(pages.max())
    nb = int(pages.sum())
    dev = torch.device("cuda")
    g = torch.Generator(device=dev)
    g.manual_seed(4000 + tiles)
    pool = torch.randn((nb, 2, BS, N_KV, D), generator=g, device=dev).to(torch.bfloat16)
    q = torch.randn((T, N_Q, D), generator=g, device=dev).to(torch.bfloat16)
    bt = np.full((n, 1, mb), -1, dtype=np.int32)
    perm = np.random.default_rng(tiles).permutation(nb).astype(np.int32)
    start = np.concatenate([[0], np.cumsum(pages)])
    for s in range(n):
        bt[s, 0, :pages[s]] = perm[start[s]:start[s + 1]]
    out = torch.full((T, N_Q, D), float("nan"), dtype=torch.bfloat16, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    _pk().pa_prefill_attention(out, q, dev_i32(cu), pool, dev_i32(bt), dev_i32(ctx), 0, SCALE,
                               err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert bool(torch.isfinite(out.float()).all()), "rows left unwritten"
    rng = np.random.default_rng(tiles + 1)
    seqs = sorted({0, extra - 1 if extra else 1, n // 2, n - 2, n - 1,
                   *rng.integers(n, size=6).tolist()})
    sub, sub_bt = gather_for_oracle(pool, bt, seqs, lens, 0)
    rows, pos, which = [], [], []
    for i, s in enumerate(seqs):
        for t in sorted({0, 31, 32, 63, int(lens[s]) - 1, int(rng.integers(lens[s]))}):
            if t < lens[s]:
                rows.append(int(cu[s]) + t)
                pos.append(t)
                which.append(i)
    rows_t = torch.from_numpy(np.array(rows)).to(dev)
    ref, e_ref = oracle.decode_attention(host_bits(q[rows_t]), sub, sub_bt[np.array(which)],
                                         np.array(pos, dtype=np.int32) + 1, 0, SCALE)
    assert e_ref == 0
    _close(host_f64(out[rows_t]), ref, f"{tiles} tiles")
