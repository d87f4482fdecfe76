"""Pins of the CPU oracle's decode attention (no GPU).

Each test ties the oracle to something other than itself: a library
attention routine on contiguous K/V, closed forms, invariants, and special
cases.  Page: "An Inference Engine in 1,500 Lines of CUDA: The Map",
"What is in the box" (16-token pages + block_table, GQA ratio 4, online
softmax in pagedAttentionKernel).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import pa_workloads as wl

N_Q, N_KV, D, BS = 32, 8, 64, 16


def _scatter_contiguous(rng, ctx_list, num_blocks, max_blocks, n_layers=1, layer=0):
    """Draw contiguous K/V per sequence, then place them into a pool through a
    random block table (the inverse of the gather the oracle performs)."""
    pool = np.full((num_blocks, 2, BS, N_KV, D), wl.BF16_NAN, dtype=np.uint16)
    bt = np.full((len(ctx_list), n_layers, max_blocks), -1, dtype=np.int32)
    perm = rng.permutation(num_blocks)
    off = 0
    Ks, Vs = [], []
    for s, T in enumerate(ctx_list):
        K = wl.normal_bf16(rng, (T, N_KV, D))
        V = wl.normal_bf16(rng, (T, N_KV, D))
        nb = (T + BS - 1) // BS
        ids = perm[off:off + nb]
        off += nb
        bt[s, layer, :nb] = ids
        for t in range(T):
            pool[ids[t // BS], 0, t % BS] = K[t]
            pool[ids[t // BS], 1, t % BS] = V[t]
        Ks.append(K)
        Vs.append(V)
    return pool, bt, Ks, Vs


def _sdpa_reference(q_bits, K_bits, V_bits, scale):
    """torch's scaled_dot_product_attention in fp64 on one sequence's
    contiguous K/V, kv heads expanded to q heads by repeat_interleave."""
    q = torch.from_numpy(oracle.bf16_to_f64(q_bits))[:, None, :]            # [32][1][64]
    K = torch.from_numpy(oracle.bf16_to_f64(K_bits)).permute(1, 0, 2)       # [8][T][64]
    V = torch.from_numpy(oracle.bf16_to_f64(V_bits)).permute(1, 0, 2)
    K = K.repeat_interleave(N_Q // N_KV, dim=0)
    V = V.repeat_interleave(N_Q // N_KV, dim=0)
    o = torch.nn.functional.scaled_dot_product_attention(q, K, V, scale=scale)
    return o[:, 0, :].numpy()


@pytest.mark.parametrize("ctx_list", [[17, 14], [1, 16, 33, 100], [257]])
@pytest.mark.parametrize("q_scale", [1.0, 4.0])
def test_matches_library_attention_on_contiguous_kv(ctx_list, q_scale):
    rng = np.random.default_rng(11)
    num_blocks = sum((t + 15) // 16 for t in ctx_list) + 5
    max_blocks = max((t + 15) // 16 for t in ctx_list) + 1
    pool, bt, Ks, Vs = _scatter_contiguous(rng, ctx_list, num_blocks, max_blocks)
    q = wl.normal_bf16(rng, (len(ctx_list), N_Q, D), scale=q_scale)
    out, err = oracle.decode_attention(q, pool, bt, np.array(ctx_list), layer=0, scale=0.125)
    assert err == 0
    for s in range(len(ctx_list)):
        ref = _sdpa_reference(q[s], Ks[s], Vs[s], 0.125)
        np.testing.assert_allclose(out[s], ref, rtol=0, atol=1e-12)


def test_block_id_permutation_invariance():
    rng = np.random.default_rng(3)
    w = wl.make_workload("tiny", context_lens=[40, 7, 16], max_blocks_per_seq=4)
    pool = wl.make_pool_numpy(w, rng)
    q = wl.normal_bf16(rng, (w.num_seqs, N_Q, D))
    out0, e0 = oracle.decode_attention(q, pool, w.block_table, w.context_lens, 0)
    perm = rng.permutation(w.num_blocks)
    pool2 = np.empty_like(pool)
    pool2[perm] = pool
    bt2 = np.where(w.block_table >= 0, perm[np.maximum(w.block_table, 0)], -1).astype(np.int32)
    out1, e1 = oracle.decode_attention(q, pool2, bt2, w.context_lens, 0)
    assert e0 == 0 and e1 == 0
    assert np.array_equal(out0, out1)


def test_single_token_returns_its_value():
    rng = np.random.default_rng(5)
    w = wl.make_workload("tiny", context_lens=[1, 1])
    pool = wl.make_pool_numpy(w, rng)
    q = wl.normal_bf16(rng, (2, N_Q, D), scale=3.0)
    out, err = oracle.decode_attention(q, pool, w.block_table, w.context_lens, 0)
    assert err == 0
    for s in range(2):
        blk = w.block_table[s, 0, 0]
        v = oracle.bf16_to_f64(pool[blk, 1, 0])                 # [8][64]
        for h in range(N_Q):
            assert np.array_equal(out[s, h], v[h // 4])


def test_constant_value_rows_return_that_value_and_fix_gqa_mapping():
    """Every token of kv head g carries V = g + 1: any softmax weights give
    g + 1, so q head h must read exactly floor(h / 4) + 1."""
    rng = np.random.default_rng(6)
    w = wl.make_workload("tiny", context_lens=[33, 9])
    pool = wl.make_pool_numpy(w, rng)
    for g in range(N_KV):
        pool[:, 1, :, g, :] = wl.to_bf16_bits(np.full((), g + 1.0, dtype=np.float32))
    q = wl.normal_bf16(rng, (2, N_Q, D))
    out, err = oracle.decode_attention(q, pool, w.block_table, w.context_lens, 0)
    assert err == 0
    for h in range(N_Q):
        np.testing.assert_allclose(out[:, h], h // 4 + 1.0, rtol=0, atol=1e-13)


def test_zero_query_gives_uniform_mean():
    rng = np.random.default_rng(7)
    ctx = [23]
    pool, bt, Ks, Vs = _scatter_contiguous(rng, ctx, 4, 3)
    q = np.zeros((1, N_Q, D), dtype=np.uint16)
    out, _ = oracle.decode_attention(q, pool, bt, np.array(ctx), 0)
    mean = oracle.bf16_to_f64(Vs[0]).mean(axis=0)                # [8][64]
    for h in range(N_Q):
        np.testing.assert_allclose(out[0, h], mean[h // 4], rtol=0, atol=1e-13)


def test_two_token_weights_three_to_one():
    """q = e0, k1 = e0, k2 = 0 and scale = ln 3: scores ln3 and 0, so the
    weights are exactly 3/4 and 1/4."""
    pool = np.zeros((2, 2, BS, N_KV, D), dtype=np.uint16)
    one = wl.to_bf16_bits(np.float32(1.0))
    pool[0, 0, 0, :, 0] = one                   # k_0 = e0 for every kv head
    rng = np.random.default_rng(8)
    v = wl.normal_bf16(rng, (2, N_KV, D))
    pool[0, 1, 0] = v[0]
    pool[0, 1, 1] = v[1]
    bt = np.array([[[0, -1]]], dtype=np.int32)
    q = np.zeros((1, N_Q, D), dtype=np.uint16)
    q[0, :, 0] = one
    out, err = oracle.decode_attention(q, pool, bt, np.array([2]), 0, scale=math.log(3.0))
    assert err == 0
    vv = oracle.bf16_to_f64(v)
    for h in range(N_Q):
        np.testing.assert_allclose(out[0, h], 0.75 * vv[0, h // 4] + 0.25 * vv[1, h // 4],
                                   rtol=0, atol=1e-14)


def test_nan_poison_outside_context_never_reaches_output():
    rng = np.random.default_rng(9)
    w = wl.make_workload("tiny")
    pool = wl.make_pool_numpy(w, rng, poison=True)
    assert np.any(pool == wl.BF16_NAN)
    q = wl.normal_bf16(rng, (w.num_seqs, N_Q, D))
    out, err = oracle.decode_attention(q, pool, w.block_table, w.context_lens, 0)
    assert err == 0 and np.all(np.isfinite(out))


def test_empty_context_writes_zeros():
    rng = np.random.default_rng(10)
    w = wl.make_workload("tiny", context_lens=[0, 5])
    pool = wl.make_pool_numpy(w, rng)
    q = wl.normal_bf16(rng, (2, N_Q, D))
    out, err = oracle.decode_attention(q, pool, w.block_table, w.context_lens, 0)
    assert err == 0
    assert np.all(out[0] == 0.0) and np.all(np.isfinite(out[1]))


@pytest.mark.parametrize("T", [1, 16, 17, 100, 300])
def test_split_partials_merge_to_whole(T):
    """Split-context merge: partials over disjoint ranges, merged by
    rescaling to the common maximum, equal the softmax over the union."""
    rng = np.random.default_rng(T)
    pool, bt, Ks, Vs = _scatter_contiguous(rng, [T], (T + 15) // 16 + 2, (T + 15) // 16 + 1)
    q = wl.normal_bf16(rng, (1, N_Q, D), scale=4.0)
    whole, _ = oracle.decode_attention(q, pool, bt, np.array([T]), 0)
    for trial in range(3):
        cuts = np.sort(rng.choice(np.arange(1, T), size=min(T - 1, 1 + trial * 3), replace=False)) if T > 1 else []
        edges = [0, *[int(c) for c in cuts], T]
        for h in (0, 5, 31):
            ms, ls, accs = [], [], []
            for a, b in zip(edges[:-1], edges[1:]):
                m, l, acc, err = oracle.attention_partial(q[0, h], pool, bt[0, 0], h // 4, a, b)
                assert err == 0
                ms.append(m)
                ls.append(l)
                accs.append(acc)
            merged = oracle.merge_partials(ms, ls, np.stack(accs))
            np.testing.assert_allclose(merged, whole[0, h], rtol=0, atol=1e-12)


def test_bad_block_and_context_range_set_error_bits():
    rng = np.random.default_rng(12)
    w = wl.make_workload("tiny")
    pool = wl.make_pool_numpy(w, rng)
    q = wl.normal_bf16(rng, (w.num_seqs, N_Q, D))
    bt = w.block_table.copy()
    bt[0, 0, 1] = -1
    _, err = oracle.decode_attention(q, pool, bt, w.context_lens, 0)
    assert err & oracle.ERR_BAD_BLOCK
    bt = w.block_table.copy()
    bt[1, 0, 0] = w.num_blocks
    _, err = oracle.decode_attention(q, pool, bt, w.context_lens, 0)
    assert err & oracle.ERR_BAD_BLOCK
    ctx = w.context_lens.copy()
    ctx[0] = w.max_blocks_per_seq * 16 + 1
    _, err = oracle.decode_attention(q, pool, w.block_table, ctx, 0)
    assert err & oracle.ERR_CTX_RANGE


def test_layer_selects_its_table_row():
    """Two layers with different blocks: layer l must read only row l."""
    rng = np.random.default_rng(13)
    w = wl.make_workload("tiny", n_layers=2, context_lens=[20, 3], max_blocks_per_seq=3)
    pool = wl.make_pool_numpy(w, rng)
    q = wl.normal_bf16(rng, (2, N_Q, D))
    o0, _ = oracle.decode_attention(q, pool, w.block_table, w.context_lens, 0)
    o1, _ = oracle.decode_attention(q, pool, w.block_table, w.context_lens, 1)
    swapped = w.block_table[:, ::-1, :].copy()
    s0, _ = oracle.decode_attention(q, pool, swapped, w.context_lens, 1)
    assert np.array_equal(o0, s0)
    assert not np.allclose(o0, o1)
