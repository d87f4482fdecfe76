"""Pins of the CPU oracle's prefill path: a prompt chunk appended to the
paged cache (RoPE, pages in (sequence, position) order) and its causal
attention.  Page: "An Inference Engine in 1,500 Lines of CUDA: The Map",
"The path of one inference" (prefill is matrix x matrix over the whole
prompt; ropeKernel_llama3 rotates every prompt token)."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import pa_workloads as wl

N_Q, N_KV, D, BS = 32, 8, 64, 16
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "prefill_append_worked_example.json")


def _rand_chunk(rng, n_rows):
    return (wl.normal_bf16(rng, (n_rows, N_KV, D)), wl.normal_bf16(rng, (n_rows, N_KV, D)),
            wl.normal_bf16(rng, (n_rows, N_Q, D)))


def test_worked_example_page_order():
    g = json.load(open(GOLDEN))
    rng = np.random.default_rng(0)
    rows = g["cu_tokens"][-1]
    k, v, q = _rand_chunk(rng, rows)
    pool = wl.normal_bf16(rng, (g["num_blocks"], 2, BS, N_KV, D))
    q2, p2, b2, f2, c2, err = oracle.prefill_append_rope(
        k, v, q, g["cu_tokens"], pool, np.array(g["block_table"]), g["context_lens"], 0,
        g["free_list"], g["free_count"])
    assert err == g["expect_err"]
    assert np.array_equal(b2, np.array(g["expect_block_table"]))
    assert c2 == g["expect_free_count"]
    for r, (blk, slot) in enumerate(g["expect_slots"]):
        assert np.array_equal(p2[blk, 1, slot], v[r])          # V copied to the right slot


def _contiguous_case(rng, ctx, n, q_scale=1.0):
    """One sequence: contiguous K/V of ctx + n tokens scattered into a pool,
    the last n tokens being the chunk (already in the cache)."""
    T = ctx + n
    nb = (T + BS - 1) // BS
    perm = rng.permutation(nb + 3)
    K = wl.normal_bf16(rng, (T, N_KV, D))
    V = wl.normal_bf16(rng, (T, N_KV, D))
    pool = np.full((nb + 3, 2, BS, N_KV, D), wl.BF16_NAN, dtype=np.uint16)
    bt = np.full((1, 1, nb + 1), -1, dtype=np.int32)
    bt[0, 0, :nb] = perm[:nb]
    for t in range(T):
        pool[perm[t // BS], 0, t % BS] = K[t]
        pool[perm[t // BS], 1, t % BS] = V[t]
    q = wl.normal_bf16(rng, (n, N_Q, D), scale=q_scale)
    return K, V, pool, bt, q


@pytest.mark.parametrize("ctx,n", [(0, 1), (0, 17), (14, 3), (100, 40), (31, 33)])
def test_causal_attention_matches_library_sdpa(ctx, n):
    rng = np.random.default_rng(ctx * 100 + n)
    K, V, pool, bt, q = _contiguous_case(rng, ctx, n, q_scale=2.0)
    out, err = oracle.prefill_attention(q, [0, n], pool, bt, [ctx], 0)
    assert err == 0
    qt = torch.from_numpy(oracle.bf16_to_f64(q)).permute(1, 0, 2)               # [32][n][64]
    Kt = torch.from_numpy(oracle.bf16_to_f64(K)).permute(1, 0, 2).repeat_interleave(4, 0)
    Vt = torch.from_numpy(oracle.bf16_to_f64(V)).permute(1, 0, 2).repeat_interleave(4, 0)
    qpos = torch.arange(ctx, ctx + n)[:, None]
    kpos = torch.arange(ctx + n)[None, :]
    mask = kpos <= qpos                                                            # True = attend
    ref = torch.nn.functional.scaled_dot_product_attention(qt, Kt, Vt, attn_mask=mask, scale=0.125)
    np.testing.assert_allclose(out, ref.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)


def test_last_chunk_token_is_the_decode_step():
    rng = np.random.default_rng(3)
    ctx, n = 50, 9
    K, V, pool, bt, q = _contiguous_case(rng, ctx, n)
    out, _ = oracle.prefill_attention(q, [0, n], pool, bt, [ctx], 0)
    dec, _ = oracle.decode_attention(q[-1:], pool, bt, [ctx + n], 0)
    np.testing.assert_allclose(out[-1], dec[0], rtol=0, atol=1e-14)


def test_one_sequence_chunk_equals_successive_decode_appends():
    rng = np.random.default_rng(4)
    ctx0, n = 13, 40
    w = wl.make_workload("tiny", seed=4, context_lens=[ctx0], max_blocks_per_seq=6, num_blocks=20)
    pool = wl.make_pool_numpy(w, rng)
    k, v, q = _rand_chunk(rng, n)
    qa, pa, ba, fa, ca, ea = oracle.prefill_append_rope(k, v, q, [0, n], pool, w.block_table,
                                                        [ctx0], 0, w.free_list, w.free_count)
    assert ea == 0
    st = (pool, w.block_table, w.free_list, w.free_count)
    qs = []
    for i in range(n):
        q1, p1, b1, f1, c1, e1 = oracle.kv_append_rope(k[i:i + 1], v[i:i + 1], q[i:i + 1], st[0],
                                                       st[1], [ctx0 + i], 0, st[2], st[3])
        assert e1 == 0
        st = (p1, b1, f1, c1)
        qs.append(q1[0])
    assert np.array_equal(pa, st[0]) and np.array_equal(ba, st[1]) and ca == st[3]
    assert np.array_equal(qa, np.stack(qs))


def test_chunk_past_capacity_is_refused_whole():
    rng = np.random.default_rng(5)
    w = wl.make_workload("tiny", context_lens=[40, 3], max_blocks_per_seq=3, num_blocks=12)
    pool = wl.make_pool_numpy(w, rng)
    k, v, q = _rand_chunk(rng, 12)
    cu = [0, 9, 12]                      # 40 + 9 > 48: refused; 3 + 3 fits
    q2, p2, b2, f2, c2, err = oracle.prefill_append_rope(k, v, q, cu, pool, w.block_table,
                                                         w.context_lens, 0, w.free_list,
                                                         w.free_count)
    assert err == oracle.ERR_CTX_RANGE
    assert np.array_equal(q2[:9], q[:9])             # not rotated
    assert np.array_equal(b2[0], w.block_table[0]) and c2 == w.free_count


def test_underflow_in_the_middle_of_a_chunk():
    rng = np.random.default_rng(6)
    pool = wl.normal_bf16(rng, (4, 2, BS, N_KV, D))
    bt = np.full((1, 1, 4), -1, dtype=np.int32)
    k, v, q = _rand_chunk(rng, 20)
    q2, p2, b2, f2, c2, err = oracle.prefill_append_rope(k, v, None, [0, 20], pool, bt, [0], 0,
                                                         [3, -1, -1, -1], 1)
    assert err == oracle.ERR_FREE_UNDERFLOW
    assert list(b2[0, 0]) == [3, -1, -1, -1] and c2 == 0
    assert np.array_equal(p2[3, 1], v[:16])          # first page stored
    untouched = np.ones(4, dtype=bool)
    untouched[3] = False
    assert np.array_equal(p2[untouched], pool[untouched])
