"""Pins of the CPU oracle's KV append (allocation + RoPE + store) and free.

Page: "An Inference Engine in 1,500 Lines of CUDA: The Map", "The path of
one inference": the KV cache cut into 16-token blocks numbered by an iota
free list, and a block_table of -1 ("not assigned yet") per sequence and
layer.  The hand-worked fixture in tests/golden carries its own citation.
"""
import json
import os

import numpy as np
import pytest

import oracle
import pa_workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "append_free_worked_example.json")
N_Q, N_KV, D, BS = 32, 8, 64, 16


def _golden():
    return json.load(open(GOLDEN))


def test_worked_example_append_then_free():
    g = _golden()
    nbk = g["num_blocks"]
    bt = np.array(g["block_table"], dtype=np.int32)
    fl = np.array(g["free_list"], dtype=np.int32)
    fc = g["free_count"]
    rng = np.random.default_rng(0)
    pool = wl.normal_bf16(rng, (nbk, 2, BS, N_KV, D))
    ctx = np.array(g["append"]["context_lens"], dtype=np.int32)
    n = len(ctx)
    for layer in g["append"]["layers"]:
        k = wl.normal_bf16(rng, (n, N_KV, D))
        v = wl.normal_bf16(rng, (n, N_KV, D))
        _, pool, bt, fl, fc, err = oracle.kv_append_rope(k, v, None, pool, bt, ctx, layer, fl, fc)
        assert err == 0
        for s, (blk, slot) in enumerate(g["append"]["expect_slots"][str(layer)]):
            assert bt[s, layer, ctx[s] // BS] == blk
            assert ctx[s] % BS == slot
            assert np.array_equal(pool[blk, 1, slot], v[s])          # V is a copy
            if ctx[s] == 0:                                           # RoPE at 0 = identity
                assert np.array_equal(pool[blk, 0, slot], k[s])
    assert np.array_equal(bt, np.array(g["append"]["expect_block_table"]))
    assert fc == g["append"]["expect_free_count"]

    f = g["free"]
    bt2, fl2, fc2, err = oracle.free(f["seq_ids"], bt, f["context_lens"], fl, fc, nbk)
    assert err == f["expect_err"]
    assert np.array_equal(bt2, np.array(f["expect_block_table"]))
    assert fc2 == f["expect_free_count"]
    assert list(fl2[:fc2]) == f["expect_free_list_head"]


def test_worked_example_underflow():
    u = _golden()["underflow"]
    bt = np.array(u["block_table"], dtype=np.int32)
    n = bt.shape[0]
    rng = np.random.default_rng(1)
    pool = wl.normal_bf16(rng, (u["num_blocks"], 2, BS, N_KV, D))
    k = wl.normal_bf16(rng, (n, N_KV, D))
    v = wl.normal_bf16(rng, (n, N_KV, D))
    _, pool2, bt2, fl2, fc2, err = oracle.kv_append_rope(k, v, None, pool, bt, u["context_lens"], 0,
                                                         u["free_list"], u["free_count"])
    assert err == u["expect_err"]
    assert np.array_equal(bt2, np.array(u["expect_block_table"]))
    assert fc2 == u["expect_free_count"]


def test_rotated_k_and_q_are_rope_of_input_rounded_once():
    """The stored K is RoPE(k, pos) rounded to bf16 once; q likewise, in
    place.  Position pos = context length; slot = pos % 16."""
    rng = np.random.default_rng(2)
    w = wl.make_workload("tiny", context_lens=[17, 14, 31, 0], max_blocks_per_seq=3)
    pool = wl.make_pool_numpy(w, rng)
    n = w.num_seqs
    k = wl.normal_bf16(rng, (n, N_KV, D))
    v = wl.normal_bf16(rng, (n, N_KV, D))
    q = wl.normal_bf16(rng, (n, N_Q, D))
    inv = oracle.llama3_inv_freq()
    q2, pool2, bt2, fl2, fc2, err = oracle.kv_append_rope(k, v, q, pool, w.block_table,
                                                          w.context_lens, 0, w.free_list,
                                                          w.free_count)
    assert err == 0
    for s in range(n):
        pos = int(w.context_lens[s])
        blk = bt2[s, 0, pos // BS]
        for h in range(N_KV):
            ref = oracle.f64_to_bf16(oracle.rope_rotate(oracle.bf16_to_f64(k[s, h]), pos, inv))
            assert np.array_equal(pool2[blk, 0, pos % BS, h], ref)
        for h in (0, 17, 31):
            ref = oracle.f64_to_bf16(oracle.rope_rotate(oracle.bf16_to_f64(q[s, h]), pos, inv))
            assert np.array_equal(q2[s, h], ref)
    # everything else in the pool is untouched
    touched = np.zeros(pool.shape[:3], dtype=bool)
    for s in range(n):
        pos = int(w.context_lens[s])
        touched[bt2[s, 0, pos // BS], :, pos % BS] = True
    same = (pool2 == pool) | ((pool2 == wl.BF16_NAN) & (pool == wl.BF16_NAN))
    assert np.all(same[~touched])


@pytest.mark.parametrize("seed", [3, 4, 5])
def test_allocation_invariants_over_many_steps(seed):
    """Blocks are conserved (free + owned = pool), no block is owned twice
    within a layer, and only positions that start a page allocate."""
    rng = np.random.default_rng(seed)
    n, L, mb, nbk = 9, 3, 6, 80
    ctx = rng.integers(0, 40, size=n).astype(np.int32)
    bt = np.full((n, L, mb), -1, dtype=np.int32)
    fl = np.full(nbk, -1, dtype=np.int32)
    fl[:] = rng.permutation(nbk)
    fc = nbk
    # give each (seq, layer) its current blocks
    for layer in range(L):
        for s in range(n):
            for j in range((ctx[s] + 15) // 16):
                fc -= 1
                bt[s, layer, j] = fl[fc]
    pool = wl.normal_bf16(rng, (nbk, 2, BS, N_KV, D))
    for step in range(20):
        before = fc
        for layer in range(L):
            k = wl.normal_bf16(rng, (n, N_KV, D))
            v = wl.normal_bf16(rng, (n, N_KV, D))
            _, pool, bt, fl, fc, err = oracle.kv_append_rope(k, v, None, pool, bt, ctx, layer, fl, fc)
            assert err == 0
        starts = int(np.sum(ctx % 16 == 0))
        assert before - fc == starts * L
        ctx = ctx + 1
        owned = bt[bt >= 0]
        assert owned.size + fc == nbk
        assert len(set(owned.tolist()) | set(fl[:fc].tolist())) == nbk
        for layer in range(L):
            ids = bt[:, layer][bt[:, layer] >= 0]
            assert len(np.unique(ids)) == ids.size
        if step == 10:
            done = [1, 4]
            bt, fl, fc, err = oracle.free(done, bt, ctx, fl, fc, nbk)
            assert err == 0
            assert np.all(bt[done] == -1)
            ctx[done] = 0


def test_context_at_capacity_is_refused():
    rng = np.random.default_rng(6)
    w = wl.make_workload("tiny", context_lens=[64, 3], max_blocks_per_seq=4)
    pool = wl.make_pool_numpy(w, rng)
    k = wl.normal_bf16(rng, (2, N_KV, D))
    v = wl.normal_bf16(rng, (2, N_KV, D))
    _, pool2, bt2, _, fc2, err = oracle.kv_append_rope(k, v, None, pool, w.block_table,
                                                       w.context_lens, 0, w.free_list, w.free_count)
    assert err == oracle.ERR_CTX_RANGE
    assert fc2 == w.free_count
    assert np.array_equal(bt2[0], w.block_table[0])


def test_free_overflow_is_reported():
    bt = np.array([[[0, 1]], [[2, -1]]], dtype=np.int32)
    fl = np.array([3, -1, -1, -1], dtype=np.int32)
    bt2, fl2, fc2, err = oracle.free([0, 1], bt, [32, 5], fl, 3, 4)
    assert err == oracle.ERR_FREE_OVERFLOW
    assert fc2 == 4
    assert list(fl2) == [3, -1, -1, 0]
