"""Pins of the oracle with the page size as a tunable (8, 16 or 32 tokens
per block; the page's BLOCK_SIZE is 16).

Page: "An Inference Engine in 1,500 Lines of CUDA: The Map" ("What is in the
box": 16-token pages + block_table; "The path of one inference": the free
list and the -1 entries).  The pins: attention over the same tokens is the
same whatever the page size (bit for bit: the oracle sums in token order),
and equal to torch's attention on the contiguous tokens; hand-worked appends
at 8 and 32 tokens per page; token-by-token appends read back at every
position; free returns ceil(ctx / page) pages per layer; prefill attention
the same at every page size and equal to causal attention on the contiguous
tokens; a prefill append equal to single-token appends of the same tokens.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import pa_workloads as wl

N_Q, N_KV, D = 32, 8, 64
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "block_size_append_example.json")


def _paged(rng, K, V, ctxs, bt_tokens, extra=3):
    """Scatter contiguous K/V [seq][t][8][64] into a pool of bt_tokens pages
    through a shuffled table."""
    pages = [(c + bt_tokens - 1) // bt_tokens for c in ctxs]
    nb = sum(pages) + extra
    mb = max(max(pages), 1) + 1
    pool = np.full((nb, 2, bt_tokens, N_KV, D), wl.BF16_NAN, dtype=np.uint16)
    table = np.full((len(ctxs), 1, mb), -1, dtype=np.int32)
    ids = rng.permutation(nb)
    off = 0
    for s, c in enumerate(ctxs):
        for j in range(pages[s]):
            blk = int(ids[off])
            off += 1
            table[s, 0, j] = blk
            n = min(bt_tokens, c - j * bt_tokens)
            pool[blk, 0, :n] = K[s][j * bt_tokens:j * bt_tokens + n]
            pool[blk, 1, :n] = V[s][j * bt_tokens:j * bt_tokens + n]
    return pool, table


def test_attention_is_the_same_for_every_page_size():
    rng = np.random.default_rng(1)
    ctxs = [1, 7, 8, 9, 31, 32, 33, 100]
    K = [wl.normal_bf16(rng, (c, N_KV, D)) for c in ctxs]
    V = [wl.normal_bf16(rng, (c, N_KV, D)) for c in ctxs]
    q = wl.normal_bf16(rng, (len(ctxs), N_Q, D), scale=2.0)
    outs = {}
    for bt in (8, 16, 32):
        pool, table = _paged(rng, K, V, ctxs, bt)
        out, err = oracle.decode_attention(q, pool, table, np.array(ctxs, np.int32), 0,
                                           block_tokens=bt)
        assert err == 0
        outs[bt] = out
    assert np.array_equal(outs[8], outs[16]) and np.array_equal(outs[32], outs[16])
    # and the contiguous tokens through torch's attention
    for s, c in enumerate(ctxs):
        qs = torch.from_numpy(oracle.bf16_to_f64(q[s])).view(N_KV, 4, 1, D)
        ks = torch.from_numpy(oracle.bf16_to_f64(K[s])).permute(1, 0, 2).unsqueeze(1)
        vs = torch.from_numpy(oracle.bf16_to_f64(V[s])).permute(1, 0, 2).unsqueeze(1)
        ref = torch.nn.functional.scaled_dot_product_attention(
            qs, ks.expand(N_KV, 4, c, D), vs.expand(N_KV, 4, c, D), scale=0.125)
        assert np.allclose(outs[8][s], ref.reshape(N_Q, D).numpy(), atol=1e-12)


@pytest.mark.parametrize("case", range(2))
def test_hand_worked_append(case):
    c = json.load(open(GOLDEN))["cases"][case]
    bt = c["block_tokens"]
    rng = np.random.default_rng(case)
    n = len(c["context_lens"])
    nb = len(c["free_list"])
    pool = wl.normal_bf16(rng, (nb, 2, bt, N_KV, D))
    k = wl.normal_bf16(rng, (n, N_KV, D))
    v = wl.normal_bf16(rng, (n, N_KV, D))
    _, p2, b2, f2, c2, err = oracle.kv_append_rope(
        k, v, None, pool, np.array(c["block_table"], np.int32), c["context_lens"], 0,
        np.array(c["free_list"], np.int32), c["free_count"], block_tokens=bt)
    assert err == 0
    assert np.array_equal(b2, np.array(c["expect_block_table"]))
    assert c2 == c["expect_free_count"]
    for s, (blk, slot) in enumerate(c["expect_slots"]):
        assert np.array_equal(p2[blk, 1, slot], v[s])
    changed = np.argwhere((p2 != pool).reshape(nb * 2 * bt, -1).any(axis=1))
    assert len(changed) <= 2 * n          # only the K and V rows of the new tokens


@pytest.mark.parametrize("bt", [8, 32])
def test_token_by_token_appends_read_back(bt):
    """Appending 70 tokens one at a time puts token t's V at block
    table[t // bt], slot t % bt, and its K equal to the rotation of k_t."""
    rng = np.random.default_rng(bt)
    T = 70
    nb = (T + bt - 1) // bt + 2
    pool = np.zeros((nb, 2, bt, N_KV, D), dtype=np.uint16)
    table = np.full((1, 1, (T + bt - 1) // bt + 1), -1, np.int32)
    fl = rng.permutation(nb).astype(np.int32)
    fc = nb
    ks = wl.normal_bf16(rng, (T, 1, N_KV, D))
    vs = wl.normal_bf16(rng, (T, 1, N_KV, D))
    for t in range(T):
        _, pool, table, fl, fc, err = oracle.kv_append_rope(ks[t], vs[t], None, pool, table, [t],
                                                            0, fl, fc, block_tokens=bt)
        assert err == 0
    assert fc == nb - (T + bt - 1) // bt
    for t in range(T):
        blk = table[0, 0, t // bt]
        assert np.array_equal(pool[blk, 1, t % bt], vs[t, 0])
        rot = np.stack([oracle.f64_to_bf16(oracle.rope_rotate(oracle.bf16_to_f64(ks[t, 0, h]), t))
                        for h in range(N_KV)])
        assert np.array_equal(pool[blk, 0, t % bt], rot)


@pytest.mark.parametrize("bt", [8, 16, 32])
def test_free_returns_ceil_pages(bt):
    ctxs = [0, 1, bt, bt + 1, 5 * bt - 1]
    L = 2
    mb = 5
    need = [(c + bt - 1) // bt for c in ctxs]
    nb = sum(need) * L + 3
    table = np.full((len(ctxs), L, mb), -1, np.int32)
    ids = iter(range(nb))
    for s, k in enumerate(need):
        for layer in range(L):
            for j in range(k):
                table[s, layer, j] = next(ids)
    fl = np.full(nb, -1, np.int32)
    fl[:3] = [nb - 3, nb - 2, nb - 1]
    b2, f2, c2, err = oracle.free(np.arange(len(ctxs), dtype=np.int32), table, ctxs, fl, 3, nb,
                                  block_tokens=bt)
    assert err == 0 and c2 == nb and (b2 == -1).all()
    assert sorted(f2.tolist()) == list(range(nb))


# ---------------------------------------------------------------- prefill
def _cu(lens):
    return np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)


def test_prefill_attention_is_the_same_for_every_page_size():
    """Prompt chunks after cached contexts: the same tokens in pools of 8-,
    16- and 32-token pages give the same output bit for bit, equal to causal
    attention over the contiguous tokens."""
    rng = np.random.default_rng(3)
    ctxs, lens = [0, 5, 31, 40], [9, 20, 2, 33]
    tot = [c + n for c, n in zip(ctxs, lens)]
    K = [wl.normal_bf16(rng, (t, N_KV, D)) for t in tot]
    V = [wl.normal_bf16(rng, (t, N_KV, D)) for t in tot]
    q = wl.normal_bf16(rng, (sum(lens), N_Q, D), scale=2.0)
    cu = _cu(lens)
    outs = {}
    for bt in (8, 16, 32):
        pool, table = _paged(rng, K, V, tot, bt)
        out, err = oracle.prefill_attention(q, cu, pool, table, np.array(ctxs, np.int32), 0,
                                            block_tokens=bt)
        assert err == 0
        outs[bt] = out
    assert np.array_equal(outs[8], outs[16]) and np.array_equal(outs[32], outs[16])
    for s, (c, n) in enumerate(zip(ctxs, lens)):
        qs = torch.from_numpy(oracle.bf16_to_f64(q[cu[s]:cu[s + 1]]))      # [n][32][64]
        ks = torch.from_numpy(oracle.bf16_to_f64(K[s]))                      # [c+n][8][64]
        vs = torch.from_numpy(oracle.bf16_to_f64(V[s]))
        qh = qs.permute(1, 0, 2)                                             # [32][n][64]
        kh = ks.permute(1, 0, 2).repeat_interleave(4, dim=0)                 # [32][c+n][64]
        vh = vs.permute(1, 0, 2).repeat_interleave(4, dim=0)
        # row i sees keys 0 .. c + i
        mask = torch.arange(c + n)[None, :] <= (c + torch.arange(n))[:, None]
        ref = torch.nn.functional.scaled_dot_product_attention(qh, kh, vh, attn_mask=mask,
                                                               scale=0.125)
        assert np.allclose(outs[16][cu[s]:cu[s + 1]], ref.permute(1, 0, 2).numpy(), atol=1e-12)


@pytest.mark.parametrize("bt", [8, 16, 32])
def test_prefill_append_equals_token_by_token_appends(bt):
    """A chunk per sequence appended at once leaves the table, free list and
    pool exactly as single-token appends of the same tokens, sequence by
    sequence in position order, do."""
    rng = np.random.default_rng(10 + bt)
    ctxs, lens = [0, bt - 1, bt, 2 * bt + 3], [bt + 5, 1, 2 * bt, 3]
    mb = max((c + n + bt - 1) // bt for c, n in zip(ctxs, lens)) + 1
    old = [(c + bt - 1) // bt for c in ctxs]
    nb = sum(old) + sum((c + n + bt - 1) // bt - o for c, n, o in zip(ctxs, lens, old)) + 3
    ids = rng.permutation(nb).astype(np.int32)
    table = np.full((len(ctxs), 1, mb), -1, np.int32)
    used = 0
    for s, o in enumerate(old):
        table[s, 0, :o] = ids[used:used + o]
        used += o
    fl = np.full(nb, -1, np.int32)
    fl[:nb - used] = ids[used:]
    fc = nb - used
    pool = wl.normal_bf16(rng, (nb, 2, bt, N_KV, D))
    T = sum(lens)
    k = wl.normal_bf16(rng, (T, N_KV, D))
    v = wl.normal_bf16(rng, (T, N_KV, D))
    q = wl.normal_bf16(rng, (T, N_Q, D))
    cu = _cu(lens)
    q1, p1, b1, f1, c1, err = oracle.prefill_append_rope(k, v, q, cu, pool, table, ctxs, 0, fl, fc,
                                                         block_tokens=bt)
    assert err == 0
    p2, b2, f2, c2 = pool, table, fl, fc
    q2 = np.empty_like(q)
    for s, (c, n) in enumerate(zip(ctxs, lens)):
        for i in range(n):
            r = cu[s] + i
            one = [s]   # a one-sequence call on table row s
            qr, p2, bs, f2, c2, e = oracle.kv_append_rope(k[r:r + 1], v[r:r + 1], q[r:r + 1], p2,
                                                          b2[one], [c + i], 0, f2, c2,
                                                          block_tokens=bt)
            assert e == 0
            b2 = b2.copy()
            b2[s] = bs[0]
            q2[r] = qr[0]
    assert np.array_equal(b1, b2) and c1 == c2 and np.array_equal(f1[:c1], f2[:c2])
    assert np.array_equal(p1, p2) and np.array_equal(q1, q2)
    # pages opened per sequence: ceil((ctx + n) / bt) - ceil(ctx / bt)
    assert fc - c1 == sum((c + n + bt - 1) // bt - (c + bt - 1) // bt for c, n in zip(ctxs, lens))
