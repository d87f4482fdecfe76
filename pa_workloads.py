"""Seeded synthetic workloads for the PagedAttention decode step.

This module only draws inputs: context lengths, block tables built by
popping block ids from a shuffled free list, and q / K / V / new-token
values drawn N(0, 1) and rounded to bf16.  It holds none of the attention,
RoPE or allocation arithmetic, so both the CPU oracle side and the CUDA side
of every test can take their inputs from it.

bf16 travels as raw ``uint16`` bit patterns in numpy; on the device the
same bits are viewed as ``torch.bfloat16``.

The five workloads follow the shapes of tiny-vllm's Llama 3.2 1B engine
("An Inference Engine in 1,500 Lines of CUDA: The Map", constants listing:
N_LAYERS = 16, BLOCK_SIZE = 16; "What is in the box": GQA ratio 4) with the
sizes the benchmark is specified on:

  tiny      1 layer, 2 sequences with contexts 17 and 14 (the two prompt
            lengths of the page), a 64-block pool, blocks from a seeded
            permutation, unused slots NaN-poisoned.
  llama1b   16 layers, 16 sequences, contexts uniform in [256, 2048],
            65,536-block pool, ids from a shuffled free list.
  pool2g    16 layers, 64 sequences x 4096, the 2 GiB 65,536-block pool; each
            layer's table is its own random 16,384-block subset of the pool.
  long32k   16 layers, 4 sequences x 32,768, 131,072-block pool, q scaled x4.
  ragged    16 layers, 256 sequences, contexts floor(exp(U(0, ln 8192)))
            clamped to [1, 8192], 262,144-block pool, shuffled free list; each
            layer first appends one token, then attends over ctx + 1.

Prefill workloads (make_prefill_workload) pack a prompt chunk per sequence:
the page's two prompts, eight fresh 2048-token prompts, and 512-token
chunks after 4096 cached tokens.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

N_Q = 32
N_KV = 8
HEAD_DIM = 64
BLOCK = 16
BLOCK_ELEMS = 2 * BLOCK * N_KV * HEAD_DIM      # one physical block, K and V
BF16_NAN = 0x7FC0


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = ((u >> 16) & 1) + 0x7FFF
    return ((u + rounding) >> 16).astype(np.uint16)


def normal_bf16(rng: np.random.Generator, shape, scale: float = 1.0) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if scale != 1.0:
        x = x * np.float32(scale)
    return to_bf16_bits(x)


@dataclasses.dataclass
class Workload:
    name: str
    n_layers: int
    context_lens: np.ndarray          # int32 [num_seqs], tokens cached before the step
    num_blocks: int
    max_blocks_per_seq: int
    block_table: np.ndarray           # int32 [num_seqs][n_layers][max_blocks_per_seq]
    free_list: np.ndarray             # int32 [num_blocks]; entries >= free_count unused
    free_count: int
    q_scale: float = 1.0
    append: bool = False              # step = append(pos=ctx) then attention over ctx+1
    scale: float = 0.125              # 1/sqrt(64)
    seed: int = 0
    block_tokens: int = BLOCK         # tokens per page (the page's BLOCK_SIZE, a tunable)

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def attn_context_lens(self) -> np.ndarray:
        """Tokens the attention of the step covers."""
        return (self.context_lens + (1 if self.append else 0)).astype(np.int32)

    def kv_bytes_per_layer(self) -> int:
        return int(self.attn_context_lens.astype(np.int64).sum()) * N_KV * HEAD_DIM * 2 * 2


def _assign_tables(rng, ctx, n_layers, num_blocks, max_blocks, per_layer_subset=None,
                   block_tokens=BLOCK):
    """Give every (sequence, layer) ceil(ctx/page) physical blocks popped from a
    shuffled free list.  With per_layer_subset, each layer instead draws its
    own random subset of the pool (blocks may then repeat across layers)."""
    n = len(ctx)
    nb = (ctx + block_tokens - 1) // block_tokens
    bt = np.full((n, n_layers, max_blocks), -1, dtype=np.int32)
    if per_layer_subset is None:
        free = rng.permutation(num_blocks).astype(np.int32)
        need = int(nb.sum()) * n_layers
        if need > num_blocks:
            raise ValueError(f"pool of {num_blocks} blocks cannot hold {need}")
        top = num_blocks
        for layer in range(n_layers):
            for s in range(n):
                k = int(nb[s])
                if k:
                    # pop k ids from the back of the shuffled free list
                    bt[s, layer, :k] = free[top - k:top][::-1]
                    top -= k
        free_list = free.copy()
        free_list[top:] = -1
        return bt, free_list, top
    for layer in range(n_layers):
        ids = rng.permutation(num_blocks)[: int(nb.sum())].astype(np.int32)
        off = 0
        for s in range(n):
            k = int(nb[s])
            bt[s, layer, :k] = ids[off:off + k]
            off += k
    free_list = np.full(num_blocks, -1, dtype=np.int32)
    return bt, free_list, 0


def make_workload(name: str, seed: int | None = None, block_tokens: int = BLOCK,
                  **over) -> Workload:
    """Table-level description of one of the five workloads (no tensors).
    With block_tokens other than 16 the pool keeps its bytes (16 / page
    times the blocks) and the tables hold pages of that many tokens."""
    seeds = {"tiny": 1, "llama1b": 2, "pool2g": 3, "long32k": 4, "ragged": 5, "pool8g": 3}
    if name == "pool8g":
        # pool2g's batch in a pool large enough for every layer's pages
        # (262,144 blocks = 8 GiB): no page is shared between layers
        over = dict(over)
        over.setdefault("num_blocks", 262144)
        over["alias"] = False
        return dataclasses.replace(make_workload("pool2g", seed=seed, block_tokens=block_tokens,
                                                 **over), name="pool8g")
    if seed is None:
        seed = seeds.get(name, 0)
    if block_tokens != BLOCK:
        if name == "tiny" or block_tokens not in (8, 32):
            raise ValueError("page sizes 8 and 32 are given for the full-size workloads")
        w = make_workload(name, seed=seed, **over)
        rng = np.random.default_rng(seed)
        ctx = w.context_lens
        nb_pool = w.num_blocks * BLOCK // block_tokens
        max_ctx = {"llama1b": 2048, "ragged": over.get("max_ctx", 8192)}.get(
            name, int(ctx.max()))
        mb = max_ctx // block_tokens + 1
        subset = True if (name == "pool2g" and over.get("alias", True)) else None
        bt, fl, fc = _assign_tables(rng, ctx, w.n_layers, nb_pool, mb, per_layer_subset=subset,
                                    block_tokens=block_tokens)
        return dataclasses.replace(w, num_blocks=nb_pool, max_blocks_per_seq=mb, block_table=bt,
                                   free_list=fl, free_count=fc, block_tokens=block_tokens)
    rng = np.random.default_rng(seed)
    if name == "tiny":
        ctx = np.array(over.get("context_lens", [17, 14]), dtype=np.int32)
        n_layers = over.get("n_layers", 1)
        num_blocks = over.get("num_blocks", 64)
        max_blocks = over.get("max_blocks_per_seq", 4)
        # tables = leading entries of one seeded permutation of the pool
        perm = rng.permutation(num_blocks).astype(np.int32)
        nb = (ctx + BLOCK - 1) // BLOCK
        bt = np.full((len(ctx), n_layers, max_blocks), -1, dtype=np.int32)
        off = 0
        for layer in range(n_layers):
            for s in range(len(ctx)):
                bt[s, layer, :nb[s]] = perm[off:off + nb[s]]
                off += int(nb[s])
        free_list = np.full(num_blocks, -1, dtype=np.int32)
        rest = perm[off:][::-1].copy()
        free_list[:len(rest)] = rest
        return Workload(name, n_layers, ctx, num_blocks, max_blocks, bt, free_list,
                        len(rest), seed=seed, append=over.get("append", False))
    if name == "llama1b":
        n = over.get("num_seqs", 16)
        ctx = rng.integers(256, 2048, size=n, endpoint=True).astype(np.int32)
        n_layers = over.get("n_layers", 16)
        num_blocks = over.get("num_blocks", 65536)
        max_blocks = 2048 // BLOCK + 1
        bt, fl, fc = _assign_tables(rng, ctx, n_layers, num_blocks, max_blocks)
        return Workload(name, n_layers, ctx, num_blocks, max_blocks, bt, fl, fc, seed=seed)
    if name == "pool2g":
        n = over.get("num_seqs", 64)
        ctx = np.full(n, over.get("ctx", 4096), dtype=np.int32)
        n_layers = over.get("n_layers", 16)
        num_blocks = over.get("num_blocks", 65536)
        max_blocks = int(ctx.max()) // BLOCK + 1
        alias = over.get("alias", True)
        bt, fl, fc = _assign_tables(rng, ctx, n_layers, num_blocks, max_blocks,
                                    per_layer_subset=True if alias else None)
        return Workload(name, n_layers, ctx, num_blocks, max_blocks, bt, fl, fc, seed=seed)
    if name == "long32k":
        n = over.get("num_seqs", 4)
        ctx = np.full(n, over.get("ctx", 32768), dtype=np.int32)
        n_layers = over.get("n_layers", 16)
        num_blocks = over.get("num_blocks", 131072)
        max_blocks = int(ctx.max()) // BLOCK + 1
        bt, fl, fc = _assign_tables(rng, ctx, n_layers, num_blocks, max_blocks)
        return Workload(name, n_layers, ctx, num_blocks, max_blocks, bt, fl, fc,
                        q_scale=4.0, seed=seed)
    if name == "ragged":
        n = over.get("num_seqs", 256)
        max_ctx = over.get("max_ctx", 8192)
        u = rng.uniform(0.0, math.log(max_ctx), size=n)
        ctx = np.clip(np.floor(np.exp(u)), 1, max_ctx).astype(np.int32)
        n_layers = over.get("n_layers", 16)
        num_blocks = over.get("num_blocks", 262144)
        max_blocks = max_ctx // BLOCK + 1
        bt, fl, fc = _assign_tables(rng, ctx, n_layers, num_blocks, max_blocks)
        return Workload(name, n_layers, ctx, num_blocks, max_blocks, bt, fl, fc,
                        append=True, seed=seed)
    raise ValueError(f"unknown workload {name!r}")


@dataclasses.dataclass
class PrefillWorkload:
    """Prompt chunks per sequence: chunk_lens[s] tokens appended after the
    context_lens[s] tokens already paged (0 for a fresh prompt)."""
    name: str
    n_layers: int
    context_lens: np.ndarray          # int32 [num_seqs], tokens cached before the chunk
    chunk_lens: np.ndarray            # int32 [num_seqs]
    num_blocks: int
    max_blocks_per_seq: int
    block_table: np.ndarray           # int32 [num_seqs][n_layers][max_blocks_per_seq]
    free_list: np.ndarray             # int32 [num_blocks]; entries >= free_count unused
    free_count: int
    scale: float = 0.125
    seed: int = 0
    block_tokens: int = BLOCK         # tokens per page

    @property
    def num_seqs(self) -> int:
        return int(self.chunk_lens.shape[0])

    @property
    def cu_tokens(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.chunk_lens.astype(np.int64))]).astype(np.int32)

    @property
    def total_tokens(self) -> int:
        return int(self.chunk_lens.astype(np.int64).sum())


PREFILL_WORKLOADS = {
    # name: (seed, layers, cached context per sequence, chunk per sequence, pool blocks)
    "prompts17_14": (6, 1, [0, 0], [17, 14], 64),
    "prefill8x2k": (7, 16, [0] * 8, [2048] * 8, 65536),
    "chunked32x512": (8, 16, [4096] * 32, [512] * 32, 262144),
}


def make_prefill_workload(name: str, seed: int | None = None,
                          block_tokens: int = BLOCK, layers: int = 0) -> PrefillWorkload:
    """prompts17_14: the page's two prompts (17 and 14 tokens), one layer.
    prefill8x2k: 8 fresh 2048-token prompts through 16 layers, 65,536-block
    pool.  chunked32x512: 32 sequences with 4096 tokens paged already append
    a 512-token chunk each, 16 layers, 262,144-block pool.  Cached pages are
    popped from a shuffled free list; the chunks' pages come from what is
    left of it.  With block_tokens other than 16 the pool keeps its bytes
    (16 / page times the blocks) and the tables hold pages of that many
    tokens.  layers > 0 keeps only the first `layers` layers, in a pool
    scaled down with them (the same work per layer call, a smaller device
    footprint)."""
    if block_tokens not in (8, 16, 32):
        raise ValueError("pages of 8, 16 or 32 tokens")
    sd, n_layers, ctx, lens, num_blocks = PREFILL_WORKLOADS[name]
    if layers > 0:
        if layers > n_layers:
            raise ValueError(f"{name} has {n_layers} layers")
        num_blocks = -(-num_blocks * layers // n_layers)
        n_layers = layers
    num_blocks = num_blocks * BLOCK // block_tokens
    rng = np.random.default_rng(sd if seed is None else seed)
    ctx = np.array(ctx, dtype=np.int32)
    lens = np.array(lens, dtype=np.int32)
    max_blocks = int(((ctx + lens + block_tokens - 1) // block_tokens).max()) + 1
    bt, free_list, top = _assign_tables(rng, ctx, n_layers, num_blocks, max_blocks,
                                        block_tokens=block_tokens)
    return PrefillWorkload(name, n_layers, ctx, lens, num_blocks, max_blocks, bt, free_list, top,
                           seed=sd if seed is None else seed, block_tokens=block_tokens)


def live_mask(w: Workload, context_lens=None) -> np.ndarray:
    """bool [num_blocks][page]: slots that hold a live token of some sequence."""
    ctx = w.context_lens if context_lens is None else context_lens
    B = w.block_tokens
    live = np.zeros((w.num_blocks, B), dtype=bool)
    for s in range(w.num_seqs):
        for layer in range(w.n_layers):
            row = w.block_table[s, layer]
            for t0 in range(0, int(ctx[s]), B):
                blk = row[t0 // B]
                live[blk, : min(B, int(ctx[s]) - t0)] = True
    return live


def make_pool_numpy(w: Workload, rng: np.random.Generator, poison: bool = True) -> np.ndarray:
    """Host pool [num_blocks][2][16][8][64] of bf16 bits; slots that hold no
    live token are NaN when poison is set."""
    pool = normal_bf16(rng, (w.num_blocks, 2, w.block_tokens, N_KV, HEAD_DIM))
    if poison:
        dead = ~live_mask(w)
        pool.transpose(0, 2, 1, 3, 4)[dead] = BF16_NAN
    return pool


def make_step_inputs(w: Workload, rng: np.random.Generator):
    """Per-layer q [L][n][32][64] and, for appending workloads, the new
    token's k and v [L][n][8][64], all bf16 bits."""
    L, n = w.n_layers, w.num_seqs
    q = normal_bf16(rng, (L, n, N_Q, HEAD_DIM), scale=w.q_scale)
    if not w.append:
        return q, None, None
    k_new = normal_bf16(rng, (L, n, N_KV, HEAD_DIM))
    v_new = normal_bf16(rng, (L, n, N_KV, HEAD_DIM))
    return q, k_new, v_new


def make_pool_torch(w: Workload, device, seed: int, poison: bool = True):
    """Device pool drawn N(0,1) in bf16 by torch's seeded CUDA generator (the
    full-size workloads are too large to draw on the host).  Returns a
    bf16 tensor [num_blocks][2][16][8][64]."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    B = w.block_tokens
    pool = torch.empty((w.num_blocks, 2, B, N_KV, HEAD_DIM), dtype=torch.bfloat16,
                       device=device)
    flat = pool.view(-1)
    chunk = 1 << 28
    for i in range(0, flat.numel(), chunk):
        seg = flat[i:i + chunk]
        seg.normal_(0.0, 1.0, generator=g)
    if poison:
        # NaN in the unused tail slots of every (sequence, layer)'s last block
        ctx = w.context_lens
        tail_blocks, tail_from = [], []
        for s in range(w.num_seqs):
            r = int(ctx[s]) % B
            if r == 0:
                continue
            for layer in range(w.n_layers):
                tail_blocks.append(int(w.block_table[s, layer, int(ctx[s]) // B]))
                tail_from.append(r)
        if tail_blocks:
            tb = torch.tensor(tail_blocks, device=device, dtype=torch.long)
            tf = torch.tensor(tail_from, device=device, dtype=torch.long)
            slot = torch.arange(B, device=device)
            mask = slot[None, :] >= tf[:, None]                  # [n_tail][page]
            nan = torch.tensor(float("nan"), dtype=torch.bfloat16, device=device)
            sub = pool[tb]                                       # [n_tail][2][16][8][64]
            sub = torch.where(mask[:, None, :, None, None], nan, sub)
            pool[tb] = sub
    return pool


def make_prefill_pool_torch(w: PrefillWorkload, device, seed: int):
    """Device pool for a prefill workload: N(0,1) bf16 from torch's seeded
    CUDA generator, with every block still on the free list set to NaN, so
    the slots past a chunk's last token in its last page read as NaN."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    pool = torch.empty((w.num_blocks, 2, w.block_tokens, N_KV, HEAD_DIM), dtype=torch.bfloat16,
                       device=device)
    flat = pool.view(-1)
    chunk = 1 << 28
    for i in range(0, flat.numel(), chunk):
        flat[i:i + chunk].normal_(0.0, 1.0, generator=g)
    free = torch.from_numpy(w.free_list[:w.free_count].astype(np.int64)).to(device)
    for i in range(0, free.numel(), 16384):
        pool[free[i:i + 16384]] = float("nan")
    return pool


# ------------------------------------------------------ continuous batching
@dataclasses.dataclass
class ServeWorkload:
    """Requests (id, prompt tokens, decode steps) fed to the serving loop."""
    name: str
    n_layers: int
    max_slots: int
    num_blocks: int
    max_blocks_per_seq: int
    prefill_budget: int               # prompt tokens prefilled per step at most
    requests: list                    # [(rid, prompt_len, decode_steps)]
    scale: float = 0.125
    seed: int = 0
    block_tokens: int = BLOCK         # tokens per page


SERVE_WORKLOADS = {
    # name: (seed, layers, slots, pool blocks, prefill budget, requests,
    #        prompt range, decode-step range)
    "serve_tiny": (9, 2, 3, 12, 32, 7, (1, 40), (1, 20)),
    "serve256": (10, 16, 64, 65536, 8192, 256, (16, 2048), (16, 512)),
}


def make_serve_workload(name: str, block_tokens: int = BLOCK) -> ServeWorkload:
    """serve_tiny: 7 requests through 3 slots of a 2-layer model with a
    12-page pool and 32 prompt tokens per step, so admissions wait for
    slots, for pages and for the prefill budget.  serve256: 256
    requests through 64 slots of the 16-layer model, prompts and decode
    lengths log-uniform in [16, 2048] and [16, 512], a 65,536-block pool and
    8192 prompt tokens per step.  With block_tokens other than 16 the pool
    keeps its bytes (16 / page times the pages)."""
    sd, L, slots, nb, budget, n_req, (p0, p1), (g0, g1) = SERVE_WORKLOADS[name]
    rng = np.random.default_rng(sd)
    p = np.floor(np.exp(rng.uniform(np.log(p0), np.log(p1 + 1), size=n_req))).astype(int)
    g = np.floor(np.exp(rng.uniform(np.log(g0), np.log(g1 + 1), size=n_req))).astype(int)
    p = np.clip(p, p0, p1)
    g = np.clip(g, g0, g1)
    reqs = [(i, int(p[i]), int(g[i])) for i in range(n_req)]
    if block_tokens not in (8, 16, 32):
        raise ValueError("pages of 8, 16 or 32 tokens")
    # the pool keeps its bytes: 16 / page times the pages
    nb = nb * BLOCK // block_tokens
    mb = int(max((a + b + block_tokens - 1) // block_tokens for _, a, b in reqs)) + 1
    return ServeWorkload(name, L, slots, nb, mb, budget, reqs, seed=sd, block_tokens=block_tokens)


def request_token_inputs(seed: int, rid: int, layer: int, positions):
    """q [n][32][64], k [n][8][64], v [n][8][64] bf16 bits of request rid's
    tokens at `positions` in `layer`: N(0,1) from a generator keyed by
    (seed, rid, layer, position), so any token can be drawn on its own."""
    positions = np.asarray(positions, dtype=np.int64).ravel()
    q = np.empty((len(positions), N_Q, HEAD_DIM), dtype=np.uint16)
    k = np.empty((len(positions), N_KV, HEAD_DIM), dtype=np.uint16)
    v = np.empty((len(positions), N_KV, HEAD_DIM), dtype=np.uint16)
    for i, pos in enumerate(positions):
        rng = np.random.default_rng([seed, rid, layer, int(pos)])
        q[i] = normal_bf16(rng, (N_Q, HEAD_DIM))
        k[i] = normal_bf16(rng, (N_KV, HEAD_DIM))
        v[i] = normal_bf16(rng, (N_KV, HEAD_DIM))
    return q, k, v
