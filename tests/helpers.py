"""Shared test plumbing: numpy <-> torch transfers of bf16 bit patterns,
comparison metrics, and oracle runs on sampled sequences of device pools.
Holds no attention / RoPE / allocation arithmetic."""
from __future__ import annotations

import numpy as np

import pa_workloads as wl

# attention output tolerances against the fp64 oracle (bf16 output)
ATOL_MAX = 1e-2
ATOL_MEAN = 1e-3
# arithmetic error allowed on top of the output's own bf16 rounding where
# that rounding alone exceeds ATOL_MAX (|output| >= 4)
ROUNDING_SLACK = 1e-3


def dev_bf16(bits: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def dev_i32(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def host_bits(t) -> np.ndarray:
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host_f64(t) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def bf16_ordinal(bits: np.ndarray) -> np.ndarray:
    b = bits.astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def ulp_diff(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    return np.abs(bf16_ordinal(a_bits) - bf16_ordinal(b_bits))


def bf16_half_ulp(x: np.ndarray) -> np.ndarray:
    """Half the spacing of bf16 numbers at |x| (8 significant bits): the
    largest error of rounding x to bf16."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.ldexp(1.0, (e - 8).astype(np.int64))


def assert_attention_close(gpu_out_f64: np.ndarray, ref: np.ndarray, what: str = "",
                           output_rounding: bool = False):
    """Max and mean absolute error of a bf16 output against the fp64 oracle.

    Decode (default): each element within 1e-2, except where the bf16 format
    itself cannot hold that: an output with |ref| >= 4 (a short context whose
    output is about one V entry) lies up to half a bf16 ulp (1/64 at [4, 8))
    from the nearest bf16 number, so there the bound is that half ulp plus
    1e-3 of arithmetic.  Below 4 this is the plain 1e-2.
    With output_rounding (prefill, whose P enters the tensor-core MMA as bf16),
    each element may carry the rounding of its exact value on top of 1e-2."""
    assert gpu_out_f64.shape == ref.shape, (gpu_out_f64.shape, ref.shape)
    assert np.all(np.isfinite(gpu_out_f64)), f"{what}: non-finite output"
    d = np.abs(gpu_out_f64 - ref)
    if output_rounding:
        dm = d - bf16_half_ulp(ref)
    else:
        dm = d - np.maximum(0.0, bf16_half_ulp(ref) + ROUNDING_SLACK - ATOL_MAX)
    if dm.max() > ATOL_MAX:
        i = np.unravel_index(int(np.argmax(dm)), d.shape)
        raise AssertionError(f"{what}: max abs err {d.max():.3e} ({dm.max():.3e} beyond the "
                             f"bound) at {tuple(int(x) for x in i)}: got {gpu_out_f64[i]!r}, "
                             f"oracle {ref[i]!r}")
    assert d.mean() <= ATOL_MEAN, f"{what}: mean abs err {d.mean():.3e}"
    return float(d.max()), float(d.mean())


def workspace_for(n, max_blocks):
    import torch
    import paged_kv_cache_205_gb300 as pk
    return pk.decode_workspace(n, max_blocks)


def gather_for_oracle(pool_dev, block_table: np.ndarray, seqs, ctx, layer, return_ids=False):
    """Copy the blocks that sequences `seqs` read in `layer` from a device pool
    [num_blocks][2][page][8][64] into a compact host pool, with the table rows
    renumbered to it.  With return_ids, also the device block id of every
    compact block."""
    import torch
    page = int(pool_dev.shape[2])
    rows = []
    ids = []
    for s in seqs:
        nb = (int(ctx[s]) + page - 1) // page
        rows.append(block_table[s, layer, :nb])
        ids.extend(block_table[s, layer, :nb].tolist())
    uniq = sorted(set(ids))
    remap = {b: i for i, b in enumerate(uniq)}
    idx = torch.tensor(uniq, dtype=torch.long, device=pool_dev.device)
    sub = host_bits(pool_dev.index_select(0, idx)) if uniq else np.zeros((0, 2, page, 8, 64), np.uint16)
    mb = max(1, max((len(r) for r in rows), default=1))
    bt = np.full((len(seqs), 1, mb), -1, dtype=np.int32)
    for i, r in enumerate(rows):
        bt[i, 0, :len(r)] = [remap[b] for b in r.tolist()]
    if sub.shape[0] == 0:
        sub = np.zeros((1, 2, page, 8, 64), np.uint16)
    if return_ids:
        return sub, bt, np.asarray(uniq, dtype=np.int64)
    return sub, bt


def oracle_attention_threads(q, pool, block_table, context_lens, layer, scale=0.125,
                             block_tokens=16, threads=None):
    """oracle.decode_attention over all sequences, the sequences shared out
    over host threads (the oracle's C runs without the GIL and keeps no
    state between calls); the result is the same as one call."""
    import os
    from concurrent.futures import ThreadPoolExecutor

    import oracle
    n = int(np.asarray(context_lens).shape[0])
    out = np.zeros((n, 32, 64), dtype=np.float64)
    if n == 0:
        return out, 0
    threads = threads or max(1, min(16, os.cpu_count() or 1))
    parts = [p for p in np.array_split(np.arange(n), min(n, 4 * threads)) if len(p)]

    def run(idx):
        o, e = oracle.decode_attention(q[idx], pool, block_table[idx], context_lens[idx], layer,
                                       scale=scale, block_tokens=block_tokens)
        return idx, o, e

    err = 0
    with ThreadPoolExecutor(threads) as ex:
        for idx, o, e in ex.map(run, parts):
            out[idx] = o
            err |= e
    return out, err
