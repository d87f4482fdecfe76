"""Shared test plumbing: numpy <-> torch transfers of bf16 bit patterns,
comparison metrics, and oracle runs on sampled sequences of device pools.
Holds no attention / RoPE / allocation arithmetic."""
from __future__ import annotations

import numpy as np

import pa_workloads as wl

# attention output tolerances against the fp64 oracle (bf16 output)
ATOL_MAX = 1e-2
ATOL_MEAN = 1e-3


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
    With output_rounding, each element may also carry the rounding of its
    exact value to bf16 (half an ulp at |ref|), which alone exceeds ATOL_MAX
    once |ref| >= 4: outputs that large come from rows attending over a few
    keys (the first tokens of a prompt)."""
    assert gpu_out_f64.shape == ref.shape, (gpu_out_f64.shape, ref.shape)
    assert np.all(np.isfinite(gpu_out_f64)), f"{what}: non-finite output"
    d = np.abs(gpu_out_f64 - ref)
    dm = d - bf16_half_ulp(ref) if output_rounding else d
    assert dm.max() <= ATOL_MAX, \
        f"{what}: max abs err {d.max():.3e} ({dm.max():.3e} beyond the output rounding)"
    assert d.mean() <= ATOL_MEAN, f"{what}: mean abs err {d.mean():.3e}"
    return float(d.max()), float(d.mean())


def workspace_for(n, max_blocks):
    import torch
    import paged_kv_cache_205_gb300 as pk
    return pk.decode_workspace(n, max_blocks)


def gather_for_oracle(pool_dev, block_table: np.ndarray, seqs, ctx, layer):
    """Copy the blocks that sequences `seqs` read in `layer` from a device pool
    [num_blocks][2][page][8][64] into a compact host pool, with the table rows
    renumbered to it."""
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
    return sub, bt
