#!/usr/bin/env python3
"""Benchmark of the PagedAttention decode step (C ABI, GB300).

One step = the whole hot path over one batch: for each of the 16 layers,
(ragged workload only: pa_kv_append_rope of the new token, then)
pa_decode_attention.  Inputs live in HBM before the timed region.  Prints
one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle as the reference arm
  python bench.py --path prefill [--workload prefill8x2k|chunked32x512]
  python bench.py --path serve [--workload serve256]

With --path prefill one step is a whole prefill of one batch of prompt
chunks: for each of the 16 layers pa_prefill_append_rope (pages, RoPE on k
and q, K/V stores) then pa_prefill_attention (causal, over the pages); the
metric is prefill tokens/s and the roofline is the attention kernel's
tensor throughput.

Workloads (pa_workloads): llama1b (default: 16 layers, 16 sequences, context
U[256, 2048]), pool2g, long32k, ragged, tiny.

Under torchrun each rank runs an independent replica of the workload on its
own GPU (the path shards by sequence with no exchange); `value` is the
throughput summed over ranks, timed as the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import pa_workloads as wl  # noqa: E402

METRIC = "decode-attention HBM GB/s and % of GB300 peak; sequence-steps/sec"
N_Q, N_KV, D, BS = 32, 8, 64, 16
DESCRIPTIONS = {
    "tiny": "1 layer, 2 sequences with contexts 17 and 14, 64-block pool",
    "llama1b": "Llama-3.2-1B decode: 16 layers, 16 sequences, context U[256,2048], "
               "65,536-block pool, 32/8 heads, head_dim 64, 16-token bf16 blocks",
    "pool2g": "2 GiB pool (65,536 blocks), 16 layers, 64 sequences x 4096, per-layer random "
              "16,384-block subsets",
    "pool8g": "pool2g's batch (16 layers, 64 sequences x 4096) in an 8 GiB pool (262,144 "
              "blocks): every layer's pages distinct, no aliasing",
    "long32k": "16 layers, 4 sequences x 32,768, 131,072-block pool, q x4",
    "ragged": "continuous batching: 256 sequences, context log-U[1,8192], 262,144-block pool; "
              "per layer append (RoPE, pos = ctx) then attention over ctx+1",
}


# ------------------------------------------------------------ byte counts
def attention_bytes(ctx: np.ndarray, page: int = BS) -> int:
    """Algorithmic HBM bytes of one decode-attention call: K and V of every
    context token (2048 B per token over 8 kv heads), q and out (4096 B each
    per sequence), the block ids read and the context lengths."""
    ctx = ctx.astype(np.int64)
    return int(ctx.sum() * 2048 + len(ctx) * (4096 + 4096) + ((ctx + page - 1) // page).sum() * 4
               + len(ctx) * 4)


def append_bytes(n: int) -> int:
    """Algorithmic bytes of one append call with q: k_new, v_new read (1 KiB
    each), K and V written (1 KiB each), q read and written (4 KiB each),
    table entry and context length."""
    return n * (1024 * 4 + 4096 * 2 + 8)


# ------------------------------------------------------ replica aggregation
def aggregate_ranks(ms_per_step: float, e2e_s: float, bytes_per_step: int, seqs: int, dist=None):
    """Whole-job numbers over independent replicas: every rank ran the same
    workload on its own GPU; the job's step time is the slowest rank's, and
    the throughput counts the work of all ranks."""
    import torch
    world = dist.get_world_size() if dist is not None else 1
    t = torch.tensor([ms_per_step, e2e_s], dtype=torch.float64)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    ms, e2e = float(t[0]), float(t[1])
    return {
        "ms_per_step": ms,
        "e2e_s": e2e,
        "gbs": world * bytes_per_step / (ms / 1e3) / 1e9,
        "e2e_gbs": world * bytes_per_step / e2e / 1e9,
        "seq_steps_per_s": world * seqs / (ms / 1e3),
        "world": world,
    }


# --------------------------------------------------------- clock sampling
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None
        self.thread = None
        self.marking = False

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        t0 = time.time()
        while not self.rows and time.time() - t0 < 5:
            time.sleep(0.02)

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.rows.append((self.marking, parts))

    def mark(self, on: bool):
        self.marking = on

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = [p for m, p in self.rows if m] or [p for _, p in self.rows]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ------------------------------------------------------------- roofline
def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def measured_tensor_peak():
    """Dense bf16 TFLOP/s of the GB300s, burst (a kernel timed alone)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback"


SPLIT_SOURCES = ("pa_decode.cu", "pa_decode_tile.cuh", "pa_device.cuh")
PAIR_SOURCES = ("pa_decode_pair.cu", "pa_decode_tile.cuh", "pa_device.cuh")


def kernel_source_hash(sources=SPLIT_SOURCES) -> str:
    h = hashlib.sha256()
    for name in sources:
        with open(os.path.join(ROOT, "paged_kv_cache_205_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, kernel: str = "decode_split_kernel",
                     sources=SPLIT_SOURCES):
    """DRAM bytes per launch from the committed ncu summary, valid only while
    the kernel source hash recorded there matches the current source."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    mh = re.search(r"kernel source hash:\s*`?([0-9a-f]{16})", text)
    mt = re.search(r"dram bytes per launch:\s*([0-9.eE+]+)", text)
    if not mh or not mt or mh.group(1) != kernel_source_hash(sources):
        return None
    return float(mt.group(1))


# ------------------------------------------------- oracle (CPU baseline)
def oracle_unit(w: wl.Workload, s: int, layer: int, rng, max_tokens=None):
    """Host inputs of one (sequence, layer) of the workload, drawn with the
    same distributions, for the oracle: a compact pool holding only that
    sequence's blocks in a shuffled order."""
    ctx = int(w.attn_context_lens[s])
    if max_tokens is not None:
        ctx = max(1, min(ctx, int(max_tokens)))
    page = w.block_tokens
    nb = (ctx + page - 1) // page + 1
    pool = wl.normal_bf16(rng, (nb, 2, page, N_KV, D))
    bt = np.full((1, 1, nb), -1, dtype=np.int32)
    bt[0, 0, :] = rng.permutation(nb).astype(np.int32)
    q = wl.normal_bf16(rng, (1, N_Q, D), scale=w.q_scale)
    k = wl.normal_bf16(rng, (1, N_KV, D))
    v = wl.normal_bf16(rng, (1, N_KV, D))
    fl = np.zeros(4, dtype=np.int32)
    return dict(q=q, pool=pool, bt=bt, ctx=ctx, k=k, v=v, fl=fl)


def oracle_run_unit(u, w: wl.Workload):
    """One unit through the oracle: append (ragged) then attention.  Returns
    the algorithmic bytes it stands for."""
    import oracle
    ctx = u["ctx"]
    page = w.block_tokens
    if w.append:
        pos = ctx - 1   # the unit's context includes the appended token
        bt = u["bt"].copy()
        # the new token's page exists already unless it starts one
        oracle.kv_append_rope(u["k"], u["v"], u["q"], u["pool"], bt, np.array([pos]), 0,
                              u["fl"], 1 if pos % page == 0 else 0, block_tokens=page)
        oracle.decode_attention(u["q"], u["pool"], u["bt"], np.array([ctx]), 0, scale=w.scale,
                                block_tokens=page)
        return attention_bytes(np.array([ctx]), page) + append_bytes(1)
    oracle.decode_attention(u["q"], u["pool"], u["bt"], np.array([ctx]), 0, scale=w.scale,
                            block_tokens=page)
    return attention_bytes(np.array([ctx]), page)


def cpu_baseline(w: wl.Workload, budget_s: float = 12.0):
    """The oracle, single-threaded, over whole (sequence, layer) units of one
    step until the budget is spent."""
    import oracle
    oracle.build()
    rng = np.random.default_rng(w.seed + 77)
    units = [(s, l) for l in range(w.n_layers) for s in range(w.num_seqs)]
    t_total, nbytes, done = 0.0, 0, 0
    for s, l in units:
        u = oracle_unit(w, s, l, rng)
        t0 = time.perf_counter()
        nbytes += oracle_run_unit(u, w)
        t_total += time.perf_counter() - t0
        done += 1
        if t_total > budget_s:
            break
    seq_layers_per_s = done / t_total
    return {
        "value": nbytes / t_total / 1e9,
        "unit": "GB/s",
        "seq_steps_per_s": seq_layers_per_s / w.n_layers,
        "cores": 1,
        "kind": "oracle",
        "sample": f"{done} of {len(units)} (sequence, layer) units of one step "
                  f"({done / len(units):.0%}), {t_total:.1f} s, single-threaded C, fp64",
        "host_cores": os.cpu_count(),
    }


def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle
    oracle.build()
    w = wl.make_workload(args.workload, block_tokens=args.block_tokens)
    rng = np.random.default_rng(w.seed + 91)
    # size each step so the whole run stays within a few minutes
    per_step_budget = min(0.5, 150.0 / max(1, args.steps + args.warmup))
    probe = oracle_unit(w, 0, 0, rng, max_tokens=256)
    t0 = time.perf_counter()
    oracle_run_unit(probe, w)
    tok_rate = probe["ctx"] / max(time.perf_counter() - t0, 1e-6)
    max_tokens = max(16, int(per_step_budget * tok_rate))
    units = [(s, l) for l in range(w.n_layers) for s in range(w.num_seqs)]
    for i in range(args.warmup):
        s, l = units[i % len(units)]
        oracle_run_unit(oracle_unit(w, s, l, rng, max_tokens), w)
    t_total, nbytes, seq_layers = 0.0, 0, 0
    for i in range(args.steps):
        s, l = units[i % len(units)]
        u = oracle_unit(w, s, l, rng, max_tokens)
        t0 = time.perf_counter()
        nbytes += oracle_run_unit(u, w)
        t_total += time.perf_counter() - t0
        seq_layers += 1
    gbs = nbytes / t_total / 1e9
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": gbs,
        "unit": "GB/s",
        "n_gpus": args.gpus,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": t_total / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"{args.workload}: {DESCRIPTIONS[args.workload]}",
                   "block_tokens": w.block_tokens,
                   "sample_per_step": f"one (sequence, layer) unit, context capped at {max_tokens} tokens"},
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"{args.steps} units, one per step, single-threaded C (fp64)",
                         "host_cores": os.cpu_count()},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


# ------------------------------------------------------------- GPU arm
def attn_launches(cluster: bool) -> int:
    """Kernel launches of one pa_decode_attention call."""
    return 1 if cluster else 2


class DeviceStep:
    """Device-resident state of one workload and the step over it."""

    def __init__(self, w: wl.Workload, seed: int):
        import torch
        import paged_kv_cache_205_gb300 as pk
        self.pk = pk
        self.w = w
        dev = torch.device("cuda")
        L, n = w.n_layers, w.num_seqs
        self.pool = wl.make_pool_torch(w, dev, seed=seed, poison=True)
        self.bt = torch.from_numpy(w.block_table).to(dev)
        self.ctx_host = w.context_lens.astype(np.int32)
        self.ctx = torch.from_numpy(self.ctx_host).to(dev)
        self.ctx_attn = torch.from_numpy(w.attn_context_lens).to(dev)
        g = torch.Generator(device=dev)
        g.manual_seed(seed + 1)
        self.q = (torch.randn((L, n, N_Q, D), generator=g, device=dev) * w.q_scale).to(torch.bfloat16)
        self.out = torch.empty((L, n, N_Q, D), dtype=torch.bfloat16, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.ws = pk.decode_workspace(n, w.max_blocks_per_seq, block_tokens=w.block_tokens)
        if w.append:
            self.k_new = torch.randn((L, n, N_KV, D), generator=g, device=dev).to(torch.bfloat16)
            self.v_new = torch.randn((L, n, N_KV, D), generator=g, device=dev).to(torch.bfloat16)
            self.fl = torch.from_numpy(w.free_list).to(dev)
            self.fc0 = torch.tensor([w.free_count], dtype=torch.int32, device=dev)
            self.fc = self.fc0.clone()
        self.launches_per_step = L * (2 + (2 if w.append else 0))

    def layer(self, l, q=None, out=None):
        pk, w = self.pk, self.w
        q = self.q[l] if q is None else q
        out = self.out[l] if out is None else out
        if w.append:
            pk.pa_kv_append_rope(self.k_new[l], self.v_new[l], q, self.pool, self.bt, self.ctx, l,
                                 self.fl, self.fc, self.err)
        pk.pa_decode_attention(out, q, self.pool, self.bt, self.ctx_attn, l, w.scale, self.ws,
                               self.err)

    def step(self):
        if self.w.append:
            # every step allocates the same pages again: the free count is
            # restored first (steady state: blocks recycled between steps)
            self.fc.copy_(self.fc0)
        for l in range(self.w.n_layers):
            self.layer(l)

    def bytes_per_step(self) -> int:
        b = attention_bytes(self.w.attn_context_lens, self.w.block_tokens) * self.w.n_layers
        if self.w.append:
            b += append_bytes(self.w.num_seqs) * self.w.n_layers
        return b


# the other workloads the decode path is specified on, measured in the same
# process as the headline one and reported under "per_config"
PER_CONFIG = ("pool2g", "long32k", "ragged")
MIN_REPLAYS = 200   # roofline and end-to-end passes: at least this many replays


def decode_kernel_name(pk, kern) -> str:
    return {pk.PA_DECODE_CLUSTER: "pa_decode_attention (decode_pair_kernel: one thread-block "
                                  "cluster per (sequence, kv head))",
            pk.PA_DECODE_SEQ: "pa_decode_attention (decode_seq_kernel: one thread-block cluster "
                              "per sequence)"}.get(
        kern, "pa_decode_attention (decode_split_kernel + decode_merge_kernel)")


def decode_traffic(pk, workload, kern, block_tokens):
    """ncu DRAM bytes per launch of the workload's attention kernel, from the
    committed summary of that kernel (16-token pages only), or None."""
    if block_tokens != BS:
        return None
    if kern == pk.PA_DECODE_CLUSTER:
        return profiled_traffic(workload, "decode_pair_kernel", PAIR_SOURCES)
    if kern == pk.PA_DECODE_SEQ:
        return profiled_traffic(workload, "decode_seq_kernel", PAIR_SOURCES)
    return profiled_traffic(workload, "decode_split_kernel", SPLIT_SOURCES)


def decode_workload(name: str, block_tokens: int = BS, layers: int = 0) -> wl.Workload:
    """The named workload; with layers > 0 only its first `layers` layers, in
    a pool just large enough for their pages (the same contexts: a small
    device footprint for profiler captures of single launches)."""
    w = wl.make_workload(name, block_tokens=block_tokens)
    if layers <= 0 or layers >= w.n_layers:
        return w
    pages = int(((w.context_lens.astype(np.int64) + 1 + block_tokens - 1) // block_tokens).sum())
    nb = pages * layers + 1024
    if name == "pool2g":   # each layer draws its own subset of the pool
        nb = max(nb, int(((w.context_lens + block_tokens - 1) // block_tokens).sum()))
    return wl.make_workload(name, block_tokens=block_tokens, n_layers=layers, num_blocks=nb)


def measure_decode(args, w, rank, dist, sampler, k_steps):
    """Device step of one workload: the timed K steps (one graph of all
    layers per step), the attention launches alone (roofline), and the
    end-to-end step with host copies.  Returns the raw figures."""
    import torch
    st = DeviceStep(w, seed=w.seed + 1000 * rank)
    pk = st.pk
    pk.pa_decode_set_grid_limit(args.grid)
    if args.decode_kernel == "auto":
        # the choice the continuous batcher makes: from the batch's lengths
        path = pk.pa_decode_kernel_for_lengths(w.attn_context_lens, w.block_tokens)
    else:
        path = {"count": pk.PA_DECODE_AUTO, "split": pk.PA_DECODE_SPLIT,
                "cluster": pk.PA_DECODE_CLUSTER, "seq": pk.PA_DECODE_SEQ}[args.decode_kernel]
    pk.pa_decode_set_path(path)
    # which decode kernel the library runs for this batch
    kern = pk.pa_decode_kernel_for(w.num_seqs, w.block_tokens)
    cluster = kern in (pk.PA_DECODE_CLUSTER, pk.PA_DECODE_SEQ)
    st.launches_per_step = attn_launches(cluster) * w.n_layers + (2 * w.n_layers if w.append else 0)
    L, n = w.n_layers, w.num_seqs

    def barrier():
        if dist is not None:
            dist.barrier()

    def check(where):
        torch.cuda.synchronize()
        if int(st.err.item()) != 0:
            raise RuntimeError(f"device error bits {int(st.err.item())} {where} ({w.name})")

    # eager warm-up (also sets the library's per-device attributes)
    for _ in range(3):
        st.step()
    check("during eager warm-up")

    # one step = one CUDA graph of the layers' launches
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g_step = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g_step, stream=side):
            st.step()
    torch.cuda.current_stream().wait_stream(side)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        g_step.replay()
    check("during warm-up")

    barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    sampler.mark(True)
    e0.record(stream)
    for _ in range(k_steps):
        g_step.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    sampler.mark(False)
    barrier()
    ms = e0.elapsed_time(e1) / k_steps
    check("in the timed region")

    # dominant kernel: the attention launches of a step alone, back to back
    # in one graph, CUDA events on the replay stream
    g_attn = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g_attn, stream=side):
            for l in range(L):
                pk.pa_decode_attention(st.out[l], st.q[l], st.pool, st.bt, st.ctx_attn, l,
                                       w.scale, st.ws, st.err)
    torch.cuda.current_stream().wait_stream(side)
    k_roof = max(MIN_REPLAYS, min(k_steps, 500))
    for _ in range(3):
        g_attn.replay()
    torch.cuda.synchronize()
    a0 = torch.cuda.Event(enable_timing=True)
    a1 = torch.cuda.Event(enable_timing=True)
    sampler.mark(True)
    a0.record(stream)
    for _ in range(k_roof):
        g_attn.replay()
    a1.record(stream)
    torch.cuda.synchronize()
    sampler.mark(False)
    attn_ms = a0.elapsed_time(a1) / (k_roof * L)
    check("in the roofline pass")

    # end to end: every step's inputs from pinned host memory and its outputs
    # back, pipelined over two sets of device inputs and outputs.  The graph
    # of step i computes from one set while a side stream brings step i + 1's
    # inputs into the other set and sends step i - 1's outputs back from it,
    # so the layers' kernels keep their dependent-launch chain and the copies
    # run beside them (one graph per set; replays on one stream follow each
    # other, so a set is free when its turn comes).  The first step's inputs
    # come in before the timed region, the last step's outputs go back
    # inside it: one input copy and one output copy per timed step.
    h_q = torch.empty((L, n, N_Q, D), dtype=torch.bfloat16).pin_memory()
    h_q.copy_(st.q.cpu())
    h_ctx = torch.from_numpy(w.attn_context_lens.copy()).pin_memory()
    h_out = torch.empty((L, n, N_Q, D), dtype=torch.bfloat16).pin_memory()
    h_kv = None
    if w.append:
        h_kv = (st.k_new.cpu().pin_memory(), st.v_new.cpu().pin_memory(),
                torch.from_numpy(st.ctx_host.copy()).pin_memory())
    sets = []
    for _ in range(2):
        ds = {"q": torch.empty_like(st.q), "out": torch.empty_like(st.out),
              "ctx_attn": torch.empty_like(st.ctx_attn)}
        if w.append:
            ds.update(k=torch.empty_like(st.k_new), v=torch.empty_like(st.v_new),
                      ctx=torch.empty_like(st.ctx))
        sets.append(ds)
    s_side = torch.cuda.Stream()

    def fill(ds):
        ds["ctx_attn"].copy_(h_ctx, non_blocking=True)
        ds["q"].copy_(h_q, non_blocking=True)
        if w.append:
            ds["ctx"].copy_(h_kv[2], non_blocking=True)
            ds["k"].copy_(h_kv[0], non_blocking=True)
            ds["v"].copy_(h_kv[1], non_blocking=True)

    def e2e_step(ds, other):
        cur = torch.cuda.current_stream()
        s_side.wait_stream(cur)
        with torch.cuda.stream(s_side):
            h_out.copy_(other["out"], non_blocking=True)   # the previous step's result
            fill(other)                                     # the next step's inputs
        if w.append:
            st.fc.copy_(st.fc0)
        for l in range(L):
            if w.append:
                pk.pa_kv_append_rope(ds["k"][l], ds["v"][l], ds["q"][l], st.pool, st.bt, ds["ctx"],
                                     l, st.fl, st.fc, st.err)
            pk.pa_decode_attention(ds["out"][l], ds["q"][l], st.pool, st.bt, ds["ctx_attn"], l,
                                   w.scale, st.ws, st.err)
        cur.wait_stream(s_side)

    graphs = []
    for i in range(2):
        g_i = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(g_i, stream=side):
                e2e_step(sets[i], sets[1 - i])
        torch.cuda.current_stream().wait_stream(side)
        graphs.append(g_i)
    k_e2e = max(MIN_REPLAYS, min(k_steps, 500))
    k_e2e += k_e2e % 2
    fill(sets[0])
    for i in range(4):
        graphs[i % 2].replay()
    torch.cuda.synchronize()
    barrier()
    sampler.mark(True)
    t0 = time.perf_counter()
    for i in range(k_e2e):
        graphs[i % 2].replay()
    h_out.copy_(sets[1]["out"], non_blocking=True)
    torch.cuda.synchronize()
    e2e_s = (time.perf_counter() - t0) / k_e2e
    sampler.mark(False)
    check("in the end-to-end pass")
    h2d = h_q.numel() * 2 + h_ctx.numel() * 4
    if w.append:
        h2d += h_kv[0].numel() * 2 + h_kv[1].numel() * 2 + h_kv[2].numel() * 4
    d2h = h_out.numel() * 2
    res = dict(ms=ms, e2e_s=e2e_s, attn_ms=attn_ms, k_roof=k_roof, k_e2e=k_e2e, h2d=h2d, d2h=d2h,
               bytes_step=st.bytes_per_step(), kern=kern, launches_per_step=st.launches_per_step)
    del st, g_step, g_attn, graphs, sets
    pk.pa_decode_set_path(pk.PA_DECODE_AUTO)
    pk.pa_decode_set_grid_limit(0)
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def decode_roofline(pk, w, workload, r, peak, peak_kind):
    attn_bytes = attention_bytes(w.attn_context_lens, w.block_tokens)
    achieved = attn_bytes / (r["attn_ms"] / 1e3) / 1e9
    return {
        "bound": "hbm",
        "kernel": decode_kernel_name(pk, r["kern"]),
        "achieved": achieved,
        "peak": peak,
        "peak_kind": f"{peak_kind} HBM copy bandwidth",
        "unit": "GB/s",
        "frac": achieved / peak,
        # (the committed ncu summaries are of 16-token pages)
        "traffic": decode_traffic(pk, workload, r["kern"], w.block_tokens),
        "bytes_per_launch": attn_bytes,
        "ms_per_launch": r["attn_ms"],
        "timing": f"{r['k_roof']} replays of a graph of the {w.n_layers} attention launches, "
                  "events on the replay stream",
    }


def decode_e2e(agg, r):
    return {
        "value": agg["e2e_gbs"],
        "unit": "GB/s",
        "h2d_bytes_per_step": r["h2d"],
        "d2h_bytes_per_step": r["d2h"],
        "ms_per_step": agg["e2e_s"] * 1e3,
        "how": f"pinned H2D of the step inputs + the step + D2H of all outputs, pipelined over two "
               f"sets of device buffers (step i's graph brings step i+1's inputs in and sends step "
               f"i-1's outputs back on a side stream beside its kernels), {r['k_e2e']} steps, one "
               f"graph replay each, the last outputs copied inside the timed region, host wall "
               f"clock",
    }


def run_gpu(args, rank, world, dist):
    import torch
    import paged_kv_cache_205_gb300 as pk
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    w = decode_workload(args.workload, args.block_tokens, args.layers)
    sampler = ClockSampler(local)
    sampler.start()
    r = measure_decode(args, w, rank, dist, sampler, args.steps)
    agg = aggregate_ranks(r["ms"], r["e2e_s"], r["bytes_step"], w.num_seqs, dist)
    # the other specified workloads, in the same process and launch configuration
    others = []
    if (args.per_config and args.workload == "llama1b" and args.block_tokens == BS
            and args.decode_kernel == "auto" and args.grid == 0 and args.layers == 0):
        for name in PER_CONFIG:
            wo = wl.make_workload(name)
            ro = measure_decode(args, wo, rank, dist, sampler, args.steps)
            others.append((name, wo, ro,
                           aggregate_ranks(ro["ms"], ro["e2e_s"], ro["bytes_step"], wo.num_seqs,
                                           dist)))
    sampler.stop()
    if rank != 0:
        return

    peak, peak_kind = measured_hbm_peak()
    ctx_a = w.attn_context_lens.astype(np.int64)
    page_fill = float(ctx_a.sum() / (((ctx_a + w.block_tokens - 1) // w.block_tokens).sum()
                                     * w.block_tokens))
    line = {
        "metric": METRIC,
        "value": agg["gbs"],
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": agg["ms_per_step"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "accumulate": "fp32",
        "data": "synthetic",
        "pct_of_peak": 100.0 * agg["gbs"] / (peak * world),
        "seq_steps_per_s": agg["seq_steps_per_s"],
        "config": {
            "workload": f"{args.workload}: {DESCRIPTIONS[args.workload]}" +
                        (f" (first {w.n_layers} layers only, {w.num_blocks}-block pool)"
                         if args.layers else ""),
            "num_seqs": w.num_seqs,
            "n_layers": w.n_layers,
            "algorithmic_bytes_per_step": r["bytes_step"],
            "l2": "inputs larger than L2: each step reads "
                  f"{r['bytes_step'] / 2**20:.0f} MiB of distinct K/V (L2 129 MB)",
            "launch": "one CUDA graph per step (the layers' C-ABI launches, captured)",
            "parallelism": f"replicas x{world}",
            "decode_grid_cap": args.grid,
            "decode_kernel": {1: "split", 2: "cluster", 3: "seq"}.get(r["kern"], str(r["kern"])),
            "decode_kernel_choice": {
                "auto": "from the batch's context lengths (pa_decode_kernel_for_lengths)",
                "count": "from the batch size (PA_DECODE_AUTO)"}.get(args.decode_kernel, "forced"),
            "block_tokens": w.block_tokens,
            "page_fill": page_fill,
        },
        "roofline": decode_roofline(pk, w, args.workload, r, peak, peak_kind),
        "e2e": decode_e2e(agg, r),
        "gpu_launches": r["launches_per_step"] * args.steps,
        "clocks": sampler.summary(),
    }
    if others:
        line["per_config"] = {}
        for name, wo, ro, ao in others:
            entry = {
                "workload": f"{name}: {DESCRIPTIONS[name]}",
                "value": ao["gbs"],
                "unit": "GB/s",
                "pct_of_peak": 100.0 * ao["gbs"] / (peak * world),
                "seq_steps_per_s": ao["seq_steps_per_s"],
                "ms_per_step": ao["ms_per_step"],
                "steps": args.steps,
                "decode_kernel": {1: "split", 2: "cluster", 3: "seq"}.get(ro["kern"],
                                                                         str(ro["kern"])),
                "roofline": decode_roofline(pk, wo, name, ro, peak, peak_kind),
                "e2e": decode_e2e(ao, ro),
            }
            if world == 1 and not args.no_cpu_baseline:
                entry["cpu_baseline"] = cpu_baseline(wo, budget_s=args.cpu_budget / 2)
            line["per_config"][name] = entry
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, budget_s=args.cpu_budget)
    print(json.dumps(line))


# ================================================================ prefill
PREFILL_METRIC = "prefill tokens/s (paged append + causal paged attention, 16 layers)"
PREFILL_SOURCES = ("pa_prefill.cu", "pa_device.cuh", "pa_tc.cuh")


def prefill_keys(ctx: np.ndarray, lens: np.ndarray) -> int:
    """Query-key pairs of one causal prefill call: row i of a chunk after ctx
    cached tokens sees ctx + i + 1 keys."""
    ctx = ctx.astype(np.int64)
    n = lens.astype(np.int64)
    return int((n * ctx + n * (n + 1) // 2).sum())


def prefill_attention_flops(ctx: np.ndarray, lens: np.ndarray) -> float:
    """Algorithmic FLOPs of one prefill-attention call: per query-key pair
    and q head, 2*64 for q.k and 2*64 for p*v."""
    return 4.0 * D * N_Q * prefill_keys(ctx, lens)


def prefill_oracle_sample(w, rng, max_tokens: int):
    """One (sequence, layer) of a prefill workload for the oracle, drawn with
    the same distributions: the sequence's cached context and the first
    max_tokens tokens of its chunk, on a compact pool.  Returns the inputs
    and the attention FLOPs they stand for."""
    ctx = int(w.context_lens[0])
    n = max(1, min(int(w.chunk_lens[0]), int(max_tokens)))
    page = w.block_tokens
    old = (ctx + page - 1) // page
    need = (ctx + n + page - 1) // page
    nb = need + 1
    ids = rng.permutation(nb).astype(np.int32)
    bt = np.full((1, 1, need + 1), -1, dtype=np.int32)
    bt[0, 0, :old] = ids[:old]
    free = ids[old:]
    pool = wl.normal_bf16(rng, (nb, 2, page, N_KV, D))
    k = wl.normal_bf16(rng, (n, N_KV, D))
    v = wl.normal_bf16(rng, (n, N_KV, D))
    q = wl.normal_bf16(rng, (n, N_Q, D))
    u = dict(k=k, v=v, q=q, pool=pool, bt=bt, ctx=np.array([ctx], np.int32),
             cu=np.array([0, n], np.int32), fl=free, fc=len(free), page=page)
    return u, prefill_attention_flops(np.array([ctx]), np.array([n]))


def prefill_oracle_run(u, scale):
    import oracle
    q2, p2, b2, _, _, _ = oracle.prefill_append_rope(u["k"], u["v"], u["q"], u["cu"], u["pool"],
                                                     u["bt"], u["ctx"], 0, u["fl"], u["fc"],
                                                     block_tokens=u["page"])
    oracle.prefill_attention(q2, u["cu"], p2, b2, u["ctx"], 0, scale, block_tokens=u["page"])


def prefill_cpu_rate(w, rng, budget_s: float):
    """Oracle attention FLOP/s on samples of the workload, growing the sample
    until one takes about budget_s."""
    import oracle
    oracle.build()
    m, t, flops = 16, 0.0, 0.0
    while True:
        u, f = prefill_oracle_sample(w, rng, m)
        t0 = time.perf_counter()
        prefill_oracle_run(u, w.scale)
        dt = time.perf_counter() - t0
        t, flops = dt, f
        if dt > budget_s / 4 or m >= int(w.chunk_lens[0]):
            return flops / t, m, t
        m *= 2


def prefill_cpu_baseline(w, budget_s: float = 12.0):
    rng = np.random.default_rng(w.seed + 77)
    rate, m, t = prefill_cpu_rate(w, rng, budget_s)
    flops_step = prefill_attention_flops(w.context_lens, w.chunk_lens) * w.n_layers
    return {
        "value": w.total_tokens / (flops_step / rate),
        "unit": "tokens/s",
        "cores": 1,
        "kind": "oracle",
        "sample": f"append + attention of the first {m} tokens of one sequence's chunk in one "
                  f"layer ({t:.1f} s, single-threaded C, fp64), scaled to the step by "
                  "attention FLOPs",
        "host_cores": os.cpu_count(),
    }


def run_prefill_reference(args, rank, world):
    if rank != 0:
        return
    w = wl.make_prefill_workload(args.workload, block_tokens=args.block_tokens,
                                  layers=args.layers)
    rng = np.random.default_rng(w.seed + 91)
    per_step_budget = min(0.5, 150.0 / max(1, args.steps + args.warmup))
    _, m, _ = prefill_cpu_rate(w, rng, per_step_budget * 4)
    for _ in range(args.warmup):
        u, _ = prefill_oracle_sample(w, rng, m)
        prefill_oracle_run(u, w.scale)
    t_total, flops = 0.0, 0.0
    for _ in range(args.steps):
        u, f = prefill_oracle_sample(w, rng, m)
        t0 = time.perf_counter()
        prefill_oracle_run(u, w.scale)
        t_total += time.perf_counter() - t0
        flops += f
    flops_step = prefill_attention_flops(w.context_lens, w.chunk_lens) * w.n_layers
    tps = w.total_tokens / (flops_step / (flops / t_total))
    line = {
        "impl": "reference",
        "metric": PREFILL_METRIC,
        "value": tps,
        "unit": "tokens/s",
        "n_gpus": args.gpus,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": t_total / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"{args.workload}: {prefill_description(args.workload, w)}",
                   "sample_per_step": f"the first {m} tokens of one chunk in one layer, "
                                      "scaled to the step by attention FLOPs"},
        "cpu_baseline": {"value": tps, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": f"{args.steps} samples, one per step, single-threaded C (fp64)",
                         "host_cores": os.cpu_count()},
        "e2e": {"value": tps, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


PREFILL_DESCRIPTIONS = {
    "prompts17_14": "the page's two prompts (17 and 14 tokens), 1 layer, 64-block pool",
    "prefill8x2k": "8 fresh 2048-token prompts, 16 layers, 65,536-block pool, Llama-3.2-1B "
                   "heads (32 q / 8 kv, head_dim 64), 16-token bf16 pages",
    "chunked32x512": "32 sequences with 4096 tokens paged append a 512-token chunk each, 16 "
                     "layers, 262,144-block pool",
}


def prefill_description(name, w):
    d = PREFILL_DESCRIPTIONS[name]
    if w.block_tokens != BS:
        d += f"; here {w.block_tokens}-token pages ({w.num_blocks:,} blocks, the same bytes)"
    if w.n_layers != wl.PREFILL_WORKLOADS[name][1]:
        d += f" (first {w.n_layers} layers only, {w.num_blocks:,}-block pool)"
    return d


def run_prefill_gpu(args, rank, world, dist):
    import torch
    import paged_kv_cache_205_gb300 as pk
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda")
    w = wl.make_prefill_workload(args.workload, block_tokens=args.block_tokens,
                                  layers=args.layers)
    L, T, n = w.n_layers, w.total_tokens, w.num_seqs
    seed = w.seed + 1000 * rank
    pool = wl.make_prefill_pool_torch(w, dev, seed)
    bt = torch.from_numpy(w.block_table).to(dev)
    fl = torch.from_numpy(w.free_list).to(dev)
    fc0 = torch.tensor([w.free_count], dtype=torch.int32, device=dev)
    fc = fc0.clone()
    cu = torch.from_numpy(w.cu_tokens).to(dev)
    ctx = torch.from_numpy(w.context_lens).to(dev)
    g = torch.Generator(device=dev)
    g.manual_seed(seed + 1)
    q = torch.randn((L, T, N_Q, D), generator=g, device=dev).to(torch.bfloat16)
    k = torch.randn((L, T, N_KV, D), generator=g, device=dev).to(torch.bfloat16)
    v = torch.randn((L, T, N_KV, D), generator=g, device=dev).to(torch.bfloat16)
    out = torch.empty_like(q)
    err = torch.zeros(1, dtype=torch.int32, device=dev)

    def step(qs=q, ks=k, vs=v):
        # every step pages the same chunks again: the free count is restored
        # first (steady state: the pages are recycled between steps)
        fc.copy_(fc0)
        for l in range(L):
            pk.pa_prefill_append_rope(ks[l], vs[l], qs[l], cu, pool, bt, ctx, l, fl, fc, err)
            pk.pa_prefill_attention(out[l], qs[l], cu, pool, bt, ctx, l, w.scale, err)

    def barrier():
        if dist is not None:
            dist.barrier()

    def check(where):
        torch.cuda.synchronize()
        if int(err.item()) != 0:
            raise RuntimeError(f"device error bits {int(err.item())} {where}")

    for _ in range(3):
        step()
    check("during eager warm-up")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g_step = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g_step, stream=side):
            step()
    torch.cuda.current_stream().wait_stream(side)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        g_step.replay()
    check("during warm-up")

    sampler = ClockSampler(local)
    sampler.start()
    barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    sampler.mark(True)
    e0.record(stream)
    for _ in range(args.steps):
        g_step.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    sampler.mark(False)
    barrier()
    ms = e0.elapsed_time(e1) / args.steps
    check("in the timed region")

    # dominant kernel: the step's attention launches alone, one graph
    g_attn = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g_attn, stream=side):
            for l in range(L):
                pk.pa_prefill_attention(out[l], q[l], cu, pool, bt, ctx, l, w.scale, err)
    torch.cuda.current_stream().wait_stream(side)
    k_roof = max(MIN_REPLAYS, min(args.steps, 500))
    for _ in range(3):
        g_attn.replay()
    torch.cuda.synchronize()
    a0 = torch.cuda.Event(enable_timing=True)
    a1 = torch.cuda.Event(enable_timing=True)
    sampler.mark(True)
    a0.record(stream)
    for _ in range(k_roof):
        g_attn.replay()
    a1.record(stream)
    torch.cuda.synchronize()
    sampler.mark(False)
    attn_ms = a0.elapsed_time(a1) / (k_roof * L)
    check("in the roofline pass")

    # end to end: the chunks' q/k/v from pinned host memory, the step, all
    # outputs back to pinned host memory, one graph per step
    h_q, h_k, h_v = (x.cpu().pin_memory() for x in (q, k, v))
    h_out = torch.empty_like(out, device="cpu").pin_memory()
    d_q, d_k, d_v = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

    # layer by layer: each layer's inputs on their own stream ahead of its
    # kernels, each layer's output on another once its attention is done, so
    # that the copies both ways run beside the kernels (a layer's kernels
    # are long enough that the per-layer waits cost nothing)
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(L)]
    ev_att = [torch.cuda.Event() for _ in range(L)]

    def e2e_step():
        cur = torch.cuda.current_stream()
        fc.copy_(fc0)
        s_in.wait_stream(cur)
        s_out.wait_stream(cur)
        with torch.cuda.stream(s_in):
            for l in range(L):
                d_q[l].copy_(h_q[l], non_blocking=True)
                d_k[l].copy_(h_k[l], non_blocking=True)
                d_v[l].copy_(h_v[l], non_blocking=True)
                ev_in[l].record(s_in)
        for l in range(L):
            cur.wait_event(ev_in[l])
            pk.pa_prefill_append_rope(d_k[l], d_v[l], d_q[l], cu, pool, bt, ctx, l, fl, fc, err)
            pk.pa_prefill_attention(out[l], d_q[l], cu, pool, bt, ctx, l, w.scale, err)
            ev_att[l].record(cur)
            s_out.wait_event(ev_att[l])
            with torch.cuda.stream(s_out):
                h_out[l].copy_(out[l], non_blocking=True)
        cur.wait_stream(s_in)
        cur.wait_stream(s_out)

    g_e2e = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g_e2e, stream=side):
            e2e_step()
    torch.cuda.current_stream().wait_stream(side)
    k_e2e = max(MIN_REPLAYS, min(args.steps, 500))
    for _ in range(2):
        g_e2e.replay()
    torch.cuda.synchronize()
    barrier()
    sampler.mark(True)
    t0 = time.perf_counter()
    for _ in range(k_e2e):
        g_e2e.replay()
    torch.cuda.synchronize()
    e2e_s = (time.perf_counter() - t0) / k_e2e
    sampler.mark(False)
    check("in the end-to-end pass")
    h2d = (h_q.numel() + h_k.numel() + h_v.numel()) * 2
    d2h = h_out.numel() * 2

    agg = aggregate_ranks(ms, e2e_s, 0, n, dist)
    ms, e2e_s, world = agg["ms_per_step"], agg["e2e_s"], agg["world"]
    sampler.stop()
    if rank != 0:
        return
    flops = prefill_attention_flops(w.context_lens, w.chunk_lens)
    peak, peak_kind = measured_tensor_peak()
    achieved = flops / (attn_ms / 1e3) / 1e12
    line = {
        "metric": PREFILL_METRIC,
        "value": world * T / (ms / 1e3),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "accumulate": "fp32",
        "data": "synthetic",
        "config": {
            "workload": f"{args.workload}: {prefill_description(args.workload, w)}",
            "num_seqs": n,
            "n_layers": L,
            "tokens_per_step": T,
            "block_tokens": w.block_tokens,
            "attention_flops_per_step": flops * L,
            "l2": "inputs larger than L2: each step reads and writes "
                  f"{(q.numel() + out.numel() + k.numel() + v.numel()) * 2 / 2**20:.0f} MiB "
                  "of q/k/v/out (L2 129 MB)",
            "launch": "one CUDA graph per step (the 16 layers' C-ABI launches, captured)",
            "parallelism": f"replicas x{world}",
        },
        "roofline": {
            "bound": "tensor",
            "kernel": "pa_prefill_attention (prefill_attention_kernel)",
            "achieved": achieved,
            "peak": peak,
            "peak_kind": f"{peak_kind} dense bf16 (burst: the kernel timed alone)",
            "unit": "TFLOP/s",
            "frac": achieved / peak,
            "traffic": (profiled_traffic(args.workload, "prefill_attention_kernel",
                                         PREFILL_SOURCES) if w.block_tokens == BS else None),
            "flops_per_launch": flops,
            "ms_per_launch": attn_ms,
            "timing": f"{k_roof} replays of a graph of the {L} attention launches, events on the "
                      "replay stream",
        },
        "e2e": {
            "value": world * T / e2e_s,
            "unit": "tokens/s",
            "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "ms_per_step": e2e_s * 1e3,
            "how": "pinned H2D of every layer's q/k/v + the step + D2H of all outputs (each "
                   "layer's inputs on an input stream ahead of its kernels, each layer's output "
                   "on an output stream once its attention is done), one graph replay per "
                   "step, host wall clock",
        },
        "gpu_launches": 3 * L * args.steps,
        "clocks": sampler.summary(),
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = prefill_cpu_baseline(w)
    print(json.dumps(line))


# ======================================================= continuous batching
SERVE_METRIC = ("serving output tokens/s (continuous batching over the paged cache: queue, "
                "slots, prefill + decode, 16 layers)")
SERVE_DESCRIPTIONS = {
    "serve_tiny": "7 requests, 3 slots, 2 layers, 12-page pool, 32 prompt tokens per step",
    "serve256": "256 requests (prompts log-U[16,2048], decode steps log-U[16,512]) through 64 "
                "slots, 16 layers, 65,536-block pool, 8192 prompt tokens per step",
}


def serve_totals(w):
    """Output tokens (the prefill's first token + one per decode step), prompt
    tokens, and the decode-attention and prefill-attention work of one run."""
    out_tokens = sum(1 + g for _, p, g in w.requests)
    prompt_tokens = sum(p for _, p, g in w.requests)
    flops = sum(prefill_attention_flops(np.array([0]), np.array([p])) for _, p, g in w.requests)
    kv_bytes = 0
    for _, p, g in w.requests:
        ctx = np.arange(p + 1, p + g + 1, dtype=np.int64)   # attention context of each decode step
        kv_bytes += attention_bytes(ctx)
    return out_tokens, prompt_tokens, flops * w.n_layers, kv_bytes * w.n_layers


class ServeLoop:
    """Device buffers of the batcher and one complete serving run."""

    def __init__(self, w, seed):
        import torch
        import paged_kv_cache_205_gb300 as pk
        self.pk, self.w = pk, w
        dev = torch.device("cuda")
        S, L, mb, B = w.max_slots, w.n_layers, w.max_blocks_per_seq, w.prefill_budget
        g = torch.Generator(device=dev)
        g.manual_seed(seed)
        self.pool = torch.randn((w.num_blocks, 2, w.block_tokens, N_KV, D), generator=g,
                                device=dev).to(torch.bfloat16)
        self.fl0 = torch.from_numpy(
            np.random.default_rng(seed).permutation(w.num_blocks).astype(np.int32)).to(dev)
        self.bt = torch.full((S, L, mb), -1, dtype=torch.int32, device=dev)
        self.bt_tmp = torch.empty_like(self.bt)
        self.ctl = torch.zeros(pk.pa_batcher_ctl_bytes(S), dtype=torch.uint8, device=dev)
        self.fl = self.fl0.clone()
        self.fc = torch.tensor([w.num_blocks], dtype=torch.int32, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.ws = pk.decode_workspace(S, mb, block_tokens=w.block_tokens)
        bf = torch.bfloat16

        def rnd(shape):
            return torch.randn(shape, generator=g, device=dev).to(bf)
        self.pq, self.pk_, self.pv = rnd((L, B, N_Q, D)), rnd((L, B, N_KV, D)), rnd((L, B, N_KV, D))
        self.po = torch.empty((L, B, N_Q, D), dtype=bf, device=dev)
        self.dq, self.dk, self.dv = rnd((L, S, N_Q, D)), rnd((L, S, N_KV, D)), rnd((L, S, N_KV, D))
        self.do = torch.empty((L, S, N_Q, D), dtype=bf, device=dev)
        self.bufs = pk.batch_buffers(self.pool, self.bt, self.bt_tmp, self.ctl, self.fl, self.fc,
                                     self.err, self.ws, self.pq, self.pk_, self.pv, self.po,
                                     self.dq, self.dk, self.dv, self.do, w.scale)

    def reset(self):
        self.bt.fill_(-1)
        self.fl.copy_(self.fl0)
        self.fc.fill_(self.w.num_blocks)

    def run(self, on_step=None, count=False):
        """One complete serving run of the workload; returns the steps taken
        and, with `count`, the launches enqueued (else 0; the schedule and so
        the count are the same on every run).  on_step(plan, before) is called
        around each pa_batcher_run."""
        w = self.w
        b = self.pk.Batcher(w.max_slots, w.n_layers, w.max_blocks_per_seq, w.num_blocks,
                            w.prefill_budget, block_tokens=w.block_tokens)
        for r in w.requests:
            b.submit(*r)
        steps = launches = 0
        while True:
            p = b.plan()
            if p.done:
                break
            if on_step:
                on_step(p, True)
            attn = 0
            if count and p.n_rows > 0:
                # the batcher's kernel for this step: from the rows' contexts
                _, pos = b.rows()
                kern = self.pk.pa_decode_kernel_for_lengths(pos[:p.n_rows] + 1, w.block_tokens)
                attn = attn_launches(kern in (self.pk.PA_DECODE_CLUSTER, self.pk.PA_DECODE_SEQ))
            b.run(self.bufs)
            if on_step:
                on_step(p, False)
            steps += 1
            launches += 1 + (3 if p.n_retired else 0) + 3 * w.n_layers * (p.n_admitted > 0) \
                + (2 + attn) * w.n_layers * (p.n_rows > 0)
        b.close()
        return steps, launches


def serve_cpu_baseline(w, budget_s: float = 12.0):
    """The oracle's attention rates, sampled on this workload's shapes (a
    decode unit at the median decode context, a prefill unit at the median
    prompt), applied to the run's decode bytes and prefill FLOPs."""
    import oracle
    oracle.build()
    rng = np.random.default_rng(w.seed + 77)
    out_tokens, _, flops, kv_bytes = serve_totals(w)
    P = np.array([p for _, p, g in w.requests])
    G = np.array([g for _, p, g in w.requests])
    ctx_med = int(np.median(P + G // 2))
    nb = (ctx_med + BS) // BS + 1
    pool = wl.normal_bf16(rng, (nb, 2, BS, N_KV, D))
    bt = rng.permutation(nb).astype(np.int32).reshape(1, 1, nb)
    q = wl.normal_bf16(rng, (1, N_Q, D))
    t_dec, n_dec = 0.0, 0
    while t_dec < budget_s / 2:
        t0 = time.perf_counter()
        oracle.decode_attention(q, pool, bt, np.array([ctx_med], np.int32), 0, w.scale)
        t_dec += time.perf_counter() - t0
        n_dec += 1
    dec_rate = attention_bytes(np.array([ctx_med])) * n_dec / t_dec
    pw = wl.make_prefill_workload("prefill8x2k")
    pw.chunk_lens = np.array([int(np.median(P))] * 8, dtype=np.int32)
    pre_rate, m, t_pre = prefill_cpu_rate(pw, rng, budget_s / 2)
    t_run = kv_bytes / dec_rate + flops / pre_rate
    return {
        "value": out_tokens / t_run,
        "unit": "tokens/s",
        "cores": 1,
        "kind": "oracle",
        "sample": f"{n_dec} decode units at context {ctx_med} ({t_dec:.1f} s) and a {m}-token "
                  f"prefill unit ({t_pre:.1f} s), single-threaded C, fp64; the run's KV bytes "
                  "and prefill FLOPs at those rates",
        "host_cores": os.cpu_count(),
    }


def run_serve_reference(args, rank, world):
    if rank != 0:
        return
    w = wl.make_serve_workload(args.workload, block_tokens=args.block_tokens)
    base = serve_cpu_baseline(w, budget_s=min(20.0, 2.0 + 0.5 * args.steps))
    out_tokens = serve_totals(w)[0]
    line = {
        "impl": "reference",
        "metric": SERVE_METRIC,
        "value": base["value"],
        "unit": "tokens/s",
        "n_gpus": args.gpus,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": out_tokens / base["value"] * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"{args.workload}: {SERVE_DESCRIPTIONS[args.workload]}",
                   "block_tokens": w.block_tokens,
                   "sample_per_step": base["sample"]},
        "cpu_baseline": base,
        "e2e": {"value": base["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def run_serve_gpu(args, rank, world, dist):
    import torch
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    w = wl.make_serve_workload(args.workload, block_tokens=args.block_tokens)
    loop = ServeLoop(w, seed=w.seed + 1000 * rank)
    stream = torch.cuda.current_stream()

    def barrier():
        if dist is not None:
            dist.barrier()

    def check(where):
        torch.cuda.synchronize()
        if int(loop.err.item()) != 0:
            raise RuntimeError(f"device error bits {int(loop.err.item())} {where}")
        if int(loop.fc.item()) != w.num_blocks:
            raise RuntimeError(f"pages not all returned {where}")

    launches_per_run = 0
    for i in range(args.warmup):
        loop.reset()
        _, n_launch = loop.run(count=(i == 0))
        launches_per_run = launches_per_run or n_launch
    check("during warm-up")

    # timed: K complete runs; the resets (three small fills) sit between runs
    sampler = ClockSampler(local)
    sampler.start()
    barrier()
    torch.cuda.synchronize()
    total_ms, launches, steps_per_run = 0.0, 0, 0
    sampler.mark(True)
    for _ in range(args.steps):
        loop.reset()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        steps_per_run, _ = loop.run()
        e1.record(stream)
        e1.synchronize()
        total_ms += e0.elapsed_time(e1)
        launches += launches_per_run
    sampler.mark(False)
    barrier()
    check("in the timed region")
    ms = total_ms / args.steps

    # dominant work: the loop's decode-only steps (no request leaves or
    # enters), timed one by one with events around pa_batcher_run
    rec = []

    def on_step(p, before):
        ev = torch.cuda.Event(enable_timing=True)
        ev.record(stream)
        if before:
            rec.append([p.n_retired, p.n_admitted, p.n_rows, ev, None])
        else:
            rec[-1][4] = ev

    loop.reset()
    loop.run(on_step)
    torch.cuda.synchronize()
    check("in the roofline pass")
    # decode-only steps: their algorithmic bytes need the rows' contexts,
    # which the plan does not return; recompute them from the policy's
    # book-keeping (the oracle-free count: every row advances one token)
    dec_ms, dec_bytes = 0.0, 0
    sim = loop.pk.Batcher(w.max_slots, w.n_layers, w.max_blocks_per_seq, w.num_blocks,
                          w.prefill_budget, block_tokens=w.block_tokens)
    for r in w.requests:
        sim.submit(*r)
    i = 0
    while True:
        p = sim.plan()
        if p.done:
            break
        _, pos = sim.rows()
        n_ret, n_adm, n_rows, ev0, ev1 = rec[i]
        if n_ret == 0 and n_adm == 0 and n_rows > 0:
            dec_ms += ev0.elapsed_time(ev1)
            dec_bytes += w.n_layers * (attention_bytes(pos.astype(np.int64) + 1)
                                       + append_bytes(n_rows))
        sim.commit()
        i += 1
    sim.close()
    achieved = dec_bytes / (dec_ms / 1e3) / 1e9 if dec_ms > 0 else 0.0

    # end to end: every step's q/k/v from pinned host memory, outputs back.
    # The host side is kept rows first ([row][layer][...]), so that a step's
    # rows are one contiguous block each way (one direct copy at the link's
    # rate; the batcher's buffers are layer first, and a device-side copy
    # moves the block between the two orders)
    names = ("pq", "pk_", "pv", "dq", "dk", "dv")
    h = {name: getattr(loop, name).transpose(0, 1).contiguous().cpu().pin_memory() for name in names}
    g = {name: torch.empty_like(h[name], device="cuda") for name in names}
    h_po = torch.empty_like(loop.po.transpose(0, 1), device="cpu").contiguous().pin_memory()
    h_do = torch.empty_like(loop.do.transpose(0, 1), device="cpu").contiguous().pin_memory()
    g_po = torch.empty_like(h_po, device="cuda")
    g_do = torch.empty_like(h_do, device="cuda")
    io = {"h2d": 0, "d2h": 0}

    # Each step's rows go in on their own stream, beside the previous step's
    # kernels (the plan of step i + 1 is known once step i is enqueued), and
    # its outputs go back on another, beside the next step's kernels; the
    # device scratch is reused only once the copy or reorder that read it is
    # done.
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = {"reordered": None, "sent": None}

    def e2e_step(p, before):
        cur = torch.cuda.current_stream()
        if before:
            moves = []
            if p.n_admitted:
                moves += [(name, p.prefill_tokens) for name in ("pq", "pk_", "pv")]
            if p.n_rows:
                moves += [(name, p.n_rows) for name in ("dq", "dk", "dv")]
            if not moves:
                return
            if ev["reordered"] is not None:
                s_in.wait_event(ev["reordered"])
            with torch.cuda.stream(s_in):
                for name, k in moves:
                    g[name][:k].copy_(h[name][:k], non_blocking=True)
                    io["h2d"] += h[name][:k].numel() * 2
                arrived = torch.cuda.Event()
                arrived.record(s_in)
            cur.wait_event(arrived)
            for name, k in moves:
                getattr(loop, name)[:, :k].copy_(g[name][:k].transpose(0, 1))
            ev["reordered"] = torch.cuda.Event()
            ev["reordered"].record(cur)
        else:
            moves = []
            if p.n_admitted:
                moves.append((loop.po, g_po, h_po, p.prefill_tokens))
            if p.n_rows:
                moves.append((loop.do, g_do, h_do, p.n_rows))
            if not moves:
                return
            if ev["sent"] is not None:
                cur.wait_event(ev["sent"])
            for src, gs, hs, k in moves:
                gs[:k].copy_(src[:, :k].transpose(0, 1))
            ready = torch.cuda.Event()
            ready.record(cur)
            s_out.wait_event(ready)
            with torch.cuda.stream(s_out):
                for src, gs, hs, k in moves:
                    hs[:k].copy_(gs[:k], non_blocking=True)
                    io["d2h"] += hs[:k].numel() * 2
                ev["sent"] = torch.cuda.Event()
                ev["sent"].record(s_out)

    loop.reset()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    loop.run(e2e_step)
    torch.cuda.synchronize()
    e2e_s = time.perf_counter() - t0
    check("in the end-to-end pass")

    out_tokens, prompt_tokens, flops, kv_bytes = serve_totals(w)
    agg = aggregate_ranks(ms, e2e_s, 0, len(w.requests), dist)
    ms, e2e_s, world = agg["ms_per_step"], agg["e2e_s"], agg["world"]
    sampler.stop()
    if rank != 0:
        return
    peak, peak_kind = measured_hbm_peak()
    line = {
        "metric": SERVE_METRIC,
        "value": world * out_tokens / (ms / 1e3),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "accumulate": "fp32",
        "data": "synthetic",
        "prompt_tokens_per_s": world * prompt_tokens / (ms / 1e3),
        "config": {
            "workload": f"{args.workload}: {SERVE_DESCRIPTIONS[args.workload]}",
            "block_tokens": w.block_tokens,
            "step": "one complete serving run of the workload (every request admitted, "
                    "prefilled, decoded and released)",
            "loop_steps_per_run": steps_per_run,
            "output_tokens_per_run": out_tokens,
            "prompt_tokens_per_run": prompt_tokens,
            "l2": f"each run reads {kv_bytes / 2**30:.1f} GiB of K/V over its decode steps "
                  "(L2 129 MB)",
            "launch": "host loop: pa_batcher_plan + pa_batcher_run per loop step, one stream; "
                      "decode-only steps replayed from CUDA graphs (one per batch size)",
            "parallelism": f"replicas x{world}",
        },
        "roofline": {
            "bound": "hbm",
            "kernel": "decode-only loop steps (pa_kv_append_rope + pa_decode_attention, "
                      f"{w.n_layers} layers), timed one by one",
            "achieved": achieved,
            "peak": peak,
            "peak_kind": f"{peak_kind} HBM copy bandwidth",
            "unit": "GB/s",
            "frac": achieved / peak,
            "traffic": None,
            "decode_only_ms_per_run": dec_ms,
            "run_ms": ms,
        },
        "e2e": {
            "value": world * out_tokens / e2e_s,
            "unit": "tokens/s",
            "h2d_bytes_per_step": io["h2d"],
            "d2h_bytes_per_step": io["d2h"],
            "ms_per_step": e2e_s * 1e3,
            "how": "one run with every loop step's q/k/v copied from pinned host memory and its "
                   "outputs copied back (one contiguous block per tensor and direction, host "
                   "buffers rows first, reordered on the device; a step's inputs on their own "
                   "stream beside the previous step's kernels, its outputs on another beside "
                   "the next step's), host wall clock",
        },
        "gpu_launches": launches,
        "clocks": sampler.summary(),
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = serve_cpu_baseline(w)
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default 2000 for decode, 200 for prefill)")
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--path", default="decode", choices=["decode", "prefill", "serve"])
    ap.add_argument("--workload", default=None,
                    help="decode: " + ", ".join(sorted(DESCRIPTIONS)) + " (default llama1b); "
                         "prefill: " + ", ".join(sorted(PREFILL_DESCRIPTIONS)) +
                         " (default prefill8x2k); serve: " +
                         ", ".join(sorted(SERVE_DESCRIPTIONS)) + " (default serve256)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of oracle time for each CPU baseline")
    ap.add_argument("--no-per-config", dest="per_config", action="store_false",
                    help="decode path: measure the headline workload only (by default the "
                         "llama1b line also carries pool2g, long32k and ragged)")
    ap.add_argument("--block-tokens", type=int, default=BS, choices=[8, 16, 32],
                    help="decode path: tokens per page (the page size as a tunable)")
    ap.add_argument("--decode-kernel", default="auto",
                    choices=["auto", "count", "split", "cluster", "seq"],
                    help="decode-attention kernel: chosen from the batch's context lengths "
                         "(pa_decode_kernel_for_lengths, as the batcher does), chosen from the "
                         "batch size alone (PA_DECODE_AUTO), the split-context kernel, one "
                         "cluster per (sequence, kv head), or one cluster per sequence")
    ap.add_argument("--layers", type=int, default=0,
                    help="decode and prefill paths: only the first N layers, in a pool sized for them "
                         "(profiler captures of one launch on a small footprint; not a bench line)")
    ap.add_argument("--grid", type=int, default=0,
                    help="cap on decode CTAs per launch (0 = two per SM)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.steps is None:
        args.steps = {"decode": 2000, "prefill": 200, "serve": 5}[args.path]
    names = {"decode": DESCRIPTIONS, "prefill": PREFILL_DESCRIPTIONS,
             "serve": SERVE_DESCRIPTIONS}[args.path]
    if args.workload is None:
        args.workload = {"decode": "llama1b", "prefill": "prefill8x2k",
                         "serve": "serve256"}[args.path]
    if args.workload not in names:
        ap.error(f"--workload {args.workload} is not a {args.path} workload")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group("gloo")
        dist = tdist
    try:
        if args.path == "serve":
            if args.impl == "reference":
                run_serve_reference(args, rank, world)
            else:
                run_serve_gpu(args, rank, world, dist)
        elif args.path == "prefill":
            if args.impl == "reference":
                run_prefill_reference(args, rank, world)
            else:
                run_prefill_gpu(args, rank, world, dist)
        elif args.impl == "reference":
            run_reference(args, rank, world)
        else:
            run_gpu(args, rank, world, dist)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
