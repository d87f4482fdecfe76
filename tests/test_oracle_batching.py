"""Pins of the oracle's continuous-batching loop (oracle/batching.py).

Page: "An Inference Engine in 1,500 Lines of CUDA: The Map", "The path of one
inference" (prompts queue, slots, prefill of a whole prompt while a slot is
free, one decode token per active slot per step, exit when nothing is active
and the queue is empty).  The pins: a schedule worked by hand (admissions,
releases, page ids, free list), the loop's invariants on seeded workloads,
and every output of a run against attention computed without pages from
the same tokens (contiguous K/V, RoPE by position).
"""
import json
import os

import numpy as np
import pytest

import oracle
from oracle import batching
import pa_workloads as wl

BS = 16
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "batching_worked_example.json")


def _run(w_layers, max_slots, num_blocks, mb, budget, requests, free_list=None, seed=0,
         pool=None, record=None, scale=0.125, block_tokens=BS):
    sched = batching.Scheduler(max_slots, w_layers, num_blocks, budget, block_tokens)
    for rid, p, g in requests:
        sched.submit(rid, p, g)
    if free_list is None:
        free_list = np.random.default_rng(seed).permutation(num_blocks).astype(np.int32)
    if pool is None:
        pool = np.full((num_blocks, 2, block_tokens, 8, 64), wl.BF16_NAN, dtype=np.uint16)
    st = batching.PagedState(pool, np.full((max_slots, w_layers, mb), -1, np.int32),
                             free_list, len(free_list))

    def inputs(rid, layer, pos):
        return wl.request_token_inputs(seed, rid, layer, pos)

    steps = []
    while True:
        plan = sched.plan()
        if plan is None:
            break
        pre, dec, err = batching.run_step(sched, st, plan, inputs, scale)
        assert err == 0
        steps.append((plan, pre, dec, st.bt.copy(), st.fc, st.fl.copy(),
                      [(r.rid, r.ctx) for r in sched.rows]))
        if record is not None:
            record(plan, pre, dec, st, sched)
    return steps, st


@pytest.mark.parametrize("golden", ["batching_worked_example.json",
                                    "batching_worked_example_8.json"])
def test_worked_example_schedule_and_pages(golden):
    """Hand-worked schedules: 16-token pages, and 8-token pages (a request's
    lifetime pages, the positions that open a page and the pages it returns
    all follow the page size)."""
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", golden)))
    steps, st = _run(g["n_layers"], g["max_slots"], g["num_blocks"], g["max_blocks_per_seq"],
                     g["prefill_budget"], [tuple(r) for r in g["requests"]],
                     free_list=np.array(g["free_list"], np.int32),
                     block_tokens=g.get("block_tokens", BS))
    assert len(steps) == len(g["expect_steps"])
    for i, ((plan, _, _, bt, fc, _, _), e) in enumerate(zip(steps, g["expect_steps"])):
        assert plan.retired == e["retired"], i
        assert plan.admitted == e["admitted"], i
        assert plan.rows == e["rows"], i
        assert np.array_equal(bt[:, 0, :], np.array(e["table"])), i
        assert fc == e["free_count"], i
    assert st.fl.tolist() == g["expect_free_list"]


def _policy_only(w):
    """Runs the loop's decisions without numbers and checks the invariants
    each step."""
    sched = batching.Scheduler(w.max_slots, w.n_layers, w.num_blocks, w.prefill_budget)
    for r in w.requests:
        sched.submit(*r)
    admitted, finished, steps = [], [], 0
    active_steps = {}
    prev_rows = []
    while True:
        plan = sched.plan()
        if plan is None:
            break
        steps += 1
        assert len(plan.rows) <= w.max_slots
        assert sched.promised <= w.num_blocks
        assert sum(p for rid, p, g in w.requests if rid in plan.admitted) <= w.prefill_budget
        # the rows left keep their order; the new ones come after them
        assert plan.rows[:plan.n_keep] == [r for r in prev_rows if r not in plan.retired]
        assert plan.rows[plan.n_keep:] == plan.admitted
        prev_rows = list(plan.rows)
        admitted += plan.admitted
        finished += plan.retired
        for rid in plan.rows:
            active_steps[rid] = active_steps.get(rid, 0) + 1
        # a queued request is blocked only by a real limit
        if sched.queue:
            rid, p, g = sched.queue[0]
            need = batching.pages_needed(p, g, w.n_layers)
            used = sum(pp for r2, pp, gg in w.requests if r2 in plan.admitted)
            assert (len(plan.rows) >= w.max_slots or sched.promised + need > w.num_blocks
                    or p > w.prefill_budget - used)
        sched.finish_step(plan)
    order = [r[0] for r in w.requests]
    assert admitted == order                      # first in, first out, each once
    assert sorted(finished) == sorted(order)
    for rid, p, g in w.requests:
        assert active_steps[rid] == g             # exactly G decode steps
    assert sched.done() and sched.promised == 0
    return steps


@pytest.mark.parametrize("name", ["serve_tiny", "serve256"])
def test_policy_invariants(name):
    _policy_only(wl.make_serve_workload(name))


def test_admission_waits_for_slots_pages_and_budget():
    """serve_tiny is sized so that each of the three limits blocks the queue
    head at some step."""
    w = wl.make_serve_workload("serve_tiny")
    sched = batching.Scheduler(w.max_slots, w.n_layers, w.num_blocks, w.prefill_budget)
    for r in w.requests:
        sched.submit(*r)
    seen = set()
    while True:
        plan = sched.plan()
        if plan is None:
            break
        if sched.queue:
            rid, p, g = sched.queue[0]
            need = batching.pages_needed(p, g, w.n_layers)
            used = sum(pp for r2, pp, gg in w.requests if r2 in plan.admitted)
            if len(plan.rows) >= w.max_slots:
                seen.add("slots")
            elif sched.promised + need > w.num_blocks:
                seen.add("pages")
            elif p > w.prefill_budget - used:
                seen.add("budget")
        sched.finish_step(plan)
    assert seen == {"slots", "pages", "budget"}


def test_submit_refuses_what_can_never_run():
    s = batching.Scheduler(2, 2, 4, 32)
    with pytest.raises(ValueError):
        s.submit(0, 33, 1)            # longer than the prefill budget
    with pytest.raises(ValueError):
        s.submit(1, 20, 20)           # 2 layers x 3 pages > 4
    with pytest.raises(ValueError):
        s.submit(2, 5, 0)             # no decode step


def _rope_rows(x_bits, positions):
    """RoPE of every head of every row at its position, rounded to bf16."""
    out = np.empty_like(x_bits)
    for i, pos in enumerate(positions):
        for h in range(x_bits.shape[1]):
            out[i, h] = oracle.f64_to_bf16(oracle.rope_rotate(oracle.bf16_to_f64(x_bits[i, h]),
                                                              int(pos)))
    return out


def _direct_attention(seed, rid, layer, pos, scale=0.125):
    """Output of request rid's token at position pos without pages: its
    tokens 0..pos, K and q rotated at their positions, softmax in fp64."""
    positions = np.arange(pos + 1)
    q, k, v = wl.request_token_inputs(seed, rid, layer, positions)
    qr = oracle.bf16_to_f64(_rope_rows(q[-1:], [pos])[0])           # [32][64]
    kr = oracle.bf16_to_f64(_rope_rows(k, positions))                # [t][8][64]
    vv = oracle.bf16_to_f64(v)
    out = np.empty((32, 64))
    for h in range(32):
        s = kr[:, h // 4, :] @ qr[h] * scale
        p = np.exp(s - s.max())
        out[h] = p @ vv[:, h // 4, :] / p.sum()
    return out


def _pages_at(w, block_tokens):
    """serve_tiny's pool in pages of block_tokens tokens (the same bytes) and
    the table row length that holds its longest request."""
    nb = w.num_blocks * BS // block_tokens
    mb = max((p + g + block_tokens - 1) // block_tokens for _, p, g in w.requests) + 1
    return nb, mb


@pytest.mark.parametrize("block_tokens", [8, 16, 32])
def test_loop_outputs_equal_attention_without_pages(block_tokens):
    """Every prefill row and decode row the loop produced on serve_tiny
    (pages recycled through the free list, rows moved as requests leave)
    equals attention over the request's own tokens laid out contiguously,
    whatever the page size."""
    w = wl.make_serve_workload("serve_tiny")
    seed = 3
    checked = 0
    worst = 0.0

    def record(plan, pre, dec, st, sched):
        nonlocal checked, worst
        rows = sched.rows
        for layer in range(w.n_layers):
            off = 0
            for i in range(plan.n_keep, len(rows)):
                r = rows[i]
                for t in (0, r.prompt_len - 1):
                    ref = _direct_attention(seed, r.rid, layer, t)
                    worst = max(worst, np.abs(pre[layer, off + t] - ref).max())
                    checked += 1
                off += r.prompt_len
            for i, r in enumerate(rows):
                pos = r.ctx - 1          # the token decoded this step
                ref = _direct_attention(seed, r.rid, layer, pos)
                worst = max(worst, np.abs(dec[layer, i] - ref).max())
                checked += 1

    nb, mb = _pages_at(w, block_tokens)
    _run(w.n_layers, w.max_slots, nb, mb, w.prefill_budget, w.requests, seed=seed, record=record,
         block_tokens=block_tokens)
    assert checked > 100
    assert worst < 1e-9, worst


@pytest.mark.parametrize("block_tokens", [8, 16, 32])
def test_pages_conserved_and_never_shared(block_tokens):
    w = wl.make_serve_workload("serve_tiny")
    nb, mb = _pages_at(w, block_tokens)

    def record(plan, pre, dec, st, sched):
        live = st.bt[st.bt >= 0]
        assert len(live) == len(set(live.tolist())), "a page is owned twice"
        assert len(live) + st.fc == nb
        for i, r in enumerate(sched.rows):
            for layer in range(w.n_layers):
                assert (st.bt[i, layer] >= 0).sum() == (r.ctx + block_tokens - 1) // block_tokens
        assert (st.bt[len(sched.rows):] == -1).all()

    _, st = _run(w.n_layers, w.max_slots, nb, mb, w.prefill_budget, w.requests, seed=4,
                 record=record, block_tokens=block_tokens)
    assert st.fc == nb and (st.bt == -1).all()
    assert sorted(st.fl.tolist()) == list(range(nb))
