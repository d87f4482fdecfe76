"""The library's continuous-batching decisions (pa_batcher_plan / _rows /
_retired / _commit, host code only, no GPU needed) against the oracle's
loop, step by step: which requests leave, which are admitted, which request
each row holds and at which position it decodes.  Also the argument checks
of the batcher's C entry points."""
import json
import os

import pytest

from oracle import batching
import pa_workloads as wl

def _compare(max_slots, n_layers, mb, pages, budget, requests, block_tokens=16):
    import paged_kv_cache_205_gb300 as pk
    nat = pk.Batcher(max_slots, n_layers, mb, pages, budget, block_tokens=block_tokens)
    ref = batching.Scheduler(max_slots, n_layers, pages, budget, block_tokens)
    for r in requests:
        nat.submit(*r)
        ref.submit(*r)
    steps = 0
    while True:
        p = nat.plan()
        rp = ref.plan()
        if rp is None:
            assert p.done == 1
            break
        assert p.done == 0
        steps += 1
        ids, pos = nat.rows()
        assert ids.tolist() == rp.rows, steps
        want_pos = [r.prompt_len if i >= rp.n_keep else r.ctx for i, r in enumerate(ref.rows)]
        assert pos.tolist() == want_pos, steps
        assert nat.retired() == rp.retired, steps
        assert p.n_keep == rp.n_keep and p.n_admitted == len(rp.admitted)
        assert p.n_rows == len(rp.rows) and p.n_retired == len(rp.retired)
        assert p.prefill_tokens == sum(r.prompt_len for r in ref.rows[rp.n_keep:])
        assert nat.pending() == len(ref.queue)
        nat.commit()
        ref.finish_step(rp)
    nat.close()
    return steps


@pytest.mark.parametrize("golden", ["batching_worked_example.json",
                                    "batching_worked_example_8.json"])
def test_worked_example(golden):
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", golden)))
    n = _compare(g["max_slots"], g["n_layers"], g["max_blocks_per_seq"], g["num_blocks"],
                 g["prefill_budget"], [tuple(r) for r in g["requests"]],
                 g.get("block_tokens", 16))
    assert n == len(g["expect_steps"])


@pytest.mark.parametrize("block_tokens", [8, 16, 32])
@pytest.mark.parametrize("name", ["serve_tiny", "serve256"])
def test_serving_workloads(name, block_tokens):
    """The serving workloads with pages of 8, 16 and 32 tokens: the pool
    keeps its bytes (16 / page times the pages)."""
    w = wl.make_serve_workload(name)
    pages = w.num_blocks * 16 // block_tokens
    mb = max((p + g + block_tokens - 1) // block_tokens for _, p, g in w.requests) + 1
    assert _compare(w.max_slots, w.n_layers, mb, pages, w.prefill_budget, w.requests,
                    block_tokens) > 0


def test_argument_checks():
    import paged_kv_cache_205_gb300 as pk
    with pytest.raises(pk.PagedKVError):
        pk.Batcher(0, 2, 4, 12, 32)
    with pytest.raises(pk.PagedKVError):
        pk.Batcher(2, 2, 4, 12, 32, block_tokens=24)
    b = pk.Batcher(2, 2, 4, 12, 32)
    for bad in [(0, 0, 1), (1, 5, 0), (2, 33, 1), (3, 40, 30), (4, 30, 40)]:
        with pytest.raises(pk.PagedKVError):
            b.submit(*bad)                      # empty, no step, budget, table, pages
    with pytest.raises(pk.PagedKVError):
        b.commit()                              # nothing planned
    assert b.plan().done == 1                   # empty queue: nothing to do
    b.submit(7, 10, 2)
    p = b.plan()
    assert p.n_rows == 1 and p.n_admitted == 1 and p.prefill_tokens == 10
    with pytest.raises(pk.PagedKVError):
        b.plan()                                # previous plan not run
    b.commit()
    b.close()
