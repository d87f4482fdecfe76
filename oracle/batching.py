"""Oracle of the continuous-batching loop over the paged cache.

TEST INFRASTRUCTURE ONLY (see the package docstring): the tests and the
benchmark's CPU legs use it; the product never does.

Page: "An Inference Engine in 1,500 Lines of CUDA: The Map", "The path of one
inference": prompts wait in a queue; while a slot is free and a prompt is
queued, prefill() takes the whole prompt at once; otherwise one decode step
produces one token for every active slot; a finished slot returns to the free
set; the loop ends when no slot is active and the queue is empty.  The
numeric work of each step is done by this package's C oracle
(``prefill_append_rope``, ``prefill_attention``, ``kv_append_rope``,
``decode_attention``, ``free``), in the order the loop runs it.

The policy, where the page leaves it open (each choice is the plainest one
the rest of the page supports):

  * A request is (id, P prompt tokens, G decode steps), G >= 1: the prefill
    yields its first token, each decode step one more, and it is finished
    after its G-th decode step.  (The engine has no model here, so a seeded
    generation length stands in for the end-of-text token.)
  * Active requests occupy rows 0..n-1 of the block table in admission
    order.  A step first releases the requests that finished in the previous
    step (``free`` over their rows in ascending row order), then closes the
    gaps: the remaining rows keep their order and move down.
  * Admission is first-in first-out and stops at the first queued request
    that does not fit: it needs a free row, ``L * ceil((P + G) / B)`` pages
    of B tokens (16, the page's BLOCK_SIZE, unless chosen otherwise) not
    promised to the requests already admitted (its whole life, so a decode
    step never runs out of pages), and P tokens of the step's prefill
    budget.
  * The admitted prompts are prefilled together (all layers), then every
    active row (the new ones included) takes one decode step (all layers):
    append at position ctx, attention over ctx + 1.
"""
from __future__ import annotations

import collections
import dataclasses

import numpy as np

BLOCK = 16


def pages_needed(prompt_len: int, decode_steps: int, n_layers: int,
                 block_tokens: int = BLOCK) -> int:
    """Pages a request holds at the end of its life: P + G tokens per layer,
    in pages of block_tokens tokens."""
    return n_layers * ((prompt_len + decode_steps + block_tokens - 1) // block_tokens)


@dataclasses.dataclass
class Row:
    rid: int
    prompt_len: int
    decode_steps: int
    ctx: int = 0          # tokens cached
    done: int = 0         # decode steps taken


@dataclasses.dataclass
class StepPlan:
    retired: list          # request ids released at the start of the step
    retired_rows: list     # their rows before the gaps closed
    retired_ctx: list      # their cached tokens (P + G)
    admitted: list         # request ids prefilled this step (rows n_keep ..)
    rows: list             # request id per row after admission (decode order)
    n_keep: int            # rows that were active before admission


class Scheduler:
    """The loop's host decisions, without numbers."""

    def __init__(self, max_slots: int, n_layers: int, pages_free: int, prefill_budget: int,
                 block_tokens: int = BLOCK):
        self.max_slots = max_slots
        self.n_layers = n_layers
        self.pages_free = pages_free
        self.prefill_budget = prefill_budget
        self.block_tokens = block_tokens
        self.queue = collections.deque()
        self.rows: list[Row] = []
        self.promised = 0

    def submit(self, rid: int, prompt_len: int, decode_steps: int):
        if prompt_len < 1 or decode_steps < 1 or prompt_len > self.prefill_budget:
            raise ValueError("request cannot be served")
        if pages_needed(prompt_len, decode_steps, self.n_layers,
                        self.block_tokens) > self.pages_free:
            raise ValueError("request needs more pages than the pool holds")
        self.queue.append((rid, prompt_len, decode_steps))

    def done(self) -> bool:
        return not self.queue and not self.rows

    def plan(self) -> StepPlan | None:
        """Decide one step; returns None when the loop is over."""
        retired_rows = [i for i, r in enumerate(self.rows) if r.done >= r.decode_steps]
        retired = [self.rows[i].rid for i in retired_rows]
        for i in retired_rows:
            r = self.rows[i]
            self.promised -= pages_needed(r.prompt_len, r.decode_steps, self.n_layers,
                                          self.block_tokens)
        retired_ctx = [self.rows[i].ctx for i in retired_rows]
        self.rows = [r for r in self.rows if r.done < r.decode_steps]
        n_keep = len(self.rows)
        admitted, budget = [], self.prefill_budget
        while self.queue:
            rid, p, g = self.queue[0]
            need = pages_needed(p, g, self.n_layers, self.block_tokens)
            if len(self.rows) >= self.max_slots or self.promised + need > self.pages_free \
                    or p > budget:
                break
            self.queue.popleft()
            self.rows.append(Row(rid, p, g))
            self.promised += need
            budget -= p
            admitted.append(rid)
        if not self.rows and not retired:
            return None
        return StepPlan(retired, retired_rows, retired_ctx, admitted, [r.rid for r in self.rows],
                        n_keep)

    def finish_step(self, plan: StepPlan):
        """Book-keeping after the step ran: prompts are cached, every row
        took one decode step."""
        for i, r in enumerate(self.rows):
            if i >= plan.n_keep:
                r.ctx = r.prompt_len
            r.ctx += 1
            r.done += 1


class PagedState:
    """The oracle's copy of the device state: pool [pages][2][B][8][64], block
    table (one row per slot), free list and count."""

    def __init__(self, pool, block_table, free_list, free_count):
        self.pool = np.array(pool, dtype=np.uint16, copy=True)
        self.bt = np.array(block_table, dtype=np.int32, copy=True)
        self.fl = np.array(free_list, dtype=np.int32, copy=True)
        self.fc = int(free_count)


def run_step(sched: Scheduler, st: PagedState, plan: StepPlan, inputs, scale: float):
    """Runs one planned step on the oracle state.

    inputs(rid, layer, positions) -> (q [n][32][64], k [n][8][64], v [n][8][64])
    bf16 bits for the request's tokens at those positions.  Returns
    (prefill_out [layers][tokens][32][64] fp64 or None, decode_out
    [layers][rows][32][64] fp64 or None when no row is left, error bits).
    The loop's last step only releases what finished in the one before."""
    import oracle
    L = sched.n_layers
    B = sched.block_tokens
    err = 0
    # 1. release the finished requests, then close the gaps (order kept)
    if plan.retired_rows:
        ctx = np.zeros(st.bt.shape[0], dtype=np.int32)
        ctx[plan.retired_rows] = plan.retired_ctx
        st.bt, st.fl, st.fc, e = oracle.free(np.array(plan.retired_rows, np.int32), st.bt, ctx,
                                             st.fl, st.fc, st.pool.shape[0], block_tokens=B)
        err |= e
        n_prev = plan.n_keep + len(plan.retired_rows)
        gone = set(plan.retired_rows)
        keep = [i for i in range(n_prev) if i not in gone]
        moved = st.bt[keep]
        st.bt[:len(keep)] = moved
        st.bt[len(keep):n_prev] = -1
    rows = sched.rows
    n = len(rows)
    k0 = plan.n_keep
    # 2. prefill of the admitted prompts, packed in row order
    pre_out = None
    if n > k0:
        lens = [rows[i].prompt_len for i in range(k0, n)]
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        zero = np.zeros(n - k0, dtype=np.int32)
        pre_out = []
        for layer in range(L):
            qs, ks, vs = [], [], []
            for i in range(k0, n):
                q, k, v = inputs(rows[i].rid, layer, np.arange(rows[i].prompt_len))
                qs.append(q)
                ks.append(k)
                vs.append(v)
            q, k, v = np.concatenate(qs), np.concatenate(ks), np.concatenate(vs)
            sub = st.bt[k0:n]
            q2, st.pool, sub2, st.fl, st.fc, e = oracle.prefill_append_rope(
                k, v, q, cu, st.pool, sub, zero, layer, st.fl, st.fc, block_tokens=B)
            st.bt[k0:n] = sub2
            err |= e
            out, e = oracle.prefill_attention(q2, cu, st.pool, st.bt[k0:n], zero, layer, scale,
                                              block_tokens=B)
            err |= e
            pre_out.append(out)
        pre_out = np.stack(pre_out)
    # 3. one decode step for every active row
    ctx = np.array([r.prompt_len if i >= k0 else r.ctx for i, r in enumerate(rows)], np.int32)
    if n == 0:
        sched.finish_step(plan)
        return pre_out, None, err
    dec_out = []
    for layer in range(L):
        qs, ks, vs = [], [], []
        for i, r in enumerate(rows):
            q, k, v = inputs(r.rid, layer, np.array([ctx[i]]))
            qs.append(q)
            ks.append(k)
            vs.append(v)
        q, k, v = np.concatenate(qs), np.concatenate(ks), np.concatenate(vs)
        sub = st.bt[:n]
        q2, st.pool, sub2, st.fl, st.fc, e = oracle.kv_append_rope(k, v, q, st.pool, sub, ctx,
                                                                   layer, st.fl, st.fc,
                                                                   block_tokens=B)
        st.bt[:n] = sub2
        err |= e
        out, e = oracle.decode_attention(q2, st.pool, st.bt[:n], ctx + 1, layer, scale,
                                         block_tokens=B)
        err |= e
        dec_out.append(out)
    sched.finish_step(plan)
    return pre_out, np.stack(dec_out), err

