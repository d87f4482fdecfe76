"""Failure detection on the GPU without a GPU fault.

Every wait of the decode kernels is bounded: one that runs out sets
PA_DEV_TIMEOUT in the caller's error word and the kernel returns, so the
CUDA context stays usable.  The test makes a wait run out on purpose through
the library's test hook (one stage of the split-context kernel published
without its copies: a barrier that nothing completes), with a 50 us limit,
checks the bit and that the call returned promptly, then checks that the next
call, with the hook cleared, matches the oracle.  Calls go through the C ABI.
"""
import time

import numpy as np
import pytest

import oracle
import pa_workloads as wl
from helpers import assert_attention_close, dev_bf16, dev_i32, host_f64, workspace_for

pytestmark = pytest.mark.gpu

N_Q, D = 32, 64


def test_wait_that_nothing_completes_runs_out_and_the_next_call_is_clean():
    import torch
    import paged_kv_cache_205_gb300 as pk
    rng = np.random.default_rng(77)
    ctx = np.array([300, 40, 900, 17, 0, 655], dtype=np.int32)
    nbk = int(((ctx + 15) // 16).sum()) + 8
    mb = int(((ctx + 15) // 16).max()) + 1
    w = wl.make_workload("tiny", seed=77, context_lens=ctx, num_blocks=nbk, max_blocks_per_seq=mb)
    pool = wl.make_pool_numpy(w, rng, poison=True)
    q = wl.normal_bf16(rng, (len(ctx), N_Q, D))
    qd, poold, btd, ctxd = dev_bf16(q), dev_bf16(pool), dev_i32(w.block_table), dev_i32(ctx)
    out = torch.zeros((len(ctx), N_Q, D), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = workspace_for(len(ctx), mb)
    pk.pa_decode_set_path(pk.PA_DECODE_SPLIT)
    pk.pa_decode_set_grid_limit(2)   # CTA 0 streams many stages
    try:
        pk.pa_decode_set_test_fault(1, 50_000)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        pk.pa_decode_attention(out, qd, poold, btd, ctxd, 0, 0.125, ws, err)
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
        assert int(err.item()) & pk.PA_DEV_TIMEOUT, int(err.item())
        assert dt < 0.5, f"the call took {dt:.3f} s"
    finally:
        pk.pa_decode_set_test_fault(-1)
    try:
        err.zero_()
        out.fill_(float("nan"))
        pk.pa_decode_attention(out, qd, poold, btd, ctxd, 0, 0.125, ws, err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        ref, e = oracle.decode_attention(q, pool, w.block_table, ctx, 0)
        assert e == 0
        assert_attention_close(host_f64(out), ref, "the call after the timeout")
    finally:
        pk.pa_decode_set_path(pk.PA_DECODE_AUTO)
        pk.pa_decode_set_grid_limit(0)


def test_prefill_wait_that_nothing_completes_runs_out_and_the_next_call_is_clean():
    """The same for the prefill attention kernel: CTA 0 announces the bytes of
    its second 128-key chunk without issuing the copies; every role's wait on
    it runs out after 50 us, the CTA waits for its own copies, stores and MMAs
    in flight before it frees its tensor memory, and the call reports
    PA_DEV_TIMEOUT; the next call, with the hook cleared, matches the
    oracle."""
    import torch
    import paged_kv_cache_205_gb300 as pk
    from test_gpu_prefill import SCALE, _attention_state, _close, _gpu_prefill_attention
    # the heaviest item (the first in the work order, CTA 0's) runs through
    # 4 chunks: 300 cached tokens and the second tile of a 100-token chunk
    pool, bt, ctx, cu, q = _attention_state(41, [300, 0, 150], [100, 64, 40])
    try:
        pk.pa_prefill_set_test_fault(1, 50_000)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        _, err = _gpu_prefill_attention(pool, bt, ctx, cu, q)
        dt = time.perf_counter() - t0
        assert err & pk.PA_DEV_TIMEOUT, err
        assert dt < 1.0, f"the call took {dt:.3f} s"
    finally:
        pk.pa_prefill_set_test_fault(-1)
    out, err = _gpu_prefill_attention(pool, bt, ctx, cu, q)
    ref, e_ref = oracle.prefill_attention(q, cu, pool, bt, ctx, 0, SCALE)
    assert err == e_ref == 0
    _close(host_f64(out), ref, "the call after the timeout")
