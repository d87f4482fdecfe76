"""GPU parity of pa_decode_attention against the fp64 CPU oracle.

Every call goes through the C ABI (libpagedkv.so via ctypes).  Tolerance
(bf16 output vs fp64 oracle): max abs error <= 1e-2, mean abs <= 1e-3.
"""
import numpy as np
import pytest

import oracle
import pa_workloads as wl
from helpers import assert_attention_close, dev_bf16, dev_i32, host_f64, workspace_for

pytestmark = pytest.mark.gpu

N_Q, N_KV, D = 32, 8, 64


def _pk():
    import paged_kv_cache_205_gb300 as pk
    return pk


@pytest.fixture(autouse=True, params=["split", "cluster", "seq"])
def decode_path(request):
    """Every test runs on each decode kernel: the split-context kernel, one
    cluster per (sequence, kv head), one cluster per sequence."""
    pk = _pk()
    pk.pa_decode_set_grid_limit(0)
    pk.pa_decode_set_path({"split": pk.PA_DECODE_SPLIT, "cluster": pk.PA_DECODE_CLUSTER,
                           "seq": pk.PA_DECODE_SEQ}[request.param])
    yield request.param
    pk.pa_decode_set_path(pk.PA_DECODE_AUTO)
    pk.pa_decode_set_grid_limit(0)


def _run_gpu(q_bits, pool_bits, bt, ctx, layer, scale=0.125, grid=0, pool_dev=None, num_seqs=None):
    import torch
    pk = _pk()
    pk.pa_decode_set_grid_limit(grid)
    n = bt.shape[0] if num_seqs is None else num_seqs
    q = dev_bf16(q_bits)
    pool = dev_bf16(pool_bits) if pool_dev is None else pool_dev
    btd = dev_i32(bt)
    ctxd = dev_i32(ctx)
    out = torch.full((max(n, 1), N_Q, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = workspace_for(max(n, 1), bt.shape[2])
    pk.pa_decode_attention(out, q, pool, btd, ctxd, layer, scale, ws, err, num_seqs=n)
    torch.cuda.synchronize()
    return host_f64(out), int(err.item())


def _small_case(seed, ctx, n_layers=1, q_scale=1.0, extra_blocks=8):
    rng = np.random.default_rng(seed)
    ctx = np.asarray(ctx, dtype=np.int32)
    nbk = int(((ctx + 15) // 16).sum()) * n_layers + extra_blocks
    mb = int(max(1, ((ctx + 15) // 16).max())) + 1
    w = wl.make_workload("tiny", seed=seed, context_lens=ctx, n_layers=n_layers,
                         num_blocks=nbk, max_blocks_per_seq=mb)
    pool = wl.make_pool_numpy(w, rng, poison=True)
    q = wl.normal_bf16(rng, (len(ctx), N_Q, D), scale=q_scale)
    return w, pool, q


def test_tiny_workload_matches_oracle():
    """Two sequences with contexts 17 and 14 over a 64-block pool."""
    w = wl.make_workload("tiny")
    rng = np.random.default_rng(100)
    pool = wl.make_pool_numpy(w, rng, poison=True)
    q = wl.normal_bf16(rng, (w.num_seqs, N_Q, D))
    ref, e_ref = oracle.decode_attention(q, pool, w.block_table, w.context_lens, 0)
    out, err = _run_gpu(q, pool, w.block_table, w.context_lens, 0)
    assert err == 0 and e_ref == 0
    assert_attention_close(out, ref, "tiny")


@pytest.mark.parametrize("grid", [0, 1, 2, 3, 7, 64])
def test_split_count_does_not_change_result(grid):
    """The same inputs cut across 1..many CTAs (1 = no split) all match."""
    w, pool, q = _small_case(7, [1, 15, 16, 17, 100, 250, 33, 64], q_scale=2.0)
    ref, _ = oracle.decode_attention(q, pool, w.block_table, w.context_lens, 0)
    out, err = _run_gpu(q, pool, w.block_table, w.context_lens, 0, grid=grid)
    assert err == 0
    assert_attention_close(out, ref, f"grid={grid}")


@pytest.mark.parametrize("ctx", [[1], [16], [17], [31, 32, 33], [0, 5], [0], [0, 0, 40, 0],
                                 [2047, 1], [4096]])
def test_edge_contexts(ctx):
    w, pool, q = _small_case(len(ctx) * 13 + sum(ctx), ctx)
    ref, _ = oracle.decode_attention(q, pool, w.block_table, w.context_lens, 0)
    out, err = _run_gpu(q, pool, w.block_table, w.context_lens, 0)
    assert err == 0
    assert_attention_close(out, ref, f"ctx={ctx}")
    for s, t in enumerate(ctx):
        if t == 0:
            assert np.all(out[s] == 0.0)


def test_many_sequences_ragged_and_layers():
    rng = np.random.default_rng(5)
    ctx = rng.integers(0, 400, size=40)
    w, pool, q = _small_case(21, ctx, n_layers=3)
    for layer in range(3):
        ref, _ = oracle.decode_attention(q, pool, w.block_table, w.context_lens, layer)
        out, err = _run_gpu(q, pool, w.block_table, w.context_lens, layer)
        assert err == 0
        assert_attention_close(out, ref, f"layer {layer}")


def test_peaked_softmax_q_times_four():
    w, pool, q = _small_case(9, [300, 1000, 77], q_scale=4.0)
    ref, _ = oracle.decode_attention(q, pool, w.block_table, w.context_lens, 0)
    out, err = _run_gpu(q, pool, w.block_table, w.context_lens, 0, grid=5)
    assert err == 0
    assert_attention_close(out, ref, "peaked")


def test_constant_value_per_kv_head_fixes_gqa_mapping():
    w, pool, q = _small_case(10, [50, 3])
    for g in range(N_KV):
        pool[:, 1, :, g, :] = wl.to_bf16_bits(np.full((), g + 1.0, dtype=np.float32))
    out, err = _run_gpu(q, pool, w.block_table, w.context_lens, 0)
    assert err == 0
    for h in range(N_Q):
        assert np.all(out[:, h] == h // 4 + 1.0)


def test_non_default_scale():
    w, pool, q = _small_case(11, [64, 9])
    ref, _ = oracle.decode_attention(q, pool, w.block_table, w.context_lens, 0, scale=0.3)
    out, err = _run_gpu(q, pool, w.block_table, w.context_lens, 0, scale=0.3)
    assert err == 0
    assert_attention_close(out, ref, "scale 0.3")


def test_fewer_sequences_than_table_rows():
    w, pool, q = _small_case(12, [40, 20, 10])
    ref, _ = oracle.decode_attention(q[:2], pool, w.block_table[:2], w.context_lens[:2], 0)
    out, err = _run_gpu(q, pool, w.block_table, w.context_lens, 0, num_seqs=2)
    assert err == 0
    assert_attention_close(out[:2], ref, "num_seqs=2")


def test_zero_sequences_is_a_no_op():
    w, pool, q = _small_case(13, [5])
    out, err = _run_gpu(q, pool, w.block_table, w.context_lens, 0, num_seqs=0)
    assert err == 0 and np.all(np.isnan(out))


def test_device_errors_are_reported_not_trapped():
    import torch
    w, pool, q = _small_case(14, [40, 20])
    bt = w.block_table.copy()
    bt[0, 0, 1] = -1
    _, err = _run_gpu(q, pool, bt, w.context_lens, 0)
    assert err & _pk().PA_DEV_BAD_BLOCK
    bt = w.block_table.copy()
    bt[1, 0, 0] = w.num_blocks + 5
    _, err = _run_gpu(q, pool, bt, w.context_lens, 0)
    assert err & _pk().PA_DEV_BAD_BLOCK
    ctx = w.context_lens.copy()
    ctx[1] = w.max_blocks_per_seq * 16 + 3
    _, err = _run_gpu(q, pool, w.block_table, ctx, 0)
    assert err & _pk().PA_DEV_CTX_RANGE
    # the context stays usable
    ref, _ = oracle.decode_attention(q, pool, w.block_table, w.context_lens, 0)
    out, err = _run_gpu(q, pool, w.block_table, w.context_lens, 0)
    assert err == 0
    assert_attention_close(out, ref, "after errors")
    torch.cuda.synchronize()


def test_host_argument_errors():
    import torch
    pk = _pk()
    w, pool, q = _small_case(15, [20])
    qd, poold, btd, ctxd = dev_bf16(q), dev_bf16(pool), dev_i32(w.block_table), dev_i32(w.context_lens)
    out = torch.empty((1, N_Q, D), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = workspace_for(1, w.max_blocks_per_seq)
    with pytest.raises(pk.PagedKVError) as e:
        pk.pa_decode_attention(out, qd, poold, btd, ctxd, 1, 0.125, ws, err)
    assert e.value.code == -3
    with pytest.raises(pk.PagedKVError) as e:
        pk.pa_decode_attention(out, qd, poold, btd, ctxd, 0, 0.125, ws[:16], err)
    assert e.value.code == -4
    flat = torch.empty(N_Q * D + 1, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pk.PagedKVError) as e:
        pk.pa_decode_attention(flat[1:].view(1, N_Q, D), qd, poold, btd, ctxd, 0, 0.125, ws, err)
    assert e.value.code == -5


def test_workspace_reused_across_calls_and_grids():
    """One zero-filled workspace serves many calls in a row (the work counter
    is returned to zero by every call), whatever the split."""
    import torch
    pk = _pk()
    rng = np.random.default_rng(31)
    ws = workspace_for(12, 40)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for trial, grid in enumerate([0, 3, 0, 17, 1, 0]):
        ctx = rng.integers(0, 600, size=12)
        w, pool, q = _small_case(40 + trial, ctx)
        pk.pa_decode_set_grid_limit(grid)
        out = torch.empty((12, N_Q, D), dtype=torch.bfloat16, device="cuda")
        bt = np.zeros((12, 1, 40), dtype=np.int32) - 1
        bt[:, :, :w.block_table.shape[2]] = w.block_table
        pk.pa_decode_attention(out, dev_bf16(q), dev_bf16(pool), dev_i32(bt), dev_i32(w.context_lens),
                               0, 0.125, ws, err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        ref, _ = oracle.decode_attention(q, pool, w.block_table, w.context_lens, 0)
        assert_attention_close(host_f64(out), ref, f"trial {trial}")


def test_graph_replay_matches_oracle():
    """The call captured in a CUDA graph and replayed gives the same result
    every replay."""
    import torch
    pk = _pk()
    w, pool, q = _small_case(51, [700, 33, 1, 250, 0, 1900], n_layers=2)
    qd, poold, btd, ctxd = dev_bf16(q), dev_bf16(pool), dev_i32(w.block_table), dev_i32(w.context_lens)
    out = torch.zeros((w.num_seqs, N_Q, D), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = workspace_for(w.num_seqs, w.max_blocks_per_seq)
    pk.pa_decode_attention(out, qd, poold, btd, ctxd, 1, 0.125, ws, err)   # warm-up
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            pk.pa_decode_attention(out, qd, poold, btd, ctxd, 1, 0.125, ws, err)
    torch.cuda.current_stream().wait_stream(side)
    ref, _ = oracle.decode_attention(q, pool, w.block_table, w.context_lens, 1)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert_attention_close(host_f64(out), ref, "graph replay")


def test_too_many_sequences_is_refused():
    import torch
    pk = _pk()
    n = 2049
    bt = torch.full((n, 1, 1), -1, dtype=torch.int32, device="cuda")
    ctx = torch.zeros(n, dtype=torch.int32, device="cuda")
    q = torch.zeros((n, N_Q, D), dtype=torch.bfloat16, device="cuda")
    pool = torch.zeros((1, 2, 16, 8, 64), dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(pk.PagedKVError) as e:
        pk.pa_decode_attention(q, q, pool, bt, ctx, 0, 0.125, ws, err)
    assert e.value.code == -2


@pytest.mark.parametrize("grid", [0, 40, 7])
def test_large_batch_merge_shape(grid):
    """A large batch where a small grid forces many sequences to be split
    into several pieces, each merged per q head."""
    rng = np.random.default_rng(61 + grid)
    ctx = rng.integers(0, 300, size=160)
    w, pool, q = _small_case(62 + grid, ctx, q_scale=2.0)
    ref, _ = oracle.decode_attention(q, pool, w.block_table, w.context_lens, 0)
    out, err = _run_gpu(q, pool, w.block_table, w.context_lens, 0, grid=grid)
    assert err == 0
    assert_attention_close(out, ref, f"160 sequences, grid {grid}")


def test_automatic_kernel_choice(decode_path):
    """Automatic choice: the per-head cluster kernel while every (sequence,
    kv head) pair gets two CTAs (two CTAs per SM in all), the split-context
    kernel beyond, for 16- and 32-token pages; a grid limit lowers the
    bound; 8-token pages take the split kernel unless the per-head kernel is
    forced (four 1 KiB copies per tile make it slower there); a forced path
    is reported as forced."""
    import torch
    pk = _pk()
    pk.pa_decode_set_path(pk.PA_DECODE_AUTO)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    fit = (2 * sms) // 16
    assert pk.pa_decode_kernel_for(1) == pk.PA_DECODE_CLUSTER
    assert pk.pa_decode_kernel_for(fit) == pk.PA_DECODE_CLUSTER
    assert pk.pa_decode_kernel_for(fit + 1) == pk.PA_DECODE_SPLIT
    assert pk.pa_decode_kernel_for(16, 8) == pk.PA_DECODE_SPLIT
    assert pk.pa_decode_kernel_for(fit, 32) == pk.PA_DECODE_CLUSTER
    assert pk.pa_decode_kernel_for(fit + 1, 32) == pk.PA_DECODE_SPLIT
    pk.pa_decode_set_grid_limit(64)
    assert pk.pa_decode_kernel_for(4) == pk.PA_DECODE_CLUSTER
    assert pk.pa_decode_kernel_for(5) == pk.PA_DECODE_SPLIT
    pk.pa_decode_set_path(pk.PA_DECODE_SEQ)
    assert pk.pa_decode_kernel_for(300) == pk.PA_DECODE_SEQ


def _tile_rho(ctx):
    """Longest context over the mean, in 16-token tiles."""
    t = (np.asarray(ctx, dtype=np.int64) + 15) // 16
    return float(t.max()) * len(t) / float(t.sum())


def test_kernel_choice_from_lengths(decode_path):
    """pa_decode_kernel_for_lengths: a batch whose longest context lies more
    than 3x above the mean (in 16-token tiles) takes the split-context kernel;
    an even batch the per-head cluster kernel while every (sequence, kv head)
    pair gets two CTAs, then (16-token pages, at most one sequence per CTA of
    the grid) the per-sequence cluster kernel, then the split kernel; 8-token
    pages the split kernel.  The answer does not depend on the forced path
    (this test runs under each) and follows the grid limit."""
    import torch
    pk = _pk()
    choose = pk.pa_decode_kernel_for_lengths
    SPLIT, CLUSTER, SEQ = pk.PA_DECODE_SPLIT, pk.PA_DECODE_CLUSTER, pk.PA_DECODE_SEQ
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    fit = (2 * sms) // 16
    # the measured workloads
    assert choose(wl.make_workload("llama1b").attn_context_lens) == CLUSTER
    assert choose(wl.make_workload("long32k").attn_context_lens) == CLUSTER
    assert choose(wl.make_workload("pool2g").attn_context_lens) == SEQ
    ragged = wl.make_workload("ragged").attn_context_lens
    assert _tile_rho(ragged) > 3 and choose(ragged) == SPLIT
    # log-uniform contexts in [1, 8192], 16 sequences
    rng = np.random.default_rng(16)
    logu = np.floor(np.exp(rng.uniform(0, np.log(8192), size=16))).astype(np.int32)
    assert choose(logu) == (SPLIT if _tile_rho(logu) > 3 else CLUSTER)
    # the heavy-tail bound is strict: max / mean = 3 is still even
    assert choose([160, 0, 0]) == CLUSTER
    assert choose([160, 0, 0, 0]) == SPLIT
    tail = np.full(16, 100, dtype=np.int32)
    tail[0] = 1600
    assert choose(tail) == SPLIT
    # even batches by size and page size
    assert choose(np.full(fit, 1000)) == CLUSTER
    assert choose(np.full(fit + 1, 1000)) == SEQ
    assert choose(np.full(2 * sms, 1000)) == SEQ
    assert choose(np.full(2 * sms + 1, 1000)) == SPLIT
    assert choose(np.full(fit, 1000), 32) == CLUSTER
    assert choose(np.full(fit + 1, 1000), 32) == SPLIT
    assert choose(np.full(4, 1000), 8) == SPLIT
    assert choose([]) == SPLIT
    pk.pa_decode_set_grid_limit(64)
    assert choose(np.full(4, 1000)) == CLUSTER
    assert choose(np.full(5, 1000)) == SEQ
    assert choose(np.full(65, 1000)) == SPLIT
    pk.pa_decode_set_grid_limit(0)


@pytest.mark.parametrize("case", ["logu16", "tail16", "even8", "even40"])
def test_chosen_kernel_matches_oracle(case):
    """The kernel the length-aware choice names, run on its batch (seeded
    lengths of the kinds the rule separates: heavy-tailed -> split kernel,
    even and few -> per-head clusters, even and many -> per-sequence
    clusters), matches the oracle."""
    pk = _pk()
    rng = np.random.default_rng({"logu16": 61, "tail16": 63, "even8": 64, "even40": 62}[case])
    if case == "logu16":
        ctx = np.floor(np.exp(rng.uniform(0, np.log(4096), size=16))).astype(np.int64)
    elif case == "tail16":
        ctx = rng.integers(1, 200, size=16)
        ctx[5] = 3000
    else:
        ctx = rng.integers(600, 700, size=8 if case == "even8" else 40)
    w, pool, q = _small_case(3100 + len(ctx), ctx)
    path = pk.pa_decode_kernel_for_lengths(w.context_lens)
    assert path == {"logu16": pk.PA_DECODE_SPLIT, "tail16": pk.PA_DECODE_SPLIT,
                    "even8": pk.PA_DECODE_CLUSTER, "even40": pk.PA_DECODE_SEQ}[case]
    pk.pa_decode_set_path(path)
    ref, _ = oracle.decode_attention(q, pool, w.block_table, w.context_lens, 0)
    out, err = _run_gpu(q, pool, w.block_table, w.context_lens, 0)
    assert err == 0
    assert_attention_close(out, ref, f"{case}, kernel {path}")


@pytest.mark.parametrize("n,law", [(10, "u"), (16, "u"), (19, "u"), (16, "logu"), (12, "even")])
def test_packed_plan_that_moves_after_the_wait(decode_path, n, law):
    """The per-head kernel's packed plan (two CTAs per pair on average) first
    worked out from a wrong length (the test hook makes every sequence look
    like the first), so that after the dependency wait the plan moves: CTAs
    take another (sequence, kv head) or part mid-call, or are left idle.  The
    result still matches the oracle."""
    pk = _pk()
    rng = np.random.default_rng(500 + n)
    if law == "u":
        ctx = rng.integers(256, 2049, size=n)
    elif law == "logu":
        ctx = np.floor(np.exp(rng.uniform(0, np.log(3000), size=n))).astype(np.int64)
        ctx[0] = 1
    else:
        ctx = np.full(n, 700)
        ctx[0] = 40
    w, pool, q = _small_case(4100 + n, ctx, q_scale=2.0)
    ref, _ = oracle.decode_attention(q, pool, w.block_table, w.context_lens, 0)
    pk.pa_decode_set_path(pk.PA_DECODE_CLUSTER)
    pk.pa_decode_set_test_plan(1)
    try:
        out, err = _run_gpu(q, pool, w.block_table, w.context_lens, 0)
    finally:
        pk.pa_decode_set_test_plan(0)
    assert err == 0
    assert_attention_close(out, ref, f"moved plan n={n} {law}")


@pytest.mark.parametrize("grid", [0, 24, 64, 152, 304])
@pytest.mark.parametrize("n", [1, 2, 3, 7, 16, 19, 32])
def test_mixed_lengths_every_cluster_size(decode_path, n, grid):
    """Batches of 1..32 sequences with heavy-tailed lengths (empty, single
    tokens, page edges, long), under grid limits that give the per-head
    cluster kernel clusters of 1, 2, 4 and 8 CTAs (or hand larger batches to
    the split-context kernel)."""
    rng = np.random.default_rng(1000 + 37 * n + grid)
    ctx = np.floor(np.exp(rng.uniform(0, np.log(3000), size=n))).astype(np.int64)
    ctx[rng.random(n) < 0.15] = 0
    if n >= 3:
        ctx[:3] = [1, 16, 2900]
    w, pool, q = _small_case(2000 + n + grid, ctx, q_scale=2.0)
    ref, _ = oracle.decode_attention(q, pool, w.block_table, w.context_lens, 0)
    out, err = _run_gpu(q, pool, w.block_table, w.context_lens, 0, grid=grid)
    assert err == 0
    assert_attention_close(out, ref, f"n={n} grid={grid}")
    for s, t in enumerate(ctx):
        if t == 0:
            assert np.all(out[s] == 0.0)
