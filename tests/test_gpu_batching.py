"""GPU parity of the continuous-batching loop (pa_batcher_run) against the
oracle's loop, through the C ABI.

Page: "An Inference Engine in 1,500 Lines of CUDA: The Map", "The path of one
inference" (queue, slots, prefill while a slot is free, one decode token per
active slot per step).  serve_tiny runs step by step on both sides with the
same keyed token inputs: plans equal, block tables, free list and count
bit-exact after every step, V pages bit-exact and K pages within the RoPE
bound, prefill and decode outputs within the attention tolerance (beyond the
output's bf16 rounding).  serve256 runs at full size as the benchmark runs
it: pages conserved after every step, sampled decode rows against the
oracle's attention over the pages the GPU wrote, everything returned at the
end.
"""
import numpy as np
import pytest

from oracle import batching
import pa_workloads as wl
from helpers import assert_attention_close, dev_i32, gather_for_oracle, host_bits, host_f64
from test_gpu_append import _compare_pools

pytestmark = pytest.mark.gpu

N_Q, N_KV, D, BS = 32, 8, 64, 16


def _pk():
    import paged_kv_cache_205_gb300 as pk
    return pk


class DeviceLoop:
    """The buffers of one batcher on the GPU."""

    def __init__(self, w, pool, free_list, block_tokens=BS, max_blocks_per_seq=None):
        import torch
        pk = _pk()
        dev = torch.device("cuda")
        S, L, B = w.max_slots, w.n_layers, w.prefill_budget
        mb = w.max_blocks_per_seq if max_blocks_per_seq is None else max_blocks_per_seq
        self.w = w
        self.pool = pool
        self.bt = torch.full((S, L, mb), -1, dtype=torch.int32, device=dev)
        self.bt_tmp = torch.empty_like(self.bt)
        self.ctl = torch.zeros(pk.pa_batcher_ctl_bytes(S), dtype=torch.uint8, device=dev)
        self.fl = dev_i32(free_list)
        self.fc = torch.tensor([len(free_list)], dtype=torch.int32, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.ws = pk.decode_workspace(S, mb, block_tokens=block_tokens)
        bf = torch.bfloat16
        self.pq = torch.zeros((L, B, N_Q, D), dtype=bf, device=dev)
        self.pk_ = torch.zeros((L, B, N_KV, D), dtype=bf, device=dev)
        self.pv = torch.zeros((L, B, N_KV, D), dtype=bf, device=dev)
        self.po = torch.zeros((L, B, N_Q, D), dtype=bf, device=dev)
        self.dq = torch.zeros((L, S, N_Q, D), dtype=bf, device=dev)
        self.dk = torch.zeros((L, S, N_KV, D), dtype=bf, device=dev)
        self.dv = torch.zeros((L, S, N_KV, D), dtype=bf, device=dev)
        self.do = torch.zeros((L, S, N_Q, D), dtype=bf, device=dev)
        self.bufs = pk.batch_buffers(self.pool, self.bt, self.bt_tmp, self.ctl, self.fl, self.fc,
                                     self.err, self.ws, self.pq, self.pk_, self.pv, self.po,
                                     self.dq, self.dk, self.dv, self.do, w.scale)
        self.b = pk.Batcher(S, L, mb, len(free_list), B, block_tokens=block_tokens)
        for r in w.requests:
            self.b.submit(*r)


def _put(t, bits):
    import torch
    t.copy_(torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16))


def _step_by_step(w, block_tokens, seed=11, kernels=None):
    """Runs workload w through the library's loop and the oracle's, step by
    step with the same keyed token inputs, comparing plans, tables, free
    list, pool and outputs after every step.  With `kernels` (a list), the
    decode kernel the length rule picks for each step's rows is appended.
    Returns (steps, prefill steps)."""
    import torch
    pk = _pk()
    nb = w.num_blocks * BS // block_tokens
    mb = max((p + g + block_tokens - 1) // block_tokens for _, p, g in w.requests) + 1
    rng = np.random.default_rng(w.seed)
    free_list = rng.permutation(nb).astype(np.int32)
    pool0 = np.full((nb, 2, block_tokens, N_KV, D), wl.BF16_NAN, dtype=np.uint16)
    dl = DeviceLoop(w, torch.from_numpy(pool0.view(np.int16)).view(torch.bfloat16).cuda(),
                    free_list, block_tokens, mb)
    ref = batching.Scheduler(w.max_slots, w.n_layers, nb, w.prefill_budget, block_tokens)
    for r in w.requests:
        ref.submit(*r)
    st = batching.PagedState(pool0, np.full(tuple(dl.bt.shape), -1, np.int32), free_list,
                             len(free_list))

    def inputs(rid, layer, pos):
        return wl.request_token_inputs(seed, rid, layer, pos)

    steps = prefills = 0
    while True:
        p = dl.b.plan()
        rp = ref.plan()
        if rp is None:
            assert p.done == 1
            break
        steps += 1
        ids, pos = dl.b.rows()
        assert ids.tolist() == rp.rows and dl.b.retired() == rp.retired
        if kernels is not None and p.n_rows > 0:
            kernels.append(pk.pa_decode_kernel_for_lengths(pos[:p.n_rows] + 1, block_tokens))
        # the step's inputs, from the rows the library planned
        for layer in range(w.n_layers):
            off = 0
            for i in range(p.n_keep, p.n_rows):
                q, k, v = inputs(int(ids[i]), layer, np.arange(pos[i]))
                n = q.shape[0]
                _put(dl.pq[layer, off:off + n], q)
                _put(dl.pk_[layer, off:off + n], k)
                _put(dl.pv[layer, off:off + n], v)
                off += n
            for i in range(p.n_rows):
                q, k, v = inputs(int(ids[i]), layer, [pos[i]])
                _put(dl.dq[layer, i:i + 1], q)
                _put(dl.dk[layer, i:i + 1], k)
                _put(dl.dv[layer, i:i + 1], v)
        dl.b.run(dl.bufs)
        pre, dec, e = batching.run_step(ref, st, rp, inputs, w.scale)
        torch.cuda.synchronize()
        assert e == 0 and int(dl.err.item()) == 0, steps
        assert np.array_equal(dl.bt.cpu().numpy(), st.bt), steps
        assert int(dl.fc.item()) == st.fc, steps
        assert np.array_equal(dl.fl.cpu().numpy()[:st.fc], st.fl[:st.fc]), steps
        _compare_pools(host_bits(dl.pool), st.pool)
        if pre is not None:
            prefills += 1
            got = host_f64(dl.po[:, :p.prefill_tokens])
            assert_attention_close(got, pre, f"prefill step {steps}", output_rounding=True)
        if dec is not None:
            got = host_f64(dl.do[:, :p.n_rows])
            assert_attention_close(got, dec, f"decode step {steps}")
    assert int(dl.fc.item()) == nb and (dl.bt.cpu().numpy() == -1).all()
    dl.b.close()
    return steps, prefills


@pytest.mark.parametrize("block_tokens", [8, 16, 32])
def test_serve_tiny_step_by_step(block_tokens):
    """serve_tiny with pages of 8, 16 and 32 tokens (the pool keeps its
    bytes), step by step against the oracle's loop."""
    steps, prefills = _step_by_step(wl.make_serve_workload("serve_tiny"), block_tokens)
    assert steps > 10 and prefills > 2


def test_decode_steps_switch_kernels():
    """A loop whose decode steps take all three kernels, step by step against
    the oracle: 24 even rows (the per-sequence kernel), then 5 short rows and
    one 1200-token prompt (a heavy tail: the split kernel), then the long
    request alone (the per-head kernel).  The batcher picks each step's
    kernel from its rows' contexts and captures one graph per (rows,
    kernel)."""
    import torch
    pk = _pk()
    # 24 rows exceed the per-head kernel's bound (two CTAs per (row, kv head))
    assert 24 * 16 > 2 * torch.cuda.get_device_properties(0).multi_processor_count
    reqs = [(i, 120, 4) for i in range(19)] + [(19 + i, 120, 12) for i in range(5)]
    reqs.append((24, 1200, 16))
    w = wl.ServeWorkload("switch", 1, 24, 400, 0, 4096, reqs, seed=12)
    kernels = []
    steps, prefills = _step_by_step(w, BS, seed=13, kernels=kernels)
    seen = set(kernels)
    assert seen == {pk.PA_DECODE_SPLIT, pk.PA_DECODE_CLUSTER, pk.PA_DECODE_SEQ}, kernels
    assert prefills >= 2


def test_serve256_full_size_sampled():
    """The benchmark's serving workload at full size (256 requests, 64 slots,
    16 layers), device-drawn inputs: after every step the free count equals
    the pool minus the pages the active requests hold, and on sampled steps
    three decode rows match the oracle's attention over the pages the GPU
    wrote (rotated q read back from the step's buffer)."""
    import torch
    w = wl.make_serve_workload("serve256")
    dev = torch.device("cuda")
    rng = np.random.default_rng(w.seed)
    free_list = rng.permutation(w.num_blocks).astype(np.int32)
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed)
    pool = torch.randn((w.num_blocks, 2, BS, N_KV, D), generator=g, device=dev).to(torch.bfloat16)
    dl = DeviceLoop(w, pool, free_list)
    for t in (dl.pq, dl.pk_, dl.pv, dl.dq, dl.dk, dl.dv):
        t.normal_(generator=g)
    sample_rng = np.random.default_rng(5)
    steps = checked = 0
    while True:
        p = dl.b.plan()
        if p.done:
            break
        ids, pos = dl.b.rows()
        dl.b.run(dl.bufs)
        steps += 1
        torch.cuda.synchronize()
        assert int(dl.err.item()) == 0, steps
        ctx_after = pos.astype(np.int64) + 1
        held = int(sum(w.n_layers * ((c + BS - 1) // BS) for c in ctx_after))
        assert int(dl.fc.item()) == w.num_blocks - held, steps
        if p.n_rows and steps % 97 == 1:
            table = dl.bt.cpu().numpy()
            rows = sorted(set(sample_rng.integers(p.n_rows, size=3).tolist()))
            ctxs = np.zeros(w.max_slots, dtype=np.int32)
            ctxs[:p.n_rows] = ctx_after
            for layer in (0, w.n_layers - 1):
                sub, sub_bt = gather_for_oracle(dl.pool, table, rows, ctxs, layer)
                import oracle
                q = host_bits(dl.dq[layer, rows])
                ref, e = oracle.decode_attention(q, sub, sub_bt, ctxs[rows], 0, w.scale)
                assert e == 0
                assert_attention_close(host_f64(dl.do[layer, rows]), ref,
                                       f"step {steps} layer {layer}")
                checked += 1
    assert dl.b.pending() == 0 and steps > 100 and checked >= 4
    assert int(dl.fc.item()) == w.num_blocks and (dl.bt.cpu().numpy() == -1).all()
    dl.b.close()


def test_graph_replayed_steps_equal_direct_launches():
    """Decode-only steps replayed from CUDA graphs (the default) give
    bit-identical tables, free lists and outputs to the same loop run with
    direct launches, step by step (batch sizes change as requests come and
    go, so several graphs are captured and replayed)."""
    import torch
    w = wl.make_serve_workload("serve_tiny")
    rng = np.random.default_rng(w.seed)
    free_list = rng.permutation(w.num_blocks).astype(np.int32)
    runs = []
    for graphs in (False, True):
        g = torch.Generator(device="cuda")
        g.manual_seed(5)
        pool = torch.randn((w.num_blocks, 2, BS, N_KV, D), generator=g,
                           device="cuda").to(torch.bfloat16)
        dl = DeviceLoop(w, pool, free_list)
        dl.b.set_graphs(graphs)
        steps = []
        while True:
            p = dl.b.plan()
            if p.done:
                break
            for t in (dl.pq, dl.pk_, dl.pv, dl.dq, dl.dk, dl.dv):
                t.normal_(generator=g)
            dl.b.run(dl.bufs)
            torch.cuda.synchronize()
            steps.append((p.n_rows, p.n_admitted, p.n_retired, dl.bt.cpu().numpy().copy(),
                          int(dl.fc.item()), host_bits(dl.do[:, :p.n_rows]),
                          host_bits(dl.po[:, :p.prefill_tokens]), int(dl.err.item())))
        dl.b.close()
        runs.append(steps)
    assert len(runs[0]) == len(runs[1]) > 10
    decode_only = 0
    for a, b in zip(*runs):
        assert a[:3] == b[:3] and a[4] == b[4] and a[7] == b[7] == 0
        assert np.array_equal(a[3], b[3]) and np.array_equal(a[5], b[5])
        assert np.array_equal(a[6], b[6])
        decode_only += a[1] == 0 and a[2] == 0 and a[0] > 0
    assert decode_only > 5
