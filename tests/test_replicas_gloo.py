"""The multi-GPU path is replicas only: each rank runs its own workload and
nothing is exchanged on the data path.  What the ranks share is the timing
rule -- the job's step time is the slowest rank's and throughput counts the
work of every rank -- checked here with two gloo ranks on CPU."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = 2.0 if rank == 0 else 3.0          # rank 1 is the slow one
    e2e = 0.004 if rank == 0 else 0.005
    out = bench.aggregate_ranks(ms, e2e, bytes_per_step=6_000_000, seqs=16, dist=dist)
    q.put((rank, out))
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank_and_sum_the_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in (0, 1):
        out = res[r]
        assert out["world"] == 2
        assert out["ms_per_step"] == pytest.approx(3.0)
        assert out["e2e_s"] == pytest.approx(0.005)
        assert out["gbs"] == pytest.approx(2 * 6_000_000 / 3e-3 / 1e9)
        assert out["seq_steps_per_s"] == pytest.approx(2 * 16 / 3e-3)


def test_single_process_needs_no_group():
    import bench
    out = bench.aggregate_ranks(1.5, 0.002, 3_000_000, 4, None)
    assert out["world"] == 1 and out["ms_per_step"] == 1.5
    assert out["gbs"] == pytest.approx(3_000_000 / 1.5e-3 / 1e9)
