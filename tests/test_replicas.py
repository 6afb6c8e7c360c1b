"""The multi-rank path of bench.py on CPU: two gloo ranks, each with its own
timing; the job's time is the slowest rank's and its throughput counts the
work of every rank (weak scaling of independent replicas)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank: int, world: int, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    w, r, local = bench.dist_env()
    assert (w, r, local) == (world, rank, rank)
    secs = [0.25, 0.40][rank]                       # rank 1 is the slow one
    worst = bench.max_over_ranks(secs, world)
    tput = bench.job_throughput(1e12, world, worst)
    q.put((rank, worst, tput))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_max_and_throughput():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, worst, tput in got:
        assert worst == pytest.approx(0.40)
        assert tput == pytest.approx(2 * 1e12 / 0.40 / 1e12)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(1.5, 1) == 1.5
    assert bench.job_throughput(2e12, 1, 2.0) == pytest.approx(1.0)


def test_clock_rejection_rule():
    import bench
    ok = {"sm_mhz": 1900.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]}
    assert not bench.ClockSampler.rejected(ok)
    assert bench.ClockSampler.rejected({"sm_mhz": 1900.0, "sm_max_mhz": 2070.0,
                                        "reasons": ["hw_slowdown"]})
    assert bench.ClockSampler.rejected({"sm_mhz": 600.0, "sm_max_mhz": 2070.0, "reasons": []})
