"""Multi-rank logic of bench.py on CPU (gloo, world size 2): no GPU needed.

The path shards by packs: every rank runs its own pack with no collective on the data path;
the only cross-rank step is the reduction of the timings to the slowest rank, and the
reported rate is the work of all ranks over that time (weak scaling).
"""

import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys

    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    # rank r measured step time 1 + r and qkv time 5 - r
    times = bench.reduce_max([1.0 + rank, 5.0 - rank], world)
    rate = bench.whole_job_rate(world, 10.0, times[0])

    class Args:
        steps, warmup = 4, 3

    ref = bench.run_reference(Args, rank, world) if rank != 0 else "rank0"
    q.put((rank, times, rate, ref))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_reduce_to_the_slowest_and_report_weak_scaling():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, times, rate, ref in got:
        assert times == [2.0, 5.0]           # element-wise max over the two ranks
        assert rate == pytest.approx(10.0)   # 2 ranks x 10 units / 2.0 s
    assert got[1][3] is None                 # the reference arm runs on rank 0 only


def test_single_rank_is_identity():
    import sys

    sys.path.insert(0, ROOT)
    import bench

    assert bench.reduce_max([3.0, 1.5], 1) == [3.0, 1.5]
    assert bench.whole_job_rate(1, 8.0, 2.0) == 4.0
