"""World-size-2 gloo test of bench.py's multi-rank host logic on the CPU:
rendezvous from the torchrun environment, barrier, the max over ranks of the
per-rank time and the whole-job throughput formula (weak scaling)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    import torch.distributed as dist
    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank)
    bench.barrier(w)
    slowest = bench.max_over_ranks(10.0 + 5.0 * rank, w, "cpu")
    rate = bench.whole_job_rate(w, 1000, 4, slowest)
    q.put((rank, slowest, rate))
    dist.destroy_process_group()


def test_two_rank_max_time_and_weak_scaling_rate():
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
    for rank, slowest, rate in got:
        assert slowest == 15.0
        assert rate == pytest.approx(2 * 1000 * 4 / 15e-3)
