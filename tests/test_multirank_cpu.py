"""Multi-rank host logic of bench.py on the CPU.

World-size-2 gloo runs check the rendezvous from the torchrun environment,
the barrier, the max over ranks of the per-rank time and the whole-job
throughput of both launch modes: replicas (every rank runs the whole
workload, weak scaling) and --shard (the ranks deal one batch's (sequence,
kv head) units among themselves, strong scaling), including that the shards
cover every unit exactly once and that the whole-job rate counts each unit
once. The partition functions are also checked on their own for many
shapes and world sizes."""
import os
import random
import socket

import pytest
import torch.multiprocessing as mp

import bench
from parametrized_local_linear_gb300 import inputs


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _prefill_units(calls, G):
    """(b, kv head) units of a rank's calls, and the query heads they read."""
    units, heads = [], []
    for b, kv0, kv1 in calls:
        assert 0 <= kv0 < kv1
        units += [(b, g) for g in range(kv0, kv1)]
        heads += [(b, h) for h in range(kv0 * G, kv1 * G)]
    return units, heads


def _worker(rank, world, port, q):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import torch.distributed as dist
    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank)
    bench.barrier(w)
    slowest = bench.max_over_ranks(10.0 + 5.0 * rank, w, "cpu")
    rate = bench.whole_job_rate(w, 1000, 4, slowest)
    # --shard: this rank's share of the benchmark's batches.
    wp, wd = inputs.PREFILL_0P6B, inputs.DECODE_RAGGED
    calls = bench.prefill_shard(wp.B, wp.Hkv, w, r)
    units, heads = _prefill_units(calls, wp.Hq // wp.Hkv)
    lens = wd.seqlens().tolist()
    b0, b1 = bench.decode_shard(lens, w, r)
    gathered = [None] * w
    dist.all_gather_object(gathered, (units, heads, (b0, b1)))
    own = 8 * wp.d * len(heads) * wp.L * (wp.L + 1) // 2
    tot = [0.0]
    t = bench.max_over_ranks(2.0 + rank, w, "cpu")
    import torch
    s = torch.tensor([float(own)], dtype=torch.float64)
    dist.all_reduce(s)
    tot[0] = float(s.item())
    srate = bench.sharded_rate(wp.flops, 3, t)
    q.put((rank, slowest, rate, gathered, tot[0], srate, t))
    dist.destroy_process_group()


def test_two_ranks_replicas_and_shards():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted((q.get(timeout=10) for _ in range(2)), key=lambda x: x[0])
    wp, wd = inputs.PREFILL_0P6B, inputs.DECODE_RAGGED
    for rank, slowest, rate, gathered, tot, srate, t in got:
        # Replicas: every rank ran the whole workload; the job took the slowest.
        assert slowest == 15.0
        assert rate == pytest.approx(2 * 1000 * 4 / 15e-3)
        # Shards: every (sequence, kv head) unit and every query head exactly once.
        units = [u for g in gathered for u in g[0]]
        heads = [h for g in gathered for h in g[1]]
        assert sorted(units) == [(b, g) for b in range(wp.B) for g in range(wp.Hkv)]
        assert sorted(heads) == [(b, h) for b in range(wp.B) for h in range(wp.Hq)]
        ranges = [g[2] for g in gathered]
        assert ranges[0][0] == 0 and ranges[-1][1] == wd.B
        assert all(a[1] == b[0] for a, b in zip(ranges, ranges[1:]))
        # The ranks' own flops add up to the batch's, counted once, and the
        # whole-job rate divides that by the slowest rank's time.
        assert tot == wp.flops
        assert t == 3.0
        assert srate == pytest.approx(wp.flops * 3 / 3.0e-3)


@pytest.mark.parametrize("B,Hkv,world", [(4, 8, 2), (4, 8, 3), (4, 8, 8), (4, 8, 5), (1, 8, 8),
                                         (3, 2, 7), (2, 1, 4), (64, 8, 8), (1, 1, 2)])
def test_prefill_shards_cover_every_unit_once(B, Hkv, world):
    G = 2
    all_units = []
    sizes = []
    for rank in range(world):
        calls = bench.prefill_shard(B, Hkv, world, rank)
        units, heads = _prefill_units(calls, G)
        assert len(heads) == G * len(units)
        # Calls are cut at sequence boundaries and never straddle one.
        assert all(0 <= b < B and kv1 <= Hkv for b, _, kv1 in calls)
        all_units += units
        sizes.append(len(units))
    assert sorted(all_units) == [(b, g) for b in range(B) for g in range(Hkv)]
    assert max(sizes) - min(sizes) <= 1
    # Contiguous in the sequence-major unit order.
    assert all_units == sorted(all_units)


@pytest.mark.parametrize("world", [1, 2, 3, 8, 13])
def test_decode_shards_partition_the_sequences(world):
    rng = random.Random(world)
    for lens in ([8192] * 64, inputs.DECODE_RAGGED.seqlens().tolist(), [0, 5, 0, 0, 7, 1],
                 [rng.randrange(0, 5000) for _ in range(40)], [0, 0, 0]):
        ranges = [bench.decode_shard(lens, world, r) for r in range(world)]
        assert ranges[0][0] == 0 and ranges[-1][1] == len(lens)
        assert all(a[1] == b[0] and a[0] <= a[1] for a, b in zip(ranges, ranges[1:]))
        total = sum(lens)
        # Each cut is the first sequence boundary at or past k / world of the
        # tokens: a rank's tokens exceed an even share by less than the
        # longest sequence.
        longest = max(lens) if lens else 0
        for b0, b1 in ranges:
            assert sum(lens[b0:b1]) <= total / world + longest
    # A uniform batch splits evenly whenever the world size divides it.
    assert [bench.decode_shard([8192] * 64, 8, r) for r in range(8)] == \
        [(8 * r, 8 * r + 8) for r in range(8)]


def test_config_selection_covers_the_five_workloads():
    """--config 1..5 names each of the five workloads once, and --seed gives
    the same shape with another seed."""
    import dataclasses
    assert sorted(bench.CONFIGS) == [1, 2, 3, 4, 5]
    assert sorted(w.name for w in bench.CONFIGS.values()) == sorted(inputs.WORKLOADS)
    w = dataclasses.replace(bench.CONFIGS[4], seed=7)
    assert w.seed == 7 and w.B == inputs.DECODE_B64.B and w.name == inputs.DECODE_B64.name
