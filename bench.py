"""Benchmark of the Parallax forward hot path on GB300 (one JSON line on stdout).

A step is one pass of the whole hot path over one batch of synthetic input:
the causal prefill of the 0.6B-shaped workload (B=4, Hq=16, Hkv=8, L=4096,
d=128, bf16) followed by a decode of the batched workload (B=64, Hq=16,
Hkv=8, d=128, 8192 cached tokens each). ``value`` is the prefill throughput
in algorithmic TFLOP/s (8 d flops per causal pair); the decode throughput in
algorithmic HBM GB/s is the ``decode`` object. Both are timed per launch with
CUDA events on the launching stream; inputs are resident in HBM and larger
than L2, so no flush is needed between steps. The 1.7B-shaped prefill and
the ragged long-context decode are timed after the steps (``extra``).

``--impl reference`` times the fp64 CPU oracle instead (the only other
implementation of this method here), on a bounded row sample per step.

``--config N`` (1-5: the fp32 tiny prefill, the 0.6B- and 1.7B-shaped
prefills, the batched and the ragged decode) times that one workload alone and
prints one line for it; ``--seed`` replaces the workload's input seed and
``--nsplit`` fixes the decode's share count (0: the library's default). The
prefill and decode launches of a timed step sit in NVTX ranges.

Under torchrun each rank runs the same per-rank workload on its own GPU
(weak scaling, no collective on the data path); rank 0 prints the line.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from parametrized_local_linear_gb300 import inputs  # noqa: E402

METRIC = "Parallax fwd: prefill TFLOP/s, decode HBM GB/s; % of GB300 roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# dram__bytes_read.sum + dram__bytes_write.sum per launch, from the ncu
# captures summarised in profiles/ (prefill: the bench's own workload;
# decode: a quarter-size batch scaled by 4, the traffic being proportional to
# the cache streamed). Set to None whenever a kernel changes after its capture.
NCU_TRAFFIC_BYTES = {"prefill_tc_kernel": 392.79e6, "decode_split_kernel": 4 * 540.57e6}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def _peak(peaks, key):
    v = peaks.get(key)
    if isinstance(v, dict):
        v = v.get("value")
    return float(v) if v is not None else FALLBACK_PEAKS[key]


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1])); mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world, units_per_rank_per_step, steps, max_ms):
    """Whole-job throughput: every rank processed the same units; the job took
    the slowest rank's time (max over ranks)."""
    return world * units_per_rank_per_step * steps / (max_ms * 1e-3)


def sharded_rate(units_per_step, steps, max_ms):
    """Whole-job throughput when the ranks share one batch: every unit of the
    batch was processed once, by one rank, and the job took the slowest
    rank's time."""
    return units_per_step * steps / (max_ms * 1e-3)


# ---------------------------------------------------------------- sharding
# The path partitions into independent (sequence, kv head) units: a kv head's
# keys and values and the query heads that read them touch nothing else. With
# --shard the ranks deal one batch's units among themselves, contiguous and
# balanced, with no collective on the data path (each rank keeps its own
# outputs).
def shard_range(n_units, world, rank):
    """Contiguous share [start, end) of n_units for `rank`: sizes differ by at
    most one, the first n_units % world ranks taking the larger."""
    base, extra = divmod(n_units, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def prefill_shard(B, Hkv, world, rank):
    """The prefill units of `rank`: its contiguous range of the sequence-major
    (sequence, kv head) list, cut at sequence boundaries into calls
    (b, kv0, kv1), each one contiguous slice of the batch (sequence b, kv
    heads kv0 .. kv1 - 1 and their query heads)."""
    s, e = shard_range(B * Hkv, world, rank)
    calls = []
    u = s
    while u < e:
        b, kv0 = divmod(u, Hkv)
        kv1 = min(Hkv, kv0 + (e - u))
        calls.append((b, kv0, kv1))
        u += kv1 - kv0
    return calls


def decode_shard(seqlens, world, rank):
    """The decode sequences [b0, b1) of `rank`. The packed cache holds a
    sequence's kv heads interleaved token by token, so a rank takes whole
    sequences: contiguous ranges whose ends are the first sequence boundaries
    at or past k / world of the batch's cached tokens (k = 1 .. world - 1),
    so cached tokens, the decode's work, spread as evenly as whole sequences
    allow."""
    lens = [max(0, int(x)) for x in seqlens]
    cum = [0]
    for n in lens:
        cum.append(cum[-1] + n)
    total = cum[-1]

    def cut(k):
        if k >= world:
            return len(lens)
        goal = total * k / world
        return next(i for i, c in enumerate(cum) if c >= goal)

    return cut(rank), cut(rank + 1)


def oracle_prefill_sample(w, q, k, v, r, budget_s, seed, threads=None):
    """Time the fp64 oracle on seeded random causal rows of workload w until
    about budget_s seconds of oracle time; return (algorithmic flops of the
    rows done, oracle seconds, rows, threads). Host copies are not timed."""
    import random

    import oracle
    rng = random.Random(seed)
    threads = oracle.default_threads() if threads is None else threads
    done_flops, rows_done, secs = 0, 0, 0.0
    while secs < budget_s:
        b, h = rng.randrange(w.B), rng.randrange(w.Hq)
        g = h // (w.Hq // w.Hkv)
        rows = [(0, 0, rng.randrange(w.L)) for _ in range(threads)]
        qs = q[b:b + 1, h:h + 1].cpu(); rs = r[b:b + 1, h:h + 1].cpu()
        ks = k[b:b + 1, g:g + 1].cpu(); vs = v[b:b + 1, g:g + 1].cpu()
        ts = time.perf_counter()
        oracle.prefill(qs, ks, vs, rs, rows=rows, threads=threads)
        secs += time.perf_counter() - ts
        done_flops += sum(8 * w.d * (i + 1) for _, _, i in rows)
        rows_done += len(rows)
    return done_flops, secs, rows_done, threads


def oracle_extra_samples(w, q, k, v, r, budget_s, seed=12):
    """The gradient and projection oracles timed on bounded samples of the
    0.6B-shaped workload: {row name: cpu_baseline dict}."""
    import random

    import numpy as np

    import oracle
    from oracle import grad as ograd
    rng = random.Random(seed)
    out = {}
    # Gradient oracle: whole gradients of random causal rows (autograd through
    # the explicit Sigma of the row), 16 d flops per (query, key) pair.
    dout = torch.randn(q.shape[2:], device=q.device).to(q.dtype)
    flops, secs, n = 0, 0.0, 0
    while secs < budget_s:
        b, h, i = rng.randrange(w.B), rng.randrange(w.Hq), rng.randrange(w.L)
        g = h // (w.Hq // w.Hkv)
        args = [q[b, h, i].cpu(), r[b, h, i].cpu(), k[b, g, :i + 1].cpu(), v[b, g, :i + 1].cpu(),
                dout[i].cpu()]
        ts = time.perf_counter()
        ograd.row_grads(*args)
        secs += time.perf_counter() - ts
        flops += 16 * w.d * (i + 1)
        n += 1
    out[w.name + "_backward"] = {
        "value": flops / secs / 1e12, "unit": "TFLOP/s", "cores": torch.get_num_threads(),
        "kind": "oracle", "sample": f"whole gradients of {n} random causal rows (torch fp64 "
                                    f"autograd through explicit Sigma), {secs:.1f} s"}
    # Projection oracle: fp64 product for random token rows of the layer.
    D, F = 1024, (2 * w.Hq + 2 * w.Hkv) * w.d
    xs = np.random.default_rng(seed).standard_normal((256, D))
    ws = np.random.default_rng(seed + 1).standard_normal((F, D))
    flops, secs, n = 0, 0.0, 0
    while secs < budget_s / 4:
        ts = time.perf_counter()
        oracle.qkvr_projection(xs, ws, 1, xs.shape[0], w.Hq, w.Hkv, w.d)
        secs += time.perf_counter() - ts
        flops += 2 * xs.shape[0] * D * F
        n += xs.shape[0]
    out[f"qkvr_projection_0p6b_T{w.B * w.L}_D{D}_F{F}"] = {
        "value": flops / secs / 1e12, "unit": "TFLOP/s", "cores": torch.get_num_threads(),
        "kind": "oracle", "sample": f"{n} token rows (numpy fp64 product), {secs:.1f} s"}
    return out


def cpu_baseline_plan(dev, explicit_budget_s=4.0, seed=21):
    """The CPU oracles timed on each of the five workloads, on this host's
    cores: the explicit-Sigma C oracle (configs 1, 4, 5 on the whole workload
    or a stated sample of it; configs 2, 3 on random rows, extrapolated by
    pair count) and the expanded fp64 form on the whole workload. Inputs are
    the same distributions, drawn on the device and copied to the host; the
    copies are not timed. Returns {workload: {oracle: result}}."""
    import random

    import oracle
    from oracle import expanded
    rng = random.Random(seed)
    threads = oracle.default_threads()
    tthreads = torch.get_num_threads()
    res = {}

    def timed(fn):
        ts = time.perf_counter()
        fn()
        return time.perf_counter() - ts

    # Config 1: the whole tiny fp32 prefill, both oracles.
    w = inputs.TINY_PREFILL_F32
    q, k, v, r = inputs.prefill_inputs_for(w)
    t_exp = timed(lambda: oracle.prefill(q, k, v, r, threads=threads))
    t_dense = timed(lambda: expanded.prefill(q, k, v, r))
    res[w.name] = {
        "explicit": {"value": w.flops / t_exp / 1e12, "unit": "TFLOP/s", "seconds": t_exp,
                     "cores": threads, "sample": "whole workload"},
        "expanded": {"value": w.flops / t_dense / 1e12, "unit": "TFLOP/s", "seconds": t_dense,
                     "cores": tthreads, "sample": "whole workload"}}
    # Configs 2, 3: explicit on random rows, extrapolated; expanded in full.
    for w in (inputs.PREFILL_0P6B, inputs.PREFILL_1P7B):
        q, k, v, r = (t.cpu() for t in inputs.prefill_inputs_for(w, device=dev))
        f, secs, rows, _ = oracle_prefill_sample(w, q, k, v, r, explicit_budget_s,
                                                 seed=rng.randrange(1 << 30), threads=threads)
        t_dense = timed(lambda: expanded.prefill(q, k, v, r))
        res[w.name] = {
            "explicit": {"value": f / secs / 1e12, "unit": "TFLOP/s", "seconds": secs,
                         "cores": threads, "extrapolated_full_s": w.flops / (f / secs),
                         "sample": f"{rows} random causal rows, extrapolated by pair count"},
            "expanded": {"value": w.flops / t_dense / 1e12, "unit": "TFLOP/s",
                         "seconds": t_dense, "cores": tthreads, "sample": "whole workload"}}
        del q, k, v, r
    # Configs 4, 5: explicit on whole (sequence, head) pairs until the budget
    # is spent, reported per pair and as the cache rate it implies for the
    # whole batch; expanded in full.
    for w in (inputs.DECODE_B64, inputs.DECODE_RAGGED):
        q, r, kc, vc, sl = inputs.decode_inputs_for(w, device=dev)
        q, r, kc, vc = (t.cpu() for t in (q, r, kc, vc))
        lens = sl.tolist()
        pairs, secs, keys = 0, 0.0, 0
        while secs < explicit_budget_s:
            batch = [(rng.randrange(w.B), rng.randrange(w.Hq)) for _ in range(threads)]
            secs += timed(lambda: oracle.decode(q, r, kc, vc, sl, pairs=batch, threads=threads))
            pairs += len(batch)
            keys += sum(lens[b] for b, _ in batch)
        full_keys = sum(lens) * w.Hq
        full_s = secs * full_keys / keys
        by = w.bytes_moved()
        t_dense = timed(lambda: expanded.decode(q, r, kc, vc, sl))
        res[w.name] = {
            "explicit": {"value": by / full_s / 1e9, "unit": "GB/s", "seconds": secs,
                         "cores": threads, "pairs_per_s": pairs / secs,
                         "extrapolated_full_s": full_s,
                         "sample": f"{pairs} random (sequence, head) pairs, extrapolated by "
                                   "cached keys"},
            "expanded": {"value": by / t_dense / 1e9, "unit": "GB/s", "seconds": t_dense,
                         "cores": tthreads, "sample": "whole workload"}}
        del q, r, kc, vc
    return res


def run_reference(args, world, rank):
    """The oracle as the reference arm: each step is a bounded row sample."""
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    w = inputs.PREFILL_0P6B
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    q, k, v, r = inputs.prefill_inputs_for(w, device=dev)
    per_step = max(3.0, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_prefill_sample(w, q, k, v, r, 1.0, seed=7)
    flops, secs, rows, threads = 0, 0.0, 0, 1
    for s in range(args.steps):
        f, t, n, threads = oracle_prefill_sample(w, q, k, v, r, per_step, seed=100 + s)
        flops += f; secs += t; rows += n
    value = flops / secs / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * secs / max(1, args.steps), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "oracle": "explicit Sigma_KV per query, fp64, C"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"{rows} random causal rows of {w.name}, "
                                   f"~{per_step:.0f} s of CPU work per step"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


CONFIGS = {1: inputs.TINY_PREFILL_F32, 2: inputs.PREFILL_0P6B, 3: inputs.PREFILL_1P7B,
           4: inputs.DECODE_B64, 5: inputs.DECODE_RAGGED}


def run_config(args, world, rank, local):
    """Times one workload alone (one launch a step) and prints its JSON line.
    A prefill reports algorithmic TFLOP/s (8 d flops per causal pair), a decode
    algorithmic HBM GB/s; each rank runs the whole workload (replicas)."""
    from parametrized_local_linear_gb300 import (build, plx_check_device_error, plx_decode_fwd,
                                                 plx_prefill_fwd, plx_prefill_fwd_f32)
    w = CONFIGS[args.config]
    if args.seed is not None:
        w = dataclasses.replace(w, seed=args.seed)
    if rank == 0 or world == 1:
        build.build()
    barrier(world)
    build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    peaks, peaks_src = load_peaks()
    cfg = {"workload": w.name, "seed": w.seed}
    if isinstance(w, inputs.PrefillShape):
        q, k, v, r = inputs.prefill_inputs_for(w, device=dev)
        out = torch.empty_like(q)
        f32 = w.dtype == torch.float32
        call = plx_prefill_fwd_f32 if f32 else plx_prefill_fwd
        fn = lambda: call(q, k, v, r, out)  # noqa: E731
        units, scale, unit, tag = w.flops, 1e12, "TFLOP/s", "prefill"
        kernel = "prefill_f32_kernel" if f32 else "prefill_tc_kernel"
        roof = None if f32 else ("tensor", _peak(peaks, "bf16_tflops"), f"bf16_tflops ({peaks_src})")
        dtype = "f32" if f32 else "bf16"
    else:
        dq, dr, kc, vc, sl = inputs.decode_inputs_for(w, device=dev)
        lens = sl
        sl = sl.to(dev)
        out = torch.empty_like(dq)
        fn = lambda: plx_decode_fwd(dq, dr, kc, vc, sl, out, nsplit=args.nsplit)  # noqa: E731
        units, scale, unit, tag = w.bytes_moved(lens), 1e9, "GB/s", "decode"
        kernel = "decode_split_kernel + combine"
        roof = ("hbm", _peak(peaks, "hbm_gbs"), f"hbm_gbs ({peaks_src})")
        dtype = "bf16"
        cfg["nsplit"] = args.nsplit
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize(dev)
    plx_check_device_error()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        t_end = time.time() + 0.6
        while time.time() < t_end:
            fn()
            torch.cuda.synchronize(dev)
        for e0, e1 in evs:
            torch.cuda.nvtx.range_push(tag)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize(dev)
    barrier(world)
    plx_check_device_error()
    ms = sum(e0.elapsed_time(e1) for e0, e1 in evs)
    ms_max = max_over_ranks(ms, world, dev)
    K = args.steps
    value = whole_job_rate(world, units, K, ms_max) / scale
    per_launch = units / (ms / K * 1e-3) / scale
    line = {"metric": f"{w.name} {tag} {unit}", "value": value, "unit": unit, "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": ms_max / K, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": dtype, "data": "synthetic",
            "config": dict(cfg, l2="inputs fit in L2 (tiny workload)"
                           if w.name == inputs.TINY_PREFILL_F32.name else "inputs larger than L2"),
            "clocks": clk.summary(), "gpu_launches": K * (2 if tag == "decode" else 1)}
    if roof is not None:
        bound, peak, src = roof
        line["roofline"] = {"bound": bound, "kernel": kernel, "achieved": per_launch, "peak": peak,
                            "unit": unit, "frac": per_launch / peak, "peak_source": src,
                            "traffic": None}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def run_ncu_case(case):
    """Profiling-sized cases for ncu (one kernel, few launches, inputs > L2)."""
    from parametrized_local_linear_gb300 import (build, plx_check_device_error, plx_decode_fwd,
                                                 plx_prefill_fwd)
    build.build()
    dev = torch.device("cuda", 0)
    if case == "prefill":
        w = inputs.PREFILL_0P6B  # 256 MB of inputs and output
        q, k, v, r = inputs.prefill_inputs_for(w, device=dev)
        out = torch.empty_like(q)
        fn = lambda: plx_prefill_fwd(q, k, v, r, out)  # noqa: E731
    elif case == "backward":
        from parametrized_local_linear_gb300 import plx_prefill_bwd, plx_prefill_fwd_train
        w = inputs.PREFILL_0P6B  # about 0.6 GB of inputs, saved tensors and gradients
        q, k, v, r = inputs.prefill_inputs_for(w, device=dev)
        o, lse, o1, sb = plx_prefill_fwd_train(q, k, v, r)
        do = torch.randn(q.shape, device=dev).to(q.dtype)
        g = [torch.empty_like(x) for x in (q, k, v, r)]
        fn = lambda: plx_prefill_bwd(q, k, v, r, o, o1, lse, sb, do, *g)  # noqa: E731
    elif case == "projection":
        from parametrized_local_linear_gb300 import plx_qkvr_proj
        w = inputs.PREFILL_0P6B  # x 32 MB, W 12 MB, q/k/v/r 201 MB
        F = (2 * w.Hq + 2 * w.Hkv) * w.d
        x = torch.randn(w.B * w.L, 1024, device=dev).to(torch.bfloat16)
        wt = (torch.randn(F, 1024, device=dev) / 32.0).to(torch.bfloat16)
        fn = lambda: plx_qkvr_proj(x, wt, w.B, w.L, w.Hq, w.Hkv, w.d)  # noqa: E731
    else:
        if case == "decode":
            lens = [8192] * 16  # 16 x 8192 tokens x 8 heads: 537 MB of cache
        elif case == "decode_long":
            lens = [131072]  # one sequence of 131072 tokens x 8 heads: 537 MB of cache
        else:
            lens = [1024, 40000, 3000, 17000]  # ragged, 250 MB of cache
        dq, dr, kc, vc, sl = inputs.decode_inputs(len(lens), 16, 8, 128, lens, torch.bfloat16,
                                                  0.05, 5, device=dev)
        sl = sl.to(dev)
        out = torch.empty_like(dq)
        fn = lambda: plx_decode_fwd(dq, dr, kc, vc, sl, out)  # noqa: E731
    for _ in range(6):
        fn()
    torch.cuda.synchronize(dev)
    plx_check_device_error()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="plx", choices=["plx", "reference"])
    ap.add_argument("--no-extra", action="store_true", help="skip the 1.7B / ragged timings")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--shard", action="store_true",
                    help="under torchrun, deal one batch's (sequence, kv head) units among the "
                         "ranks (strong scaling) instead of a full replica per rank")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--config", type=int, choices=sorted(CONFIGS), default=None,
                    help="time one workload alone: 1 fp32 tiny prefill, 2 0.6B-shaped prefill, "
                         "3 1.7B-shaped prefill, 4 batched decode, 5 ragged decode")
    ap.add_argument("--seed", type=int, default=None, help="input seed for --config")
    ap.add_argument("--nsplit", type=int, default=0,
                    help="decode share count for --config 4/5 (0: the library's default)")
    ap.add_argument("--ncu-case", choices=["prefill", "decode", "decode_ragged", "decode_long", "backward",
                                           "projection"], default=None,
                    help="run 3 warm-up + 3 launches of one kernel on a profiling-sized case "
                         "(inputs > L2, < 1 GB) and exit; prints nothing")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.ncu_case:
        return run_ncu_case(args.ncu_case)
    world, rank, local = dist_setup()
    if args.impl == "reference":
        return run_reference(args, world, rank)
    if args.config is not None:
        return run_config(args, world, rank, local)

    from parametrized_local_linear_gb300 import (build, plx_check_device_error, plx_decode_fwd,
                                                 plx_prefill_fwd)
    if rank == 0 or world == 1:
        build.build()
    barrier(world)
    build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    peaks, peaks_src = load_peaks()

    wp, wd = inputs.PREFILL_0P6B, inputs.DECODE_B64
    q, k, v, r = inputs.prefill_inputs_for(wp, device=dev)
    out = torch.empty_like(q)
    lse = torch.empty(wp.B, wp.Hq, wp.L, device=dev)
    dq, dr, kc, vc, sl = inputs.decode_inputs_for(wd, device=dev)
    lens = sl.tolist()
    sl = sl.to(dev)
    dout = torch.empty_like(dq)
    dbytes = wd.bytes_moved()
    G = wp.Hq // wp.Hkv
    # This rank's prefill calls (b, kv0, kv1) and decode sequences [b0, b1):
    # with --shard its share of the one batch; otherwise (replicas) the whole
    # batch, whose timed prefill is one batched call and whose end-to-end leg
    # calls the prefill once per sequence.
    if args.shard:
        pcalls = prefill_shard(wp.B, wp.Hkv, world, rank)
        b0, b1 = decode_shard(lens, world, rank)
    else:
        pcalls = [(b, 0, wp.Hkv) for b in range(wp.B)]
        b0, b1 = 0, wd.B
    tok0, tok1 = sum(lens[:b0]), sum(lens[:b1])
    own_flops = sum(8 * wp.d * (c[2] - c[1]) * G * wp.L * (wp.L + 1) // 2 for c in pcalls)
    own_dbytes = (2 * (tok1 - tok0) * wd.Hkv * wd.d + 3 * (b1 - b0) * wd.Hq * wd.d) * 2

    def pviews(b, kv0, kv1, ts=(q, k, v, r, out, lse)):
        qq, kk, vv, rr, oo, ll = ts
        h0, h1 = kv0 * G, kv1 * G
        return (qq[b:b + 1, h0:h1], kk[b:b + 1, kv0:kv1], vv[b:b + 1, kv0:kv1], rr[b:b + 1, h0:h1],
                oo[b:b + 1, h0:h1], ll[b:b + 1, h0:h1])

    dviews = (dq[b0:b1], dr[b0:b1], kc[tok0:tok1], vc[tok0:tok1], sl[b0:b1], dout[b0:b1])

    def step(ev):
        torch.cuda.nvtx.range_push("prefill")
        ev[0].record(stream)
        if args.shard:
            for c in pcalls:
                plx_prefill_fwd(*pviews(*c))
        else:
            plx_prefill_fwd(q, k, v, r, out, lse)
        ev[1].record(stream)
        torch.cuda.nvtx.range_pop()
        torch.cuda.nvtx.range_push("decode")
        if b1 > b0:
            plx_decode_fwd(*dviews)
        ev[2].record(stream)
        torch.cuda.nvtx.range_pop()

    for _ in range(args.warmup):
        step([torch.cuda.Event(enable_timing=True) for _ in range(3)])
    torch.cuda.synchronize(dev)
    plx_check_device_error()

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        # Keep the GPU busy while the sampler starts, so its samples are taken
        # under load; these steps are not timed.
        t_end = time.time() + 0.6
        while time.time() < t_end:
            step([torch.cuda.Event(enable_timing=True) for _ in range(3)])
            torch.cuda.synchronize(dev)
        t0 = torch.cuda.Event(enable_timing=True); t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for i in range(args.steps):
            step(evs[i])
        t1.record(stream)
        torch.cuda.synchronize(dev)
    barrier(world)
    plx_check_device_error()
    pre_ms = sum(e[0].elapsed_time(e[1]) for e in evs)
    dec_ms = sum(e[1].elapsed_time(e[2]) for e in evs)
    total_ms = t0.elapsed_time(t1)
    pre_ms_max = max_over_ranks(pre_ms, world, dev)
    dec_ms_max = max_over_ranks(dec_ms, world, dev)
    total_ms_max = max_over_ranks(total_ms, world, dev)
    K = args.steps
    if args.shard:
        value = sharded_rate(wp.flops, K, pre_ms_max) / 1e12
        dec_gbs = sharded_rate(dbytes, K, dec_ms_max) / 1e9
    else:
        value = whole_job_rate(world, wp.flops, K, pre_ms_max) / 1e12
        dec_gbs = whole_job_rate(world, dbytes, K, dec_ms_max) / 1e9
    # Per-launch rates of this rank's own work (rank 0 prints them).
    pre_launch_s = pre_ms / K * 1e-3
    dec_launch_s = dec_ms / K * 1e-3
    pre_launch_flops = wp.flops if not args.shard else own_flops
    dec_launch_bytes = dbytes if not args.shard else own_dbytes
    tc_peak = _peak(peaks, "bf16_tflops")
    hbm_peak = _peak(peaks, "hbm_gbs")

    # ---------------------------------------------------------------- e2e
    # Through the same C-ABI calls, from pinned host buffers, with the copies
    # inside the timing: each sequence's q, k, v, r go to the device on a copy
    # stream while the previous sequence's prefill runs (one plx_prefill_fwd
    # call per sequence), the decode's new q, r follow, and each output comes
    # back while later work runs. A step ends when its last copy has landed.
    # Measured on GB300: the host link moves about 210 GB/s host to device and
    # 192 GB/s back, the same with 1 to 8 DMA streams or an SM copy kernel, so
    # the copies, not the kernels, bound this leg (201 MB up, 67 MB back: 1.31
    # ms of link time against 1.45 ms a step). Sending the outputs back on a
    # second stream, concurrently with the inputs, was slower (1.51 ms): both
    # directions at once drop to about 169 GB/s each, and the inputs are on
    # the critical path.
    hq = [t.cpu().pin_memory() for t in (q, k, v, r)]
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    hd = [t[b0:b1].cpu().pin_memory() for t in (dq, dr)]
    hdout = torch.empty(dout[b0:b1].shape, dtype=dout.dtype).pin_memory()

    def hviews(b, kv0, kv1):
        h0, h1 = kv0 * G, kv1 * G
        return (hq[0][b:b + 1, h0:h1], hq[1][b:b + 1, kv0:kv1], hq[2][b:b + 1, kv0:kv1],
                hq[3][b:b + 1, h0:h1])

    nbytes = lambda t: t.numel() * t.element_size()  # noqa: E731
    h2d = sum(nbytes(t) for c in pcalls for t in hviews(*c)) + sum(nbytes(t) for t in hd)
    d2h = sum(nbytes(pviews(*c)[4]) for c in pcalls) + nbytes(hdout)
    copy_stream = torch.cuda.Stream(dev)
    dseq = [[torch.empty_like(t, device=dev) for t in hviews(*c)] for c in pcalls]
    dseq_out = [torch.empty_like(pviews(*c)[4]) for c in pcalls]
    ddec = [torch.empty_like(t, device=dev) for t in hd]
    ddec_out = torch.empty_like(hdout, device=dev)
    hout_views = [pviews(*c, ts=(hq[0], hq[1], hq[2], hq[3], hout, hout))[4] for c in pcalls]

    def e2e_step():
        ev_in = []
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_stream(stream)  # the previous step is done with the buffers
            for c, dst_c in zip(pcalls, dseq):
                for dst, src in zip(dst_c, hviews(*c)):
                    dst.copy_(src, non_blocking=True)
                ev_in.append(torch.cuda.Event())
                ev_in[-1].record(copy_stream)
            for dst, src in zip(ddec, hd):
                dst.copy_(src, non_blocking=True)
            ev_dec = torch.cuda.Event()
            ev_dec.record(copy_stream)
        ev_out = []
        for n in range(len(pcalls)):
            stream.wait_event(ev_in[n])
            plx_prefill_fwd(*dseq[n], dseq_out[n])
            ev_out.append(torch.cuda.Event())
            ev_out[-1].record(stream)
        stream.wait_event(ev_dec)
        if b1 > b0:
            plx_decode_fwd(ddec[0], ddec[1], kc[tok0:tok1], vc[tok0:tok1], sl[b0:b1], ddec_out)
        ev_d = torch.cuda.Event()
        ev_d.record(stream)
        with torch.cuda.stream(copy_stream):
            for n in range(len(pcalls)):
                copy_stream.wait_event(ev_out[n])
                hout_views[n].copy_(dseq_out[n], non_blocking=True)
            copy_stream.wait_event(ev_d)
            hdout.copy_(ddec_out, non_blocking=True)
        stream.wait_stream(copy_stream)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True); e1 = torch.cuda.Event(enable_timing=True)
    ke = max(3, min(K, 10))
    barrier(world)
    e0.record(stream)
    for _ in range(ke):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev) / ke
    # The slices called separately give bit for bit the batched call's output.
    for c, hv in zip(pcalls, hout_views):
        if not torch.equal(hv, pviews(*c)[4].cpu()):
            raise RuntimeError(f"e2e prefill output of call {c} differs from the batched call")
    # The e2e step also contains the decode; count its time, credit only prefill flops.
    if args.shard:
        e2e_value = wp.flops / (e2e_ms * 1e-3) / 1e12
    else:
        e2e_value = world * wp.flops / (e2e_ms * 1e-3) / 1e12

    # ---------------------------------------------------------------- extra
    extra = {}
    if not args.no_extra and not args.shard:
        del hq, hd
        from parametrized_local_linear_gb300 import (plx_decode_fwd_cor, plx_prefill_fwd_chunk,
                                                     plx_prefill_fwd_cor)
        a = torch.cuda.Event(enable_timing=True); b = torch.cuda.Event(enable_timing=True)

        def launch_s(fn, n):
            """Mean seconds per call of fn() over n back-to-back calls after 3
            untimed ones (CUDA events on the launching stream)."""
            for _ in range(3):
                fn()
            a.record(stream)
            for _ in range(n):
                fn()
            b.record(stream)
            torch.cuda.synchronize(dev)
            return a.elapsed_time(b) / n * 1e-3

        l2_flush = torch.ones(128 << 20, dtype=torch.float32, device=dev)  # 512 MB

        def flush_l2():
            # A read-only pass over 512 MB: L2 ends up holding clean lines of
            # this buffer. A write (memset) would leave up to an L2 of dirty
            # lines whose write-back the next kernel would pay for: about
            # 25 us more for a 537 MB decode, against its ncu time.
            l2_flush.sum()

        def launch_cold_s(fn, n):
            """Mean seconds per call of fn() with L2 flushed before each call
            (a 512 MB read outside the timed interval), 3 untimed calls first.
            Eight flushes go ahead of the loop so that the host, enqueueing
            through the Python binding, stays ahead of the GPU: a gap between
            the first event and a short kernel would otherwise be timed."""
            for _ in range(3):
                fn()
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(n)]
            for _ in range(8):
                flush_l2()
            for e0, e1 in evs:
                flush_l2()
                e0.record(stream)
                fn()
                e1.record(stream)
            torch.cuda.synchronize(dev)
            return sum(e0.elapsed_time(e1) for e0, e1 in evs) / n * 1e-3

        def tflops(name, flops, t):
            extra[name] = {"value": flops / t / 1e12, "unit": "TFLOP/s", "ms": t * 1e3,
                           "frac_of_peak": flops / t / 1e12 / tc_peak}

        w3 = inputs.PREFILL_1P7B
        q3, k3, v3, r3 = inputs.prefill_inputs_for(w3, device=dev)
        o3 = torch.empty_like(q3)
        tflops(w3.name, w3.flops, launch_s(lambda: plx_prefill_fwd(q3, k3, v3, r3, o3), 5))
        # Chunked prefill: the last 2048 positions of a 16384-token sequence
        # (a new chunk against an existing cache), 1.7B-shaped heads.
        lq, lk = 2048, w3.L
        qc, rc = q3[:, :, -lq:].contiguous(), r3[:, :, -lq:].contiguous()
        oc = torch.empty_like(qc)
        cflops = 8 * w3.d * w3.B * w3.Hq * (lq * (lk - lq) + lq * (lq + 1) // 2)
        tflops("prefill_chunk_Lq2048_Lk16384_B1_Hq16_Hkv8_d128", cflops,
               launch_s(lambda: plx_prefill_fwd_chunk(qc, k3, v3, rc, oc), 5))
        del q3, k3, v3, r3, o3, qc, rc, oc
        # The correction-to-output ratio as a side output of the same calls.
        cor = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
        tflops(wp.name + "_with_cor", wp.flops,
               launch_s(lambda: plx_prefill_fwd_cor(q, k, v, r, out, None, cor), 10))
        dcor = torch.empty(dq.shape[:2], dtype=torch.float32, device=dev)
        td = launch_s(lambda: plx_decode_fwd_cor(dq, dr, kc, vc, sl, dout, dcor), 10)
        extra[wd.name + "_with_cor"] = {"value": dbytes / td / 1e9, "unit": "GB/s", "ms": td * 1e3,
                                        "frac_of_peak": dbytes / td / 1e9 / hbm_peak}
        # Training: the forward that saves o^SA and sbar, and the backward
        # (algorithmic flops: 8 length-d dot products per causal pair, twice
        # the forward's).
        from parametrized_local_linear_gb300 import plx_prefill_bwd, plx_prefill_fwd_train
        o_t, lse_t, o1_t, sb_t = plx_prefill_fwd_train(q, k, v, r)
        do_t = torch.randn(q.shape, device=dev, dtype=torch.float32).to(q.dtype)
        gq, gk, gv, gr = (torch.empty_like(x) for x in (q, k, v, r))
        tflops(wp.name + "_forward_train", wp.flops,
               launch_s(lambda: plx_prefill_fwd_train(q, k, v, r, o_t, lse_t, o1_t, sb_t), 10))
        tflops(wp.name + "_backward", 2 * wp.flops,
               launch_s(lambda: plx_prefill_bwd(q, k, v, r, o_t, o1_t, lse_t, sb_t, do_t,
                                                gq, gk, gv, gr), 10))
        del o_t, lse_t, o1_t, sb_t, do_t, gq, gk, gv, gr
        # The fused input projection x [W_Q; W_K; W_V; W_R]^T of the 0.6B- and
        # 1.7B-shaped layers (model dims 1024 and 2048), all B L tokens.
        from parametrized_local_linear_gb300 import plx_qkvr_proj
        for dm, tag in ((1024, "0p6b"), (2048, "1p7b")):
            F = (2 * wp.Hq + 2 * wp.Hkv) * wp.d
            xt = torch.randn(wp.B * wp.L, dm, device=dev).to(torch.bfloat16)
            wt = (torch.randn(F, dm, device=dev) / dm ** 0.5).to(torch.bfloat16)
            po = [torch.empty_like(t) for t in (q, k, v, r)]
            tflops(f"qkvr_projection_{tag}_T{wp.B * wp.L}_D{dm}_F{F}", 2 * wp.B * wp.L * dm * F,
                   launch_s(lambda: plx_qkvr_proj(xt, wt, wp.B, wp.L, wp.Hq, wp.Hkv, wp.d, *po), 10))
            del xt, wt, po
        # Sweeps (head layout of the 0.6B / 1.7B models: Hq 16, Hkv 8, d 128):
        # prefill at several context lengths with 16384 tokens per call, and
        # decode across batch sizes (8192 cached tokens) and contexts (16
        # sequences), each decode call after an L2 flush (several of these
        # caches fit in L2).
        for B_, L_ in ((16, 1024), (8, 2048), (2, 8192), (1, 32768)):
            qs, ks, vs, rs = inputs.prefill_inputs(B_, 16, 8, L_, 128, torch.bfloat16, 0.05, 2000 + L_,
                                                   device=dev)
            os_ = torch.empty_like(qs)
            fl = 8 * 128 * B_ * 16 * L_ * (L_ + 1) // 2
            tflops(f"prefill_sweep_B{B_}_L{L_}", fl,
                   launch_s(lambda: plx_prefill_fwd(qs, ks, vs, rs, os_), 5))
            del qs, ks, vs, rs, os_
        for B_, ctx in ((1, 512), (1, 2048), (1, 8192), (1, 131072), (4, 8192), (8, 8192),
                        (32, 8192), (128, 8192), (16, 2048), (16, 32768)):
            ds = inputs.decode_inputs(B_, 16, 8, 128, [ctx] * B_, torch.bfloat16, 0.05, 3000 + B_,
                                      device=dev)
            sls = ds[4].to(dev)
            ods = torch.empty_like(ds[0])
            by = 2 * B_ * ctx * 8 * 128 * 2 + 3 * B_ * 16 * 128 * 2
            td = launch_cold_s(lambda: plx_decode_fwd(ds[0], ds[1], ds[2], ds[3], sls, ods), 10)
            extra[f"decode_sweep_B{B_}_ctx{ctx}"] = {"value": by / td / 1e9, "unit": "GB/s",
                                                     "ms": td * 1e3,
                                                     "frac_of_peak": by / td / 1e9 / hbm_peak,
                                                     "l2": "flushed (512 MB read) before each call"}
            del ds, sls, ods
        w5 = inputs.DECODE_RAGGED
        d5 = inputs.decode_inputs_for(w5, device=dev)
        sl5 = d5[4].to(dev)
        o5 = torch.empty_like(d5[0])
        t5 = launch_s(lambda: plx_decode_fwd(d5[0], d5[1], d5[2], d5[3], sl5, o5), 10)
        by5 = w5.bytes_moved()
        extra[w5.name] = {"value": by5 / t5 / 1e9, "unit": "GB/s", "ms": t5 * 1e3,
                          "bytes": by5, "seqlens": w5.seqlens().tolist(),
                          "frac_of_peak": by5 / t5 / 1e9 / hbm_peak}
        del d5
        plx_check_device_error()

    # ---------------------------------------------------------------- cpu baseline
    cpu, cpu_plan = None, None
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        import oracle
        oracle.build()
        f, secs, rows, threads = oracle_prefill_sample(wp, q, k, v, r, args.cpu_seconds, seed=11)
        cpu = {"value": f / secs / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "sample": f"{rows} random causal rows of {wp.name} (explicit Sigma_KV, fp64), "
                         f"{secs:.1f} s"}
        if extra:
            for name, base in oracle_extra_samples(wp, q, k, v, r, args.cpu_seconds / 4).items():
                if name in extra:
                    extra[name]["cpu_baseline"] = base
        cpu_plan = cpu_baseline_plan(dev, explicit_budget_s=args.cpu_seconds / 3)

    clocks = clk.summary()
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": total_ms_max / K,
        "higher_is_better": True,
        "scaling": "strong" if args.shard else "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": wp.name, "decode_workload": wd.name,
                   "step": "prefill 0.6B-shaped + decode B64 ctx8192",
                   "l2": "inputs larger than L2 (prefill 256 MB, decode 2.1 GB); no flush",
                   "parallelism": (f"one batch sharded over (sequence, kv head) units x{world}"
                                   if args.shard else
                                   f"replicas x{world}" if world > 1 else "single GPU")},
        "roofline": {"bound": "tensor", "kernel": "prefill_tc_kernel",
                     "achieved": pre_launch_flops / pre_launch_s / 1e12, "peak": tc_peak,
                     "unit": "TFLOP/s", "frac": pre_launch_flops / pre_launch_s / 1e12 / tc_peak,
                     "peak_source": f"bf16_tflops ({'of measured' if peaks_src == 'measured' else 'of fallback'})",
                     "traffic": NCU_TRAFFIC_BYTES["prefill_tc_kernel"],
                     "algorithmic_flops_per_launch": pre_launch_flops},
        "decode": {"workload": wd.name, "value": dec_gbs, "unit": "GB/s",
                   "ms": dec_launch_s * 1e3,
                   "roofline": {"bound": "hbm", "kernel": "decode_split_kernel + combine",
                                "achieved": dec_launch_bytes / dec_launch_s / 1e9,
                                "peak": hbm_peak, "unit": "GB/s",
                                "frac": dec_launch_bytes / dec_launch_s / 1e9 / hbm_peak,
                                "peak_source": f"hbm_gbs ({peaks_src})",
                                "traffic": NCU_TRAFFIC_BYTES["decode_split_kernel"],
                                "algorithmic_bytes_per_launch": dec_launch_bytes}},
        "extra": extra,
        "cpu_baseline": cpu,
        "cpu_baselines": cpu_plan,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "method": "one prefill call per sequence; host copies on a second stream, "
                          "overlapped with the kernels, inside the timing; the host link "
                          "(about 210 GB/s up, 192 GB/s down) bounds it"},
        "gpu_launches": K * ((len(pcalls) if args.shard else 1) + (2 if b1 > b0 else 0)),
        "clocks": clocks,
        "gpu": torch.cuda.get_device_name(dev),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
