#!/usr/bin/env python3
"""Benchmark of the group-quantized 4-bit matmul library on GB300.

Headline workload (one line of JSON on rank 0): the M = 1 decode projections of
a Gemma-shaped decoder (gate_up 1536->12288, down 6144->1536, q 1536->2048,
o 2048->1536), W4A8 with group 64, 64-wide Hadamard rotation of the
activations, x ~ N(0,1) with 1% +-20 outliers. One step is one decode pass
over LAYERS layers with their own weights: for each projection one fused
launch (activation prepass + GEMV in one kernel). The metric is weight+scale
bytes streamed per second.
The per-step weights (> 2x L2) are larger than L2, so no flush is needed.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference] [--no-sweep]
  python bench.py --profile-case prefill_gemm:1068     (a few GEMM launches, for ncu; also prep_rotated:M,
                                                        lm_head_gemv:1, lm_head_gemv_cq4:1, lm_head_gemm:M,
                                                        lm_head_gemm_f16:M, affine_gemm:M)

The step is captured once in a CUDA graph (the kernels are launched with
programmatic dependent launch, so each GEMV streams its weights while the
previous kernel drains) and replayed K times between CUDA events. Under
torchrun each rank runs its own replica (weak scaling); the time is the max
over ranks. ``--impl reference`` times the CPU oracle on the host instead.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import qmm_synth  # noqa: E402

LAYERS = 32
PROJ = [("gate_up", 12288, 1536), ("down", 1536, 6144), ("q", 2048, 1536), ("o", 1536, 2048)]
GROUP = 64
W4A8, AFFINE, CQ4 = 0, 1, 2
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "gemv_fused_w4a8_gemma_decode.txt")
GEMV_SOURCE = os.path.join(ROOT, "bit_group_quantized_qmm_gb300", "csrc", "qmm_gemv_fused.cu")


# ------------------------------------------------------------------ plumbing

def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--layers", type=int, default=LAYERS)
    p.add_argument("--no-sweep", action="store_true", help="skip the other workloads' extra figures")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-cpu-all-cores", action="store_true", help="skip the all-core oracle figure")
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--peaks", action="store_true",
                   help="compile and run the FP32 / mma.sync peak microbenchmark and exit (one JSON line)")
    p.add_argument("--profile-case", default=None, metavar="prefill_gemm:M|prep_rotated:M|lm_head_gemv[_cq4]:1|lm_head_gemm[_f16]:M|affine_gemm:M",
                   help="run one prefill GEMM shape a few times and exit (for profilers; prints one JSON line)")
    return p.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(world, use_cuda):
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend="nccl" if use_cuda else "gloo")


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """Largest value of x over all ranks (x itself when world == 1)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples every 100 ms while running."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        rows = []
        if self.path and os.path.exists(self.path):
            with open(self.path) as f:
                for ln in f:
                    parts = [p.strip() for p in ln.split(",")]
                    if len(parts) >= 10:
                        rows.append(parts)
            os.unlink(self.path)
        return rows

    @staticmethod
    def summarize(rows):
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        smax = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for name, val in zip(names, r[6:10]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        power = [float(r[4]) for r in rows if r[4].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_median": statistics.median(power) if power else None}


# ------------------------------------------------------------------ workload

def layer_inputs(seed, rank, layer, name, N, K):
    prefix = f"gemma_decode/r{rank}/l{layer}/{name}"
    lay = qmm_synth.Layer(name, W4A8, N, K, GROUP, GROUP, outlier_frac=0.01)
    qb, sw, _ = qmm_synth.layer_weights(seed, prefix, lay)
    x = qmm_synth.layer_activations(seed, prefix, lay, 1)
    return lay, qb, sw, x


class DecodeModel:
    """Packed weights and per-projection buffers of LAYERS decoder layers."""

    def __init__(self, layers, rank, keep_host=False):
        import torch
        import bit_group_quantized_qmm_gb300 as q
        self.q = q
        dev = torch.device("cuda", torch.cuda.current_device())
        self.projs = []
        self.host = []
        xs, ys = [], []
        x_off = y_off = 0
        for l in range(layers):
            for name, N, K in PROJ:
                lay, qb, sw, x = layer_inputs(0, rank, l, name, N, K)
                d = q.weight_desc(W4A8, N, K, GROUP)
                packed = torch.empty(q.qmm_packed_size(d), dtype=torch.uint8, device=dev)
                q.qmm_pack_weights(d, torch.from_numpy(qb).to(dev), torch.from_numpy(sw.view(np.int16)).to(dev),
                                   None, packed)
                self.projs.append(dict(name=name, N=N, K=K, d=d, packed=packed, x_off=x_off, y_off=y_off))
                if keep_host:
                    self.host.append((qb, sw, x))
                xs.append(x.reshape(-1))
                x_off += K
                y_off += N
        torch.cuda.synchronize()
        self.x_host = torch.from_numpy(np.concatenate(xs)).pin_memory()
        self.x = self.x_host.to(dev)
        self.y = torch.zeros(y_off, dtype=torch.float32, device=dev)
        self.y_host = torch.empty(y_off, dtype=torch.float32).pin_memory()
        kmax = max(K for _, _, K in PROJ)
        self.a = [torch.empty(K, dtype=torch.int8, device=dev) for _, _, K in PROJ]
        self.sx = [torch.empty(K // GROUP, dtype=torch.float32, device=dev) for _, _, K in PROJ]
        ws_bytes = max(q.qmm_gemv_workspace_size(p["d"]) for p in self.projs)
        self.ws = torch.zeros(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
        self.ws_bytes = ws_bytes
        self.kmax = kmax
        # bytes
        self.weight_bytes = sum(q.qmm_packed_size(p["d"]) for p in self.projs)
        self.act_bytes = sum(p["K"] * 1 + (p["K"] // GROUP) * 4 + p["N"] * 4 for p in self.projs)
        self.h2d_bytes = self.x.numel() * 4
        self.d2h_bytes = self.y.numel() * 4

    def enqueue_step(self, x_all=None, y_all=None):
        """One decode pass: one fused prepass + GEMV launch per projection
        (on the model's own x / y buffers unless others are given)."""
        q = self.q
        x_all = self.x if x_all is None else x_all
        y_all = self.y if y_all is None else y_all
        for p in self.projs:
            x = x_all[p["x_off"]:p["x_off"] + p["K"]]
            q.qmm_gemv_fused(p["d"], p["packed"], x, 0, GROUP, y_all[p["y_off"]:p["y_off"] + p["N"]])

    def enqueue_step_two_kernels(self):
        """The same pass through qmm_prep_act + qmm_gemv (two launches per projection)."""
        q = self.q
        for i, p in enumerate(self.projs):
            j = i % len(PROJ)
            x = self.x[p["x_off"]:p["x_off"] + p["K"]]
            q.qmm_prep_act(W4A8, 1, p["K"], GROUP, GROUP, x, 0, a=self.a[j], sx=self.sx[j])
            q.qmm_gemv(p["d"], p["packed"], self.a[j], self.sx[j], self.y[p["y_off"]:p["y_off"] + p["N"]],
                       self.ws, self.ws_bytes)

    def fused_algorithmic_bytes(self):
        """Per step: packed nibbles + scales, fp32 x in, fp32 y out."""
        return self.weight_bytes + sum(4 * p["K"] + 4 * p["N"] for p in self.projs)


def capture(fn):
    import torch
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()          # eager warm-up: first-call set-up happens outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def time_graph(g, steps, warmup, world):
    """Seconds for `steps` replays, CUDA events on the replay stream, max over ranks."""
    import torch
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    barrier(world)
    return e0.elapsed_time(e1) / 1e3


def gemv_traffic_per_step(model):
    """DRAM bytes of the GEMV launches of one step, from the committed ncu
    summary, or None when the kernel changed since it was taken."""
    if not os.path.exists(PROFILE_TRAFFIC):
        return None
    src_hash = hashlib.sha256(open(GEMV_SOURCE, "rb").read()).hexdigest()[:16]
    vals = {}
    with open(PROFILE_TRAFFIC) as f:
        for ln in f:
            if ":" in ln and not ln.startswith("#"):
                k, _, v = ln.partition(":")
                vals[k.strip()] = v.strip()
    if vals.get("gemv_source_sha256_16") != src_hash:
        return None
    try:
        per_weight_byte = float(vals["dram_bytes_per_weight_byte"])
    except (KeyError, ValueError):
        return None
    return per_weight_byte * model.weight_bytes


# ------------------------------------------------------------------ CPU baseline (oracle)

def cpu_oracle_rate(host, seconds, rows_cap=None):
    """Oracle (single-threaded C) on the decode projections, cycling through
    them until `seconds` pass: prepass of x, then the outputs of the sampled
    rows. Returns (weight+scale bytes per second, description)."""
    import oracle
    orc = oracle.default()
    t0 = time.perf_counter()
    done_bytes = 0
    n_proj = 0
    while True:
        for qb, sw, x in host:
            N, K = qb.shape[0], qb.shape[1] * 2
            rows = None
            nr = N
            if rows_cap and rows_cap < N:
                rows = np.arange(0, N, max(1, N // rows_cap), dtype=np.int32)[:rows_cap]
                nr = rows.size
            a, sx, _ = orc.prep_w4a8(x, GROUP, GROUP)
            orc.gemm_w4a8(qb, sw, a, sx, GROUP, rows=rows)
            done_bytes += nr * (K // 2 + 2 * (K // GROUP))
            n_proj += 1
            if time.perf_counter() - t0 >= seconds:
                el = time.perf_counter() - t0
                return done_bytes / el / 1e9, n_proj, el


_CPU_HOST = None


def _cpu_pool_init(host):
    global _CPU_HOST
    _CPU_HOST = host


def _cpu_pool_work(seconds):
    rate, n, el = cpu_oracle_rate(_CPU_HOST, seconds)
    return rate * el * 1e9, n, el


def cpu_oracle_rate_all_cores(host, seconds):
    """The same oracle passes in one process per host core (spawned), each
    timing itself for `seconds`. Returns (aggregate GB/s, processes, passes)."""
    import multiprocessing as mp
    n = os.cpu_count() or 1
    with mp.get_context("spawn").Pool(n, initializer=_cpu_pool_init, initargs=(host,)) as pool:
        res = pool.map(_cpu_pool_work, [seconds] * n)
    total = sum(r[0] for r in res)
    return total / max(r[2] for r in res) / 1e9, n, sum(r[1] for r in res)


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle, as it stands, on the host cores."""
    if rank != 0:
        return      # rank 0 alone times the oracle; the other ranks exit without work
    host = []
    for l in range(2):
        for name, N, K in PROJ:
            _, qb, sw, x = layer_inputs(0, 0, l, name, N, K)
            host.append((qb, sw, x))
    import oracle
    orc = oracle.default()
    # one step = the prepass and 64 sampled output rows of one projection
    rows_per_step = 64
    times, nbytes = [], 0
    total = args.warmup + args.steps
    t_budget = 150.0
    t_start = time.perf_counter()
    for s in range(total):
        qb, sw, x = host[s % len(host)]
        N, K = qb.shape[0], qb.shape[1] * 2
        rows = np.linspace(0, N - 1, rows_per_step).astype(np.int32)
        t0 = time.perf_counter()
        a, sx, _ = orc.prep_w4a8(x, GROUP, GROUP)
        orc.gemm_w4a8(qb, sw, a, sx, GROUP, rows=rows)
        dt = time.perf_counter() - t0
        if s >= args.warmup:
            times.append(dt)
            nbytes += rows_per_step * (K // 2 + 2 * (K // GROUP))
        if time.perf_counter() - t_start > t_budget:
            break
    el = sum(times) if times else float("nan")
    value = nbytes / el / 1e9 if times else None
    line = {
        "impl": "reference", "metric": "GEMV weight GB/s (decode projections, M=1)", "value": value, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": len(times), "warmup": args.warmup,
        "ms_per_step": 1e3 * el / max(1, len(times)), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int8", "data": "synthetic",
        "config": {"workload": "gemma_decode (sampled rows)", "sample": f"{rows_per_step} output rows per step"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"prepass + {rows_per_step} sampled rows of one projection per step, "
                                   f"cycling through 8 projections"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ sweep of the other workloads

# Peak of the legacy warp-level int8 MMA (mma.sync.m16n8k32.s8, int32
# accumulators) on this GPU, measured with `python bench.py --peaks`: 223 MACs
# per clock per SM (the tcgen05 kind::f16 MMA the GEMM issues does 4096). The
# sweep reports every GEMM's TOPS against it beside the bf16 figure.
MMA_SYNC_S8_MAC_PER_CLK_SM = 223.0


def s8_peak_tops(sm_mhz=None):
    """mma.sync s8 peak in TOPS at the given SM clock (default: the measured maximum)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    mhz = sm_mhz
    if mhz is None:
        mhz = 2070.0
        if os.path.exists(path):
            with open(path) as f:
                mhz = float(json.load(f).get("sm_max_mhz", mhz))
    return 2.0 * MMA_SYNC_S8_MAC_PER_CLK_SM * 152 * mhz * 1e6 / 1e12


def ab_time(fns, calls, rounds=6, iters=10):
    """Alternating best-of timing: one CUDA graph per function, replayed
    `iters` times per round; the rounds alternate the order (A B, B A, A B,
    ...) so that a drift of the clock or of the other users hits every
    function alike. Per function: the best round's time per call, the median,
    the spread ((worst - best) / best) and the number of rounds."""
    graphs = {k: capture(f) for k, f in fns.items()}
    keys = list(fns)
    samples = {k: [] for k in keys}
    for r in range(rounds):
        for k in (keys if r % 2 == 0 else keys[::-1]):
            samples[k].append(time_graph(graphs[k], iters, 2, 1) / iters / calls[k])
    out = {}
    for k, v in samples.items():
        best = min(v)
        out[k] = {"us_per_call": best * 1e6, "us_median": statistics.median(v) * 1e6,
                  "spread": (max(v) - best) / best, "rounds": rounds}
    del graphs
    return out


def eager_us(fn, calls, reps=3):
    """Time per call of eager (not captured) calls: CUDA events around `calls`
    back-to-back calls from Python, best of `reps` (host launch cost included)."""
    import torch
    best = float("inf")
    fn()
    torch.cuda.synchronize()
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1) * 1e3 / calls)
    return best


# --- oracle tasks (the CPU baseline beside every sweep row)

def _oracle_run(task):
    """One pass of a row's sampled oracle work; returns seconds."""
    import oracle
    orc = oracle.default()
    t0 = time.perf_counter()
    kind = task["kind"]
    if kind == "w4a8":
        a, sx, _ = orc.prep_w4a8(task["x"], task["group"], task["had"])
        for qb, sw in task["mats"]:
            orc.gemm_w4a8(qb, sw, a, sx, task["group"])
    elif kind == "affine":
        orc.gemm_affine(task["qb"], task["s"], task["b"], task["x16"])
    elif kind == "rotated_cq4":
        a, sx, _, _ = orc.prep_rotated(task["R"], task["x"], 128)
        orc.gemm_cq4(task["idx"], task["C"], task["cb"], task["sw"], a, sx, 128)
    return time.perf_counter() - t0


def _oracle_loop(args):
    task, seconds = args
    n, t0 = 0, time.perf_counter()
    while True:
        _oracle_run(task)
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            return n, el


def oracle_baselines(rows, pool, seconds=0.6):
    """For every (row, task): the oracle's sampled work timed single-threaded
    in this process and, in parallel, in one spawned process per host core.
    The task's `bytes` / `ops` are the weight bytes and operations of the
    sampled work; `full_bytes` those of the whole call."""
    ncores = os.cpu_count() or 1
    for row, task in rows:
        n1, el1 = _oracle_loop((task, seconds))
        rate1 = task["bytes"] * n1 / el1
        base = {"kind": "oracle", "cores": 1, "sample": task["sample"],
                "weight_GBps": rate1 / 1e9,
                "us_per_call_est": task["full_bytes"] / rate1 * 1e6}
        if task.get("ops"):
            base["GOPS"] = task["ops"] * n1 / el1 / 1e9
        if pool is not None:
            res = pool.map(_oracle_loop, [(task, seconds)] * ncores)
            el = max(r[1] for r in res)
            nall = sum(r[0] for r in res)
            allc = {"cores": ncores, "weight_GBps": task["bytes"] * nall / el / 1e9}
            if task.get("ops"):
                allc["GOPS"] = task["ops"] * nall / el / 1e9
            base["all_cores"] = allc
        if "all_cores" in base:
            base["all_cores"]["us_per_call_est"] = task["full_bytes"] / (base["all_cores"]["weight_GBps"] * 1e9) * 1e6
        gpu_gbps = row.get("weight_GBps")
        if gpu_gbps:
            base["gpu_speedup_vs_1_core"] = gpu_gbps / base["weight_GBps"]
            if "all_cores" in base:
                base["gpu_speedup_vs_all_cores"] = gpu_gbps / base["all_cores"]["weight_GBps"]
        row["cpu_baseline"] = base
        # the same figures flat on the row, beside the GPU's
        row["oracle_us"] = base["us_per_call_est"]
        row["oracle_GBps"] = base["weight_GBps"]
        row["oracle_cores"] = 1
        if "all_cores" in base:
            row["oracle_all_cores_us"] = base["all_cores"]["us_per_call_est"]
            row["oracle_all_cores_GBps"] = base["all_cores"]["weight_GBps"]
            row["oracle_all_cores"] = base["all_cores"]["cores"]


def _sample_rows(N, n=64):
    return np.unique(np.linspace(0, N - 1, n).astype(np.int64))


def sweep(world, cpu=True):
    """Extra figures for the other workloads (not the headline): GEMV at
    K = N = 1024, sibling GEMVs (q | k | v) in one launch vs three, prefill
    GEMM TOPS vs M, affine GEMM, lm_head sweep, orthogonal lm_head. Each call
    rotates over enough weight copies to exceed L2 twice. Every row is timed
    by alternating best-of rounds (with its spread), once more as eager calls,
    and beside the oracle on a row-sampled slice of the same shape (one core
    and all host cores)."""
    import torch
    import bit_group_quantized_qmm_gb300 as q
    dev = torch.device("cuda", torch.cuda.current_device())
    out = {}
    pool_bytes = 320 << 20
    tasks = []   # (row dict, oracle task)

    def pack_pool(variant, N, K, group, name, had=None):
        lay = qmm_synth.Layer(name, variant, N, K, group,
                              (group if variant == W4A8 else 0) if had is None else had)
        qb, s, b = qmm_synth.layer_weights(0, name, lay)
        d = q.weight_desc(variant, N, K, group)
        size = q.qmm_packed_size(d)
        copies = max(2, math.ceil(pool_bytes / size))
        first = torch.empty(size, dtype=torch.uint8, device=dev)
        q.qmm_pack_weights(d, torch.from_numpy(qb).to(dev), torch.from_numpy(s.view(np.int16)).to(dev),
                           None if b is None else torch.from_numpy(b.view(np.int16)).to(dev), first)
        pool = [first] + [first.clone() for _ in range(copies - 1)]
        return lay, d, pool, size, (qb, s, b)

    def w4a8_task(hostw, x, group, had, N, K, M, label, mats=None):
        rows = _sample_rows(N)
        qb, sw, _ = hostw
        mats = mats or [(qb[rows], sw[rows])]
        nr = sum(m[0].shape[0] for m in mats)
        per_row = K // 2 + 2 * (K // group)
        return {"kind": "w4a8", "x": np.ascontiguousarray(x), "group": group, "had": had, "mats": mats,
                "bytes": nr * per_row, "ops": 2 * M * nr * K, "full_bytes": N * per_row,
                "sample": f"{label}: prepass of all {M} activation rows + {nr} of {N} output rows"}

    # K = N = 1024 GEMV
    lay, d, pool, size, hostw = pack_pool(W4A8, 1024, 1024, 64, "gemv_k1024_n1024", had=0)
    x = torch.from_numpy(qmm_synth.layer_activations(0, "gemv_k1024_n1024", lay, 1)).to(dev)
    a = torch.empty(1024, dtype=torch.int8, device=dev)
    sx = torch.empty(16, dtype=torch.float32, device=dev)
    y = torch.empty(1024, dtype=torch.float32, device=dev)
    ws = torch.zeros(max(16, q.qmm_gemv_workspace_size(d)), dtype=torch.uint8, device=dev)
    q.qmm_prep_act(W4A8, 1, 1024, 64, 0, x, 0, a=a, sx=sx)

    def gemv_pool():
        for p in pool:
            q.qmm_gemv(d, p, a, sx, y, ws, ws.numel())

    def fused_pool():   # quantization of x included
        for p in pool:
            q.qmm_gemv_fused(d, p, x[0], 0, 0, y)
    n = len(pool)
    t = ab_time({"gemv": gemv_pool, "fused": fused_pool}, {"gemv": n, "fused": n})
    row = dict(t["gemv"])
    row["weight_GBps"] = size / (row["us_per_call"] * 1e-6) / 1e9
    row["eager_us_per_call"] = eager_us(gemv_pool, n)
    row["fused"] = dict(t["fused"], weight_GBps=size / (t["fused"]["us_per_call"] * 1e-6) / 1e9,
                        eager_us_per_call=eager_us(fused_pool, n))
    out["gemv_k1024_n1024"] = row
    tasks.append((row, w4a8_task(hostw, x.cpu().numpy(), 64, 0, 1024, 1024, 1, "K = N = 1024")))
    del pool

    # sibling GEMVs sharing x (q | k | v of one layer, K = 1536): one launch vs three
    Ns, K = (2048, 512, 512), 1536
    sib = []
    for i, N in enumerate(Ns):
        lay_i, d_i, pool_i, size_i, host_i = pack_pool(W4A8, N, K, 64, f"siblings/{i}")
        sib.append((d_i, pool_i, size_i, host_i))
    ncopy = min(len(p[1]) for p in sib)
    xs_np = qmm_synth.layer_activations(0, "siblings/x", lay_i, 1)
    x = torch.from_numpy(xs_np).to(dev)[0].contiguous()
    ys = [torch.empty(N, dtype=torch.float32, device=dev) for N in Ns]
    descs = [p[0] for p in sib]
    set_bytes = sum(p[2] for p in sib)

    def separate():
        for c in range(ncopy):
            for (d_i, pool_i, _, _), y_i in zip(sib, ys):
                q.qmm_gemv_fused(d_i, pool_i[c], x, 0, 64, y_i)

    def together():
        for c in range(ncopy):
            q.qmm_gemv_fused_siblings(descs, [p[1][c] for p in sib], x, 0, 64, ys)
    t = ab_time({"separate": separate, "together": together}, {"separate": ncopy, "together": ncopy})
    row = {"one_launch_us": t["together"]["us_per_call"], "separate_us": t["separate"]["us_per_call"],
           "one_launch_spread": t["together"]["spread"], "separate_spread": t["separate"]["spread"],
           "rounds": t["together"]["rounds"],
           "weight_GBps": set_bytes / (t["together"]["us_per_call"] * 1e-6) / 1e9,
           "eager_one_launch_us": eager_us(together, ncopy), "eager_separate_us": eager_us(separate, ncopy)}
    out["siblings_qkv"] = row
    mats = []
    for (_, _, _, (qb_i, sw_i, _)), N in zip(sib, Ns):
        r_i = _sample_rows(N, 22)
        mats.append((qb_i[r_i], sw_i[r_i]))
    per_row = K // 2 + 2 * (K // 64)
    nr = sum(m[0].shape[0] for m in mats)
    tasks.append((row, {"kind": "w4a8", "x": np.ascontiguousarray(xs_np), "group": 64, "had": 64, "mats": mats,
                        "bytes": nr * per_row, "ops": 2 * nr * K, "full_bytes": sum(Ns) * per_row,
                        "sample": f"q|k|v: one prepass + {nr} of {sum(Ns)} output rows"}))
    del sib

    # prefill GEMM K=1536 N=12288 vs M
    lay, d, pool, size, hostw = pack_pool(W4A8, 12288, 1536, 64, "prefill_gemm")
    res = {}
    for M in (16, 64, 128, 512, 1068):
        x_np = qmm_synth.layer_activations(0, f"prefill_gemm/x{M}", lay, M)
        x = torch.from_numpy(x_np).to(dev)
        a16 = torch.empty((M, 1536), dtype=torch.float16, device=dev)
        sxm = torch.empty((M, 24), dtype=torch.float32, device=dev)
        Y = torch.empty((M, 12288), dtype=torch.float32, device=dev)
        q.qmm_prep_act(W4A8, M, 1536, 64, 64, x, 0, a16=a16, sx=sxm)
        use = pool[:max(2, min(len(pool), 8))]

        def gemm_pool():
            for p in use:
                q.qmm_gemm(d, p, M, a16, sxm, Y)
        row = dict(ab_time({"g": gemm_pool}, {"g": len(use)})["g"])
        tsec = row["us_per_call"] * 1e-6
        row.update({"TOPS": 2 * M * 12288 * 1536 / tsec / 1e12, "weight_GBps": size / tsec / 1e9,
                    "eager_us_per_call": eager_us(gemm_pool, len(use)), "kernel": q.qmm_last_kernel_id()})
        res[str(M)] = row
        tasks.append((row, w4a8_task(hostw, x_np, 64, 64, 12288, 1536, M, f"prefill M = {M}")))
    out["prefill_gemm"] = res
    del pool

    # affine GEMM K=5120 N=34816
    lay, d, pool, size, (qb_a, s_a, b_a) = pack_pool(AFFINE, 34816, 5120, 64, "affine_gemm")
    res = {}
    for M in (64, 65, 128):
        x16_np = qmm_synth.layer_activations(0, f"affine_gemm/x{M}", lay, M)
        x16 = torch.from_numpy(x16_np.view(np.float16)).to(dev)
        S = torch.empty((M, 80), dtype=torch.float32, device=dev)
        Y = torch.empty((M, 34816), dtype=torch.float32, device=dev)
        q.qmm_prep_act(AFFINE, M, 5120, 64, 0, x16, 1, gsum=S)

        def aff_pool():
            for p in pool:
                q.qmm_gemm(d, p, M, x16, S, Y)
        row = dict(ab_time({"g": aff_pool}, {"g": len(pool)}, iters=4)["g"])
        tsec = row["us_per_call"] * 1e-6
        row.update({"TFLOPS": 2 * M * 34816 * 5120 / tsec / 1e12, "weight_GBps": size / tsec / 1e9,
                    "eager_us_per_call": eager_us(aff_pool, len(pool)), "kernel": q.qmm_last_kernel_id()})
        # the element-wise error beside the norm-wise tolerance, on sampled columns
        rows = _sample_rows(34816, 48)
        import oracle
        Yr, Ym = oracle.default().gemm_affine(qb_a, s_a, b_a, x16_np, rows=rows.astype(np.int32))
        Yg = Y[:, torch.from_numpy(rows).to(dev)].double().cpu().numpy()
        err = np.abs(Yg - Yr)
        floor = 1e-3 * float(np.abs(Yr).max())
        big = np.abs(Yr) > floor
        row["max_rel_err_elementwise"] = float((err[big] / np.abs(Yr[big])).max())
        row["rel_err_floor"] = floor
        row["max_err_over_normwise_bound"] = float((err / (2e-3 * Ym)).max())
        res[str(M)] = row
        nr = rows.size
        per_row = 5120 // 2 + 4 * 80
        tasks.append((row, {"kind": "affine", "qb": qb_a[rows], "s": s_a[rows], "b": b_a[rows],
                            "x16": np.ascontiguousarray(x16_np), "bytes": nr * per_row, "ops": 2 * M * nr * 5120,
                            "full_bytes": 34816 * per_row,
                            "sample": f"affine M = {M}: group sums + {nr} of 34816 output rows"}))
    out["affine_gemm"] = res
    del pool

    # lm_head sweep K=1536 N=262144 group 128
    lay, d, pool, size, hostw = pack_pool(W4A8, 262144, 1536, 128, "lm_head")
    res = {}
    for M in (1, 2, 4, 8, 16, 32):
        x_np = qmm_synth.layer_activations(0, f"lm_head/x{M}", lay, M)
        x = torch.from_numpy(x_np).to(dev)
        a = torch.empty((M, 1536), dtype=torch.int8, device=dev)
        a16 = torch.empty((M, 1536), dtype=torch.float16, device=dev)
        sxm = torch.empty((M, 12), dtype=torch.float32, device=dev)
        Y = torch.empty((M, 262144), dtype=torch.float32, device=dev)
        q.qmm_prep_act(W4A8, M, 1536, 128, 128, x, 0, a=a, a16=a16, sx=sxm)
        entry = {}

        def gemm_pool():
            for p in pool:
                q.qmm_gemm(d, p, M, a16, sxm, Y)
        fns, calls = {"gemm": gemm_pool}, {"gemm": len(pool)}
        if M == 1:
            ws1 = torch.zeros(max(16, q.qmm_gemv_workspace_size(d)), dtype=torch.uint8, device=dev)

            def gemv_pool2():
                for p in pool:
                    q.qmm_gemv(d, p, a, sxm, Y, ws1, ws1.numel())
            fns["gemv"], calls["gemv"] = gemv_pool2, len(pool)
        t = ab_time(fns, calls, iters=4)
        for k in fns:
            r_ = dict(t[k])
            r_["weight_GBps"] = size / (r_["us_per_call"] * 1e-6) / 1e9
            r_["eager_us_per_call"] = eager_us(fns[k], calls[k])
            if k == "gemm":
                fns[k]()
                r_["kernel"] = q.qmm_last_kernel_id()
                r_["TOPS"] = 2 * M * 262144 * 1536 / (r_["us_per_call"] * 1e-6) / 1e12
            entry[k] = r_
        res[str(M)] = entry
        tasks.append((entry["gemv" if M == 1 else "gemm"],
                      w4a8_task(hostw, x_np, 128, 128, 262144, 1536, M, f"lm_head M = {M}")))
    out["lm_head"] = res
    del pool

    # orthogonal lm_head: full-K rotation prepass + CQ4 GEMV/GEMM on weights
    # stored rotated, one norm per row viewed as 128-wide groups
    N, K = 262144, 1536
    lay = qmm_synth.Layer("lm_head_orth", CQ4, N, K, 128, 0)
    idx, _, _ = qmm_synth.layer_weights(0, "lm_head_orth", lay)
    C, cb = qmm_synth.layer_codebook(0, "lm_head_orth")
    norms = qmm_synth.uniform_f16(0, "lm_head_orth/norms", (N, 1), 0.005, 0.02)
    sw = np.ascontiguousarray(np.repeat(norms, K // 128, axis=1))
    d = q.weight_desc(CQ4, N, K, 128)
    size = q.qmm_packed_size(d)
    first = torch.empty(size, dtype=torch.uint8, device=dev)
    q.qmm_pack_weights_cq4(d, torch.from_numpy(idx).to(dev), C, cb, torch.from_numpy(sw.view(np.int16)).to(dev),
                           first)
    pool = [first] + [first.clone() for _ in range(max(1, math.ceil(pool_bytes / size)) - 1)]
    R_np = qmm_synth.orthogonal_f32(0, "lm_head_orth/R", K)
    R = torch.from_numpy(R_np).to(dev)
    res = {}
    for M in (1, 8):
        x_np = qmm_synth.layer_activations(0, f"lm_head_orth/x{M}", lay, M)
        x = torch.from_numpy(x_np).to(dev)
        a = torch.empty((M, K), dtype=torch.int8, device=dev)
        a16 = torch.empty((M, K), dtype=torch.float16, device=dev)
        sxm = torch.empty((M, K // 128), dtype=torch.float32, device=dev)
        Y = torch.empty((M, N), dtype=torch.float32, device=dev)
        ws1 = torch.zeros(max(16, q.qmm_gemv_workspace_size(d)), dtype=torch.uint8, device=dev)

        def prep_only():
            for _ in pool:
                q.qmm_prep_act_rotated(M, K, 128, R, x, 0, a=a, a16=a16, sx=sxm)

        def prep_and_matmul():
            for p in pool:
                q.qmm_prep_act_rotated(M, K, 128, R, x, 0, a=a, a16=a16, sx=sxm)
                if M == 1:
                    q.qmm_gemv(d, p, a, sxm, Y, ws1, ws1.numel())
                else:
                    q.qmm_gemm(d, p, M, a16, sxm, Y)
        t = ab_time({"prep": prep_only, "call": prep_and_matmul}, {"prep": len(pool), "call": len(pool)}, iters=4)
        row = dict(t["call"])
        row.update({"prep_rotated_us": t["prep"]["us_per_call"], "prep_rotated_spread": t["prep"]["spread"],
                    "weight_GBps": size / (row["us_per_call"] * 1e-6) / 1e9,
                    "rotation_GBps": K * K * 4 / (t["prep"]["us_per_call"] * 1e-6) / 1e9,
                    "eager_us_per_call": eager_us(prep_and_matmul, len(pool))})
        res[str(M)] = row
        rows = _sample_rows(N)
        per_row = K // 2 + 2 * (K // 128)
        tasks.append((row, {"kind": "rotated_cq4", "R": R_np, "x": np.ascontiguousarray(x_np), "idx": idx[rows],
                            "C": C, "cb": cb, "sw": sw[rows], "bytes": rows.size * per_row,
                            "ops": 2 * M * rows.size * K, "full_bytes": N * per_row,
                            "sample": f"orthogonal lm_head M = {M}: full-K rotation of x + {rows.size} of {N} "
                                      f"output rows"}))
    out["lm_head_orth"] = res
    del pool
    torch.cuda.empty_cache()
    if cpu:
        import multiprocessing as mp
        with mp.get_context("spawn").Pool(os.cpu_count() or 1) as cpu_pool:
            oracle_baselines(tasks, cpu_pool)
    _add_fractions(out)
    return out


def _add_fractions(node):
    """Beside every figure of the sweep, its fraction of the peaks: weight
    bytes per second over the measured copy bandwidth; TOPS / TFLOPS over the
    measured dense bf16 rate (the rate of the kind::f16 MMAs the GEMM issues)
    and over the mma.sync s8 peak (the int8 warp MMA, measured on this GPU)."""
    hbm, tflops, _ = measured_peaks()
    s8 = s8_peak_tops()
    if isinstance(node, dict):
        for k in list(node):
            v = node[k]
            if k.endswith("weight_GBps") and isinstance(v, (int, float)):
                node[k.replace("weight_GBps", "frac_copy_bw")] = v / hbm
            elif k in ("TOPS", "TFLOPS"):
                node["frac_bf16_peak"] = v / tflops
                node["frac_s8_peak"] = v / s8
            elif k != "cpu_baseline":
                _add_fractions(v)


# ------------------------------------------------------------------ per-projection figures of the headline

def projection_rows(model):
    """Per projection of the decode step: one fused launch per layer of that
    projection alone, over enough weight copies to exceed L2 twice, the four
    projections timed by alternating best-of rounds. Algorithmic bytes per
    launch: packed nibbles and scales, fp32 x in, fp32 y out."""
    q = model.q
    fns, calls, nbytes, keep = {}, {}, {}, []
    for name, N, K in PROJ:
        ps = [p for p in model.projs if p["name"] == name]
        blobs = [p["packed"] for p in ps]
        size = q.qmm_packed_size(ps[0]["d"])
        while len(blobs) * size < (256 << 20):
            blobs = blobs + [b.clone() for b in blobs[:len(ps)]]
        keep.append(blobs)
        d = ps[0]["d"]
        x = model.x[ps[0]["x_off"]:ps[0]["x_off"] + K]
        y = model.y[ps[0]["y_off"]:ps[0]["y_off"] + N]

        def f(blobs=blobs, d=d, x=x, y=y):
            for b in blobs:
                q.qmm_gemv_fused(d, b, x, 0, GROUP, y)
        fns[name], calls[name], nbytes[name] = f, len(blobs), size
    t = ab_time(fns, calls, rounds=6, iters=20)
    hbm, _, _ = measured_peaks()
    out = {}
    for name, N, K in PROJ:
        r = t[name]
        alg = nbytes[name] + 4 * K + 4 * N
        gbps = alg / (r["us_per_call"] * 1e-6) / 1e9
        out[name] = {"N": N, "K": K, "us_per_launch": r["us_per_call"], "us_median": r["us_median"],
                     "spread": r["spread"], "rounds": r["rounds"], "algorithmic_bytes": alg, "GBps": gbps,
                     "frac_copy_bw": gbps / hbm, "copies": calls[name]}
    return out


# ------------------------------------------------------------------ peaks of the non-tensor-memory units

PEAKS_CU = r'''
// FP32 FMA (scalar and packed pairs) and legacy warp-MMA (mma.sync) rates:
// one CTA per SM, clock64 per CTA, the slowest CTA counts; the warp-MMA rates
// are the best over 4, 8 and 16 warps per SM.
#include <cstdio>
#include <cstdint>
#include <cuda_runtime.h>
__global__ void __launch_bounds__(1024, 1) fp32(int iters, int packed, long long* cyc, float* sink)
{
    float a[16];
    for (int i = 0; i < 16; ++i) a[i] = threadIdx.x * 1e-7f + i;
    const float b = 0.999f, c = 1e-6f;
    __syncthreads();
    const long long t0 = clock64();
    if (!packed) {
        for (int it = 0; it < iters; ++it)
#pragma unroll
            for (int i = 0; i < 16; ++i) asm volatile("fma.rn.f32 %0, %0, %1, %2;" : "+f"(a[i]) : "f"(b), "f"(c));
    } else {
        unsigned long long p[8], bb, cc;
        for (int i = 0; i < 8; ++i) asm("mov.b64 %0, {%1, %2};" : "=l"(p[i]) : "f"(a[2 * i]), "f"(a[2 * i + 1]));
        asm("mov.b64 %0, {%1, %1};" : "=l"(bb) : "f"(b));
        asm("mov.b64 %0, {%1, %1};" : "=l"(cc) : "f"(c));
        for (int it = 0; it < iters; ++it)
#pragma unroll
            for (int i = 0; i < 8; ++i) asm volatile("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(p[i]) : "l"(bb), "l"(cc));
        for (int i = 0; i < 8; ++i) asm("mov.b64 {%0, %1}, %2;" : "=f"(a[2 * i]), "=f"(a[2 * i + 1]) : "l"(p[i]));
    }
    __syncthreads();
    const long long t1 = clock64();
    float s = 0.f;
    for (int i = 0; i < 16; ++i) s += a[i];
    if (s == 12345.f) sink[threadIdx.x] = s;
    if (threadIdx.x == 0) cyc[blockIdx.x] = t1 - t0;
}
__global__ void __launch_bounds__(512, 1) mmas(int iters, int mode, long long* cyc, int* sink)
{
    uint32_t a0 = threadIdx.x, a1 = a0 * 3, a2 = a0 * 5, a3 = a0 * 7, b0 = a0 * 11, b1 = a0 * 13;
    uint32_t d[8][4];
    for (int i = 0; i < 8; ++i)
        for (int j = 0; j < 4; ++j) d[i][j] = 0;
    if (mode == 1) { a0 &= 0x3C003C00u; a1 &= 0x3C003C00u; a2 &= 0x3C003C00u; a3 &= 0x3C003C00u; b0 &= 0x3C003C00u; b1 &= 0x3C003C00u; }
    __syncthreads();
    const long long t0 = clock64();
    for (int it = 0; it < iters; ++it)
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (mode == 0)
                asm volatile("mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                             : "+r"(d[i][0]), "+r"(d[i][1]), "+r"(d[i][2]), "+r"(d[i][3])
                             : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
            else
                asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                             : "+r"(d[i][0]), "+r"(d[i][1]), "+r"(d[i][2]), "+r"(d[i][3])
                             : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
        }
    __syncthreads();
    const long long t1 = clock64();
    int s = 0;
    for (int i = 0; i < 8; ++i)
        for (int j = 0; j < 4; ++j) s += (int)d[i][j];
    if (s == 12345) sink[threadIdx.x] = s;
    if (threadIdx.x == 0) cyc[blockIdx.x] = t1 - t0;
}
static long long slowest(long long* dcyc, int n)
{
    long long h[1024], mx = 0;
    cudaMemcpy(h, dcyc, 8 * n, cudaMemcpyDeviceToHost);
    for (int i = 0; i < n; ++i) mx = h[i] > mx ? h[i] : mx;
    return mx;
}
int main()
{
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
    long long* cyc; float* fs; int* is;
    cudaMalloc(&cyc, 8 * 1024); cudaMalloc(&fs, 4 * 1024); cudaMalloc(&is, 4 * 1024);
    double best[4] = {0, 0, 0, 0};
    for (int rep = 0; rep < 3; ++rep) {
        for (int packed = 0; packed < 2; ++packed) {
            fp32<<<sms, 1024>>>(4096, packed, cyc, fs);
            if (cudaDeviceSynchronize() != cudaSuccess) return 1;
            const double r = 1024.0 * 4096 * 16 / slowest(cyc, sms);
            if (r > best[packed]) best[packed] = r;
        }
        for (int mode = 0; mode < 2; ++mode)
            for (int threads = 128; threads <= 512; threads *= 2) {
                mmas<<<sms, threads>>>(1024, mode, cyc, is);
                if (cudaDeviceSynchronize() != cudaSuccess) return 1;
                const double r = (threads / 32) * 1024.0 * 8 * (mode == 0 ? 16 * 8 * 32 : 16 * 8 * 16) / slowest(cyc, sms);
                if (r > best[2 + mode]) best[2 + mode] = r;
            }
    }
    printf("{\"sms\": %d, \"fma_f32_lane_ops_per_clk_sm\": %.1f, \"fma_f32x2_lane_ops_per_clk_sm\": %.1f, "
           "\"mma_sync_s8_mac_per_clk_sm\": %.1f, \"mma_sync_f16_mac_per_clk_sm\": %.1f}\n",
           sms, best[0], best[1], best[2], best[3]);
    return 0;
}
'''


def run_peaks():
    """Compile and run the FP32 / mma.sync microbenchmark; print its JSON line
    with the s8 peak in TOPS at the measured maximum SM clock."""
    import shutil
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    with tempfile.TemporaryDirectory() as tmp:
        src = os.path.join(tmp, "peaks.cu")
        exe = os.path.join(tmp, "peaks")
        with open(src, "w") as f:
            f.write(PEAKS_CU)
        subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-o", exe, src], check=True)
        res = subprocess.run([exe], capture_output=True, text=True, check=True)
    d = json.loads(res.stdout.strip().splitlines()[-1])
    d["mma_sync_s8_tops_at_max_clock"] = 2.0 * d["mma_sync_s8_mac_per_clk_sm"] * d["sms"] * 2070e6 / 1e12
    d["tcgen05_kind_f16_mac_per_clk_sm_nominal"] = 4096
    print(json.dumps(d), flush=True)


def profile_case(spec):
    """A few launches of one prefill GEMM shape (K = 1536, N = 12288, group 64,
    Hadamard-64): prepass, then 2 + 3 GEMM calls on one packed weight. Small
    enough to capture under a profiler; the timing printed is informational."""
    import torch
    import bit_group_quantized_qmm_gb300 as q
    name, _, m = spec.partition(":")
    if name not in ("prefill_gemm", "prep_rotated", "lm_head_gemv", "lm_head_gemv_cq4", "lm_head_gemm",
                    "lm_head_gemm_f16", "affine_gemm") or not m.isdigit():
        raise SystemExit(f"unknown profile case {spec!r} (expected prefill_gemm:M, prep_rotated:M, "
                         "lm_head_gemv:1, lm_head_gemv_cq4:1, lm_head_gemm[_f16]:M or affine_gemm:M)")
    if name == "lm_head_gemm_f16":
        # the same GEMM with the weights-in-N kernel held to its fp16 form (M 9..32)
        q.qmm_set_gemm_narrow(q.NARROW_F16)
        name = "lm_head_gemm"
    if name == "affine_gemm":
        # the affine GEMM of the fused gate_up shape (K = 5120, N = 34816, group 64, fp16 x)
        M, N, K = int(m), 34816, 5120
        dev = torch.device("cuda", torch.cuda.current_device())
        lay = qmm_synth.Layer("affine_gemm", AFFINE, N, K, 64, 0)
        qb, s, b = qmm_synth.layer_weights(0, "affine_gemm", lay)
        d = q.weight_desc(AFFINE, N, K, 64)
        packed = torch.empty(q.qmm_packed_size(d), dtype=torch.uint8, device=dev)
        q.qmm_pack_weights(d, torch.from_numpy(qb).to(dev), torch.from_numpy(s.view(np.int16)).to(dev),
                           torch.from_numpy(b.view(np.int16)).to(dev), packed)
        x16 = torch.from_numpy(qmm_synth.layer_activations(0, f"affine_gemm/x{M}", lay, M).view(np.float16)).to(dev)
        S = torch.empty((M, K // 64), dtype=torch.float32, device=dev)
        Y = torch.empty((M, N), dtype=torch.float32, device=dev)
        q.qmm_prep_act(AFFINE, M, K, 64, 0, x16, 1, gsum=S)
        for _ in range(2):
            q.qmm_gemm(d, packed, M, x16, S, Y)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(3):
            q.qmm_gemm(d, packed, M, x16, S, Y)
        e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / 3
        print(json.dumps({"profile_case": spec, "us_per_call": us, "TFLOPS": 2 * M * N * K / us / 1e6,
                          "kernel": q.qmm_last_kernel_id(), "device_status": q.qmm_device_status()}))
        return
    if name == "lm_head_gemm":
        # the GEMM at lm_head size (K = 1536, N = 262144, group 128); M <= 8 runs
        # the dp4a kernel's streaming form
        M, N, K, g = int(m), 262144, 1536, 128
        dev = torch.device("cuda", torch.cuda.current_device())
        lay = qmm_synth.Layer("lm_head", W4A8, N, K, g, g)
        qb, sw, _ = qmm_synth.layer_weights(0, "lm_head", lay)
        d = q.weight_desc(W4A8, N, K, g)
        packed = torch.empty(q.qmm_packed_size(d), dtype=torch.uint8, device=dev)
        q.qmm_pack_weights(d, torch.from_numpy(qb).to(dev), torch.from_numpy(sw.view(np.int16)).to(dev), None, packed)
        x = torch.from_numpy(qmm_synth.layer_activations(0, f"lm_head/x{M}", lay, M)).to(dev)
        a16 = torch.empty((M, K), dtype=torch.float16, device=dev)
        sx = torch.empty((M, K // g), dtype=torch.float32, device=dev)
        Y = torch.empty((M, N), dtype=torch.float32, device=dev)
        q.qmm_prep_act(W4A8, M, K, g, g, x, 0, a16=a16, sx=sx)
        for _ in range(2):
            q.qmm_gemm(d, packed, M, a16, sx, Y)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(3):
            q.qmm_gemm(d, packed, M, a16, sx, Y)
        e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / 3
        print(json.dumps({"profile_case": spec, "us_per_call": us, "weight_GBps": packed.numel() / us / 1e3,
                          "kernel": q.qmm_last_kernel_id(), "device_status": q.qmm_device_status()}))
        return
    if name in ("lm_head_gemv", "lm_head_gemv_cq4"):
        # the plain GEMV on prepared codes at lm_head size (K = 1536, N = 262144,
        # group 128), symmetric or codebook weights
        N, K, g = 262144, 1536, 128
        variant = CQ4 if name.endswith("cq4") else W4A8
        dev = torch.device("cuda", torch.cuda.current_device())
        lay = qmm_synth.Layer("lm_head", variant, N, K, g, g)
        qb, sw, _ = qmm_synth.layer_weights(0, "lm_head", lay)
        d = q.weight_desc(variant, N, K, g)
        packed = torch.empty(q.qmm_packed_size(d), dtype=torch.uint8, device=dev)
        if variant == CQ4:
            C, cb = qmm_synth.layer_codebook(0, "lm_head")
            q.qmm_pack_weights_cq4(d, torch.from_numpy(qb).to(dev), C, cb,
                                   torch.from_numpy(sw.view(np.int16)).to(dev), packed)
        else:
            q.qmm_pack_weights(d, torch.from_numpy(qb).to(dev), torch.from_numpy(sw.view(np.int16)).to(dev), None,
                               packed)
        x = torch.from_numpy(qmm_synth.layer_activations(0, "lm_head/x1", lay, 1)).to(dev)
        a = torch.empty(K, dtype=torch.int8, device=dev)
        sx = torch.empty(K // g, dtype=torch.float32, device=dev)
        y = torch.empty(N, dtype=torch.float32, device=dev)
        ws = torch.zeros(max(16, q.qmm_gemv_workspace_size(d)), dtype=torch.uint8, device=dev)
        q.qmm_prep_act(W4A8, 1, K, g, g, x, 0, a=a, sx=sx)
        for _ in range(2):
            q.qmm_gemv(d, packed, a, sx, y, ws, ws.numel())
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(3):
            q.qmm_gemv(d, packed, a, sx, y, ws, ws.numel())
        e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / 3
        print(json.dumps({"profile_case": spec, "us_per_call": us, "weight_GBps": packed.numel() / us / 1e3,
                          "device_status": q.qmm_device_status()}))
        return
    if name == "prep_rotated":
        # full-K rotation prepass of the orthogonal lm_head (K = 1536, group 128)
        M, K = int(m), 1536
        dev = torch.device("cuda", torch.cuda.current_device())
        R = torch.from_numpy(qmm_synth.orthogonal_f32(0, "lm_head_orth/R", K)).to(dev)
        x = torch.from_numpy(qmm_synth.activations_f32(0, f"lm_head_orth/x{M}", M, K, 0.01)).to(dev)
        a = torch.empty((M, K), dtype=torch.int8, device=dev)
        sx = torch.empty((M, K // 128), dtype=torch.float32, device=dev)
        for _ in range(2):
            q.qmm_prep_act_rotated(M, K, 128, R, x, 0, a=a, sx=sx)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(3):
            q.qmm_prep_act_rotated(M, K, 128, R, x, 0, a=a, sx=sx)
        e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / 3
        print(json.dumps({"profile_case": spec, "us_per_call": us, "rotation_GBps": K * K * 4 / us / 1e3,
                          "device_status": q.qmm_device_status()}))
        return
    M, N, K, g = int(m), 12288, 1536, 64
    dev = torch.device("cuda", torch.cuda.current_device())
    lay = qmm_synth.Layer("prefill_gemm", W4A8, N, K, g, g)
    qb, s, _ = qmm_synth.layer_weights(0, "prefill_gemm", lay)
    d = q.weight_desc(W4A8, N, K, g)
    packed = torch.empty(q.qmm_packed_size(d), dtype=torch.uint8, device=dev)
    q.qmm_pack_weights(d, torch.from_numpy(qb).to(dev), torch.from_numpy(s.view(np.int16)).to(dev), None, packed)
    x = torch.from_numpy(qmm_synth.layer_activations(0, f"prefill_gemm/x{M}", lay, M)).to(dev)
    a16 = torch.empty((M, K), dtype=torch.float16, device=dev)
    sx = torch.empty((M, K // g), dtype=torch.float32, device=dev)
    Y = torch.empty((M, N), dtype=torch.float32, device=dev)
    q.qmm_prep_act(W4A8, M, K, g, g, x, 0, a16=a16, sx=sx)
    for _ in range(2):
        q.qmm_gemm(d, packed, M, a16, sx, Y)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(3):
        q.qmm_gemm(d, packed, M, a16, sx, Y)
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / 3
    print(json.dumps({"profile_case": spec, "us_per_call": us, "TOPS": 2 * M * N * K / us / 1e6,
                      "device_status": q.qmm_device_status()}))


# ------------------------------------------------------------------ main

def main():
    args = parse_args()
    rank, world, local = dist_env()
    if args.peaks:
        run_peaks()
        return
    if args.profile_case:
        import torch
        torch.cuda.set_device(local)
        profile_case(args.profile_case)
        return
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    import torch
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device for the library arm (use --impl reference for the oracle)")
    torch.cuda.set_device(local)
    dist_init(world, use_cuda=True)
    import bit_group_quantized_qmm_gb300 as q

    hbm_peak, bf16_peak, peak_kind = measured_peaks()
    model = DecodeModel(args.layers, rank, keep_host=(rank == 0 and world == 1))
    g_step = capture(model.enqueue_step)
    g_two = capture(model.enqueue_step_two_kernels)
    n_kernels_per_step = len(model.projs)

    sampler = ClockSampler(local)
    sampler.start()
    t_step = time_graph(g_step, args.steps, args.warmup, world)
    clock_rows = sampler.stop()
    t_step = max_over_ranks(t_step, world)

    # the step is nothing but the fused GEMV launches: average launch time
    gemv_launch_s = t_step / (args.steps * len(model.projs))
    # the same pass as two launches per projection (prepass, then GEMV)
    two_iters = max(10, min(args.steps, 2000))
    t_two = max_over_ranks(time_graph(g_two, two_iters, 3, world), world) / two_iters

    # end to end: every step copies its x in from pinned host memory and its y
    # out to pinned host memory; two device buffer sets let the copies of one
    # step overlap the launches of the neighbouring steps (h2d and d2h on
    # their own streams, ordered by events)
    xs = [model.x, model.x.clone()]
    ys = [model.y, torch.empty_like(model.y)]
    yh = [model.y_host, torch.empty_like(model.y_host).pin_memory()]
    g_e2e = [g_step, capture(lambda: model.enqueue_step(xs[1], ys[1]))]
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    main = torch.cuda.current_stream()
    ev = {k: [torch.cuda.Event(), torch.cuda.Event()] for k in ("in", "done", "out")}
    torch.cuda.synchronize()
    barrier(world)
    e2e_steps = max(10, min(args.steps, 2000))
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        b = i & 1
        if i >= 2:
            h2d.wait_event(ev["done"][b])          # the graph two steps back has read x[b]
        with torch.cuda.stream(h2d):
            xs[b].copy_(model.x_host, non_blocking=True)
            ev["in"][b].record(h2d)
        main.wait_event(ev["in"][b])
        if i >= 2:
            main.wait_event(ev["out"][b])          # y[b] of two steps back is out
        g_e2e[b].replay()
        ev["done"][b].record(main)
        d2h.wait_event(ev["done"][b])
        with torch.cuda.stream(d2h):
            yh[b].copy_(ys[b], non_blocking=True)
            ev["out"][b].record(d2h)
    torch.cuda.synchronize()
    t_e2e = time.perf_counter() - t0
    barrier(world)
    t_e2e = max_over_ranks(t_e2e, world)

    per_projection = projection_rows(model) if rank == 0 and not args.no_sweep else None

    total_weight = sum_over_ranks(model.weight_bytes * args.steps, world)
    value = total_weight / t_step / 1e9
    e2e_value = sum_over_ranks(model.weight_bytes * e2e_steps, world) / t_e2e / 1e9
    gemv_bytes = model.fused_algorithmic_bytes() / len(model.projs)
    achieved = gemv_bytes / gemv_launch_s / 1e9
    traffic = gemv_traffic_per_step(model)
    status = q.qmm_device_status()

    sweep_out = None
    if not args.no_sweep and rank == 0:
        sweep_out = sweep(1 if world == 1 else world, cpu=not args.no_cpu_baseline)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, nproj, el = cpu_oracle_rate(model.host[:8], args.cpu_seconds)
        cpu = {"value": rate, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"{nproj} projection passes (prepass + all output rows) of the first two layers, "
                         f"{el:.1f} s, single-threaded C"}
        if not args.no_cpu_all_cores:
            rate_all, procs, nall = cpu_oracle_rate_all_cores(model.host[:8], args.cpu_seconds / 2)
            cpu["all_cores"] = {"value": rate_all, "unit": "GB/s", "cores": procs,
                                "sample": f"{nall} projection passes in {procs} spawned processes, "
                                          f"{args.cpu_seconds / 2:.1f} s each"}

    if rank == 0:
        clocks = ClockSampler.summarize(clock_rows)
        line = {
            "metric": "GEMV weight GB/s (decode projections, M=1)",
            "value": value,
            "unit": "GB/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": 1e3 * t_step / args.steps,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "int8",
            "data": "synthetic",
            "config": {
                "workload": f"gemma_decode: {args.layers} layers x (gate_up 1536->12288, down 6144->1536, "
                            "q 1536->2048, o 2048->1536), M=1, W4A8 group 64, Hadamard-64, "
                            "x N(0,1) + 1% +-20 outliers, seed 0",
                "layers": args.layers,
                "weight_bytes_per_step": model.weight_bytes,
                "l2": "per-step weights larger than L2 (no flush)",
                "launch": "CUDA graph of the step (one qmm_gemv_fused per projection); programmatic dependent launch",
                "two_kernel_ms_per_step": 1e3 * t_two,
                "parallelism": f"replicas x{world}",
            },
            "roofline": {
                "kernel": "gemv_fused_kernel (W4A8 prepass + GEMV, M=1)",
                "bound": "hbm",
                "achieved": achieved,
                "peak": hbm_peak,
                "unit": "GB/s",
                "frac": achieved / hbm_peak,
                "peak_kind": f"{peak_kind} copy bandwidth",
                "traffic": None if traffic is None else traffic / len(model.projs),
                "algorithmic_bytes_per_launch": gemv_bytes,
                "avg_launch_us": gemv_launch_s * 1e6,
                "frac_of_8TBps": achieved / 8000.0,
            },
            "per_projection": per_projection,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": model.h2d_bytes,
                    "d2h_bytes_per_step": model.d2h_bytes, "steps": e2e_steps,
                    "copies": "pinned host x in and y out every step, on their own streams, two device "
                              "buffer sets: a step's copies overlap its neighbours' launches"},
            "gpu_launches": n_kernels_per_step * args.steps,
            "clocks": clocks,
            "device_status": status,
            "sweep": sweep_out,
        }
        print(json.dumps(line), flush=True)
    barrier(world)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
