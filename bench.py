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
                                                        affine_gemm:M)

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
    p.add_argument("--profile-case", default=None, metavar="prefill_gemm:M|prep_rotated:M|lm_head_gemv[_cq4]:1|lm_head_gemm:M|affine_gemm:M",
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

def sweep(world):
    """Extra figures for the other workloads (not the headline): GEMV at
    K = N = 1024, sibling GEMVs (q | k | v) in one launch vs three, prefill
    GEMM TOPS vs M, affine GEMM, lm_head sweep. Each call rotates over enough
    weight copies to exceed L2 twice."""
    import torch
    import bit_group_quantized_qmm_gb300 as q
    dev = torch.device("cuda", torch.cuda.current_device())
    out = {}
    pool_bytes = 320 << 20

    def pack_pool(variant, N, K, group, name):
        lay = qmm_synth.Layer(name, variant, N, K, group, group if variant == W4A8 else 0)
        qb, s, b = qmm_synth.layer_weights(0, name, lay)
        d = q.weight_desc(variant, N, K, group)
        size = q.qmm_packed_size(d)
        copies = max(2, math.ceil(pool_bytes / size))
        first = torch.empty(size, dtype=torch.uint8, device=dev)
        q.qmm_pack_weights(d, torch.from_numpy(qb).to(dev), torch.from_numpy(s.view(np.int16)).to(dev),
                           None if b is None else torch.from_numpy(b.view(np.int16)).to(dev), first)
        pool = [first] + [first.clone() for _ in range(copies - 1)]
        return lay, d, pool, size

    def timed(fn, iters=20, warm=3):
        g = capture(fn)
        return time_graph(g, iters, warm, 1) / iters

    # K = N = 1024 GEMV
    lay, d, pool, size = pack_pool(W4A8, 1024, 1024, 64, "gemv_k1024_n1024")
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
    t = timed(gemv_pool) / len(pool)
    tf = timed(fused_pool) / len(pool)
    out["gemv_k1024_n1024"] = {"us_per_call": t * 1e6, "weight_GBps": size / t / 1e9,
                               "fused_us_per_call": tf * 1e6, "fused_weight_GBps": size / tf / 1e9}
    del pool

    # sibling GEMVs sharing x (q | k | v of one layer, K = 1536): one launch vs three
    Ns, K = (2048, 512, 512), 1536
    sib = []
    for i, N in enumerate(Ns):
        lay_i, d_i, pool_i, size_i = pack_pool(W4A8, N, K, 64, f"siblings/{i}")
        sib.append((d_i, pool_i, size_i))
    ncopy = min(len(p[1]) for p in sib)
    x = torch.from_numpy(qmm_synth.layer_activations(0, "siblings/x", lay_i, 1)).to(dev)[0].contiguous()
    ys = [torch.empty(N, dtype=torch.float32, device=dev) for N in Ns]
    descs = [p[0] for p in sib]
    set_bytes = sum(p[2] for p in sib)

    def separate():
        for c in range(ncopy):
            for (d_i, pool_i, _), y_i in zip(sib, ys):
                q.qmm_gemv_fused(d_i, pool_i[c], x, 0, 64, y_i)

    def together():
        for c in range(ncopy):
            q.qmm_gemv_fused_siblings(descs, [p[1][c] for p in sib], x, 0, 64, ys)
    t_sep = timed(separate) / ncopy
    t_tog = timed(together) / ncopy
    out["siblings_qkv"] = {"separate_us": t_sep * 1e6, "one_launch_us": t_tog * 1e6,
                           "weight_GBps_one_launch": set_bytes / t_tog / 1e9}
    del sib

    # prefill GEMM K=1536 N=12288 vs M
    lay, d, pool, size = pack_pool(W4A8, 12288, 1536, 64, "prefill_gemm")
    res = {}
    for M in (16, 64, 128, 512, 1068):
        x = torch.from_numpy(qmm_synth.layer_activations(0, f"prefill_gemm/x{M}", lay, M)).to(dev)
        a16 = torch.empty((M, 1536), dtype=torch.float16, device=dev)
        sxm = torch.empty((M, 24), dtype=torch.float32, device=dev)
        Y = torch.empty((M, 12288), dtype=torch.float32, device=dev)
        q.qmm_prep_act(W4A8, M, 1536, 64, 64, x, 0, a16=a16, sx=sxm)
        use = pool[:max(2, min(len(pool), 8))]

        def gemm_pool():
            for p in use:
                q.qmm_gemm(d, p, M, a16, sxm, Y)
        t = timed(gemm_pool) / len(use)
        res[str(M)] = {"us_per_call": t * 1e6, "TOPS": 2 * M * 12288 * 1536 / t / 1e12,
                       "weight_GBps": size / t / 1e9}
    out["prefill_gemm"] = res
    del pool

    # affine GEMM K=5120 N=34816
    lay, d, pool, size = pack_pool(AFFINE, 34816, 5120, 64, "affine_gemm")
    res = {}
    for M in (64, 65, 128):
        x16 = torch.from_numpy(qmm_synth.layer_activations(0, f"affine_gemm/x{M}", lay, M).view(np.float16)).to(dev)
        S = torch.empty((M, 80), dtype=torch.float32, device=dev)
        Y = torch.empty((M, 34816), dtype=torch.float32, device=dev)
        q.qmm_prep_act(AFFINE, M, 5120, 64, 0, x16, 1, gsum=S)

        def aff_pool():
            for p in pool:
                q.qmm_gemm(d, p, M, x16, S, Y)
        t = timed(aff_pool) / len(pool)
        res[str(M)] = {"us_per_call": t * 1e6, "TFLOPS": 2 * M * 34816 * 5120 / t / 1e12,
                       "weight_GBps": size / t / 1e9}
    out["affine_gemm"] = res
    del pool

    # lm_head sweep K=1536 N=262144 group 128
    lay, d, pool, size = pack_pool(W4A8, 262144, 1536, 128, "lm_head")
    res = {}
    for M in (1, 2, 4, 8, 16, 32):
        x = torch.from_numpy(qmm_synth.layer_activations(0, f"lm_head/x{M}", lay, M)).to(dev)
        a = torch.empty((M, 1536), dtype=torch.int8, device=dev)
        a16 = torch.empty((M, 1536), dtype=torch.float16, device=dev)
        sxm = torch.empty((M, 12), dtype=torch.float32, device=dev)
        Y = torch.empty((M, 262144), dtype=torch.float32, device=dev)
        q.qmm_prep_act(W4A8, M, 1536, 128, 128, x, 0, a=a, a16=a16, sx=sxm)
        entry = {}

        def gemm_pool():
            for p in pool:
                q.qmm_gemm(d, p, M, a16, sxm, Y)
        t = timed(gemm_pool) / len(pool)
        entry["gemm"] = {"us_per_call": t * 1e6, "weight_GBps": size / t / 1e9}
        if M == 1:
            ws1 = torch.zeros(max(16, q.qmm_gemv_workspace_size(d)), dtype=torch.uint8, device=dev)

            def gemv_pool2():
                for p in pool:
                    q.qmm_gemv(d, p, a, sxm, Y, ws1, ws1.numel())
            t = timed(gemv_pool2) / len(pool)
            entry["gemv"] = {"us_per_call": t * 1e6, "weight_GBps": size / t / 1e9}
        res[str(M)] = entry
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
    R = torch.from_numpy(qmm_synth.orthogonal_f32(0, "lm_head_orth/R", K)).to(dev)
    res = {}
    for M in (1, 8):
        x = torch.from_numpy(qmm_synth.layer_activations(0, f"lm_head_orth/x{M}", lay, M)).to(dev)
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
        tp = timed(prep_only) / len(pool)
        t = timed(prep_and_matmul) / len(pool)
        res[str(M)] = {"prep_rotated_us": tp * 1e6, "us_per_call": t * 1e6, "weight_GBps": size / t / 1e9,
                       "rotation_GBps": K * K * 4 / tp / 1e9}
    out["lm_head_orth"] = res
    del pool
    torch.cuda.empty_cache()
    _add_fractions(out)
    return out


def _add_fractions(node):
    """Beside every figure of the sweep, its fraction of the measured peaks:
    weight bytes per second over the copy bandwidth, TOPS / TFLOPS over the
    dense bf16 rate (the rate of the kind::f16 MMAs the GEMM issues)."""
    hbm, tflops, _ = measured_peaks()
    if isinstance(node, dict):
        for k in list(node):
            v = node[k]
            if k.endswith("weight_GBps"):
                node[k.replace("weight_GBps", "frac_copy_bw")] = v / hbm
            elif k in ("TOPS", "TFLOPS"):
                node["frac_bf16_peak"] = v / tflops
            else:
                _add_fractions(v)


def profile_case(spec):
    """A few launches of one prefill GEMM shape (K = 1536, N = 12288, group 64,
    Hadamard-64): prepass, then 2 + 3 GEMM calls on one packed weight. Small
    enough to capture under a profiler; the timing printed is informational."""
    import torch
    import bit_group_quantized_qmm_gb300 as q
    name, _, m = spec.partition(":")
    if name not in ("prefill_gemm", "prep_rotated", "lm_head_gemv", "lm_head_gemv_cq4", "lm_head_gemm",
                    "affine_gemm") or not m.isdigit():
        raise SystemExit(f"unknown profile case {spec!r} (expected prefill_gemm:M, prep_rotated:M, "
                         "lm_head_gemv:1, lm_head_gemv_cq4:1, lm_head_gemm:M or affine_gemm:M)")
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

    total_weight = sum_over_ranks(model.weight_bytes * args.steps, world)
    value = total_weight / t_step / 1e9
    e2e_value = sum_over_ranks(model.weight_bytes * e2e_steps, world) / t_e2e / 1e9
    gemv_bytes = model.fused_algorithmic_bytes() / len(model.projs)
    achieved = gemv_bytes / gemv_launch_s / 1e9
    traffic = gemv_traffic_per_step(model)
    status = q.qmm_device_status()

    sweep_out = None
    if not args.no_sweep and rank == 0:
        sweep_out = sweep(1 if world == 1 else world)

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
