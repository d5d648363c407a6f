#!/usr/bin/env python
"""Throughput of the multi-LoRA batched linear layer on GB300.

One step = one pass of the whole layer over one batch (lora_linear_fused):
for this decode batch the tcgen05 base GEMM writes fp32 partials split over
d_in, then one kernel computes each token's (BGMV) adapter term (shrink,
cluster sum, expand), adds the summed partials and stores y once -- on the
decode workload: one 4096->4096 layer, rank 16, 256 resident adapters, 64
one-token requests with Zipf(1.1) adapter ids and 8 base-only rows.  Inputs
are seeded and synthetic; weights and activations are resident in HBM before
timing.

Reported on one JSON line (rank 0):
  value     tokens/s over K steps (CUDA-graph replays; 4 rotating buffer sets
            whose total is > 2x L2, so every step reads HBM)
  e2e       the same metric through the public call with host buffers: each
            step copies x and the ids from pinned memory, runs the layer and
            copies y back
  roofline  the dominant kernel (the split-K base GEMM): its mean launch
            duration over back-to-back launches timed with CUDA events,
            against the measured HBM copy peak
  sweep     tokens/s and achieved GB/s over distinct adapters per batch
            (4096->4096, rank 16, 1024-slot pool; T = 32 and 256)
  configs   the decode layer over a 4-bit base, the prefill workload, and
            the 8B-shaped stack (224 layers), padded and with ragged ranks
  cpu_baseline  the fp64 CPU oracle on the host cores (a bounded sample):
            the whole decode batch per pass, BLAS threads set explicitly,
            median of 3 runs with all cores and with one thread
  clocks    nvidia-smi SM clocks and throttle reasons sampled every 50 ms
            over the whole run (the timed regions included)

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                      (--gpus N > 1 without a launcher: re-runs itself under
                      torch.distributed.run with N ranks, one replica per GPU)
    python bench.py --profile CASE    a few untimed launches of one workload's
                                      kernels, for a profiler (no JSON line)
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "LoRA-layer tokens/s and achieved HBM GB/s vs roofline, swept over distinct adapters/batch"
UNIT = "tokens/s"
NSETS = 4
E2E_GROUP = 4     # steps per group of the pipelined end-to-end loop
GRAPH_STEPS = 500

DECODE_DESC = ("decode_bgmv: one 4096->4096 layer, rank 16, 256 resident adapters, 64 one-token "
               "requests, ids Zipf(1.1) over the pool, 8 rows base-only")


# ----------------------------------------------------------------- helpers
def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100000)
    p.add_argument("--warmup", type=int, default=5000)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-sweep", action="store_true")
    p.add_argument("--no-prefill", action="store_true")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--no-stack", action="store_true",
                   help="skip the 224-layer 8B-shaped stack (timed by default)")
    p.add_argument("--profile", choices=["decode", "prefill", "decode4bit", "ragged", "sweep256"],
                   help="run 3 untimed passes of one workload and exit (for ncu)")
    p.add_argument("--oracle-child", type=int, default=0, help=argparse.SUPPRESS)
    p.add_argument("--oracle-budget", type=float, default=12.0, help=argparse.SUPPRESS)
    a = p.parse_args(argv)
    if a.warmup < 3:
        p.error("--warmup must be >= 3")
    if a.steps < 1:
        p.error("--steps must be >= 1")
    return a


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def dist_setup(backend):
    import torch.distributed as dist
    rank, world, _ = dist_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return rank, world


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def reduce_max(x: float, device=None) -> float:
    """Max of a host float over all ranks (the slowest rank sets the time)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        return {"hbm_gbs": float(m["hbm_gbs"]), "bf16_tflops": float(m["bf16_tflops"]),
                "bf16_tflops_sustained": float(m.get("bf16_tflops_sustained", m["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


def kernel_src_sha():
    h = hashlib.sha256()
    for f in ("k_decode_tc.cu", "ptx.cuh", "common.cuh"):
        with open(os.path.join(ROOT, "lora_serving_device_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def dram_traffic_per_launch():
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, or None when the kernel source changed since it was taken."""
    p = os.path.join(ROOT, "profiles", "decode_gemm_traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    if d.get("src_sha") != kernel_src_sha():
        return None
    return d.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every `period_ms`."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: str, period_ms: int = 50):
        self.proc = None
        self.lines = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(period_ms), "-i", gpu_index], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self, window=None):
        return parse_clocks(self.lines, window)


def _smi_time(stamp):
    """Seconds since the epoch of an nvidia-smi timestamp (local time)."""
    import datetime
    for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
        try:
            return datetime.datetime.strptime(stamp.strip(), fmt).timestamp()
        except ValueError:
            pass
    return None


def parse_clocks(lines, window=None):
    """Median busy SM clock, max clock and throttle reasons of nvidia-smi
    lines; `window` = (t0, t1) wall seconds keeps only samples inside it."""
    sm, mx, reasons = [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for ln in lines:
        parts = [p.strip() for p in ln.split(",")]
        if len(parts) < 10:
            continue
        if window is not None:
            ts = _smi_time(parts[0])
            if ts is None or not (window[0] <= ts <= window[1]):
                continue
        try:
            s, m = float(parts[2]), float(parts[3])
        except ValueError:
            continue
        sm.append(s)
        mx.append(m)
        for n, v in zip(names, parts[6:10]):
            if v.lower() in ("active", "1", "yes"):
                reasons.add(n)
    if not sm:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
    busy = [s for s in sm if s >= 0.5 * max(sm)] or sm
    return {"sm_mhz": statistics.median(busy), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
            "samples": len(sm)}


# d_in splits for the standalone SGMV rows on the prefill workload: the shrink,
# with its three-CTA ring, is fastest at 4 (29.0 us; 38.0 at 2, 30.5 at 3, 30.7
# at 5, 30.0 at 6, 32.0 at 8); the expand, which sums the partials in its V
# build at the start of every CTA, on one (131.4 us; 136.9 on two)
SGMV_SHRINK_KSPLIT = 4
SGMV_EXPAND_KSPLIT = 1


def fused_ksplit(T, d_in, d_out, n_slots, r, num_sms=152):
    """The shrink split the fused path uses (mirrors the library's choice;
    tests/test_bench_host.py checks it against lora_workspace_bytes)."""
    if T <= 256:      # decode-sized batch: per-token shrink, ~256 CTAs
        return max(1, min(-(-256 // max(T, 1)), 16, max(d_in // 512, 1)))
    cap = min(T, n_slots)
    if r in (64, 128):  # tensor-core shrink, splits folded into one partial
        est = -(-T // 128) + (cap + 1) // 2
        return max(1, min(-(-3 * num_sms // max(est, 1)), 4, max(d_in // 128, 1)))
    if n_slots <= 32767 and -(-d_out // 256) * -(-T // 256) >= 2 * num_sms:
        return 1      # 256 x 256 prefill tiles: v as one partial
    est = (T + 63) // 64 + (cap + 1) // 2
    ks = -(-2 * num_sms // max(est, 1))
    return max(1, min(ks, 16, max(d_in // 128, 1)))


def layer_bytes(T, d_in, d_out, r, D, elem=2):
    """Algorithmic HBM bytes of one fused layer: W0 once, each distinct
    adapter's A and B once, x read, y written, the ids."""
    return (d_in * d_out + D * r * (d_in + d_out) + T * d_in + T * d_out) * elem + T * 4


def gemm_bytes(T, d_in, d_out, elem=2):
    """Algorithmic HBM bytes of the decode base GEMM: W0 and x read once.
    Its fp32 partial tiles are written to L2 and read back from there by
    the next kernel (ncu counts no DRAM writes for them), so they are not
    counted."""
    return (d_in * d_out + T * d_in) * elem


# ------------------------------------------------------------ reference arm
REF_BUDGET_S = 150.0


def set_blas_threads(n):
    """Pin the BLAS / OpenMP thread count (read when numpy loads its BLAS, so
    this must run before the first numpy import of the process)."""
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS",
              "BLIS_NUM_THREADS"):
        os.environ[k] = str(n)


def cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith("model name"):
                    return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine() or "unknown"


def run_reference(args):
    """The CPU fp64 oracle as it stands, timed on the host cores with the BLAS
    thread count set to every core of the affinity mask.  One step is a pass
    of the oracle's per-request loop over a window of the decode batch: the
    whole 64-token batch when K + W passes fit in ~150 s (the usual case),
    else the largest window that does (at least one token).  Only rank 0
    runs; the other ranks exit at once."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    cores = len(os.sched_getaffinity(0))
    set_blas_threads(cores)
    from lora_serving_device_gb300 import workloads as W
    from oracle import lora_ref as O
    w = W.decode_bgmv()

    def window(t0, n):
        idx = [(t0 + i) % w.T for i in range(n)]
        O.lora_linear(w.x[idx], w.W0, w.A_pool, w.B_pool, w.scale, w.slot_ids[idx])

    t0 = time.perf_counter()
    window(0, w.T)                       # calibration pass (untimed)
    est = time.perf_counter() - t0
    n = w.T if (args.steps + args.warmup) * est <= REF_BUDGET_S else \
        max(1, int(w.T * REF_BUDGET_S / ((args.steps + args.warmup) * est)))
    for j in range(args.warmup):
        window(j * n, n)
    t0 = time.perf_counter()
    for j in range(args.steps):
        window((args.warmup + j) * n, n)
    dt = time.perf_counter() - t0
    value = args.steps * n / dt
    sample = ("per step: the whole 64-token decode batch" if n == w.T else
              f"per step: {n} of the decode batch's 64 tokens (one-token requests), "
              f"all 4096 output columns") + \
        f", numpy fp64 per-request loop, BLAS threads = {cores}"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded)",
            "config": {"workload": DECODE_DESC, "T": w.T, "d_in": w.d_in, "d_out": w.d_out,
                       "r": w.r, "n_slots": w.n_slots, "distinct": w.distinct,
                       "parallelism": "host", "tokens_per_step": n},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample, "cpu_model": cpu_model(), "blas_threads": cores},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def oracle_child(threads, budget_s):
    """Child process of cpu_baseline: BLAS threads already set in its
    environment.  Times three runs of whole-batch oracle passes, each run
    about budget_s / 3 long, and prints one JSON line."""
    from lora_serving_device_gb300 import workloads as W
    from oracle import lora_ref as O
    w = W.decode_bgmv()

    def one():
        O.lora_linear(w.x, w.W0, w.A_pool, w.B_pool, w.scale, w.slot_ids)

    t0 = time.perf_counter()
    one()                                # untimed warm pass, sizes the runs
    est = time.perf_counter() - t0
    passes = max(1, int(budget_s / 3 / est))
    runs = []
    for _ in range(3):
        t0 = time.perf_counter()
        for _ in range(passes):
            one()
        runs.append(passes * w.T / (time.perf_counter() - t0))
    print(json.dumps({"threads": threads, "passes_per_run": passes, "runs": runs}), flush=True)
    return 0


def cpu_baseline(budget_s=12.0):
    """The oracle on the host cores: whole-batch passes of the decode workload,
    median of 3 runs with the BLAS thread count set to every core, and the
    same with one thread.  Each measurement runs in a fresh process, so the
    thread count is set before numpy loads its BLAS (and nothing is forked
    from this CUDA process)."""
    cores = len(os.sched_getaffinity(0))
    out = {}
    for label, n in (("all", cores), ("single", 1)):
        env = dict(os.environ)
        for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS",
                  "BLIS_NUM_THREADS"):
            env[k] = str(n)
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-child", str(n),
                            "--oracle-budget", str(budget_s)], env=env, capture_output=True,
                           text=True, timeout=600)
        if r.returncode != 0:
            raise RuntimeError(f"oracle timing failed: {r.stderr[-400:]}")
        out[label] = json.loads(r.stdout.strip().splitlines()[-1])
    med = statistics.median(out["all"]["runs"])
    return {"value": med, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"the whole 64-token decode batch per pass, numpy fp64 per-request loop; "
                      f"median of 3 runs of {out['all']['passes_per_run']} passes, BLAS threads "
                      f"= {cores}",
            "cpu_model": cpu_model(), "blas_threads": cores, "runs": out["all"]["runs"],
            "single_thread": {"value": statistics.median(out["single"]["runs"]), "unit": UNIT,
                              "blas_threads": 1, "runs": out["single"]["runs"],
                              "passes_per_run": out["single"]["passes_per_run"]}}


# --------------------------------------------------------------- our arm
def _up(a, dev):
    import numpy as np
    import torch
    from lora_serving_device_gb300 import workloads as W
    return torch.from_numpy(W.bf16_bits(a).view(np.int16)).view(torch.bfloat16).to(dev)


class LayerSet:
    """Device tensors of one layer instance (one of the rotating sets)."""

    def __init__(self, x, W0, A, B, ids, scale, y):
        self.x, self.W0, self.A, self.B, self.ids, self.scale, self.y = x, W0, A, B, ids, scale, y

    def clone(self):
        return LayerSet(self.x.clone(), self.W0.clone(), self.A.clone(), self.B.clone(),
                        self.ids.clone(), self.scale.clone(), self.y.clone())


def capture(fn, n_steps, stream):
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            for i in range(n_steps):
                fn(i)
    return g


def graph_mean_ms(fn, n_steps, stream):
    """Mean ms per call of fn(i): n_steps calls replayed back to back from one
    CUDA graph (after an eager warm-up and a warm replay), CUDA events on the
    launching stream around the replay."""
    import torch
    with torch.cuda.stream(stream):
        for i in range(3):
            fn(i)
    stream.synchronize()
    g = capture(fn, n_steps, stream)
    with torch.cuda.stream(stream):
        g.replay()
    stream.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    with torch.cuda.stream(stream):
        g.replay()
    e1.record(stream)
    stream.synchronize()
    return e0.elapsed_time(e1) / n_steps


def block_row(ms, nbytes, pk):
    """One standalone kernel against the HBM roofline of its algorithmic bytes;
    points whose roofline time is under 5 us are launch/ramp floored."""
    us = ms * 1e3
    roof_us = nbytes / (pk["hbm_gbs"] * 1e9) * 1e6
    gbs = nbytes / (us * 1e-6) / 1e9
    return {"us": us, "gbs": gbs, "frac": gbs / pk["hbm_gbs"], "algorithmic_bytes": nbytes,
            "roofline_us": roof_us, "latency_floored": roof_us < 5.0}


def graph_chunk(K, W):
    """Steps per CUDA graph when the timed graph cannot be uploaded ahead:
    the largest divisor of K that is at most W (and GRAPH_STEPS), so the K
    timed steps are whole replays of one graph and the W warm-up steps
    replay that same graph at least once (a graph's first launch pays for
    its upload; none is left inside the timed region)."""
    top = max(1, min(W, K, GRAPH_STEPS))
    return max(g for g in range(1, top + 1) if K % g == 0)


def graph_upload(g, stream):
    """Upload an instantiated CUDA graph to the device without running it
    (driver cuGraphUpload on torch's graph exec).  False where this torch
    does not expose the exec handle."""
    import ctypes
    try:
        exe = g.raw_cuda_graph_exec()
        drv = ctypes.CDLL("libcuda.so.1")
        drv.cuGraphUpload.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
        drv.cuGraphUpload.restype = ctypes.c_int
        return drv.cuGraphUpload(ctypes.c_void_p(int(exe)),
                                 ctypes.c_void_p(int(stream.cuda_stream))) == 0
    except (AttributeError, OSError, TypeError, RuntimeError):
        return False


SPACER_CYCLES = 400000  # ~0.2 ms of GPU spin ahead of the start event
_FLUSH = {}


def l2_flush():
    """Reduce a zeroed 256 MB buffer (about twice the L2) on the current
    stream: L2 is left holding clean lines of it only."""
    import torch
    dev = torch.cuda.current_device()
    if dev not in _FLUSH:
        _FLUSH[dev] = torch.zeros(64 << 20, dtype=torch.int32, device=dev)
    torch.amax(_FLUSH[dev])


def timed_graph_steps(fn, K, W, stream):
    """Run W warm-up steps then time exactly K steps of `fn(i)` from CUDA
    graphs; returns (elapsed ms of the K steps, (wall start, wall end)).

    K <= GRAPH_STEPS: the K steps are one graph, uploaded before the timed
    region (so one launch, one pipeline start); the W warm-up steps run
    from their own graph.  Where the upload is not available, or K is
    larger, the K steps are whole replays of a graph of graph_chunk(K, W)
    steps that the warm-up also replays.  After the barrier and the
    synchronize, a read of a buffer twice the L2 size (which leaves L2
    holding only clean lines of that buffer) and a short GPU spin are queued
    ahead of the start event: nothing the warm-up left in L2 is hit, the
    host's launch latency falls before the start event, and the events
    bracket only the K steps."""
    import torch
    with torch.cuda.stream(stream):
        for i in range(2):          # eager warm-up before capture
            fn(i)
    stream.synchronize()
    g_timed, reps, g_warm = None, 0, []
    if K <= GRAPH_STEPS:
        g = capture(fn, K, stream)
        if graph_upload(g, stream):
            g_timed, reps = g, 1
            gw = min(W, GRAPH_STEPS)
            g_warm = [(capture(fn, gw, stream), W // gw)]
            if W % gw:
                g_warm.append((capture(fn, W % gw, stream), 1))
    if g_timed is None:
        G = graph_chunk(K, W)
        g_timed, reps = capture(fn, G, stream), K // G
        g_warm = [(g_timed, W // G)]
        if W % G:
            g_warm.append((capture(fn, W % G, stream), 1))
    with torch.cuda.stream(stream):
        for g, n in g_warm:
            for _ in range(n):
                g.replay()
        # the flush buffer, the spin kernel and the events are set up here, so
        # nothing is allocated or loaded for the first time once the start
        # event is queued
        l2_flush()
        torch.cuda._sleep(SPACER_CYCLES)
        torch.cuda.Event(enable_timing=True).record(stream)
    stream.synchronize()
    barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    with torch.cuda.stream(stream):
        l2_flush()
        torch.cuda._sleep(SPACER_CYCLES)
        e0.record(stream)
        for _ in range(reps):
            g_timed.replay()
        e1.record(stream)
    stream.synchronize()
    torch.cuda.synchronize()
    wall1 = time.time()
    barrier()
    TIMING["graph_uploaded"] = reps == 1 and K <= GRAPH_STEPS and g_warm and g_warm[0][0] is not g_timed
    TIMING["replays"] = reps
    return e0.elapsed_time(e1), (wall0, wall1)


TIMING = {}


def per_kernel_times(sets, L, T, d_in, d_out, r, n_slots, n_steps, stream):
    """Mean launch duration of each kernel of the fused decode path, each
    launched on its own through its public call: n_steps back-to-back
    launches replayed from one CUDA graph, CUDA events on the launching
    stream around the replay, rotating buffer sets.  The kernels are the
    split-K base GEMM (the dominant one) and the kernel that computes the
    BGMV adapter term, adds the GEMM's partials and stores y.  Launched on
    their own they do not overlap, so each mean includes the start-up and
    tail that the fused chain hides."""
    import torch
    dev = sets[0].x.device
    S = L.lora_decode_split(T, d_in, d_out)
    partial = torch.zeros((S, T, d_out), dtype=torch.float32, device=dev)
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)

    def gemm(i):
        s = sets[i % len(sets)]
        L.base_gemm_splitk_t(s.x, s.W0, ws, ksplit=0, partial=partial, stream=stream)

    def merge(i):
        s = sets[i % len(sets)]
        L.bgmv_adapter_merge_t(s.x, s.A, s.B, s.ids, s.scale, partial, ws, y=s.y, stream=stream)

    out = {"split": S, "n": n_steps}
    for name, fn in (("gemm_ms", gemm), ("adapter_merge_ms", merge)):
        out[name] = graph_mean_ms(fn, n_steps, stream)
    return out


def decode_blocks(sets, L, w, stream, pk, n_steps=400):
    """The scope table's a2 / a3 rows on their own, on the decode workload
    (rotating buffer sets): BGMV shrink, BGMV expand (accumulating into y),
    and the one-launch adapter term (shrink + cluster sum + expand, fp32 out).
    Algorithmic bytes: each distinct adapter's A or B once, x or v, y."""
    import numpy as np
    import torch
    T, d_in, d_out, r, n_slots, D = w.T, w.d_in, w.d_out, w.r, w.n_slots, w.distinct
    T_lora = int(((w.slot_ids >= 0) & (w.slot_ids < n_slots)).sum())
    dev = sets[0].x.device
    ks = fused_ksplit(T, d_in, d_out, n_slots, r)
    vpart = torch.zeros((ks, T, r), dtype=torch.float32, device=dev)
    delta = torch.zeros((T, d_out), dtype=torch.float32, device=dev)
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)

    def shrink(i):
        s = sets[i % len(sets)]
        L.bgmv_shrink_t(s.x, s.A, s.ids, s.scale, ks, ws, v_partial=vpart, stream=stream)

    def expand(i):
        s = sets[i % len(sets)]
        L.bgmv_expand_t(vpart, s.B, s.ids, s.y, ws, stream=stream)

    def adapter(i):
        s = sets[i % len(sets)]
        L.bgmv_adapter_t(s.x, s.A, s.B, s.ids, s.scale, ws, delta=delta, stream=stream)

    b_shrink = D * d_in * r * 2 + T * d_in * 2 + ks * T * r * 4
    b_expand = D * r * d_out * 2 + ks * T * r * 4 + 2 * T * d_out * 2
    b_adapter = D * r * (d_in + d_out) * 2 + T * d_in * 2 + T_lora * d_out * 4
    return {"workload": "decode_bgmv", "ksplit": ks,
            "bgmv_shrink": block_row(graph_mean_ms(shrink, n_steps, stream), b_shrink, pk),
            "bgmv_expand": block_row(graph_mean_ms(expand, n_steps, stream), b_expand, pk),
            "bgmv_adapter": block_row(graph_mean_ms(adapter, n_steps, stream), b_adapter, pk)}


def upload_point(L, sets, w, stream, n_steps=500, rounds=16):
    """The slot-upload path (lora_slot_upload) from pinned host memory: its
    H2D rate alone, and while the decode layer runs on another stream, with
    the layer's time per step alone and with the uploads running (the
    uploads go to slots the batch does not use)."""
    import numpy as np
    import torch
    T, d_in, d_out, r, n_slots = w.T, w.d_in, w.d_out, w.r, w.n_slots
    used = set(int(i) for i in w.slot_ids.tolist())
    free = [sl for sl in range(n_slots) if sl not in used][:64]
    g = torch.Generator().manual_seed(1002)
    A_h = (torch.randn((d_in, r), generator=g) / 64).to(torch.bfloat16).pin_memory()
    B_h = (torch.randn((r, d_out), generator=g) * 0.02).to(torch.bfloat16).pin_memory()
    per = (d_in * r + r * d_out) * 2
    side = torch.cuda.Stream(device=sets[0].x.device)
    pool = sets[1]     # the other sets keep their own pools

    def uploads():
        for _ in range(rounds):
            for sl in free:
                L.slot_upload_t(pool.A, pool.B, None, sl, A_h, B_h, 2.0, stream=side)

    nbytes = per * len(free) * rounds
    uploads()                               # warm
    side.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(side)
    uploads()
    e1.record(side)
    side.synchronize()
    alone_ms = e0.elapsed_time(e1)
    ws = L.workspace(L.OP_LINEAR_FUSED, T, d_in, d_out, r, n_slots, device=sets[0].x.device)

    def step(i):
        s = sets[[0, 2, 3][i % 3]]
        L.linear_fused_t(s.x, s.W0, s.A, s.B, s.ids, s.scale, ws, y=s.y, stream=stream)

    layer_ms = graph_mean_ms(step, n_steps, stream)
    gr = capture(step, n_steps, stream)
    torch.cuda.synchronize()
    f0 = torch.cuda.Event(enable_timing=True)
    f1 = torch.cuda.Event(enable_timing=True)
    u0 = torch.cuda.Event(enable_timing=True)
    u1 = torch.cuda.Event(enable_timing=True)
    u0.record(side)
    uploads()
    u1.record(side)
    f0.record(stream)
    with torch.cuda.stream(stream):
        gr.replay()
    f1.record(stream)
    torch.cuda.synchronize()
    both_ms = f0.elapsed_time(f1) / n_steps
    up_ms = u0.elapsed_time(u1)
    return {"adapter_bytes": per, "uploads": len(free) * rounds,
            "upload_gbs": nbytes / (alone_ms * 1e-3) / 1e9,
            "upload_gbs_during_layer": nbytes / (up_ms * 1e-3) / 1e9,
            "layer_us": layer_ms * 1e3, "layer_us_during_upload": both_ms * 1e3,
            "overlap_ms": min(up_ms, both_ms * n_steps)}


def e2e_pipelined(sets, L, T, d_in, d_out, r, n_slots, n_steps, stream, warm=300, group=4):
    """The public call with host buffers as a serving loop runs it, a group of
    `group` steps at a time: the group's H2D of x and ids (pinned memory) on a
    copy-in stream, its layers back to back on the compute stream, its D2H of
    y on a copy-out stream, over two groups' worth of device buffer sets, so
    group g + 1's H2D and group g - 1's D2H overlap group g's layers.  Groups
    depend on each other through events only (a group's buffers are reloaded
    once the layers of the group two back have read them, and its y rewritten
    once their D2H has read it), so the compute stream waits for copies once
    per group and consecutive layers inside a group keep their programmatic
    overlap.  Every step still copies its own inputs in and its own y out.
    n_steps steps (a multiple of `group`) are one CUDA graph, replayed after a
    warm-up replay; CUDA events on the compute stream around the replay.
    Returns ms for the n_steps steps."""
    import torch
    n = len(sets)
    G = group
    nb = 2 * G
    x_h = [s.x.cpu().pin_memory() for s in sets]
    ids_h = [s.ids.cpu().pin_memory() for s in sets]
    y_h = [torch.empty((T, d_out), dtype=sets[0].y.dtype).pin_memory() for _ in sets]
    x_d = [torch.empty_like(sets[0].x) for _ in range(nb)]
    ids_d = [torch.empty_like(sets[0].ids) for _ in range(nb)]
    y_d = [torch.empty_like(sets[0].y) for _ in range(nb)]
    ws = L.workspace(L.OP_LINEAR_FUSED, T, d_in, d_out, r, n_slots)
    s_in = torch.cuda.Stream(device=x_d[0].device)
    s_out = torch.cuda.Stream(device=x_d[0].device)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_c = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def steps(k):
        for g in range(k // G):
            e = g % 2
            with torch.cuda.stream(s_in):
                if g >= 2:
                    s_in.wait_event(ev_c[e])
                for j in range(G):
                    i = g * G + j
                    x_d[i % nb].copy_(x_h[i % n], non_blocking=True)
                    ids_d[i % nb].copy_(ids_h[i % n], non_blocking=True)
                ev_in[e].record(s_in)
            stream.wait_event(ev_in[e])
            if g >= 2:
                stream.wait_event(ev_out[e])
            for j in range(G):
                i = g * G + j
                s = sets[i % n]
                L.linear_fused_t(x_d[i % nb], s.W0, s.A, s.B, ids_d[i % nb], s.scale, ws,
                                 y=y_d[i % nb], stream=stream)
            ev_c[e].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_c[e])
                for j in range(G):
                    i = g * G + j
                    y_h[i % n].copy_(y_d[i % nb], non_blocking=True)
                ev_out[e].record(s_out)

    def graph(k):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                s_in.wait_stream(stream)
                s_out.wait_stream(stream)
                steps(k)
                stream.wait_stream(s_in)
                stream.wait_stream(s_out)
        return g

    with torch.cuda.stream(stream):
        steps(2 * G)
    torch.cuda.synchronize()
    g_warm, g = graph(warm - warm % G), graph(n_steps)
    graph_upload(g, stream)
    with torch.cuda.stream(stream):
        g_warm.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        l2_flush()
        torch.cuda._sleep(SPACER_CYCLES)
        e0.record(stream)
        g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    # the last group's host outputs against the same call on device buffers
    # (the kernels are deterministic, so the bits must agree)
    y_ref = torch.empty_like(sets[0].y)
    for j in range(G):
        i = n_steps - G + j
        s = sets[i % n]
        L.linear_fused_t(s.x, s.W0, s.A, s.B, s.ids, s.scale, ws, y=y_ref, stream=stream)
        stream.synchronize()
        if not torch.equal(y_h[i % n], y_ref.cpu()):
            raise RuntimeError(f"pipelined end-to-end loop: step {i}'s host output differs")
    return e0.elapsed_time(e1)


def e2e_steps(sets, L, T, d_in, d_out, r, n_slots, n_steps, stream, warm=300):
    """The public call with host buffers, every step inside the timed region:
    the H2D of that step's x and ids from pinned memory, the layer, the D2H of
    y.  Timed as a serving loop runs the call: the steps captured in CUDA
    graphs (memcpy nodes and the layer's kernels), timed like `value` with the
    weights rotating over the same sets, so W0 comes from HBM every step.  The
    same steps issued one by one from Python are timed as well (host launch
    overhead included).  Returns (graph ms, eager ms, h2d and d2h bytes per
    step)."""
    import torch
    n = len(sets)
    x_h = [s.x.cpu().pin_memory() for s in sets]
    ids_h = [s.ids.cpu().pin_memory() for s in sets]
    y_h = [torch.empty((T, d_out), dtype=sets[0].y.dtype).pin_memory() for _ in sets]
    x_d = torch.empty_like(sets[0].x)
    ids_d = torch.empty_like(sets[0].ids)
    y_d = torch.empty_like(sets[0].y)
    ws = L.workspace(L.OP_LINEAR_FUSED, T, d_in, d_out, r, n_slots)

    def step(i):
        s = sets[i % n]
        x_d.copy_(x_h[i % n], non_blocking=True)
        ids_d.copy_(ids_h[i % n], non_blocking=True)
        L.linear_fused_t(x_d, s.W0, s.A, s.B, ids_d, s.scale, ws, y=y_d, stream=stream)
        y_h[i % n].copy_(y_d, non_blocking=True)

    ms_graph, _ = timed_graph_steps(step, n_steps, warm, stream)
    with torch.cuda.stream(stream):
        for i in range(20):
            step(i)
    stream.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(n_steps):
            step(i)
        e1.record(stream)
    stream.synchronize()
    ms_eager = e0.elapsed_time(e1)
    h2d = x_h[0].numel() * x_h[0].element_size() + ids_h[0].numel() * 4
    return ms_graph, ms_eager, h2d, y_h[0].numel() * y_h[0].element_size()


def device_normal(shape, std, seed, dev):
    import torch
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    t = torch.empty(shape, dtype=torch.float32, device=dev)
    t.normal_(0.0, std, generator=g)
    return t.to(torch.bfloat16)


def sweep(L, stream, pk, dev, steps=2000, warm=300):
    """Distinct adapters per batch: tokens/s and achieved GB/s of the fused
    layer over the diversity workload (weights drawn on the device)."""
    import numpy as np
    import torch
    from lora_serving_device_gb300 import workloads as W
    d_in = d_out = 4096
    r, n_slots = 16, 1024
    bases = []
    for s in range(NSETS):
        W0 = device_normal((d_in, d_out), W.W0_STD, 40400 + s, dev)
        A = device_normal((n_slots, d_in, r), W.A_STD, 40410 + s, dev)
        B = device_normal((n_slots, r, d_out), W.B_STD, 40420 + s, dev)
        bases.append((W0, A, B))
    scale = torch.full((n_slots,), W.SCALE, dtype=torch.float32, device=dev)
    out = []
    for T, k in W.SWEEP_POINTS:
        ids = torch.from_numpy(W.sweep_ids(T, k)).to(dev)
        x = device_normal((T, d_in), 1.0, 40430 + T, dev)
        sets = [LayerSet(x, b[0], b[1], b[2], ids, scale,
                         torch.empty((T, d_out), dtype=torch.bfloat16, device=dev)) for b in bases]
        ws = L.workspace(L.OP_LINEAR_FUSED, T, d_in, d_out, r, n_slots)

        def fn(i):
            s = sets[i % NSETS]
            L.linear_fused_t(s.x, s.W0, s.A, s.B, s.ids, s.scale, ws, y=s.y, stream=stream)

        ms, _ = timed_graph_steps(fn, steps, warm, stream)
        t_step = ms / 1e3 / steps
        nbytes = layer_bytes(T, d_in, d_out, r, k)
        gbs = nbytes / t_step / 1e9
        roof_s = nbytes / (pk["hbm_gbs"] * 1e9)
        out.append({"T": T, "distinct": k, "us_per_step": t_step * 1e6,
                    "tokens_per_s": T / t_step, "gbs": gbs, "frac": gbs / pk["hbm_gbs"],
                    "roofline_us": roof_s * 1e6, "latency_floored": roof_s < 5e-6})
    del bases
    torch.cuda.empty_cache()
    return out


def prefill_point(L, stream, pk, dev, steps=30, warm=5):
    import numpy as np
    import torch
    from lora_serving_device_gb300 import workloads as W
    lengths, slots = W.prefill_ids()
    ids_np = np.repeat(np.array(slots, np.int32), np.array(lengths))
    T = int(ids_np.size)
    d_in, d_out, r, n_slots = 4096, 14336, 64, 64
    x = device_normal((T, d_in), 1.0, 30301, dev)
    W0 = device_normal((d_in, d_out), W.W0_STD, 30302, dev)
    A = device_normal((n_slots, d_in, r), W.A_STD, 30303, dev)
    B = device_normal((n_slots, r, d_out), W.B_STD, 30304, dev)
    ids = torch.from_numpy(ids_np).to(dev)
    scale = torch.full((n_slots,), W.SCALE, dtype=torch.float32, device=dev)
    y = torch.empty((T, d_out), dtype=torch.bfloat16, device=dev)
    ws = L.workspace(L.OP_LINEAR_FUSED, T, d_in, d_out, r, n_slots)

    def fn(i):
        L.linear_fused_t(x, W0, A, B, ids, scale, ws, y=y, stream=stream)

    ms, _ = timed_graph_steps(fn, steps, warm, stream)
    t = ms / 1e3 / steps
    D = int(np.unique(ids_np).size)
    flops = 2.0 * T * d_in * d_out + 2.0 * T * r * (d_in + d_out)
    nbytes = layer_bytes(T, d_in, d_out, r, D)
    tf = flops / t / 1e12
    # the scope table's a1 / a2 / a3 rows on their own on this workload
    ks, kx = SGMV_SHRINK_KSPLIT, SGMV_EXPAND_KSPLIT
    wss = torch.zeros(256, dtype=torch.uint8, device=dev)
    segs = L.build_segments_t(ids, n_slots, wss, stream=stream)
    vpart = torch.zeros((ks, T, r), dtype=torch.float32, device=dev)
    vpart_x = torch.zeros((kx, T, r), dtype=torch.float32, device=dev)
    L.sgmv_shrink_t(x, A, segs, scale, kx, wss, v_partial=vpart_x, stream=stream)
    b_seg = 4 * T + 4 * T + 8 * D + 8
    b_shrink = D * d_in * r * 2 + T * d_in * 2 + ks * T * r * 4
    b_expand = D * r * d_out * 2 + kx * T * r * 4 + 2 * T * d_out * 2
    blocks = {
        "ksplit": {"sgmv_shrink": ks, "sgmv_expand": kx},
        "build_segments": block_row(graph_mean_ms(
            lambda i: L.build_segments_t(ids, n_slots, wss, stream=stream), 50, stream), b_seg, pk),
        "sgmv_shrink": block_row(graph_mean_ms(
            lambda i: L.sgmv_shrink_t(x, A, segs, scale, ks, wss, v_partial=vpart, stream=stream),
            30, stream), b_shrink, pk),
        "sgmv_expand": block_row(graph_mean_ms(
            lambda i: L.sgmv_expand_t(vpart_x, B, segs, y, wss, stream=stream), 30, stream),
            b_expand, pk)}
    # the same layer over a 4-bit base: W0 dequantised once per call into the
    # workspace, then the bf16 prefill path
    cb = _up(W.nf4_like_codebook(), dev)
    base4 = L.Base4bit.quantize(W0, cb, stream=stream)
    ws4 = L.workspace(L.OP_LINEAR_FUSED_4BIT, T, d_in, d_out, r, n_slots)
    ms4, _ = timed_graph_steps(
        lambda i: L.linear_fused_4bit_t(x, base4, A, B, ids, scale, ws4, y=y, stream=stream),
        steps, warm, stream)
    t4 = ms4 / 1e3 / steps
    prefill_4bit = {"workload": "prefill_sgmv with W0 as 4-bit codes + bf16 absmax per 64-row "
                                "block, dequantised once per call into the workspace",
                    "ms_per_step": t4 * 1e3, "tokens_per_s": T / t4,
                    "tflops": flops / t4 / 1e12, "frac_burst_bf16": flops / t4 / 1e12 / pk["bf16_tflops"],
                    "device_error": L.get_error_t(ws4, stream=stream)}
    del base4, ws4
    # the same layer over a ragged-rank pool (ranks drawn from 8 / 16 / 64 per
    # slot, as in workload 5): with its own workspace it takes the prefill
    # route over a compact padded copy of the batch's adapters; with a
    # workspace for 256 tokens, 256-token chunks of the decode path
    ranks = W.stack_ranks(n_slots)
    pool = L.RaggedPool.from_padded(A, B, ranks)
    wsr = L.workspace(L.OP_LINEAR_FUSED_RAGGED, T, d_in, d_out, pool.r_max, n_slots)
    msr, _ = timed_graph_steps(
        lambda i: L.linear_fused_ragged_t(x, W0, pool, ids, scale, wsr, y=y, stream=stream),
        steps, warm, stream)
    err_r = L.get_error_t(wsr, stream=stream)
    del wsr
    wsc = L.workspace(L.OP_LINEAR_FUSED, 256, d_in, d_out, pool.r_max, n_slots)
    msc, _ = timed_graph_steps(
        lambda i: L.linear_fused_ragged_t(x, W0, pool, ids, scale, wsc, y=y, stream=stream),
        max(3, steps // 10), 2, stream)
    tr = msr / 1e3 / steps
    tc = msc / 1e3 / max(3, steps // 10)
    prefill_ragged = {"workload": "prefill_sgmv over a ragged-rank pool (ranks 8 / 16 / 64 per "
                                  "slot), the prefill route (the batch's adapters padded to the "
                                  "pool's rank 64 in the workspace)",
                      "ms_per_step": tr * 1e3, "tokens_per_s": T / tr,
                      "tflops": flops / tr / 1e12, "frac_burst_bf16": flops / tr / 1e12 / pk["bf16_tflops"],
                      "device_error": err_r,
                      "chunked_decode_path_ms": tc * 1e3}
    del pool, wsc
    res = {"workload": "prefill_sgmv: 4096->14336, rank 64, 64 slots, 16 prefill requests "
                       "(U[64,1024] tokens) + 48 decode tokens",
           "T": T, "distinct": D, "ms_per_step": t * 1e3, "tokens_per_s": T / t,
           "tflops": tf, "gbs": nbytes / t / 1e9,
           # timed alone for well under a second: the burst peak applies
           "roofline": {"bound": "tensor", "achieved": tf, "peak": pk["bf16_tflops"],
                        "unit": "TFLOP/s", "frac": tf / pk["bf16_tflops"],
                        "peak_kind": "burst (cuBLAS bf16, measured)",
                        "frac_vs_sustained": tf / pk["bf16_tflops_sustained"]},
           "blocks": blocks, "prefill_4bit": prefill_4bit, "prefill_ragged": prefill_ragged}
    del x, W0, A, B
    torch.cuda.empty_cache()
    return res


def q4_point(L, sets, w, stream, pk, steps=4000, warm=400):
    """The decode layer with its base matrix in 4 bits (codebook + bf16
    absmax per 64-row block, quantised by the library), bf16 adapters."""
    import torch
    from lora_serving_device_gb300 import workloads as W
    T, d_in, d_out, r, n_slots = w.T, w.d_in, w.d_out, w.r, w.n_slots
    cb = _up(W.nf4_like_codebook(), sets[0].x.device)
    bases = [L.Base4bit.quantize(s.W0, cb, stream=stream) for s in sets]
    stream.synchronize()
    ws = L.workspace(L.OP_LINEAR_FUSED_4BIT, T, d_in, d_out, r, n_slots, device=sets[0].x.device)
    n = len(sets)

    def step(i):
        s = sets[i % n]
        L.linear_fused_4bit_t(s.x, bases[i % n], s.A, s.B, s.ids, s.scale, ws, y=s.y,
                              stream=stream)

    ms, _ = timed_graph_steps(step, steps, warm, stream)
    err = L.get_error_t(ws, stream=stream)
    t = ms / 1e3 / steps
    qbytes = d_in * d_out // 2 + (d_in // 64) * d_out * 2
    D = w.distinct
    lb = qbytes + (D * r * (d_in + d_out) + T * d_in + T * d_out) * 2 + T * 4
    split = L.lora_decode_split(T, d_in, d_out)
    part = torch.empty((split, T, d_out), dtype=torch.float32, device=sets[0].x.device)
    gemm_ms = graph_mean_ms(lambda i: L.base_gemm_4bit_splitk_t(
        sets[i % n].x, bases[i % n], ws, ksplit=split, partial=part, stream=stream), 400, stream)
    gb = qbytes + T * d_in * 2 + T * d_out * 4
    res = {"workload": "decode_4bit: " + DECODE_DESC + "; W0 as 4-bit codes + bf16 absmax per "
                       "64-row block (0.53 B/weight)",
           "us_per_step": t * 1e6, "tokens_per_s": T / t, "layer_bytes": lb,
           "gbs": lb / t / 1e9, "frac": lb / t / 1e9 / pk["hbm_gbs"], "device_error": err,
           "gemm": dict(block_row(gemm_ms, gb, pk),
                        kernel="decode_q4_kernel (4-bit dequant in the mainloop, tcgen05)")}
    del bases
    torch.cuda.empty_cache()
    return res


def stack_point(L, stream, pk, dev, steps=5, warm=3, ragged=False):
    """The 8B-shaped stack: 32 layers x 7 projections, one fused call each.
    ragged: every adapter kept at its own rank (8, 16 or 64) in a ragged pool
    instead of zero-padded to 64."""
    import numpy as np
    import torch
    from lora_serving_device_gb300 import workloads as W
    ranks = W.stack_ranks()
    ids_np = W.stack_ids()
    ids = torch.from_numpy(ids_np).to(dev)
    scale = torch.full((250,), W.SCALE, dtype=torch.float32, device=dev)
    layers = []
    for layer in range(W.STACK_LAYERS):
        for p in range(7):
            t = W.stack_layer_device(layer, p, device=dev, ranks=ranks)
            _, d_in, d_out = W.STACK_PROJECTIONS[p]
            pool = None
            if ragged:
                pool = L.RaggedPool.from_padded(t.pop("A_pool"), t.pop("B_pool"), ranks)
            ws = L.workspace(L.OP_LINEAR_FUSED, 256, d_in, d_out, 64, 250)
            y = torch.empty((256, d_out), dtype=torch.bfloat16, device=dev)
            layers.append((t, pool, ws, y))

    def fn(i):
        for t, pool, ws, y in layers:
            if pool is None:
                L.linear_fused_t(t["x"], t["W0"], t["A_pool"], t["B_pool"], ids, scale, ws, y=y,
                                 stream=stream)
            else:
                L.linear_fused_ragged_t(t["x"], t["W0"], pool, ids, scale, ws, y=y,
                                        stream=stream)

    ms, _ = timed_graph_steps(fn, steps, warm, stream)
    t = ms / 1e3 / steps
    used = np.unique(ids_np[ids_np >= 0])
    D = int(used.size)
    # each distinct adapter's A and B once, at the rank the pool stores it
    rank_sum = int(sum(int(ranks[a]) for a in used)) if ragged else 64 * D
    nbytes = sum((di * do + rank_sum * (di + do) + 256 * (di + do)) * 2 + 256 * 4
                 for _, di, do in W.STACK_PROJECTIONS) * W.STACK_LAYERS
    form = "ranks 8/16/64 each at its own rank (ragged pool)" if ragged else \
        "ranks 8/16/64 padded to 64"
    res = {"workload": f"stack_8b: 32 layers x 7 projections, 250 slots ({form}), T=256",
           "distinct": D, "adapter_rank_sum": rank_sum, "ms_per_step": t * 1e3,
           "tokens_per_s": 256 / t, "gbs": nbytes / t / 1e9,
           "frac": nbytes / t / 1e9 / pk["hbm_gbs"]}
    del layers
    torch.cuda.empty_cache()
    return res


def run_ours(args):
    import numpy as np
    import torch
    from lora_serving_device_gb300 import build as B
    from lora_serving_device_gb300 import lora as L
    from lora_serving_device_gb300 import workloads as W

    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_setup("nccl")
    if rank == 0 and not os.path.exists(L.LIB_PATH):
        B.build()
    barrier()
    L.load()
    pk = peaks()
    stream = torch.cuda.Stream(device=dev)

    # clocks and throttle reasons over the whole run, timed regions included
    gpu_index = os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[0] or str(local)
    clk = ClockSampler(gpu_index if world == 1 else str(local))

    w = W.decode_bgmv()
    T, d_in, d_out, r, n_slots = w.T, w.d_in, w.d_out, w.r, w.n_slots
    D = w.distinct
    s0 = LayerSet(_up(w.x, dev), _up(w.W0, dev), _up(w.A_pool, dev), _up(w.B_pool, dev),
                  torch.from_numpy(w.slot_ids).to(dev), torch.from_numpy(w.scale).to(dev),
                  torch.empty((T, d_out), dtype=torch.bfloat16, device=dev))
    sets = [s0] + [s0.clone() for _ in range(NSETS - 1)]
    ws = L.workspace(L.OP_LINEAR_FUSED, T, d_in, d_out, r, n_slots, device=dev)

    def step(i):
        s = sets[i % NSETS]
        L.linear_fused_t(s.x, s.W0, s.A, s.B, s.ids, s.scale, ws, y=s.y, stream=stream)

    ms, wall = timed_graph_steps(step, args.steps, args.warmup, stream)
    timing = dict(TIMING)
    ms_max = reduce_max(ms, device=dev)
    err = L.get_error_t(ws, stream=stream)
    if err:
        raise SystemExit(f"device error word {err:#x}")
    value = world * T * args.steps / (ms_max / 1e3)

    try:
        kt = per_kernel_times(sets, L, T, d_in, d_out, r, n_slots, 400, stream)
        blocks = decode_blocks(sets, L, w, stream, pk)
    except RuntimeError as e:
        print(f"per-kernel timing unavailable: {e}", file=sys.stderr)
        kt, blocks = None, None
    e2e_ms, e2e_eager_ms, h2d, d2h = e2e_steps(sets, L, T, d_in, d_out, r, n_slots, 2000, stream)
    e2e_ms = reduce_max(e2e_ms, device=dev)
    e2e_eager_ms = reduce_max(e2e_eager_ms, device=dev)
    e2e_pipe_ms = reduce_max(e2e_pipelined(sets, L, T, d_in, d_out, r, n_slots, 2000, stream,
                                           group=E2E_GROUP), device=dev)
    e2e_step_ms = reduce_max(e2e_pipelined(sets, L, T, d_in, d_out, r, n_slots, 2000, stream,
                                           group=1), device=dev)
    if rank != 0:
        clk.stop()
        barrier()
        return 0

    step_s = ms_max / 1e3 / args.steps
    gb = gemm_bytes(T, d_in, d_out)
    roof = None
    if kt is not None:
        ach = gb / (kt["gemm_ms"] / 1e3) / 1e9
        traffic = dram_traffic_per_launch()
        roof = {"bound": "hbm", "achieved": ach, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": ach / pk["hbm_gbs"], "traffic": traffic,
                "kernel": "decode_gemm_kernel (tcgen05 swap-AB base GEMM, split over d_in)",
                "algorithmic_bytes_per_launch": gb, "launch_us": kt["gemm_ms"] * 1e3,
                "peak_source": pk["source"], "frac_vs_8tbs": ach / 8000.0}
    lb = layer_bytes(T, d_in, d_out, r, D)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded)",
        "config": {"workload": DECODE_DESC, "T": T, "d_in": d_in, "d_out": d_out, "r": r,
                   "n_slots": n_slots, "distinct": D,
                   "l2": f"{NSETS} rotating buffer sets (>2x L2); a clean read of 256 MB before the start event", "parallelism": "replicas",
                   "graph": ("one CUDA graph of the K steps, uploaded before the timed region"
                             if timing.get("graph_uploaded") else
                             f"{timing.get('replays')} replays of one graph the warm-up also "
                             f"replays"),
                   "launch_latency": "hidden behind a GPU spin queued before the start event"},
        "layer_gbs": lb / step_s / 1e9, "layer_frac": lb / step_s / 1e9 / pk["hbm_gbs"],
        "gpu_launches": 2 * args.steps,
        "e2e": {"value": world * T * 2000 / (e2e_pipe_ms / 1e3), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_pipe_ms / 2000,
                "mode": f"2000 steps from one CUDA graph, as a serving loop runs them, "
                        f"{E2E_GROUP} steps at a time: per step the H2D of x and ids from "
                        f"pinned memory (copy-in stream), lora_linear_fused, the D2H of y "
                        f"(copy-out stream); the compute stream waits for a group's copies "
                        f"once, and the next group's H2D and the previous group's D2H "
                        f"overlap its layers ({2 * E2E_GROUP} device buffer sets); weights "
                        f"rotate over the 4 sets",
                "per_step": {"value": world * T * 2000 / (e2e_step_ms / 1e3),
                             "ms_per_step": e2e_step_ms / 2000,
                             "mode": "the same loop with the compute stream waiting for "
                                     "copies at every step (two buffer sets)"},
                "serial": {"value": world * T * 2000 / (e2e_ms / 1e3),
                           "ms_per_step": e2e_ms / 2000,
                           "mode": "the same steps in one stream, each step's copies and "
                                   "layer one after another (CUDA graphs)"},
                "eager": {"value": world * T * 2000 / (e2e_eager_ms / 1e3),
                          "ms_per_step": e2e_eager_ms / 2000,
                          "mode": "the serial steps issued from Python one by one"}},
        "roofline": roof,
        "kernels_ms": kt, "blocks": blocks,
    }
    line["slot_upload"] = upload_point(L, sets, w, stream)
    cfgs = {"decode_4bit": q4_point(L, sets, w, stream, pk)}
    if not args.no_sweep:
        line["sweep"] = sweep(L, stream, pk, dev)
    if not args.no_prefill:
        cfgs["prefill_sgmv"] = prefill_point(L, stream, pk, dev)
    if not args.no_stack:
        cfgs["stack_8b"] = stack_point(L, stream, pk, dev)
        cfgs["stack_8b_ragged"] = stack_point(L, stream, pk, dev, ragged=True)
    if cfgs:
        line["configs"] = cfgs
    clk.stop()
    line["clocks"] = clk.summary()
    line["clocks"]["period_ms"] = 50
    line["clocks"]["timed_region"] = clk.summary((wall[0] - 0.06, wall[1] + 0.06))
    if world == 1 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline()
    print(json.dumps(line), flush=True)
    barrier()
    return 0


def relaunch(n, argv=None):
    """--gpus N > 1 without a launcher: run this script under
    torch.distributed.run with N ranks on this node (one replica per GPU)."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__)]
    cmd += list(sys.argv[1:] if argv is None else argv)
    return subprocess.call(cmd)


def run_profile(case):
    """Three untimed passes of one workload's kernels, nothing else: a short
    command for a profiler's launch list or a single-kernel capture."""
    import numpy as np
    import torch
    from lora_serving_device_gb300 import build as B
    from lora_serving_device_gb300 import lora as L
    from lora_serving_device_gb300 import workloads as W
    if not os.path.exists(L.LIB_PATH):
        B.build()
    L.load()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.Stream(device=dev)
    if case == "prefill":
        lengths, slots = W.prefill_ids()
        ids_np = np.repeat(np.array(slots, np.int32), np.array(lengths))
        T, d_in, d_out, r, n_slots = int(ids_np.size), 4096, 14336, 64, 64
        x = device_normal((T, d_in), 1.0, 30301, dev)
        W0 = device_normal((d_in, d_out), W.W0_STD, 30302, dev)
        A = device_normal((n_slots, d_in, r), W.A_STD, 30303, dev)
        Bp = device_normal((n_slots, r, d_out), W.B_STD, 30304, dev)
        ids = torch.from_numpy(ids_np).to(dev)
        scale = torch.full((n_slots,), W.SCALE, dtype=torch.float32, device=dev)
        y = torch.empty((T, d_out), dtype=torch.bfloat16, device=dev)
        ws = L.workspace(L.OP_LINEAR_FUSED, T, d_in, d_out, r, n_slots)
        ks, kx = SGMV_SHRINK_KSPLIT, SGMV_EXPAND_KSPLIT
        wss = torch.zeros(256, dtype=torch.uint8, device=dev)
        vpart = torch.zeros((ks, T, r), dtype=torch.float32, device=dev)
        vpart_x = torch.zeros((kx, T, r), dtype=torch.float32, device=dev)
        for _ in range(3):
            L.linear_fused_t(x, W0, A, Bp, ids, scale, ws, y=y, stream=stream)
            segs = L.build_segments_t(ids, n_slots, wss, stream=stream)
            L.sgmv_shrink_t(x, A, segs, scale, ks, wss, v_partial=vpart, stream=stream)
            L.sgmv_shrink_t(x, A, segs, scale, kx, wss, v_partial=vpart_x, stream=stream)
            L.sgmv_expand_t(vpart_x, Bp, segs, y, wss, stream=stream)
        err = L.get_error_t(ws, stream=stream)
    elif case == "sweep256":
        # the T = 256 sweep point with 16 distinct adapters (weights drawn on
        # the device as in the sweep)
        T, d_in, d_out, r, n_slots = 256, 4096, 4096, 16, 1024
        W0 = device_normal((d_in, d_out), W.W0_STD, 40400, dev)
        A = device_normal((n_slots, d_in, r), W.A_STD, 40410, dev)
        Bp = device_normal((n_slots, r, d_out), W.B_STD, 40420, dev)
        x = device_normal((T, d_in), 1.0, 40430 + T, dev)
        ids = torch.from_numpy(W.sweep_ids(T, 16)).to(dev)
        scale = torch.full((n_slots,), W.SCALE, dtype=torch.float32, device=dev)
        y = torch.empty((T, d_out), dtype=torch.bfloat16, device=dev)
        ws = L.workspace(L.OP_LINEAR_FUSED, T, d_in, d_out, r, n_slots)
        for _ in range(3):
            L.linear_fused_t(x, W0, A, Bp, ids, scale, ws, y=y, stream=stream)
        err = L.get_error_t(ws, stream=stream)
    else:
        w = W.decode_bgmv()
        s0 = LayerSet(_up(w.x, dev), _up(w.W0, dev), _up(w.A_pool, dev), _up(w.B_pool, dev),
                      torch.from_numpy(w.slot_ids).to(dev), torch.from_numpy(w.scale).to(dev),
                      torch.empty((w.T, w.d_out), dtype=torch.bfloat16, device=dev))
        ws = L.workspace(L.OP_LINEAR_FUSED, w.T, w.d_in, w.d_out, w.r, w.n_slots, device=dev)
        if case == "decode4bit":
            base = L.Base4bit.quantize(s0.W0, _up(W.nf4_like_codebook(), dev), stream=stream)
            run = lambda: L.linear_fused_4bit_t(s0.x, base, s0.A, s0.B, s0.ids, s0.scale, ws,
                                                y=s0.y, stream=stream)
        elif case == "ragged":
            ranks = W.stack_ranks(w.n_slots) // 4          # 2, 4 or 16 -> classes 8, 8, 16
            pool = L.RaggedPool.from_padded(s0.A, s0.B, np.minimum(ranks, w.r))
            run = lambda: L.linear_fused_ragged_t(s0.x, s0.W0, pool, s0.ids, s0.scale, ws,
                                                  y=s0.y, stream=stream)
        else:
            run = lambda: L.linear_fused_t(s0.x, s0.W0, s0.A, s0.B, s0.ids, s0.scale, ws,
                                           y=s0.y, stream=stream)
        for _ in range(3):
            run()
        err = L.get_error_t(ws, stream=stream)
    stream.synchronize()
    if err:
        raise SystemExit(f"device error word {err:#x}")
    print(f"profile case {case}: 3 passes done")
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.oracle_child:
        return oracle_child(args.oracle_child, args.oracle_budget)
    rank, world, _ = dist_env()
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        return relaunch(args.gpus, argv)
    if world != args.gpus:
        raise SystemExit(f"--gpus {args.gpus} but the launcher started {world} ranks")
    if args.profile:
        return run_profile(args.profile)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
