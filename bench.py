#!/usr/bin/env python
"""Benchmark of the per-token-group fp8 e4m3 quantization hot path on GB300.

One step = one pass of the whole path over one batch of synthetic input:
  colwise   X (65536, 4096) bf16, 16 token groups along dim0 -> e4m3 + scales
  rowwise_t A (8192, 16640) bf16, 64 token groups along dim1 (two empty,
            0.5% outlier columns) -> e4m3 A^T + scales
the two large workloads of the pytorch/ao PR pages (#2668's (65536, 4096)
benchmark shape, #2863's (Mg, N) = (16640, 8192) shape).

Metric: achieved HBM GB/s counted algorithmically -- 2 bytes read + 1 byte
written per element plus 4 bytes per scale (the ideal of one read) -- over
the device time of the timed steps; also us per call.  Inputs (512 MB and
272 MB) are larger than L2 (126 MB) and disjoint, so no L2 flush is needed.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mine|reference]

N > 1 runs under torchrun, one rank per GPU, each rank on its own batch
(weak scaling, no data-path collective); time is the max over ranks.
``--impl reference`` times the CPU oracle (the plain C statement of the
method) on bounded samples of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = ("achieved HBM GB/s and % of GB300 peak for per-group fp8 quant "
          "(algorithmic bytes: 2 B read + 1 B written per element + 4 B per "
          "scale); us/call")
UNIT = "GB/s"
COLWISE_SHAPE = (65536, 4096, 16)   # M, K, groups
ROWWISE_SHAPE = (8192, 16640, 64)   # N, Mg, groups
FALLBACK_HBM_GBS = 6800.0
# pytorch/ao PR pages, hardware unstated: context only
PAGES_CONTEXT = {
    "colwise_65536x4096_g16_triton_us": 1603.23,
    "rowwise_16640x8192_g64_triton_transpose_us": 784.288,
    "source": "pytorch/ao #2668 new-autotune table; #2863 Benchmarks table",
}
POW2 = False  # --pow2-scales
# the sources each kernel's recorded DRAM traffic depends on
KERNEL_SOURCES = {"colwise": ["gq_device.cuh", "gq_colwise.cu"],
                  "rowwise_t": ["gq_device.cuh", "gq_rowwise.cu"]}


# ------------------------------------------------------------- helpers --

def colwise_bytes(M, K, G):
    return 3 * M * K + 4 * G * K


def rowwise_bytes(N, Mg, G):
    return 3 * N * Mg + 4 * N * G


def step_bytes():
    return colwise_bytes(*COLWISE_SHAPE) + rowwise_bytes(*ROWWISE_SHAPE)


def kernel_source_hash(kernel: str) -> str:
    h = hashlib.sha256()
    d = os.path.join(ROOT, "fp8_quantization_moe_gb300", "csrc")
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(d, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def traffic_record(kernel: str):
    """dram bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    rec = d.get(kernel)
    if not rec or rec.get("kernel_source_hash") != kernel_source_hash(kernel):
        return None
    return rec


def reduce_over_ranks(ms: float, nbytes: int, dist_ok: bool):
    """Max of the per-rank timed milliseconds and sum of the per-rank bytes."""
    if not dist_ok:
        return ms, nbytes
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([ms], dtype=torch.float64, device=dev)
    b = torch.tensor([nbytes], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(b, op=dist.ReduceOp.SUM)
    return float(t.item()), int(b.item())


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples in a background process."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
             "sw_power_cap")

    def __init__(self, gpu_id: str):
        self.samples = []  # (time, sm, max, reasons)
        self.proc = None
        self.gpu_id = gpu_id
        self.t_load = [None, None]

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100", "-i",
                 self.gpu_id], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
        except OSError:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm, mx = float(parts[0]), float(parts[1])
            except ValueError:
                continue
            reasons = [n for n, v in zip(self.NAMES, parts[4:8]) if v == "Active"]
            self.samples.append((time.time(), sm, mx, reasons))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        t0, t1 = self.t_load
        load = [s for s in self.samples
                if t0 is not None and t1 is not None and t0 <= s[0] <= t1]
        if not load:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "samples": 0, "note": "no nvidia-smi samples"}
        reasons = sorted({r for s in load for r in s[3]})
        return {"sm_mhz": statistics.median(s[1] for s in load),
                "sm_max_mhz": max(s[2] for s in load), "reasons": reasons,
                "samples": len(load),
                "window": "sustained run of the same step around the timed "
                          "region"}


# -------------------------------------------------------- the CPU oracle --

def oracle_sample_gbs(budget_s: float = 12.0):
    """The oracle, as it stands, on bounded samples of the workload: the
    colwise path on a 512-column slice of X (all 65536 rows, the same 16
    groups) and the rowwise_t path on a 512-row slice of A (all 16640
    columns, the same 64 groups).  Returns (GB/s, seconds, sample text)."""
    import numpy as np

    import oracle
    from fp8_quantization_moe_gb300 import synth

    M, K, G = COLWISE_SHAPE
    N, Mg, Gr = ROWWISE_SHAPE
    kc, nr = 512, 512
    c = synth.colwise_large(G, rows=M, cols=kc)
    r = synth.rowwise_outliers(Gr, N=nr, Mg=Mg)
    o = oracle.get()
    nbytes, secs = 0, 0.0
    reps = 0
    while secs < budget_s or reps == 0:
        t = time.perf_counter()
        o.colwise(c.x, c.offs)
        o.rowwise_t(r.x, r.offs)
        secs += time.perf_counter() - t
        nbytes += colwise_bytes(M, kc, G) + rowwise_bytes(nr, Mg, Gr)
        reps += 1
        if secs > budget_s / 2 and reps >= 1:
            break
    sample = (f"colwise {M}x{kc} (16 groups) + rowwise_t {nr}x{Mg} (64 groups), "
              f"{reps} pass(es), {secs:.1f} s single-threaded")
    return nbytes / secs / 1e9, secs, sample


def oracle_parallel_gbs(budget_s: float = 4.0):
    """The same oracle on the same samples, split into independent units over
    every host core: column slices of X (each with all rows and the same
    groups) and row slices of A (each with all token columns); threads call
    the C oracle, which runs without the interpreter lock.  Returns (GB/s,
    threads, sample text)."""
    import concurrent.futures as cf

    import numpy as np

    import oracle
    from fp8_quantization_moe_gb300 import synth

    M, K, G = COLWISE_SHAPE
    N, Mg, Gr = ROWWISE_SHAPE
    kc, nr = 512, 512
    c = synth.colwise_large(G, rows=M, cols=kc)
    r = synth.rowwise_outliers(Gr, N=nr, Mg=Mg)
    o = oracle.get()
    n = max(1, os.cpu_count() or 1)
    cols = [np.ascontiguousarray(c.x[:, j::n]) for j in range(n) if c.x[:, j::n].shape[1] > 0]
    rows = [np.ascontiguousarray(r.x[j::n]) for j in range(n) if r.x[j::n].shape[0] > 0]
    nbytes, secs, reps = 0, 0.0, 0
    with cf.ThreadPoolExecutor(n) as ex:
        while secs < budget_s or reps == 0:
            t = time.perf_counter()
            jobs = [ex.submit(o.colwise, x, c.offs) for x in cols]
            jobs += [ex.submit(o.rowwise_t, a, r.offs) for a in rows]
            for j in jobs:
                j.result()
            secs += time.perf_counter() - t
            nbytes += colwise_bytes(M, kc, G) + rowwise_bytes(nr, Mg, Gr)
            reps += 1
    sample = (f"the same samples split into {len(cols)} column slices + {len(rows)} row "
              f"slices on {n} threads, {reps} pass(es), {secs:.1f} s")
    return nbytes / secs / 1e9, n, sample


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import numpy as np  # noqa: F401

    import oracle
    from fp8_quantization_moe_gb300 import synth

    oracle.build()
    o = oracle.get()
    M, K, G = COLWISE_SHAPE
    N, Mg, Gr = ROWWISE_SHAPE
    kc, nr = 128, 128  # per-step sample: ~1 s of oracle work
    c = synth.colwise_large(G, rows=M, cols=kc)
    r = synth.rowwise_outliers(Gr, N=nr, Mg=Mg)
    per_step = colwise_bytes(M, kc, G) + rowwise_bytes(nr, Mg, Gr)
    for _ in range(args.warmup):
        o.colwise(c.x, c.offs)
        o.rowwise_t(r.x, r.offs)
    t = time.perf_counter()
    for _ in range(args.steps):
        o.colwise(c.x, c.offs)
        o.rowwise_t(r.x, r.offs)
    secs = time.perf_counter() - t
    gbs = per_step * args.steps / secs / 1e9
    sample = (f"per step: colwise {M}x{kc} of X (16 groups) + rowwise_t "
              f"{nr}x{Mg} of A (64 groups), single-threaded C oracle")
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": secs * 1e3 / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16->e4m3 (fp32 scale math)",
        "data": "synthetic (seeded)",
        "config": {"workload": "colwise 65536x4096 g16 + rowwise_t 8192x16640 g64 "
                   "(bounded column/row samples on the CPU)",
                   "parallelism": "single CPU thread"},
        "cpu_baseline": {"value": gbs, "unit": UNIT, "cores": oracle.threads_used(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": gbs, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------- GPU path --

EXPERT_SHAPE = (8, 4096, 4096)  # --expert-dim1: E experts of (K, N) weights


def run_expert(args):
    """Times the stacked expert-weight path (scales along dim1) on one GPU:
    one call = one step; same metric and timing rules as the main bench."""
    import numpy as np
    import torch

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    import __graft_entry__

    __graft_entry__.build()
    import fp8_quantization_moe_gb300 as gq
    from fp8_quantization_moe_gb300 import synth

    E, K, N = EXPERT_SHAPE
    rng = np.random.default_rng(1700)
    x = rng.standard_normal((E, K, N), dtype=np.float32)
    x *= np.power(np.float32(10), rng.uniform(-2, 2, size=(E, 1, N))).astype(np.float32)
    w = torch.from_numpy(synth.to_bf16_bits(x).view(np.int16)).view(torch.bfloat16).to(dev)
    del x
    q = torch.empty((E, K, N), dtype=torch.float8_e4m3fn, device=dev)
    sc = torch.empty((E, N), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        gq.expert_dim1(w, out=q, scales=sc, stream=stream, pow2_scales=POW2)
    torch.cuda.synchronize(dev)
    gq.check_device_error()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    ev[0].record(stream)
    for i in range(args.steps):
        gq.expert_dim1(w, out=q, scales=sc, stream=stream, pow2_scales=POW2)
        ev[i + 1].record(stream)
    torch.cuda.synchronize(dev)
    gq.check_device_error()
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(args.steps)]
    total_ms = ev[0].elapsed_time(ev[-1])
    nbytes = 3 * E * K * N + 4 * E * N
    value = nbytes * args.steps / (total_ms * 1e-3) / 1e9
    peak, peak_kind = measured_peaks()
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16->e4m3 (fp32 scale math)", "data": "synthetic (seeded)",
        "config": {"workload": f"expert weights W {E}x{K}x{N} bf16, scales along dim1 "
                               "(per expert and column); columns scaled 10^U(-2,2)",
                   "scales": "rounded down to powers of two" if POW2
                             else "448 / max(amax, 1e-12)",
                   "l2": f"input {2 * E * K * N / 2**20:.0f} MiB larger than L2; no flush"},
        "per_call": {"us_median": statistics.median(per) * 1e3,
                     "timing": "CUDA events on the launching stream around each C-ABI "
                               "call (workspace clear + kernel)"},
        "roofline": {"bound": "hbm", "kernel": "colwise (E groups of K rows)",
                     "achieved": value, "peak": peak, "unit": "GB/s",
                     "frac": value / peak, "peak_kind": peak_kind, "traffic": None,
                     "algorithmic_bytes": nbytes},
        "gpu_launches": args.steps,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_mxfp8(args):
    """Times the mxfp8 dim0 cast on the colwise benchmark input X (65536,
    4096): one call = one step."""
    import numpy as np
    import torch

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    import __graft_entry__

    __graft_entry__.build()
    import fp8_quantization_moe_gb300 as gq
    from fp8_quantization_moe_gb300 import synth

    M, K, G = COLWISE_SHAPE
    c = synth.colwise_large(G, rows=M, cols=K)
    x = torch.from_numpy(c.x.view(np.int16)).view(torch.bfloat16).to(dev)
    q = torch.empty((M, K), dtype=torch.float8_e4m3fn, device=dev)
    sc = torch.empty((M, K // 32), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        gq.mxfp8_dim0(x, args.mxfp8, out=q, scales=sc, stream=stream)
    torch.cuda.synchronize(dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    ev[0].record(stream)
    for i in range(args.steps):
        gq.mxfp8_dim0(x, args.mxfp8, out=q, scales=sc, stream=stream)
        ev[i + 1].record(stream)
    torch.cuda.synchronize(dev)
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(args.steps)]
    total_ms = ev[0].elapsed_time(ev[-1])
    nbytes = 3 * M * K + M * K // 32
    value = nbytes * args.steps / (total_ms * 1e-3) / 1e9
    peak, peak_kind = measured_peaks()
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16->e4m3 + e8m0 block scales", "data": "synthetic (seeded)",
        "config": {"workload": f"mxfp8 dim0 cast ({args.mxfp8.upper()}) of X {M}x{K} bf16, "
                               "32-element row blocks; rows scaled 10^U(-2,2)",
                   "l2": f"input {2 * M * K / 2**20:.0f} MiB larger than L2; no flush"},
        "per_call": {"us_median": statistics.median(per) * 1e3,
                     "timing": "CUDA events on the launching stream around each call"},
        "roofline": {"bound": "hbm", "kernel": "mx_kernel", "achieved": value, "peak": peak,
                     "unit": "GB/s", "frac": value / peak, "peak_kind": peak_kind,
                     "traffic": None,
                     "algorithmic_bytes": nbytes},
        "gpu_launches": args.steps,
    }
    print(json.dumps(line), flush=True)
    return 0


WGRAD_SHAPE = (16640, 8192, 4096, 16)  # tokens T, N, K, groups


def run_wgrad(args):
    """Times the grouped grad_weight GEMM on the tensor cores: T = 16640 tokens
    in 16 groups (the rowwise_t workload's tokens), N = 8192, K = 4096, e4m3
    operands with fp32 scales, bf16 out.  One call = one step."""
    import numpy as np
    import torch

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    import __graft_entry__

    __graft_entry__.build()
    import fp8_quantization_moe_gb300 as gq
    from fp8_quantization_moe_gb300 import synth

    T, N, K, G = (tuple(int(v) for v in args.wgrad_shape.split(",")) if args.wgrad_shape
                  else WGRAD_SHAPE)
    rng = np.random.default_rng(1700)
    offs_np = synth.random_partition(rng, T, G)
    c = synth.wgrad_case(T, N, K, offs_np, seed=1701)
    qa = torch.from_numpy(c.qa_t).to(dev)
    qx = torch.from_numpy(c.qx).to(dev)
    sa = torch.from_numpy(c.sa).to(dev)
    sx = torch.from_numpy(c.sx).to(dev)
    offs = torch.from_numpy(c.offs).to(dev)
    out = torch.empty((G, N, K), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        gq.grouped_wgrad(qa, sa, qx, sx, offs, out=out, stream=stream)
    torch.cuda.synchronize(dev)
    props = torch.cuda.get_device_properties(dev)
    sampler = ClockSampler(f"GPU-{props.uuid}")
    sampler.start()
    time.sleep(0.3)
    sampler.t_load[0] = time.time()
    t_end = time.time() + args.clock_window
    while time.time() < t_end:
        for _ in range(5):
            gq.grouped_wgrad(qa, sa, qx, sx, offs, out=out, stream=stream)
        torch.cuda.synchronize(dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    ev[0].record(stream)
    for i in range(args.steps):
        gq.grouped_wgrad(qa, sa, qx, sx, offs, out=out, stream=stream)
        ev[i + 1].record(stream)
    torch.cuda.synchronize(dev)
    sampler.t_load[1] = time.time()
    sampler.stop()
    gq.check_device_error()
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(args.steps)]
    total_ms = ev[0].elapsed_time(ev[-1])
    flops = 2.0 * N * K * int(offs_np[-1])
    tflops = flops * args.steps / (total_ms * 1e-3) / 1e12
    peak, peak_kind = measured_tensor_peak_fp8()
    out_bytes = G * N * K * 2
    line = {
        "metric": "grouped fp8 grad_weight GEMM throughput (tensor cores)", "value": tflops,
        "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 x e4m3 -> fp32 accumulate -> bf16", "data": "synthetic (seeded e4m3 codes)",
        "config": {"workload": f"grad_weight per token group: T={T} tokens in {G} groups, "
                               f"N={N}, K={K}; out bf16 ({G}, {N}, {K})",
                   "l2": f"output {out_bytes / 2**30:.2f} GiB larger than L2 per call; no flush"},
        "per_call": {"us_median": statistics.median(per) * 1e3,
                     "timing": "CUDA events on the launching stream around each call"},
        "roofline": {"bound": "tensor", "kernel": "wgrad_kernel", "achieved": tflops,
                     "peak": peak, "unit": "TFLOP/s", "frac": tflops / peak,
                     "peak_kind": peak_kind, "traffic": None, "algorithmic_flops": flops,
                     "hbm_floor_us": (out_bytes + T * (N + K)) / (measured_peaks()[0] * 1e3)},
        "clocks": sampler.summary(),
        "gpu_launches": args.steps,
    }
    print(json.dumps(line), flush=True)
    return 0


def _time_calls(fn, steps, flush=None):
    """Median and mean microseconds of `steps` calls of fn, each bracketed by
    CUDA events on the current stream; `flush` (untimed) runs before each.
    Everything is enqueued back to back and synchronised once, so that the
    host's launch latency stays outside the events."""
    import torch

    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    ev = []
    for _ in range(steps):
        if flush is not None:
            flush()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        ev.append((e0, e1))
    torch.cuda.synchronize()
    per = [e0.elapsed_time(e1) * 1e3 for e0, e1 in ev]
    return statistics.median(per), statistics.mean(per)


def per_config_block(dev, steps: int = 20):
    """Every listed workload and group count, and the built NEXT rows, each
    timed on its own: us per call (mean of `steps`, CUDA events around each
    C-ABI call), algorithmic GB/s (2 B read + 1 B written per element + 4 B
    per fp32 scale, 1 B per e8m0 scale) and % of the measured copy peak; the
    grouped grad_weight GEMM as TFLOP/s against the measured bf16 figures
    times the nominal fp8/bf16 ratio.  Inputs that fit L2 (workloads 1 and
    2) get an L2 flush (a 256 MiB write) before each timed call."""
    import numpy as np
    import torch

    import fp8_quantization_moe_gb300 as gq
    from fp8_quantization_moe_gb300 import synth

    peak, _ = measured_peaks()
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def flush():
        flush_buf.zero_()

    def rec(us_med, us_mean, nbytes, **extra):
        # the mean: event timestamps come in steps of about 1 us, which the
        # median keeps and the mean averages out
        gbs = nbytes / (us_mean * 1e-6) / 1e9
        d = {"us": round(us_mean, 2), "us_median": round(us_med, 2), "gbs": round(gbs, 1),
             "pct_peak": round(100 * gbs / peak, 1)}
        d.update(extra)
        return d

    def bf16(bits):
        return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(dev)

    out = {}
    # colwise: workloads 1, 2 (and 2 with every strip two-phase), 3 at 4 / 8 / 16 groups
    for idx, groups in ((1, 4), (2, 16), (3, 4), (3, 8), (3, 16)):
        case = synth.workload(idx, groups)
        M, K = case.x.shape
        x, o = bf16(case.x), torch.from_numpy(case.offs).to(dev)
        q = torch.empty((M, K), dtype=torch.float8_e4m3fn, device=dev)
        sc = torch.empty((groups, K), dtype=torch.float32, device=dev)
        small = 2 * M * K < (64 << 20)
        for two in ((False, True) if idx == 2 else (False,)):
            med, mean = _time_calls(lambda: gq.colwise(x, o, out=q, scales=sc, two_phase=two),
                                    steps, flush if small else None)
            name = f"colwise_{M}x{K}_g{groups}" + ("_two_phase" if two else "")
            out[name] = rec(med, mean, colwise_bytes(M, K, groups),
                            l2="flushed before each call" if small else "input larger than L2")
        del x, q
    torch.cuda.empty_cache()
    # rowwise_t: workload 4 (16 groups), 5 at 1 and 64 groups
    for idx, groups in ((4, 16), (5, 1), (5, 64)):
        case = synth.workload(idx, groups)
        N, Mg = case.x.shape
        a, o = bf16(case.x), torch.from_numpy(case.offs).to(dev)
        qt = torch.empty((Mg, N), dtype=torch.float8_e4m3fn, device=dev)
        sc = torch.empty((N, groups), dtype=torch.float32, device=dev)
        med, mean = _time_calls(lambda: gq.rowwise_t(a, o, out=qt, scales=sc), steps)
        out[f"rowwise_t_{N}x{Mg}_g{groups}"] = rec(med, mean, rowwise_bytes(N, Mg, groups),
                                                   l2="input larger than L2")
        del a, qt
    torch.cuda.empty_cache()
    # mxfp8 dim0 on workload 3's X
    case = synth.workload(3, 16)
    M, K = case.x.shape
    x = bf16(case.x)
    q = torch.empty((M, K), dtype=torch.float8_e4m3fn, device=dev)
    sm = torch.empty((M, K // 32), dtype=torch.uint8, device=dev)
    for mode in ("floor", "rceil"):
        med, mean = _time_calls(lambda: gq.mxfp8_dim0(x, mode, out=q, scales=sm), steps)
        out[f"mxfp8_{mode}_{M}x{K}"] = rec(med, mean, 3 * M * K + M * K // 32,
                                          l2="input larger than L2")
    del x, q, sm
    # stacked expert weights along dim1
    E, Ke, Ne = EXPERT_SHAPE
    rng = np.random.default_rng(1700)
    w = rng.standard_normal((E, Ke, Ne), dtype=np.float32)
    w *= np.power(np.float32(10), rng.uniform(-2, 2, size=(E, 1, Ne))).astype(np.float32)
    wd = bf16(synth.to_bf16_bits(w))
    del w
    qe = torch.empty((E, Ke, Ne), dtype=torch.float8_e4m3fn, device=dev)
    se = torch.empty((E, Ne), dtype=torch.float32, device=dev)
    med, mean = _time_calls(lambda: gq.expert_dim1(wd, out=qe, scales=se), steps)
    out[f"expert_dim1_{E}x{Ke}x{Ne}"] = rec(med, mean, 3 * E * Ke * Ne + 4 * E * Ne,
                                            l2="input larger than L2")
    # the same weights read as (E, N, K) and scaled per (expert, row)
    sr = torch.empty((E, Ke), dtype=torch.float32, device=dev)
    med, mean = _time_calls(lambda: gq.expert_rowwise(wd, out=qe, scales=sr), steps)
    out[f"expert_rowwise_{E}x{Ke}x{Ne}"] = rec(med, mean, 3 * E * Ke * Ne + 4 * E * Ke,
                                               l2="input larger than L2")
    del wd, qe, sr
    torch.cuda.empty_cache()
    # the grouped grad_weight GEMM
    T, N, K, G = WGRAD_SHAPE
    rng = np.random.default_rng(1700)
    c = synth.wgrad_case(T, N, K, synth.random_partition(rng, T, G), seed=1701)
    d = lambda v: torch.from_numpy(v).to(dev)
    qa, sa, qx, sx, offs = d(c.qa_t), d(c.sa), d(c.qx), d(c.sx), d(c.offs)
    og = torch.empty((G, N, K), dtype=torch.bfloat16, device=dev)
    med, mean = _time_calls(lambda: gq.grouped_wgrad(qa, sa, qx, sx, offs, out=og), 10)
    flops = 2.0 * N * K * T
    tf = flops / (mean * 1e-6) / 1e12
    sus, _ = measured_tensor_peak_fp8()
    burst = 2.0 * measured_bf16_burst()
    out[f"grouped_wgrad_T{T}_N{N}_K{K}_g{G}"] = {
        "us": round(mean, 1), "us_median": round(med, 1), "tflops": round(tf, 1),
        "frac_of_sustained_fp8": round(tf / sus, 3), "frac_of_burst_fp8": round(tf / burst, 3),
        "peak_note": "fp8 = measured bf16 x 2 (nominal fp8/bf16 ratio)"}
    del qa, qx, og
    torch.cuda.empty_cache()
    gq.check_device_error()
    return out


def measured_bf16_burst():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["bf16_tflops"])
    except (OSError, KeyError, ValueError):
        return 1900.0


def measured_tensor_peak_fp8():
    """fp8 dense peak for a kernel timed inside a sustained run (the timed
    calls follow seconds of the same load, under the power cap): the measured
    sustained cuBLAS bf16 figure times the nominal fp8 / bf16 ratio (4.5 /
    2.25 PFLOP/s), else the fallback sustained bf16 figure times that ratio."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return (2.0 * float(json.load(f)["bf16_tflops_sustained"]),
                    "measured sustained bf16 x 2 (nominal fp8/bf16)")
    except (OSError, KeyError, ValueError):
        return 2.0 * 1700.0, "fallback sustained bf16 x 2 (nominal fp8/bf16)"


def run_only(args):
    """Times one kernel alone on its benchmark workload, launched back to
    back on the stream (--only colwise | rowwise_t), the outputs alternating
    between two buffers.  For profiling: in the middle of such a run, the
    output lines a launch leaves dirty in L2 are written back during the
    next, which leaves as many of its own behind (to other addresses, so
    none is merged with a later write), and one launch's DRAM counters count
    one output."""
    import numpy as np
    import torch

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    import __graft_entry__

    __graft_entry__.build()
    import fp8_quantization_moe_gb300 as gq
    from fp8_quantization_moe_gb300 import synth

    if args.rowwise_no_split:
        gq.debug_set(no_split=True)
    if args.only == "colwise":
        M, K, G = COLWISE_SHAPE
        G = args.only_groups or G
        case = synth.colwise_large(G, rows=M, cols=K)
        nbytes = colwise_bytes(M, K, G)
        x = torch.from_numpy(case.x.view(np.int16)).view(torch.bfloat16).to(dev)
        o = torch.from_numpy(case.offs).to(dev)
        qs = [torch.empty((M, K), dtype=torch.float8_e4m3fn, device=dev) for _ in range(2)]
        ss = [torch.empty((G, K), dtype=torch.float32, device=dev) for _ in range(2)]
        call = lambda i: gq.colwise(x, o, out=qs[i % 2], scales=ss[i % 2], pow2_scales=POW2)
        workload = f"colwise X {M}x{K} bf16, {G} groups"
    else:
        N, Mg, G = ROWWISE_SHAPE
        G = args.only_groups or G
        case = (synth.rowwise_g16() if G == 16 and (N, Mg) == (8192, 16640)
                else synth.rowwise_outliers(G, N=N, Mg=Mg))
        nbytes = rowwise_bytes(N, Mg, G)
        a = torch.from_numpy(case.x.view(np.int16)).view(torch.bfloat16).to(dev)
        o = torch.from_numpy(case.offs).to(dev)
        qs = [torch.empty((Mg, N), dtype=torch.float8_e4m3fn, device=dev) for _ in range(2)]
        ss = [torch.empty((N, G), dtype=torch.float32, device=dev) for _ in range(2)]
        call = lambda i: gq.rowwise_t(a, o, out=qs[i % 2], scales=ss[i % 2], pow2_scales=POW2)
        workload = f"rowwise_t A {N}x{Mg} bf16, {G} groups"
    for i in range(args.warmup):
        call(i)
    torch.cuda.synchronize(dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    ev[0].record()
    for i in range(args.steps):
        call(args.warmup + i)
        ev[i + 1].record()
    torch.cuda.synchronize(dev)
    gq.check_device_error()
    per = [ev[i].elapsed_time(ev[i + 1]) * 1e3 for i in range(args.steps)]
    peak, peak_kind = measured_peaks()
    us = ev[0].elapsed_time(ev[args.steps]) * 1e3 / args.steps
    print(json.dumps({"only": args.only, "workload": workload, "us_mean": us,
                      "us_median": statistics.median(per),
                      "gbs": nbytes / (us * 1e-6) / 1e9,
                      "frac": nbytes / (us * 1e-6) / 1e9 / peak, "peak_kind": peak_kind,
                      "steps": args.steps, "warmup": args.warmup,
                      "gpu_launches": args.steps}), flush=True)
    return 0


def run_mine(args):
    import numpy as np
    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist_ok = world > 1
    if dist_ok:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)

    import __graft_entry__

    __graft_entry__.build()
    import fp8_quantization_moe_gb300 as gq
    from fp8_quantization_moe_gb300 import synth

    M, K, G = COLWISE_SHAPE
    N, Mg, Gr = ROWWISE_SHAPE
    seed_off = 7919 * rank  # each rank its own batch
    c = synth.colwise_large(G, seed=1300 + G + seed_off, rows=M, cols=K)
    r = synth.rowwise_outliers(Gr, seed=1500 + Gr + seed_off, N=N, Mg=Mg)

    def to_dev(bits):
        return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(dev)

    x, a = to_dev(c.x), to_dev(r.x)
    xo = torch.from_numpy(c.offs).to(dev)
    ao = torch.from_numpy(r.offs).to(dev)
    q = torch.empty((M, K), dtype=torch.float8_e4m3fn, device=dev)
    qs = torch.empty((G, K), dtype=torch.float32, device=dev)
    qt = torch.empty((Mg, N), dtype=torch.float8_e4m3fn, device=dev)
    ts = torch.empty((N, Gr), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        gq.colwise(x, xo, out=q, scales=qs, stream=stream, pow2_scales=POW2)
        gq.rowwise_t(a, ao, out=qt, scales=ts, stream=stream, pow2_scales=POW2)

    props = torch.cuda.get_device_properties(dev)
    sampler = ClockSampler(f"GPU-{props.uuid}")
    sampler.start()
    time.sleep(0.3)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    gq.check_device_error()

    # sustained load around the timed region, for the clock samples
    sampler.t_load[0] = time.time()
    t_end = time.time() + args.clock_window
    while time.time() < t_end:
        for _ in range(20):
            step()
        torch.cuda.synchronize(dev)

    if dist_ok:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)]
          for _ in range(args.steps)]
    for i in range(args.steps):
        ev[i][0].record(stream)
        gq.colwise(x, xo, out=q, scales=qs, stream=stream, pow2_scales=POW2)
        ev[i][1].record(stream)
        gq.rowwise_t(a, ao, out=qt, scales=ts, stream=stream, pow2_scales=POW2)
        ev[i][2].record(stream)
    torch.cuda.synchronize(dev)
    stream_col = [ev[i][0].elapsed_time(ev[i][1]) for i in range(args.steps)]
    stream_row = [ev[i][1].elapsed_time(ev[i][2]) for i in range(args.steps)]
    stream_ms = ev[0][0].elapsed_time(ev[-1][2])

    # The step captured once into a CUDA graph and replayed: the library's
    # host work (checks, tensor-map encoding) runs at capture, every replay
    # does the full device work of both calls.
    graph = not args.no_graph
    if graph:
        gs = torch.cuda.Stream(dev)
        with torch.cuda.stream(gs):
            gq.colwise(x, xo, out=q, scales=qs, stream=gs, pow2_scales=POW2)
            gq.rowwise_t(a, ao, out=qt, scales=ts, stream=gs, pow2_scales=POW2)
        torch.cuda.synchronize(dev)
        g_step = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_step, stream=gs):
            gq.colwise(x, xo, out=q, scales=qs, stream=gs, pow2_scales=POW2)
            gq.rowwise_t(a, ao, out=qt, scales=ts, stream=gs, pow2_scales=POW2)
        torch.cuda.synchronize(dev)
        gev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
        with torch.cuda.stream(gs):
            for _ in range(args.warmup):
                g_step.replay()
            torch.cuda.synchronize(dev)
            if dist_ok:
                torch.distributed.barrier()
            torch.cuda.synchronize(dev)
            gev[0].record(gs)
            for i in range(args.steps):
                g_step.replay()
                gev[i + 1].record(gs)
        torch.cuda.synchronize(dev)
    if dist_ok:
        torch.distributed.barrier()
    sampler.t_load[1] = time.time()
    time.sleep(0.25)
    sampler.stop()
    gq.check_device_error()

    # per-call times (and the kernels' rooflines) from the stream launches
    col_ms, row_ms = stream_col, stream_row
    total_ms = gev[0].elapsed_time(gev[-1]) if graph else stream_ms
    nbytes = step_bytes() * args.steps
    max_ms, all_bytes = reduce_over_ranks(total_ms, nbytes, dist_ok)
    value = all_bytes / (max_ms * 1e-3) / 1e9
    smax_ms, _ = reduce_over_ranks(stream_ms, nbytes, dist_ok)

    # end to end through the host-buffer API: H2D inputs, kernels, D2H outputs
    xh = torch.from_numpy(c.x.view(np.int16)).view(torch.bfloat16).pin_memory()
    ah = torch.from_numpy(r.x.view(np.int16)).view(torch.bfloat16).pin_memory()
    xoh = torch.from_numpy(c.offs).pin_memory()
    aoh = torch.from_numpy(r.offs).pin_memory()
    qh = torch.empty((M, K), dtype=torch.float8_e4m3fn, pin_memory=True)
    qsh = torch.empty((G, K), dtype=torch.float32, pin_memory=True)
    qth = torch.empty((Mg, N), dtype=torch.float8_e4m3fn, pin_memory=True)
    tsh = torch.empty((N, Gr), dtype=torch.float32, pin_memory=True)

    def e2e_step():
        gq.colwise_host(xh, xoh, qh, qsh, device=dev, stream=stream, pow2_scales=POW2)
        gq.rowwise_t_host(ah, aoh, qth, tsh, device=dev, stream=stream, pow2_scales=POW2)

    e2e_step()
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1)
    e2e_max, e2e_bytes = reduce_over_ranks(e2e_ms, step_bytes() * args.e2e_steps,
                                           dist_ok)
    h2d = (c.x.nbytes + r.x.nbytes + c.offs.nbytes + r.offs.nbytes)
    d2h = (M * K + G * K * 4 + Mg * N + N * Gr * 4)

    peak, peak_kind = measured_peaks()
    col_b = colwise_bytes(M, K, G)
    row_b = rowwise_bytes(N, Mg, Gr)
    col_avg = statistics.mean(col_ms)
    row_avg = statistics.mean(row_ms)
    col_gbs = col_b / (col_avg * 1e-3) / 1e9
    row_gbs = row_b / (row_avg * 1e-3) / 1e9
    tr = traffic_record("colwise")
    tr_row = traffic_record("rowwise_t")

    if rank != 0:
        if dist_ok:
            torch.distributed.destroy_process_group()
        return 0

    per_config = None
    if world == 1 and not args.no_per_config:
        per_config = per_config_block(dev)

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        gbs, secs, sample = oracle_sample_gbs()
        import oracle
        pgbs, pthreads, psample = oracle_parallel_gbs()
        cpu = {"value": gbs, "unit": UNIT, "cores": oracle.threads_used(),
               "kind": "oracle", "sample": sample,
               "all_cores": {"value": pgbs, "unit": UNIT, "cores": pthreads,
                             "sample": psample}}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": max_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16->e4m3 (fp32 scale math)", "data": "synthetic (seeded)",
        "config": {
            "workload": f"colwise X {M}x{K} bf16, {G} groups (rows scaled "
                        f"10^U(-2,2)) + rowwise_t A {N}x{Mg} bf16, {Gr} groups "
                        "(2 empty, 0.5% outlier columns x1000)",
            "global_batch": M + Mg, "parallelism": f"replicas x{world}",
            "scales": "rounded down to powers of two" if POW2 else "448 / max(amax, 1e-12)",
            "l2": f"inputs ({2 * M * K / 2**20:.0f} MiB, {2 * N * Mg / 2**20:.0f} MiB) larger "
                  "than L2 and disjoint; no flush",
            "launch": ("the step (both calls) captured once into a CUDA graph, "
                       "replayed per step" if graph else "stream launches"),
        },
        "per_call": {
            "colwise_us": col_avg * 1e3, "colwise_gbs": col_gbs,
            "colwise_pct_peak": 100 * col_gbs / peak,
            "rowwise_t_us": row_avg * 1e3, "rowwise_t_gbs": row_gbs,
            "rowwise_t_pct_peak": 100 * row_gbs / peak,
            "timing": "CUDA events on the launching stream around each C-ABI "
                      "call launched on the stream (workspace clear + kernel)",
        },
        "stream_launch": {
            "value": all_bytes / (smax_ms * 1e-3) / 1e9, "unit": UNIT,
            "colwise_us": statistics.mean(stream_col) * 1e3,
            "rowwise_t_us": statistics.mean(stream_row) * 1e3,
            "note": "the same steps launched on the stream (no graph)",
        },
        "roofline": {
            "bound": "hbm", "kernel": "colwise", "achieved": col_gbs,
            "peak": peak, "unit": "GB/s", "frac": col_gbs / peak,
            "peak_kind": f"{peak_kind} copy bandwidth (hbm_gbs)",
            "traffic": (tr["dram_bytes_per_launch"] if tr else None),
            "algorithmic_bytes": col_b,
        },
        "roofline_rowwise_t": {
            "bound": "hbm", "kernel": "rowwise_t", "achieved": row_gbs,
            "peak": peak, "unit": "GB/s", "frac": row_gbs / peak,
            "traffic": (tr_row["dram_bytes_per_launch"] if tr_row else None),
            "algorithmic_bytes": row_b,
        },
        "per_config": per_config,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_bytes / (e2e_max * 1e-3) / 1e9, "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": args.e2e_steps,
                "path": "colwise_host + rowwise_t_host (pinned host buffers)"},
        "gpu_launches": 2 * args.steps,
        "clocks": sampler.summary(),
        "pages_context": PAGES_CONTEXT,
        "gpu": props.name,
    }
    print(json.dumps(line), flush=True)
    if dist_ok:
        torch.distributed.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["mine", "reference"], default="mine")
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--clock-window", type=float, default=1.5,
                    help="seconds of sustained load around the timed region")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per-configuration block (every workload and group "
                         "count, mxfp8, expert dim1 and the grouped GEMM, each timed alone)")
    ap.add_argument("--pow2-scales", action="store_true",
                    help="round every scale down to a power of two (the "
                         "round_scales_to_power_of_2 option); same bytes moved")
    ap.add_argument("--expert-dim1", action="store_true",
                    help="time the stacked expert-weight path (8 experts of "
                         "4096x4096, scales along dim1) instead of the main step")
    ap.add_argument("--mxfp8", choices=["floor", "rceil"], default=None,
                    help="time the mxfp8 dim0 cast of the colwise input instead "
                         "of the main step")
    ap.add_argument("--wgrad", action="store_true",
                    help="time the grouped fp8 grad_weight GEMM instead of the main step")
    ap.add_argument("--wgrad-shape", default=None,
                    help="T,N,K,groups for --wgrad (a smaller case for profiling)")
    ap.add_argument("--only", choices=["colwise", "rowwise_t"], default=None,
                    help="time one kernel alone on its benchmark workload, launched "
                         "back to back (for profiling)")
    ap.add_argument("--only-groups", type=int, default=0,
                    help="with --only: the workload's group count (default: the benchmark's)")
    ap.add_argument("--rowwise-no-split", action="store_true",
                    help="with --only rowwise_t: never split units across blocks "
                         "(the gq_debug_set flag), to compare the two paths")
    ap.add_argument("--no-graph", action="store_true",
                    help="time stream launches only (default: the step's two calls "
                         "replayed from CUDA graphs, stream launches reported beside)")
    ap.add_argument("--half", action="store_true",
                    help="profiling case: half the tokens of each workload "
                         "(inputs 256 MB and 136 MB, still larger than L2); "
                         "not the benchmark configuration")
    args = ap.parse_args(argv)
    global POW2
    POW2 = bool(args.pow2_scales)
    if args.half:
        global COLWISE_SHAPE, ROWWISE_SHAPE
        COLWISE_SHAPE = (COLWISE_SHAPE[0] // 2,) + COLWISE_SHAPE[1:]
        ROWWISE_SHAPE = (ROWWISE_SHAPE[0], ROWWISE_SHAPE[1] // 2, ROWWISE_SHAPE[2])
    if args.warmup < 3:
        args.warmup = 3  # timing rule: at least three warm-up steps
    if args.impl == "reference":
        return run_reference(args)
    if args.expert_dim1:
        return run_expert(args)
    if args.mxfp8:
        return run_mxfp8(args)
    if args.wgrad:
        return run_wgrad(args)
    if args.only:
        return run_only(args)
    return run_mine(args)


if __name__ == "__main__":
    sys.exit(main())
