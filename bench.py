#!/usr/bin/env python3
"""Benchmark of the Q4_G64_FP16 linear layer on one GB300 (or N replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--samples S] [--impl ours|reference]
                    [--workload NAME] [--t T] [--qtype FMT] [--route R] [--op OP] [--profile]
    python bench.py --workload q4_6144x5120 --sweep 1:128:1,384,385,512,640,641,1024 [--csv-out F]

A step is one call of the layer on one batch of the workload's synthetic input.
With no --workload the run times three records of the 6144 x 5120 layer: the
decode GEMV at T = 1 (the headline), T = 8 (the small-T route) and T = 1024 (the
large-T tile route); otherwise one record of the named workload.

Timing of a record: W untimed warm-up calls, then S samples (at least 50).  A
sample is exactly K back-to-back calls captured in one CUDA graph (call i on
rotating copy i mod R of the weights, X and Y, R copies larger than 2.5 x L2 in
total, so every call streams from HBM), queued right after a 256 MiB L2 flush
(the buffer is written, then read back so no dirty line is written back inside
the sample), with CUDA events on the launching stream around the graph launch.
ms_per_step = median sample / K; value = the metric at that time; min and p95
are reported too.  The linear-benchmark contract's own method (section 6: one
call per sample behind the flush, median) is reported as cold_call.  Metrics
follow the contract's sections 4-5 (weight_only_bit_q4_gb300.metrics).

--sweep times a contiguous T range (and single T values) of one workload under the
contract's cold-cache method only (section 6: per T, the first call untimed, 3 warm-up
calls, then 20 samples of one public call behind a 256 MiB flush; median, min, p95), and
prints the contract's console header and one line per T (section 7) with the change of the
median against the previous T (delta_%), optionally to a CSV file as well.

The first record also carries e2e: the step with X and Y in pinned host memory through
q4lin_linear_host (the library stages X in and the layer stores Y into the pinned
buffer), one CUDA graph replay per step, median of 200; the same step with
cudaMemcpyAsync copies around the device-buffer call (memcpy_us) and issued eagerly from
Python (eager_us) is reported beside it.

--qtype times a sibling weight format (Q5G64, Q6G64, W8G32) on the same geometry
through q4lin_linear_qtype; its bytes are that format's.  --op times a fused operation
(LinearAdd, LinearSwiGLU, LinearPair).  Under torchrun (N > 1)
every rank runs an independent replica on its own GPU (the layer does not exchange
data between GPUs); value = the units all ranks processed / the slowest rank's time.
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

from weight_only_bit_q4_gb300 import metrics, synth  # noqa: E402

METRIC = "Q4 linear µs + logical GB/s (small T) / eff. TFLOP/s (large T) vs GB300 roofline"
FLUSH_BYTES = 256 << 20

# name -> (N, K, T, scale distribution, outlier channels, weight seed, x seed)
WORKLOADS = {
    "q4_512x1024_t8": (512, 1024, 8, "halfnormal", False, 0, 0),
    "q4_6144x5120_t1": (6144, 5120, 1, "halfnormal", False, 0, 0),
    "q4_6144x5120": (6144, 5120, None, "halfnormal", False, 0, None),       # --t, X seed = T
    "q4_14336x5120": (14336, 5120, None, "lognormal", True, 0, None),       # --t in {1,16,128,1024}
    "q4_34816x5120_t1024": (34816, 5120, 1024, "halfnormal", False, 0, 0),
    "q4_5120x17408_t1024": (5120, 17408, 1024, "halfnormal", False, 0, 0),
    "q4_34816x5120": (34816, 5120, None, "halfnormal", False, 0, None),      # --t (profiling long weights)
    "q4_5120x17408": (5120, 17408, None, "halfnormal", False, 0, None),      # --t (profiling deep K)
    # the suites' other Q4 geometries: draft heads (T class 1, 16, 128, 1024) and
    # vision projections (T class 4, 128, 1024)
    "q4_131072x5120": (131072, 5120, None, "halfnormal", False, 0, None),
    "q4_131072x2048": (131072, 2048, None, "halfnormal", False, 0, None),
    "q4_3456x1152": (3456, 1152, None, "halfnormal", False, 0, None),
    "q4_4304x1152": (4304, 1152, None, "halfnormal", False, 0, None),
}
DEFAULT_WORKLOAD = "q4_6144x5120_t1"


# the records of the default run: the decode GEMV headline, then the small-T and the
# large-T routes on the same 6144 x 5120 weight
DEFAULT_RECORDS = (("q4_6144x5120_t1", None), ("q4_6144x5120", 8), ("q4_6144x5120", 1024))
MIN_SAMPLES = 50


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20, help="calls per timed sample (K)")
    p.add_argument("--warmup", type=int, default=10, help="untimed warm-up calls per record (W >= 3)")
    p.add_argument("--samples", type=int, default=MIN_SAMPLES, help=f"timed samples per record (>= {MIN_SAMPLES})")
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=None, choices=sorted(WORKLOADS),
                   help=f"time this workload alone (default: the three records of {DEFAULT_WORKLOAD} at T = 1, 8, 1024)")
    p.add_argument("--t", type=int, default=None, help="T for the sweep workloads")
    p.add_argument("--qtype", default="q4g64", choices=sorted(metrics.GROUP_BYTES),
                   help="weight format (the sibling formats run for 1..4 tokens)")
    p.add_argument("--op", default="linear", choices=["linear", "add", "swiglu", "pair"],
                   help="linear: Y = W.X; add: LinearAdd, Y = W.X + R; swiglu: LinearSwiGLU on the workload's "
                        "weight as a gate/up pair (F = N / 2); pair: LinearPair, two weights of the workload's "
                        "shape on one X (the fused forms run the exact tile route for every T)")
    p.add_argument("--route", default="auto", choices=["auto", "tc_fp16", "gemv", "stream_mma", "tc_splitk"],
                   help="auto: the library's choice; tc_fp16: the opt-in tile route on fp16-rounded weights; "
                        "the others force that route (q4lin_linear_route)")
    p.add_argument("--profile", action="store_true",
                   help="one call between cudaProfilerStart/Stop after warm-up and flush (for ncu --profile-from-start off)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-probe", action="store_true", help="skip the HBM read probe")
    p.add_argument("--sweep", default=None,
                   help="T values of one workload: comma-separated A:B:S ranges and single values "
                        "(cold-cache per-call timing, one line per T with delta_%%)")
    p.add_argument("--repeat", type=int, default=20, help="--sweep: timed samples per T")
    p.add_argument("--csv-out", default=None, help="--sweep: also write the lines to this CSV file")
    a = p.parse_args(argv)
    a.warmup = max(a.warmup, 3)
    a.steps = max(a.steps, 1)
    a.samples = max(a.samples, MIN_SAMPLES)
    return a


def record_specs(args):
    """(workload name, T) of every record this run times; the first is the headline."""
    single = (args.workload is not None or args.qtype != "q4g64" or args.route != "auto" or args.op != "linear"
              or args.t is not None)
    if single:
        return [(args.workload or DEFAULT_WORKLOAD, args.t)]
    return list(DEFAULT_RECORDS)


def workload(args, name=None, t=None):
    name = name if name is not None else (args.workload or DEFAULT_WORKLOAD)
    t = t if t is not None else args.t
    N, K, T, dist, outl, ws, xs = WORKLOADS[name]
    if T is None:
        T = t if t is not None else 1
    elif t is not None and t != T:
        raise SystemExit(f"workload {name} has fixed T={T}")
    if xs is None:
        xs = T
    wname = name if WORKLOADS[name][2] is not None else f"{name}_t{T}"
    qtype = getattr(args, "qtype", "q4g64")
    if qtype != "q4g64":
        wname = qtype + wname[2:]            # q4_6144x5120_t1 -> q5g64_6144x5120_t1
    route = getattr(args, "route", "auto")
    if route != "auto":
        if qtype != "q4g64":
            raise SystemExit(f"--route {route} runs the Q4 format only")
        wname += "_" + route
    op = getattr(args, "op", "linear")
    if op != "linear":
        if qtype != "q4g64" or route != "auto":
            raise SystemExit(f"--op {op} runs the Q4 format on its own route")
        if op == "swiglu" and N % 2:
            raise SystemExit("--op swiglu needs an even number of weight rows")
        wname += "_" + op
    return dict(name=wname, N=N, K=K, T=T, dist=dist, outliers=outl, w_seed=ws, x_seed=xs, qtype=qtype, op=op,
                route=route)


def op_bytes(wl):
    """Logical bytes of one call: the layer's model bytes; LinearAdd reads the residual too,
    LinearSwiGLU writes F = N / 2 outputs per token, LinearPair reads two weights and writes
    two outputs."""
    N, K, T = wl["N"], wl["K"], wl["T"]
    op = wl.get("op")
    if op == "swiglu":
        return metrics.model_bytes(N, K, T, wl["qtype"]) - 2 * N * T + 2 * (N // 2) * T
    if op == "pair":
        return 2 * metrics.model_bytes(N, K, T, wl["qtype"]) - 2 * K * T
    return metrics.model_bytes(N, K, T, wl["qtype"]) + (2 * N * T if op == "add" else 0)


def op_flops(wl):
    """Useful FLOPs of one call (LinearPair: both weights)."""
    f = metrics.useful_flops(wl["N"], wl["K"], wl["T"])
    return 2 * f if wl.get("op") == "pair" else f


def format_problem(wl, rows=None):
    """(planes, scales, x) of a sibling-format workload (its first ``rows`` rows)."""
    planes, sc, x = synth.make_problem_fmt(wl["qtype"], wl["N"], wl["K"], wl["T"],
                                           w_seed=wl["w_seed"], x_seed=wl["x_seed"])
    if rows is not None:
        planes, sc = tuple(p[:rows] for p in planes), sc[:rows]
    return planes, sc, x


def small_t(wl):
    # HBM-bound below the ridge (~280 FLOP/B at 6.8 TB/s and 1.9 PF/s): T <~ 75
    return wl["T"] <= 64


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured")
    except (OSError, KeyError, ValueError):
        return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_max(values, world, device=None):
    """Elementwise max over ranks of a list of floats (identity when world == 1)."""
    if world == 1:
        return list(values)
    import torch
    import torch.distributed as dist
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms in the background;
    summary() reports the samples inside one window of time.monotonic()."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self._reader = threading.Thread(target=self._read, daemon=True)
        self._reader.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def stop(self):
        if self.proc is None:
            return
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()

    def summary(self, t0, t1):
        rows = [l for (t, l) in self.lines if t0 <= t <= t1 + 0.1]
        if not rows:   # a window shorter than the sampling period: the samples around it
            near = sorted(self.lines, key=lambda e: abs(e[0] - 0.5 * (t0 + t1)))[:2]
            rows = [l for (_, l) in near]
        sm, mx, reasons = [], [], set()
        for r in rows:
            f = [x.strip() for x in r.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"), f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- traffic record
def kernel_source_digest(source: str = "q4_gemv.cu"):
    """Digest of one kernel's translation unit: its .cu file and the device-code headers
    (.cuh).  The .h headers hold host declarations only and are left out."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "weight_only_bit_q4_gb300", "csrc")
    for f in [source] + sorted(f for f in os.listdir(csrc) if f.endswith(".cuh")):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + b"\0" + fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(wl_name):
    """DRAM bytes per launch from the committed ncu summary, if taken on the current kernels."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d.get(wl_name)
        if e and e.get("src_digest") == kernel_source_digest(e.get("source", "q4_gemv.cu")):
            return float(e["dram_bytes_per_launch"]), e.get("kernel")
    except (OSError, ValueError, KeyError):
        pass
    return None, None


# ----------------------------------------------------------------------------- our arm
def measure_ours(args, wl, rank, world, local, sampler=None, with_e2e=True):
    """Times one record of the layer on this rank's GPU.

    R copies of the weight planes, X and Y (R * logical bytes >= 2.5 x L2) rotate
    call by call.  One CUDA graph holds K = args.steps back-to-back calls (call i on
    copy i mod R); a sample is a 256 MiB write+read L2 flush, then the graph launch
    bracketed by CUDA events on the launching stream; S = args.samples samples, all
    queued without host synchronisation.  Reported per sample: its time / K.

    Cold single call (the linear-benchmark contract's method, reported beside it):
    the flush, then events around one graph launch of one call; median / min / p95.
    """
    import numpy as np
    import torch
    from weight_only_bit_q4_gb300 import build, q4lin

    build.build()
    q4lin.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    N, K, T = wl["N"], wl["K"], wl["T"]
    qtype = wl["qtype"]
    if qtype == "q4g64":
        planes = (synth.packed_codes(N, K, wl["w_seed"]),)
        sc = synth.group_scales(N, K, wl["w_seed"], wl["dist"])
        x = synth.activations(T, K, wl["x_seed"], wl["outliers"])
    else:
        planes, sc, x = format_problem(wl)
    per_copy = op_bytes(wl)
    op = wl.get("op", "linear")
    add = op == "add"
    r = synth.activations(T, N, wl["x_seed"] + 7919) if add else None   # LinearAdd's bf16 residual [T, N]
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size or (128 << 20)
    R = int(max(2, min(64, -(-int(2.5 * l2) // per_copy))))
    pl_d = tuple(torch.from_numpy(p).to(dev) for p in planes)
    sc_d = torch.from_numpy(sc.view(np.int16)).to(dev)
    x_d = torch.from_numpy(x.view(np.int16)).to(dev).view(torch.bfloat16)
    pls = [pl_d] + [tuple(p.clone() for p in pl_d) for _ in range(R - 1)]
    scs = [sc_d] + [sc_d.clone() for _ in range(R - 1)]
    xs = [x_d] + [x_d.clone() for _ in range(R - 1)]
    n_out = N // 2 if op == "swiglu" else N
    ys = [torch.empty((T, n_out), dtype=torch.bfloat16, device=dev) for _ in range(R)]
    if op == "pair":   # the second weight (seed + 1) and its outputs
        pl_b = torch.from_numpy(synth.packed_codes(N, K, wl["w_seed"] + 1)).to(dev)
        sc_b = torch.from_numpy(synth.group_scales(N, K, wl["w_seed"] + 1, wl["dist"]).view(np.int16)).to(dev)
        pls_b = [pl_b] + [pl_b.clone() for _ in range(R - 1)]
        scs_b = [sc_b] + [sc_b.clone() for _ in range(R - 1)]
        ys_b = [torch.empty((T, N), dtype=torch.bfloat16, device=dev) for _ in range(R)]
    rs = [torch.from_numpy(r.view(np.int16)).to(dev).view(torch.bfloat16) for _ in range(R)] if add else None
    route_arg = {"tc_fp16": q4lin.ROUTE_TC_FP16, "gemv": q4lin.ROUTE_GEMV, "stream_mma": q4lin.ROUTE_STREAM_MMA,
                 "tc_splitk": q4lin.ROUTE_TC_SPLITK}.get(wl.get("route"), q4lin.ROUTE_AUTO)
    ws_n = q4lin.workspace_bytes(N, K, T, route_arg)
    ws_d = torch.empty(max(ws_n, 256), dtype=torch.uint8, device=dev)
    route = q4lin.select_route(N, K, T) if route_arg == q4lin.ROUTE_AUTO else route_arg
    launches = q4lin.kernel_launches(N, K, T)
    if route_arg == q4lin.ROUTE_TC_FP16:   # operand pass + main launch (+ tail launch)
        pl = q4lin.tile_plan_full(N, K, T, route_arg)
        launches = 1 + (2 if pl["main_tiles"] < -(-N // 128) * -(-T // pl["n"]) else 1)
    elif route_arg == q4lin.ROUTE_STREAM_MMA:   # operand pass + streaming kernel, per 32 tokens
        launches = 2 * -(-T // 32)
    elif route_arg == q4lin.ROUTE_TC_SPLITK:
        pl = q4lin.tile_plan_full(N, K, T, route_arg)
        launches = 2 if pl["main_tiles"] < -(-N // 128) * -(-T // pl["n"]) else 1
    elif route_arg == q4lin.ROUTE_GEMV:
        launches = 1 if T <= 4 else -(-T // 4)
    stream = torch.cuda.Stream(dev)

    if qtype != "q4g64":   # the library's own choice for the format (GEMV, warp-MMA or tile route)
        launches = q4lin.kernel_launches(N, K, T, qtype)
        route = q4lin.qtype_route(qtype, N, K, T)

    if op != "linear" and q4lin.fused_route(op, n_out, K, T) == q4lin.ROUTE_STREAM_MMA:
        # a few tokens: the warp-MMA route's one-launch form, one launch per weight
        route = q4lin.ROUTE_STREAM_MMA
        launches = 2 if op == "pair" else 1
    elif op != "linear":   # the exact tile route: one launch, or two with a tail launch
        n_plan = 128 * 2 * -(-N // 128) if op == "pair" else N
        pl = q4lin.tile_plan_full(n_plan, K, T, q4lin.ROUTE_TC_SPLITK)
        route = q4lin.ROUTE_TC_SPLITK
        launches = 2 if pl["main_tiles"] < -(-n_plan // 128) * -(-T // pl["n"]) else 1

    def call(i):
        i %= R
        if add:
            q4lin.linear_add(pls[i][0], scs[i], xs[i], rs[i], y=ys[i], stream=stream)
        elif op == "swiglu":
            q4lin.linear_swiglu(pls[i][0], scs[i], xs[i], y=ys[i], stream=stream)
        elif op == "pair":
            q4lin.linear_pair(pls[i][0], scs[i], pls_b[i], scs_b[i], xs[i], y_a=ys[i], y_b=ys_b[i], stream=stream)
        elif qtype == "q4g64":
            q4lin.linear(pls[i][0], scs[i], xs[i], y=ys[i], workspace=ws_d if ws_n else None, stream=stream,
                         route=route_arg)
        else:
            q4lin.linear_qtype(qtype, pls[i], scs[i], xs[i], y=ys[i], stream=stream)

    K_steps, S = args.steps, args.samples
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    sink = torch.empty((), dtype=torch.int32, device=dev)

    def flush_l2(i):
        flush.fill_(i & 0x7FFF)                 # write 256 MiB: evicts L2
        torch.sum(flush, dim=0, out=sink)       # read it back: no dirty lines left to write back

    with torch.cuda.stream(stream):
        for i in range(R):
            call(i)
        torch.cuda.synchronize(dev)
        g_k = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_k, stream=stream):
            for i in range(K_steps):
                call(i)
        g_one = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_one, stream=stream):
            call(0)
        torch.cuda.synchronize(dev)

        if args.profile:
            for _ in range(args.warmup):
                g_one.replay()
            flush_l2(0)
            torch.cuda.synchronize(dev)
            torch.cuda.profiler.start()
            call(0)
            torch.cuda.synchronize(dev)
            torch.cuda.profiler.stop()
            return None

        # ---- warm-up: W untimed calls, then one untimed sample, whose length sets the
        # sample count so the timed region lasts about 0.4 s (the clock sampler reads every
        # 100 ms): at least args.samples samples
        for _ in range(args.warmup):
            g_one.replay()
        wa, wb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        flush_l2(1)
        wa.record(stream)
        g_k.replay()
        wb.record(stream)
        torch.cuda.synchronize(dev)
        sample_ms = max(wa.elapsed_time(wb), 1e-3) + 0.08     # + the flush
        S = int(min(5000, max(S, -(-400.0 // sample_ms))))

        # ---- timed: S samples of exactly K calls, each behind an L2 flush
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(S)]
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)
        t0 = time.monotonic()
        for i in range(S):
            flush_l2(i)
            ev[i][0].record(stream)
            g_k.replay()
            ev[i][1].record(stream)
        torch.cuda.synchronize(dev)
        t1 = time.monotonic()
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        clocks = sampler.summary(t0, t1) if sampler is not None else None
        sample_us = sorted(a.elapsed_time(b) * 1e3 / K_steps for a, b in ev)

        # ---- cold single call behind the flush (linear-benchmark contract, section 6)
        n_cold = 200
        ce = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_cold)]
        for i in range(5 + n_cold):
            flush_l2(i)
            if i >= 5:
                ce[i - 5][0].record(stream)
            g_one.replay()
            if i >= 5:
                ce[i - 5][1].record(stream)
        torch.cuda.synchronize(dev)
        cold_us = sorted(a.elapsed_time(b) * 1e3 for a, b in ce)

        # ---- end to end through the public call: pinned host X -> device, call, device Y -> pinned host
        e2e = None
        if with_e2e:
            x_h = [torch.from_numpy(x.view(np.int16)).pin_memory() for _ in range(2)]
            y_h = [torch.empty((T, n_out), dtype=torch.int16).pin_memory() for _ in range(2)]
            r_h = [torch.from_numpy(r.view(np.int16)).pin_memory() for _ in range(2)] if add else None
            n_e2e = 200
            ee = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_e2e)]
            for i in range(20 + n_e2e):
                c = i % R
                if i >= 20:
                    ee[i - 20][0].record(stream)
                xs[c].view(torch.int16).copy_(x_h[i & 1], non_blocking=True)
                if add:
                    rs[c].view(torch.int16).copy_(r_h[i & 1], non_blocking=True)
                call(c)
                y_h[i & 1].copy_(ys[c].view(torch.int16), non_blocking=True)
                if i >= 20:
                    ee[i - 20][1].record(stream)
            torch.cuda.synchronize(dev)
            eager_us = sorted(a.elapsed_time(b) * 1e3 for a, b in ee)
            # The same step captured in a CUDA graph per weight copy (the library call is
            # capturable): the copies and the call run as issued above, but one replay per
            # step keeps the host ahead of the GPU, so a step's events time the device work
            # rather than the Python-side enqueue of three operations.
            gs = []
            for c in range(R):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    xs[c].view(torch.int16).copy_(x_h[c & 1], non_blocking=True)
                    if add:
                        rs[c].view(torch.int16).copy_(r_h[c & 1], non_blocking=True)
                    call(c)
                    y_h[c & 1].copy_(ys[c].view(torch.int16), non_blocking=True)
                gs.append(g)
            ge = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_e2e)]
            for i in range(20 + n_e2e):
                c = i % R
                if i >= 20:
                    ge[i - 20][0].record(stream)
                gs[c].replay()
                if i >= 20:
                    ge[i - 20][1].record(stream)
            torch.cuda.synchronize(dev)
            memcpy_us = sorted(a.elapsed_time(b) * 1e3 for a, b in ge)
            host_us = None
            if op == "linear" and qtype == "q4g64" and route_arg == q4lin.ROUTE_AUTO:
                # The library's own host-buffer entry (q4lin_linear_host): X staged from the
                # pinned buffer and Y written back to it by the library's kernels, the same
                # bytes each step; one graph per weight copy, replayed once per step.
                wsh = torch.empty(max(q4lin.host_workspace_bytes(N, K, T), 256), dtype=torch.uint8, device=dev)
                hs = []
                for c in range(R):
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g, stream=stream):
                        q4lin.linear_host(pls[c][0], scs[c], x_h[c & 1], y_host=y_h[c & 1], workspace=wsh,
                                          stream=stream)
                    hs.append(g)
                he = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                      for _ in range(n_e2e)]
                for i in range(20 + n_e2e):
                    c = i % R
                    if i >= 20:
                        he[i - 20][0].record(stream)
                    hs[c].replay()
                    if i >= 20:
                        he[i - 20][1].record(stream)
                torch.cuda.synchronize(dev)
                host_us = sorted(a.elapsed_time(b) * 1e3 for a, b in he)
            e2e = dict(us=host_us if host_us is not None else memcpy_us, memcpy_us=memcpy_us, eager_us=eager_us,
                       host_entry=host_us is not None,
                       h2d=2 * K * T + (2 * N * T if add else 0), d2h=2 * n_out * T)
    del flush
    return dict(sample_us=sample_us, steps=K_steps, samples=S, copies=R, cold_us=cold_us, clocks=clocks,
                route=q4lin.ROUTE_NAMES.get(route, str(route)), launches=launches, e2e=e2e,
                tile=((pl if route == q4lin.ROUTE_TC_SPLITK else None) if op != "linear" else
                      q4lin.tile_plan_full(N, K, T, route_arg) if qtype == "q4g64" else None), ws_bytes=ws_n)


def measure_read_probe(local, logical_bytes):
    """The HBM read probe (q4lin_hbm_read_probe): back-to-back passes over 4 GiB, and
    back-to-back passes over rotating slices of ``logical_bytes`` (the headline call's
    bytes; the slices together exceed L2), timed with CUDA events."""
    import torch
    from weight_only_bit_q4_gb300 import q4lin

    dev = torch.device("cuda", local)
    big_n = 4 << 30
    big = torch.empty(big_n, dtype=torch.uint8, device=dev)
    big.fill_(1)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    sink = torch.empty(8 * sms, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(dev)
    out = {}
    with torch.cuda.stream(stream):
        for _ in range(3):
            q4lin.hbm_read_probe(big, sink, stream=stream)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(10)]
        for a, b in ev:
            a.record(stream)
            q4lin.hbm_read_probe(big, sink, stream=stream)
            b.record(stream)
        torch.cuda.synchronize(dev)
        ms = statistics.median(a.elapsed_time(b) for a, b in ev)
        out["gbs_4gib"] = round(big_n / (ms * 1e-3) / 1e9, 1)
        # slices of the headline's size, 48 of them (~800 MB), each launch on the next slice
        nb = (logical_bytes + 15) // 16 * 16
        nslice = 48
        views = [big[i * nb:(i + 1) * nb] for i in range(nslice)]
        for v in views:
            q4lin.hbm_read_probe(v, sink, stream=stream)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for rep in range(4):
            for v in views:
                q4lin.hbm_read_probe(v, sink, stream=stream)
        b.record(stream)
        torch.cuda.synchronize(dev)
        us = a.elapsed_time(b) * 1e3 / (4 * nslice)
        out["bytes_per_launch"] = nb
        out["us_per_launch"] = round(us, 3)
        out["gbs_per_launch"] = round(nb / (us * 1e-6) / 1e9, 1)
    del big
    out["method"] = ("q4lin_hbm_read_probe: 16-byte non-allocating loads, 4 CTAs of 512 threads per SM; "
                     "4 GiB: median of 10 launches; per launch: back-to-back launches over 48 rotating slices")
    return out


# ----------------------------------------------------------------------------- oracle (CPU) arms
def oracle_rows_for_budget(wl, seconds_per_step):
    """Rows of W per oracle sample so one sample costs about ``seconds_per_step``."""
    N, K, T = wl["N"], wl["K"], wl["T"]
    # decode + FP64 matmul, measured on this class of host at roughly 2e8 weight*token/s per call
    per_row = K * (1.0 + T / 8.0) / 2.0e8
    if wl["qtype"] != "q4g64":
        per_row *= 3.5          # two planes (or int8 codes at twice the count) to decode
    return int(max(1, min(N, seconds_per_step / max(per_row, 1e-12))))


def time_oracle(wl, rows, reps_budget_s, max_reps, exact=False):
    import numpy as np
    import oracle

    N, K, T = wl["N"], wl["K"], wl["T"]
    op = wl.get("op", "linear")
    if wl["qtype"] == "q4g64":
        x = synth.activations(T, K, wl["x_seed"], wl["outliers"])
        if op == "swiglu":
            # the first rows // 2 gate rows and their up rows (rows F .. F + rows // 2 of the weight)
            h = max(1, rows // 2)
            F = N // 2
            full_wq = synth.packed_codes(N, K, wl["w_seed"])
            full_sc = synth.group_scales(N, K, wl["w_seed"], wl["dist"])
            wq = np.concatenate([full_wq[:h], full_wq[F:F + h]])
            sc = np.concatenate([full_sc[:h], full_sc[F:F + h]])

            def run():
                return oracle.fused_ops.linear_swiglu(wq, sc, x)
            out_cols = h
        elif op == "pair":
            h = max(1, rows // 2)
            wa = synth.packed_codes(h, K, wl["w_seed"])
            sa = synth.group_scales(N, K, wl["w_seed"], wl["dist"])[:h]
            wb = synth.packed_codes(h, K, wl["w_seed"] + 1)
            sb = synth.group_scales(N, K, wl["w_seed"] + 1, wl["dist"])[:h]

            def run():
                ya, yb = oracle.fused_ops.linear_pair(wa, sa, wb, sb, x)
                return np.concatenate([ya, yb], axis=1)
            out_cols = 2 * h
        else:
            wq = synth.packed_codes(rows, K, wl["w_seed"])   # the first `rows` rows of the same weight stream
            sc = synth.group_scales(N, K, wl["w_seed"], wl["dist"])[:rows]
            out_cols = rows
            if op == "add":
                r = synth.activations(T, N, wl["x_seed"] + 7919)[:, :rows]

                def run():
                    return oracle.fused_ops.linear_add(wq, sc, x, r)
            else:
                def run():
                    return oracle.linear(wq, sc, x)
    else:
        planes, sc, x = format_problem(wl, rows)
        out_cols = rows

        def run():
            return oracle.sibling_formats.linear(wl["qtype"], planes, sc, x)
    times = []
    t_end = time.monotonic() + reps_budget_s
    while len(times) < max_reps and (exact or len(times) < 3 or time.monotonic() < t_end):
        t0 = time.perf_counter()
        y = run()
        times.append(time.perf_counter() - t0)
        assert y.shape == (T, out_cols) and np.isfinite(y).all()
    return times


def oracle_units(wl, rows):
    """Logical bytes and useful FLOPs of the oracle's sub-problem (rows weight rows; the fused
    forms: rows // 2 gate + up rows, or rows // 2 rows of each of the two weights)."""
    K, T = wl["K"], wl["T"]
    op = wl.get("op", "linear")
    if op in ("swiglu", "pair"):
        h = max(1, rows // 2)
        sub = dict(wl, N=2 * h if op == "swiglu" else h)
        return op_bytes(sub), op_flops(sub)
    b = metrics.model_bytes(rows, K, T, wl["qtype"]) + (2 * rows * T if op == "add" else 0)
    return b, metrics.useful_flops(rows, K, T)


def blas_threads():
    """(threads, how it was found) of the BLAS numpy calls: the thread count the loaded
    OpenBLAS reports, else the environment's setting, else the host's core count."""
    import ctypes

    import numpy as np
    np.dot(np.ones((64, 64)), np.ones((64, 64)))   # make sure the BLAS library is loaded
    try:
        with open("/proc/self/maps") as f:
            libs = sorted({l.split()[-1] for l in f if "blas" in l.lower() and l.split()[-1].startswith("/")})
    except OSError:
        libs = []
    for path in libs:
        try:
            lib = ctypes.CDLL(path)
        except OSError:
            continue
        for sym in ("scipy_openblas_get_num_threads64_", "openblas_get_num_threads64_",
                    "scipy_openblas_get_num_threads", "openblas_get_num_threads"):
            fn = getattr(lib, sym, None)
            if fn is not None:
                fn.restype = ctypes.c_int
                return int(fn()), f"{os.path.basename(path)}: {sym}()"
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        v = os.environ.get(var)
        if v and v.isdigit():
            return int(v), var
    return os.cpu_count() or 1, "os.cpu_count() (BLAS thread count not readable)"


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def cpu_baseline(wl):
    rows = oracle_rows_for_budget(wl, 2.0)
    times = time_oracle(wl, rows, 12.0, 30)
    med = statistics.median(times)
    b, f = oracle_units(wl, rows)
    value = b / med / 1e9 if small_t(wl) else f / med / 1e12
    threads, how = blas_threads()
    return {"value": round(value, 4), "unit": "GB/s" if small_t(wl) else "TFLOP/s",
            "cores": threads, "threads_source": how, "cpu_model": cpu_model(), "host_cores": os.cpu_count(),
            "kind": "oracle",
            "sample": f"FP64 oracle (numpy decode + BLAS matmul) on rows 0..{rows - 1} of the {wl['name']} weight "
                      f"with all {wl['T']} tokens; median of {len(times)} runs; logical units of that sub-problem"}


def reference_arm(args, wl, rank, world):
    if rank != 0:
        return 0
    budget = 150.0
    per_step = min(2.0, budget / (args.steps + args.warmup))
    rows = oracle_rows_for_budget(wl, per_step)
    times = time_oracle(wl, rows, 0.0, args.warmup + args.steps, exact=True)[args.warmup:]
    med = statistics.median(times)
    b, f = oracle_units(wl, rows)
    small = small_t(wl)
    value = b / med / 1e9 if small else f / med / 1e12
    unit = "GB/s" if small else "TFLOP/s"
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": unit,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(med * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl["name"], "N": wl["N"], "K": wl["K"], "T": wl["T"], "qtype": wl["qtype"]},
        "cpu_baseline": {"value": round(value, 4), "unit": unit, "cores": blas_threads()[0],
                         "cpu_model": cpu_model(), "kind": "oracle",
                         "sample": f"each step: FP64 oracle on rows 0..{rows - 1} of the weight, all {wl['T']} tokens"},
        "e2e": {"value": round(value, 4), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- main
def record_summary(wl, res, peaks, world, dev):
    """The figures of one timed record (rates are whole-job: all ranks' units over the
    slowest rank's median sample)."""
    N, K, T = wl["N"], wl["K"], wl["T"]
    su = res["sample_us"]
    med, lo, p95 = statistics.median(su), su[0], metrics.percentile(su, 95)
    med_max, lo_max, p95_max = reduce_max([med, lo, p95], world, dev)
    mb, fl = op_bytes(wl), op_flops(wl)
    small = small_t(wl)
    unit = "GB/s" if small else "TFLOP/s"

    def rate(us):
        return mb / (us * 1e-6) / 1e9 if small else fl / (us * 1e-6) / 1e12

    # roofline of the dominant kernel: algorithmic bytes (FLOPs) per launch / its mean launch duration
    nl = max(1, res["launches"])
    per_launch_us = med_max / nl
    if small:
        roof = {"bound": "hbm", "achieved": round(mb / nl / (per_launch_us * 1e-6) / 1e9, 2),
                "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    else:
        roof = {"bound": "tensor", "achieved": round(fl / nl / (per_launch_us * 1e-6) / 1e12, 2),
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s"}
    roof["frac"] = round(roof["achieved"] / roof["peak"], 4)
    roof["peak_source"] = peaks["source"]
    traffic, tkernel = recorded_traffic(wl["name"])
    roof["traffic"] = traffic
    if tkernel:
        roof["traffic_kernel"] = tkernel
    cold = res["cold_us"]
    cold_med = statistics.median(cold)
    return {
        "workload": wl["name"], "N": N, "K": K, "T": T, "qtype": wl["qtype"], "route": res["route"],
        "tile": res["tile"], "launches_per_step": res["launches"],
        "steps": res["steps"], "samples": res["samples"],
        "value": round(rate(med_max) * world, 3), "unit": unit, "ms_per_step": round(med_max * 1e-3, 6),
        "us": {"median": round(med_max, 3), "min": round(lo_max, 3), "p95": round(p95_max, 3)},
        "logical_gbs": round(mb / (med_max * 1e-6) / 1e9, 2), "tflops": round(fl / (med_max * 1e-6) / 1e12, 3),
        "roofline": roof,
        "cold_call": {"method": "256 MiB write+read L2 flush, events around one graph launch of one call",
                      "median_us": round(cold_med, 3), "min_us": round(cold[0], 3),
                      "p95_us": round(metrics.percentile(cold, 95), 3), "samples": len(cold),
                      "value": round(rate(cold_med), 3), "unit": unit},
        "clocks": res["clocks"],
        "gpu_launches": res["launches"] * res["steps"] * res["samples"],
        "l2": f"{res['copies']} rotating copies of weights, X and Y ({res['copies'] * mb / 1e6:.0f} MB) "
              f"and a 256 MiB write+read flush before every sample",
    }


# ----------------------------------------------------------------------------- T sweep
DRAM_SPEC_GBS = 7900.0   # GB300 HBM3e, nominal


def parse_sweep(spec):
    """T values of a --sweep spec: comma-separated A:B:S ranges (inclusive) and single values."""
    ts = []
    for part in spec.split(","):
        part = part.strip()
        if not part:
            continue
        if ":" in part:
            f = [int(v) for v in part.split(":")]
            a, b, st = (f + [1])[:3] if len(f) == 2 else f
            if st < 1 or a < 1 or b < a:
                raise SystemExit(f"bad sweep range {part}")
            ts.extend(range(a, b + 1, st))
        else:
            ts.append(int(part))
    out = []
    for t in ts:
        if t < 1:
            raise SystemExit(f"bad sweep value {t}")
        if t not in out:
            out.append(t)
    return out


SWEEP_COLUMNS = ("label", "qtype", "policy", "N", "K", "T", "median_us", "min_us", "p95_us", "model_GB",
                 "effective_GB/s", "DRAM_%", "READ_%", "useful_TFLOP/s", "memory_floor_pct", "delta_%")


def sweep_row(label, qtype, N, K, T, us_sorted, sustained_read, prev_median):
    """One line of the sweep (the contract's section 7 fields, from section 4-5 formulas)."""
    med = statistics.median(us_sorted)
    mb = metrics.model_bytes(N, K, T, qtype)
    eff = mb / (med * 1e-6) / 1e9
    floor_us = mb / (DRAM_SPEC_GBS * 1e9) * 1e6
    return {
        "label": label, "qtype": qtype, "policy": "a16", "N": N, "K": K, "T": T,
        "median_us": round(med, 3), "min_us": round(us_sorted[0], 3),
        "p95_us": round(metrics.percentile(us_sorted, 95), 3), "model_GB": round(mb / 1e9, 6),
        "effective_GB/s": round(eff, 1), "DRAM_%": round(100.0 * eff / DRAM_SPEC_GBS, 2),
        "READ_%": round(100.0 * eff / sustained_read, 2) if sustained_read else None,
        "useful_TFLOP/s": round(metrics.useful_flops(N, K, T) / (med * 1e-6) / 1e12, 3),
        "memory_floor_pct": round(100.0 * floor_us / med, 2),
        "delta_%": None if prev_median is None else round(100.0 * (med - prev_median) / prev_median, 2),
    }


def measure_sweep_point(wl, ts_repeat, dev, stream, flush, sink, weights):
    """Cold-cache per-call samples (us, sorted) of one sweep point through the public call."""
    import numpy as np
    import torch
    from weight_only_bit_q4_gb300 import q4lin

    N, K, T = wl["N"], wl["K"], wl["T"]
    x = synth.activations(T, K, wl["x_seed"], outliers=wl["outliers"])
    x_d = torch.from_numpy(x.view(np.int16)).to(dev).view(torch.bfloat16)
    y = torch.empty((T, N), dtype=torch.bfloat16, device=dev)
    ws_n = q4lin.workspace_bytes(N, K, T)
    ws = torch.empty(max(ws_n, 256), dtype=torch.uint8, device=dev)
    wq_d, sc_d = weights

    def call():
        q4lin.linear(wq_d, sc_d, x_d, y=y, workspace=ws if ws_n else None, stream=stream)

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(ts_repeat)]
    with torch.cuda.stream(stream):
        call()                      # first public call: not timed
        for _ in range(3):          # warm-up
            call()
        for i, (a, b) in enumerate(ev):
            flush.fill_(i & 0x7FFF)                 # 256 MiB written, then read: L2 holds none of the call's data
            torch.sum(flush, dim=0, out=sink)
            a.record(stream)
            call()
            b.record(stream)
    torch.cuda.synchronize(dev)
    return sorted(a.elapsed_time(b) * 1e3 for a, b in ev)


def run_sweep(args):
    import numpy as np
    import torch
    from weight_only_bit_q4_gb300 import q4lin

    if args.qtype != "q4g64" or args.op != "linear" or args.route != "auto":
        raise SystemExit("--sweep times the Q4 layer (q4lin_linear) only")
    name = args.workload or "q4_6144x5120"
    if WORKLOADS[name][2] is not None:
        raise SystemExit(f"--sweep needs a workload whose T is free (not {name})")
    ts = parse_sweep(args.sweep)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.Stream(dev)
    wl0 = workload(args, name, ts[0])
    N, K = wl0["N"], wl0["K"]
    wq = synth.packed_codes(N, K, wl0["w_seed"])
    sc = synth.group_scales(N, K, wl0["w_seed"], wl0["dist"])
    weights = (torch.from_numpy(wq).to(dev), torch.from_numpy(sc.view(np.int16)).to(dev))
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    sink = torch.empty((), dtype=torch.int32, device=dev)
    probe = measure_read_probe(0, metrics.model_bytes(N, K, 1))
    sustained = probe["gbs_4gib"]
    print(f"gpu={torch.cuda.get_device_name(dev)}")
    print(f"dram_spec={DRAM_SPEC_GBS:.1f} GB/s")
    print(f"sustained_read={sustained:.1f} GB/s")
    print("cache=cold")
    print(" ".join(SWEEP_COLUMNS))
    rows, prev = [], None
    for t in ts:
        wl = workload(args, name, t)
        us = measure_sweep_point(wl, args.repeat, dev, stream, flush, sink, weights)
        row = sweep_row(f"{name}_t{t}", "q4g64", N, K, t, us, sustained, prev)
        prev = row["median_us"]
        rows.append(row)
        print(" ".join("-" if row[c] is None else str(row[c]) for c in SWEEP_COLUMNS), flush=True)
    if args.csv_out:
        import csv
        with open(args.csv_out, "w", newline="") as f:
            w = csv.DictWriter(f, fieldnames=list(SWEEP_COLUMNS))
            w.writeheader()
            w.writerows(rows)
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.sweep is not None:
        return run_sweep(args)
    rank, world, local = dist_env()
    specs = record_specs(args)
    wls = [workload(args, n, t) for (n, t) in specs]
    if args.impl == "reference":
        return reference_arm(args, wls[0], rank, world)

    import torch
    # NCCL on the GPUs; gloo with CPU tensors where there is no GPU (the multi-rank
    # host path, exercised by the CPU tests with the measurement stubbed)
    on_gpu = torch.cuda.is_available()
    if world > 1:
        import torch.distributed as dist
        if on_gpu:
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group("gloo")
    dev = torch.device("cuda", local) if on_gpu else None
    cvd = [v for v in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if v.strip()]
    sampler = ClockSampler(cvd[local].strip() if local < len(cvd) else str(local)) if on_gpu else None
    if sampler is not None:
        sampler.start()
        time.sleep(0.5)   # let the sampler's first readings arrive
    peaks = load_peaks()
    recs = []
    try:
        for i, wl in enumerate(wls):
            res = measure_ours(args, wl, rank, world, local, sampler=sampler,
                               with_e2e=(i == 0 and not args.no_e2e))
            if res is None:
                return 0
            recs.append((wl, res))
        probe = None
        if on_gpu and not args.no_probe and args.workload is None and world == 1:
            probe = measure_read_probe(local, op_bytes(wls[0]))
    finally:
        if sampler is not None:
            sampler.stop()
    summaries = [record_summary(wl, res, peaks, world, dev) for wl, res in recs]
    wl0, res0 = recs[0]
    head = summaries[0]
    e2e = None
    if res0["e2e"]:
        e = res0["e2e"]
        emed = reduce_max([statistics.median(e["us"])], world, dev)[0]
        mb0, fl0 = op_bytes(wl0), op_flops(wl0)
        ev = mb0 / (emed * 1e-6) / 1e9 if small_t(wl0) else fl0 / (emed * 1e-6) / 1e12
        eager = reduce_max([statistics.median(e["eager_us"])], world, dev)[0]
        mcp = reduce_max([statistics.median(e["memcpy_us"])], world, dev)[0]
        e2e = {"value": round(ev * world, 3), "unit": head["unit"], "us": round(emed, 3),
               "h2d_bytes_per_step": e["h2d"], "d2h_bytes_per_step": e["d2h"],
               "memcpy_us": round(mcp, 3), "eager_us": round(eager, 3),
               "method": ("per step: q4lin_linear_host on pinned host X and Y (the library's kernels copy X "
                          "in and Y out around the layer), " if e.get("host_entry") else
                          "per step: pinned host X -> device (cudaMemcpyAsync), the public call, device Y -> "
                          "pinned host, ") +
                         "captured in one CUDA graph per weight copy and replayed once per step; events around "
                         "each replay; median of 200.  memcpy_us: the step with cudaMemcpyAsync copies around "
                         "the device-buffer call, graphed the same way; eager_us: those three issued from "
                         "Python each step"}
    if rank != 0:
        return 0
    line = {
        "metric": METRIC, "value": head["value"], "unit": head["unit"],
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "samples": head["samples"],
        "ms_per_step": head["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": {"gemv": "f32", "tc_fp16": "fp16xfp16->f32",
                  "stream_mma": "fp16xfp16->f32 (exact operands)"}.get(head["route"], "bf16xbf16->f32"),
        "data": "synthetic",
        "config": {"workload": wl0["name"], "N": wl0["N"], "K": wl0["K"], "T": wl0["T"], "qtype": wl0["qtype"],
                   "route": head["route"], "tile": head["tile"],
                   "timing": f"median of {head['samples']} samples; a sample is one CUDA graph of {args.steps} "
                             f"back-to-back calls behind an L2 flush, events on the launching stream",
                   "l2": head["l2"],
                   "parallelism": "replicas" if world > 1 else "single"},
        "us": head["us"], "logical_gbs": head["logical_gbs"], "tflops": head["tflops"],
        "cold_call": head["cold_call"],
        "roofline": head["roofline"],
        "e2e": e2e,
        "gpu_launches": head["gpu_launches"],
        "clocks": head["clocks"],
        "records": summaries[1:],
    }
    if probe is not None:
        probe["frac_4gib_of_copy"] = round(probe["gbs_4gib"] / peaks["hbm_gbs"], 4)
        line["hbm_read_probe"] = probe
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl0)
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
