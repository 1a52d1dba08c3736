#!/usr/bin/env python3
"""Benchmark of the Q4_G64_FP16 linear layer on one GB300 (or N replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--t T] [--qtype FMT] [--route R] [--op OP] [--profile]

Timing (the linear-benchmark contract, section 6, and the Q4 measurement
report's header table): every sample is one complete public call captured in
a CUDA graph; before each sample a 256 MiB buffer is written and then read
back (the write evicts L2, the read leaves it clean so no dirty lines are
written back inside the sample); CUDA events on the launching stream bracket
only the graph launch; the flush and the graph are queued back to back with
no host synchronisation.  The primary figure is the median; min and p95 are
reported too.  Metrics follow the contract's sections 4-5 (weight_only_bit_q4_gb300.metrics).

A step is one call of the layer on one batch of the workload's synthetic
input.  Default workload: the decode GEMV, N=6144 K=5120 T=1.  --qtype times
a sibling weight format (Q5G64, Q6G64, W8G32) on the same geometry through
q4lin_linear_qtype (W8G32 for 1..4 tokens); its bytes are that format's.
Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(the layer does not exchange data between GPUs); value = the units all ranks
processed / the slowest rank's time.
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


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=None,
                   help="timed calls (default: enough for about a second of GPU time)")
    p.add_argument("--warmup", type=int, default=100)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    p.add_argument("--t", type=int, default=None, help="T for the sweep workloads")
    p.add_argument("--qtype", default="q4g64", choices=sorted(metrics.GROUP_BYTES),
                   help="weight format (the sibling formats run for 1..4 tokens)")
    p.add_argument("--op", default="linear", choices=["linear", "add"],
                   help="linear: Y = W.X; add: LinearAdd, Y = W.X + R (the tile route for every T)")
    p.add_argument("--route", default="auto", choices=["auto", "tc_fp16"],
                   help="auto: the library's choice; tc_fp16: the opt-in tile route on fp16-rounded weights")
    p.add_argument("--profile", action="store_true",
                   help="one call between cudaProfilerStart/Stop after warm-up and flush (for ncu --profile-from-start off)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    a = p.parse_args(argv)
    a.warmup = max(a.warmup, 3)
    if a.steps is not None:
        a.steps = max(a.steps, 1)
    return a


def workload(args):
    N, K, T, dist, outl, ws, xs = WORKLOADS[args.workload]
    if T is None:
        T = args.t if args.t is not None else 1
    elif args.t is not None and args.t != T:
        raise SystemExit(f"workload {args.workload} has fixed T={T}")
    if xs is None:
        xs = T
    name = args.workload if WORKLOADS[args.workload][2] is not None else f"{args.workload}_t{T}"
    qtype = getattr(args, "qtype", "q4g64")
    if qtype != "q4g64":
        if T > 4 and qtype == "w8g32":
            raise SystemExit(f"{qtype} runs for 1..4 tokens")
        name = qtype + name[2:]            # q4_6144x5120_t1 -> q5g64_6144x5120_t1
    route = getattr(args, "route", "auto")
    if route != "auto":
        if qtype != "q4g64":
            raise SystemExit(f"--route {route} runs the Q4 format only")
        name += "_" + route
    op = getattr(args, "op", "linear")
    if op == "add":
        if qtype != "q4g64" or route != "auto":
            raise SystemExit("--op add runs the Q4 format on its own route")
        name += "_add"
    return dict(name=name, N=N, K=K, T=T, dist=dist, outliers=outl, w_seed=ws, x_seed=xs, qtype=qtype, op=op)


def op_bytes(wl):
    """Logical bytes of one call: the layer's model bytes, plus the residual read by LinearAdd."""
    N, K, T = wl["N"], wl["K"], wl["T"]
    return metrics.model_bytes(N, K, T, wl["qtype"]) + (2 * N * T if wl.get("op") == "add" else 0)


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
    """nvidia-smi clocks and throttle reasons sampled every 100 ms in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t_start = self.t_stop = None

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

    def mark_start(self):
        self.t_start = time.monotonic()

    def mark_stop(self):
        self.t_stop = time.monotonic()

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = [l for (t, l) in self.lines if self.t_start is not None and self.t_start <= t <= (self.t_stop or t) + 0.1]
        if not rows:
            rows = [l for (_, l) in self.lines[-3:]]
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
def measure_ours(args, wl, rank, world, local):
    """Times the layer on this rank's GPU.

    Steady state (the primary figure): R copies of the weight planes and of X
    (and R outputs) whose total exceeds 2.5x the L2 size, so every call streams
    its operands from HBM; one CUDA graph holds R consecutive calls (call i on
    copy i) and the timed region replays it back to back, with CUDA events on
    the launching stream around every replay.  ms_per_step = total / calls.

    Cold single call (the linear-benchmark contract's method, reported beside
    it): before each sample a 256 MiB buffer is written then read back, then
    events bracket one graph launch of one call; median / min / p95.
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
    add = wl.get("op") == "add"
    r = synth.activations(T, N, wl["x_seed"] + 7919) if add else None   # LinearAdd's bf16 residual [T, N]
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size or (128 << 20)
    R = int(max(2, min(64, -(-int(2.5 * l2) // per_copy))))
    pl_d = tuple(torch.from_numpy(p).to(dev) for p in planes)
    sc_d = torch.from_numpy(sc.view(np.int16)).to(dev)
    x_d = torch.from_numpy(x.view(np.int16)).to(dev).view(torch.bfloat16)
    pls = [pl_d] + [tuple(p.clone() for p in pl_d) for _ in range(R - 1)]
    scs = [sc_d] + [sc_d.clone() for _ in range(R - 1)]
    xs = [x_d] + [x_d.clone() for _ in range(R - 1)]
    ys = [torch.empty((T, N), dtype=torch.bfloat16, device=dev) for _ in range(R)]
    rs = [torch.from_numpy(r.view(np.int16)).to(dev).view(torch.bfloat16) for _ in range(R)] if add else None
    route_arg = q4lin.ROUTE_TC_FP16 if args.route == "tc_fp16" else q4lin.ROUTE_AUTO
    ws_n = q4lin.workspace_bytes(N, K, T, route_arg)
    ws_d = torch.empty(max(ws_n, 256), dtype=torch.uint8, device=dev)
    route = q4lin.select_route(N, K, T) if route_arg == q4lin.ROUTE_AUTO else route_arg
    launches = q4lin.kernel_launches(N, K, T)
    if route_arg != q4lin.ROUTE_AUTO:   # operand pass + main launch (+ tail launch)
        pl = q4lin.tile_plan_full(N, K, T, route_arg)
        launches = 1 + (2 if pl["main_tiles"] < -(-N // 128) * -(-T // pl["n"]) else 1)
    stream = torch.cuda.Stream(dev)

    if qtype != "q4g64":   # the streaming GEMV (1..4 tokens), else Q5 / Q6 on the exact tile route
        launches = q4lin.kernel_launches(N, K, T, qtype)
        route = q4lin.ROUTE_GEMV if (T <= 4 and q4lin.select_route(N, K, T) == q4lin.ROUTE_GEMV) \
            else q4lin.ROUTE_TC_SPLITK

    if add:   # the exact tile route for every T: one launch, or two with a tail launch
        pl = q4lin.tile_plan_full(N, K, T, q4lin.ROUTE_TC_SPLITK)
        route = q4lin.ROUTE_TC_SPLITK
        launches = 2 if pl["main_tiles"] < -(-N // 128) * -(-T // pl["n"]) else 1

    def call(i):
        if add:
            q4lin.linear_add(pls[i][0], scs[i], xs[i], rs[i], y=ys[i], stream=stream)
        elif qtype == "q4g64":
            q4lin.linear(pls[i][0], scs[i], xs[i], y=ys[i], workspace=ws_d if ws_n else None, stream=stream,
                         route=route_arg)
        else:
            q4lin.linear_qtype(qtype, pls[i], scs[i], xs[i], y=ys[i], stream=stream)

    with torch.cuda.stream(stream):
        for i in range(R):
            call(i)
        torch.cuda.synchronize(dev)
        g_all = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_all, stream=stream):
            for i in range(R):
                call(i)
        g_one = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_one, stream=stream):
            call(0)
        torch.cuda.synchronize(dev)

        if args.profile:
            flush = torch.empty((256 << 20) // 4, dtype=torch.int32, device=dev)
            sink = torch.empty((), dtype=torch.int32, device=dev)
            for _ in range(args.warmup):
                g_one.replay()
            flush.fill_(1)
            torch.sum(flush, dim=0, out=sink)
            torch.cuda.synchronize(dev)
            torch.cuda.profiler.start()
            call(0)
            torch.cuda.synchronize(dev)
            torch.cuda.profiler.stop()
            return None

        # ---- steady state
        reps = max(1, -(-args.steps // R))
        calls = reps * R
        for _ in range(max(1, -(-args.warmup // R))):
            g_all.replay()
        torch.cuda.synchronize(dev)
        cvd = [v for v in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if v.strip()]
        sampler = ClockSampler(cvd[local].strip() if local < len(cvd) else str(local))
        sampler.start()
        t_wait = time.monotonic() + 0.6
        while time.monotonic() < t_wait:   # keep the GPU busy while the sampler starts
            g_all.replay()
            torch.cuda.synchronize(dev)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)
        sampler.mark_start()
        ev[0].record(stream)
        for r in range(reps):
            g_all.replay()
            ev[r + 1].record(stream)
        torch.cuda.synchronize(dev)
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        sampler.mark_stop()
        clocks = sampler.stop()
        rep_ms = [ev[r].elapsed_time(ev[r + 1]) for r in range(reps)]
        total_ms = ev[0].elapsed_time(ev[reps])
        per_call_us = sorted(m * 1e3 / R for m in rep_ms)

        # ---- cold single call behind a 256 MiB write+read flush (linear-benchmark contract, section 6)
        flush = torch.empty((256 << 20) // 4, dtype=torch.int32, device=dev)
        sink = torch.empty((), dtype=torch.int32, device=dev)
        n_cold = 200
        ce = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_cold)]
        for i in range(5 + n_cold):
            flush.fill_(i & 0x7FFF)
            torch.sum(flush, dim=0, out=sink)
            if i >= 5:
                ce[i - 5][0].record(stream)
            g_one.replay()
            if i >= 5:
                ce[i - 5][1].record(stream)
        torch.cuda.synchronize(dev)
        cold_us = sorted(a.elapsed_time(b) * 1e3 for a, b in ce)
        del flush

        # ---- end to end through the public call: pinned host X -> device, call, device Y -> pinned host
        e2e = None
        if not args.no_e2e:
            x_h = [torch.from_numpy(x.view(np.int16)).pin_memory() for _ in range(2)]
            y_h = [torch.empty((T, N), dtype=torch.int16).pin_memory() for _ in range(2)]
            r_h = [torch.from_numpy(r.view(np.int16)).pin_memory() for _ in range(2)] if add else None
            n_e2e = min(max(args.steps // 10, 100), 2000)
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
            e2e = dict(us=sorted(a.elapsed_time(b) * 1e3 for a, b in ee), h2d=2 * K * T + (2 * N * T if add else 0),
                       d2h=2 * N * T)

    return dict(per_call_us=per_call_us, total_ms=total_ms, calls=calls, copies=R, cold_us=cold_us,
                clocks=clocks, route=q4lin.ROUTE_NAMES.get(route, str(route)), launches=launches, e2e=e2e,
                tile=q4lin.tile_plan_full(N, K, T, q4lin.ROUTE_TC_SPLITK if add else route_arg),
                ws_bytes=ws_n)


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
    if wl["qtype"] == "q4g64":
        wq = synth.packed_codes(rows, K, wl["w_seed"])   # the first `rows` rows of the same weight stream
        sc = synth.group_scales(N, K, wl["w_seed"], wl["dist"])[:rows]
        x = synth.activations(T, K, wl["x_seed"], wl["outliers"])

        if wl.get("op") == "add":
            r = synth.activations(T, N, wl["x_seed"] + 7919)[:, :rows]

            def run():
                return oracle.fused_ops.linear_add(wq, sc, x, r)
        else:
            def run():
                return oracle.linear(wq, sc, x)
    else:
        planes, sc, x = format_problem(wl, rows)

        def run():
            return oracle.sibling_formats.linear(wl["qtype"], planes, sc, x)
    times = []
    t_end = time.monotonic() + reps_budget_s
    while len(times) < max_reps and (exact or len(times) < 3 or time.monotonic() < t_end):
        t0 = time.perf_counter()
        y = run()
        times.append(time.perf_counter() - t0)
        assert y.shape == (T, rows) and np.isfinite(y).all()
    return times


def oracle_units(wl, rows):
    K, T = wl["K"], wl["T"]
    b = metrics.model_bytes(rows, K, T, wl["qtype"]) + (2 * rows * T if wl.get("op") == "add" else 0)
    f = metrics.useful_flops(rows, K, T)
    return b, f


def blas_threads():
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        v = os.environ.get(var)
        if v and v.isdigit():
            return int(v)
    return os.cpu_count() or 1


def cpu_baseline(wl):
    rows = oracle_rows_for_budget(wl, 2.0)
    times = time_oracle(wl, rows, 12.0, 30)
    med = statistics.median(times)
    b, f = oracle_units(wl, rows)
    value = b / med / 1e9 if small_t(wl) else f / med / 1e12
    return {"value": round(value, 4), "unit": "GB/s" if small_t(wl) else "TFLOP/s",
            "cores": blas_threads(), "kind": "oracle",
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
        "cpu_baseline": {"value": round(value, 4), "unit": unit, "cores": blas_threads(), "kind": "oracle",
                         "sample": f"each step: FP64 oracle on rows 0..{rows - 1} of the weight, all {wl['T']} tokens"},
        "e2e": {"value": round(value, 4), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- main
def main(argv=None):
    args = parse_args(argv)
    rank, world, local = dist_env()
    wl = workload(args)
    if args.steps is None:
        # about a second of GPU time at the expected rate, so the clock sampler sees the timed region
        us_guess = max(2.0, metrics.model_bytes(wl["N"], wl["K"], wl["T"], wl["qtype"]) / 5e3 / 1e3,
                       metrics.useful_flops(wl["N"], wl["K"], wl["T"]) / 1.0e15 * 1e6)
        args.steps = int(min(200000, max(1000, 1.0e6 / us_guess)))
    if args.impl == "reference":
        return reference_arm(args, wl, rank, world)

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
    res = measure_ours(args, wl, rank, world, local)
    if res is None:
        return 0
    dev = torch.device("cuda", local) if on_gpu else None
    mean_us = res["total_ms"] * 1e3 / res["calls"]          # steady state, all calls of the timed region
    med_rep = statistics.median(res["per_call_us"])         # median over graph replays
    mean_max, med_max = reduce_max([mean_us, med_rep], world, dev)
    N, K, T = wl["N"], wl["K"], wl["T"]
    mb, fl = op_bytes(wl), metrics.useful_flops(N, K, T)
    small = small_t(wl)
    unit = "GB/s" if small else "TFLOP/s"

    def rate(us):
        return mb / (us * 1e-6) / 1e9 if small else fl / (us * 1e-6) / 1e12

    value = rate(mean_max) * world
    peaks = load_peaks()
    # roofline of the dominant kernel: algorithmic bytes (FLOPs) per launch / its mean launch duration
    nl = max(1, res["launches"])
    per_launch_us = mean_max / nl
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
    e2e = None
    if res["e2e"]:
        e = res["e2e"]
        emed = reduce_max([statistics.median(e["us"])], world, dev)[0]
        e2e = {"value": round(rate(emed) * world, 3), "unit": unit, "us": round(emed, 3),
               "h2d_bytes_per_step": e["h2d"], "d2h_bytes_per_step": e["d2h"]}
    if rank != 0:
        return 0
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": unit,
        "n_gpus": world, "steps": res["calls"], "warmup": args.warmup, "ms_per_step": round(mean_max * 1e-3, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": {"gemv": "f32", "tc_fp16": "fp16xfp16->f32"}.get(res["route"], "bf16xbf16->f32"),
        "data": "synthetic",
        "config": {"workload": wl["name"], "N": N, "K": K, "T": T, "qtype": wl["qtype"], "route": res["route"],
                   "tile": res["tile"],
                   "timing": f"steady state: CUDA graph of {res['copies']} back-to-back calls replayed, events per replay",
                   "l2": f"inputs larger than L2: {res['copies']} rotating copies of weights, X and Y "
                         f"({res['copies'] * mb / 1e6:.0f} MB)",
                   "parallelism": "replicas" if world > 1 else "single"},
        "us": {"mean": round(mean_us, 3), "median_replay": round(med_rep, 3),
               "min_replay": round(res["per_call_us"][0], 3)},
        "logical_gbs": round(mb / (mean_us * 1e-6) / 1e9, 2),
        "tflops": round(fl / (mean_us * 1e-6) / 1e12, 3),
        "cold_call": {"method": "256 MiB write+read L2 flush, events around one graph launch of one call",
                      "median_us": round(cold_med, 3), "min_us": round(cold[0], 3),
                      "p95_us": round(metrics.percentile(cold, 95), 3), "samples": len(cold),
                      "value": round(rate(cold_med), 3), "unit": unit},
        "roofline": roof,
        "e2e": e2e,
        "gpu_launches": res["launches"] * res["calls"],
        "clocks": res["clocks"],
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl)
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
