"""Benchmark metrics for the Q4_G64_FP16 linear layer.

Definitions follow the linear-benchmark contract (linear-benchmark.md,
section 4 "theoretical traffic" and section 5 "useful work") and the Q4
measurement report (q4-linear.md, metric definitions):

    weight_bytes  = groups * 34,  groups = N * align_up(K, 128) / 64
    model_bytes   = weight_bytes + 2*K*T + 2*N*T      (one logical pass)
    logical GB/s  = model_bytes / seconds / 1e9
    useful FLOPs  = 2*N*K*T  (decode, padding and split-K work not counted)
    TFLOP/s       = useful FLOPs / seconds / 1e12
    memory floor  = model_bytes / bandwidth

The sibling formats of the same table count their own bytes per group:
Q5G64 42 and Q6G64 50 per 64 weights, W8G32 34 per 32 weights.
"""
from __future__ import annotations


def align_up(v: int, a: int) -> int:
    return (v + a - 1) // a * a


def q4_weight_bytes(N: int, K: int) -> int:
    return N * align_up(K, 128) // 64 * (32 + 2)


# qtype -> (weights per group, bytes per group, scale included)
GROUP_BYTES = {"q4g64": (64, 34), "q5g64": (64, 42), "q6g64": (64, 50), "w8g32": (32, 34)}


def weight_bytes(qtype: str, N: int, K: int) -> int:
    group, per_group = GROUP_BYTES[qtype]
    return N * align_up(K, 128) // group * per_group


def model_bytes(N: int, K: int, T: int, qtype: str = "q4g64") -> int:
    return weight_bytes(qtype, N, K) + 2 * K * T + 2 * N * T


def useful_flops(N: int, K: int, T: int) -> int:
    return 2 * N * K * T


def logical_gbs(N: int, K: int, T: int, seconds: float) -> float:
    return model_bytes(N, K, T) / seconds / 1e9


def tflops(N: int, K: int, T: int, seconds: float) -> float:
    return useful_flops(N, K, T) / seconds / 1e12


def memory_floor_us(N: int, K: int, T: int, gbs: float) -> float:
    return model_bytes(N, K, T) / (gbs * 1e9) * 1e6


def percentile(sorted_vals, p: float) -> float:
    """Nearest-rank percentile of an already sorted list."""
    if not sorted_vals:
        return float("nan")
    import math
    rank = math.ceil(p / 100.0 * len(sorted_vals))
    return sorted_vals[max(0, min(len(sorted_vals), rank) - 1)]
