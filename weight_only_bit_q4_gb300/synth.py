"""Seeded synthetic inputs for the Q4_G64_FP16 linear layer.

This module only draws numbers: it holds none of the layer's arithmetic (no
decode, no dequantisation, no matmul).  Both the CUDA path's tests/benchmark
and the CPU oracle's tests take their inputs from here, so the two sides see
the same bytes.

Random source
-------------
A counter-based splitmix64 (Steele, Lea & Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014): output ``i`` of a stream whose
state starts at ``s0`` is ``mix64(s0 + (i + 1) * GAMMA)`` -- exactly the
sequence the sequential generator produces, but computable for any ``i``.
Each tensor draws from its own stream; the stream's start state is
``mix64(seed * GAMMA ^ tag)`` with a fixed 64-bit tag per tensor.

Uniforms take the top 53 bits: ``u = (z >> 11) * 2**-53`` in [0, 1).
Normals use the Box-Muller transform on consecutive uniform pairs
``(u1, u2)``: ``r = sqrt(-2 ln(1 - u1))``, giving ``r cos(2 pi u2)`` and
``r sin(2 pi u2)``.

Workloads (the linear-benchmark contract's fixture is not published, so these
stand in for it; the recipe is the one the benchmark configurations name):

* codes: uniform integers 0..15, two per byte (even k in the low nibble);
  the packed bytes are the little-endian bytes of the stream's outputs, which
  makes both nibbles independent and uniform.
* scales: fp16 of ``|N(0,1)| * 0.02 + 1e-3`` ("halfnormal"), or of
  ``exp(ln 0.02 + 0.5 * N(0,1))`` ("lognormal"), rounded to nearest even.
* activations X[T, K]: bf16 of N(0,1) (double -> float32 -> bf16, each
  round-to-nearest-even); with ``outliers=True`` round(0.01 * K) channels
  (columns k of X, chosen without replacement from the seed) are multiplied
  by 20 for every token before rounding.
"""
from __future__ import annotations

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# One tag per tensor so the streams never overlap in practice.
TAG_CODES = 0x436F646573000001
TAG_SCALES = 0x5363616C65000002
TAG_X = 0x4163747300000003
TAG_OUTLIER = 0x4F75746C69000004
TAG_HIGH = 0x4869676800000005
TAG_W8 = 0x5738436F64000006


def mix64(z: np.ndarray) -> np.ndarray:
    """splitmix64 output function on a uint64 array (wrapping arithmetic)."""
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def stream_state(seed: int, tag: int) -> np.uint64:
    with np.errstate(over="ignore"):
        s = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) * GAMMA ^ np.uint64(tag)
    return mix64(np.array([s], dtype=np.uint64))[0]


def splitmix64(state: int | np.uint64, count: int, start: int = 0) -> np.ndarray:
    """Outputs ``start .. start+count-1`` of the splitmix64 sequence seeded with ``state``."""
    idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(state) + idx * GAMMA
    return mix64(z)


def uniform(state, count: int) -> np.ndarray:
    z = splitmix64(state, count)
    return (z >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal(state, count: int) -> np.ndarray:
    pairs = (count + 1) // 2
    u = uniform(state, 2 * pairs).reshape(pairs, 2)
    r = np.sqrt(-2.0 * np.log1p(-u[:, 0]))
    th = 2.0 * np.pi * u[:, 1]
    out = np.empty((pairs, 2), dtype=np.float64)
    out[:, 0] = r * np.cos(th)
    out[:, 1] = r * np.sin(th)
    return out.reshape(-1)[:count]


def float32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    return float32_to_bf16_bits(np.asarray(a, dtype=np.float64).astype(np.float32))


def to_fp16_bits(a: np.ndarray) -> np.ndarray:
    return np.asarray(a, dtype=np.float64).astype(np.float16).view(np.uint16)


def packed_codes(N: int, K: int, seed: int = 0) -> np.ndarray:
    """uint8 [N, K/2]: uniform nibbles, even k in the low nibble."""
    assert K % 2 == 0
    nbytes = N * (K // 2)
    words = splitmix64(stream_state(seed, TAG_CODES), (nbytes + 7) // 8)
    return words.astype("<u8").view(np.uint8)[:nbytes].reshape(N, K // 2).copy()


def group_scales(N: int, K: int, seed: int = 0, dist: str = "halfnormal", group: int = 64) -> np.ndarray:
    """fp16 bit patterns [N, K/group]."""
    G = K // group
    z = normal(stream_state(seed, TAG_SCALES), N * G).reshape(N, G)
    if dist == "halfnormal":
        s = np.abs(z) * 0.02 + 1e-3
    elif dist == "lognormal":
        s = np.exp(np.log(0.02) + 0.5 * z)
    else:
        raise ValueError(dist)
    return to_fp16_bits(s)


def outlier_channels(K: int, seed: int) -> np.ndarray:
    """round(0.01*K) distinct channel indices in [0, K), drawn from the seed."""
    n = int(round(0.01 * K))
    keys = splitmix64(stream_state(seed, TAG_OUTLIER), K)
    return np.sort(np.argsort(keys, kind="stable")[:n])


def activations(T: int, K: int, seed: int, outliers: bool = False) -> np.ndarray:
    """bf16 bit patterns [T, K] (row-major: K contiguous)."""
    z = normal(stream_state(seed, TAG_X), T * K).reshape(T, K)
    if outliers:
        z[:, outlier_channels(K, seed)] *= 20.0
    return to_bf16_bits(z)


# The benchmark configurations, by what they are.
WORKLOADS = {
    "q4_512x1024_t8": dict(N=512, K=1024, T=8, scales="halfnormal", outliers=False),
    "q4_6144x5120_t1": dict(N=6144, K=5120, T=1, scales="halfnormal", outliers=False),
    "q4_14336x5120": dict(N=14336, K=5120, T=(1, 16, 128, 1024), scales="lognormal", outliers=True),
    "q4_34816x5120_t1024": dict(N=34816, K=5120, T=1024, scales="halfnormal", outliers=False),
    "q4_5120x17408_t1024": dict(N=5120, K=17408, T=1024, scales="halfnormal", outliers=False),
}

# The 6144x5120 sweep: every T in 1..128 plus the large-T anchors and seams.
SWEEP_6144x5120_T = tuple(range(1, 129)) + (384, 385, 512, 640, 641, 1024)


def make_problem(N: int, K: int, T: int, *, w_seed: int = 0, x_seed: int | None = None,
                 scales: str = "halfnormal", outliers: bool = False):
    """(wq uint8 [N,Kp/2], scales uint16 [N,Kp/64], x uint16 [T,K]), Kp = K rounded up to 128.

    The weight planes are stored for K rounded up to a multiple of 128 (the
    storage layout of the format); for K a multiple of 128 that is K itself.
    The weight is seeded ``w_seed`` (shared across a T sweep); X is seeded
    ``x_seed``, which defaults to T ("one seed per T").
    """
    if x_seed is None:
        x_seed = T
    Kp = (K + 127) // 128 * 128
    wq = packed_codes(N, Kp, w_seed)
    s = group_scales(N, Kp, w_seed, scales)
    x = activations(T, K, x_seed, outliers)
    return wq, s, x


def uniform_bytes(rows: int, cols: int, seed: int, tag: int) -> np.ndarray:
    """uint8 [rows, cols] from the splitmix64 stream of (seed, tag)."""
    nbytes = rows * cols
    words = splitmix64(stream_state(seed, tag), (nbytes + 7) // 8)
    return words.astype("<u8").view(np.uint8)[:nbytes].reshape(rows, cols).copy()


# sibling formats: bits per weight in the high plane (0: W8, one int8 code per weight)
FORMAT_HIGH_BITS = {"q4g64": None, "q5g64": 1, "q6g64": 2, "w8g32": 0}


def make_problem_fmt(qtype: str, N: int, K: int, T: int, *, w_seed: int = 0, x_seed: int | None = None):
    """(planes, scales, x) for a sibling weight format, planes stored for Kp = K rounded
    up to 128 columns: q5g64 / q6g64 (low [N, Kp/2], high [N, Kp*bits/8]), w8g32
    (codes [N, Kp]); uniform bytes in every plane, half-normal fp16 scales per group."""
    if x_seed is None:
        x_seed = T
    Kp = (K + 127) // 128 * 128
    x = activations(T, K, x_seed)
    if qtype == "w8g32":
        return (uniform_bytes(N, Kp, w_seed, TAG_W8),), group_scales(N, Kp, w_seed, group=32), x
    bits = FORMAT_HIGH_BITS[qtype]
    low = packed_codes(N, Kp, w_seed)
    high = uniform_bytes(N, Kp * bits // 8, w_seed, TAG_HIGH)
    return (low, high), group_scales(N, Kp, w_seed), x
