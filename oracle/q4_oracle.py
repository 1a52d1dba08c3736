"""CPU FP64 oracle for the Q4_G64_FP16 weight-only linear layer.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import or call this
module; only the tests, the smoke check and the benchmark's CPU-baseline /
reference leg do.  It shares no code with the CUDA library (no kernels, no
headers, no tables, no helpers) and imports nothing from it.

What it computes (plain definitions, no blocking, fusion or reordering):

    y[t, n] = sum_k  w[n, k] * x[t, k]                   (FP64)
    w[n, k] = (q[n, k] - 8) * s[n, floor(k / 64)]

* Weight format "Q4G64_F16S", called Q4_G64_FP16 row-split in the Q4 linear
  measurement report (q4-linear.md, header table): 4-bit codes, groups of 64
  consecutive weights along K, one FP16 scale per group, 32 code bytes +
  2 scale bytes = 34 bytes per group (linear-benchmark.md, section 4
  "theoretical traffic", format table).  The pages do not fix nibble order or
  zero point; the layer's specification does: codes are stored as [N, K/2]
  bytes with element 2j in the low nibble and 2j+1 in the high nibble, the
  scales as a separate [N, K/64] FP16 plane, and w = (q - 8) * s.
* X is BF16 [T, K] row-major (the report's X[K, T] with K contiguous), Y is
  [T, N] row-major.  The result is exact up to FP64 rounding; the GPU path is
  accepted when |y - y_ref| <= 8e-3 |y_ref| + 1e-3 rms(y_ref), with rms taken
  over the whole output (the report's test paragraph: independent decode of
  codes and scales, FP64 matmul as the oracle, full-output check).

The FP16 and BF16 decoders below work from the bit fields (sign, exponent,
mantissa) and do not rely on any library half-precision type.

Parity pins: every function here is pinned by tests/test_oracle_pins.py
against values the pages print (byte counts), closed forms, invariants and
exact brute force on tiny integer-valued inputs.
"""
from __future__ import annotations

import numpy as np

GROUP = 64            # weights per scale group along K
ZERO_POINT = 8        # w = (q - 8) * s
CODE_BYTES_PER_GROUP = GROUP // 2
SCALE_BYTES_PER_GROUP = 2


# --------------------------------------------------------------------------
# Format bookkeeping (linear-benchmark.md, section 4: K_pad, groups, bytes)
# --------------------------------------------------------------------------
def k_pad(K: int) -> int:
    """K rounded up to a multiple of 128 (linear-benchmark.md section 4)."""
    return (K + 127) // 128 * 128


def weight_bytes(N: int, K: int) -> int:
    """Bytes of the code plane plus the scale plane: groups * (32 + 2)."""
    groups = N * k_pad(K) // GROUP
    return groups * (CODE_BYTES_PER_GROUP + SCALE_BYTES_PER_GROUP)


# --------------------------------------------------------------------------
# Bit-pattern decoders
# --------------------------------------------------------------------------
def fp16_bits_to_f64(bits) -> np.ndarray:
    """IEEE-754 binary16 bit patterns -> float64 (sign, 5-bit exponent, 10-bit mantissa)."""
    b = np.asarray(bits, dtype=np.int64) & 0xFFFF
    sign = np.where((b >> 15) & 1, -1.0, 1.0)
    e = (b >> 10) & 0x1F
    m = (b & 0x3FF).astype(np.float64)
    normal = (1.0 + m / 1024.0) * np.exp2(e.astype(np.float64) - 15.0)
    subnormal = m * 2.0 ** -24
    special = np.where(m == 0, np.inf, np.nan)
    out = np.where(e == 0, subnormal, np.where(e == 31, special, normal))
    return sign * out


def bf16_bits_to_f64(bits) -> np.ndarray:
    """bfloat16 bit patterns -> float64 (sign, 8-bit exponent, 7-bit mantissa)."""
    b = np.asarray(bits, dtype=np.int64) & 0xFFFF
    sign = np.where((b >> 15) & 1, -1.0, 1.0)
    e = (b >> 7) & 0xFF
    m = (b & 0x7F).astype(np.float64)
    normal = (1.0 + m / 128.0) * np.exp2(e.astype(np.float64) - 127.0)
    subnormal = m * 2.0 ** -133
    special = np.where(m == 0, np.inf, np.nan)
    out = np.where(e == 0, subnormal, np.where(e == 255, special, normal))
    return sign * out


# --------------------------------------------------------------------------
# Decode and dequantise
# --------------------------------------------------------------------------
def unpack_codes(wq: np.ndarray) -> np.ndarray:
    """uint8 [N, K/2] -> int64 codes q [N, K]; byte j holds q[2j] (low) and q[2j+1] (high)."""
    wq = np.asarray(wq, dtype=np.uint8)
    N, half = wq.shape
    q = np.empty((N, 2 * half), dtype=np.int64)
    q[:, 0::2] = wq & 0x0F
    q[:, 1::2] = wq >> 4
    return q


def dequantize(wq: np.ndarray, scale_bits: np.ndarray) -> np.ndarray:
    """FP64 weights w[n, k] = (q[n, k] - 8) * s[n, k // 64] for every k the code plane holds
    (the last group may be partial: ceil(K / 64) scales for K codes)."""
    q = unpack_codes(wq)
    N, K = q.shape
    s = fp16_bits_to_f64(scale_bits)
    assert s.shape == (N, (K + GROUP - 1) // GROUP), (s.shape, N, K)
    group_of_k = np.arange(K) // GROUP
    return (q - ZERO_POINT).astype(np.float64) * s[:, group_of_k]


def logical_planes(wq: np.ndarray, scale_bits: np.ndarray, K: int):
    """The part of the stored planes that holds W[:, :K].

    The planes are stored for K_pad = k_pad(K) columns (linear-benchmark.md
    section 4: groups = N * K_pad / 64); the positions k >= K are padding, not
    part of W, and whatever bits they hold never enter y.  Planes stored for
    exactly K columns (K a multiple of 128, or a caller that did not pad) are
    accepted as they are.
    """
    wq = np.asarray(wq)
    scale_bits = np.asarray(scale_bits)
    assert K % 2 == 0 and 2 * wq.shape[1] in (K, k_pad(K)), (wq.shape, K)
    return wq[:, :K // 2], scale_bits[:, :(K + GROUP - 1) // GROUP]


def linear(wq: np.ndarray, scale_bits: np.ndarray, x_bits: np.ndarray,
           rows: np.ndarray | None = None) -> np.ndarray:
    """y_ref [T, N] (or [T, len(rows)] for a row subset) in FP64.

    ``x_bits`` is bf16 bit patterns [T, K].  The contraction over K is one
    library matmul in FP64 on independently decoded operands.
    """
    if rows is not None:
        wq = np.asarray(wq)[rows]
        scale_bits = np.asarray(scale_bits)[rows]
    x = bf16_bits_to_f64(x_bits)                 # [T, K]
    wq, scale_bits = logical_planes(wq, scale_bits, x.shape[1])
    w = dequantize(wq, scale_bits)               # [N, K]
    assert x.shape[1] == w.shape[1]
    return x @ w.T                               # [T, N]


def linear_loops(wq, scale_bits, x_bits) -> list:
    """The same definition as plain Python loops (tiny shapes only); the sum runs over the
    K columns of X, so padded plane positions never enter."""
    wq = np.asarray(wq)
    x = bf16_bits_to_f64(x_bits)
    N = wq.shape[0]
    K = x.shape[1]
    s = fp16_bits_to_f64(scale_bits)
    T = x.shape[0]
    y = [[0.0] * N for _ in range(T)]
    for t in range(T):
        for n in range(N):
            acc = 0.0
            for k in range(K):
                byte = int(wq[n, k // 2])
                q = byte % 16 if k % 2 == 0 else byte // 16
                acc += (q - ZERO_POINT) * float(s[n, k // GROUP]) * float(x[t, k])
            y[t][n] = acc
    return y


# --------------------------------------------------------------------------
# Acceptance
# --------------------------------------------------------------------------
REL_TOL = 8e-3
RMS_TOL = 1e-3


def rms(y_ref: np.ndarray) -> float:
    y_ref = np.asarray(y_ref, dtype=np.float64)
    return float(np.sqrt(np.mean(y_ref * y_ref))) if y_ref.size else 0.0


def within_tolerance(y: np.ndarray, y_ref: np.ndarray, rms_ref: float | None = None) -> np.ndarray:
    """Elementwise |y - y_ref| <= 8e-3 |y_ref| + 1e-3 rms(y_ref)."""
    y = np.asarray(y, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    if rms_ref is None:
        rms_ref = rms(y_ref)
    return np.abs(y - y_ref) <= REL_TOL * np.abs(y_ref) + RMS_TOL * rms_ref


def check(y_bits: np.ndarray, y_ref: np.ndarray, rms_ref: float | None = None) -> dict:
    """Compare bf16 output bits with y_ref; returns a summary dict (ok, n_bad, worst)."""
    y = bf16_bits_to_f64(y_bits)
    ok = within_tolerance(y, y_ref, rms_ref)
    if rms_ref is None:
        rms_ref = rms(y_ref)
    err = np.abs(y - np.asarray(y_ref, dtype=np.float64))
    bound = REL_TOL * np.abs(y_ref) + RMS_TOL * rms_ref
    ratio = err / np.maximum(bound, 1e-300)
    worst = int(np.argmax(ratio)) if ratio.size else -1
    return dict(ok=bool(ok.all()), n_bad=int((~ok).sum()), size=int(ok.size),
                worst_ratio=float(ratio.reshape(-1)[worst]) if ratio.size else 0.0,
                nonfinite=int((~np.isfinite(y)).sum()), rms=rms_ref)
