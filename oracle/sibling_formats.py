"""CPU FP64 oracle for the sibling weight formats Q5G64, Q6G64 and W8G32.

TEST INFRASTRUCTURE ONLY, like the rest of this package: only the tests, the
smoke check and the benchmark's CPU legs may use it, and it shares no code
with the CUDA library.

The formats are the other rows of the format table of linear-benchmark.md,
section 4 ("theoretical traffic"), which fixes their group sizes and bytes
per group, and nothing else:

    Q5G64_F16S   64 weights: 32 low bytes + 8 high bytes + 2 scale bytes = 42
    Q6G64_F16S   64 weights: 32 low bytes + 16 high bytes + 2 scale bytes = 50
    W8G32_F16S   32 weights: 32 code bytes + 2 scale bytes = 34

Readings (the plainest ones the table and the Q4 format support):

* Planes are separate and row-major, stored for K_pad = align_up(K, 128)
  columns like Q4 (groups = N * K_pad / group size); plane positions k >= K
  are padding and never enter y.
* Q5/Q6: the low plane is the Q4 code plane (weight 2j in the low nibble of
  byte j, 2j+1 in the high nibble).  The high plane holds the remaining bits
  of every weight in k order from the least significant bit of each byte:
  Q5, 1 bit per weight, weight 8i + b in bit b of byte i; Q6, 2 bits per
  weight, weight 4i + b in bits 2b..2b+1 of byte i.  q = low | high << 4.
* Zero points are the middle code, as Q4's 8 is for 4 bits: w = (q - 16) * s
  for Q5, w = (q - 32) * s for Q6.
* W8: one signed (two's complement) int8 code per weight, w = code * s, with
  one FP16 scale per 32 consecutive weights.

y[t, n] = sum_{k<K} w[n, k] x[t, k] in FP64, X bf16 [T, K] as for Q4.
"""
from __future__ import annotations

import numpy as np

from .q4_oracle import bf16_bits_to_f64, fp16_bits_to_f64, k_pad

# qtype -> (group size, zero point, bits in the high plane per weight)
FORMATS = {
    "q5g64": (64, 16, 1),
    "q6g64": (64, 32, 2),
    "w8g32": (32, 0, 0),
}
BYTES_PER_GROUP = {"q4g64": 34, "q5g64": 42, "q6g64": 50, "w8g32": 34}


def weight_bytes(qtype: str, N: int, K: int) -> int:
    """Bytes of all planes: groups * bytes per group, groups = N * K_pad / group size."""
    group = 32 if qtype == "w8g32" else 64
    return N * k_pad(K) // group * BYTES_PER_GROUP[qtype]


def unpack_low(low: np.ndarray) -> np.ndarray:
    """uint8 [N, K/2] -> low 4 bits [N, K] (weight 2j: low nibble of byte j)."""
    low = np.asarray(low, dtype=np.uint8)
    q = np.empty((low.shape[0], 2 * low.shape[1]), dtype=np.int64)
    q[:, 0::2] = low & 0x0F
    q[:, 1::2] = low >> 4
    return q


def unpack_high(high: np.ndarray, bits: int) -> np.ndarray:
    """uint8 [N, K * bits / 8] -> high fields [N, K]: weight (8 / bits) i + b in bits
    bits*b .. bits*b + bits - 1 of byte i."""
    high = np.asarray(high, dtype=np.int64)
    per_byte = 8 // bits
    mask = (1 << bits) - 1
    fields = [(high >> (bits * b)) & mask for b in range(per_byte)]
    out = np.stack(fields, axis=-1)                  # [N, bytes, per_byte]
    return out.reshape(high.shape[0], -1)


def codes(qtype: str, planes: tuple) -> np.ndarray:
    """Integer codes q [N, K] of the stored columns (W8: the signed int8 values)."""
    if qtype == "w8g32":
        (c,) = planes
        return np.asarray(c, dtype=np.uint8).view(np.int8).astype(np.int64)
    _, _, bits = FORMATS[qtype]
    low, high = planes
    return unpack_low(low) | (unpack_high(high, bits) << 4)


def logical(qtype: str, planes: tuple, scale_bits: np.ndarray, K: int):
    """The plane parts that hold W[:, :K] (planes stored for K or K_pad columns)."""
    group, _, bits = FORMATS[qtype]
    scale_bits = np.asarray(scale_bits)
    ng = (K + group - 1) // group
    if qtype == "w8g32":
        (c,) = planes
        c = np.asarray(c)
        assert c.shape[1] in (K, k_pad(K)), (c.shape, K)
        return (c[:, :K],), scale_bits[:, :ng]
    low, high = (np.asarray(p) for p in planes)
    assert K % 8 == 0 and 2 * low.shape[1] in (K, k_pad(K)), (low.shape, K)
    assert high.shape[1] * 8 // bits == 2 * low.shape[1], (high.shape, low.shape)
    return (low[:, :K // 2], high[:, :K * bits // 8]), scale_bits[:, :ng]


def dequantize(qtype: str, planes: tuple, scale_bits: np.ndarray) -> np.ndarray:
    """FP64 w[n, k] = (q[n, k] - zero) * s[n, k // group] for every stored column."""
    group, zero, _ = FORMATS[qtype]
    q = codes(qtype, planes)
    N, K = q.shape
    s = fp16_bits_to_f64(scale_bits)
    assert s.shape == (N, (K + group - 1) // group), (s.shape, N, K)
    return (q - zero).astype(np.float64) * s[:, np.arange(K) // group]


def linear(qtype: str, planes: tuple, scale_bits: np.ndarray, x_bits: np.ndarray,
           rows: np.ndarray | None = None) -> np.ndarray:
    """y_ref [T, N] (or [T, len(rows)]) in FP64; one library matmul on decoded operands."""
    if rows is not None:
        planes = tuple(np.asarray(p)[rows] for p in planes)
        scale_bits = np.asarray(scale_bits)[rows]
    x = bf16_bits_to_f64(x_bits)
    planes, scale_bits = logical(qtype, planes, scale_bits, x.shape[1])
    w = dequantize(qtype, planes, scale_bits)
    assert w.shape[1] == x.shape[1]
    return x @ w.T
