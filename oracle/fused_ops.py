"""CPU FP64 oracle for the fused operations next to the Q4 linear layer.

TEST INFRASTRUCTURE ONLY, like the rest of this package: only the tests, the
smoke check and the benchmark's CPU legs may use it, and it shares no code
with the CUDA library.

The linear-benchmark page names three fused operations that its pure Linear
benchmark leaves to their own benchmarks (section "status and scope": Q4/Q5/Q6/W8
LinearAdd, LinearSwiGLU and LinearPair), and lists the 34816 x 5120 weight as the
MLP gate/up parent.  The pages define none of them.  Readings (the plainest the
names and that geometry support):

* LinearAdd:  Y = W . X + R, R a bf16 residual with Y's shape [T, N] (the add is
  part of the same FP32 result before the one bf16 rounding of Y).
* LinearSwiGLU:  one packed weight of 2F rows, the first F the gate projection and
  the next F the up projection (34816 = 2 x 17408, the MLP width that the
  5120 x 17408 down projection consumes); Y[t, f] = silu(g[t, f]) * u[t, f] with
  g = W[:F] . X, u = W[F:] . X and silu(z) = z / (1 + e^-z).  Y is [T, F].
* LinearPair:  two weights applied to one X in one call, (W_a . X, W_b . X).

All in FP64 from the decoded operands of q4_oracle.
"""
from __future__ import annotations

import numpy as np

from . import q4_oracle


def silu(z: np.ndarray) -> np.ndarray:
    """z / (1 + e^-z) in FP64, written so that neither branch overflows."""
    z = np.asarray(z, dtype=np.float64)
    out = np.empty_like(z)
    pos = z >= 0
    out[pos] = z[pos] / (1.0 + np.exp(-z[pos]))
    e = np.exp(z[~pos])                       # z < 0: z e^z / (1 + e^z)
    out[~pos] = z[~pos] * e / (1.0 + e)
    return out


def linear_add(wq: np.ndarray, scale_bits: np.ndarray, x_bits: np.ndarray, r_bits: np.ndarray) -> np.ndarray:
    """LinearAdd: y_ref [T, N] = W . X + R in FP64 (R bf16 bits [T, N])."""
    y = q4_oracle.linear(wq, scale_bits, x_bits)
    r = q4_oracle.bf16_bits_to_f64(np.asarray(r_bits))
    assert r.shape == y.shape, (r.shape, y.shape)
    return y + r


def linear_swiglu(wq: np.ndarray, scale_bits: np.ndarray, x_bits: np.ndarray) -> np.ndarray:
    """LinearSwiGLU: y_ref [T, F] = silu(gate) * up, gate = rows [0, F), up = rows [F, 2F)."""
    n2 = np.asarray(wq).shape[0]
    assert n2 % 2 == 0, n2
    f = n2 // 2
    y = q4_oracle.linear(wq, scale_bits, x_bits)
    return silu(y[:, :f]) * y[:, f:]


def linear_pair(wq_a, scale_bits_a, wq_b, scale_bits_b, x_bits):
    """LinearPair: (W_a . X, W_b . X), each y_ref [T, N_a] / [T, N_b] in FP64."""
    return (q4_oracle.linear(wq_a, scale_bits_a, x_bits),
            q4_oracle.linear(wq_b, scale_bits_b, x_bits))
