"""Pins for the fused-operation oracle (LinearAdd, LinearSwiGLU, LinearPair): identities
of the SiLU, a library logistic function the oracle does not use, exact brute force
on integer-valued inputs, the packing of the gate/up weight, and planted mistakes."""
import math
import struct
from fractions import Fraction

import numpy as np
import pytest
from scipy.special import expit

import oracle
from oracle import fused_ops as fo
from weight_only_bit_q4_gb300 import synth


# ---------------------------------------------------------------- SiLU
def test_silu_against_library_logistic():
    z = np.concatenate([np.linspace(-60, 60, 2401), [0.0, -1e-300, 1e-300, 700.0, -700.0]])
    want = z * expit(z)
    got = fo.silu(z)
    assert np.all(np.isfinite(got))
    assert np.allclose(got, want, rtol=1e-15, atol=1e-300)


def test_silu_identities():
    z = np.linspace(-30, 30, 601)
    # silu(z) - silu(-z) = z (sigma(z) + sigma(-z) = 1)
    assert np.allclose(fo.silu(z) - fo.silu(-z), z, rtol=0, atol=1e-13)
    assert fo.silu(np.array([0.0]))[0] == 0.0
    # slope 1/2 at 0, and silu(z) -> z for large z, -> 0 from below for very negative z
    h = 1e-8
    assert fo.silu(np.array([h]))[0] / h == pytest.approx(0.5, abs=1e-8)
    assert fo.silu(np.array([40.0]))[0] == pytest.approx(40.0, rel=1e-16, abs=1e-15)
    v = fo.silu(np.array([-40.0]))[0]
    assert v < 0 and v == pytest.approx(-40.0 * math.exp(-40.0), rel=1e-12)
    # the minimum: silu'(z) = 0 near z = -1.27846, value about -0.27846
    zz = np.linspace(-1.4, -1.15, 250001)
    i = int(np.argmin(fo.silu(zz)))
    assert zz[i] == pytest.approx(-1.27846, abs=1e-4)
    assert fo.silu(zz)[i] == pytest.approx(-0.27846, abs=1e-4)


# ---------------------------------------------------------------- exact brute force
def _int_problem(N, K, T, seed):
    """Scales in {1, 2, 1/2, -1}, x and r small integers: every sum is exact in FP64."""
    rng = np.random.default_rng(seed)
    wq = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    s = np.array([0x3C00, 0x4000, 0x3800, 0xBC00], np.uint16)[rng.integers(0, 4, (N, K // 64))]
    x = (rng.integers(-4, 5, (T, K)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    r = (rng.integers(-50, 51, (T, N)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    return wq, s, x, r


def _bits_f(b, fmt):
    if fmt == "e":
        return Fraction(struct.unpack("<e", struct.pack("<H", int(b)))[0])
    return Fraction(struct.unpack("<f", struct.pack("<I", int(b) << 16))[0])


def _exact_linear(wq, s, x):
    N, T, K = wq.shape[0], x.shape[0], x.shape[1]
    out = [[Fraction(0)] * N for _ in range(T)]
    for n in range(N):
        q = [(int(wq[n, k // 2]) >> (4 * (k % 2))) & 15 for k in range(K)]
        for t in range(T):
            out[t][n] = sum((q[k] - 8) * _bits_f(s[n, k // 64], "e") * _bits_f(x[t, k], "b") for k in range(K))
    return out


@pytest.mark.parametrize("N,K,T", [(3, 128, 2), (5, 256, 1), (2, 192, 3)])
def test_linear_add_exact(N, K, T):
    wq, s, x, r = _int_problem(N, K, T, seed=N * 7 + K + T)
    ref = _exact_linear(wq, s, x)
    y = fo.linear_add(wq, s, x, r)
    for t in range(T):
        for n in range(N):
            assert Fraction(y[t, n]) == ref[t][n] + _bits_f(r[t, n], "b")


def test_linear_add_zero_residual_is_linear():
    wq, s, x = synth.make_problem(40, 1152, 7, w_seed=2)
    r = np.zeros((7, 40), np.uint16)
    assert np.array_equal(fo.linear_add(wq, s, x, r), oracle.linear(wq, s, x))


# ---------------------------------------------------------------- gate/up packing
def test_swiglu_one_hot_selects_gate_and_up_columns():
    F, K = 6, 256
    wq, s, _ = synth.make_problem(2 * F, K, 1, w_seed=5)
    w = oracle.dequantize(wq, s)                      # [2F, K], rows 0..F-1 gate, F..2F-1 up
    for k0 in (0, 63, 64, 200, 255):
        x = np.zeros((1, K), np.uint16)
        x[0, k0] = 0x3F80                             # 1.0
        want = [float(w[f, k0]) * float(expit(w[f, k0])) * float(w[F + f, k0]) for f in range(F)]
        assert np.allclose(fo.linear_swiglu(wq, s, x)[0], want, rtol=1e-15, atol=0)


def test_swiglu_with_unit_up_half_is_silu_of_gate():
    # up half all q = 9 with scale 1 and x one-hot: u = 1, so y = silu(g)
    F, K = 4, 128
    wq, s, _ = synth.make_problem(2 * F, K, 1, w_seed=6)
    wq[F:] = 0x99
    s[F:] = 0x3C00
    x = np.zeros((1, K), np.uint16)
    x[0, 7] = 0x3F80
    g = oracle.dequantize(wq, s)[:F, 7]
    assert np.allclose(fo.linear_swiglu(wq, s, x)[0], g * expit(g), rtol=1e-15, atol=0)


# ---------------------------------------------------------------- pair
def test_pair_is_two_linears():
    wa, sa, x = synth.make_problem(33, 512, 5, w_seed=1)
    wb, sb, _ = synth.make_problem(70, 512, 5, w_seed=2)
    ya, yb = fo.linear_pair(wa, sa, wb, sb, x)
    assert np.array_equal(ya, oracle.linear(wa, sa, x)) and np.array_equal(yb, oracle.linear(wb, sb, x))
    ya2, yb2 = fo.linear_pair(wa, sa, wa, sa, x)
    assert np.array_equal(ya2, yb2)


# ---------------------------------------------------------------- planted mistakes
def test_planted_mistakes_are_caught(monkeypatch):
    # gate and up halves swapped
    with monkeypatch.context() as m:
        real = oracle.linear
        m.setattr(fo, "linear_swiglu", lambda wq, s, x: fo.silu(real(wq, s, x)[:, wq.shape[0] // 2:])
                  * real(wq, s, x)[:, :wq.shape[0] // 2])
        with pytest.raises(AssertionError):
            test_swiglu_one_hot_selects_gate_and_up_columns()
    # sigmoid in place of silu
    with monkeypatch.context() as m:
        m.setattr(fo, "silu", lambda z: expit(np.asarray(z, np.float64)))
        with pytest.raises(AssertionError):
            test_silu_against_library_logistic()
    # residual dropped
    with monkeypatch.context() as m:
        m.setattr(fo, "linear_add", lambda wq, s, x, r: oracle.linear(wq, s, x))
        with pytest.raises(AssertionError):
            test_linear_add_exact(3, 128, 2)
