"""Pins for the sibling-format oracle (Q5G64, Q6G64, W8G32): the byte counts of the
format table (linear-benchmark.md section 4), bit fields decoded by library routines
the oracle does not use, invariants, exact brute force, and planted mistakes."""
import struct
from fractions import Fraction

import numpy as np
import pytest

from oracle import sibling_formats as sf

FMTS = ["q5g64", "q6g64", "w8g32"]


def test_weight_bytes_per_group_table():
    # 6144 x 5120: 80 groups of 64 per row (42 / 50 bytes each), W8: 160 groups of 32 (34 bytes each)
    assert sf.weight_bytes("q5g64", 6144, 5120) == 6144 * 80 * 42 == 20_643_840
    assert sf.weight_bytes("q6g64", 6144, 5120) == 6144 * 80 * 50 == 24_576_000
    assert sf.weight_bytes("w8g32", 6144, 5120) == 6144 * 160 * 34 == 33_423_360
    # K_pad: 1152 + 0, 4304 -> 4352
    assert sf.weight_bytes("q5g64", 1152, 4304) == 1152 * 68 * 42


def test_high_plane_fields_against_unpackbits():
    v = np.arange(256, dtype=np.uint8).reshape(1, 256)
    bits = np.unpackbits(v, axis=1, bitorder="little").reshape(256, 8)    # bits[i, b] = bit b of byte i
    q5 = sf.unpack_high(v, 1).reshape(256, 8)
    assert np.array_equal(q5, bits)
    q6 = sf.unpack_high(v, 2).reshape(256, 4)
    assert np.array_equal(q6, bits[:, 0::2] + 2 * bits[:, 1::2])


def test_w8_codes_against_struct():
    c = np.arange(256, dtype=np.uint8).reshape(1, 256)
    got = sf.codes("w8g32", (c,)).reshape(256)
    want = [struct.unpack("<b", bytes([i]))[0] for i in range(256)]
    assert got.tolist() == want


def test_q5_q6_codes_span_and_order():
    low = np.array([[0x21, 0x43, 0x00, 0x00]], np.uint8)     # weights 0..7: 1, 2, 3, 4, 0, 0, 0, 0
    high5 = np.array([[0b1010]], np.uint8)                   # weights 1 and 3 get bit 4
    assert sf.codes("q5g64", (low, high5))[0].tolist() == [1, 18, 3, 20, 0, 0, 0, 0]
    high6 = np.array([[0b11_10_01_00, 0b00_00_00_11]], np.uint8)   # weights 0..3: fields 0..3, weight 4: 3
    assert sf.codes("q6g64", (low, high6))[0].tolist() == [1, 18, 35, 52, 48, 0, 0, 0]


def _zero_point_planes(qtype, N, K):
    if qtype == "w8g32":
        return (np.zeros((N, K), np.uint8),)
    bits = 1 if qtype == "q5g64" else 2
    fill = 0xFF if bits == 1 else 0xAA                          # q = 16 / q = 32
    return np.zeros((N, K // 2), np.uint8), np.full((N, K * bits // 8), fill, np.uint8)


@pytest.mark.parametrize("qtype", FMTS)
def test_zero_point_codes_give_exact_zero(qtype):
    N, K, T = 4, 256, 3
    group = 32 if qtype == "w8g32" else 64
    s = np.full((N, K // group), 0x3C00, np.uint16)
    x = np.full((T, K), 0x3F80, np.uint16)                       # 1.0
    assert np.all(sf.linear(qtype, _zero_point_planes(qtype, N, K), s, x) == 0.0)


@pytest.mark.parametrize("qtype", FMTS)
def test_one_hot_x_selects_dequantised_column(qtype):
    from weight_only_bit_q4_gb300 import synth
    planes, s, _ = synth.make_problem_fmt(qtype, 6, 256, 1, w_seed=3)
    w = sf.dequantize(qtype, planes, s)
    for k0 in (0, 31, 32, 63, 64, 200, 255):
        x = np.zeros((1, 256), np.uint16)
        x[0, k0] = 0x3F80
        assert np.array_equal(sf.linear(qtype, planes, s, x)[0], w[:, k0])


# ---------------------------------------------------------------- exact brute force
def _exact_problem(qtype, N, K, T, seed):
    rng = np.random.default_rng(seed)
    Kp = (K + 127) // 128 * 128
    group = 32 if qtype == "w8g32" else 64
    choices = np.array([0x3C00, 0x4000, 0x3800, 0x4200, 0x3400, 0xBC00], np.uint16)
    s = choices[rng.integers(0, len(choices), (N, Kp // group))]
    s[:, (K + group - 1) // group:] = 0x7E00                     # NaN scales in wholly padded groups
    if qtype == "w8g32":
        planes = (rng.integers(0, 256, (N, Kp), dtype=np.uint8),)
    else:
        bits = 1 if qtype == "q5g64" else 2
        planes = (rng.integers(0, 256, (N, Kp // 2), dtype=np.uint8),
                  rng.integers(0, 256, (N, Kp * bits // 8), dtype=np.uint8))
    xv = rng.integers(-4, 5, (T, K)).astype(np.float32)
    x = (xv.view(np.uint32) >> 16).astype(np.uint16)
    return planes, s, x


def _exact_reference(qtype, planes, s, x):
    """Fractions over k < K; struct and unpackbits decoders, plain loops."""
    T, K = x.shape
    N = s.shape[0]
    group = 32 if qtype == "w8g32" else 64
    zero = {"q5g64": 16, "q6g64": 32, "w8g32": 0}[qtype]
    xv = [[Fraction(struct.unpack("<f", struct.pack("<I", int(b) << 16))[0]) for b in row] for row in x]
    out = [[Fraction(0)] * N for _ in range(T)]
    for n in range(N):
        if qtype == "w8g32":
            q = [struct.unpack("<b", bytes([int(b)]))[0] for b in planes[0][n, :K]]
        else:
            bits = 1 if qtype == "q5g64" else 2
            hb = np.unpackbits(planes[1][n:n + 1], axis=1, bitorder="little")[0]
            q = []
            for k in range(K):
                byte = int(planes[0][n, k // 2])
                lo = byte % 16 if k % 2 == 0 else byte // 16
                hi = sum(int(hb[bits * k + i]) << i for i in range(bits))
                q.append(lo + 16 * hi)
        sv = [Fraction(struct.unpack("<e", struct.pack("<H", int(b)))[0]) for b in s[n, :(K + group - 1) // group]]
        for t in range(T):
            out[t][n] = sum((q[k] - zero) * sv[k // group] * xv[t][k] for k in range(K))
    return out


CASES = [(q, N, K, T) for q in FMTS for (N, K, T) in [(2, 128, 1), (3, 256, 2), (2, 72, 2), (3, 200, 1)]]


@pytest.mark.parametrize("qtype,N,K,T", CASES)
def test_brute_force_exact(qtype, N, K, T):
    planes, s, x = _exact_problem(qtype, N, K, T, seed=N * 131 + K + T)
    ref = _exact_reference(qtype, planes, s, x)
    y = sf.linear(qtype, planes, s, x)
    for t in range(T):
        for n in range(N):
            assert Fraction(y[t, n]) == ref[t][n]


# ---------------------------------------------------------------- planted mistakes
def _pins_fail(monkeypatch, qtype, **patch):
    for name, value in patch.items():
        monkeypatch.setattr(sf, name, value)
    try:
        for (q, N, K, T) in CASES:
            if q == qtype:
                test_brute_force_exact(q, N, K, T)
    except AssertionError:
        return True
    return False


def test_planted_mistakes_are_caught(monkeypatch):
    real_high, real_codes = sf.unpack_high, sf.codes
    reversed_bits = lambda high, bits: real_high(high, bits)[:, ::-1]
    with monkeypatch.context() as m:
        assert _pins_fail(m, "q5g64", unpack_high=reversed_bits)
    with monkeypatch.context() as m:
        assert _pins_fail(m, "q6g64", unpack_high=reversed_bits)
    with monkeypatch.context() as m:
        assert _pins_fail(m, "q5g64", FORMATS={**sf.FORMATS, "q5g64": (64, 15, 1)})
    with monkeypatch.context() as m:
        assert _pins_fail(m, "w8g32", codes=lambda q, p: (np.asarray(p[0], np.int64) if q == "w8g32"
                                                          else real_codes(q, p)))
    with monkeypatch.context() as m:   # high bits placed below the low nibble
        assert _pins_fail(m, "q6g64", codes=lambda q, p: (sf.unpack_low(p[0]) << 2 | sf.unpack_high(p[1], 2))
                          if q == "q6g64" else real_codes(q, p))
