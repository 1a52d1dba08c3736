"""Pins for the CPU FP64 oracle: values the pages print, closed forms,
invariants, exact brute force on tiny inputs, and planted mistakes that the
pins must catch.  No GPU needed."""
import struct
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import q4_oracle as O
from weight_only_bit_q4_gb300 import synth


# ---------------------------------------------------------------- bytes
def test_weight_bytes_printed_values(golden):
    rows = golden("format_bytes.txt")
    assert len(rows) == 2
    for N, K, b, *_ in rows:
        assert oracle.weight_bytes(int(N), int(K)) == int(b)


def test_weight_bytes_closed_form_and_padding():
    # N*K/64*34 when K is a multiple of 128; K is padded to 128 otherwise.
    for N, K in [(512, 1024), (14336, 5120), (34816, 5120), (5120, 17408), (3456, 1152)]:
        assert oracle.weight_bytes(N, K) == N * K // 64 * 34
    assert oracle.weight_bytes(1, 64) == 2 * 34
    assert oracle.weight_bytes(3, 130) == 3 * 256 // 64 * 34


# ---------------------------------------------------------------- decoders
def test_fp16_decoder_special_values():
    cases = {0x3C00: 1.0, 0x0001: 2.0 ** -24, 0x7BFF: 65504.0, 0xC000: -2.0,
             0x0400: 2.0 ** -14, 0x03FF: 1023 * 2.0 ** -24, 0x3555: 0.333251953125,
             0x0000: 0.0, 0x3800: 0.5}
    for bits, v in cases.items():
        assert oracle.fp16_bits_to_f64(bits) == v, hex(bits)
    assert oracle.fp16_bits_to_f64(0x7C00) == np.inf
    assert np.isnan(oracle.fp16_bits_to_f64(0x7E00))


def test_fp16_decoder_all_patterns_vs_struct():
    bits = np.arange(1 << 16, dtype=np.uint16)
    ours = oracle.fp16_bits_to_f64(bits)
    ref = np.array([struct.unpack("<e", struct.pack("<H", int(b)))[0] for b in bits])
    fin = np.isfinite(ref)
    assert np.array_equal(ours[fin], ref[fin])
    assert np.array_equal(np.isnan(ours), np.isnan(ref))


def test_bf16_decoder_all_patterns_vs_float32():
    bits = np.arange(1 << 16, dtype=np.uint32)
    ours = oracle.bf16_bits_to_f64(bits)
    with np.errstate(invalid="ignore"):
        ref = (bits << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    fin = np.isfinite(ref)
    assert np.array_equal(ours[fin], ref[fin])
    assert oracle.bf16_bits_to_f64(0x3F80) == 1.0
    assert oracle.bf16_bits_to_f64(0x4049) == 3.140625
    assert oracle.bf16_bits_to_f64(0x0001) == 2.0 ** -133


# ---------------------------------------------------------------- decode
def test_unpack_all_bytes_against_divmod_table():
    table = [(b % 16, b // 16) for b in range(256)]
    wq = np.arange(256, dtype=np.uint8).reshape(1, 256)
    q = oracle.unpack_codes(wq)[0]
    for b in range(256):
        assert (q[2 * b], q[2 * b + 1]) == table[b]


def test_dequant_hand_example():
    # byte 0x8F: even k -> 15, odd k -> 8; w = (15-8)*s, (8-8)*s.
    wq = np.full((1, 32), 0x8F, dtype=np.uint8)
    for sbits, s in [(0x3C00, 1.0), (0x4000, 2.0), (0x3800, 0.5)]:
        w = oracle.dequantize(wq, np.array([[sbits]], dtype=np.uint16))
        assert np.all(w[0, 0::2] == 7 * s) and np.all(w[0, 1::2] == 0.0)
    # code 0 is the most negative weight
    w = oracle.dequantize(np.zeros((1, 32), np.uint8), np.array([[0x3C00]], np.uint16))
    assert np.all(w == -8.0)


def test_scale_group_boundaries():
    # group g covers k in [64g, 64g+64): distinct scales per group show up exactly there.
    K = 256
    wq = np.full((1, K // 2), 0x99, dtype=np.uint8)           # q = 9 everywhere -> w = s
    sbits = np.array([[0x3C00, 0x4000, 0x4200, 0x4400]], np.uint16)  # 1, 2, 3, 4
    w = oracle.dequantize(wq, sbits)[0]
    for k in range(K):
        assert w[k] == float(k // 64 + 1)


# ---------------------------------------------------------------- invariants
def _rand_problem(N, K, T, seed):
    return synth.make_problem(N, K, T, w_seed=seed, x_seed=seed + 1)


def test_all_codes_eight_gives_exact_zero():
    _, s, x = _rand_problem(17, 256, 5, 3)
    wq = np.full((17, 128), 0x88, dtype=np.uint8)
    y = oracle.linear(wq, s, x)
    assert np.all(y == 0.0)


def test_linear_in_each_scale():
    wq, s, x = _rand_problem(9, 384, 4, 5)
    y0 = oracle.linear(wq, s, x)
    n, g = 4, 3
    s2 = s.copy()
    s2[n, g] = s[n, g] + 0x0400          # exponent + 1: exactly doubles a normal fp16
    assert oracle.fp16_bits_to_f64(s2[n, g]) == 2 * oracle.fp16_bits_to_f64(s[n, g])
    y1 = oracle.linear(wq, s2, x)
    # only column n changes, by exactly group g's contribution
    others = [i for i in range(9) if i != n]
    assert np.array_equal(y1[:, others], y0[:, others])
    q = oracle.unpack_codes(wq)[n, 64 * g:64 * g + 64] - 8
    xs = oracle.bf16_bits_to_f64(x)[:, 64 * g:64 * g + 64]
    contrib = (xs * q).sum(axis=1) * oracle.fp16_bits_to_f64(s[n, g])
    np.testing.assert_allclose(y1[:, n] - y0[:, n], contrib, rtol=1e-12, atol=1e-12)


def test_one_hot_x_selects_dequantised_column():
    wq, s, _ = _rand_problem(11, 256, 1, 7)
    K = 256
    for k0 in [0, 1, 63, 64, 127, 200, 255]:
        x = np.zeros((1, K), np.uint16)
        x[0, k0] = 0x3F80                 # bf16 1.0
        y = oracle.linear(wq, s, x)[0]
        byte = wq[:, k0 // 2].astype(int)
        q = np.where(k0 % 2 == 0, byte & 15, byte >> 4)
        assert np.array_equal(y, (q - 8) * oracle.fp16_bits_to_f64(s[:, k0 // 64]))


def test_q9_unit_scale_unit_x_gives_K():
    for K in [128, 1024, 5120]:
        wq = np.full((3, K // 2), 0x99, dtype=np.uint8)
        s = np.full((3, K // 64), 0x3C00, dtype=np.uint16)
        x = np.full((2, K), 0x3F80, dtype=np.uint16)
        assert np.all(oracle.linear(wq, s, x) == float(K))


def test_row_subset_matches_full():
    wq, s, x = _rand_problem(40, 512, 3, 9)
    full = oracle.linear(wq, s, x)
    rows = np.array([0, 7, 39])
    assert np.array_equal(oracle.linear(wq, s, x, rows=rows), full[:, rows])


# ---------------------------------------------------------------- brute force
def _exact_problem(N, K, T, seed):
    rng = np.random.default_rng(seed)
    wq = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    # scales that are exact small dyadics in fp16; x small integers in bf16
    choices = np.array([0x3C00, 0x4000, 0x3800, 0x4200, 0x3400, 0xBC00], np.uint16)  # 1,2,.5,3,.25,-1
    s = choices[rng.integers(0, len(choices), (N, K // 64))]
    xv = rng.integers(-4, 5, (T, K)).astype(np.float32)
    x = ((xv.view(np.uint32) >> 16)).astype(np.uint16)     # exact in bf16
    return wq, s, x


def _exact_reference(wq, s, x):
    """Fractions; decoders from struct (library) rather than the oracle's own."""
    N, half = wq.shape
    K = 2 * half
    T = x.shape[0]
    sv = [[Fraction(struct.unpack("<e", struct.pack("<H", int(b)))[0]) for b in row] for row in s]
    xv = [[Fraction(struct.unpack("<f", struct.pack("<I", int(b) << 16))[0]) for b in row] for row in x]
    out = [[Fraction(0)] * N for _ in range(T)]
    for n in range(N):
        codes = []
        for byte in wq[n]:
            byte = int(byte)
            codes += [byte - 16 * (byte // 16), byte // 16]
        for t in range(T):
            out[t][n] = sum((codes[k] - 8) * sv[n][k // 64] * xv[t][k] for k in range(K))
    return out


@pytest.mark.parametrize("N,K,T", [(1, 128, 1), (3, 128, 2), (8, 256, 3), (3, 256, 1)])
def test_brute_force_tiny_exact(N, K, T):
    wq, s, x = _exact_problem(N, K, T, seed=N * 1000 + K + T)
    ref = _exact_reference(wq, s, x)
    y = oracle.linear(wq, s, x)
    for t in range(T):
        for n in range(N):
            assert Fraction(y[t, n]) == ref[t][n]
    loops = oracle.linear_loops(wq, s, x)
    for t in range(T):
        for n in range(N):
            assert Fraction(loops[t][n]) == ref[t][n]


# ---------------------------------------------------------------- K not a multiple of 128
def _exact_padded_problem(N, K, T, seed):
    """Planes stored for K_pad = align_up(K, 128) columns (linear-benchmark.md section 4).
    The padded codes are random and every wholly padded group gets NaN or Inf scale
    bits, so anything that lets padding into y shows up."""
    rng = np.random.default_rng(seed)
    Kp = (K + 127) // 128 * 128
    wq = rng.integers(0, 256, (N, Kp // 2), dtype=np.uint8)
    choices = np.array([0x3C00, 0x4000, 0x3800, 0x4200, 0x3400, 0xBC00], np.uint16)
    s = choices[rng.integers(0, len(choices), (N, Kp // 64))]
    g_real = (K + 63) // 64
    s[:, g_real:] = np.where(rng.integers(0, 2, (N, Kp // 64 - g_real)) == 0, 0x7E00, 0x7C00)
    xv = rng.integers(-4, 5, (T, K)).astype(np.float32)
    x = ((xv.view(np.uint32) >> 16)).astype(np.uint16)
    return wq, s, x


def _exact_reference_logical(wq, s, x):
    """Fractions over k < K, K = the width of X; struct decoders, plain loops."""
    N = wq.shape[0]
    T, K = x.shape
    xv = [[Fraction(struct.unpack("<f", struct.pack("<I", int(b) << 16))[0]) for b in row] for row in x]
    out = [[Fraction(0)] * N for _ in range(T)]
    for n in range(N):
        sv = [Fraction(struct.unpack("<e", struct.pack("<H", int(b)))[0]) for b in s[n, :(K + 63) // 64]]
        codes = []
        for j in range(K // 2):
            byte = int(wq[n, j])
            codes += [byte % 16, byte // 16]
        for t in range(T):
            out[t][n] = sum((codes[k] - 8) * sv[k // 64] * xv[t][k] for k in range(K))
    return out


@pytest.mark.parametrize("N,K,T", [(2, 8, 1), (3, 72, 2), (4, 200, 2), (1, 136, 3), (2, 64, 2)])
def test_brute_force_padded_k_exact(N, K, T):
    wq, s, x = _exact_padded_problem(N, K, T, seed=N * 977 + K + T)
    ref = _exact_reference_logical(wq, s, x)
    y = oracle.linear(wq, s, x)
    loops = oracle.linear_loops(wq, s, x)
    for t in range(T):
        for n in range(N):
            assert Fraction(y[t, n]) == ref[t][n]
            assert Fraction(loops[t][n]) == ref[t][n]


def test_padding_bits_do_not_enter():
    wq, s, x = _exact_padded_problem(5, 200, 3, seed=11)
    y = oracle.linear(wq, s, x)
    wq2, s2 = wq.copy(), s.copy()
    wq2[:, 100:] = 0        # codes of k >= 200
    s2[:, 4:] = 0           # scales of groups 4.. (k >= 256; group 3 holds k = 192..255)
    assert np.array_equal(oracle.linear(wq2, s2, x), y)
    # K a multiple of 128 stores exactly K columns: unchanged behaviour
    wq3, s3, x3 = _exact_problem(3, 256, 2, seed=5)
    assert oracle.linear(wq3, s3, x3).shape == (2, 3)


# ---------------------------------------------------------------- tolerance
def test_tolerance_definition():
    y_ref = np.array([[1.0, -2.0, 0.0, 4.0]])
    r = np.sqrt((1 + 4 + 0 + 16) / 4)
    # just inside the bound passes, just beyond fails
    bound = 8e-3 * np.abs(y_ref) + 1e-3 * r
    assert oracle.within_tolerance(y_ref + bound * 0.999, y_ref).all()
    assert not oracle.within_tolerance(y_ref + bound * 1.001, y_ref).any()
    assert oracle.rms(y_ref) == pytest.approx(r)


# ---------------------------------------------------------------- planted mistakes
def _mutant_unpack_swapped(wq):
    wq = np.asarray(wq, dtype=np.uint8)
    q = np.empty((wq.shape[0], 2 * wq.shape[1]), np.int64)
    q[:, 0::2] = wq >> 4
    q[:, 1::2] = wq & 15
    return q


def _run_pins_against(monkeypatch, **patches):
    """Run a subset of the pins with the oracle patched; return the names that failed."""
    for name, fn in patches.items():
        monkeypatch.setattr(O, name, fn)
    failed = []
    pins = {
        "hand": test_dequant_hand_example,
        "groups": test_scale_group_boundaries,
        "onehot": test_one_hot_x_selects_dequantised_column,
        "q9": test_q9_unit_scale_unit_x_gives_K,
        "brute": lambda: test_brute_force_tiny_exact(3, 128, 2),
        "zero": test_all_codes_eight_gives_exact_zero,
    }
    for name, pin in pins.items():
        try:
            pin()
        except AssertionError:
            failed.append(name)
    return failed


def test_planted_mistakes_are_caught(monkeypatch):
    orig_dequant = O.dequantize
    mutants = {
        "swapped nibbles": dict(unpack_codes=_mutant_unpack_swapped),
        "zero point 7": dict(dequantize=lambda wq, sb: orig_dequant(wq, sb) + O.fp16_bits_to_f64(sb)[:, np.arange(2 * wq.shape[1]) // 64]),
        "scale index k//32": dict(dequantize=lambda wq, sb: (O.unpack_codes(wq) - 8) * O.fp16_bits_to_f64(sb)[:, np.minimum(np.arange(2 * wq.shape[1]) // 32, sb.shape[1] - 1)]),
        "scale dropped": dict(dequantize=lambda wq, sb: (O.unpack_codes(wq) - 8).astype(np.float64)),
        "sign flipped": dict(dequantize=lambda wq, sb: -orig_dequant(wq, sb)),
    }
    for label, patch in mutants.items():
        with monkeypatch.context() as m:
            failed = _run_pins_against(m, **patch)
        assert failed, f"planted mistake not caught: {label}"


def test_planted_transpose_is_caught():
    wq, s, x = _exact_problem(3, 128, 2, seed=11)
    ref = _exact_reference(wq, s, x)
    y = oracle.linear(wq, s, x)
    assert y.shape == (2, 3)
    bad = (oracle.dequantize(wq, s) @ oracle.bf16_bits_to_f64(x).T)  # [N, T]: the transposed layout
    assert bad.shape != y.shape or any(Fraction(bad[t][n]) != ref[t][n] for t in range(2) for n in range(3))
