"""GPU parity of the streaming warp-MMA route (Q4LIN_ROUTE_STREAM_MMA) against the FP64 oracle.

The route feeds the tensor cores exact operands: each nibble becomes the fp16
subnormal q * 2^-24 (or 16 q * 2^-24), X is taken per token at a power of two in
fp16, and the group scale and zero point are applied to FP32 partial sums.  It is
held to the layer's own bound, |y - y_ref| <= 8e-3 |y_ref| + 1e-3 rms(y_ref),
including operands far outside fp16's range, every token count through the passes
of 32 tokens, and the row bands, chunks and sub-boxes of its shared-memory plan.
"""
import numpy as np
import pytest

import oracle
from weight_only_bit_q4_gb300 import q4lin, synth

from gpu_util import assert_close, reference, to_dev, torch, weights, x_to_dev, y_bits

pytestmark = pytest.mark.gpu

R = q4lin.ROUTE_STREAM_MMA


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from weight_only_bit_q4_gb300 import build
    build.build()
    q4lin.load()
    assert q4lin.clear_device_status() == 0
    yield
    assert q4lin.device_status() == 0


def run(d, route=R):
    y = q4lin.linear(*d, route=route)
    torch().cuda.synchronize()
    return y_bits(y)


def test_every_token_count_6144x5120():
    # 1..40 tokens: one, two, three and four token tiles, then passes of 32
    wq, s, w = weights(6144, 5120)
    wq_d, s_d, _ = to_dev(wq, s, np.zeros((1, 5120), np.uint16))
    for T in list(range(1, 41)) + [63, 64, 65, 100]:
        x = synth.activations(T, 5120, T)
        assert_close(run((wq_d, s_d, x_to_dev(x))), reference(w, x), f"stream_mma T={T}")


def test_library_routes_small_token_counts_here():
    for T in range(2, 33):
        assert q4lin.select_route(6144, 5120, T) == R, T
    assert q4lin.workspace_bytes(6144, 5120, 8) > 0


@pytest.mark.parametrize("N,K,T", [(1, 8, 1), (7, 72, 3), (8, 128, 8), (33, 1152, 9), (129, 640, 16),
                                   (1000, 384, 24), (300, 17408, 5), (10, 65536, 2), (4097, 512, 31),
                                   (2000, 5120, 32), (153, 1152, 33), (999, 8192, 12)])
def test_shapes(N, K, T):
    wq, s, x = synth.make_problem(N, K, T, w_seed=N + K, x_seed=T)
    assert_close(run(to_dev(wq, s, x)), oracle.linear(wq, s, x), f"stream_mma {N}x{K} T={T}")


@pytest.mark.parametrize("N,K,T", [(14336, 5120, 16), (34816, 5120, 8), (5120, 17408, 8)])
def test_benchmark_geometries(N, K, T):
    dist = "lognormal" if N == 14336 else "halfnormal"
    wq, s, w = weights(N, K, 0, dist)
    x = synth.activations(T, K, T, outliers=(N == 14336))
    assert_close(run(to_dev(wq, s, x)), reference(w, x), f"stream_mma {N}x{K} T={T}")


def test_draft_head_sampled_rows():
    # 131072 rows: several row bands per CTA; oracle on sampled rows
    N, K, T = 131072, 5120, 16
    wq = synth.packed_codes(N, K, 5)
    s = synth.group_scales(N, K, 5)
    x = synth.activations(T, K, 6)
    yb = run(to_dev(wq, s, x))
    rows = np.unique(np.concatenate([np.arange(0, 300), np.arange(N - 300, N),
                                     np.linspace(0, N - 1, 1500).astype(np.int64)]))
    y_ref = oracle.linear(wq, s, x, rows=rows)
    assert_close(yb[:, rows], y_ref, "131072x5120 T=16", rms_ref=oracle.rms(y_ref))


def test_operands_outside_fp16_range():
    # rows of very large and of subnormal scales, tokens of very large and very small x
    N, K, T = 512, 1024, 24
    wq, s, x = synth.make_problem(N, K, T, w_seed=7, x_seed=8)
    sf = s.view(np.float16).astype(np.float32)
    sf[:64] *= 3.0e4 / max(float(np.abs(sf[:64]).max()), 1e-30)
    sf[64:128] *= 2.0e-7 / max(float(np.abs(sf[64:128]).max()), 1e-30)
    s = sf.astype(np.float16).view(np.uint16)
    xf = oracle.bf16_bits_to_f64(x).astype(np.float32)
    xf[:8] *= 1.0e6
    xf[8:16] *= 1.0e-30
    x = synth.float32_to_bf16_bits(xf)
    y_ref = oracle.linear(wq, s, x)
    yb = run(to_dev(wq, s, x))
    for lo, hi in ((0, 8), (8, 16), (16, T)):   # each token block against its own rms
        assert_close(yb[lo:hi], y_ref[lo:hi], f"tokens {lo}..{hi - 1}")


def test_tokens_spanning_many_binades():
    # one token whose values run from 1e-20 to 1e4: bf16 -> fp16 at the token's power of two
    # keeps every value that matters against the token's largest
    K = 2048
    wq, s, x = synth.make_problem(256, K, 3, w_seed=9, x_seed=10)
    xf = oracle.bf16_bits_to_f64(x).astype(np.float32)
    xf[0] *= np.logspace(-20, 4, K).astype(np.float32)
    x = synth.float32_to_bf16_bits(xf)
    y_ref = oracle.linear(wq, s, x)
    yb = run(to_dev(wq, s, x))
    assert_close(yb[:1], y_ref[:1], "wide token")
    assert_close(yb[1:], y_ref[1:], "plain tokens")


def test_deterministic_guarded_and_inputs_preserved():
    t = torch()
    N, K, T = 3000, 2048, 19
    wq, s, x = synth.make_problem(N, K, T, w_seed=12, x_seed=13)
    d = to_dev(wq, s, x)
    before = [a.clone() for a in d]
    pad = 4096
    buf = t.full((pad + T * N + pad,), -3.0, dtype=t.bfloat16, device="cuda")
    y = buf[pad:pad + T * N].view(T, N)
    q4lin.linear(*d, y=y, route=R)
    t.cuda.synchronize()
    a = y_bits(y)
    assert bool((buf[:pad] == -3.0).all()) and bool((buf[pad + T * N:] == -3.0).all())
    for u, v in zip(before, d):
        assert t.equal(u, v)
    assert np.array_equal(a, run(d))
    assert_close(a, oracle.linear(wq, s, x), "guarded")


def test_needs_its_workspace():
    t = torch()
    wq, s, x = synth.make_problem(1024, 2048, 8, w_seed=3, x_seed=4)
    d = to_dev(wq, s, x)
    y = t.empty((8, 1024), dtype=t.bfloat16, device="cuda")
    assert q4lin.workspace_bytes(1024, 2048, 8, R) > 0
    st = q4lin.linear_raw(*(q4lin._ptr(a) for a in d), q4lin._ptr(y), 1024, 2048, 8, None, None, R)
    assert st == 4  # Q4LIN_ERR_WORKSPACE
