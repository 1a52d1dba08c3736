"""GPU parity of the fused operations against the FP64 fused-operation oracle within the
layer's tolerance.  LinearAdd (q4lin_linear_add): Y = W . X + R with the bf16 residual R
added to the FP32 sum before Y's bf16 rounding -- one token to 1024 (the warp-MMA route's
one-launch form up to 8 tokens, the tile route beyond or where that form does not fit),
padded K, a K split across a cluster, the in-place form (R is Y) and K = 0 (Y = R).
LinearSwiGLU and LinearPair (one launch per weight up to 8 tokens) likewise."""
import numpy as np
import pytest

from oracle import fused_ops as fo
from weight_only_bit_q4_gb300 import q4lin, synth

from gpu_util import assert_close, to_dev, torch, x_to_dev, y_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from weight_only_bit_q4_gb300 import build
    build.build()
    q4lin.load()
    assert q4lin.clear_device_status() == 0
    yield
    assert q4lin.device_status() == 0


@pytest.mark.parametrize("N,K,T", [(6144, 5120, 1), (1000, 1152, 37), (640, 4304, 300), (77, 17408, 8),
                                   (6144, 5120, 1024), (6144, 5120, 8), (333, 640, 7), (129, 1160, 2),
                                   (1000, 2048, 5), (34816, 5120, 4)])
def test_linear_add_matches_oracle(N, K, T):
    t = torch()
    wq, s, x = synth.make_problem(N, K, T, w_seed=N + 2, x_seed=K + T)
    r = synth.activations(T, N, seed=T + 11)           # bf16 residual [T, N]
    d = to_dev(wq, s, x)
    r_d = x_to_dev(r)
    y = q4lin.linear_add(*d, r_d)
    t.cuda.synchronize()
    y_ref = fo.linear_add(wq, s, x, r)
    assert_close(y_bits(y), y_ref, f"LinearAdd {N}x{K} T={T}")
    # in place: R is Y
    y2 = r_d.clone()
    q4lin.linear_add(*d, y2, y=y2)
    t.cuda.synchronize()
    assert np.array_equal(y_bits(y2), y_bits(y))


def test_fused_ops_routes():
    # up to 8 tokens the one-launch warp-MMA form where its whole-K operands fit, the tile route otherwise
    assert q4lin.fused_route("add", 6144, 5120, 8) == q4lin.ROUTE_STREAM_MMA
    assert q4lin.fused_route("add", 6144, 5120, 1) == q4lin.ROUTE_STREAM_MMA
    assert q4lin.fused_route("add", 6144, 5120, 9) == q4lin.ROUTE_TC_SPLITK
    assert q4lin.fused_route("add", 77, 17408, 8) == q4lin.ROUTE_TC_SPLITK    # 278 KB of operands
    assert q4lin.fused_route("pair", 6144, 5120, 8) == q4lin.ROUTE_STREAM_MMA
    assert q4lin.fused_route("swiglu", 17408, 5120, 8) == q4lin.ROUTE_STREAM_MMA
    assert q4lin.fused_route("swiglu", 17408, 5120, 9) == q4lin.ROUTE_TC_SPLITK


def test_linear_add_empty_k_copies_the_residual():
    t = torch()
    r = x_to_dev(synth.activations(3, 64, seed=5))
    y = t.zeros((3, 64), dtype=t.bfloat16, device="cuda")
    st = q4lin.load().q4lin_linear_add(None, None, None, q4lin._ptr(r), q4lin._ptr(y), 64, 0, 3, None)
    t.cuda.synchronize()
    assert st == 0 and t.equal(y.view(t.int16), r.view(t.int16))


@pytest.mark.parametrize("F,K,T", [(64, 128, 1), (100, 1152, 37), (5, 72, 17), (300, 4304, 8), (2176, 5120, 300),
                                   (17408, 5120, 1024), (129, 17408, 3), (17408, 5120, 8), (1000, 2048, 5),
                                   (3, 8, 2), (500, 1160, 1)])
def test_linear_swiglu_matches_oracle(F, K, T):
    """LinearSwiGLU on a 2F-row gate/up weight (34816 x 5120 at T = 1024 among them):
    y = silu(gate) * up in FP32 before the bf16 rounding, held to the layer's bound."""
    t = torch()
    wq, s, x = synth.make_problem(2 * F, K, T, w_seed=F + 5, x_seed=K + T)
    d = to_dev(wq, s, x)
    y = q4lin.linear_swiglu(*d)
    t.cuda.synchronize()
    assert tuple(y.shape) == (T, F)
    assert_close(y_bits(y), fo.linear_swiglu(wq, s, x), f"LinearSwiGLU F={F} K={K} T={T}")
    assert np.array_equal(y_bits(q4lin.linear_swiglu(*d)), y_bits(y))   # deterministic


def test_linear_swiglu_guard_bands():
    t = torch()
    F, K, T = 200, 1024, 40
    wq, s, x = synth.make_problem(2 * F, K, T, w_seed=3, x_seed=4)
    pad = 2048
    buf = t.full((pad + T * F + pad,), -3.0, dtype=t.bfloat16, device="cuda")
    y = buf[pad:pad + T * F].view(T, F)
    q4lin.linear_swiglu(*to_dev(wq, s, x), y=y)
    t.cuda.synchronize()
    assert bool((buf[:pad] == -3.0).all()) and bool((buf[pad + T * F:] == -3.0).all())
    assert_close(y_bits(y), fo.linear_swiglu(wq, s, x), "guarded")


@pytest.mark.parametrize("Na,Nb,K,T", [(6144, 1024, 5120, 8), (300, 77, 1152, 100), (128, 128, 256, 1024),
                                       (1000, 3000, 2048, 257), (5, 7, 72, 2), (0, 64, 256, 3), (64, 0, 256, 3),
                                       (6144, 6144, 5120, 1), (200, 300, 17408, 4)])
def test_linear_pair_matches_oracle(Na, Nb, K, T):
    """LinearPair: two weights on one X in one call, each output against its own oracle."""
    t = torch()
    wq_a, s_a, x = synth.make_problem(Na, K, T, w_seed=Na + 1, x_seed=K + T)
    wq_b, s_b, _ = synth.make_problem(Nb, K, 1, w_seed=Nb + 2, x_seed=0)
    da, db = to_dev(wq_a, s_a, x), to_dev(wq_b, s_b, x)
    ya = t.full((T, Na), 7.0, dtype=t.bfloat16, device="cuda")
    yb = t.full((T, Nb), 7.0, dtype=t.bfloat16, device="cuda")
    q4lin.linear_pair(da[0], da[1], db[0], db[1], da[2], y_a=ya, y_b=yb)
    t.cuda.synchronize()
    ra, rb = fo.linear_pair(wq_a, s_a, wq_b, s_b, x)
    if Na:
        assert_close(y_bits(ya), ra, f"LinearPair a {Na}x{K} T={T}")
    if Nb:
        assert_close(y_bits(yb), rb, f"LinearPair b {Nb}x{K} T={T}")
