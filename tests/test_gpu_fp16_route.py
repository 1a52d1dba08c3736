"""GPU checks of the opt-in tile route on fp16-rounded weights (Q4LIN_ROUTE_TC_FP16).

That route folds the group scale into the weight, w = fp16((q - 8) * s), so its
outputs carry one fp16 rounding per weight on top of FP32 accumulation.  Its
documented bound is |y - y_ref| <= 8e-3 |y_ref| + 4e-3 rms(y_ref) (the layer's
default routes meet the tighter 1e-3 rms floor); these tests hold it to that bound
against the FP64 oracle, including operands far outside fp16's range (the route
takes X per token and the scales per row at a power of two).
"""
import numpy as np
import pytest

import oracle
from weight_only_bit_q4_gb300 import q4lin, synth

from gpu_util import to_dev, torch, y_bits

pytestmark = pytest.mark.gpu

REL, FLOOR = 8e-3, 4e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from weight_only_bit_q4_gb300 import build
    build.build()
    q4lin.load()
    assert q4lin.clear_device_status() == 0
    yield
    assert q4lin.device_status() == 0


def run_fp16(wq, s, x):
    t = torch()
    d = to_dev(wq, s, x)
    y = q4lin.linear(*d, route=q4lin.ROUTE_TC_FP16)
    t.cuda.synchronize()
    return y_bits(y)


def check_fp16(yb, y_ref, what):
    y = oracle.bf16_bits_to_f64(yb)
    assert np.isfinite(y).all(), what
    rms = oracle.rms(y_ref)
    ratio = np.abs(y - y_ref) / (REL * np.abs(y_ref) + FLOOR * rms)
    assert ratio.max() <= 1.0, f"{what}: worst {ratio.max():.3g}x the route's bound"
    return ratio.max()


@pytest.mark.parametrize("N,K,T", [(6144, 5120, 1024), (3456, 1152, 1024), (1000, 1152, 37), (77, 72, 5),
                                   (300, 200, 70), (640, 4304, 130), (2048, 17408, 16)])
def test_fp16_route_matches_oracle(N, K, T):
    wq, s, x = synth.make_problem(N, K, T, w_seed=N + 1, x_seed=K + T)
    check_fp16(run_fp16(wq, s, x), oracle.linear(wq, s, x), f"{N}x{K} T={T}")


def test_fp16_route_lognormal_scales_outlier_channels():
    N, K, T = 14336, 5120, 128
    wq = synth.packed_codes(N, K, 0)
    s = synth.group_scales(N, K, 0, "lognormal")
    x = synth.activations(T, K, T, outliers=True)
    check_fp16(run_fp16(wq, s, x), oracle.linear(wq, s, x), "14336x5120 lognormal + outliers")


def test_fp16_route_operands_outside_fp16_range():
    # rows of very large and of subnormal scales, tokens of very large and very small x:
    # the per-row and per-token powers of two keep every operand in fp16's range
    N, K, T = 512, 1024, 40
    wq, s, x = synth.make_problem(N, K, T, w_seed=7, x_seed=8)
    sf = s.view(np.float16).astype(np.float32)
    sf[:64] *= 3.0e4 / max(float(np.abs(sf[:64]).max()), 1e-30)      # up to 30000
    sf[64:128] *= 2.0e-7 / max(float(np.abs(sf[64:128]).max()), 1e-30)  # fp16 subnormals
    s = sf.astype(np.float16).view(np.uint16)
    xf = oracle.bf16_bits_to_f64(x).astype(np.float32)
    xf[:8] *= 1.0e6
    xf[8:16] *= 1.0e-30
    x = synth.float32_to_bf16_bits(xf)
    y_ref = oracle.linear(wq, s, x)
    yb = run_fp16(wq, s, x)
    # token blocks of very different magnitude: hold each to the bound of its own rms
    for lo, hi in ((0, 8), (8, 16), (16, T)):
        check_fp16(yb[lo:hi], y_ref[lo:hi], f"tokens {lo}..{hi - 1}")


def test_fp16_route_deterministic_and_needs_workspace():
    t = torch()
    wq, s, x = synth.make_problem(1024, 2048, 96, w_seed=3, x_seed=4)
    assert run_fp16(wq, s, x).tobytes() == run_fp16(wq, s, x).tobytes()
    d = to_dev(wq, s, x)
    y = t.empty((96, 1024), dtype=t.bfloat16, device="cuda")
    st = q4lin.linear_raw(*(q4lin._ptr(a) for a in d), q4lin._ptr(y), 1024, 2048, 96, None, None,
                          q4lin.ROUTE_TC_FP16)
    assert st == 4  # Q4LIN_ERR_WORKSPACE
