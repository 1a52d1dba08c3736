"""GPU parity for LinearAdd (q4lin_linear_add): Y = W . X + R with the bf16 residual R
added to the FP32 sum before Y's bf16 rounding, against the FP64 fused-operation
oracle within the layer's tolerance.  Covers one token to 1024, padded K, a K split
across a cluster, the in-place form (R is Y) and K = 0 (Y = R)."""
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
                                   (6144, 5120, 1024)])
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


def test_linear_add_empty_k_copies_the_residual():
    t = torch()
    r = x_to_dev(synth.activations(3, 64, seed=5))
    y = t.zeros((3, 64), dtype=t.bfloat16, device="cuda")
    st = q4lin.load().q4lin_linear_add(None, None, None, q4lin._ptr(r), q4lin._ptr(y), 64, 0, 3, None)
    t.cuda.synchronize()
    assert st == 0 and t.equal(y.view(t.int16), r.view(t.int16))
