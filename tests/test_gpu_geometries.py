"""GPU parity on the other Q4 geometries of the linear-benchmark suites, through the
same path: the draft heads (131072 x 5120 and 131072 x 2048, "Continuous" T class
1, 16, 128, 1024) and the vision projections (3456 x 1152 and 4304 x 1152,
"VisionStep4" T class 4, 128, 1024) of the Q4 geometry tables
(linear-benchmark.md section 2).  K = 1152 = 9 x 128 is not a power of two and
is not a multiple of the 1024-wide column groups of the decode GEMV.

The vision shapes are compared element by element with the FP64 oracle over the
whole output.  The draft heads' weights (up to 357 MB) are checked on sampled
rows (the first 64, the last 300 and 1,500 spread over N), computed by the
oracle row by row, with rms(y_ref) taken over the sampled rows.
"""
import numpy as np
import pytest

import oracle
from weight_only_bit_q4_gb300 import q4lin, synth

from gpu_util import assert_close, to_dev, torch, y_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from weight_only_bit_q4_gb300 import build
    build.build()
    q4lin.load()
    assert q4lin.clear_device_status() == 0
    yield
    assert q4lin.device_status() == 0


def _run(d):
    y = q4lin.linear(*d)
    torch().cuda.synchronize()
    return y_bits(y)


@pytest.mark.parametrize("N,K", [(3456, 1152), (4304, 1152)])
def test_vision_projections(N, K):
    wq = synth.packed_codes(N, K, 0)
    s = synth.group_scales(N, K, 0)
    for T in (4, 128, 1024):
        x = synth.activations(T, K, T)
        y_ref = oracle.linear(wq, s, x)
        assert_close(_run(to_dev(wq, s, x)), y_ref, f"{N}x{K} T={T} route {q4lin.select_route(N, K, T)}")


@pytest.mark.parametrize("N,K", [(131072, 5120), (131072, 2048)])
def test_draft_heads_sampled_rows(N, K):
    t = torch()
    wq = synth.packed_codes(N, K, 0)
    s = synth.group_scales(N, K, 0)
    rows = np.unique(np.concatenate([np.arange(0, 64), np.arange(N - 300, N),
                                     np.linspace(0, N - 1, 1500).astype(np.int64)]))
    wq_d, s_d, _ = to_dev(wq, s, np.zeros((1, K), np.uint16))
    for T in (1, 16, 128, 1024):
        x = synth.activations(T, K, T)
        x_d = to_dev(wq[:1], s[:1], x)[2]
        y_ref = oracle.linear(wq, s, x, rows=rows)
        yb = _run((wq_d, s_d, x_d))
        assert_close(yb[:, rows], y_ref, f"{N}x{K} T={T} route {q4lin.select_route(N, K, T)}",
                     rms_ref=oracle.rms(y_ref))
    del wq_d, s_d
    t.cuda.empty_cache()
