"""The allocation-free entry point, q4lin_linear_fp16_static.

Some callers cannot allocate device memory around the layer: work issued inside a
stream capture that must not allocate, an allocator that owns the whole device, or
a host program with no allocator at all.  This entry runs the fp16 tile route with
its scratch in a fixed array inside the library.  It is checked here, through the
C ABI, against the workspace entry of the same route (q4lin_linear_route with
Q4LIN_ROUTE_TC_FP16) on two calls in a row that share the array.  The file sorts
last so that a run stopping at the first failure has run every other test first.
"""
import ctypes

import numpy as np
import pytest

import oracle
from weight_only_bit_q4_gb300 import q4lin, synth

from gpu_util import to_dev, torch, y_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from weight_only_bit_q4_gb300 import build
    build.build()
    q4lin.load()
    assert q4lin.clear_device_status() == 0
    yield
    assert q4lin.device_status() == 0


def _static(d, y, N, K, T):
    t = torch()
    p = [ctypes.c_void_p(a.data_ptr()) for a in d]
    st = q4lin.load().q4lin_linear_fp16_static(p[0], p[1], p[2], ctypes.c_void_p(y.data_ptr()), N, K, T, None)
    t.cuda.synchronize()
    return st


def _within_route_bound(a_bits, b_bits):
    # the fp16 route's bound, |a - b| <= 8e-3 |b| + 4e-3 rms(b), taking b as the reference
    a, b = oracle.bf16_bits_to_f64(a_bits), oracle.bf16_bits_to_f64(b_bits)
    return bool(np.all(np.abs(a - b) <= 8e-3 * np.abs(b) + 4e-3 * oracle.rms(b)))


def test_static_scratch_entry_matches_workspace_entry():
    t = torch()
    cases = [(6144, 5120, 256, 1), (1000, 1152, 37, 2)]
    problems, outs = [], []
    for N, K, T, seed in cases:               # two calls in a row on the shared array
        wq, s, x = synth.make_problem(N, K, T, w_seed=seed, x_seed=seed + 10)
        d = to_dev(wq, s, x)
        y = t.full((T, N), 7.0, dtype=t.bfloat16, device="cuda")
        assert _static(d, y, N, K, T) == 0, q4lin.last_error_detail()
        problems.append(d)
        outs.append(y_bits(y))
    for (N, K, T, _), d, yb in zip(cases, problems, outs):
        y_ws = q4lin.linear(*d, route=q4lin.ROUTE_TC_FP16)
        t.cuda.synchronize()
        ref = y_bits(y_ws)
        assert _within_route_bound(yb, ref), (N, K, T)
        assert np.array_equal(yb, ref), (N, K, T)   # the same kernels: the same bits


def test_static_scratch_entry_refuses_shapes_beyond_its_array():
    t = torch()
    N, K, T = 256, 5120, 2048                 # 2*T*K alone is 20 MiB
    wq, s, x = synth.make_problem(N, K, T, w_seed=3)
    d = to_dev(wq, s, x)
    y = t.full((T, N), 7.0, dtype=t.bfloat16, device="cuda")
    assert _static(d, y, N, K, T) == 2
    assert "16 MiB" in q4lin.last_error_detail()
    assert bool((y == 7.0).all())
