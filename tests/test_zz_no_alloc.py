"""The allocation-free entry point, q4lin_linear_fp16_static.

Some callers cannot allocate device memory around the layer: work issued inside a
stream capture that must not allocate, an allocator that owns the whole device, or
a host program with no allocator at all.  This entry runs the fp16 tile route with
its scratch in a fixed array inside the library.  It is checked here, through the
C ABI, against the FP64 oracle at that route's documented bound and against the
workspace entry of the same route (q4lin_linear_route with Q4LIN_ROUTE_TC_FP16),
on two calls in a row that share the array; its capacity limit is checked at the
boundary, and free device memory must not change across a call.  The file sorts
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


def _within_route_bound(a_bits, y_ref):
    # the fp16 route's bound: |y - y_ref| <= 8e-3 |y_ref| + 4e-3 rms(y_ref)
    a = oracle.bf16_bits_to_f64(a_bits)
    return bool(np.all(np.abs(a - y_ref) <= 8e-3 * np.abs(y_ref) + 4e-3 * oracle.rms(y_ref)))


def test_static_scratch_entry_matches_oracle_and_workspace_entry():
    t = torch()
    cases = [(6144, 5120, 256, 1), (1000, 1152, 37, 2)]
    problems, outs = [], []
    for N, K, T, seed in cases:               # two calls in a row on the shared array
        wq, s, x = synth.make_problem(N, K, T, w_seed=seed, x_seed=seed + 10)
        d = to_dev(wq, s, x)
        y = t.full((T, N), 7.0, dtype=t.bfloat16, device="cuda")
        assert _static(d, y, N, K, T) == 0, q4lin.last_error_detail()
        problems.append((wq, s, x, d))
        outs.append(y_bits(y))
    for (N, K, T, _), (wq, s, x, d), yb in zip(cases, problems, outs):
        assert _within_route_bound(yb, oracle.linear(wq, s, x)), (N, K, T)
        y_ws = q4lin.linear(*d, route=q4lin.ROUTE_TC_FP16)
        t.cuda.synchronize()
        assert np.array_equal(yb, y_bits(y_ws)), (N, K, T)   # the same kernels: the same bits


def test_static_scratch_entry_capacity_boundary():
    # 2*T*K + 4*T + 4*N bytes, each part rounded up to 256, against 16 MiB: at N = 6144,
    # K = 5120 the largest T that fits is 1635
    t = torch()
    N, K = 6144, 5120
    wq, s, x = synth.make_problem(N, K, 1636, w_seed=4, x_seed=5)
    d = to_dev(wq, s, x)
    y = t.full((1636, N), 7.0, dtype=t.bfloat16, device="cuda")
    assert _static(d, y, N, K, 1636) == 2
    assert "16 MiB" in q4lin.last_error_detail()
    assert bool((y == 7.0).all())
    y2 = t.full((1635, N), 7.0, dtype=t.bfloat16, device="cuda")
    assert _static(d, y2, N, K, 1635) == 0, q4lin.last_error_detail()   # x rows 0..1634
    assert _within_route_bound(y_bits(y2), oracle.linear(wq, s, x[:1635]))


def test_static_scratch_entry_refuses_shapes_beyond_its_array():
    t = torch()
    N, K, T = 256, 5120, 2048                 # 2*T*K alone is 20 MiB
    wq, s, x = synth.make_problem(N, K, T, w_seed=3)
    d = to_dev(wq, s, x)
    y = t.full((T, N), 7.0, dtype=t.bfloat16, device="cuda")
    assert _static(d, y, N, K, T) == 2
    assert "16 MiB" in q4lin.last_error_detail()
    assert bool((y == 7.0).all())


def test_static_scratch_entry_allocates_nothing():
    # after a first call (which loads the library's kernels into the context), a call
    # leaves the device's free memory exactly as it was
    t = torch()
    N, K, T = 2048, 4096, 64
    wq, s, x = synth.make_problem(N, K, T, w_seed=6, x_seed=7)
    d = to_dev(wq, s, x)
    y = t.empty((T, N), dtype=t.bfloat16, device="cuda")
    assert _static(d, y, N, K, T) == 0
    free0 = t.cuda.mem_get_info()[0]
    assert _static(d, y, N, K, T) == 0
    assert t.cuda.mem_get_info()[0] == free0
    assert _within_route_bound(y_bits(y), oracle.linear(wq, s, x))
