"""GPU parity of q4lin_linear_host (X and Y in page-locked host memory) against the FP64 oracle.

The entry stages X from page-locked host memory into the workspace with a kernel,
runs q4lin_linear on it, and copies Y back with a kernel; the layer's bound and the
output contract (every element of y written, nothing outside it) are those of
q4lin_linear.  Pageable or device pointers are refused with INVALID_ARG before any
launch.
"""
import ctypes

import numpy as np
import pytest

import oracle
from weight_only_bit_q4_gb300 import q4lin, synth

from gpu_util import assert_close, to_dev, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from weight_only_bit_q4_gb300 import build
    build.build()
    q4lin.load()
    assert q4lin.clear_device_status() == 0
    yield
    assert q4lin.device_status() == 0


def pinned(a: np.ndarray):
    t = torch()
    return t.from_numpy(np.ascontiguousarray(a).view(np.int16)).pin_memory()


def host_bits(y) -> np.ndarray:
    return y.view(torch().int16).numpy().view(np.uint16).copy()


@pytest.mark.parametrize("N,K,T", [(6144, 5120, 1), (6144, 5120, 8), (1000, 2048, 64), (333, 640, 37),
                                   (129, 1152, 5), (77, 72, 3)])
def test_matches_oracle(N, K, T):
    wq, s, x = synth.make_problem(N, K, T, w_seed=N + 1, x_seed=K + T)
    wq_d, s_d, _ = to_dev(wq, s, x[:1])
    y = q4lin.linear_host(wq_d, s_d, pinned(x))
    torch().cuda.synchronize()
    assert_close(host_bits(y), oracle.linear(wq, s, x), f"host entry {N}x{K} T={T}")


def test_output_written_exactly():
    # y_host is a window of a larger pinned buffer: every element of the window is
    # written, the guard bands around it are not (2 T N bytes = 24642: a 2-byte tail)
    t = torch()
    N, K, T = 333, 640, 37
    wq, s, x = synth.make_problem(N, K, T, w_seed=5, x_seed=6)
    wq_d, s_d, _ = to_dev(wq, s, x[:1])
    guard = 64
    buf = t.full((T * N + 2 * guard,), 0x7FC1, dtype=t.int16).pin_memory()
    y = buf[guard:guard + T * N].view(T, N)
    assert y.data_ptr() % 16 == 0
    q4lin.linear_host(wq_d, s_d, pinned(x), y_host=y)
    t.cuda.synchronize()
    b = buf.numpy().view(np.uint16)
    assert (b[:guard] == 0x7FC1).all() and (b[guard + T * N:] == 0x7FC1).all()
    assert_close(host_bits(y), oracle.linear(wq, s, x), "windowed y_host")


def test_empty_k_writes_zeros():
    t = torch()
    N, T = 40, 3
    wq_d = t.zeros((N, 0), dtype=t.uint8, device="cuda")
    s_d = t.zeros((N, 0), dtype=t.int16, device="cuda")
    x = t.zeros((T, 0), dtype=t.int16).pin_memory()
    y = t.full((T, N), 0x3F80, dtype=t.int16).pin_memory()
    q4lin.linear_host(wq_d, s_d, x, y_host=y)
    t.cuda.synchronize()
    assert (y.numpy() == 0).all()


def test_refuses_pageable_and_device_buffers():
    t = torch()
    N, K, T = 64, 256, 4
    wq, s, x = synth.make_problem(N, K, T, w_seed=1, x_seed=2)
    wq_d, s_d, x_d = to_dev(wq, s, x)
    ws = t.empty(q4lin.host_workspace_bytes(N, K, T), dtype=t.uint8, device="cuda")
    lib = q4lin.load()
    p = q4lin._ptr
    x_page = t.from_numpy(np.ascontiguousarray(x).view(np.int16).copy())   # pageable
    y_pin = t.empty((T, N), dtype=t.int16).pin_memory()
    y_dev = t.empty((T, N), dtype=t.int16, device="cuda")
    assert lib.q4lin_linear_host(p(wq_d), p(s_d), p(x_page), p(y_pin), N, K, T, p(ws), None) == 1
    assert "page-locked" in q4lin.last_error_detail()
    assert lib.q4lin_linear_host(p(wq_d), p(s_d), p(x_d), p(y_pin), N, K, T, p(ws), None) == 1
    assert lib.q4lin_linear_host(p(wq_d), p(s_d), p(pinned(x)), p(y_dev), N, K, T, p(ws), None) == 1
    t.cuda.synchronize()
    # the context is still usable
    y = q4lin.linear_host(wq_d, s_d, pinned(x))
    t.cuda.synchronize()
    assert_close(host_bits(y), oracle.linear(wq, s, x), "after the refusals")


def test_graph_replay_with_new_host_input():
    t = torch()
    N, K = 6144, 5120
    for T in (1, 8, 64):
        wq, s, x1 = synth.make_problem(N, K, T, w_seed=0, x_seed=300 + T)
        x2 = synth.activations(T, K, 400 + T)
        wq_d, s_d, _ = to_dev(wq, s, x1[:1])
        xh = pinned(x1)
        yh = t.empty((T, N), dtype=t.int16).pin_memory()
        ws = t.empty(q4lin.host_workspace_bytes(N, K, T), dtype=t.uint8, device="cuda")
        stream = t.cuda.Stream()
        with t.cuda.stream(stream):
            q4lin.linear_host(wq_d, s_d, xh, y_host=yh, workspace=ws, stream=stream)   # warm-up
            stream.synchronize()
            g = t.cuda.CUDAGraph()
            with t.cuda.graph(g, stream=stream):
                q4lin.linear_host(wq_d, s_d, xh, y_host=yh, workspace=ws, stream=stream)
            g.replay()
            stream.synchronize()
            assert_close(host_bits(yh), oracle.linear(wq, s, x1), f"graph T={T} first input")
            xh.copy_(t.from_numpy(np.ascontiguousarray(x2).view(np.int16)))
            g.replay()
            stream.synchronize()
            assert_close(host_bits(yh), oracle.linear(wq, s, x2), f"graph T={T} refilled host input")
