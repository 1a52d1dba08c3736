"""Seeded random shapes through every entry point and route, against the FP64 oracles.

Sixty cases drawn once from a fixed seed: N from 1 to about 3000, K any multiple of 8 up to
about 12000 (so K_pad padding, partial last groups and every split of K appear), T from 1
to about 600 on a log scale (every route and tile width, and their seams), over q4lin_linear
with the library's route and with a forced route, the sibling formats and the three fused
operations.  Each output is held to the layer's bound; the cases are sized so the FP64
oracle takes well under a second each.
"""
import numpy as np
import pytest

import oracle
from oracle import fused_ops as fo
from oracle import sibling_formats as sf
from weight_only_bit_q4_gb300 import q4lin, synth

from gpu_util import assert_close, to_dev, torch, x_to_dev, y_bits

pytestmark = pytest.mark.gpu

KINDS = ["linear", "linear", "route", "route", "q5g64", "q6g64", "w8g32", "w8g32", "add", "swiglu", "pair"]


def _cases(n=60, seed=2024):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        kind = KINDS[rng.integers(len(KINDS))]
        N = int(rng.integers(1, 3000))
        K = 8 * int(rng.integers(1, 1500))
        T = int(np.exp(rng.uniform(0.0, np.log(600.0))))
        T = max(1, T)
        if N * K * T > 6e8:          # keep the FP64 oracle quick
            continue
        route = ["gemv", "tc", "tc_splitk", "stream_mma"][int(rng.integers(4))] if kind == "route" else None
        if route == "gemv" and T > 4:
            route = "tc_splitk"
        out.append((kind, N, K, T, route))
    return out


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from weight_only_bit_q4_gb300 import build
    build.build()
    q4lin.load()
    assert q4lin.clear_device_status() == 0
    yield
    assert q4lin.device_status() == 0


def _dev(a):
    t = torch()
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return t.from_numpy(a).cuda()


ROUTES = {"gemv": q4lin.ROUTE_GEMV, "tc": q4lin.ROUTE_TC, "tc_splitk": q4lin.ROUTE_TC_SPLITK,
          "stream_mma": q4lin.ROUTE_STREAM_MMA}


@pytest.mark.parametrize("kind,N,K,T,route", _cases())
def test_random_shape(kind, N, K, T, route):
    t = torch()
    seed = N * 7 + K * 3 + T
    label = f"{kind} {N}x{K} T={T}" + (f" route={route}" if route else "")
    if kind in ("q5g64", "q6g64", "w8g32"):
        planes, s, x = synth.make_problem_fmt(kind, N, K, T, w_seed=seed, x_seed=seed + 1)
        try:
            y = q4lin.linear_qtype(kind, tuple(_dev(p) for p in planes), _dev(s), _dev(x).view(t.bfloat16))
        except q4lin.Q4LinError as e:   # a shape no route of that format can plan: refused, never approximated
            assert e.status == 2, (label, e)
            return
        t.cuda.synchronize()
        assert_close(y_bits(y), sf.linear(kind, planes, s, x), label)
        return
    if kind == "swiglu":
        F = max(1, N // 2)
        wq, s, x = synth.make_problem(2 * F, K, T, w_seed=seed, x_seed=seed + 1)
        y = q4lin.linear_swiglu(*to_dev(wq, s, x))
        t.cuda.synchronize()
        assert_close(y_bits(y), fo.linear_swiglu(wq, s, x), label)
        return
    if kind == "pair":
        Nb = max(1, N // 3)
        wq_a, s_a, x = synth.make_problem(N, K, T, w_seed=seed, x_seed=seed + 1)
        wq_b, s_b, _ = synth.make_problem(Nb, K, 1, w_seed=seed + 2, x_seed=0)
        da, db = to_dev(wq_a, s_a, x), to_dev(wq_b, s_b, x)
        ya, yb = q4lin.linear_pair(da[0], da[1], db[0], db[1], da[2])
        t.cuda.synchronize()
        ra, rb = fo.linear_pair(wq_a, s_a, wq_b, s_b, x)
        assert_close(y_bits(ya), ra, label + " (a)")
        assert_close(y_bits(yb), rb, label + " (b)")
        return
    wq, s, x = synth.make_problem(N, K, T, w_seed=seed, x_seed=seed + 1)
    d = to_dev(wq, s, x)
    if kind == "add":
        r = synth.activations(T, N, seed=seed + 2)
        y = q4lin.linear_add(*d, x_to_dev(r))
        t.cuda.synchronize()
        assert_close(y_bits(y), fo.linear_add(wq, s, x, r), label)
        return
    if kind == "route":
        rt = ROUTES[route]
        if rt == q4lin.ROUTE_STREAM_MMA and q4lin.workspace_bytes(N, K, T, rt) == 0:
            return   # no plan for this shape on the warp-MMA route
        try:
            y = q4lin.linear(*d, route=rt)
        except q4lin.Q4LinError as e:
            assert e.status == 2, (label, e)   # no plan on the forced route: refused
            return
    else:
        y = q4lin.linear(*d)
    t.cuda.synchronize()
    assert_close(y_bits(y), oracle.linear(wq, s, x), label)
