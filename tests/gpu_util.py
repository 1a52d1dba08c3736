"""Helpers for the GPU parity tests: device upload, oracle caching, comparison."""
from __future__ import annotations

import functools

import numpy as np

import oracle
from weight_only_bit_q4_gb300 import synth


def torch():
    import torch as _t
    return _t


def to_dev(wq, s, x):
    t = torch()
    return (t.from_numpy(np.ascontiguousarray(wq)).cuda(),
            t.from_numpy(np.ascontiguousarray(s).view(np.int16)).cuda(),
            t.from_numpy(np.ascontiguousarray(x).view(np.int16)).cuda().view(t.bfloat16))


def x_to_dev(x):
    t = torch()
    return t.from_numpy(np.ascontiguousarray(x).view(np.int16)).cuda().view(t.bfloat16)


def y_bits(y) -> np.ndarray:
    t = torch()
    return y.view(t.int16).cpu().numpy().view(np.uint16)


@functools.lru_cache(maxsize=2)
def weights(N: int, K: int, w_seed: int = 0, dist: str = "halfnormal"):
    """(wq, scales, w_f64) for a seeded weight; the FP64 weight comes from the oracle."""
    wq = synth.packed_codes(N, K, w_seed)
    s = synth.group_scales(N, K, w_seed, dist)
    return wq, s, oracle.dequantize(wq, s)


def reference(w_f64: np.ndarray, x_bits: np.ndarray) -> np.ndarray:
    """Oracle y_ref [T, N] from the oracle's dequantised weight and decoded X."""
    return oracle.bf16_bits_to_f64(x_bits) @ w_f64.T


def assert_close(yb: np.ndarray, y_ref: np.ndarray, what: str = "", rms_ref=None):
    r = oracle.check(yb, y_ref, rms_ref)
    assert r["nonfinite"] == 0, f"{what}: {r}"
    assert r["ok"], f"{what}: {r['n_bad']} of {r['size']} elements out of tolerance (worst {r['worst_ratio']:.3g}x bound)"
    return r
