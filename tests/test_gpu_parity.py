"""GPU parity: the CUDA path against the FP64 oracle, element by element.

Tolerance (the layer's acceptance bound): |y - y_ref| <= 8e-3 |y_ref| + 1e-3 rms(y_ref),
rms over the whole output.  Every route is compared with the oracle, not with
the other routes (different compute organisations need not agree bitwise).
"""
import numpy as np
import pytest

import oracle
from weight_only_bit_q4_gb300 import q4lin, synth

from gpu_util import assert_close, reference, to_dev, torch, weights, x_to_dev, y_bits

pytestmark = pytest.mark.gpu

ROUTES = [q4lin.ROUTE_GEMV, q4lin.ROUTE_TC_SPLITK, q4lin.ROUTE_TC, q4lin.ROUTE_STREAM_MMA]


def implemented(route):
    return route in q4lin.implemented_routes()


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from weight_only_bit_q4_gb300 import build
    build.build()
    q4lin.load()
    assert q4lin.clear_device_status() == 0
    yield
    assert q4lin.device_status() == 0


def run(wq_d, s_d, x_d, route=q4lin.ROUTE_AUTO):
    y = q4lin.linear(wq_d, s_d, x_d, route=route)
    torch().cuda.synchronize()
    return y_bits(y)


# ------------------------------------------------------------ benchmark configurations
def test_config_512x1024_t8_all_routes():
    wq, s, x = synth.make_problem(512, 1024, 8, w_seed=0, x_seed=0)
    y_ref = oracle.linear(wq, s, x)
    d = to_dev(wq, s, x)
    assert_close(run(*d), y_ref, "auto")
    for r in ROUTES:
        if implemented(r):
            assert_close(run(*d, route=r), y_ref, q4lin.ROUTE_NAMES[r])


def test_config_6144x5120_t1():
    wq, s, w = weights(6144, 5120)
    x = synth.activations(1, 5120, 0)
    d = to_dev(wq, s, x)
    assert_close(run(*d), reference(w, x), "decode T=1")


def test_sweep_6144x5120_every_t():
    """T = 1..128 every integer, plus 384, 385, 512, 640, 641, 1024; X seed = T."""
    wq, s, w = weights(6144, 5120)
    wq_d, s_d, _ = to_dev(wq, s, np.zeros((1, 5120), np.uint16))
    for T in synth.SWEEP_6144x5120_T:
        x = synth.activations(T, 5120, T)
        assert_close(run(wq_d, s_d, x_to_dev(x)), reference(w, x), f"T={T}")


@pytest.mark.parametrize("T", [1, 16, 128, 1024])
def test_config_14336x5120_lognormal_outliers(T):
    wq, s, w = weights(14336, 5120, 0, "lognormal")
    x = synth.activations(T, 5120, T, outliers=True)
    d = to_dev(wq, s, x)
    assert_close(run(*d), reference(w, x), f"14336x5120 T={T}")


@pytest.mark.parametrize("N,K", [(34816, 5120), (5120, 17408)])
def test_config_prefill_t1024(N, K):
    wq, s, w = weights(N, K)
    x = synth.activations(1024, K, 0)
    d = to_dev(wq, s, x)
    assert_close(run(*d), reference(w, x), f"{N}x{K} T=1024")


# ------------------------------------------------------------ every route, route seams
@pytest.mark.parametrize("route", ROUTES)
def test_each_route_across_t(route):
    if not implemented(route):
        pytest.skip("route not built")
    wq, s, w = weights(6144, 5120)
    wq_d, s_d, _ = to_dev(wq, s, np.zeros((1, 5120), np.uint16))
    for T in [1, 2, 3, 4, 5, 7, 8, 9, 15, 16, 17, 24, 25, 31, 32, 33, 48, 63, 64, 65, 96, 97,
              127, 128, 129, 192, 255, 256, 257, 300, 384, 385, 511, 512, 513, 640, 641, 1000, 1024]:
        x = synth.activations(T, 5120, T)
        assert_close(run(wq_d, s_d, x_to_dev(x), route), reference(w, x), f"{q4lin.ROUTE_NAMES[route]} T={T}")


@pytest.mark.parametrize("route", ROUTES)
@pytest.mark.parametrize("N,K,T", [(1, 128, 1), (3, 128, 2), (127, 256, 5), (129, 1152, 17),
                                   (1000, 384, 33), (200, 640, 130), (300, 2048, 257),
                                   (129, 128, 3), (4097, 512, 64), (96, 8192, 100)])
def test_ragged_shapes(route, N, K, T):
    if not implemented(route):
        pytest.skip("route not built")
    wq, s, x = synth.make_problem(N, K, T, w_seed=N + K, x_seed=T)
    y_ref = oracle.linear(wq, s, x)
    assert_close(run(*to_dev(wq, s, x), route), y_ref, f"{q4lin.ROUTE_NAMES[route]} {N}x{K} T={T}")


@pytest.mark.parametrize("T", [1, 2, 3, 4])
@pytest.mark.parametrize("N,K", [(1, 128), (3, 128), (5, 128), (607, 384), (153, 1152), (1001, 4096),
                                 (999, 8192), (333, 8320), (150, 14336), (257, 17408), (77, 28672),
                                 (61, 49152), (10, 65536)])
def test_decode_gemv_shapes(N, K, T):
    """T = 1..4 on the GEMV route across K: 8-, 4- and 2-row blocks, 32- and
    16-weight lane chunks, warps that keep or reload their x values, scale runs
    that end inside the plane's last 16-byte granule (N K / 32 not a multiple of
    16), one row per CTA, and shapes beyond the streaming kernel's shared memory."""
    wq, s, x = synth.make_problem(N, K, T, w_seed=N + K, x_seed=K + T)
    y_ref = oracle.linear(wq, s, x)
    assert_close(run(*to_dev(wq, s, x), q4lin.ROUTE_GEMV), y_ref, f"decode gemv {N}x{K} T={T}")
    if T == 1:
        assert_close(run(*to_dev(wq, s, x)), y_ref, f"decode {N}x{K}")


@pytest.mark.parametrize("route", ROUTES)
@pytest.mark.parametrize("N,K", [(5, 8), (130, 64), (300, 72), (257, 200), (1000, 1000), (640, 4304), (129, 8200)])
def test_k_not_multiple_of_128(route, N, K):
    """K a multiple of 8 but not of 128: planes stored for K_pad = align_up(K, 128)
    columns (linear-benchmark.md section 4), padded codes random and every wholly
    padded group's scale NaN or Inf, which must not reach y."""
    Kp = (K + 127) // 128 * 128
    rng = np.random.default_rng(K)
    for T in [1, 2, 4, 5, 17, 100, 300]:
        wq, s, x = synth.make_problem(N, K, T, w_seed=N + K, x_seed=T)
        assert wq.shape[1] == Kp // 2 and s.shape[1] == Kp // 64 and x.shape[1] == K
        wq[:, K // 2:] = rng.integers(0, 256, (N, Kp // 2 - K // 2), dtype=np.uint8)
        g = (K + 63) // 64
        s[:, g:] = np.where(rng.integers(0, 2, (N, Kp // 64 - g)) == 0, 0x7E00, 0x7C00)
        y_ref = oracle.linear(wq, s, x)
        assert_close(run(*to_dev(wq, s, x), route), y_ref, f"{q4lin.ROUTE_NAMES[route]} {N}x{K} T={T}")


# ------------------------------------------------------------ edge cases and guards
def test_empty_and_degenerate():
    t = torch()
    wq, s, x = synth.make_problem(64, 256, 4)
    wq_d, s_d, x_d = to_dev(wq, s, x)
    y = t.full((4, 64), 7.0, dtype=t.bfloat16, device="cuda")
    # T == 0 and N == 0: no work, nothing written
    assert q4lin.linear_raw(q4lin._ptr(wq_d), q4lin._ptr(s_d), q4lin._ptr(x_d), q4lin._ptr(y), 64, 256, 0) == 0
    assert q4lin.linear_raw(q4lin._ptr(wq_d), q4lin._ptr(s_d), q4lin._ptr(x_d), q4lin._ptr(y), 0, 256, 4) == 0
    t.cuda.synchronize()
    assert bool((y == 7.0).all())
    # K == 0: the empty sum, y = +0
    assert q4lin.linear_raw(None, None, None, q4lin._ptr(y), 64, 0, 4) == 0
    t.cuda.synchronize()
    assert bool((y.view(t.int16) == 0).all())
    # all codes 8: exactly zero output
    z = np.full_like(wq, 0x88)
    yb = run(*to_dev(z, s, x))
    assert np.all(yb == 0)


def test_output_guard_and_input_preservation():
    t = torch()
    N, K, T = 1000, 1024, 37
    wq, s, x = synth.make_problem(N, K, T, w_seed=4, x_seed=5)
    wq_d, s_d, x_d = to_dev(wq, s, x)
    pad = 4096
    buf = t.full((pad + T * N + pad,), -3.0, dtype=t.bfloat16, device="cuda")
    y = buf[pad:pad + T * N].view(T, N)
    before = [a.clone() for a in (wq_d, s_d, x_d)]
    for r in [q4lin.ROUTE_AUTO] + [r for r in ROUTES if implemented(r)]:
        q4lin.linear(wq_d, s_d, x_d, y=y, route=r)
        t.cuda.synchronize()
        assert bool((buf[:pad] == -3.0).all()) and bool((buf[pad + T * N:] == -3.0).all()), r
        for a, b in zip(before, (wq_d, s_d, x_d)):
            assert t.equal(a, b)
        assert_close(y_bits(y), oracle.linear(wq, s, x), f"route {r}")


def test_deterministic_and_nondefault_stream():
    t = torch()
    wq, s, x = synth.make_problem(2048, 2048, 96, w_seed=1, x_seed=2)
    d = to_dev(wq, s, x)
    for r in [q4lin.ROUTE_AUTO] + [r for r in ROUTES if implemented(r)]:
        a = run(*d, route=r)
        b = run(*d, route=r)
        assert np.array_equal(a, b)
        st = t.cuda.Stream()
        with t.cuda.stream(st):
            y = q4lin.linear(*d, route=r, stream=st)
        st.synchronize()
        assert np.array_equal(y_bits(y), a)


def test_graph_replay_after_input_change():
    t = torch()
    N, K = 6144, 5120
    wq, s, w = weights(N, K)
    for T in [1, 4, 8, 64, 1024]:
        x1 = synth.activations(T, K, 100 + T)
        x2 = synth.activations(T, K, 200 + T)
        wq_d, s_d, x_d = to_dev(wq, s, x1)
        y = t.empty((T, N), dtype=t.bfloat16, device="cuda")
        ws_n = q4lin.workspace_bytes(N, K, T)
        ws = t.empty(max(ws_n, 256), dtype=t.uint8, device="cuda")
        q4lin.linear(wq_d, s_d, x_d, y=y, workspace=ws)   # warm-up outside capture
        t.cuda.synchronize()
        g = t.cuda.CUDAGraph()
        with t.cuda.graph(g):
            q4lin.linear(wq_d, s_d, x_d, y=y, workspace=ws)
        g.replay()
        t.cuda.synchronize()
        assert_close(y_bits(y), reference(w, x1), f"graph T={T} first inputs")
        x_d.copy_(x_to_dev(x2))
        g.replay()
        t.cuda.synchronize()
        assert_close(y_bits(y), reference(w, x2), f"graph T={T} replay after refill")


def test_large_offsets_beyond_2gb():
    """Code plane larger than 2^31 bytes: 64-bit addressing; sampled rows, oracle row by row."""
    t = torch()
    N, K, T = 524288 + 77, 8192, 3
    wq = synth.packed_codes(N, K, 9)
    s = synth.group_scales(N, K, 9)
    x = synth.activations(T, K, 9)
    d = to_dev(wq, s, x)
    rows = np.unique(np.concatenate([np.arange(0, 64), np.arange(N - 300, N),
                                     np.linspace(0, N - 1, 2000).astype(np.int64)]))
    y_ref = oracle.linear(wq, s, x, rows=rows)
    for r in [q4lin.ROUTE_AUTO] + [r for r in ROUTES if implemented(r)]:
        yb = run(*d, route=r)
        assert_close(yb[:, rows], y_ref, f"route {r}", rms_ref=oracle.rms(y_ref))
    del d
    t.cuda.empty_cache()
