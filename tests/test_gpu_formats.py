"""GPU parity for the sibling weight formats Q5G64, Q6G64 and W8G32 (linear-benchmark.md
section 4, format table) against the FP64 oracle for those formats: the decode GEMV (one
token for Q5 / Q6, 1..4 for W8; K a multiple of 128 or padded, ragged N), the streaming
warp-MMA route (Q5 / Q6 at 2..32 tokens with the high bits joined to the nibble operands,
W8 at 5..24), and the exact tile route beyond (token tiles up to 128 wide, K split across
clusters where the planner chooses it).  Q4 through the same entry point is q4lin_linear
itself."""
import numpy as np
import pytest

from oracle import sibling_formats as sf
from weight_only_bit_q4_gb300 import q4lin, synth

from gpu_util import assert_close, torch, y_bits

pytestmark = pytest.mark.gpu

FMTS = ["q5g64", "q6g64", "w8g32"]


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


def _run(qtype, planes, s, x):
    t = torch()
    y = q4lin.linear_qtype(qtype, tuple(_dev(p) for p in planes), _dev(s), _dev(x).view(t.bfloat16))
    t.cuda.synchronize()
    return y_bits(y)


@pytest.mark.parametrize("qtype", FMTS)
@pytest.mark.parametrize("N,K", [(5, 128), (300, 200), (1001, 4096), (257, 5120), (640, 4304), (77, 17408),
                                 (6144, 5120)])
def test_formats_match_oracle(qtype, N, K):
    for T in (1, 2, 3, 4):
        planes, s, x = synth.make_problem_fmt(qtype, N, K, T, w_seed=N + K, x_seed=K + T)
        y_ref = sf.linear(qtype, planes, s, x)
        if T * K * 2 > 100 * 1024:
            # x of every token must fit in shared memory next to at least two ring slots
            try:
                yb = _run(qtype, planes, s, x)
            except q4lin.Q4LinError as e:
                assert e.status == 2, e
                continue
        else:
            yb = _run(qtype, planes, s, x)
        assert_close(yb, y_ref, f"{qtype} {N}x{K} T={T}")


def test_q4_through_the_format_entry_is_q4lin_linear():
    wq, s, x = synth.make_problem(1000, 1152, 3, w_seed=4)
    t = torch()
    y_fmt = _run("q4g64", (wq,), s, x)
    y = q4lin.linear(_dev(wq), _dev(s), _dev(x).view(t.bfloat16))
    t.cuda.synchronize()
    assert np.array_equal(y_fmt, y_bits(y))


@pytest.mark.parametrize("N,K,T", [(64, 256, 5), (300, 200, 37), (1001, 4096, 130), (640, 4304, 33),
                                   (77, 17408, 8), (6144, 5120, 24), (257, 1152, 517), (5, 128, 1000),
                                   (6144, 5120, 1024), (129, 8192, 25), (1000, 2048, 40), (333, 640, 70)])
def test_w8_beyond_four_tokens_matches_oracle(N, K, T):
    """W8G32 beyond the decode GEMV: up to 24 tokens the streaming warp-MMA route (signed
    codes offset by 128 as exact fp16 subnormals, two MMAs per 32-wide group), beyond it the
    exact tile route (codes as exact bf16, one tensor-memory accumulator per 32-wide scale
    group, token tiles up to 64 wide)."""
    planes, s, x = synth.make_problem_fmt("w8g32", N, K, T, w_seed=N + 5, x_seed=K + T)
    if T <= 24:
        assert q4lin.kernel_launches(N, K, T, "w8g32") == 2
    else:
        assert q4lin.kernel_launches(N, K, T, "w8g32") in (1, 2)   # the tile route (and a tail launch)
        assert q4lin.load().q4lin_qtype_workspace_bytes(3, N, K, T) == 0
    assert_close(_run("w8g32", planes, s, x), sf.linear("w8g32", planes, s, x), f"w8g32 {N}x{K} T={T}")


def test_w8_beyond_four_tokens_needs_workspace():
    t = torch()
    planes, s, x = synth.make_problem_fmt("w8g32", 64, 256, 5)
    y = t.empty((5, 64), dtype=t.bfloat16, device="cuda")
    d = [_dev(p) for p in planes] + [_dev(s), _dev(x)]
    st = q4lin.load().q4lin_linear_qtype(3, q4lin._ptr(d[0]), None, q4lin._ptr(d[1]), q4lin._ptr(d[2]),
                                         q4lin._ptr(y), 64, 256, 5, None, None)
    assert st == 4  # Q4LIN_ERR_WORKSPACE


@pytest.mark.parametrize("qtype", ["q5g64", "q6g64"])
@pytest.mark.parametrize("N,K,T", [(64, 256, 5), (300, 200, 37), (1001, 4096, 130), (640, 4304, 300),
                                   (77, 17408, 8), (6144, 5120, 128), (257, 1152, 517), (5, 128, 1000),
                                   (6144, 5120, 1024), (1000, 2048, 257)])
def test_q5_q6_tile_route_matches_oracle(qtype, N, K, T):
    # beyond 128 tokens 256-wide tiles (two A stages beside the high-bit stages) or 128-wide ones
    planes, s, x = synth.make_problem_fmt(qtype, N, K, T, w_seed=N + 3, x_seed=K + T)
    assert_close(_run(qtype, planes, s, x), sf.linear(qtype, planes, s, x), f"{qtype} {N}x{K} T={T}")


@pytest.mark.parametrize("qtype", ["q5g64", "q6g64"])
@pytest.mark.parametrize("N,K,T", [(6144, 5120, 8), (6144, 5120, 2), (1001, 4096, 16), (300, 200, 7),
                                   (257, 1152, 32), (640, 4304, 24), (77, 17408, 9), (4097, 512, 31),
                                   (33, 1160, 3), (2000, 5120, 17)])
def test_q5_q6_warp_mma_route_matches_oracle(qtype, N, K, T):
    """Q5G64 / Q6G64 on the streaming warp-MMA route (2..32 tokens): the high bits of each
    weight join its nibble as 16 h in the exact fp16-subnormal operand (16 q <= 1008 stays
    subnormal), zero points 16 and 32 in the operand pass's term."""
    qt = {"q5g64": 1, "q6g64": 2}[qtype]
    assert q4lin.kernel_launches(N, K, T, qtype) == 2
    assert q4lin.load().q4lin_qtype_workspace_bytes(qt, N, K, T) > 0
    planes, s, x = synth.make_problem_fmt(qtype, N, K, T, w_seed=N + 7, x_seed=K + T)
    assert_close(_run(qtype, planes, s, x), sf.linear(qtype, planes, s, x), f"{qtype} {N}x{K} T={T}")


@pytest.mark.parametrize("qtype", ["q5g64", "q6g64"])
def test_q5_q6_gemv_without_plan_goes_to_tiles(qtype):
    # four tokens of a long K: whichever route has a plan (the warp-MMA route here)
    N, K, T = 128, 17408, 4
    planes, s, x = synth.make_problem_fmt(qtype, N, K, T, w_seed=9, x_seed=10)
    assert_close(_run(qtype, planes, s, x), sf.linear(qtype, planes, s, x), f"{qtype} {N}x{K} T={T}")
