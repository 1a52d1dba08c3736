"""The C-ABI library builds, loads and exports what include/q4lin.h declares;
host-side argument checks work without a GPU (no compute calls here)."""
import ctypes
import os
import re
import subprocess

import pytest

from weight_only_bit_q4_gb300 import build as q4build
from weight_only_bit_q4_gb300 import q4lin

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "q4lin.h")


@pytest.fixture(scope="module")
def lib():
    q4build.build()
    return q4lin.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(q4lin_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("q4lin_workspace_bytes", "q4lin_linear", "q4lin_status_string",
                     "q4lin_device_status"):
        assert required in names
    assert set(names) == set(q4lin.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", q4lin.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (q4lin_\w+)", out))
    assert set(declared_functions()) <= exported


def test_c_client_compiles_links_and_runs(lib, tmp_path):
    # the boundary from C, without Python in between: header alone, library linked
    src = os.path.join(ROOT, "tests", "c_abi", "abi_host_checks.c")
    exe = str(tmp_path / "abi_host_checks")
    libdir = os.path.dirname(q4lin.LIB_PATH)
    cmd = ["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), src, "-o", exe,
           "-L" + libdir, "-lq4lin", "-Wl,-rpath," + libdir]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    run = subprocess.run([exe], capture_output=True, text=True)
    assert run.returncode == 0, run.stdout + run.stderr
    assert "FAIL" not in run.stdout


def test_status_strings(lib):
    for code in range(8):
        assert q4lin.status_string(code) and q4lin.status_string(code) != "unknown status"
    assert q4lin.status_string(99) == "unknown status"
    assert re.match(r"\d+\.\d+\.\d+$", q4lin.version())


def _call(N, K, T, wq=16, s=16, x=16, y=16, ws=None, route=0):
    vp = lambda v: None if v is None else ctypes.c_void_p(v)
    return q4lin.linear_raw(vp(wq), vp(s), vp(x), vp(y), N, K, T, vp(ws), None, route)


def test_argument_errors_detected_on_host(lib):
    # None of these reach the CUDA runtime: the fake pointers are never dereferenced.
    assert _call(-1, 128, 1) == 1
    assert _call(4, -128, 1) == 1
    assert _call(4, 128, -1) == 1
    assert _call(4, 100, 1) == 2          # K % 8 != 0: X rows would not start 16-byte aligned
    assert _call(4, 60, 1) == 2
    assert _call(4, 4, 1) == 2
    assert _call(4, 128, 1, wq=None) == 1
    assert _call(4, 128, 1, s=None) == 1
    assert _call(4, 128, 1, x=None) == 1
    assert _call(4, 128, 1, y=None) == 1
    assert _call(4, 128, 1, wq=17) == 3
    assert _call(4, 128, 1, s=18) == 3
    assert _call(4, 128, 1, x=24) == 3
    assert _call(4, 128, 1, y=8) == 3
    assert _call(1 << 41, 128, 1) == 1    # beyond the size limit
    assert _call(1 << 30, 1 << 30, 1) == 1  # N*K would overflow the byte counts
    assert _call(4, 128, 1, route=9) == 1  # no such route


def _call_qtype(qtype, N, K, T, codes=16, high=16, s=16, x=16, y=16):
    vp = lambda v: None if v is None else ctypes.c_void_p(v)
    return int(lib_fn().q4lin_linear_qtype(qtype, vp(codes), vp(high), vp(s), vp(x), vp(y), N, K, T, None, None))


def lib_fn():
    return q4lin.load()


def test_linear_add_host_checks(lib):
    vp = ctypes.c_void_p
    f = lib.q4lin_linear_add
    assert f(vp(16), vp(16), vp(16), None, vp(16), 64, 256, 8, None) == 1      # no residual
    assert f(vp(16), vp(16), vp(16), vp(24), vp(16), 64, 256, 8, None) == 3    # misaligned residual
    assert f(vp(16), vp(16), vp(16), vp(16), vp(16), 64, 100, 8, None) == 2    # K % 8 != 0
    assert f(None, None, None, None, None, 0, 256, 8, None) == 0               # empty


def test_qtype_launch_counts_on_host(lib):
    # q4g64 is q4lin_kernel_launches; unknown formats and refused shapes launch nothing
    assert q4lin.kernel_launches(6144, 5120, 1024, "q4g64") == q4lin.kernel_launches(6144, 5120, 1024)
    assert lib.q4lin_qtype_kernel_launches(9, 64, 256, 8) == 0
    assert q4lin.kernel_launches(64, 100, 8, "q5g64") == 0            # K % 8 != 0
    assert q4lin.kernel_launches(0, 256, 8, "q6g64") == 0             # empty
    assert q4lin.kernel_launches(64, 0, 8, "q6g64") == 1              # the zero fill
    # W8 beyond the GEMV: the warp-MMA route up to 24 tokens (an operand pass and a kernel,
    # workspace for the operands), the exact tile route beyond (no workspace)
    assert q4lin.kernel_launches(6144, 5120, 16, "w8g32") == 2
    assert lib.q4lin_qtype_workspace_bytes(3, 6144, 5120, 16) > 0
    assert q4lin.kernel_launches(6144, 5120, 1024, "w8g32") in (1, 2)
    assert lib.q4lin_qtype_workspace_bytes(3, 6144, 5120, 1024) == 0
    assert lib.q4lin_qtype_workspace_bytes(3, 6144, 5120, 1) == 0   # the decode GEMV
    assert lib.q4lin_qtype_workspace_bytes(1, 6144, 5120, 1024) == 0  # Q5: the exact tile route
    for q in ("q5g64", "q6g64"):                                      # the tile route (one wave or a tail)
        assert q4lin.kernel_launches(6144, 5120, 1024, q) in (1, 2)


def test_qtype_argument_errors_detected_on_host(lib):
    assert _call_qtype(9, 4, 128, 1) == 1                 # no such format
    assert _call_qtype(-1, 4, 128, 1) == 1
    assert _call_qtype(1, 4, 128, 1, high=None) == 1      # Q5 without its high plane
    assert _call_qtype(2, 4, 128, 1, high=None) == 1      # Q6 without its high plane
    assert _call_qtype(1, 4, 128, 1, high=24) == 3        # misaligned high plane
    assert _call_qtype(3, 4, 100, 1) == 2                 # K % 8 != 0
    assert _call_qtype(3, 4, 128, 1, codes=None) == 1
    assert _call_qtype(2, 4, 128, 1, s=8) == 3
    assert _call_qtype(1, 0, 128, 5, codes=None, high=None, s=None, x=None, y=None) == 0   # empty


def test_empty_problems_are_noops(lib):
    # N == 0 or T == 0: nothing to compute, nothing launched, even with null pointers.
    assert _call(0, 128, 5, wq=None, s=None, x=None, y=None) == 0
    assert _call(5, 128, 0, wq=None, s=None, x=None, y=None) == 0
    assert _call(0, 0, 0, wq=None, s=None, x=None, y=None) == 0


def test_workspace_query_and_route_selection(lib):
    for N, K, T in [(6144, 5120, 1), (6144, 5120, 16), (6144, 5120, 1024), (512, 1024, 8)]:
        ws = q4lin.workspace_bytes(N, K, T)
        assert ws % 256 == 0
        assert q4lin.select_route(N, K, T) in (1, 2, 3, 5)
    # 2..32 tokens: the streaming warp-MMA route, whose operand pass needs workspace
    for T in (2, 8, 16, 24, 32):
        assert q4lin.select_route(6144, 5120, T) == q4lin.ROUTE_STREAM_MMA
        assert q4lin.workspace_bytes(6144, 5120, T) > 0
    assert q4lin.select_route(6144, 5120, 33) == q4lin.ROUTE_TC_SPLITK
    assert q4lin.workspace_bytes(-1, 128, 1) == 0
    assert q4lin.workspace_bytes(4, 100, 1) == 0
    assert q4lin.workspace_bytes(0, 128, 1) == 0
    assert q4lin.select_route(6144, 5120, 1) == q4lin.ROUTE_GEMV
    assert q4lin.workspace_bytes(6144, 5120, 1) == 0


def test_fp16_tile_route_workspace_checked_on_host(lib):
    # the opt-in fp16 route refuses a NULL or misaligned workspace before any CUDA call
    assert _call(64, 256, 8, route=q4lin.ROUTE_TC_FP16) == 4
    assert _call(64, 256, 8, ws=16 + 128, route=q4lin.ROUTE_TC_FP16) == 3
    assert _call(64, 256, 8, route=q4lin.ROUTE_STREAM_MMA) == 4   # its operand pass needs workspace
    assert _call(64, 256, 8, route=6) == 1


def test_static_scratch_entry_host_checks(lib):
    vp = ctypes.c_void_p
    f = lib.q4lin_linear_fp16_static
    assert f(vp(16), vp(16), vp(16), vp(16), 256, 5120, 2048, None) == 2   # beyond its 16 MiB array
    assert "16 MiB" in q4lin.last_error_detail()
    assert f(vp(16), vp(16), vp(16), vp(16), 256, 100, 8, None) == 2       # K % 8 != 0
    assert f(None, None, None, None, 0, 5120, 8, None) == 0                # empty
    assert f(vp(16), vp(16), vp(16), vp(8), 64, 256, 8, None) == 3         # misaligned y


def test_fp16_tile_route_workspace(lib):
    # the opt-in fp16 route: fp16 X [T, K], then a per-token and a per-row int, each
    # part rounded up to 256 bytes; the default routes take none
    def r256(b):
        return -(-b // 256) * 256
    for N, K, T in [(6144, 5120, 1024), (1000, 1152, 37), (77, 72, 5)]:
        want = r256(2 * T * K) + r256(4 * T) + r256(4 * N)
        assert q4lin.workspace_bytes(N, K, T, q4lin.ROUTE_TC_FP16) == want
        for r in (q4lin.ROUTE_TC, q4lin.ROUTE_TC_SPLITK, q4lin.ROUTE_GEMV):
            assert q4lin.workspace_bytes(N, K, T, r) == 0
    # it plans like the split route (clusters along K allowed)
    assert q4lin.tile_plan(1024, 65536, 16, q4lin.ROUTE_TC_FP16)[1] > 1
    assert q4lin.tile_plan(1024, 65536, 16, q4lin.ROUTE_TC)[1] == 1


def test_valid_call_without_gpu_reports_error_not_crash(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st = _call(4, 128, 1)
    assert st in (5, 6)   # device unsupported / CUDA error: no device here


def test_tile_plan_query(lib):
    # Host-only: the planner reads device attributes when there is a device and
    # falls back to a nominal SM count when there is none.
    assert q4lin.tile_plan(6144, 5120, 1) == (0, 1)                      # GEMV route
    assert q4lin.tile_plan(6144, 5120, 64, q4lin.ROUTE_GEMV) == (0, 1)
    assert q4lin.tile_plan(6144, 5120, 0) == (0, 1)                      # empty problem
    for T, widths in ((8, {16}), (24, {32}), (48, {64}), (100, {128}), (1024, {128, 256})):
        bn, sk = q4lin.tile_plan(6144, 5120, T, q4lin.ROUTE_TC_SPLITK)
        assert bn in widths and 1 <= sk <= 8, (T, bn, sk)
        bn, sk = q4lin.tile_plan(6144, 5120, T, q4lin.ROUTE_TC)
        assert bn in widths and sk == 1, (T, bn, sk)
    # a deep K with few row tiles is split; a long N that fills the GPU is not
    assert q4lin.tile_plan(1024, 65536, 16, q4lin.ROUTE_TC_SPLITK)[1] > 1
    assert q4lin.tile_plan(65536, 1024, 16, q4lin.ROUTE_TC_SPLITK)[1] == 1
    assert q4lin.tile_plan(6144, 5120, 8) == (0, 1)   # the streaming warp-MMA route: no tiles
    with pytest.raises(q4lin.Q4LinError):
        q4lin.tile_plan(6144, 100, 8)
    with pytest.raises(q4lin.Q4LinError):
        q4lin.tile_plan(6144, 5120, 8, route=9)
    bn = ctypes.c_int(0)
    assert lib.q4lin_tile_plan(0, 6144, 5120, 8, ctypes.byref(bn), None, None, None) == 1
    sk = ctypes.c_int(0)
    assert lib.q4lin_tile_plan(0, 6144, 5120, 8, ctypes.byref(bn), ctypes.byref(sk), None, None) == 0
    # a tail launch covers exactly the tiles the main launch leaves, split along K
    for N, K, T in ((6144, 5120, 1024), (5120, 17408, 1024), (34816, 5120, 1024), (6144, 5120, 100)):
        p = q4lin.tile_plan_full(N, K, T)
        tiles = -(-N // 128) * -(-T // p["n"])
        assert 0 < p["main_tiles"] <= tiles
        if p["main_tiles"] < tiles:
            assert p["split_k"] == 1 and p["tail_split_k"] >= 2
            assert q4lin.kernel_launches(N, K, T) == 2
        else:
            assert p["tail_split_k"] == 0 and q4lin.kernel_launches(N, K, T) == 1
    assert q4lin.tile_plan_full(6144, 5120, 1) == {"n": 0, "split_k": 1, "main_tiles": 0, "tail_split_k": 0}


def test_diagnostics_host_checks(lib):
    import ctypes
    vp = ctypes.c_void_p
    # null source or sink, size not a multiple of 16: refused before any CUDA call
    assert lib.q4lin_hbm_read_probe(None, 1024, vp(256), 0, None) == 1
    assert lib.q4lin_hbm_read_probe(vp(256), 1024, None, 0, None) == 1
    assert lib.q4lin_hbm_read_probe(vp(256), 1000, vp(256), 0, None) == 1
    assert lib.q4lin_hbm_read_probe(vp(264), 1024, vp(256), 0, None) == 3
    # wait-expiry bound outside 1 .. 2^20, or no output word
    assert lib.q4lin_diag_wait_expiry(0, vp(256), None) == 1
    assert lib.q4lin_diag_wait_expiry((1 << 20) + 1, vp(256), None) == 1
    assert lib.q4lin_diag_wait_expiry(100, None, None) == 1


def test_fused_entry_points_host_checks(lib):
    vp = ctypes.c_void_p
    sw, pr = lib.q4lin_linear_swiglu, lib.q4lin_linear_pair
    a, b = vp(256), vp(512)
    # null weight, misaligned output, K not a multiple of 8, negative F: refused before any CUDA call
    assert sw(None, a, a, b, 64, 256, 4, None) == 1
    assert sw(a, a, a, vp(8), 64, 256, 4, None) == 3
    assert sw(a, a, a, b, 64, 100, 4, None) == 2
    assert sw(a, a, a, b, -1, 256, 4, None) == 1
    assert sw(None, None, None, None, 0, 256, 4, None) == 0     # empty
    assert pr(a, a, None, a, a, b, b, 64, 64, 256, 4, None) == 1
    assert pr(a, a, a, a, a, b, vp(8), 64, 64, 256, 4, None) == 3
    assert pr(a, a, a, a, a, b, b, 64, 64, 100, 4, None) == 2
    assert pr(None, None, None, None, None, None, None, 0, 0, 256, 4, None) == 0


def test_host_entry_workspace_and_host_checks(lib):
    # q4lin_linear_host: X staging, Y staging (each rounded up to 256), then the layer's own workspace
    def r256(b):
        return -(-b // 256) * 256
    for N, K, T in [(6144, 5120, 1), (6144, 5120, 16), (333, 640, 37), (40, 0, 3)]:
        want = r256(2 * T * K) + r256(2 * T * N) + q4lin.workspace_bytes(N, K, T)
        assert q4lin.host_workspace_bytes(N, K, T) == want
    assert q4lin.host_workspace_bytes(0, 128, 4) == 0 and q4lin.host_workspace_bytes(4, 100, 1) == 0
    f, vp = lib.q4lin_linear_host, ctypes.c_void_p
    assert f(vp(16), vp(16), vp(16), vp(16), 64, 256, 4, None, None) == 4        # no workspace
    assert f(vp(16), vp(16), vp(16), vp(16), 64, 256, 4, vp(128), None) == 3     # workspace not 256-aligned
    assert f(vp(16), vp(16), None, vp(16), 64, 256, 4, vp(256), None) == 1       # no X
    assert f(vp(16), vp(16), vp(16), vp(8), 64, 256, 4, vp(256), None) == 3      # y not 16-byte aligned
    assert f(None, None, None, None, 0, 256, 4, None, None) == 0                 # empty


def test_format_routes(lib):
    # Q5 / Q6: GEMV for one token, warp-MMA for 2..32, tiles beyond; W8: GEMV 1..4, warp-MMA 5..24, tiles beyond
    for q in ("q5g64", "q6g64"):
        assert q4lin.qtype_route(q, 6144, 5120, 1) == q4lin.ROUTE_GEMV
        for T in (2, 8, 32):
            assert q4lin.qtype_route(q, 6144, 5120, T) == q4lin.ROUTE_STREAM_MMA, (q, T)
            assert q4lin.kernel_launches(6144, 5120, T, q) == 2
        assert q4lin.qtype_route(q, 6144, 5120, 33) == q4lin.ROUTE_TC_SPLITK
    assert q4lin.qtype_route("w8g32", 6144, 5120, 4) == q4lin.ROUTE_GEMV
    assert q4lin.qtype_route("w8g32", 6144, 5120, 8) == q4lin.ROUTE_STREAM_MMA
    assert q4lin.qtype_route("w8g32", 6144, 5120, 25) == q4lin.ROUTE_TC_SPLITK
    assert q4lin.qtype_route("q4g64", 6144, 5120, 8) == q4lin.select_route(6144, 5120, 8)
    assert lib.q4lin_qtype_route(9, 64, 256, 8) == -1 and lib.q4lin_qtype_route(1, 64, 100, 8) == -1


def test_fused_operation_routes(lib):
    # no workspace: up to 8 tokens the warp-MMA route's one-launch form where its whole-K
    # operands fit in shared memory, the tile route otherwise
    for op in ("add", "swiglu", "pair"):
        N = 17408 if op == "swiglu" else 34816
        assert q4lin.fused_route(op, N, 5120, 1) == q4lin.ROUTE_STREAM_MMA, op
        assert q4lin.fused_route(op, N, 5120, 8) == q4lin.ROUTE_STREAM_MMA, op
        assert q4lin.fused_route(op, N, 5120, 9) == q4lin.ROUTE_TC_SPLITK, op
    assert q4lin.fused_route("add", 77, 17408, 8) == q4lin.ROUTE_TC_SPLITK    # 278 KB of operands
    assert q4lin.fused_route("add", 77, 17408, 2) == q4lin.ROUTE_STREAM_MMA   # 70 KB at 8 lanes
    assert lib.q4lin_fused_route(0, 64, 256, 4) == -1 and lib.q4lin_fused_route(4, 64, 256, 4) == -1
    assert lib.q4lin_fused_route(1, 64, 100, 4) == -1                          # K % 8 != 0
