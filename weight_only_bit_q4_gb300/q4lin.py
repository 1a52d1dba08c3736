"""ctypes binding of libq4lin.so (argument marshalling only).

Every step of the layer runs in the library's CUDA kernels; this module only
turns torch tensors into pointers and sizes and raises on a nonzero status.
If the library has not been built it raises: there is no other path.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libq4lin.so")

OK = 0
STATUS = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED_SHAPE", 3: "MISALIGNED", 4: "WORKSPACE",
          5: "DEVICE", 6: "CUDA", 7: "TIMEOUT"}
ROUTE_AUTO, ROUTE_GEMV, ROUTE_TC_SPLITK, ROUTE_TC, ROUTE_TC_FP16, ROUTE_STREAM_MMA = 0, 1, 2, 3, 4, 5
ROUTE_NAMES = {ROUTE_AUTO: "auto", ROUTE_GEMV: "gemv", ROUTE_TC_SPLITK: "tc_splitk", ROUTE_TC: "tc",
               ROUTE_TC_FP16: "tc_fp16", ROUTE_STREAM_MMA: "stream_mma"}

QTYPES = {"q4g64": 0, "q5g64": 1, "q6g64": 2, "w8g32": 3}

EXPORTS = ("q4lin_workspace_bytes", "q4lin_linear", "q4lin_linear_route", "q4lin_linear_qtype",
           "q4lin_linear_fp16_static", "q4lin_qtype_kernel_launches", "q4lin_linear_add",
           "q4lin_route_workspace_bytes", "q4lin_select_route", "q4lin_tile_plan", "q4lin_kernel_launches",
           "q4lin_status_string",
           "q4lin_device_status", "q4lin_clear_device_status", "q4lin_last_error_detail",
           "q4lin_hbm_read_probe", "q4lin_diag_wait_expiry", "q4lin_linear_swiglu", "q4lin_linear_pair",
           "q4lin_qtype_workspace_bytes", "q4lin_host_workspace_bytes", "q4lin_linear_host", "q4lin_fused_route", "q4lin_qtype_route", "q4lin_version")

_lib = None


class Q4LinError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        detail = last_error_detail()
        super().__init__(f"q4lin: {what}{STATUS.get(status, status)}: {status_string(status)}"
                         + (f" [{detail}]" if detail else ""))


def last_error_detail() -> str:
    return load().q4lin_last_error_detail().decode(errors="replace")


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the library (once).  Raises if it is missing: build it first."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"{p} not found: build it with `python -m weight_only_bit_q4_gb300.build`")
    lib = ctypes.CDLL(p)
    i64, sz, vp = ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p
    lib.q4lin_workspace_bytes.argtypes = [i64, i64, i64]
    lib.q4lin_workspace_bytes.restype = sz
    lib.q4lin_route_workspace_bytes.argtypes = [ctypes.c_int, i64, i64, i64]
    lib.q4lin_route_workspace_bytes.restype = sz
    lib.q4lin_linear.argtypes = [vp, vp, vp, vp, i64, i64, i64, vp, vp]
    lib.q4lin_linear.restype = ctypes.c_int
    lib.q4lin_linear_route.argtypes = [ctypes.c_int, vp, vp, vp, vp, i64, i64, i64, vp, vp]
    lib.q4lin_linear_qtype.argtypes = [ctypes.c_int, vp, vp, vp, vp, vp, i64, i64, i64, vp, vp]
    lib.q4lin_linear_qtype.restype = ctypes.c_int
    lib.q4lin_linear_fp16_static.argtypes = [vp, vp, vp, vp, i64, i64, i64, vp]
    lib.q4lin_linear_fp16_static.restype = ctypes.c_int
    lib.q4lin_linear_route.restype = ctypes.c_int
    lib.q4lin_select_route.argtypes = [i64, i64, i64]
    lib.q4lin_select_route.restype = ctypes.c_int
    lib.q4lin_tile_plan.argtypes = [ctypes.c_int, i64, i64, i64, ctypes.POINTER(ctypes.c_int),
                                    ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int64),
                                    ctypes.POINTER(ctypes.c_int)]
    lib.q4lin_tile_plan.restype = ctypes.c_int
    lib.q4lin_kernel_launches.argtypes = [i64, i64, i64]
    lib.q4lin_kernel_launches.restype = ctypes.c_int
    lib.q4lin_linear_add.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, vp]
    lib.q4lin_linear_add.restype = ctypes.c_int
    lib.q4lin_qtype_kernel_launches.argtypes = [ctypes.c_int, i64, i64, i64]
    lib.q4lin_qtype_kernel_launches.restype = ctypes.c_int
    lib.q4lin_status_string.argtypes = [ctypes.c_int]
    lib.q4lin_status_string.restype = ctypes.c_char_p
    lib.q4lin_device_status.argtypes = []
    lib.q4lin_device_status.restype = ctypes.c_int
    lib.q4lin_clear_device_status.argtypes = []
    lib.q4lin_clear_device_status.restype = ctypes.c_int
    lib.q4lin_last_error_detail.argtypes = []
    lib.q4lin_last_error_detail.restype = ctypes.c_char_p
    lib.q4lin_hbm_read_probe.argtypes = [vp, sz, vp, ctypes.c_int, vp]
    lib.q4lin_hbm_read_probe.restype = ctypes.c_int
    lib.q4lin_diag_wait_expiry.argtypes = [ctypes.c_uint32, vp, vp]
    lib.q4lin_diag_wait_expiry.restype = ctypes.c_int
    lib.q4lin_qtype_workspace_bytes.argtypes = [ctypes.c_int, i64, i64, i64]
    lib.q4lin_qtype_workspace_bytes.restype = sz
    lib.q4lin_linear_swiglu.argtypes = [vp, vp, vp, vp, i64, i64, i64, vp]
    lib.q4lin_linear_swiglu.restype = ctypes.c_int
    lib.q4lin_linear_pair.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, vp]
    lib.q4lin_linear_pair.restype = ctypes.c_int
    lib.q4lin_host_workspace_bytes.argtypes = [i64, i64, i64]
    lib.q4lin_host_workspace_bytes.restype = sz
    lib.q4lin_linear_host.argtypes = [vp, vp, vp, vp, i64, i64, i64, vp, vp]
    lib.q4lin_linear_host.restype = ctypes.c_int
    lib.q4lin_qtype_route.argtypes = [ctypes.c_int, i64, i64, i64]
    lib.q4lin_qtype_route.restype = ctypes.c_int
    lib.q4lin_fused_route.argtypes = [ctypes.c_int, i64, i64, i64]
    lib.q4lin_fused_route.restype = ctypes.c_int
    lib.q4lin_version.argtypes = []
    lib.q4lin_version.restype = ctypes.c_char_p
    if path is None:
        _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().q4lin_status_string(int(status)).decode()


def version() -> str:
    return load().q4lin_version().decode()


def workspace_bytes(N: int, K: int, T: int, route: int = ROUTE_AUTO) -> int:
    if route == ROUTE_AUTO:
        return int(load().q4lin_workspace_bytes(N, K, T))
    return int(load().q4lin_route_workspace_bytes(route, N, K, T))


def select_route(N: int, K: int, T: int) -> int:
    return int(load().q4lin_select_route(N, K, T))


def tile_plan(N: int, K: int, T: int, route: int = ROUTE_AUTO) -> tuple:
    """(token-tile width, split-K cluster size) of the tensor-core route's main launch; (0, 1) for the GEMV."""
    p = tile_plan_full(N, K, T, route)
    return p["n"], p["split_k"]


def tile_plan_full(N: int, K: int, T: int, route: int = ROUTE_AUTO) -> dict:
    """The whole tensor-core plan: tile width, main-launch split, main-launch tiles, tail split (0 = none)."""
    bn, sk, mt, ts = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int64(0), ctypes.c_int(0)
    st = load().q4lin_tile_plan(route, N, K, T, ctypes.byref(bn), ctypes.byref(sk), ctypes.byref(mt),
                                ctypes.byref(ts))
    if st != OK:
        raise Q4LinError(st, "tile plan: ")
    return {"n": int(bn.value), "split_k": int(sk.value), "main_tiles": int(mt.value), "tail_split_k": int(ts.value)}


def kernel_launches(N: int, K: int, T: int, qtype: str = "q4g64") -> int:
    """Kernels one call launches (q4lin_linear, or q4lin_linear_qtype for another format)."""
    if qtype == "q4g64":
        return int(load().q4lin_kernel_launches(N, K, T))
    return int(load().q4lin_qtype_kernel_launches(QTYPES[qtype], N, K, T))


_IMPLEMENTED = (ROUTE_GEMV, ROUTE_TC_SPLITK, ROUTE_TC, ROUTE_TC_FP16, ROUTE_STREAM_MMA)


def implemented_routes():
    """Routes the library can run (the others return INVALID_ARG)."""
    return _IMPLEMENTED


def device_status() -> int:
    return int(load().q4lin_device_status())


def clear_device_status() -> int:
    return int(load().q4lin_clear_device_status())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def linear_raw(wq_ptr, scales_ptr, x_ptr, y_ptr, N, K, T, ws_ptr=None, stream=None,
               route: int = ROUTE_AUTO) -> int:
    """Pointer-level call; returns the status code (no exception)."""
    lib = load()
    if route == ROUTE_AUTO:
        return int(lib.q4lin_linear(wq_ptr, scales_ptr, x_ptr, y_ptr, N, K, T, ws_ptr, stream))
    return int(lib.q4lin_linear_route(route, wq_ptr, scales_ptr, x_ptr, y_ptr, N, K, T, ws_ptr, stream))


def linear(wq, scales, x, y=None, workspace=None, stream=None, route: int = ROUTE_AUTO):
    """Y[T, N] (bf16) = dequant(wq, scales) applied to X[T, K] (bf16) on the GPU.

    wq: uint8 [N, Kp/2]; scales: fp16 (or int16/uint16 bit patterns) [N, Kp/64],
    Kp = K rounded up to 128 (the planes' stored width; columns k >= K are
    padding); x: bf16 [T, K]; all CUDA, contiguous.  ``y`` (bf16 [T, N]) and
    ``workspace`` (uint8, >= workspace_bytes) are allocated here with torch if
    not given.  Runs on ``stream`` (a torch.cuda.Stream) or the current stream.
    """
    import torch

    T, K = x.shape
    N = wq.shape[0]
    Kp = (K + 127) // 128 * 128
    if tuple(wq.shape) != (N, Kp // 2) or tuple(scales.shape) != (N, Kp // 64):
        raise ValueError(f"shape mismatch: wq {tuple(wq.shape)} scales {tuple(scales.shape)} x {tuple(x.shape)}")
    for name, t in (("wq", wq), ("scales", scales), ("x", x)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if wq.dtype != torch.uint8 or x.dtype != torch.bfloat16 or scales.element_size() != 2:
        raise ValueError("dtypes: wq uint8, scales fp16 bits, x bf16")
    if y is None:
        y = torch.empty((T, N), dtype=torch.bfloat16, device=x.device)
    elif y.shape != (T, N) or y.dtype != torch.bfloat16 or not y.is_contiguous():
        raise ValueError("y must be a contiguous bf16 [T, N] tensor")
    need = workspace_bytes(N, K, T, route)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    s = (stream or torch.cuda.current_stream(x.device)).cuda_stream
    st = linear_raw(_ptr(wq), _ptr(scales), _ptr(x), _ptr(y), N, K, T,
                    _ptr(workspace) if need else None, ctypes.c_void_p(s), route)
    if st != OK:
        raise Q4LinError(st)
    return y


FUSED_OPS = {"add": 1, "swiglu": 2, "pair": 3}


def qtype_route(qtype: str, N: int, K: int, T: int) -> int:
    """Route q4lin_linear_qtype takes for this format and shape."""
    return int(load().q4lin_qtype_route(QTYPES[qtype], N, K, T))


def fused_route(op: str, N: int, K: int, T: int) -> int:
    """Route of a fused operation ("add", "swiglu", "pair"; N = F for swiglu, rows per weight for pair)."""
    return int(load().q4lin_fused_route(FUSED_OPS[op], N, K, T))


def host_workspace_bytes(N: int, K: int, T: int) -> int:
    return int(load().q4lin_host_workspace_bytes(N, K, T))


def linear_host(wq, scales, x_host, y_host=None, workspace=None, stream=None):
    """q4lin_linear_host: X and Y in page-locked host memory, the weights on the GPU.

    x_host: pinned CPU bf16 [T, K] (or int16 bit patterns); ``y_host`` (pinned CPU bf16
    [T, N]) and ``workspace`` (CUDA uint8, >= host_workspace_bytes) are allocated here if
    not given.  The call is stream-ordered: y_host holds the result once ``stream`` (a
    torch.cuda.Stream, default the current one) has passed it.
    """
    import torch

    T, K = x_host.shape
    N = wq.shape[0]
    Kp = (K + 127) // 128 * 128
    if tuple(wq.shape) != (N, Kp // 2) or tuple(scales.shape) != (N, Kp // 64):
        raise ValueError(f"shape mismatch: wq {tuple(wq.shape)} scales {tuple(scales.shape)} x {tuple(x_host.shape)}")
    for name, t in (("wq", wq), ("scales", scales)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if x_host.is_cuda or not x_host.is_contiguous() or x_host.element_size() != 2:
        raise ValueError("x_host must be a contiguous 2-byte CPU tensor (pinned)")
    if y_host is None:
        y_host = torch.empty((T, N), dtype=torch.bfloat16).pin_memory()
    elif y_host.is_cuda or tuple(y_host.shape) != (T, N) or y_host.element_size() != 2 or not y_host.is_contiguous():
        raise ValueError("y_host must be a contiguous 2-byte CPU [T, N] tensor (pinned)")
    if workspace is None:
        workspace = torch.empty(max(host_workspace_bytes(N, K, T), 256), dtype=torch.uint8, device=wq.device)
    s = (stream or torch.cuda.current_stream(wq.device)).cuda_stream
    st = int(load().q4lin_linear_host(_ptr(wq), _ptr(scales), _ptr(x_host), _ptr(y_host), N, K, T,
                                      _ptr(workspace), ctypes.c_void_p(s)))
    if st != OK:
        raise Q4LinError(st)
    return y_host


def linear_add(wq, scales, x, r, y=None, stream=None):
    """LinearAdd: Y = W . X + R (bf16 [T, N]); ``y`` may be ``r`` itself for an in-place add."""
    import torch

    T, K = x.shape
    N = wq.shape[0]
    Kp = (K + 127) // 128 * 128
    if tuple(wq.shape) != (N, Kp // 2) or tuple(scales.shape) != (N, Kp // 64) or tuple(r.shape) != (T, N):
        raise ValueError(f"shape mismatch: wq {tuple(wq.shape)} scales {tuple(scales.shape)} x {tuple(x.shape)} "
                         f"r {tuple(r.shape)}")
    for name, t in (("wq", wq), ("scales", scales), ("x", x), ("r", r)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if y is None:
        y = torch.empty((T, N), dtype=torch.bfloat16, device=x.device)
    s = (stream or torch.cuda.current_stream(x.device)).cuda_stream
    st = int(load().q4lin_linear_add(_ptr(wq), _ptr(scales), _ptr(x), _ptr(r), _ptr(y), N, K, T, ctypes.c_void_p(s)))
    if st != OK:
        raise Q4LinError(st)
    return y


def linear_qtype(qtype: str, planes, scales, x, y=None, stream=None):
    """Y[T, N] (bf16) for a sibling weight format ("q4g64", "q5g64", "q6g64", "w8g32").

    planes: (codes,) for q4g64 / w8g32, (low codes, high bits) for q5g64 / q6g64;
    planes and scales stored for Kp = K rounded up to 128 columns (see q4lin.h);
    all CUDA, contiguous.  Workspace (W8 beyond the decode GEMV) is allocated here.
    """
    import torch

    qt = QTYPES[qtype]
    T, K = x.shape
    Kp = (K + 127) // 128 * 128
    codes = planes[0]
    N = codes.shape[0]
    code_cols = Kp if qtype == "w8g32" else Kp // 2
    group = 32 if qtype == "w8g32" else 64
    bits = {"q5g64": 1, "q6g64": 2}.get(qtype, 0)
    if tuple(codes.shape) != (N, code_cols) or tuple(scales.shape) != (N, Kp // group):
        raise ValueError(f"shape mismatch: codes {tuple(codes.shape)} scales {tuple(scales.shape)} x {tuple(x.shape)}")
    high = planes[1] if bits else None
    if bits and tuple(high.shape) != (N, Kp * bits // 8):
        raise ValueError(f"shape mismatch: high {tuple(high.shape)}")
    for name, t in (("codes", codes), ("scales", scales), ("x", x)) + ((("high", high),) if bits else ()):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if y is None:
        y = torch.empty((T, N), dtype=torch.bfloat16, device=x.device)
    need = int(load().q4lin_qtype_workspace_bytes(qt, N, K, T))
    ws = torch.empty(need, dtype=torch.uint8, device=x.device) if need else None
    s = (stream or torch.cuda.current_stream(x.device)).cuda_stream
    st = int(load().q4lin_linear_qtype(qt, _ptr(codes), _ptr(high) if bits else None, _ptr(scales), _ptr(x),
                                       _ptr(y), N, K, T, _ptr(ws), ctypes.c_void_p(s)))
    if st != OK:
        raise Q4LinError(st)
    return y


def hbm_read_probe(buf, sink, blocks: int = 0, stream=None) -> None:
    """Enqueue one pass of the HBM read probe over ``buf`` (a CUDA tensor, 16-byte
    aligned, size a multiple of 16 bytes); ``sink`` is an int32 CUDA tensor with at
    least ``blocks`` (default four per SM) elements."""
    import torch

    s = (stream or torch.cuda.current_stream(buf.device)).cuda_stream
    st = int(load().q4lin_hbm_read_probe(_ptr(buf), buf.numel() * buf.element_size(), _ptr(sink), int(blocks),
                                         ctypes.c_void_p(s)))
    if st != OK:
        raise Q4LinError(st, "hbm read probe: ")


def diag_wait_expiry(limit: int, out, stream=None) -> None:
    """Enqueue the wait-expiry check (see q4lin.h); ``out`` is an int32 CUDA tensor."""
    import torch

    s = (stream or torch.cuda.current_stream(out.device)).cuda_stream
    st = int(load().q4lin_diag_wait_expiry(int(limit), _ptr(out), ctypes.c_void_p(s)))
    if st != OK:
        raise Q4LinError(st, "wait expiry check: ")


def _check_planes(wq, scales, K, what):
    Kp = (K + 127) // 128 * 128
    if wq.shape[1] != Kp // 2 or tuple(scales.shape) != (wq.shape[0], Kp // 64):
        raise ValueError(f"{what}: shape mismatch wq {tuple(wq.shape)} scales {tuple(scales.shape)} K {K}")
    for name, t in (("wq", wq), ("scales", scales)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{what}: {name} must be a contiguous CUDA tensor")


def linear_swiglu(wq, scales, x, y=None, stream=None):
    """LinearSwiGLU: Y[T, F] = silu(W[:F] . X) * (W[F:] . X) for a packed weight of 2F rows."""
    import torch

    T, K = x.shape
    n2 = wq.shape[0]
    if n2 % 2:
        raise ValueError("the gate/up weight has an even number of rows")
    F = n2 // 2
    _check_planes(wq, scales, K, "linear_swiglu")
    if y is None:
        y = torch.empty((T, F), dtype=torch.bfloat16, device=x.device)
    s = (stream or torch.cuda.current_stream(x.device)).cuda_stream
    st = int(load().q4lin_linear_swiglu(_ptr(wq), _ptr(scales), _ptr(x), _ptr(y), F, K, T, ctypes.c_void_p(s)))
    if st != OK:
        raise Q4LinError(st)
    return y


def linear_pair(wq_a, scales_a, wq_b, scales_b, x, y_a=None, y_b=None, stream=None):
    """LinearPair: (W_a . X, W_b . X) in one call; returns (Y_a [T, N_a], Y_b [T, N_b])."""
    import torch

    T, K = x.shape
    _check_planes(wq_a, scales_a, K, "linear_pair a")
    _check_planes(wq_b, scales_b, K, "linear_pair b")
    Na, Nb = wq_a.shape[0], wq_b.shape[0]
    if y_a is None:
        y_a = torch.empty((T, Na), dtype=torch.bfloat16, device=x.device)
    if y_b is None:
        y_b = torch.empty((T, Nb), dtype=torch.bfloat16, device=x.device)
    s = (stream or torch.cuda.current_stream(x.device)).cuda_stream
    st = int(load().q4lin_linear_pair(_ptr(wq_a), _ptr(scales_a), _ptr(wq_b), _ptr(scales_b), _ptr(x), _ptr(y_a),
                                      _ptr(y_b), Na, Nb, K, T, ctypes.c_void_p(s)))
    if st != OK:
        raise Q4LinError(st)
    return y_a, y_b
