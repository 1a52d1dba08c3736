// C-ABI entry points of q4lin: argument checks, route selection, dispatch.
//
// The public call mirrors the linear-benchmark contract's operation
// (linear-benchmark.md, "status and scope": linear(x, w, out, policy,
// workspace, stream)) with a workspace capacity query (section 1.1) and a
// format selector that rejects unsupported points (section 1.1) and returns
// one host launcher per exact (N, K, T) (section 8.2).
#include <cstdio>
#include <cstring>

#include "q4lin.h"
#include "q4_internal.h"

namespace q4 {

static thread_local char g_detail[512];

void set_error_detail(const char* what) {
  std::snprintf(g_detail, sizeof(g_detail), "%s", what);
}

int cuda_check(cudaError_t e, const char* where) {
  if (e == cudaSuccess) return 0;
  std::snprintf(g_detail, sizeof(g_detail), "%s: %s (%s)", where, cudaGetErrorString(e), cudaGetErrorName(e));
  return 6;  // Q4LIN_ERR_CUDA
}

}  // namespace q4

extern "C" const char* q4lin_status_string(int status);

namespace {

constexpr int64_t kMaxDim = (int64_t)1 << 40;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int validate_sizes(int64_t N, int64_t K, int64_t T) {
  if (N < 0 || K < 0 || T < 0) return Q4LIN_ERR_INVALID_ARG;
  if (N > kMaxDim || K > kMaxDim || T > kMaxDim) return Q4LIN_ERR_INVALID_ARG;
  // every byte count derived from the sizes must stay far from int64 overflow
  if ((double)N * (double)K > 9.0e17 || (double)T * (double)K > 9.0e17 ||
      (double)N * (double)T > 9.0e17)
    return Q4LIN_ERR_INVALID_ARG;
  // any K whose X rows stay 16-byte aligned; the weight planes are stored for K
  // rounded up to 128 (K_pad) and the padded positions are ignored
  if (K % 8 != 0) return Q4LIN_ERR_UNSUPPORTED_SHAPE;
  return Q4LIN_OK;
}

// Host-only argument validation; touches no CUDA API.
int validate(const uint8_t* wq, const uint16_t* scales, const uint16_t* x, uint16_t* y,
             int64_t N, int64_t K, int64_t T) {
  const int st = validate_sizes(N, K, T);
  if (st != Q4LIN_OK) return st;
  if (N == 0 || T == 0) return Q4LIN_OK;
  if (y == nullptr) return Q4LIN_ERR_INVALID_ARG;
  if (!aligned16(y)) return Q4LIN_ERR_MISALIGNED;
  if (K == 0) return Q4LIN_OK;
  if (wq == nullptr || scales == nullptr || x == nullptr) return Q4LIN_ERR_INVALID_ARG;
  if (!aligned16(wq) || !aligned16(scales) || !aligned16(x)) return Q4LIN_ERR_MISALIGNED;
  return Q4LIN_OK;
}

// The library is built for sm_103a only (compute capability 10.3); any other device
// would fail every launch with "no kernel image", so it is refused up front.
int check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return Q4LIN_ERR_CUDA;
  static int cached[128];   // 0 unknown, 1 ok, 2 not supported
  if (dev >= 0 && dev < 128 && cached[dev] != 0) {
    if (cached[dev] == 2) q4::set_error_detail("device is not compute capability 10.3 (the library is built for sm_103a)");
    return cached[dev] == 1 ? Q4LIN_OK : Q4LIN_ERR_DEVICE;
  }
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return Q4LIN_ERR_CUDA;
  const int ok = (major == 10 && minor == 3) ? 1 : 2;
  if (dev >= 0 && dev < 128) cached[dev] = ok;
  if (ok != 1) {
    char msg[160];
    std::snprintf(msg, sizeof(msg), "device is compute capability %d.%d; the library is built for sm_103a (10.3)",
                  major, minor);
    q4::set_error_detail(msg);
  }
  return ok == 1 ? Q4LIN_OK : Q4LIN_ERR_DEVICE;
}

// Tokens at or below which the streaming warp-MMA route is chosen (where it has a plan):
// measured on 6144 x 5120 against the tile route, 12.5 against 18.1 us at T = 8, 16.5 us
// at T = 24, level at T = 32.
constexpr int64_t kMmaMaxT = 32;     // Q4: one pass of the warp-MMA route (measured faster than 32-token tiles)
constexpr int64_t kW8MmaMaxT = 24;   // W8G32: the warp-MMA route up to here, the tile route beyond

int route_for(int64_t N, int64_t K, int64_t T) {
  // One token: the streaming CUDA-core GEMV.  Two to kMmaMaxT tokens: the streaming
  // warp-MMA route (every weight read once and decoded once for all the tokens);
  // above, the tcgen05 tile route, whose planner splits K only where that fills the
  // GPU better.  Shapes a route has no plan for fall through to the next one.
  if (T == 1 && q4::gemv_stream_ok(N, K, T)) return Q4LIN_ROUTE_GEMV;
  if (T <= kMmaMaxT && q4::mma_supported(N, K, T)) return Q4LIN_ROUTE_STREAM_MMA;
  if (!q4::tc_supported(N, K, T)) return Q4LIN_ROUTE_GEMV;
  if (T <= 4 && q4::gemv_stream_ok(N, K, T)) return Q4LIN_ROUTE_GEMV;
  return Q4LIN_ROUTE_TC_SPLITK;
}

size_t round256(size_t b) { return (b + 255) / 256 * 256; }

size_t route_ws(int route, int64_t N, int64_t K, int64_t T) {
  switch (route) {
    case Q4LIN_ROUTE_GEMV: return round256(q4::gemv_workspace_bytes(N, K, T));
    case Q4LIN_ROUTE_TC:
    case Q4LIN_ROUTE_TC_SPLITK:
    case Q4LIN_ROUTE_TC_FP16: return round256(q4::tc_workspace_bytes(route, N, K, T));
    case Q4LIN_ROUTE_STREAM_MMA: return round256(q4::mma_workspace_bytes(N, K, T));
    default: return 0;
  }
}

int run_impl(int route, const uint8_t* wq, const uint16_t* scales, const uint16_t* x, uint16_t* y,
             int64_t N, int64_t K, int64_t T, void* workspace, void* stream) {
  int st = validate(wq, scales, x, y, N, K, T);
  if (st != Q4LIN_OK) return st;
  if (N == 0 || T == 0) return Q4LIN_OK;
  if (route == Q4LIN_ROUTE_AUTO) route = route_for(N, K, T);
  if (route < Q4LIN_ROUTE_GEMV || route > Q4LIN_ROUTE_STREAM_MMA) return Q4LIN_ERR_INVALID_ARG;
  if (route == Q4LIN_ROUTE_STREAM_MMA && K > 0 && !q4::mma_supported(N, K, T)) {
    q4::set_error_detail("streaming warp-MMA route: no shared-memory plan for this shape");
    return Q4LIN_ERR_UNSUPPORTED_SHAPE;
  }
  const size_t ws = route_ws(route, N, K, T);
  if (ws > 0 && workspace == nullptr) return Q4LIN_ERR_WORKSPACE;
  if (ws > 0 && (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return Q4LIN_ERR_MISALIGNED;
  st = check_device();
  if (st != Q4LIN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (K == 0) return q4::cuda_check(cudaMemsetAsync(y, 0, (size_t)N * (size_t)T * 2, s), "zero fill of y");
  q4::LinearArgs a{wq, scales, x, y, N, K, T, workspace, s};
  switch (route) {
    case Q4LIN_ROUTE_GEMV: return q4::gemv_launch(a);
    case Q4LIN_ROUTE_TC:
    case Q4LIN_ROUTE_TC_SPLITK:
    case Q4LIN_ROUTE_TC_FP16: return q4::tc_launch(a, route);
    case Q4LIN_ROUTE_STREAM_MMA: return q4::mma_launch(a);
    default: return Q4LIN_ERR_INVALID_ARG;
  }
}

// Sibling formats: the same checks as the Q4 layer, plus the high-bit plane for
// Q5G64 / Q6G64, then the streaming GEMV (1..4 tokens) or UNSUPPORTED_SHAPE.
// W8G32 beyond the warp-MMA route's token range takes the tile route.
bool w8_tile(int64_t N, int64_t K, int64_t T) { return T > kW8MmaMaxT && q4::tc_supported(N, K, T); }

// Route of a sibling format (K > 0):
//   Q5G64 / Q6G64: the decode GEMV for one token; the streaming warp-MMA route for 2..32
//     tokens (the high bits joined to the nibble operands; its operand pass needs
//     workspace); the exact tile route beyond (token tiles up to 128 wide); where a route
//     has no plan, the GEMV up to 4 tokens, else the tile route.
//   W8G32: the decode GEMV for 1..4 tokens, the warp-MMA route up to 24, the tile route beyond.
int qtype_route(int qtype, int64_t N, int64_t K, int64_t T) {
  const bool q56 = qtype == Q4LIN_QTYPE_Q5G64 || qtype == Q4LIN_QTYPE_Q6G64;
  if (q56) {
    if (T == 1 && q4::gemv_stream_ok(N, K, T, qtype)) return Q4LIN_ROUTE_GEMV;
    if (T <= kMmaMaxT && q4::mma_supported(N, K, T, qtype)) return Q4LIN_ROUTE_STREAM_MMA;
    if (q4::gemv_stream_ok(N, K, T, qtype) || !q4::tc_supported(N, K, T)) return Q4LIN_ROUTE_GEMV;
    return Q4LIN_ROUTE_TC_SPLITK;
  }
  if (q4::gemv_stream_ok(N, K, T, qtype)) return Q4LIN_ROUTE_GEMV;
  if (w8_tile(N, K, T)) return Q4LIN_ROUTE_TC_SPLITK;
  if (q4::mma_supported(N, K, T, qtype)) return Q4LIN_ROUTE_STREAM_MMA;
  return Q4LIN_ROUTE_GEMV;   // refused there (UNSUPPORTED_SHAPE)
}

int run_qtype_impl(int qtype, const uint8_t* codes, const uint8_t* high, const uint16_t* scales,
                   const uint16_t* x, uint16_t* y, int64_t N, int64_t K, int64_t T, void* workspace, void* stream) {
  int st = validate(codes, scales, x, y, N, K, T);
  if (st != Q4LIN_OK) return st;
  if (N == 0 || T == 0) return Q4LIN_OK;
  const bool needs_high = qtype == Q4LIN_QTYPE_Q5G64 || qtype == Q4LIN_QTYPE_Q6G64;
  if (K > 0 && needs_high && high == nullptr) return Q4LIN_ERR_INVALID_ARG;
  if (K > 0 && needs_high && !aligned16(high)) return Q4LIN_ERR_MISALIGNED;
  st = check_device();
  if (st != Q4LIN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (K == 0) return q4::cuda_check(cudaMemsetAsync(y, 0, (size_t)N * (size_t)T * 2, s), "zero fill of y");
  q4::LinearArgs a{codes, scales, x, y, N, K, T, nullptr, s};
  a.fmt = qtype;
  a.wh = needs_high ? high : nullptr;
  switch (qtype_route(qtype, N, K, T)) {
    case Q4LIN_ROUTE_TC_SPLITK: return q4::tc_launch(a, Q4LIN_ROUTE_TC_SPLITK);
    case Q4LIN_ROUTE_STREAM_MMA: {
      const size_t ws = round256(q4::mma_workspace_bytes(N, K, T, qtype));
      if (ws > 0 && workspace == nullptr) return Q4LIN_ERR_WORKSPACE;
      if (ws > 0 && (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return Q4LIN_ERR_MISALIGNED;
      a.workspace = workspace;
      return q4::mma_launch(a);
    }
    default: return q4::gemv_launch_fmt(a);
  }
}

int run(int route, const uint8_t* wq, const uint16_t* scales, const uint16_t* x, uint16_t* y, int64_t N,
        int64_t K, int64_t T, void* workspace, void* stream) {
  q4::set_error_detail("");
  const int st = run_impl(route, wq, scales, x, y, N, K, T, workspace, stream);
  if (st != Q4LIN_OK && q4::g_detail[0] == 0) q4::set_error_detail(q4lin_status_string(st));
  return st;
}

// The device-side address of page-locked host memory of this process (nullptr for
// pageable or device memory): what the staging kernels of q4lin_linear_host access.
const void* host_device_ptr(const void* p) {
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
}

int run_host_impl(const uint8_t* wq, const uint16_t* scales, const uint16_t* x_host, uint16_t* y_host, int64_t N,
                  int64_t K, int64_t T, void* workspace, void* stream) {
  int st = validate(wq, scales, x_host, y_host, N, K, T);
  if (st != Q4LIN_OK || N == 0 || T == 0) return st;
  if (workspace == nullptr) return Q4LIN_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return Q4LIN_ERR_MISALIGNED;
  st = check_device();
  if (st != Q4LIN_OK) return st;
  const void* xd = K > 0 ? host_device_ptr(x_host) : nullptr;   // K == 0: X is not read
  void* yd = const_cast<void*>(host_device_ptr(y_host));
  if ((K > 0 && xd == nullptr) || yd == nullptr) {
    q4::set_error_detail("x_host and y_host must be page-locked host memory of this process "
                         "(cudaHostAlloc, or cudaHostRegister and mapped)");
    return Q4LIN_ERR_INVALID_ARG;
  }
  const size_t xb = round256((size_t)T * (size_t)K * 2), yb = round256((size_t)T * (size_t)N * 2);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint16_t* xs = reinterpret_cast<uint16_t*>(ws);
  uint16_t* ys = reinterpret_cast<uint16_t*>(ws + xb);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (K == 0) {  // the empty sum: zeros staged on the device, then copied out
    if ((st = run_impl(Q4LIN_ROUTE_AUTO, wq, scales, xs, ys, N, K, T, ws + xb + yb, stream)) != Q4LIN_OK) return st;
    return q4::stage_copy(ys, yd, (size_t)T * (size_t)N * 2, s);
  }
  // X is staged (the routes read it with bulk and tensor copies); every route stores Y with
  // plain stores, which write the page-locked buffer directly
  if ((st = q4::stage_copy(xd, xs, (size_t)T * (size_t)K * 2, s)) != Q4LIN_OK) return st;
  return run_impl(Q4LIN_ROUTE_AUTO, wq, scales, xs, static_cast<uint16_t*>(yd), N, K, T, ws + xb + yb, stream);
}

// The fused operations take no workspace: up to 8 tokens they run the warp-MMA route's
// one-launch form (the streaming kernel converts X itself) where its shared memory fits,
// otherwise the exact tile route.
constexpr int64_t kFusedMmaMaxT = 8;

bool fused_op_on_mma(int64_t N, int64_t K, int64_t T, bool swiglu = false) {
  return N > 0 && K > 0 && T > 0 && T <= kFusedMmaMaxT && q4::mma_fused_supported(N, K, T, 0, swiglu);
}

}  // namespace

extern "C" {

int q4lin_qtype_route(int qtype, int64_t N, int64_t K, int64_t T) {
  if (qtype == Q4LIN_QTYPE_Q4G64) return q4lin_select_route(N, K, T);
  if (qtype < Q4LIN_QTYPE_Q5G64 || qtype > Q4LIN_QTYPE_W8G32 || validate_sizes(N, K, T) != Q4LIN_OK) return -1;
  return qtype_route(qtype, N, K, T);
}

int q4lin_fused_route(int op, int64_t N, int64_t K, int64_t T) {
  if (op < 1 || op > 3 || validate_sizes(N, K, T) != Q4LIN_OK) return -1;
  return fused_op_on_mma(N, K, T, op == 2) ? Q4LIN_ROUTE_STREAM_MMA : Q4LIN_ROUTE_TC_SPLITK;
}

size_t q4lin_host_workspace_bytes(int64_t N, int64_t K, int64_t T) {
  if (validate_sizes(N, K, T) != Q4LIN_OK || N == 0 || T == 0) return 0;
  return round256((size_t)T * (size_t)K * 2) + round256((size_t)T * (size_t)N * 2) + q4lin_workspace_bytes(N, K, T);
}

int q4lin_linear_host(const uint8_t* wq, const uint16_t* scales, const uint16_t* x_host, uint16_t* y_host,
                      int64_t N, int64_t K, int64_t T, void* workspace, void* stream) {
  q4::set_error_detail("");
  const int st = run_host_impl(wq, scales, x_host, y_host, N, K, T, workspace, stream);
  if (st != Q4LIN_OK && q4::g_detail[0] == 0) q4::set_error_detail(q4lin_status_string(st));
  return st;
}

size_t q4lin_workspace_bytes(int64_t N, int64_t K, int64_t T) {
  if (validate_sizes(N, K, T) != Q4LIN_OK || N == 0 || K == 0 || T == 0) return 0;
  return route_ws(route_for(N, K, T), N, K, T);
}

size_t q4lin_route_workspace_bytes(int route, int64_t N, int64_t K, int64_t T) {
  if (validate_sizes(N, K, T) != Q4LIN_OK || N == 0 || K == 0 || T == 0) return 0;
  if (route == Q4LIN_ROUTE_AUTO) route = route_for(N, K, T);
  return route_ws(route, N, K, T);
}

int q4lin_select_route(int64_t N, int64_t K, int64_t T) { return route_for(N, K, T); }

int q4lin_tile_plan(int route, int64_t N, int64_t K, int64_t T, int* tile_n, int* split_k, int64_t* main_tiles,
                    int* tail_split_k) {
  if (tile_n == nullptr || split_k == nullptr) return Q4LIN_ERR_INVALID_ARG;
  if (route < Q4LIN_ROUTE_AUTO || route > Q4LIN_ROUTE_STREAM_MMA) return Q4LIN_ERR_INVALID_ARG;
  if (validate_sizes(N, K, T) != Q4LIN_OK) return Q4LIN_ERR_INVALID_ARG;
  if (route == Q4LIN_ROUTE_AUTO) route = route_for(N, K, T);
  q4::TcPlan pl{0, 1, 0, 0};
  if (route != Q4LIN_ROUTE_GEMV && route != Q4LIN_ROUTE_STREAM_MMA && N > 0 && T > 0 && K > 0 &&
      q4::tc_supported(N, K, T))
    pl = q4::tc_plan_current_device(route, N, K, T);
  *tile_n = pl.bn;
  *split_k = pl.splitk;
  if (main_tiles != nullptr) *main_tiles = pl.main_tiles;
  if (tail_split_k != nullptr) *tail_split_k = pl.tail_splitk;
  return Q4LIN_OK;
}

int q4lin_kernel_launches(int64_t N, int64_t K, int64_t T) {
  if (validate_sizes(N, K, T) != Q4LIN_OK || N == 0 || T == 0) return 0;
  if (K == 0) return 1;  // the zero fill
  const int route = route_for(N, K, T);
  switch (route) {
    case Q4LIN_ROUTE_GEMV: return q4::gemv_launch_count(N, K, T);
    case Q4LIN_ROUTE_TC:
    case Q4LIN_ROUTE_TC_SPLITK:
    case Q4LIN_ROUTE_TC_FP16: return q4::tc_launch_count(route, N, K, T);
    case Q4LIN_ROUTE_STREAM_MMA: return q4::mma_launch_count(N, K, T);
    default: return 0;
  }
}

int q4lin_linear_add(const uint8_t* wq, const uint16_t* scales, const uint16_t* x, const uint16_t* r, uint16_t* y,
                     int64_t N, int64_t K, int64_t T, void* stream) {
  q4::set_error_detail("");
  int st = validate(wq, scales, x, y, N, K, T);
  const bool warp_mma = fused_op_on_mma(N, K, T);
  if (st == Q4LIN_OK && N > 0 && T > 0) {
    if (r == nullptr) st = Q4LIN_ERR_INVALID_ARG;
    else if (!aligned16(r)) st = Q4LIN_ERR_MISALIGNED;
    else if (K > 0 && !warp_mma && !q4::tc_supported(N, K, T)) st = Q4LIN_ERR_INVALID_ARG;
  }
  if (st == Q4LIN_OK && N > 0 && T > 0) st = check_device();
  if (st == Q4LIN_OK && N > 0 && T > 0) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0) {  // the empty sum: Y = R
      if (r != y)
        st = q4::cuda_check(cudaMemcpyAsync(y, r, (size_t)N * (size_t)T * 2, cudaMemcpyDeviceToDevice, s),
                            "copy of the residual");
    } else {
      q4::LinearArgs a{wq, scales, x, y, N, K, T, nullptr, s};
      a.r = r;
      st = warp_mma ? q4::mma_launch(a, true) : q4::tc_launch(a, Q4LIN_ROUTE_TC_SPLITK);
    }
  }
  if (st != Q4LIN_OK && q4::g_detail[0] == 0) q4::set_error_detail(q4lin_status_string(st));
  return st;
}

int q4lin_linear_swiglu(const uint8_t* wq, const uint16_t* scales, const uint16_t* x, uint16_t* y, int64_t F,
                        int64_t K, int64_t T, void* stream) {
  q4::set_error_detail("");
  int st = Q4LIN_OK;
  if (F < 0 || F > kMaxDim / 2) st = Q4LIN_ERR_INVALID_ARG;
  if (st == Q4LIN_OK) st = validate(wq, scales, x, y, 2 * F, K, T);
  const bool warp_mma = st == Q4LIN_OK && fused_op_on_mma(F, K, T, true);
  if (st == Q4LIN_OK && F > 0 && T > 0 && K > 0 && !warp_mma && !q4::tc_supported(2 * F, K, T))
    st = Q4LIN_ERR_INVALID_ARG;
  if (st == Q4LIN_OK && F > 0 && T > 0) st = check_device();
  if (st == Q4LIN_OK && F > 0 && T > 0) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0) {  // gate = up = 0: silu(0) * 0 = +0
      st = q4::cuda_check(cudaMemsetAsync(y, 0, (size_t)F * (size_t)T * 2, s), "zero fill of y");
    } else {
      q4::LinearArgs a{wq, scales, x, y, F, K, T, nullptr, s};
      a.mode = 1;
      st = warp_mma ? q4::mma_launch(a, true) : q4::tc_launch(a, Q4LIN_ROUTE_TC_SPLITK);
    }
  }
  if (st != Q4LIN_OK && q4::g_detail[0] == 0) q4::set_error_detail(q4lin_status_string(st));
  return st;
}

int q4lin_linear_pair(const uint8_t* wq_a, const uint16_t* scales_a, const uint8_t* wq_b, const uint16_t* scales_b,
                      const uint16_t* x, uint16_t* y_a, uint16_t* y_b, int64_t N_a, int64_t N_b, int64_t K, int64_t T,
                      void* stream) {
  q4::set_error_detail("");
  int st = validate(wq_a, scales_a, x, y_a, N_a, K, T);
  if (st == Q4LIN_OK) st = validate(wq_b, scales_b, x, y_b, N_b, K, T);
  const int64_t n_plan = 128 * ((N_a + 127) / 128 + (N_b + 127) / 128);
  // a few tokens: each weight on the one-launch warp-MMA form, one launch after the other
  const bool warp_mma = (N_a == 0 || fused_op_on_mma(N_a, K, T)) && (N_b == 0 || fused_op_on_mma(N_b, K, T));
  if (st == Q4LIN_OK && T > 0 && K > 0 && N_a + N_b > 0 && !warp_mma && !q4::tc_supported(n_plan, K, T))
    st = Q4LIN_ERR_INVALID_ARG;
  const bool work = st == Q4LIN_OK && T > 0 && N_a + N_b > 0;
  if (work) st = check_device();
  if (st == Q4LIN_OK && work) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0) {
      if (N_a > 0) st = q4::cuda_check(cudaMemsetAsync(y_a, 0, (size_t)N_a * (size_t)T * 2, s), "zero fill of y_a");
      if (st == Q4LIN_OK && N_b > 0)
        st = q4::cuda_check(cudaMemsetAsync(y_b, 0, (size_t)N_b * (size_t)T * 2, s), "zero fill of y_b");
    } else if (warp_mma) {
      if (N_a > 0) st = q4::mma_launch(q4::LinearArgs{wq_a, scales_a, x, y_a, N_a, K, T, nullptr, s}, true);
      if (st == Q4LIN_OK && N_b > 0)
        st = q4::mma_launch(q4::LinearArgs{wq_b, scales_b, x, y_b, N_b, K, T, nullptr, s}, true);
    } else if (N_a == 0 || N_b == 0) {  // one weight: the plain layer on its exact tile route
      q4::LinearArgs a = N_a > 0 ? q4::LinearArgs{wq_a, scales_a, x, y_a, N_a, K, T, nullptr, s}
                                 : q4::LinearArgs{wq_b, scales_b, x, y_b, N_b, K, T, nullptr, s};
      st = q4::tc_launch(a, Q4LIN_ROUTE_TC_SPLITK);
    } else {
      q4::LinearArgs a{wq_a, scales_a, x, y_a, N_a, K, T, nullptr, s};
      a.mode = 2;
      a.wq_b = wq_b;
      a.scales_b = scales_b;
      a.y_b = y_b;
      a.n_b = N_b;
      st = q4::tc_launch(a, Q4LIN_ROUTE_TC_SPLITK);
    }
  }
  if (st != Q4LIN_OK && q4::g_detail[0] == 0) q4::set_error_detail(q4lin_status_string(st));
  return st;
}

int q4lin_qtype_kernel_launches(int qtype, int64_t N, int64_t K, int64_t T) {
  if (qtype == Q4LIN_QTYPE_Q4G64) return q4lin_kernel_launches(N, K, T);
  if (qtype < Q4LIN_QTYPE_Q5G64 || qtype > Q4LIN_QTYPE_W8G32) return 0;
  if (validate_sizes(N, K, T) != Q4LIN_OK || N == 0 || T == 0) return 0;
  if (K == 0) return 1;  // the zero fill
  switch (qtype_route(qtype, N, K, T)) {
    case Q4LIN_ROUTE_TC_SPLITK: return q4::tc_launch_count(Q4LIN_ROUTE_TC_SPLITK, N, K, T, qtype);
    case Q4LIN_ROUTE_STREAM_MMA: return q4::mma_launch_count(N, K, T, qtype);
    default: return q4::gemv_stream_ok(N, K, T, qtype) ? 1 : 0;   // 0: refused
  }
}

size_t q4lin_qtype_workspace_bytes(int qtype, int64_t N, int64_t K, int64_t T) {
  if (qtype == Q4LIN_QTYPE_Q4G64) return q4lin_workspace_bytes(N, K, T);
  if (qtype < Q4LIN_QTYPE_Q5G64 || qtype > Q4LIN_QTYPE_W8G32) return 0;
  if (validate_sizes(N, K, T) != Q4LIN_OK || N == 0 || K == 0 || T == 0) return 0;
  if (qtype_route(qtype, N, K, T) != Q4LIN_ROUTE_STREAM_MMA) return 0;
  return round256(q4::mma_workspace_bytes(N, K, T, qtype));
}

int q4lin_linear(const uint8_t* wq, const uint16_t* scales, const uint16_t* x, uint16_t* y,
                 int64_t N, int64_t K, int64_t T, void* workspace, void* stream) {
  return run(Q4LIN_ROUTE_AUTO, wq, scales, x, y, N, K, T, workspace, stream);
}

int q4lin_linear_fp16_static(const uint8_t* wq, const uint16_t* scales, const uint16_t* x, uint16_t* y,
                             int64_t N, int64_t K, int64_t T, void* stream) {
  q4::set_error_detail("");
  int st = validate(wq, scales, x, y, N, K, T);
  if (st == Q4LIN_OK && N > 0 && T > 0 && K > 0 && !q4::tc_fp16_static_fits(N, K, T)) {
    q4::set_error_detail("fp16 route without allocation: 2*T*K + 4*T + 4*N bytes (each rounded up to 256) "
                         "exceed its 16 MiB static scratch");
    return Q4LIN_ERR_UNSUPPORTED_SHAPE;
  }
  if (st == Q4LIN_OK && N > 0 && T > 0) st = check_device();
  if (st == Q4LIN_OK && N > 0 && T > 0) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0) {
      st = q4::cuda_check(cudaMemsetAsync(y, 0, (size_t)N * (size_t)T * 2, s), "zero fill of y");
    } else {
      const q4::LinearArgs a{wq, scales, x, y, N, K, T, nullptr, s};
      st = q4::tc_fp16_static_launch(a);
    }
  }
  if (st != Q4LIN_OK && q4::g_detail[0] == 0) q4::set_error_detail(q4lin_status_string(st));
  return st;
}

int q4lin_linear_qtype(int qtype, const uint8_t* codes, const uint8_t* high, const uint16_t* scales,
                       const uint16_t* x, uint16_t* y, int64_t N, int64_t K, int64_t T, void* workspace,
                       void* stream) {
  if (qtype == Q4LIN_QTYPE_Q4G64) return run(Q4LIN_ROUTE_AUTO, codes, scales, x, y, N, K, T, workspace, stream);
  if (qtype < Q4LIN_QTYPE_Q5G64 || qtype > Q4LIN_QTYPE_W8G32) {
    q4::set_error_detail("unknown weight format");
    return Q4LIN_ERR_INVALID_ARG;
  }
  q4::set_error_detail("");
  const int st = run_qtype_impl(qtype, codes, high, scales, x, y, N, K, T, workspace, stream);
  if (st != Q4LIN_OK && q4::g_detail[0] == 0) q4::set_error_detail(q4lin_status_string(st));
  return st;
}

int q4lin_linear_route(int route, const uint8_t* wq, const uint16_t* scales, const uint16_t* x,
                       uint16_t* y, int64_t N, int64_t K, int64_t T, void* workspace, void* stream) {
  return run(route, wq, scales, x, y, N, K, T, workspace, stream);
}

const char* q4lin_status_string(int status) {
  switch (status) {
    case Q4LIN_OK: return "ok";
    case Q4LIN_ERR_INVALID_ARG: return "invalid argument (null pointer, negative or overflowing size)";
    case Q4LIN_ERR_UNSUPPORTED_SHAPE: return "unsupported shape (K not a multiple of 8, or a format and shape the decode GEMV cannot plan)";
    case Q4LIN_ERR_MISALIGNED: return "misaligned pointer (16-byte buffers, 256-byte workspace)";
    case Q4LIN_ERR_WORKSPACE: return "workspace required but NULL";
    case Q4LIN_ERR_DEVICE: return "unsupported device (needs compute capability 10.3, sm_103a)";
    case Q4LIN_ERR_CUDA: return "CUDA error";
    case Q4LIN_ERR_TIMEOUT: return "device-side bounded wait expired";
    default: return "unknown status";
  }
}

static int read_status(bool clear) {
  int worst = 0, v = 0;
  if (q4::gemv_status(&v, clear) != Q4LIN_OK) return Q4LIN_ERR_CUDA;
  if (v) worst = v;
  if (q4::tc_status(&v, clear) != Q4LIN_OK) return Q4LIN_ERR_CUDA;
  if (v) worst = v;
  if (q4::probe_status(&v, clear) != Q4LIN_OK) return Q4LIN_ERR_CUDA;
  if (v) worst = v;
  if (q4::mma_status(&v, clear) != Q4LIN_OK) return Q4LIN_ERR_CUDA;
  if (v) worst = v;
  return worst;
}

int q4lin_device_status(void) {
  if (cudaDeviceSynchronize() != cudaSuccess) return Q4LIN_ERR_CUDA;
  return read_status(false);
}

int q4lin_clear_device_status(void) {
  if (cudaDeviceSynchronize() != cudaSuccess) return Q4LIN_ERR_CUDA;
  return read_status(true) == Q4LIN_ERR_CUDA ? Q4LIN_ERR_CUDA : Q4LIN_OK;
}

int q4lin_hbm_read_probe(const void* src, size_t bytes, uint32_t* sink, int blocks, void* stream) {
  q4::set_error_detail("");
  if (src == nullptr || sink == nullptr || bytes == 0 || bytes % 16 != 0) return Q4LIN_ERR_INVALID_ARG;
  if (!aligned16(src) || (reinterpret_cast<uintptr_t>(sink) & 3u) != 0) return Q4LIN_ERR_MISALIGNED;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return Q4LIN_ERR_CUDA;
  if (blocks <= 0) blocks = 4 * sms;
  return q4::hbm_read_probe(src, bytes, sink, blocks, static_cast<cudaStream_t>(stream));
}

int q4lin_diag_wait_expiry(uint32_t limit, int* out, void* stream) {
  q4::set_error_detail("");
  if (out == nullptr || limit == 0 || limit > (1u << 20)) return Q4LIN_ERR_INVALID_ARG;
  const int st = check_device();
  if (st != Q4LIN_OK) return st;
  return q4::wait_expiry(limit, out, static_cast<cudaStream_t>(stream));
}

const char* q4lin_version(void) { return "0.2.0"; }

const char* q4lin_last_error_detail(void) { return q4::g_detail; }

}  // extern "C"
