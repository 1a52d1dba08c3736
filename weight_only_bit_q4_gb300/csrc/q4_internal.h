// Host-side declarations shared by the q4lin translation units.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace q4 {

// Records why a call failed (thread-local; read by q4lin_last_error_detail)
// and returns Q4LIN_ERR_CUDA when `e` is an error, Q4LIN_OK otherwise.
int cuda_check(cudaError_t e, const char* where);
void set_error_detail(const char* what);

struct LinearArgs {
  const uint8_t* wq;
  const uint16_t* scales;
  const uint16_t* x;
  uint16_t* y;
  int64_t N, K, T;
  void* workspace;
  cudaStream_t stream;
  int fmt = 0;                   // weight format (0: Q4G64; 1: Q5G64, 2: Q6G64, 3: W8G32)
  const uint8_t* wh = nullptr;   // Q5G64 / Q6G64: the high-bit plane
  const uint16_t* r = nullptr;   // LinearAdd: bf16 residual [T, N] (tile route)
  // fused forms on the exact tile route: 1 = LinearSwiGLU (wq / scales hold 2N rows, gate then
  // up; y is [T, N]), 2 = LinearPair (a second weight wq_b / scales_b of n_b rows into y_b)
  int mode = 0;
  const uint8_t* wq_b = nullptr;
  const uint16_t* scales_b = nullptr;
  uint16_t* y_b = nullptr;
  int64_t n_b = 0;
};

// The weight planes are stored for K rounded up to a multiple of 128
// (linear-benchmark.md section 4, K_pad); columns k >= K are padding.
inline int64_t k_pad(int64_t K) { return (K + 127) / 128 * 128; }

// CUDA-core GEMV: each weight is decoded once per block of up to 4 tokens.
int gemv_launch(const LinearArgs& a);
size_t gemv_workspace_bytes(int64_t N, int64_t K, int64_t T);
int gemv_launch_count(int64_t N, int64_t K, int64_t T);
// Whether the streaming kernel (1..4 tokens, one launch) has a shared-memory plan for
// (N, K, T) on the current device.
bool gemv_stream_ok(int64_t N, int64_t K, int64_t T, int fmt = 0);
// The sibling formats (fmt 1..3) run on the streaming GEMV only.
int gemv_launch_fmt(const LinearArgs& a);

// tcgen05 tile routes: one CTA per 128-row x BN-token output tile (per K
// share when split across a cluster), group partials in tensor memory.
struct TcPlan {
  int bn;              // token tile (MMA N)
  int splitk;          // cluster size along K of the main launch
  int64_t main_tiles;  // output tiles of the main launch (all of them without a tail launch)
  int tail_splitk;     // cluster size along K of the tail launch over the other tiles (0 = none)
};
// fmt: 0 Q4G64, 1 Q5G64, 2 Q6G64 (the latter two on token tiles up to 128 wide)
TcPlan tc_plan(int route, int64_t N, int64_t K, int64_t T, int sms, int fmt = 0);
TcPlan tc_plan_current_device(int route, int64_t N, int64_t K, int64_t T, int fmt = 0);
int tc_launch(const LinearArgs& a, int route);
// The folded tile routes (Q4LIN_ROUTE_TC, Q4LIN_ROUTE_TC_SPLITK) need workspace for
// their fp16 operands and launch a prep kernel first; the exact route needs none.
size_t tc_workspace_bytes(int route, int64_t N, int64_t K, int64_t T);
int tc_launch_count(int route, int64_t N, int64_t K, int64_t T, int fmt = 0);
// The fp16 tile route with its operand scratch in a fixed device array instead of
// a caller workspace (q4lin_linear_fp16_static): whether (N, K, T) fits, and the call.
bool tc_fp16_static_fits(int64_t N, int64_t K, int64_t T);
int tc_fp16_static_launch(const LinearArgs& a);
bool tc_supported(int64_t N, int64_t K, int64_t T);

// A 2-D tensor map (inner extent, outer extent, row pitch in bytes, box); false if the
// driver's encoder is unavailable or refuses the arguments.
bool encode_map_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                   uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle);

// Streaming warp-MMA route (a few tokens; any T in passes of 32): an operand pass
// writes X as fp16 MMA fragments into the workspace, then one persistent kernel
// streams the weights.  Whether it has a shared-memory plan for (N, K, T), its
// workspace, its launch count and the call.
// fmt: 0 Q4G64, 1 Q5G64, 2 Q6G64, 3 W8G32
bool mma_supported(int64_t N, int64_t K, int64_t T, int fmt = 0);
size_t mma_workspace_bytes(int64_t N, int64_t K, int64_t T, int fmt = 0);
int mma_launch_count(int64_t N, int64_t K, int64_t T, int fmt = 0);
// fused: the one-launch form without workspace (up to 8 tokens, where the whole-K operands
// fit in shared memory), for the entry points that take no workspace
// (swiglu: LinearSwiGLU with N = F output rows over a 2F-row weight)
bool mma_fused_supported(int64_t N, int64_t K, int64_t T, int fmt = 0, bool swiglu = false);
int mma_launch(const LinearArgs& a, bool fused = false);
int mma_status(int* value, bool clear);

// Reads (and optionally clears) the device error word of one translation unit.
int gemv_status(int* value, bool clear);
int tc_status(int* value, bool clear);
int probe_status(int* value, bool clear);

// Diagnostics: HBM read probe and the bounded-wait expiry check.
int hbm_read_probe(const void* src, size_t bytes, uint32_t* sink, int blocks, cudaStream_t stream);
// Copies `bytes` (a multiple of 2; both pointers 16-byte aligned and device-accessible,
// page-locked host memory included) in stream order, chained by programmatic launch.
int stage_copy(const void* src, void* dst, size_t bytes, cudaStream_t stream);
int wait_expiry(uint32_t limit, int* out, cudaStream_t stream);

}  // namespace q4
