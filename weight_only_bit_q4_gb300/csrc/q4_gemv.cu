// CUDA-core GEMV route of the Q4_G64_FP16 linear layer.
//
// The single-token case is the decode GEMV of the Q4 linear measurement
// report (q4-linear.md, route notes: T=1 uses a dedicated GEMV) and of the
// linear-benchmark contract's NCU example (linear-benchmark.md section 9,
// the q4_rowsplit_gemv_kernel instance): the weight planes are streamed once
// with 128-bit loads, decoded in registers and reduced along K with warp
// shuffles.  Up to four tokens share one decode of each weight.
//
// Decode: for a 16-byte chunk of one row (32 consecutive k, half a group),
// the low/high nibbles of each byte are isolated with two masks, and each
// nibble becomes the float (128 + q) with one byte permute (bytes
// {0, 0, q, 0x43}).  The chunk's partial sum is
//     sum_k (q_k - 8) x_k  =  sum_k (128 + q_k) x_k  -  136 * sum_k x_k,
// which costs one FMA per weight and token; the group scale multiplies the
// chunk partial once.  All arithmetic is FP32.
#include "q4_common.cuh"
#include "q4_internal.h"

namespace q4 {

namespace {

__device__ int g_gemv_status = 0;

constexpr int kRows = 4;     // rows per warp (x registers are shared by them)
constexpr int kWarps = 8;    // warps per CTA

template <int TT>
__global__ void __launch_bounds__(kWarps * 32)
q4_gemv_kernel(const uint8_t* __restrict__ wq, const uint16_t* __restrict__ scales,
               const uint16_t* __restrict__ x, uint16_t* __restrict__ y,
               int64_t N, int64_t K, int64_t t0) {
  const int lane = threadIdx.x & 31;
  const int64_t r0 = ((int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5)) * kRows;
  if (r0 >= N) return;
  const int64_t chunks = K >> 5;        // 16-byte chunks (32 weights) per row
  const int64_t row_bytes = K >> 1;
  const int64_t groups = K >> 6;

  const uint8_t* wrow[kRows];
  const uint16_t* srow[kRows];
#pragma unroll
  for (int r = 0; r < kRows; ++r) {
    const int64_t row = (r0 + r < N) ? (r0 + r) : (N - 1);   // tail rows re-read the last row
    wrow[r] = wq + row * row_bytes;
    srow[r] = scales + row * groups;
  }
  const uint16_t* xrow[TT];
#pragma unroll
  for (int t = 0; t < TT; ++t) xrow[t] = x + (t0 + t) * K;

  float acc[kRows][TT];
#pragma unroll
  for (int r = 0; r < kRows; ++r)
#pragma unroll
    for (int t = 0; t < TT; ++t) acc[r][t] = 0.f;

  for (int64_t c = lane; c < chunks; c += 32) {
    uint4 wv[kRows];
    float sc[kRows];
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      wv[r] = ld_stream_u4(wrow[r] + c * 16);
      sc[r] = fp16_bits_to_float(srow[r][c >> 1]);
    }
    float part[kRows][TT];
    float sx[TT];
#pragma unroll
    for (int t = 0; t < TT; ++t) {
      sx[t] = 0.f;
#pragma unroll
      for (int r = 0; r < kRows; ++r) part[r][t] = 0.f;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float xf[TT][8];
#pragma unroll
      for (int t = 0; t < TT; ++t) {
        const uint4 xv = ld_nc_u4(xrow[t] + c * 32 + i * 8);
        xf[t][0] = bf16lo(xv.x); xf[t][1] = bf16hi(xv.x);
        xf[t][2] = bf16lo(xv.y); xf[t][3] = bf16hi(xv.y);
        xf[t][4] = bf16lo(xv.z); xf[t][5] = bf16hi(xv.z);
        xf[t][6] = bf16lo(xv.w); xf[t][7] = bf16hi(xv.w);
#pragma unroll
        for (int j = 0; j < 8; ++j) sx[t] += xf[t][j];
      }
#pragma unroll
      for (int r = 0; r < kRows; ++r) {
        const uint32_t w = (i == 0) ? wv[r].x : (i == 1) ? wv[r].y : (i == 2) ? wv[r].z : wv[r].w;
        const uint32_t lo = w & 0x0F0F0F0Fu;          // q[2j]   in byte j
        const uint32_t hi = (w >> 4) & 0x0F0F0F0Fu;   // q[2j+1] in byte j
        float f[8];
        f[0] = f128_plus_byte<0>(lo); f[1] = f128_plus_byte<0>(hi);
        f[2] = f128_plus_byte<1>(lo); f[3] = f128_plus_byte<1>(hi);
        f[4] = f128_plus_byte<2>(lo); f[5] = f128_plus_byte<2>(hi);
        f[6] = f128_plus_byte<3>(lo); f[7] = f128_plus_byte<3>(hi);
#pragma unroll
        for (int t = 0; t < TT; ++t)
#pragma unroll
          for (int j = 0; j < 8; ++j) part[r][t] = fmaf(f[j], xf[t][j], part[r][t]);
      }
    }
#pragma unroll
    for (int r = 0; r < kRows; ++r)
#pragma unroll
      for (int t = 0; t < TT; ++t)
        acc[r][t] = fmaf(sc[r], fmaf(-136.f, sx[t], part[r][t]), acc[r][t]);
  }

#pragma unroll
  for (int r = 0; r < kRows; ++r)
#pragma unroll
    for (int t = 0; t < TT; ++t) acc[r][t] = warp_sum(acc[r][t]);

  if (lane == 0) {
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      if (r0 + r < N) {
#pragma unroll
        for (int t = 0; t < TT; ++t) y[(t0 + t) * N + r0 + r] = float_to_bf16_bits(acc[r][t]);
      }
    }
  }
}

}  // namespace

size_t gemv_workspace_bytes(int64_t, int64_t, int64_t) { return 0; }

int gemv_launch_count(int64_t, int64_t, int64_t T) { return (int)((T + 3) / 4); }

int gemv_launch(const LinearArgs& a) {
  const int64_t rows_per_cta = (int64_t)kRows * kWarps;
  const int64_t grid = (a.N + rows_per_cta - 1) / rows_per_cta;
  if (grid > 0x7fffffff) return Q4LIN_ERR_INVALID_ARG;
  for (int64_t t0 = 0; t0 < a.T; t0 += 4) {
    const int64_t tt = (a.T - t0 < 4) ? (a.T - t0) : 4;
    switch (tt) {
      case 1: q4_gemv_kernel<1><<<(unsigned)grid, kWarps * 32, 0, a.stream>>>(a.wq, a.scales, a.x, a.y, a.N, a.K, t0); break;
      case 2: q4_gemv_kernel<2><<<(unsigned)grid, kWarps * 32, 0, a.stream>>>(a.wq, a.scales, a.x, a.y, a.N, a.K, t0); break;
      case 3: q4_gemv_kernel<3><<<(unsigned)grid, kWarps * 32, 0, a.stream>>>(a.wq, a.scales, a.x, a.y, a.N, a.K, t0); break;
      default: q4_gemv_kernel<4><<<(unsigned)grid, kWarps * 32, 0, a.stream>>>(a.wq, a.scales, a.x, a.y, a.N, a.K, t0); break;
    }
    if (cuda_check(cudaGetLastError(), "gemv: kernel launch")) return Q4LIN_ERR_CUDA;
  }
  return Q4LIN_OK;
}

int gemv_status(int* value, bool clear) {
  if (cudaMemcpyFromSymbol(value, g_gemv_status, sizeof(int)) != cudaSuccess) return Q4LIN_ERR_CUDA;
  if (clear) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_gemv_status, &zero, sizeof(int)) != cudaSuccess) return Q4LIN_ERR_CUDA;
  }
  return Q4LIN_OK;
}

}  // namespace q4
