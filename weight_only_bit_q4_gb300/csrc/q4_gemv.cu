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
#include "q4_internal.h"
#include "q4_sm100.cuh"

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

// ---------------------------------------------------------------------------
// Single-token streaming GEMV.  One persistent CTA per SM owns a contiguous
// range of rows (balanced to one row).  Thread 0 first copies x into shared
// memory (one bulk copy per CTA), then streams the rows' code bytes into a ring
// of shared-memory slots with 1-D bulk async copies (8 rows per copy), so the
// CTA's share is in flight from the start.
//
// K is cut into column groups of 32 chunks (a chunk = 16 code bytes = 32
// weights = half a scale group); warp j of a row stream owns column group j,
// so lane l always handles chunk 32 j + l: its 32 x values (and their sum)
// are read once from the shared copy of x and stay in registers for every row.
// Per 8-row slot a warp reads one conflict-free 16-byte code chunk per row,
// decodes it to (128 + q) floats with byte permutes, accumulates with packed
// FP32 FMAs, applies (partial - 136 * sum x) * s, and reduces across the warp.
// The NJ column-group partials of a row are summed in a fixed order at the end
// (deterministic), then rounded to bf16.
constexpr int kBulkThreads = 512;
constexpr int kBulkConsumers = 15;   // warps 1..15
constexpr int64_t kBulkSmemBudget = 232448 - 1024;
constexpr int kBulkRows = 8;

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// Pull global bytes into L2 (no destination, no completion): a hint that never
// changes what a later load returns -- L2 is where every SM's view meets.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

struct StreamLayout {
  uint32_t x_off, part_off, bar_off, slot_off, slot_bytes, bytes;
};

// x (bf16, K elements), partial sums [rows_cap][nj] fp32, the x barrier and the
// full/empty barriers, then the slots (128-byte aligned)
__host__ __device__ inline StreamLayout stream_layout(int64_t K, int64_t rows_cap, int nj, int slots) {
  StreamLayout L;
  L.x_off = 0;
  L.part_off = (uint32_t)(K * 2);
  L.bar_off = (uint32_t)((L.part_off + rows_cap * nj * 4 + 15) / 16 * 16);
  L.slot_off = (L.bar_off + 8 + (uint32_t)slots * 16 + 127) / 128 * 128;
  L.slot_bytes = (uint32_t)(kBulkRows * (K / 2));
  L.bytes = L.slot_off + (uint32_t)slots * L.slot_bytes;
  return L;
}

__global__ void __launch_bounds__(kBulkThreads, 1)
q4_gemv_stream_kernel(const uint8_t* __restrict__ wq, const uint16_t* __restrict__ scales,
                      const uint16_t* __restrict__ x, uint16_t* __restrict__ y, int64_t N, int64_t K,
                      int64_t rows_cap, int nj, int slots) {
  extern __shared__ __align__(128) uint8_t smem[];
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    // While the previous kernel finishes, start this CTA's rows on their way into L2
    // (codes and scales, 16-byte granules, 32 KB per prefetch).
    const int64_t p0 = (int64_t)blockIdx.x * N / gridDim.x, p1 = (int64_t)(blockIdx.x + 1) * N / gridDim.x;
    const uint8_t* cb = wq + p0 * (K / 2);
    for (int64_t off = 0, len = (p1 - p0) * (K / 2); off < len; off += 32768)
      bulk_prefetch_l2(cb + off, (uint32_t)(len - off < 32768 ? len - off : 32768));
    // scales: the 16-byte-aligned interior of this CTA's rows only (never past them)
    const uintptr_t s0 = reinterpret_cast<uintptr_t>(scales + p0 * (K / 64));
    const uintptr_t s1 = reinterpret_cast<uintptr_t>(scales + p1 * (K / 64));
    const uintptr_t a0 = (s0 + 15) & ~uintptr_t(15), a1 = s1 & ~uintptr_t(15);
    for (uintptr_t a = a0; a < a1; a += 32768)
      bulk_prefetch_l2(reinterpret_cast<const void*>(a), (uint32_t)(a1 - a < 32768 ? a1 - a : 32768));
  }
  pdl_wait_previous();  // before any global-memory read that must see the previous kernel's writes
  const StreamLayout L = stream_layout(K, rows_cap, nj, slots);
  float* part = reinterpret_cast<float*>(smem + L.part_off);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t xbar = sbase + L.bar_off;
  const uint32_t full0 = xbar + 8, empty0 = full0 + 8u * slots;
  __shared__ int abort_word;
  volatile int* abort_flag = &abort_word;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // CTA c owns the contiguous rows [c N / G, (c+1) N / G), balanced to one row, in
  // blocks of kBulkRows (the last one may be shorter).
  const int64_t r0 = (int64_t)blockIdx.x * N / gridDim.x;
  const int64_t r1 = (int64_t)(blockIdx.x + 1) * N / gridDim.x;
  const int nb = (int)((r1 - r0 + kBulkRows - 1) / kBulkRows);
  auto blk_row = [&](int b) { return r0 + (int64_t)b * kBulkRows; };
  auto blk_rows = [&](int b) { const int64_t ra = blk_row(b); return (int)((r1 - ra < kBulkRows) ? (r1 - ra) : kBulkRows); };
  const int64_t row_bytes = K / 2, groups = K / 64, nchunk = K / 32;
  const int streams = kBulkConsumers / nj;   // row streams; warp (j, stream) = 1 + stream * nj + j

  // Barrier setup and the first copies are issued before the CTA-wide barrier,
  // so the loads start while the other warps are still being set up.
  const int first = nb < slots ? nb : slots;
  if (threadIdx.x == 0) {
    mbar_init(xbar, 1);
    for (int s = 0; s < first; ++s) {
      mbar_init(full0 + 8u * s, 1);
      mbar_init(empty0 + 8u * s, nj);   // one arrival per column-group warp
    }
    abort_word = 0;
    fence_mbar_init();
    // x first (one copy per CTA: every warp reading it from global memory would hammer
    // the same few L2 lines from every SM at once), then the weight blocks
    mbar_expect_tx(xbar, (uint32_t)(K * 2));
    bulk_g2s(sbase + L.x_off, x, (uint32_t)(K * 2), xbar);
    for (int b = 0; b < first; ++b) {
      const int64_t ra = blk_row(b);
      const uint32_t bytes = (uint32_t)(blk_rows(b) * row_bytes);
      mbar_expect_tx(full0 + 8u * b, bytes);
      bulk_g2s(sbase + L.slot_off + (uint32_t)b * L.slot_bytes, wq + ra * row_bytes, bytes, full0 + 8u * b);
    }
  }
  __syncthreads();

  if (warp == 0) {
    // ---- producer (whole warp runs the loop; lane 0 issues): refill freed slots
    int b = first;
    for (; b < nb; ++b) {
      const int s = b % slots;
      if (!warp_wait(empty0 + 8u * s, ((b / slots) & 1) ^ 1, abort_flag, &g_gemv_status)) break;
      if (lane == 0) {
        const int64_t ra = blk_row(b);
        const uint32_t bytes = (uint32_t)(blk_rows(b) * row_bytes);
        mbar_expect_tx(full0 + 8u * s, bytes);
        bulk_g2s(sbase + L.slot_off + (uint32_t)s * L.slot_bytes, wq + ra * row_bytes, bytes, full0 + 8u * s);
      }
      __syncwarp();
    }
    if (b < nb && lane == 0) {  // aborted: let the copies already issued land before the CTA exits
      mbar_drain(xbar, 0);
      for (int d = (b - slots > 0 ? b - slots : 0); d < b; ++d)
        mbar_drain(full0 + 8u * (d % slots), (d / slots) & 1);
    }
    __syncwarp();
  } else if (warp - 1 < streams * nj) {
    const int j = (warp - 1) % nj, stream = (warp - 1) / nj;
    const int64_t c = (int64_t)j * 32 + lane;     // this lane's chunk
    const bool c_ok = c < nchunk;
    // this lane's 32 x values and their sum, kept in registers for every row
    float2 xv[16];
    float xsum = 0.f;
    const bool x_ok = warp_wait(xbar, 0, abort_flag, &g_gemv_status);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 v = (c_ok && x_ok) ? ld_shared_v4(sbase + L.x_off + (uint32_t)(c * 64 + q * 16))
                                     : make_uint4(0, 0, 0, 0);
      xv[4 * q + 0] = make_float2(bf16lo(v.x), bf16hi(v.x));
      xv[4 * q + 1] = make_float2(bf16lo(v.y), bf16hi(v.y));
      xv[4 * q + 2] = make_float2(bf16lo(v.z), bf16hi(v.z));
      xv[4 * q + 3] = make_float2(bf16lo(v.w), bf16hi(v.w));
    }
#pragma unroll
    for (int q = 0; q < 16; ++q) xsum += xv[q].x + xv[q].y;
    const float bias = -136.f * xsum;

    for (int b = stream; b < nb; b += streams) {
      const int s = b % slots;
      const int64_t ra = blk_row(b);
      const int nr = blk_rows(b);
      float sc[kBulkRows];
#pragma unroll
      for (int i = 0; i < kBulkRows; ++i)
        sc[i] = (c_ok && i < nr) ? fp16_bits_to_float(scales[(ra + i) * groups + (c >> 1)]) : 0.f;
      if (!warp_wait(full0 + 8u * s, (b / slots) & 1, abort_flag, &g_gemv_status)) break;
      const uint32_t slot = sbase + L.slot_off + (uint32_t)s * L.slot_bytes;
      float acc[kBulkRows];
#pragma unroll
      for (int i = 0; i < kBulkRows; ++i) {
        acc[i] = 0.f;
        if (i < nr && c_ok) {
          const uint4 cw = ld_shared_v4(slot + (uint32_t)(i * row_bytes + c * 16));
          const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
          float2 p2 = make_float2(0.f, 0.f);
#pragma unroll
          for (int wi = 0; wi < 4; ++wi) {
            const uint32_t lo = words[wi] & 0x0F0F0F0Fu, hi = (words[wi] >> 4) & 0x0F0F0F0Fu;
            p2 = ffma2(make_float2(f128_plus_byte<0>(lo), f128_plus_byte<0>(hi)), xv[4 * wi + 0], p2);
            p2 = ffma2(make_float2(f128_plus_byte<1>(lo), f128_plus_byte<1>(hi)), xv[4 * wi + 1], p2);
            p2 = ffma2(make_float2(f128_plus_byte<2>(lo), f128_plus_byte<2>(hi)), xv[4 * wi + 2], p2);
            p2 = ffma2(make_float2(f128_plus_byte<3>(lo), f128_plus_byte<3>(hi)), xv[4 * wi + 3], p2);
          }
          acc[i] = sc[i] * ((p2.x + p2.y) + bias);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8u * s);
#pragma unroll
      for (int i = 0; i < kBulkRows; ++i) {
        const float v = warp_sum(acc[i]);
        if (lane == 0 && i < nr) part[(b * kBulkRows + i) * nj + j] = v;
      }
    }
  }

  // ---- final: y[row] = bf16(sum over column groups, in order).  Every warp
  // reaches this barrier converged (all role loops are warp-uniform).
  __syncthreads();
  if (*abort_flag) return;
  for (int64_t r = threadIdx.x; r < (int64_t)nb * kBulkRows; r += kBulkThreads) {
    const int b = (int)(r / kBulkRows), i = (int)(r % kBulkRows);
    if (i >= blk_rows(b)) continue;
    float v = 0.f;
    for (int jj = 0; jj < nj; ++jj) v += part[r * nj + jj];
    y[blk_row(b) + i] = float_to_bf16_bits(v);
  }
}

}  // namespace

size_t gemv_workspace_bytes(int64_t, int64_t, int64_t) { return 0; }

bool gemv_stream_ok(int64_t N, int64_t K, int64_t T);
int gemv_launch_count(int64_t N, int64_t K, int64_t T) {
  return gemv_stream_ok(N, K, T) ? 1 : (int)((T + 3) / 4);
}

struct StreamPlan {
  int64_t grid, rows_cap;
  int nj, slots;
  uint32_t bytes;
};

static bool stream_plan(int64_t N, int64_t K, int nsm, StreamPlan* p) {
  const int64_t nchunk = K / 32;
  p->nj = (int)((nchunk + 31) / 32);
  if (p->nj > kBulkConsumers) return false;
  p->grid = (N + 3) / 4;  // at least 4 rows per CTA
  if (p->grid > nsm) p->grid = nsm;
  if (p->grid < 1) p->grid = 1;
  p->rows_cap = ((N + p->grid - 1) / p->grid + kBulkRows - 1) / kBulkRows * kBulkRows;
  const int64_t budget = kBulkSmemBudget;
  const StreamLayout L0 = stream_layout(K, p->rows_cap, p->nj, 0);
  const int64_t per = (int64_t)kBulkRows * (K / 2) + 16;
  int64_t s = (budget - L0.slot_off - 128) / per;
  if (s > 32) s = 32;
  if (s < 4) return false;
  p->slots = (int)s;
  p->bytes = stream_layout(K, p->rows_cap, p->nj, p->slots).bytes;
  return p->bytes <= budget;
}

static int device_sms() {
  static int sms[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (dev < 64 && sms[dev]) return sms[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  if (dev < 64) sms[dev] = n;
  return n;
}

static int gemv_stream_launch(const LinearArgs& a) {
  static bool attr[64] = {};
  int dev = 0;
  if (cuda_check(cudaGetDevice(&dev), "cudaGetDevice")) return Q4LIN_ERR_CUDA;
  StreamPlan pl;
  if (!stream_plan(a.N, a.K, device_sms(), &pl)) return Q4LIN_ERR_INVALID_ARG;
  if (dev >= 64 || !attr[dev]) {
    if (cuda_check(cudaFuncSetAttribute(q4_gemv_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)kBulkSmemBudget),
                   "gemv: cudaFuncSetAttribute"))
      return Q4LIN_ERR_CUDA;
    if (dev < 64) attr[dev] = true;
  }
  // programmatic dependent launch: the kernel waits for its predecessor before touching memory
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)pl.grid, 1, 1);
  cfg.blockDim = dim3(kBulkThreads, 1, 1);
  cfg.dynamicSmemBytes = pl.bytes;
  cfg.stream = a.stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cuda_check(cudaLaunchKernelEx(&cfg, q4_gemv_stream_kernel, a.wq, a.scales, a.x, a.y, a.N, a.K, pl.rows_cap,
                                       pl.nj, pl.slots),
                    "gemv: streaming kernel launch");
}

bool gemv_stream_ok(int64_t N, int64_t K, int64_t T) {
  StreamPlan pl;
  return T == 1 && stream_plan(N, K, 148, &pl);
}

int gemv_launch(const LinearArgs& a) {
  if (gemv_stream_ok(a.N, a.K, a.T)) return gemv_stream_launch(a);
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
