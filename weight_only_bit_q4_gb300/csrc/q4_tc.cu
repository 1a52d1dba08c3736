// Tensor-core route of the Q4_G64_FP16 linear layer: TMA -> on-chip decode ->
// tcgen05.mma (kind::f16, bf16 operands) with per-group accumulators in tensor
// memory and the group scales applied in FP32.
//
// This is the tiled-MMA route of the Q4 linear measurement report
// (q4-linear.md, route notes: BF16 input, FP32-accumulating dense MMA for the
// larger token counts), re-designed for sm_103a.  One CTA computes a 128-row
// x BN-token output tile (with split-K, one K share of it; the shares of a
// tile form a thread-block cluster and are summed through distributed shared
// memory):
//
//   * two TMA producer threads stream the packed code plane (128-byte swizzle,
//     4 groups per stage) and the bf16 token tile of X straight from the
//     caller's buffer (128-byte swizzle, one 64-wide group per stage);
//   * a decode warpgroup turns each group's codes into the exact bf16 values
//     q - 8, written in the MMA's 128-byte-swizzled K-major A layout;
//   * one thread issues 4 x tcgen05.mma (K = 16) per group into one of two
//     TMEM buffers, D_g[n, t] = sum_{k in g} (q[n,k] - 8) x[t,k];
//   * four accumulate warpgroups read D_g back (tcgen05.ld) and add
//     s[n,g] * D_g[n,t] to FP32 registers, then round to bf16 and store Y[t, n].
//
// Every product (q - 8) * x is exact in FP32 and the group scale multiplies
// an FP32 partial sum, so the only rounding is FP32 accumulation and the final
// bf16 store.  (Folding the scale into a 16-bit weight instead rounds
// (q - 8) * s to 11 bits -- about 2e-4 of rms(y) -- which brushes the layer's
// 1e-3 rms accuracy floor on large outputs; bf16 folding misses it outright.)
//
// Every mbarrier wait is bounded: on expiry the kernel records
// Q4LIN_ERR_TIMEOUT in its device error word, drains what it issued (again
// bounded) and exits instead of hanging.
#include <mutex>

#include "q4_internal.h"
#include "q4_sm100.cuh"

namespace q4 {

namespace {

__device__ int g_tc_status = 0;

struct TcParams {
  const uint16_t* scales;
  uint16_t* y;
  int64_t N, K, T;
  int nk;      // groups (K-steps of 64)
  int splitk;  // CTAs of a cluster sharing one output tile along K (1 = no split)
};

// Warpgroup roles (setmaxnreg works per warpgroup of 4 consecutive warps):
//   wg0: warp 0 TMA producer (X tiles), warp 1 TMEM owner + MMA issuer of the
//        even groups, warp 2 TMA producer (code plane), warp 3 MMA issuer of
//        the odd groups
//   wg1: decode, one thread per tile row, one whole code stage per iteration
//   wg2..wg5: FP32 accumulation of the scaled group partials and the
//        epilogue; warp w reads TMEM lane quadrant w % 4 and column quarter
//        (w - 8) / 4, one thread per (row, column quarter)
constexpr int kThreads = 768;
constexpr int kAccWarps = 16;
constexpr int kTileM = 128;
constexpr int kGroupsPerW = 4;               // code stage: 128 rows x 128 bytes = 4 groups
constexpr uint32_t kABytes = kTileM * 128;   // one group of A: 128 rows x 64 bf16
constexpr uint32_t kWBytes = kTileM * 128;   // one code stage
constexpr int kRegsLaunch = 80;              // 65536 / 768, rounded down to a multiple of 8
constexpr int kRegsCtl = 40;                 // wg0
constexpr int kRegsDec = 56;                 // wg1
constexpr int kRegsAcc = 96;                 // wg2..wg5
static_assert(128 * (kRegsCtl + kRegsDec) + 512 * kRegsAcc == kThreads * kRegsLaunch,
              "register split must equal the launch allocation");

template <int BN, int S, int SW>
struct TcSmem {
  static constexpr uint32_t kB = BN * 128;  // one group of X: BN rows x 64 bf16
  static constexpr uint32_t a_off = 0;
  static constexpr uint32_t b_off = a_off + S * kABytes;
  static constexpr uint32_t w_off = b_off + S * kB;
  static constexpr uint32_t bar_off = w_off + SW * kWBytes;
  // full[S], empty[S], w_full[SW], w_empty[SW], mma_done[2], tmem_free[2], done, mma_fin
  static constexpr uint32_t n_bars = 2 * S + 2 * SW + 6;
  static constexpr uint32_t misc_off = bar_off + n_bars * 8;
  static constexpr uint32_t bytes = misc_off + 16;
  static constexpr uint32_t alloc = bytes + 1024;  // slack for 1024-byte alignment
  static constexpr uint32_t tmem_cols = 2 * BN < 32 ? 32 : 2 * BN;
  // split-K partial sums of the other CTAs of the cluster reuse the pipeline buffers
  static constexpr int max_splitk = 1 + (int)(bar_off / (kTileM * BN * 4));
};

template <int BN, int S, int SW>
__global__ void __launch_bounds__(kThreads, 1)
q4_tc_kernel(const __grid_constant__ CUtensorMap tm_codes, const __grid_constant__ CUtensorMap tm_x,
             const TcParams p) {
  using L = TcSmem<BN, S, SW>;
  constexpr int kCols = BN / 4;  // accumulator columns per accumulate thread
  static_assert(kCols % 4 == 0, "BN must be a multiple of 16");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + L::bar_off;
  auto full = [&](int s) { return bars + 8u * s; };
  auto empty = [&](int s) { return bars + 8u * (S + s); };
  auto w_full = [&](int s) { return bars + 8u * (2 * S + s); };
  auto w_empty = [&](int s) { return bars + 8u * (2 * S + SW + s); };
  auto mma_done = [&](int b) { return bars + 8u * (2 * S + 2 * SW + b); };
  auto tmem_free = [&](int b) { return bars + 8u * (2 * S + 2 * SW + 2 + b); };
  const uint32_t done_bar = bars + 8u * (2 * S + 2 * SW + 4);
  const uint32_t fin_bar = bars + 8u * (2 * S + 2 * SW + 5);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::misc_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::misc_off + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int wg = warp >> 2;
  const int64_t m0 = (int64_t)blockIdx.x * kTileM;
  const int64_t t0 = (int64_t)blockIdx.y * BN;

  // This CTA's share of the K groups (the whole K without a split).
  const int splitk = p.splitk;
  uint32_t crank = 0;
  int g_begin = 0, g_end = p.nk;
  if (splitk > 1) {
    crank = cluster_ctarank();
    g_begin = (int)(((int64_t)p.nk * crank) / splitk);
    g_end = (int)(((int64_t)p.nk * (crank + 1)) / splitk);
  }
  const int ng = g_end - g_begin;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full(s), 4 + 1);   // the 4 decode warps + the X producer's expect_tx arrival
      mbar_init(empty(s), 1);
    }
    for (int s = 0; s < SW; ++s) {
      mbar_init(w_full(s), 1);
      mbar_init(w_empty(s), 4);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(mma_done(b), 1);
      mbar_init(tmem_free(b), kAccWarps);
    }
    mbar_init(done_bar, kAccWarps);
    mbar_init(fin_bar, 2);  // one final commit per MMA issuer
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_codes);
    prefetch_tmap(&tm_x);
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), L::tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (wg == 0) {
    setmaxnreg_dec<kRegsCtl>();
    // single-lane role loops; the other lanes wait at the __syncwarp below
    if (warp == 0 && lane == 0) {
      // ----------------------------------------------------------- TMA producer: token tiles of X
      int last = -1;
      bool ok = true;
      for (int i = 0; i < ng; ++i) {
        const int s = i % S;
        if (!(ok = mbar_wait(empty(s), ((i / S) & 1) ^ 1, abort_flag, &g_tc_status))) break;
        mbar_expect_tx(full(s), L::kB);
        tma_load_2d(sbase + L::b_off + s * L::kB, &tm_x, full(s), (g_begin + i) * 64, (int32_t)t0);
        last = i;
      }
      if (!ok)  // let every copy already issued land before shared memory is released
        for (int i = (last - S + 1 > 0 ? last - S + 1 : 0); i <= last; ++i) mbar_drain(full(i % S), (i / S) & 1);
    } else if (warp == 2 && lane == 0) {
      // ----------------------------------------------------------- TMA producer: code plane stages
      const int nws = (ng + kGroupsPerW - 1) / kGroupsPerW;
      int last = -1;
      bool ok = true;
      for (int ws = 0; ws < nws; ++ws) {
        const int slot = ws % SW;
        if (!(ok = mbar_wait(w_empty(slot), ((ws / SW) & 1) ^ 1, abort_flag, &g_tc_status))) break;
        mbar_expect_tx(w_full(slot), kWBytes);
        tma_load_2d(sbase + L::w_off + slot * kWBytes, &tm_codes, w_full(slot), (g_begin + ws * kGroupsPerW) * 32,
                    (int32_t)m0);
        last = ws;
      }
      if (!ok)
        for (int ws = (last - SW + 1 > 0 ? last - SW + 1 : 0); ws <= last; ++ws)
          mbar_drain(w_full(ws % SW), (ws / SW) & 1);
    } else if ((warp == 1 || warp == 3) && lane == 0) {
      // ----------------------------------------------------------- MMA issuers
      // Group i goes to TMEM buffer i & 1 and is issued by warp 1 (even i) or warp 3
      // (odd i).  A thread's first shared-memory access after a tcgen05.commit waits
      // for the MMAs that commit covers, so one thread issuing every group would
      // leave the tensor pipe idle for the completion latency of each group; with
      // two issuers the next group is already queued while the current one drains.
      constexpr uint32_t idesc = idesc_kind_f16(kTileM, BN, 1);  // bf16 x bf16 -> f32
      const uint64_t a_desc0 = sw128_desc(sbase + L::a_off), b_desc0 = sw128_desc(sbase + L::b_off);
      const int buf = warp == 1 ? 0 : 1;
      for (int i = buf; i < ng; i += 2) {
        const int s = i % S;
        if (!mbar_wait(full(s), (i / S) & 1, abort_flag, &g_tc_status)) break;
        if (i >= 2 && !mbar_wait(tmem_free(buf), ((i >> 1) - 1) & 1, abort_flag, &g_tc_status)) break;
        tc_fence_after();
        // descriptor start address advances in 16-byte units: stage offsets and the 32-byte K steps
        const uint64_t a_desc = a_desc0 + (uint64_t)((s * kABytes) >> 4);
        const uint64_t b_desc = b_desc0 + (uint64_t)((s * L::kB) >> 4);
        const uint32_t d = tmem_base + (uint32_t)(buf * BN);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) mma_f16(d, a_desc + 2 * kk, b_desc + 2 * kk, idesc, kk != 0);
        mma_commit(empty(s));
        mma_commit(mma_done(buf));
      }
      mma_commit(fin_bar);  // arrives once every MMA this thread issued has completed
    }
    __syncwarp();
    if (splitk > 1) {  // the accumulate warpgroups reduce between these two cluster barriers
      cluster_sync();
      cluster_sync();
    }
    if (warp == 1) {
      // ----------------------------------------------------------- teardown: release TMEM once the
      // accumulate warps are done with it (they arrive on `done` after their last tcgen05.ld)
      if (lane == 0) {
        mbar_drain(done_bar, 0);
        mbar_drain(fin_bar, 0);  // no MMA may still be writing TMEM when it is released
      }
      __syncwarp();
      tc_fence_after();
      tmem_dealloc(tmem_base, L::tmem_cols);
    }
  } else if (wg == 1) {
    setmaxnreg_dec<kRegsDec>();
    // ------------------------------------------------------------- decode
    // One code stage (4 groups of this thread's row) per outer iteration; each
    // group is released to the MMA as soon as it is written.
    const int r = (warp - 4) * 32 + lane;  // tile row
    const int nws = (ng + kGroupsPerW - 1) / kGroupsPerW;
    bool ok = true;
    for (int ws = 0; ws < nws && ok; ++ws) {
      const int slot = ws % SW;
      if (!(ok = warp_wait(w_full(slot), (ws / SW) & 1, abort_flag, &g_tc_status))) break;
      const uint32_t csrc = sbase + L::w_off + slot * kWBytes + r * 128;
      uint4 cw[2 * kGroupsPerW];
#pragma unroll
      for (int c = 0; c < 2 * kGroupsPerW; ++c) cw[c] = ld_shared_v4(csrc + ((c ^ (r & 7)) << 4));
      const int gcount = (ng - ws * kGroupsPerW < kGroupsPerW) ? (ng - ws * kGroupsPerW) : kGroupsPerW;
#pragma unroll
      for (int gi = 0; gi < kGroupsPerW; ++gi) {
        if (gi >= gcount) break;
        const int i = ws * kGroupsPerW + gi, s = i % S;
        if (!(ok = warp_wait(empty(s), ((i / S) & 1) ^ 1, abort_flag, &g_tc_status))) break;
        const uint32_t adst = sbase + L::a_off + s * kABytes + r * 128;
        const uint32_t words[8] = {cw[2 * gi].x,     cw[2 * gi].y,     cw[2 * gi].z,     cw[2 * gi].w,
                                   cw[2 * gi + 1].x, cw[2 * gi + 1].y, cw[2 * gi + 1].z, cw[2 * gi + 1].w};
#pragma unroll
        for (int j = 0; j < 8; ++j) st_shared_v4(adst + ((j ^ (r & 7)) << 4), decode_word_bf16(words[j]));
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) mbar_arrive(full(s));
      }
      // Release the code stage only after its bytes were consumed: a TMA (async proxy) refill
      // must not race the shared-memory reads above.
      __syncwarp();
      if (lane == 0) mbar_arrive(w_empty(slot));
    }
    __syncwarp();
    if (splitk > 1) {
      cluster_sync();
      cluster_sync();
    }
  } else {
    setmaxnreg_inc<kRegsAcc>();
    // ------------------------------------------------------------- accumulate
    const int quad = warp & 3;                  // TMEM lane quadrant
    const int cq = (warp - 8) >> 2;             // column quarter
    const int r_acc = quad * 32 + lane;         // tile row
    float2 acc[kCols / 2];
#pragma unroll
    for (int i = 0; i < kCols / 2; ++i) acc[i] = make_float2(0.f, 0.f);
    bool acc_ok = true;
    const int64_t row = m0 + r_acc;
    const bool row_ok = row < p.N;
    const uint16_t* srow = p.scales + (row_ok ? row : 0) * (p.K >> 6);
    uint16_t s_cur[kGroupsPerW], s_nxt[kGroupsPerW];
#pragma unroll
    for (int j = 0; j < kGroupsPerW; ++j) {
      s_cur[j] = 0;
      s_nxt[j] = (row_ok && j < ng) ? srow[g_begin + j] : (uint16_t)0;
    }
    const uint32_t tlane = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(cq * kCols);
    constexpr int kLd = kCols >= 16 ? 16 : kCols;    // columns per tcgen05.ld
    for (int i = 0; i < ng; ++i) {
      const int buf = i & 1, gi = i % kGroupsPerW;
      if (gi == 0) {
#pragma unroll
        for (int j = 0; j < kGroupsPerW; ++j) {
          s_cur[j] = s_nxt[j];
          const int ii = i + kGroupsPerW + j;
          s_nxt[j] = (row_ok && ii < ng) ? srow[g_begin + ii] : (uint16_t)0;
        }
      }
      uint16_t sb = s_cur[0];
#pragma unroll
      for (int j = 1; j < kGroupsPerW; ++j) sb = (gi == j) ? s_cur[j] : sb;
      const float sf = fp16_bits_to_float(sb);
      const float2 s2 = make_float2(sf, sf);
      if (!(acc_ok = warp_wait(mma_done(buf), (i >> 1) & 1, abort_flag, &g_tc_status))) break;
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < kCols; c += kLd) {
        uint32_t v[kLd];
        if constexpr (kLd == 16) tmem_ld16(tlane + buf * BN + c, v);
        else if constexpr (kLd == 8) tmem_ld8(tlane + buf * BN + c, v);
        else tmem_ld4(tlane + buf * BN + c, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < kLd; j += 2)
          acc[(c + j) / 2] =
              ffma2(make_float2(__uint_as_float(v[j]), __uint_as_float(v[j + 1])), s2, acc[(c + j) / 2]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tmem_free(buf));
    }

    // ----------------------------------------------------------- split-K reduction across the cluster
    __syncwarp();
    if (splitk > 1) {
      cluster_sync();  // every CTA of the cluster is past its main loop: rank 0's buffers are free
      if (crank > 0) {
        const uint32_t remote0 = mapa_shared(sbase, 0);
#pragma unroll
        for (int c = 0; c < kCols; c += 4) {
          const uint32_t off = (((crank - 1) * (BN / 4) + (cq * kCols + c) / 4) * kTileM + r_acc) * 16;
          st_cluster_v4(remote0 + off, acc[c / 2].x, acc[c / 2].y, acc[c / 2 + 1].x, acc[c / 2 + 1].y);
        }
      }
      cluster_sync();  // partial sums have landed in rank 0
      if (crank == 0) {
#pragma unroll 1
        for (int q = 1; q < splitk; ++q) {
#pragma unroll
          for (int c = 0; c < kCols; c += 4) {
            const uint32_t off = (((q - 1) * (BN / 4) + (cq * kCols + c) / 4) * kTileM + r_acc) * 16;
            const float4 v = ld_shared_f4(sbase + off);
            acc[c / 2] = fadd2(acc[c / 2], make_float2(v.x, v.y));
            acc[c / 2 + 1] = fadd2(acc[c / 2 + 1], make_float2(v.z, v.w));
          }
        }
      }
    }

    // ----------------------------------------------------------- epilogue: Y[t, row] = bf16(acc)
    if (crank == 0 && acc_ok && !*abort_flag && row_ok) {
#pragma unroll
      for (int j = 0; j < kCols; ++j) {
        const int64_t t = t0 + cq * kCols + j;
        const float v = (j & 1) ? acc[j / 2].y : acc[j / 2].x;
        if (t < p.T) p.y[t * p.N + row] = float_to_bf16_bits(v);
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(done_bar);
  }
}

// ----------------------------------------------------------------- host side
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

bool make_map_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                 uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, int S, int SW>
int set_kernel_attrs() {
  using L = TcSmem<BN, S, SW>;
  static bool attr_set[64] = {};
  int dev = 0;
  if (cuda_check(cudaGetDevice(&dev), "cudaGetDevice")) return Q4LIN_ERR_CUDA;
  if (dev < 64 && attr_set[dev]) return Q4LIN_OK;
  if (cuda_check(cudaFuncSetAttribute(q4_tc_kernel<BN, S, SW>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::alloc),
                 "tc: cudaFuncSetAttribute(max dynamic shared memory)"))
    return Q4LIN_ERR_CUDA;
  if (cuda_check(cudaFuncSetAttribute(q4_tc_kernel<BN, S, SW>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1),
                 "tc: cudaFuncSetAttribute(cluster size)"))
    return Q4LIN_ERR_CUDA;
  if (dev < 64) attr_set[dev] = true;
  return Q4LIN_OK;
}

// How many clusters of `size` CTAs of this kernel can be resident at once (0 on
// error).  Clusters are placed within one GPC, so this is below sms / size when
// the GPCs' SM counts are not multiples of the cluster size.
template <int BN, int S, int SW>
int resident_clusters(int size) {
  using L = TcSmem<BN, S, SW>;
  static int cache[64][9] = {};
  int dev = 0;
  if (size < 1 || size > 8 || cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev < 64 && cache[dev][size]) return cache[dev][size];
  if (set_kernel_attrs<BN, S, SW>() != Q4LIN_OK) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1, 1, (unsigned)size);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = L::alloc;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = (unsigned)size;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, q4_tc_kernel<BN, S, SW>, &cfg) != cudaSuccess || n < 0) {
    cudaGetLastError();
    n = 0;
  }
  if (dev < 64 && n > 0) cache[dev][size] = n;
  return n;
}

template <int BN, int S, int SW>
int launch_tile(const LinearArgs& a, int splitk) {
  using L = TcSmem<BN, S, SW>;
  static_assert(L::alloc <= 232448, "shared memory budget");
  if (splitk < 1 || splitk > 8 || splitk > L::max_splitk) {
    set_error_detail("tc: split-K factor out of range for this tile");
    return Q4LIN_ERR_INVALID_ARG;
  }
  if (const int rc = set_kernel_attrs<BN, S, SW>()) return rc;
  CUtensorMap tm_codes, tm_x;
  if (!make_map_2d(&tm_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.wq, (uint64_t)(a.K / 2), (uint64_t)a.N,
                   (uint64_t)(a.K / 2), 128, kTileM) ||
      !make_map_2d(&tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.x, (uint64_t)a.K, (uint64_t)a.T, (uint64_t)a.K * 2,
                   64, BN)) {
    set_error_detail("tc: cuTensorMapEncodeTiled failed (or is unavailable)");
    return Q4LIN_ERR_CUDA;
  }
  const TcParams p{a.scales, a.y, a.N, a.K, a.T, (int)(a.K / 64), splitk};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((a.N + kTileM - 1) / kTileM), (unsigned)((a.T + BN - 1) / BN), (unsigned)splitk);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = L::alloc;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = (unsigned)splitk;
  cfg.attrs = attr;
  cfg.numAttrs = splitk > 1 ? 1 : 0;
  return cuda_check(cudaLaunchKernelEx(&cfg, q4_tc_kernel<BN, S, SW>, tm_codes, tm_x, p), "tc: kernel launch");
}

int max_splitk_for(int bn) {
  switch (bn) {
    case 256: return TcSmem<256, 4, 2>::max_splitk;
    case 128: return TcSmem<128, 5, 3>::max_splitk;
    case 64: return TcSmem<64, 6, 4>::max_splitk;
    case 32: return TcSmem<32, 6, 6>::max_splitk;
    default: return TcSmem<16, 6, 6>::max_splitk;
  }
}

int resident_clusters_for(int bn, int size) {
  switch (bn) {
    case 256: return resident_clusters<256, 4, 2>(size);
    case 128: return resident_clusters<128, 5, 3>(size);
    case 64: return resident_clusters<64, 6, 4>(size);
    case 32: return resident_clusters<32, 6, 6>(size);
    default: return resident_clusters<16, 6, 6>(size);
  }
}

int sm_count() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (dev < 64 && cached[dev]) return cached[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  if (dev < 64) cached[dev] = n;
  return n;
}

}  // namespace

TcPlan tc_plan(int route, int64_t N, int64_t K, int64_t T, int sms) {
  TcPlan pl{};
  // token tile: the smallest MMA N (multiple of 16, <= 256) covering T, else 256
  if (T > 128) pl.bn = 256;
  else if (T > 64) pl.bn = 128;
  else if (T > 32) pl.bn = 64;
  else if (T > 16) pl.bn = 32;
  else pl.bn = 16;
  pl.splitk = 1;
  if (route == Q4LIN_ROUTE_TC_SPLITK) {
    // Split K across a cluster so that the CTAs fill the GPU in as few, as full
    // waves as possible.  A wave holds as many clusters as can be resident at
    // once (queried; without a device, sms / size).
    const int64_t tiles = ((N + kTileM - 1) / kTileM) * ((T + pl.bn - 1) / pl.bn);
    const int64_t nk = K / 64;
    double best = -1.0;
    const int smax = max_splitk_for(pl.bn) < 8 ? max_splitk_for(pl.bn) : 8;
    for (int s = 1; s <= smax && s <= nk; ++s) {
      int64_t per_wave = sms / s;
      if (s > 1) {
        const int q = resident_clusters_for(pl.bn, s);
        if (q > 0 && q < per_wave) per_wave = q;
      }
      if (per_wave < 1) continue;
      const int64_t waves = (tiles + per_wave - 1) / per_wave;
      // time ~ waves x (K share of one CTA + a fixed cost per CTA of about six
      // groups: launch, first loads, epilogue); prefer fewer splits on ties
      const double cost = (double)waves * ((double)nk / (double)s + 6.0);
      if (best < 0 || cost < best - 1e-9) {
        best = cost;
        pl.splitk = s;
      }
    }
  }
  return pl;
}

size_t tc_workspace_bytes(int64_t, int64_t, int64_t) { return 0; }

int tc_launch_count(int64_t, int64_t, int64_t) { return 1; }

bool tc_supported(int64_t N, int64_t K, int64_t T) {
  // TMA coordinates are 32-bit signed and the grid's y extent is limited.
  return N < ((int64_t)1 << 31) && K < ((int64_t)1 << 31) && T < ((int64_t)1 << 31) && (T + 15) / 16 < 65535;
}

int tc_launch(const LinearArgs& a, int route) {
  if (!tc_supported(a.N, a.K, a.T)) {
    set_error_detail("tc: shape beyond the tensor-core route's limits");
    return Q4LIN_ERR_INVALID_ARG;
  }
  const TcPlan pl = tc_plan(route, a.N, a.K, a.T, sm_count());
  switch (pl.bn) {
    case 256: return launch_tile<256, 4, 2>(a, pl.splitk);
    case 128: return launch_tile<128, 5, 3>(a, pl.splitk);
    case 64: return launch_tile<64, 6, 4>(a, pl.splitk);
    case 32: return launch_tile<32, 6, 6>(a, pl.splitk);
    default: return launch_tile<16, 6, 6>(a, pl.splitk);
  }
}

int tc_status(int* value, bool clear) {
  if (cudaMemcpyFromSymbol(value, g_tc_status, sizeof(int)) != cudaSuccess) return Q4LIN_ERR_CUDA;
  if (clear) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_tc_status, &zero, sizeof(int)) != cudaSuccess) return Q4LIN_ERR_CUDA;
  }
  return Q4LIN_OK;
}

}  // namespace q4
