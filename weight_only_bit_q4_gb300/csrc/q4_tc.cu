// Tensor-core route of the Q4_G64_FP16 linear layer: TMA -> on-chip decode ->
// tcgen05.mma (kind::f16) with the FP32 accumulator in tensor memory.
//
// This is the tiled-MMA route of the Q4 linear measurement report
// (q4-linear.md, route notes: BF16 input, FP32-accumulating dense MMA for the
// larger token counts), re-designed for sm_103a:
//
//   * one CTA computes a 128-row x BN-token tile D[n, t] = sum_k W[n,k] X[t,k]
//     (the MMA's M is the weight row, its N the token); D lives in TMEM;
//   * warp 0 streams the packed code plane (TMA, 128-B swizzle, 4 groups per
//     stage) and the token tile of X (TMA, 128-B swizzle, one group per stage);
//   * warps 2..9 decode one 64-wide group per step: codes -> fp16
//     (q - 8) * s written into the MMA's 128-B-swizzled K-major A layout;
//   * one thread of warp 1 issues 4 x tcgen05.mma (K = 16) per group and
//     commits each stage back to the producers;
//   * warps 2..9 then read D from TMEM, round to bf16 and store Y[t, n].
//
// Operand precision: the MMA runs on fp16 operands.  A bf16 rounding of the
// dequantised weight (q - 8) * s needs ~14 significant bits and misses the
// layer's 1e-3 rms accuracy bound on a few percent of outputs, while fp16's
// 11-bit rounding stays well inside it; X is converted bf16 -> fp16, exact in
// fp16's normal range.  A kind::f16 MMA takes A and B of one type, so X is
// converted first (q4_x_to_f16 below), and its K order inside every 8-element
// block is permuted to [0,2,4,6,1,3,5,7] -- the order in which the decoder
// produces weights from one 32-bit code word with four byte-permutes.  The
// contraction is invariant under a common permutation of K.
//
// Every mbarrier wait is bounded: on expiry the kernel records
// Q4LIN_ERR_TIMEOUT in its device error word, drains what it issued (again
// bounded) and exits instead of hanging.
#include <cuda.h>

#include <mutex>

#include "q4_common.cuh"
#include "q4_internal.h"

namespace q4 {

namespace {

__device__ int g_tc_status = 0;

// ----------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase of `parity` to complete.  Returns false if the
// CTA is aborting (another thread timed out) or this wait itself timed out.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  for (uint32_t i = 0; i < kSpinLimit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
  }
  *abort_flag = 1;
  atomicExch(&g_tc_status, (int)Q4LIN_ERR_TIMEOUT);
  return false;
}

// Drain wait used after an abort: bounded, ignores the abort flag.
__device__ __forceinline__ void mbar_drain(uint32_t bar, uint32_t parity) {
  for (uint32_t i = 0; i < kSpinLimit; ++i)
    if (mbar_try_wait(bar, parity)) return;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int32_t c0,
                                            int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// D[tmem] (+)= A[smem] . B[smem]^T, both K-major, fp16 in, fp32 accumulate.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once all tcgen05 operations this thread issued so far complete.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// 16 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor (tcgen05 format): K-major operand whose rows
// are 128-byte lines in the 128-byte swizzle, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);  // start address
  d |= (uint64_t)1 << 16;                             // leading byte offset (unused here)
  d |= (uint64_t)(1024 >> 4) << 32;                   // stride byte offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;                             // descriptor version
  d |= (uint64_t)2 << 61;                             // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: D f32, A f16, B f16, both K-major, M x N.
constexpr uint32_t idesc_f16(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// One 32-bit code word (8 weights, byte j = q[2j] | q[2j+1] << 4) -> 8 fp16
// (q - 8) * s in the order [q0,q2,q4,q6,q1,q3,q5,q7]: bytes {q, 0x64} form the
// exact half 1024 + q, minus 1032 gives q - 8 exactly, times s rounds once.
__device__ __forceinline__ uint4 decode_word_f16(uint32_t w, __half2 s2) {
  const uint32_t lo = w & 0x0F0F0F0Fu;
  const uint32_t hi = (w >> 4) & 0x0F0F0F0Fu;
  const uint32_t m = 0x64646464u;
  const __half2 bias = __half2half2(__ushort_as_half(0x6408));  // 1032
  uint32_t h[4] = {__byte_perm(lo, m, 0x4140), __byte_perm(lo, m, 0x4342), __byte_perm(hi, m, 0x4140),
                   __byte_perm(hi, m, 0x4342)};
  uint4 out;
  uint32_t* o = reinterpret_cast<uint32_t*>(&out);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __half2 v = __hsub2(*reinterpret_cast<__half2*>(&h[i]), bias);
    v = __hmul2(v, s2);
    o[i] = *reinterpret_cast<uint32_t*>(&v);
  }
  return out;
}

// ----------------------------------------------------------------- X pre-pass
// bf16 [T, K] -> fp16 [T, K] with each 8-element block reordered to [0,2,4,6,1,3,5,7].
__global__ void __launch_bounds__(256) q4_x_to_f16(const uint16_t* __restrict__ x, uint16_t* __restrict__ xh,
                                                   int64_t n8) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x) {
    const uint4 v = ld_stream_u4(x + i * 8);
    const __half2 a = __floats2half2_rn(bf16lo(v.x), bf16lo(v.y));
    const __half2 b = __floats2half2_rn(bf16lo(v.z), bf16lo(v.w));
    const __half2 c = __floats2half2_rn(bf16hi(v.x), bf16hi(v.y));
    const __half2 d = __floats2half2_rn(bf16hi(v.z), bf16hi(v.w));
    uint4 o;
    o.x = *reinterpret_cast<const uint32_t*>(&a);
    o.y = *reinterpret_cast<const uint32_t*>(&b);
    o.z = *reinterpret_cast<const uint32_t*>(&c);
    o.w = *reinterpret_cast<const uint32_t*>(&d);
    *reinterpret_cast<uint4*>(xh + i * 8) = o;
  }
}

// ----------------------------------------------------------------- the tile kernel
struct TcParams {
  const uint16_t* scales;
  uint16_t* y;
  int64_t N, K, T;
  int nk;  // groups (K-steps of 64)
};

constexpr int kThreads = 320;        // warp 0 TMA, warp 1 MMA/TMEM, warps 2..9 decode + epilogue
constexpr int kDqThreads = 256;
constexpr int kTileM = 128;
constexpr int kGroupsPerW = 4;       // code stage: 128 rows x 128 bytes = 4 groups
constexpr uint32_t kABytes = kTileM * 128;   // one group of decoded A: 128 rows x 64 fp16
constexpr uint32_t kWBytes = kTileM * 128;   // one code stage

template <int BN, int S, int SW>
struct TcSmem {
  static constexpr uint32_t kB = BN * 128;  // one group of X: BN rows x 64 fp16
  static constexpr uint32_t a_off = 0;
  static constexpr uint32_t b_off = a_off + S * kABytes;
  static constexpr uint32_t w_off = b_off + S * kB;
  static constexpr uint32_t bar_off = w_off + SW * kWBytes;
  // barriers: full_a[S], full_b[S], empty[S], w_full[SW], w_empty[SW], acc_full
  static constexpr uint32_t n_bars = 3 * S + 2 * SW + 1;
  static constexpr uint32_t misc_off = bar_off + n_bars * 8;
  static constexpr uint32_t bytes = misc_off + 16;
  static constexpr uint32_t alloc = bytes + 1024;  // slack for 1024-byte alignment
  static constexpr uint32_t tmem_cols = BN < 32 ? 32 : BN;
};

template <int BN, int S, int SW>
__global__ void __launch_bounds__(kThreads, 1)
q4_tc_kernel(const __grid_constant__ CUtensorMap tm_codes, const __grid_constant__ CUtensorMap tm_x,
             const TcParams p) {
  using L = TcSmem<BN, S, SW>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + L::bar_off;
  auto full_a = [&](int s) { return bars + 8u * s; };
  auto full_b = [&](int s) { return bars + 8u * (S + s); };
  auto empty = [&](int s) { return bars + 8u * (2 * S + s); };
  auto w_full = [&](int s) { return bars + 8u * (3 * S + s); };
  auto w_empty = [&](int s) { return bars + 8u * (3 * S + SW + s); };
  const uint32_t acc_full = bars + 8u * (3 * S + 2 * SW);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::misc_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::misc_off + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t m0 = (int64_t)blockIdx.x * kTileM;
  const int64_t t0 = (int64_t)blockIdx.y * BN;
  const int nk = p.nk;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_a(s), kDqThreads / 32);
      mbar_init(full_b(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int s = 0; s < SW; ++s) {
      mbar_init(w_full(s), 1);
      mbar_init(w_empty(s), kDqThreads / 32);
    }
    mbar_init(acc_full, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_codes);
    prefetch_tmap(&tm_x);
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), L::tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_d = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------- TMA producer
    if (lane == 0) {
      int last_w = -1, last_b = -1;
      bool ok = true;
      for (int ks = 0; ks < nk && ok; ++ks) {
        if (ks % kGroupsPerW == 0) {
          const int ws = ks / kGroupsPerW, slot = ws % SW;
          ok = mbar_wait(w_empty(slot), ((ws / SW) & 1) ^ 1, abort_flag);
          if (!ok) break;
          mbar_expect_tx(w_full(slot), kWBytes);
          tma_load_2d(sbase + L::w_off + slot * kWBytes, &tm_codes, w_full(slot), ws * 128, (int32_t)m0);
          last_w = ws;
        }
        const int s = ks % S;
        ok = mbar_wait(empty(s), ((ks / S) & 1) ^ 1, abort_flag);
        if (!ok) break;
        mbar_expect_tx(full_b(s), L::kB);
        tma_load_2d(sbase + L::b_off + s * L::kB, &tm_x, full_b(s), ks * 64, (int32_t)t0);
        last_b = ks;
      }
      if (!ok) {
        // let every copy already issued land before the CTA's shared memory goes away
        for (int ws = (last_w - SW + 1 > 0 ? last_w - SW + 1 : 0); ws <= last_w; ++ws)
          mbar_drain(w_full(ws % SW), (ws / SW) & 1);
        for (int ks = (last_b - S + 1 > 0 ? last_b - S + 1 : 0); ks <= last_b; ++ks)
          mbar_drain(full_b(ks % S), (ks / S) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16(kTileM, BN);
      for (int ks = 0; ks < nk; ++ks) {
        const int s = ks % S;
        const uint32_t par = (ks / S) & 1;
        if (!mbar_wait(full_a(s), par, abort_flag)) break;
        if (!mbar_wait(full_b(s), par, abort_flag)) break;
        tc_fence_after();
        const uint32_t a_addr = sbase + L::a_off + s * kABytes;
        const uint32_t b_addr = sbase + L::b_off + s * L::kB;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_f16(tmem_d, sw128_desc(a_addr + kk * 32), sw128_desc(b_addr + kk * 32), idesc, (ks | kk) != 0);
        mma_commit(empty(s));
      }
      mma_commit(acc_full);  // also on abort: lets the teardown wait for MMAs in flight
    }
  } else {
    // ------------------------------------------------------------- decode warps
    const int dq = threadIdx.x - 64;
    const int r = dq & (kTileM - 1);   // row within the tile
    const int h = dq >> 7;             // which 32-wide half of each group
    const int64_t row = m0 + r;
    const bool row_ok = row < p.N;
    const uint16_t* srow = p.scales + (row_ok ? row : 0) * (p.K >> 6);
    uint16_t s_cur[kGroupsPerW], s_nxt[kGroupsPerW];
#pragma unroll
    for (int g = 0; g < kGroupsPerW; ++g) {
      s_cur[g] = (row_ok && g < nk) ? srow[g] : (uint16_t)0;
      s_nxt[g] = 0;
    }
    bool ok = true;
    for (int ks = 0; ks < nk && ok; ++ks) {
      const int ws = ks / kGroupsPerW, gi = ks % kGroupsPerW, slot = ws % SW;
      if (gi == 0) {
        ok = mbar_wait(w_full(slot), (ws / SW) & 1, abort_flag);
        if (!ok) break;
#pragma unroll
        for (int g = 0; g < kGroupsPerW; ++g) {
          const int gg = (ws + 1) * kGroupsPerW + g;
          s_nxt[g] = (row_ok && gg < nk) ? srow[gg] : (uint16_t)0;
        }
      }
      const int s = ks % S;
      ok = mbar_wait(empty(s), ((ks / S) & 1) ^ 1, abort_flag);
      if (!ok) break;
      uint16_t sb = s_cur[0];
#pragma unroll
      for (int g = 1; g < kGroupsPerW; ++g) sb = (gi == g) ? s_cur[g] : sb;
      const __half2 s2 = __half2half2(__ushort_as_half(sb));
      // 16 code bytes of this row: logical 16-byte chunk (2*gi + h) of the 128-byte line
      const uint32_t csrc = sbase + L::w_off + slot * kWBytes + r * 128 + ((((2 * gi + h) ^ (r & 7))) << 4);
      const uint4 cw = ld_shared_v4(csrc);
      const uint32_t adst = sbase + L::a_off + s * kABytes + r * 128;
      const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 o = decode_word_f16(words[i], s2);
        st_shared_v4(adst + ((((4 * h + i) ^ (r & 7))) << 4), o.x, o.y, o.z, o.w);
      }
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) mbar_arrive(full_a(s));
      if (gi == kGroupsPerW - 1 || ks == nk - 1) {
        if (lane == 0) mbar_arrive(w_empty(slot));
#pragma unroll
        for (int g = 0; g < kGroupsPerW; ++g) s_cur[g] = s_nxt[g];
      }
    }

    // ------------------------------------------------------------- epilogue
    if (ok && mbar_wait(acc_full, 0, abort_flag)) {
      tc_fence_after();
      const int quad = warp & 3;                 // TMEM lanes this warp may access
      const int half = (warp - 2) >> 2;          // which half of the BN columns
      const int64_t orow = m0 + quad * 32 + lane;
      const bool orow_ok = orow < p.N;
      constexpr int kCols = BN / 2;
#pragma unroll 1
      for (int c = half * kCols; c < (half + 1) * kCols; c += 16) {
        float v[16];
        tmem_ld16(tmem_d + ((uint32_t)(quad * 32) << 16) + (uint32_t)c, v);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int64_t t = t0 + c + j;
          if (orow_ok && t < p.T) p.y[t * p.N + orow] = float_to_bf16_bits(v[j]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    if (*abort_flag) mbar_drain(acc_full, 0);  // MMAs in flight must finish before TMEM is freed
    tc_fence_after();
    tmem_dealloc(tmem_d, L::tmem_cols);
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
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
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
int launch_tile(const LinearArgs& a, const uint16_t* xh) {
  using L = TcSmem<BN, S, SW>;
  static_assert(L::alloc <= 232448, "shared memory budget");
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(q4_tc_kernel<BN, S, SW>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::alloc) !=
        cudaSuccess)
      return Q4LIN_ERR_CUDA;
    attr_set[dev] = true;
  }
  CUtensorMap tm_codes, tm_x;
  if (!make_map_2d(&tm_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.wq, (uint64_t)(a.K / 2), (uint64_t)a.N,
                   (uint64_t)(a.K / 2), 128, kTileM) ||
      !make_map_2d(&tm_x, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, xh, (uint64_t)a.K, (uint64_t)a.T, (uint64_t)a.K * 2, 64,
                   BN))
    return Q4LIN_ERR_CUDA;
  TcParams p{a.scales, a.y, a.N, a.K, a.T, (int)(a.K / 64)};
  const dim3 grid((unsigned)((a.N + kTileM - 1) / kTileM), (unsigned)((a.T + BN - 1) / BN));
  q4_tc_kernel<BN, S, SW><<<grid, kThreads, L::alloc, a.stream>>>(tm_codes, tm_x, p);
  return cudaGetLastError() == cudaSuccess ? Q4LIN_OK : Q4LIN_ERR_CUDA;
}

int pick_bn(int64_t T) {
  if (T > 128) return 256;
  if (T > 64) return 128;
  if (T > 32) return 64;
  return 32;
}

}  // namespace

size_t tc_workspace_bytes(int64_t, int64_t K, int64_t T) { return (size_t)T * (size_t)K * 2; }

int tc_launch_count(int64_t, int64_t, int64_t) { return 2; }

bool tc_supported(int64_t N, int64_t K, int64_t T) {
  // TMA coordinates are 32-bit and the grid's y extent is limited.
  return N < ((int64_t)1 << 31) && K / 2 < ((int64_t)1 << 31) && T < ((int64_t)1 << 31) && (T + 31) / 32 < 65535 &&
         K / 64 < ((int64_t)1 << 30);
}

int tc_launch(const LinearArgs& a) {
  if (!tc_supported(a.N, a.K, a.T)) return Q4LIN_ERR_INVALID_ARG;
  uint16_t* xh = static_cast<uint16_t*>(a.workspace);
  const int64_t n8 = a.T * a.K / 8;
  int64_t blocks = (n8 + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  q4_x_to_f16<<<(unsigned)blocks, 256, 0, a.stream>>>(a.x, xh, n8);
  if (cudaGetLastError() != cudaSuccess) return Q4LIN_ERR_CUDA;
  switch (pick_bn(a.T)) {
    case 256: return launch_tile<256, 4, 2>(a, xh);
    case 128: return launch_tile<128, 5, 3>(a, xh);
    case 64: return launch_tile<64, 6, 4>(a, xh);
    default: return launch_tile<32, 6, 6>(a, xh);
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
