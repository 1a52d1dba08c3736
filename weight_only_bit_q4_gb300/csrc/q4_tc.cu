// Tensor-core route of the Q4_G64_FP16 linear layer: TMA -> on-chip decode ->
// tcgen05.mma (kind::f16, bf16 operands) with per-group accumulators in
// tensor memory and the group scales applied in FP32.
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
//   * two decode warpgroups ("teams") take alternate groups and turn each
//     group's codes into the exact bf16 values q - 8: written into a
//     tensor-memory A stage with tcgen05.st where tensor memory has room
//     (token tiles up to 128 wide), else into a 128-byte-swizzled
//     shared-memory A stage;
//   * one MMA issuer thread issues 4 x tcgen05.mma (K = 16) per group into a
//     tensor-memory accumulator buffer,
//     D_g[n, t] = sum_{k in g} (q[n,k] - 8) x[t,k];
//   * the accumulate warpgroups read D_g back (tcgen05.ld) and add
//     s[n,g] * D_g[n,t] to FP32 registers, then round to bf16 and store Y[t, n].
//
// Every product (q - 8) * x is exact in FP32 and the group scale multiplies
// an FP32 partial sum, so the only rounding is FP32 accumulation and the final
// bf16 store.
//
// The same kernel has a folded form (template flag kFold, the opt-in route
// Q4LIN_ROUTE_TC_FP16): a prep kernel writes X as fp16 (per token at a power of
// two, exact) and a power of two per weight row; the decode teams write
// fp16((q - 8) * s * 2^-rf) as the A operand, the MMAs accumulate the whole K
// share into one tensor-memory buffer, and the accumulate warps read it back once,
// undoing the powers of two.  Rounding each weight to 11 bits costs about 2e-4 of
// rms(y) per output, which brushes the layer's 1e-3 rms accuracy floor (measured:
// one element in 3.5 million at 1.03x the bound), so the folded form is never the
// library's choice; bf16 folding would miss the floor outright.
//
// Two more template parameters reuse the same pipeline.  FMT = 1 / 2 (Q5G64 /
// Q6G64, exact form, token tiles up to 128 wide) adds a second TMA stream per code
// stage for the high-bit plane; the decode teams move each weight's high bits to
// bit 4 of its nibble before taking the exact bf16 q - 16 / q - 32.  The epilogue
// optionally adds a bf16 residual R[t, n] to the FP32 sum before the store
// (LinearAdd).
//
// Synchronisation, shaped by what the hardware charges for it:
//   * while the tensor core streams its shared-memory operands an mbarrier
//     wait costs a few hundred cycles even when the phase has long completed,
//     and a thread with tcgen05.mma operations in flight pays that on every
//     shared-memory access; so the issuer never touches shared memory.  The
//     decode team of group i (after writing its A stage and seeing its X tile
//     land) and every accumulate warp (after reading back the accumulator
//     buffer that group i will overwrite) arrive on a hardware named barrier,
//     on which the issuer waits;
//   * tcgen05.mma is issued by that one thread only (concurrent issue from two
//     threads corrupted results);
//   * one tcgen05.commit per group, into a ring of mbarriers that everything
//     downstream waits on: the X producer and the decode team (the group's X
//     and A stages are free again) and the accumulate warps (D_i is ready);
//   * a parity wait cannot tell phase k from phase k + 2, so no waiter may fall
//     two phases behind: the rings cover every buffer ring, and the A and X
//     rings have even depths so that each slot belongs to one decode team;
//   * named barriers cannot time out, so every role keeps arriving on them for
//     every group even after an abort: the issuer always runs to completion.
//
// Every mbarrier wait is bounded: on expiry the kernel records
// Q4LIN_ERR_TIMEOUT in its device error word, skips the remaining work
// (still arriving where others wait), drains what it issued (again bounded)
// and exits instead of hanging.
#include <mutex>

#include "q4_internal.h"
#include "q4_sm100.cuh"

namespace q4 {

namespace {

__device__ int g_tc_status = 0;

struct TcParams {
  const uint16_t* scales;
  uint16_t* y;
  const int* xe;  // folded form: per token, X was stored as fp16 x * 2^-xe[t]
  const int* rf;  // folded form: per weight row, the scales enter as s * 2^-rf[n]
  const uint16_t* r;  // LinearAdd: bf16 residual [T, N] added before the bf16 store (may be y itself)
  int64_t N, Kp, T;   // Kp: the planes' stored width, K rounded up to 128
  int nk;      // groups (K-steps of 64) holding columns < K
  int splitk;  // CTAs of a cluster sharing one output tile along K (1 = no split)
  uint32_t tile_base;  // first output tile of this launch (tiles are numbered m-major)
  uint32_t tiles_m;    // row tiles, ceil(N / 128)
  // Fused forms of the exact tile route (FMT = 0):
  //   mode 1, LinearSwiGLU: the weight has 2F rows (gate rows [0, F), up rows [F, 2F)) and a
  //     tile stacks gate rows [f0, f0 + 64) over up rows [F + f0, F + f0 + 64); y is [T, F],
  //     y = silu(gate) * up.  N holds F, tiles_m = ceil(F / 64).
  //   mode 2, LinearPair: row tiles [0, tiles_a) are W_a's (codes tm_codes, scales, y, N),
  //     the rest W_b's (codes in the high-plane map slot, scales_b, y_b, n_b).
  int mode;
  uint32_t tiles_a;
  const uint16_t* scales_b;
  uint16_t* y_b;
  int64_t n_b;
};

// Named barrier of the accumulate warps for the SwiGLU exchange (after the issue ring and kAccBar).
constexpr uint32_t kSwiBar = 10;

constexpr int kTileM = 128;
constexpr int kGroupsPerW = 4;              // code stage: 128 rows x 128 bytes = 4 groups
constexpr uint32_t kWBytes = kTileM * 128;  // one code stage
constexpr uint32_t kABytes = kTileM * 128;  // one shared-memory A stage: 128 rows x 64 bf16
constexpr int kRing = 8;                    // depth of the per-group MMA-done / issue rings
constexpr uint32_t kIssueBar0 = 1;          // named barriers kIssueBar0 .. kIssueBar0 + kRing - 1
constexpr uint32_t kAccBar = kIssueBar0 + kRing;  // folded form: the accumulate warps' start barrier

// Per token-tile width: X stages, A stages, accumulator buffers, accumulate
// warpgroups, code stages and where A lives.  Tensor memory holds NB * BN
// accumulator columns, followed (A in tensor memory) by SA * 32 A columns.
template <int BN> struct TcCfg;
template <> struct TcCfg<256> { static constexpr int SX = 4, SA = 4, NB = 2, NACC = 4, SW = 2; static constexpr bool kATmem = false; };
template <> struct TcCfg<128> { static constexpr int SX = 8, SA = 8, NB = 2, NACC = 4, SW = 4; static constexpr bool kATmem = true; };
template <> struct TcCfg<64> { static constexpr int SX = 8, SA = 8, NB = 4, NACC = 1, SW = 4; static constexpr bool kATmem = true; };
template <> struct TcCfg<32> { static constexpr int SX = 8, SA = 8, NB = 8, NACC = 1, SW = 4; static constexpr bool kATmem = true; };
template <> struct TcCfg<16> { static constexpr int SX = 8, SA = 8, NB = 8, NACC = 1, SW = 4; static constexpr bool kATmem = true; };

// Warpgroup roles (setmaxnreg works per warpgroup of 4 consecutive warps):
//   wg0: warp 0 TMA producer (X tiles), warp 1 TMA producer (code stages) and
//        tensor-memory owner, warp 3 MMA issuer (warp 2 idles)
//   wg1 / wg2: decode teams of the even / odd groups, one thread per tile row
//   wg3..: FP32 accumulation of the scaled group partials and the epilogue;
//        warp w reads TMEM lane quadrant w % 4 and column chunk (w - 12) / 4
// FMT: 0 = Q4G64; 1 = Q5G64 and 2 = Q6G64 add a high-bit plane of 1 or 2 bits per
// weight, staged beside the codes (exact form only, token tiles up to 128 wide).
template <int BN, bool kFold, int FMT = 0>
struct TcSmem {
  using C = TcCfg<BN>;
  static constexpr int kHB = (FMT == 1 || FMT == 2) ? FMT : 0;  // high bits per weight (Q5 / Q6)
  static constexpr bool kW8 = FMT == 3;  // W8G32: one code byte per weight, two 32-wide scale groups per 64-wide group
  static_assert(FMT == 0 || (!kFold && (BN <= 128 || kHB > 0)), "sibling formats: exact form, BN <= 128 (Q5 / Q6: 256)");
  static_assert(!kW8 || BN <= 128, "W8G32: token tiles up to 128 wide");
  // W8G32 at 128-token tiles: two accumulators per group in flight fill tensor memory, so A
  // is staged in shared memory (four X, A and code stages fit beside it)
  static constexpr bool kW8Wide = kW8 && BN == 128;
  // The folded form keeps one accumulator for the whole K share, which leaves tensor
  // memory room for A at BN = 256 too; the shared memory freed there holds six X
  // stages instead of four (measured 8-12 % faster at T = 1024).
  static constexpr bool kWide = kFold && BN == 256;
  // W8G32 keeps two accumulators per group in flight (one per 32-wide scale group)
  // Q5 / Q6 at 256-token tiles: the high-bit stages take the room of two A stages
  static constexpr int SX = kWide ? 6 : kW8Wide ? 4 : C::SX,
                       SA = kW8Wide ? 4 : (kHB > 0 && BN == 256) ? 2 : C::SA, NB = kFold ? 1 : kW8 ? 2 : C::NB,
                       NACC = C::NACC, SW = kW8Wide ? 2 : C::SW;
  static constexpr int kAccPerGroup = kW8 ? 2 : 1;
  static constexpr uint32_t kCB = kW8 ? 2 * kWBytes : kWBytes;  // one code stage (4 groups)
  static constexpr bool kATmem = kWide ? true : kW8Wide ? false : C::kATmem;
  static_assert(SA % 2 == 0 && SX % 2 == 0, "the A and X ring depths must be even (one decode team per slot)");
  static_assert(kRing % 2 == 0 && kRing >= SX && kRing >= SA && kRing >= NB,
                "the barrier rings must cover every buffer ring (no waiter two phases behind)");
  static_assert(kAccPerGroup * NB * BN + (kATmem ? SA * 32 : 0) <= 512, "tensor memory budget");
  static constexpr int threads = 128 * (3 + NACC);
  // decode team + issuer, and (exact form) the accumulate warps handing back a buffer
  static constexpr uint32_t issue_threads = 128 + (kFold ? 0 : 128 * NACC) + 32;
  static constexpr uint32_t kB = BN * 128;  // one group of X: BN rows x 64 bf16
  static constexpr uint32_t x_off = 0;
  static constexpr uint32_t a_off = x_off + SX * kB;  // shared-memory A stages (A not in tensor memory)
  static constexpr uint32_t c_off = a_off + (kATmem ? 0 : SA * kABytes);
  static constexpr uint32_t kHBytes = kTileM * kGroupsPerW * 8 * kHB;  // one high-bit stage
  static constexpr uint32_t h_off = c_off + SW * kCB;
  static constexpr uint32_t bar_off = h_off + SW * kHBytes;
  // x_full[SX], c_full[SW], c_empty[SW], mma_done[kRing], done, fin
  static constexpr uint32_t n_bars = SX + 2 * SW + kRing + 2;
  static constexpr uint32_t misc_off = bar_off + n_bars * 8;
  static constexpr uint32_t bytes = misc_off + 16;
  static constexpr uint32_t alloc = bytes + 1024;  // slack for 1024-byte alignment
  static constexpr uint32_t a_col = kAccPerGroup * NB * BN;  // first A column in tensor memory
  static constexpr uint32_t tmem_cols = 512;
  // split-K partial sums of the other CTAs of the cluster reuse the pipeline buffers: that
  // many partial tiles fit at once, and larger clusters reduce in rounds of that many
  static constexpr int kRedSlots = (int)(bar_off / (kTileM * BN * 4));
  static_assert(kRedSlots >= 1, "one partial tile must fit in the pipeline buffers");
  static constexpr int max_splitk = 8;  // portable cluster size
};

// Registers per thread after the split (four accumulate warpgroups only; with
// one, the launch allocation of 128 per thread covers every role).  The split
// sums to at most the launch allocation: 896 threads x 72.  Chosen so that no role
// spills (ptxas -v): with shared-memory A stages the decode teams need 48 and the
// producers and issuer more than 40 (a decode split of 40 spilled in the decode
// loop and cost about 10 % at T = 1024); with A in tensor memory the decode teams
// need 72.
template <bool kATmem> struct TcRegs;
template <> struct TcRegs<true> { static constexpr int ctl = 32, dec = 72, acc = 80; };
template <> struct TcRegs<false> { static constexpr int ctl = 56, dec = 48, acc = 88; };
static_assert(128 * TcRegs<true>::ctl + 256 * TcRegs<true>::dec + 512 * TcRegs<true>::acc <= 896 * 72, "register split");
static_assert(128 * TcRegs<false>::ctl + 256 * TcRegs<false>::dec + 512 * TcRegs<false>::acc <= 896 * 72, "register split");

// W8G32: the four signed codes of one code word (weights k .. k + 3, byte j = weight
// k + j) as two exact bf16 pairs, even k in the low half: |code| <= 128 fits bf16's
// 8-bit significand.
__device__ __forceinline__ void w8_word_bf16(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const float f0 = (float)(int8_t)(w & 0xFFu), f1 = (float)(int8_t)((w >> 8) & 0xFFu);
  const float f2 = (float)(int8_t)((w >> 16) & 0xFFu), f3 = (float)(int8_t)(w >> 24);
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(lo) : "f"(f1), "f"(f0));  // upper half: the first operand
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(hi) : "f"(f3), "f"(f2));
}

template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t* v) {
  if constexpr (N == 16) tmem_ld16(taddr, *reinterpret_cast<uint32_t(*)[16]>(v));
  else if constexpr (N == 8) tmem_ld8(taddr, *reinterpret_cast<uint32_t(*)[8]>(v));
  else tmem_ld4(taddr, *reinterpret_cast<uint32_t(*)[4]>(v));
}

template <int BN, bool kFold, int FMT, int MODE = 0>
__global__ void __launch_bounds__(TcSmem<BN, kFold, FMT>::threads, 1)
q4_tc_kernel(const __grid_constant__ CUtensorMap tm_codes, const __grid_constant__ CUtensorMap tm_x,
             const __grid_constant__ CUtensorMap tm_high, const TcParams p) {
  using L = TcSmem<BN, kFold, FMT>;
  constexpr int kHB = L::kHB;
  constexpr bool kW8 = L::kW8;
  using R = TcRegs<L::kATmem>;
  constexpr int SX = L::SX, SA = L::SA, NB = L::NB, NACC = L::NACC, SW = L::SW;
  constexpr int kAccWarps = 4 * NACC;
  constexpr int kCols = BN / NACC;  // accumulator columns per accumulate thread
  static_assert(kCols % 4 == 0, "column chunk must be a multiple of 4");

  // Programmatic dependent launch: the next kernel in the stream may begin launching now;
  // this CTA's setup below overlaps the previous kernel's tail, and every global-memory
  // access waits for that kernel (pdl_wait_previous after the setup barrier).
  pdl_launch_dependents();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + L::bar_off;
  // Group i uses X slot i % SX, A slot i % SA, accumulator buffer i % NB, named
  // barrier kIssueBar0 + i % kRing and mma_done entry i % kRing (one commit per
  // group: its X and A slots are free again and its accumulator buffer holds D_i).
  auto x_full = [&](int s) { return bars + 8u * s; };
  auto c_full = [&](int s) { return bars + 8u * (SX + s); };
  auto c_empty = [&](int s) { return bars + 8u * (SX + SW + s); };
  auto mma_done = [&](int i) { return bars + 8u * (SX + 2 * SW + i % kRing); };
  auto ring_par = [](int i) { return (uint32_t)((i / kRing) & 1); };
  auto issue_bar = [](int i) { return kIssueBar0 + (uint32_t)(i % kRing); };
  const uint32_t done_bar = bars + 8u * (SX + 2 * SW + kRing);
  const uint32_t fin_bar = done_bar + 8u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::misc_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::misc_off + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int wg = warp >> 2;
  // Output tile of this CTA (cluster): tiles are numbered m-major, so consecutive
  // CTAs share a token tile and its X stays in L2.  32-bit arithmetic (the host
  // keeps tile numbers below 2^31): a 64-bit division would be a subroutine call.
  const uint32_t tile = p.tile_base + blockIdx.x;
  const uint32_t mt = tile % p.tiles_m;
  const int64_t t0 = (int64_t)(tile / p.tiles_m) * BN;
  // the weight this tile reads: first row (the gate rows' first row for SwiGLU), row count,
  // and for LinearPair which of the two weights
  // (MODE, a template parameter so that the plain layer's code is untouched by the fused forms)
  const bool wsel_b = MODE == 2 && mt >= p.tiles_a;
  const int64_t m0 = MODE == 1 ? (int64_t)mt * 64 : (int64_t)(wsel_b ? mt - p.tiles_a : mt) * kTileM;
  const int64_t n_rows = wsel_b ? p.n_b : p.N;   // rows of this tile's output (SwiGLU: F)

  // This CTA's share of the K groups (the whole K without a split).
  const int splitk = p.splitk;
  uint32_t crank = 0;
  int g_begin = 0, g_end = p.nk;
  if (splitk > 1) {
    crank = cluster_ctarank();
    // Q5's high plane holds 8 bytes per group: shares start on even groups so every
    // TMA x coordinate into it is a multiple of 16 bytes
    auto split_at = [&](uint32_t rk) {
      if (rk >= (uint32_t)splitk) return p.nk;
      const int g = (int)(((int64_t)p.nk * rk) / splitk);
      return kHB == 1 ? (g & ~1) : g;
    };
    g_begin = split_at(crank);
    g_end = split_at(crank + 1);
  }
  const int ng = g_end - g_begin;
  const int nws = (ng + kGroupsPerW - 1) / kGroupsPerW;
  const int red_rounds = splitk > 1 ? (splitk - 1 + L::kRedSlots - 1) / L::kRedSlots : 0;  // split-K reduction rounds

  if (threadIdx.x == 0) {
    for (int s = 0; s < SX; ++s) mbar_init(x_full(s), 1);
    for (int s = 0; s < SW; ++s) {
      mbar_init(c_full(s), 1);
      mbar_init(c_empty(s), 8);  // every code stage is read by both teams' 4 warps
    }
    for (int r = 0; r < kRing; ++r) mbar_init(mma_done(r), 1);
    mbar_init(done_bar, kAccWarps);
    mbar_init(fin_bar, 1);  // the issuer's final commit
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_codes);
    prefetch_tmap(&tm_x);
    if constexpr (kHB > 0 || MODE == 2) prefetch_tmap(&tm_high);
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), L::tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait_previous();  // before the first TMA load, scale load or output store

  if (wg == 0) {
    if constexpr (NACC == 4) setmaxnreg_dec<R::ctl>();
    // the producers run on one lane (the others wait at the __syncwarp below);
    // the issuer loop is warp-uniform
    if (warp == 0 && lane == 0) {
      // ----------------------------------------------------------- TMA producer: token tiles of X
      int last = -1;
      bool ok = true;
      for (int i = 0; i < ng; ++i) {
        const int s = i % SX;
        if (i >= SX && !(ok = mbar_wait(mma_done(i - SX), ring_par(i - SX), abort_flag, &g_tc_status))) break;
        mbar_expect_tx(x_full(s), L::kB);
        tma_load_2d(sbase + L::x_off + s * L::kB, &tm_x, x_full(s), (g_begin + i) * 64, (int32_t)t0);
        last = i;
      }
      if (!ok)  // let every copy already issued land before shared memory is released
        for (int i = (last - SX + 1 > 0 ? last - SX + 1 : 0); i <= last; ++i) mbar_drain(x_full(i % SX), (i / SX) & 1);
    } else if (warp == 1 && lane == 0) {
      // ----------------------------------------------------------- TMA producer: code plane stages
      int last = -1;
      bool ok = true;
      for (int ws = 0; ws < nws; ++ws) {
        const int slot = ws % SW;
        if (!(ok = mbar_wait(c_empty(slot), ((ws / SW) & 1) ^ 1, abort_flag, &g_tc_status))) break;
        mbar_expect_tx(c_full(slot), L::kCB + L::kHBytes);
        if constexpr (kW8) {  // 64 code bytes per group and row: two 128-byte boxes of two groups each
          tma_load_2d(sbase + L::c_off + slot * L::kCB, &tm_codes, c_full(slot), (g_begin + ws * kGroupsPerW) * 64,
                      (int32_t)m0);
          tma_load_2d(sbase + L::c_off + slot * L::kCB + kWBytes, &tm_codes, c_full(slot),
                      (g_begin + ws * kGroupsPerW + 2) * 64, (int32_t)m0);
        } else if constexpr (MODE == 1) {  // SwiGLU: gate rows into tile rows 0..63, up rows into 64..127 (64-row boxes)
          tma_load_2d(sbase + L::c_off + slot * kWBytes, &tm_codes, c_full(slot), (g_begin + ws * kGroupsPerW) * 32,
                      (int32_t)m0);
          tma_load_2d(sbase + L::c_off + slot * kWBytes + kWBytes / 2, &tm_codes, c_full(slot),
                      (g_begin + ws * kGroupsPerW) * 32, (int32_t)(p.N + m0));
        } else {
          if (MODE == 2 && wsel_b)
            tma_load_2d(sbase + L::c_off + slot * kWBytes, &tm_high, c_full(slot), (g_begin + ws * kGroupsPerW) * 32,
                        (int32_t)m0);
          else
            tma_load_2d(sbase + L::c_off + slot * kWBytes, &tm_codes, c_full(slot), (g_begin + ws * kGroupsPerW) * 32,
                        (int32_t)m0);
        }
        if constexpr (kHB > 0)  // the stage's high bits: 8 * kHB bytes per group and row
          tma_load_2d(sbase + L::h_off + slot * L::kHBytes, &tm_high, c_full(slot),
                      (g_begin + ws * kGroupsPerW) * 8 * kHB, (int32_t)m0);
        last = ws;
      }
      if (!ok)
        for (int ws = (last - SW + 1 > 0 ? last - SW + 1 : 0); ws <= last; ++ws)
          mbar_drain(c_full(ws % SW), (ws / SW) & 1);
    } else if (warp == 3) {
      // ----------------------------------------------------------- MMA issuer (no shared-memory access)
      // exact form bf16 x bf16 -> f32; folded form fp16 x fp16 -> f32
      constexpr uint32_t idesc = idesc_kind_f16(kTileM, BN, kFold ? 0u : 1u);
      // descriptors as 32-bit halves: the start address (low half) advances in 16-byte
      // units by the stage offset and by 2 per 32-byte K step
      const uint64_t bd = sw128_desc(sbase + L::x_off), ad = sw128_desc(sbase + L::a_off);
      const uint32_t b_lo0 = (uint32_t)bd, b_hi = (uint32_t)(bd >> 32);
      const uint32_t a_lo0 = (uint32_t)ad, a_hi = (uint32_t)(ad >> 32);
      for (int i = 0; i < ng; ++i) {
        named_bar_sync(issue_bar(i), L::issue_threads);  // A stage written, X landed, buffer free
        tc_fence_after();
        if (lane == 0) {
          const int s = i % SX, sa = i % SA, b = i % NB;
          const uint32_t b_lo = b_lo0 + ((uint32_t)(s * L::kB) >> 4);
          const uint32_t d = tmem_base + (uint32_t)(b * L::kAccPerGroup * BN);
          // exact form: each group starts its own buffer; folded form: one sum over the share
          const bool first = kFold ? i == 0 : true;
          if constexpr (kW8 && L::kATmem) {
            // W8G32: K 0..31 of the group into buffer d, K 32..63 into d + BN (one per scale group)
            const uint32_t a = tmem_base + L::a_col + (uint32_t)(sa * 32);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_f16_ts32(d + (uint32_t)((kk >> 1) * BN), a + 8 * kk, b_lo + 2 * kk, b_hi, idesc, (kk & 1) != 0);
          } else if constexpr (kW8) {
            const uint32_t a_lo = a_lo0 + ((uint32_t)(sa * kABytes) >> 4);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_f16_ss(d + (uint32_t)((kk >> 1) * BN), a_lo + 2 * kk, a_hi, b_lo + 2 * kk, b_hi, idesc, (kk & 1) != 0);
          } else if constexpr (L::kATmem) {
            const uint32_t a = tmem_base + L::a_col + (uint32_t)(sa * 32);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_f16_ts32(d, a + 8 * kk, b_lo + 2 * kk, b_hi, idesc, !(first && kk == 0));
          } else {
            const uint32_t a_lo = a_lo0 + ((uint32_t)(sa * kABytes) >> 4);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_f16_ss(d, a_lo + 2 * kk, a_hi, b_lo + 2 * kk, b_hi, idesc, !(first && kk == 0));
          }
          mma_commit(mma_done(i));
        }
        __syncwarp();
      }
      if (lane == 0) mma_commit(fin_bar);  // arrives once every MMA issued here has completed
    }
    __syncwarp();
    for (int rr = 0; rr < red_rounds; ++rr) {  // the accumulate warpgroups reduce between these cluster barriers
      cluster_sync();
      cluster_sync();
    }
    if (warp == 1) {
      // ----------------------------------------------------------- teardown: release tensor memory once
      // the accumulate warps are done with it and no MMA is still running
      if (lane == 0) {
        mbar_drain(done_bar, 0);
        mbar_drain(fin_bar, 0);
      }
      __syncwarp();
      tc_fence_after();
      tmem_dealloc(tmem_base, L::tmem_cols);
    }
  } else if (wg == 1 || wg == 2) {
    if constexpr (NACC == 4) setmaxnreg_dec<R::dec>();
    // ------------------------------------------------------------- decode (team = wg - 1)
    // Team t decodes groups 4 ws + t and 4 ws + t + 2 of every code stage ws,
    // one tile row per thread, into the A stage of the group's ring slot.
    const int team = wg - 1;
    const int q = warp & 3;
    const int r = q * 32 + lane;  // tile row = tensor-memory lane
    const uint32_t a_lane = tmem_base + ((uint32_t)(q * 32) << 16) + L::a_col;
    // folded form: this row's scales, and the power of two they are taken at (rows past N:
    // scale 0, and their codes read as zeros)
    const int64_t drow = m0 + r;
    const bool drow_ok = drow < p.N;
    const uint16_t* dsrow = p.scales + (drow_ok ? drow : 0) * (p.Kp >> 6) + g_begin;
    float smul = 0.f;
    if constexpr (kFold) smul = drow_ok ? exp2i(-__ldg(p.rf + drow)) : 0.f;
    bool ok = true;
    for (int ws = 0; ws < nws; ++ws) {
      const int slot = ws % SW;
      uint32_t sbits[2] = {0u, 0u};
      if constexpr (kFold) {  // issued before the wait, used after it
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int i = ws * kGroupsPerW + team + 2 * h;
          if (drow_ok && i < ng) sbits[h] = __ldg(dsrow + i);
        }
      }
      ok = ok && warp_wait(c_full(slot), (ws / SW) & 1, abort_flag, &g_tc_status);
      const uint32_t csrc = sbase + L::c_off + slot * L::kCB + r * 128;
      uint4 cw[4] = {};
      // W8G32: group gl of the stage is 64 code bytes of the row, 16-byte chunks
      // 4 (gl % 2) .. + 3 of the 128-byte box gl / 2, read where the group is decoded (the
      // stage is released after the team's last group)
      auto w8_chunk = [&](int gl, int j) -> uint4 {
        return ld_shared_v4(csrc + (uint32_t)((gl >> 1) * kWBytes) + ((uint32_t)((4 * (gl & 1) + j) ^ (r & 7)) << 4));
      };
      if constexpr (!kW8) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int c0 = 2 * (team + 2 * h);  // first 16-byte chunk of group team + 2h
          cw[2 * h] = ok ? ld_shared_v4(csrc + ((c0 ^ (r & 7)) << 4)) : make_uint4(0, 0, 0, 0);
          cw[2 * h + 1] = ok ? ld_shared_v4(csrc + (((c0 + 1) ^ (r & 7)) << 4)) : make_uint4(0, 0, 0, 0);
        }
      }
      // Q5 / Q6: the two groups' high bits (8 * kHB bytes per group in a row of the
      // unswizzled high-bit stage)
      uint4 hw[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
      if constexpr (kHB > 0) {
        const uint32_t hsrc = sbase + L::h_off + slot * L::kHBytes + r * (32 * kHB);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t ga = hsrc + (uint32_t)((team + 2 * h) * 8 * kHB);
          if (!ok) continue;
          if constexpr (kHB == 1) {
            const uint2 v = ld_shared_u64(ga);
            hw[h] = make_uint4(v.x, v.y, 0, 0);
          } else {
            hw[h] = ld_shared_v4(ga);
          }
        }
      }
      // The code slot is free once both teams have their chunks in registers (a TMA
      // refill must not race the reads above); W8G32 reads its chunks below.
      if constexpr (!kW8) {
        __syncwarp();
        if (lane == 0) mbar_arrive(c_empty(slot));
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int i = ws * kGroupsPerW + team + 2 * h;
        if (i >= ng) break;
        const int sa = i % SA;
        // the slot's previous group (i - SA, same team) must have been consumed by its MMA
        if (i >= SA) ok = ok && warp_wait(mma_done(i - SA), ring_par(i - SA), abort_flag, &g_tc_status);
        if (ok) {
          tc_fence_after();
          const uint32_t words[8] = {cw[2 * h].x,     cw[2 * h].y,     cw[2 * h].z,     cw[2 * h].w,
                                     cw[2 * h + 1].x, cw[2 * h + 1].y, cw[2 * h + 1].z, cw[2 * h + 1].w};
          // high bits of code word j of this group, in weight order
          const uint32_t hv[4] = {hw[h].x, hw[h].y, hw[h].z, hw[h].w};
          auto high_of = [&](int j) -> uint32_t {
            return kHB == 1 ? (hv[j >> 2] >> (8 * (j & 3))) & 0xFFu : (hv[j >> 1] >> (16 * (j & 1))) & 0xFFFFu;
          };
          auto decode = [&](int j, uint32_t sc2) -> uint4 {
            if constexpr (kFold) return decode_word_f16s(words[j], sc2);
            else if constexpr (kHB > 0) return decode_word_bf16_hi<kHB>(words[j], high_of(j));
            else return decode_word_bf16(words[j]);
          };
          uint32_t s2 = 0u;  // folded form: fp16(s * 2^-rf) twice
          if constexpr (kFold) {
            const uint32_t hb =
                __half_as_ushort(__float2half_rn(fp16_bits_to_float((uint16_t)sbits[h]) * smul));
            s2 = hb | (hb << 16);
          }
          if constexpr (L::kATmem) {
            uint32_t v[32];  // column j = (k = 2j, k = 2j + 1) of the group
            if constexpr (kW8) {
#pragma unroll
              for (int j = 0; j < 4; ++j) {  // chunk j: k = 16 j .. 16 j + 15
                const uint4 c4 = w8_chunk(team + 2 * h, j);
                w8_word_bf16(c4.x, v[8 * j + 0], v[8 * j + 1]);
                w8_word_bf16(c4.y, v[8 * j + 2], v[8 * j + 3]);
                w8_word_bf16(c4.z, v[8 * j + 4], v[8 * j + 5]);
                w8_word_bf16(c4.w, v[8 * j + 6], v[8 * j + 7]);
              }
            } else {
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const uint4 d4 = decode(j, s2);
                v[4 * j + 0] = d4.x;
                v[4 * j + 1] = d4.y;
                v[4 * j + 2] = d4.z;
                v[4 * j + 3] = d4.w;
              }
            }
            tmem_st32(a_lane + (uint32_t)(sa * 32), v);
            tmem_st_wait();
          } else {
            // row r of the 128-byte-swizzled K-major A stage: 16-byte chunk j holds k = 8j .. 8j + 7
            const uint32_t adst = sbase + L::a_off + sa * kABytes + r * 128;
            if constexpr (kW8) {
#pragma unroll
              for (int j = 0; j < 4; ++j) {  // code chunk j (k = 16 j .. + 15) -> A chunks 2 j, 2 j + 1
                const uint4 c4 = w8_chunk(team + 2 * h, j);
                uint32_t q[8];
                w8_word_bf16(c4.x, q[0], q[1]);
                w8_word_bf16(c4.y, q[2], q[3]);
                w8_word_bf16(c4.z, q[4], q[5]);
                w8_word_bf16(c4.w, q[6], q[7]);
                st_shared_v4(adst + ((uint32_t)((2 * j) ^ (r & 7)) << 4), make_uint4(q[0], q[1], q[2], q[3]));
                st_shared_v4(adst + ((uint32_t)((2 * j + 1) ^ (r & 7)) << 4), make_uint4(q[4], q[5], q[6], q[7]));
              }
            } else {
#pragma unroll
              for (int j = 0; j < 8; ++j)
                st_shared_v4(adst + ((j ^ (r & 7)) << 4), decode(j, s2));
            }
            fence_proxy_async();  // generic-proxy stores -> the tensor core's (async-proxy) reads
          }
        }
        ok = ok && warp_wait(x_full(i % SX), (i / SX) & 1, abort_flag, &g_tc_status);
        tc_fence_before();
        __syncwarp();
        named_bar_arrive(issue_bar(i), L::issue_threads);  // always: the issuer must never wait forever
      }
      if constexpr (kW8) {  // the team's chunks of this stage are read
        __syncwarp();
        if (lane == 0) mbar_arrive(c_empty(slot));
      }
    }
    __syncwarp();
    for (int rr = 0; rr < red_rounds; ++rr) {
      cluster_sync();
      cluster_sync();
    }
  } else {
    if constexpr (NACC == 4) setmaxnreg_inc<R::acc>();
    // ------------------------------------------------------------- accumulate
    const int quad = warp & 3;                  // TMEM lane quadrant
    const int cq = (warp - 12) >> 2;            // column chunk
    const int r_acc = quad * 32 + lane;         // tile row
    // Release an accumulator buffer as soon as its last 16-column chunk is read
    // (before that chunk's FMAs) where a thread reads 64 columns per group: measured
    // 10 % faster at BN = 256 and BN = 64, 3 % slower at BN = 128 (32 columns).
    constexpr bool kEarlyRelease = kCols >= 64 && kCols % 16 == 0;
    float2 acc[kCols / 2];
#pragma unroll
    for (int i = 0; i < kCols / 2; ++i) acc[i] = make_float2(0.f, 0.f);
    bool acc_ok = true;
    // weight row of this tile row (SwiGLU: gate rows then up rows), and whether it is a real row
    const int64_t row = MODE == 1 ? (r_acc < 64 ? m0 + r_acc : p.N + m0 + (r_acc - 64)) : m0 + r_acc;
    const bool row_ok = MODE == 1 ? (m0 + (r_acc & 63) < p.N) : row < n_rows;
    const uint16_t* scl = wsel_b ? p.scales_b : p.scales;
    const uint32_t tlane = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(cq * kCols);
    if constexpr (kFold) {
      // The sum over the whole K share is complete once the issuer's final commit has
      // landed: one warp polls for it, the others sleep on a named barrier.  Then one
      // readback, undoing the powers of two the operands were taken at.
      if (warp == 12) acc_ok = warp_wait(fin_bar, 0, abort_flag, &g_tc_status);
      named_bar_sync(kAccBar, 128 * NACC);
      acc_ok = acc_ok && !*abort_flag;
      const int rfr = row_ok ? __ldg(p.rf + row) : 0;
      if (acc_ok && ng > 0) {
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < kCols; c += 16) {
          uint32_t v[16];
          tmem_ld_cols<16>(tlane + c, v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; j += 2) {
            const int64_t t = t0 + cq * kCols + c + j;
            const int e0 = t < p.T ? __ldg(p.xe + t) : 0;
            const int e1 = t + 1 < p.T ? __ldg(p.xe + t + 1) : 0;
            acc[(c + j) / 2] = make_float2(__uint_as_float(v[j]) * exp2i(rfr + e0),
                                           __uint_as_float(v[j + 1]) * exp2i(rfr + e1));
          }
        }
      }
    } else if constexpr (kW8) {
      // W8G32: a row holds K_pad / 32 scales; group i (64 wide) has the pair 2 ga, 2 ga + 1,
      // one 32-bit load, fetched a group ahead.  Its two partials sit in buffers 2b, 2b + 1.
      const uint32_t* srow8 = reinterpret_cast<const uint32_t*>(scl + (row_ok ? row : 0) * (p.Kp >> 5));
      uint32_t sp_next = (row_ok && ng > 0) ? __ldg(srow8 + g_begin) : 0u;
      for (int i = 0; i < NB && i < ng; ++i) named_bar_arrive(issue_bar(i), L::issue_threads);
      for (int i = 0; i < ng; ++i) {
        const int b = i % NB;
        const uint32_t sp = sp_next;
        if (row_ok && i + 1 < ng) sp_next = __ldg(srow8 + g_begin + i + 1);
        acc_ok = acc_ok && warp_wait(mma_done(i), ring_par(i), abort_flag, &g_tc_status);
        if (acc_ok) {
          tc_fence_after();
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const float sf = fp16_bits_to_float((uint16_t)(hh ? (sp >> 16) : (sp & 0xFFFFu)));
            const float2 s2 = make_float2(sf, sf);
            const uint32_t dcol = tlane + (uint32_t)((2 * b + hh) * BN);
#pragma unroll
            for (int c = 0; c < kCols; c += 16) {
              uint32_t v[16];
              tmem_ld_cols<16>(dcol + c, v);
              tmem_ld_wait();
#pragma unroll
              for (int j = 0; j < 16; j += 2)
                acc[(c + j) / 2] = ffma2(make_float2(__uint_as_float(v[j]), __uint_as_float(v[j + 1])), s2, acc[(c + j) / 2]);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (i + NB < ng) named_bar_arrive(issue_bar(i + NB), L::issue_threads);  // buffers 2b, 2b + 1 are free
      }
    } else {
      // Scales are read as pairs of groups (a row holds K_pad / 64 scales, an even
      // 4-byte boundary); the next pair is fetched as soon as the current one is used.
      const uint32_t* srow = reinterpret_cast<const uint32_t*>(scl + (row_ok ? row : 0) * (p.Kp >> 6));
      int pcur = g_begin >> 1;
      uint32_t s_cur = row_ok ? __ldg(srow + pcur) : 0u;
      uint32_t s_nxt = (row_ok && 2 * (pcur + 1) < p.nk) ? __ldg(srow + pcur + 1) : 0u;
      // the first NB groups find their accumulator buffers free
      for (int i = 0; i < NB && i < ng; ++i) named_bar_arrive(issue_bar(i), L::issue_threads);
      for (int i = 0; i < ng; ++i) {
        const int b = i % NB, ga = g_begin + i;
        if ((ga >> 1) != pcur) {
          ++pcur;
          s_cur = s_nxt;
          s_nxt = (row_ok && 2 * (pcur + 1) < p.nk) ? __ldg(srow + pcur + 1) : 0u;
        }
        const float sf = fp16_bits_to_float((uint16_t)((ga & 1) ? (s_cur >> 16) : (s_cur & 0xFFFFu)));
        const float2 s2 = make_float2(sf, sf);
        acc_ok = acc_ok && warp_wait(mma_done(i), ring_par(i), abort_flag, &g_tc_status);
        bool released = false;
        if (acc_ok) {
          tc_fence_after();
          const uint32_t dcol = tlane + (uint32_t)(b * BN);
  #pragma unroll
          for (int c = 0; c < kCols; c += 16) {
            constexpr int kRest = kCols % 16;
            if (c + 16 <= kCols) {
              uint32_t v[16];
              tmem_ld_cols<16>(dcol + c, v);
              tmem_ld_wait();
              if (kEarlyRelease && c + 16 == kCols) {
                // the whole partial is in registers: hand buffer b back to the MMA
                // before the last chunk's FMAs
                tc_fence_before();
                __syncwarp();
                if (i + NB < ng) named_bar_arrive(issue_bar(i + NB), L::issue_threads);
                released = true;
              }
  #pragma unroll
              for (int j = 0; j < 16; j += 2)
                acc[(c + j) / 2] = ffma2(make_float2(__uint_as_float(v[j]), __uint_as_float(v[j + 1])), s2, acc[(c + j) / 2]);
            } else {
              // remainder of 4, 8 or 12 columns
              if constexpr (kRest >= 8) {
                uint32_t v[8];
                tmem_ld_cols<8>(dcol + c, v);
                tmem_ld_wait();
  #pragma unroll
                for (int j = 0; j < 8; j += 2)
                  acc[(c + j) / 2] = ffma2(make_float2(__uint_as_float(v[j]), __uint_as_float(v[j + 1])), s2, acc[(c + j) / 2]);
              }
              if constexpr (kRest % 8 == 4) {
                constexpr int c4 = (kRest >= 8) ? 8 : 0;
                uint32_t v[4];
                tmem_ld_cols<4>(dcol + c + c4, v);
                tmem_ld_wait();
  #pragma unroll
                for (int j = 0; j < 4; j += 2)
                  acc[(c + c4 + j) / 2] =
                      ffma2(make_float2(__uint_as_float(v[j]), __uint_as_float(v[j + 1])), s2, acc[(c + c4 + j) / 2]);
              }
            }
          }
        }
        if (!released) {
          tc_fence_before();
          __syncwarp();
          if (i + NB < ng) named_bar_arrive(issue_bar(i + NB), L::issue_threads);  // buffer b is free for group i + NB
        }
      }

    }

    // ----------------------------------------------------------- split-K reduction across the cluster
    __syncwarp();
    // rounds of kRedSlots partial tiles; rank 0 adds them in rank order (deterministic)
    for (int rr = 0; rr < red_rounds; ++rr) {
      const int q0 = 1 + rr * L::kRedSlots;
      const int q1 = q0 + L::kRedSlots < splitk ? q0 + L::kRedSlots : splitk;
      // every CTA of the cluster is past its main loop, and rank 0 has added the previous
      // round: rank 0's buffers are free
      cluster_sync();
      if ((int)crank >= q0 && (int)crank < q1) {
        const uint32_t remote0 = mapa_shared(sbase, 0);
#pragma unroll
        for (int c = 0; c < kCols; c += 4) {
          const uint32_t off = ((((int)crank - q0) * (BN / 4) + (cq * kCols + c) / 4) * kTileM + r_acc) * 16;
          st_cluster_v4(remote0 + off, acc[c / 2].x, acc[c / 2].y, acc[c / 2 + 1].x, acc[c / 2 + 1].y);
        }
      }
      cluster_sync();  // this round's partial sums have landed in rank 0
      if (crank == 0) {
#pragma unroll 1
        for (int q = q0; q < q1; ++q) {
#pragma unroll
          for (int c = 0; c < kCols; c += 4) {
            const uint32_t off = (((q - q0) * (BN / 4) + (cq * kCols + c) / 4) * kTileM + r_acc) * 16;
            const float4 v = ld_shared_f4(sbase + off);
            acc[c / 2] = fadd2(acc[c / 2], make_float2(v.x, v.y));
            acc[c / 2 + 1] = fadd2(acc[c / 2 + 1], make_float2(v.z, v.w));
          }
        }
      }
    }

    // ----------------------------------------------------------- epilogue: Y[t, row] = bf16(acc [+ R[t, row]])
    if constexpr (MODE == 1) {
      // SwiGLU: the up rows (tile rows 64..127) hand their FP32 sums to the gate rows through
      // shared memory (the pipeline buffers are free: every MMA and copy has completed); the
      // gate rows store y[t, f] = bf16(silu(g) * u), silu(g) = g / (1 + e^-g) in FP32
      float* xch = reinterpret_cast<float*>(smem);   // [64 rows][BN tokens]
      named_bar_sync(kSwiBar, 128 * NACC);            // the split-K partials in these buffers are consumed
      if (crank == 0 && r_acc >= 64) {
#pragma unroll
        for (int j = 0; j < kCols; ++j)
          xch[(r_acc - 64) * BN + cq * kCols + j] = (j & 1) ? acc[j / 2].y : acc[j / 2].x;
      }
      named_bar_sync(kSwiBar, 128 * NACC);
      if (crank == 0 && acc_ok && !*abort_flag && row_ok && r_acc < 64) {
#pragma unroll
        for (int j = 0; j < kCols; ++j) {
          const int64_t t = t0 + cq * kCols + j;
          const float gt = (j & 1) ? acc[j / 2].y : acc[j / 2].x;
          const float up = xch[r_acc * BN + cq * kCols + j];
          if (t < p.T) p.y[t * p.N + m0 + r_acc] = float_to_bf16_bits(gt / (1.f + expf(-gt)) * up);
        }
      }
    } else if (crank == 0 && acc_ok && !*abort_flag && row_ok) {
      uint16_t* yo = wsel_b ? p.y_b : p.y;
      // (a residual exists only for LinearAdd: the plain exact Q4 form)
      if (kFold || FMT != 0 || MODE != 0 || p.r == nullptr) {
#pragma unroll
        for (int j = 0; j < kCols; ++j) {
          const int64_t t = t0 + cq * kCols + j;
          const float v = (j & 1) ? acc[j / 2].y : acc[j / 2].x;
          if (t < p.T) yo[t * n_rows + row] = float_to_bf16_bits(v);
        }
      } else {
        // LinearAdd: the residual joins the FP32 sum.  R may be Y, so each element is read
        // before it is stored; the reads of a 4-token chunk are issued together (one round
        // trip to memory per chunk, not one per element; larger chunks spill the 256-wide
        // tile's accumulate warps).
        constexpr int kChunk = kCols < 4 ? kCols : 4;
#pragma unroll
        for (int j0 = 0; j0 < kCols; j0 += kChunk) {
          uint32_t rv[kChunk];
#pragma unroll
          for (int j = 0; j < kChunk; ++j) {
            const int64_t t = t0 + cq * kCols + j0 + j;
            rv[j] = t < p.T ? (uint32_t)p.r[t * n_rows + row] : 0u;
          }
#pragma unroll
          for (int j = 0; j < kChunk; ++j) {
            const int64_t t = t0 + cq * kCols + j0 + j;
            const float v = ((j0 + j) & 1) ? acc[(j0 + j) / 2].y : acc[(j0 + j) / 2].x;
            if (t < p.T) yo[t * n_rows + row] = float_to_bf16_bits(v + __uint_as_float(rv[j] << 16));
          }
        }
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(done_bar);
  }
}

// ----------------------------------------------------------------- folded-form operands
// One pass before the tile kernel, in two kinds of CTA:
//   * CTA t < T: token t.  Its largest |x| (compared as bf16 magnitude bits) fixes a
//     power of two 2^xe[t] that puts that maximum in [2^14, 2^15); x * 2^-xe[t] is then
//     exact in fp16 for every element down to 2^-38 of the maximum (smaller ones round
//     as fp16 subnormals), and is stored as the fp16 token row xh[t, :].
//   * the other CTAs: 8 weight rows each, one warp per row.  The row's largest scale
//     magnitude (groups holding columns < K) fixes 2^rf[n] that puts it in
//     [2^11, 2^12), so every decoded weight (q - 8) * s * 2^-rf stays below 2^15 in
//     magnitude (no fp16 overflow) and small scales keep their precision.
// Rows and tokens holding Inf or NaN keep a shift of 0 so those values propagate.
constexpr int kPrepRowsPerCta = 8;

__global__ void __launch_bounds__(256) q4_tc_prep_kernel(const uint16_t* __restrict__ x,
                                                         const uint16_t* __restrict__ scales, uint16_t* __restrict__ xh,
                                                         int* __restrict__ xe, int* __restrict__ rf, int64_t T, int64_t K,
                                                         int64_t N, int64_t sc_pitch, int nk) {
  pdl_launch_dependents();
  pdl_wait_previous();  // x and the scales may come from the previous kernel; xh may still be read by it
  __shared__ uint32_t red[8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if ((int64_t)blockIdx.x < T) {
    const int64_t t = blockIdx.x;
    const uint4* src = reinterpret_cast<const uint4*>(x + t * K);
    uint4* dst = reinterpret_cast<uint4*>(xh + t * K);
    const int64_t nc = K / 8;  // K is a multiple of 8
    uint32_t m2 = 0;           // two 16-bit maxima of |x| bits
    for (int64_t c = threadIdx.x; c < nc; c += 256) {
      const uint4 v = __ldg(src + c);
      m2 = __vmaxu2(m2, v.x & 0x7FFF7FFFu);
      m2 = __vmaxu2(m2, v.y & 0x7FFF7FFFu);
      m2 = __vmaxu2(m2, v.z & 0x7FFF7FFFu);
      m2 = __vmaxu2(m2, v.w & 0x7FFF7FFFu);
    }
    uint32_t m = __reduce_max_sync(0xffffffffu, max(m2 & 0xFFFFu, m2 >> 16));
    if (lane == 0) red[warp] = m;
    __syncthreads();
#pragma unroll
    for (int w = 0; w < 8; ++w) m = max(m, red[w]);
    const int E = (int)(m >> 7);  // bf16 biased exponent of the largest |x|
    const int e = (m == 0 || E == 255) ? 0 : min(max(E - 141, -100), 100);
    const float sc = exp2i(-e);
    for (int64_t c = threadIdx.x; c < nc; c += 256) {
      const uint4 v = __ldg(src + c);
      const uint32_t in[4] = {v.x, v.y, v.z, v.w};
      uint32_t out[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(out[j]) : "f"(bf16hi(in[j]) * sc), "f"(bf16lo(in[j]) * sc));
      dst[c] = make_uint4(out[0], out[1], out[2], out[3]);
    }
    if (threadIdx.x == 0) xe[t] = e;
  } else {
    const int64_t n = ((int64_t)blockIdx.x - T) * kPrepRowsPerCta + warp;
    if (n < N) {
      const uint16_t* srow = scales + n * sc_pitch;
      uint32_t m = 0;
      for (int g = lane; g < nk; g += 32) m = max(m, (uint32_t)(__ldg(srow + g) & 0x7FFFu));
      m = __reduce_max_sync(0xffffffffu, m);
      const int E = (int)(m >> 10);  // fp16 biased exponent of the largest |s|
      if (lane == 0) rf[n] = (m == 0 || E == 31) ? 0 : E - 26;
    }
  }
}

// Folded-form workspace: xh [T, K] fp16, xe [T] int, rf [N] int, each 256-byte aligned.
size_t r256(size_t b) { return (b + 255) / 256 * 256; }
size_t fold_ws_xe(int64_t, int64_t K, int64_t T) { return r256((size_t)T * (size_t)K * 2); }
size_t fold_ws_rf(int64_t N, int64_t K, int64_t T) { return fold_ws_xe(N, K, T) + r256((size_t)T * 4); }
size_t fold_ws_bytes(int64_t N, int64_t K, int64_t T) { return fold_ws_rf(N, K, T) + r256((size_t)N * 4); }

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

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

CtxGetCurrentFn ctx_get_current_fn() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(f);
  });
  return fn;
}

}  // namespace

bool encode_map_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                   uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

bool make_map_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                 uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                 CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  return encode_map_2d(m, dt, base, inner, outer, row_bytes, box_inner, box_outer, swizzle);
}

template <int BN, bool kFold, int FMT = 0, int MODE = 0>
int set_kernel_attrs() {
  using L = TcSmem<BN, kFold, FMT>;
  static bool attr_set[64] = {};
  int dev = 0;
  if (cuda_check(cudaGetDevice(&dev), "cudaGetDevice")) return Q4LIN_ERR_CUDA;
  if (dev < 64 && attr_set[dev]) return Q4LIN_OK;
  if (cuda_check(cudaFuncSetAttribute(q4_tc_kernel<BN, kFold, FMT, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      L::alloc),
                 "tc: cudaFuncSetAttribute(max dynamic shared memory)"))
    return Q4LIN_ERR_CUDA;
  if (cuda_check(cudaFuncSetAttribute(q4_tc_kernel<BN, kFold, FMT, MODE>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1),
                 "tc: cudaFuncSetAttribute(cluster size)"))
    return Q4LIN_ERR_CUDA;
  if (dev < 64) attr_set[dev] = true;
  return Q4LIN_OK;
}

// How many clusters of `size` CTAs of this kernel can be resident at once (0 on
// error).  Clusters are placed within one GPC, so this is below sms / size when
// the GPCs' SM counts are not multiples of the cluster size.
template <int BN, bool kFold>
int resident_clusters(int size) {
  using L = TcSmem<BN, kFold>;
  static int cache[64][9] = {};
  int dev = 0;
  if (size < 1 || size > 8 || cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev < 64 && cache[dev][size]) return cache[dev][size];
  if (set_kernel_attrs<BN, kFold>() != Q4LIN_OK) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1, 1, (unsigned)size);
  cfg.blockDim = dim3(L::threads, 1, 1);
  cfg.dynamicSmemBytes = L::alloc;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = (unsigned)size;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, q4_tc_kernel<BN, kFold, 0>, &cfg) != cudaSuccess || n < 0) {
    cudaGetLastError();
    n = 0;
  }
  if (dev < 64 && n > 0) cache[dev][size] = n;
  return n;
}

template <int BN, bool kFold, int FMT = 0, int MODE = 0>
int launch_tile(const LinearArgs& a, int splitk, int64_t tile_base, int64_t n_tiles) {
  using L = TcSmem<BN, kFold, FMT>;
  static_assert(L::alloc <= 232448, "shared memory budget");
  if (splitk < 1 || splitk > 8 || splitk > L::max_splitk) {
    set_error_detail("tc: split-K factor out of range for this tile");
    return Q4LIN_ERR_INVALID_ARG;
  }
  if (const int rc = set_kernel_attrs<BN, kFold, FMT, MODE>()) return rc;
  CUtensorMap tm_codes, tm_x, tm_high;
  // code plane rows hold K_pad / 2 bytes; X rows K values, whose positions k >= K read
  // as zeros (out-of-range tile elements), so a partial last group sees x = 0 beyond K.
  // The folded form reads the fp16 token rows the prep kernel left in the workspace.
  const int64_t Kp = k_pad(a.K);
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  const void* xsrc = kFold ? static_cast<const void*>(ws) : static_cast<const void*>(a.x);
  // SwiGLU: the code plane holds 2N rows and a tile loads 64 gate rows and 64 up rows
  const uint64_t code_rows = a.mode == 1 ? (uint64_t)(2 * a.N) : (uint64_t)a.N;
  const uint64_t code_row_bytes = (uint64_t)(L::kW8 ? Kp : Kp / 2);  // W8G32: one byte per weight
  if (!make_map_2d(&tm_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.wq, code_row_bytes, code_rows, code_row_bytes, 128,
                   a.mode == 1 ? kTileM / 2 : kTileM) ||
      !make_map_2d(&tm_x, kFold ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, xsrc,
                   (uint64_t)a.K, (uint64_t)a.T, (uint64_t)a.K * 2, 64, BN)) {
    set_error_detail("tc: cuTensorMapEncodeTiled failed (or is unavailable)");
    return Q4LIN_ERR_CUDA;
  }
  // Q5 / Q6 high-bit plane: rows of K_pad * kHB / 8 bytes, boxes of 4 groups x 128 rows, unswizzled
  if constexpr (L::kHB > 0) {
    const uint64_t hrow = (uint64_t)(Kp * L::kHB / 8);
    if (!make_map_2d(&tm_high, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.wh, hrow, (uint64_t)a.N, hrow,
                     (uint32_t)(kGroupsPerW * 8 * L::kHB), kTileM, CU_TENSOR_MAP_SWIZZLE_NONE)) {
      set_error_detail("tc: cuTensorMapEncodeTiled failed for the high-bit plane");
      return Q4LIN_ERR_CUDA;
    }
  } else if (a.mode == 2) {  // LinearPair: the second weight's code plane in this slot
    if (!make_map_2d(&tm_high, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.wq_b, (uint64_t)(Kp / 2), (uint64_t)a.n_b,
                     (uint64_t)(Kp / 2), 128, kTileM)) {
      set_error_detail("tc: cuTensorMapEncodeTiled failed for the second weight");
      return Q4LIN_ERR_CUDA;
    }
  } else {
    tm_high = tm_codes;  // unused
  }
  const int* xe = kFold ? reinterpret_cast<const int*>(ws + fold_ws_xe(a.N, a.K, a.T)) : nullptr;
  const int* rf = kFold ? reinterpret_cast<const int*>(ws + fold_ws_rf(a.N, a.K, a.T)) : nullptr;
  const uint32_t tiles_a = (uint32_t)((a.N + kTileM - 1) / kTileM);
  const uint32_t tiles_m = a.mode == 1 ? (uint32_t)((a.N + kTileM / 2 - 1) / (kTileM / 2))
                         : a.mode == 2 ? tiles_a + (uint32_t)((a.n_b + kTileM - 1) / kTileM)
                                       : tiles_a;
  const TcParams p{a.scales, a.y, xe, rf, a.r, a.N, Kp, a.T, (int)((a.K + 63) / 64), splitk, (uint32_t)tile_base,
                   tiles_m, a.mode, tiles_a, a.scales_b, a.y_b, a.n_b};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)n_tiles, 1, (unsigned)splitk);
  cfg.blockDim = dim3(L::threads, 1, 1);
  cfg.dynamicSmemBytes = L::alloc;
  cfg.stream = a.stream;
  // a cluster along K for a split, and programmatic dependent launch (the kernel waits
  // for its predecessor before touching global memory; measured 1 us per call saved)
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (splitk > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = 1;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = (unsigned)splitk;
    ++na;
  }
  attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  cfg.attrs = attr;
  cfg.numAttrs = (unsigned)na;
  return cuda_check(cudaLaunchKernelEx(&cfg, q4_tc_kernel<BN, kFold, FMT, MODE>, tm_codes, tm_x, tm_high, p),
                    "tc: kernel launch");
}

// The folded form's operand pass (programmatic dependent launch like the tile kernel).
int launch_prep(const LinearArgs& a) {
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  const int64_t blocks = a.T + (a.N + kPrepRowsPerCta - 1) / kPrepRowsPerCta;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cuda_check(cudaLaunchKernelEx(&cfg, q4_tc_prep_kernel, a.x, a.scales, reinterpret_cast<uint16_t*>(ws),
                                       reinterpret_cast<int*>(ws + fold_ws_xe(a.N, a.K, a.T)),
                                       reinterpret_cast<int*>(ws + fold_ws_rf(a.N, a.K, a.T)), a.T, a.K, a.N,
                                       k_pad(a.K) / 64, (int)((a.K + 63) / 64)),
                    "tc: prep kernel launch");
}

int red_slots_for(int bn) {  // partial tiles the reduction moves per round (the folded layout's: fewest)
  switch (bn) {
    case 256: return TcSmem<256, true>::kRedSlots;
    case 128: return TcSmem<128, true>::kRedSlots;
    case 64: return TcSmem<64, true>::kRedSlots;
    case 32: return TcSmem<32, true>::kRedSlots;
    default: return TcSmem<16, true>::kRedSlots;
  }
}

int max_splitk_for(int bn) {  // the same shared-memory layout in both forms
  switch (bn) {
    case 256: return TcSmem<256, true>::max_splitk;
    case 128: return TcSmem<128, true>::max_splitk;
    case 64: return TcSmem<64, true>::max_splitk;
    case 32: return TcSmem<32, true>::max_splitk;
    default: return TcSmem<16, true>::max_splitk;
  }
}

int resident_clusters_for(int bn, int size) {  // same block size and shared memory in both forms
  switch (bn) {
    case 256: return resident_clusters<256, true>(size);
    case 128: return resident_clusters<128, true>(size);
    case 64: return resident_clusters<64, true>(size);
    case 32: return resident_clusters<32, true>(size);
    default: return resident_clusters<16, true>(size);
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

// Per-CTA costs of the tile kernel, measured on a GB300 with every (width, split)
// plan forced in turn over several shapes (ns): one 64-wide K group at full
// occupancy, the fixed part of a CTA's life (setup, pipeline fill, epilogue), and
// the cluster reduction of a split per token column of the tile.  The wave model
// built from them reproduces the measured times of those plans to within ~10%.
struct TileCost {
  int bn;
  double group_ns;
  double fixed_ns;
};
// exact form (per-group accumulators read back and scaled in FP32)
constexpr TileCost kTileCostExact[] = {
    {16, 310.0, 4300.0}, {32, 330.0, 4400.0}, {64, 335.0, 6500.0}, {128, 440.0, 5300.0}, {256, 580.0, 7800.0}};
// folded form (one accumulator per K share; the 256 entry measured at T = 1024 on
// 6144 x 5120 and 34816 x 5120, the others estimated from the exact form's)
constexpr TileCost kTileCostFold[] = {
    {16, 250.0, 4300.0}, {32, 270.0, 4400.0}, {64, 280.0, 6500.0}, {128, 330.0, 5300.0}, {256, 450.0, 7000.0}};
constexpr double kSplitNsPerColumn = 22.0;

const TileCost& tile_cost(int bn, bool fold) {
  const TileCost* t = fold ? kTileCostFold : kTileCostExact;
  for (int i = 0; i < 5; ++i)
    if (t[i].bn == bn) return t[i];
  return t[0];
}

bool route_folds(int route) { return route == Q4LIN_ROUTE_TC_FP16; }

// The second launch of a tail plan: launch latency not hidden behind a previous kernel.
constexpr double kTailLaunchNs = 1500.0;
constexpr double kTailGroupFactor = 1.3;

static int64_t tile_count(int64_t N, int64_t T, int bn) { return ((N + kTileM - 1) / kTileM) * ((T + bn - 1) / bn); }

TcPlan tc_plan(int route, int64_t N, int64_t K, int64_t T, int sms, int fmt) {
  // Token-tile width candidates: the smallest MMA N covering T up to 128
  // tokens; above that 256 or 128.  For each candidate and split factor the
  // cost is waves x per-CTA time; a wave holds as many CTAs (clusters) as can
  // be resident at once (queried; without a device, sms / size).
  //
  // Tail plans: when the tiles fill one whole wave and part of a second, the
  // whole wave can run unsplit and the remaining tiles in a second launch, split
  // along K so that they fill one wave (6144 x 5120 x 1024 with 256-wide tiles:
  // 152 tiles, then 40 tiles in clusters of 2; 100.8 us instead of 113.3 us).
  int cand[2] = {0, 0};
  int ncand = 0;
  if (fmt == 3) {  // W8G32: two accumulators per group (A in shared memory at 128-wide tiles)
    cand[0] = T > 64 ? 128 : T > 32 ? 64 : T > 16 ? 32 : 16;
    ncand = 1;
  } else if (T > 128) {
    cand[0] = 256;
    cand[1] = 128;
    ncand = 2;
  } else {
    cand[0] = T > 64 ? 128 : T > 32 ? 64 : T > 16 ? 32 : 16;
    ncand = 1;
  }
  const int64_t nk = (K + 63) / 64;   // groups holding columns < K
  TcPlan best_pl{cand[0], 1, tile_count(N, T, cand[0]), 0};
  double best = -1.0;
  for (int c = 0; c < ncand; ++c) {
    const int bn = cand[c];
    const TileCost& tc = tile_cost(bn, route_folds(route));
    const int64_t tiles = tile_count(N, T, bn);
    const int smax = route == Q4LIN_ROUTE_TC ? 1 : (max_splitk_for(bn) < 8 ? max_splitk_for(bn) : 8);
    auto wave_capacity = [&](int s) -> int64_t {
      int64_t per_wave = sms / s;
      if (s > 1) {
        const int q = resident_clusters_for(bn, s);
        if (q > 0 && q < per_wave) per_wave = q;
      }
      return per_wave;
    };
    const int slots = red_slots_for(bn);
    auto cta_ns = [&](int s) -> double {
      const int rounds = s > 1 ? (s - 1 + slots - 1) / slots : 0;
      return (double)((nk + s - 1) / s) * tc.group_ns + tc.fixed_ns + rounds * kSplitNsPerColumn * bn;
    };
    for (int s = 1; s <= smax && s <= nk; ++s) {
      const int64_t per_wave = wave_capacity(s);
      if (per_wave < 1) continue;
      const int64_t waves = (tiles + per_wave - 1) / per_wave;
      const double cost = (double)waves * cta_ns(s);
      if (best < 0 || cost < best - 1e-9) {  // ties keep the earlier (fewer splits, preferred width)
        best = cost;
        best_pl = TcPlan{bn, s, tiles, 0};
      }
    }
    // Tail plans are considered after one whole wave only: behind several waves the
    // single launch's partial last wave already overlaps the stragglers of the one
    // before.  A tail CTA was measured about 25 % slower per group than the model's
    // full-occupancy figure (kTailGroupFactor).
    const int64_t per_wave1 = wave_capacity(1);
    if (smax > 1 && per_wave1 > 0 && tiles > per_wave1 && tiles < 2 * per_wave1) {
      const int64_t main_tiles = per_wave1, rest = tiles - main_tiles;
      const double main_cost = cta_ns(1);
      for (int st = 2; st <= smax && st <= nk; ++st) {
        if (rest > wave_capacity(st)) continue;
        const double cost = main_cost + kTailGroupFactor * cta_ns(st) + kTailLaunchNs;
        if (cost < best - 1e-9) {
          best = cost;
          best_pl = TcPlan{bn, 1, main_tiles, st};
        }
      }
    }
  }
  return best_pl;
}

TcPlan tc_plan_current_device(int route, int64_t N, int64_t K, int64_t T, int fmt) {
  return tc_plan(route, N, K, T, sm_count(), fmt);
}

size_t tc_workspace_bytes(int route, int64_t N, int64_t K, int64_t T) {
  return route_folds(route) ? fold_ws_bytes(N, K, T) : 0;
}

int tc_launch_count(int route, int64_t N, int64_t K, int64_t T, int fmt) {
  const TcPlan pl = tc_plan_current_device(route, N, K, T, fmt);
  return (pl.main_tiles < tile_count(N, T, pl.bn) ? 2 : 1) + (route_folds(route) ? 1 : 0);
}

bool tc_supported(int64_t N, int64_t K, int64_t T) {
  // TMA coordinates are 32-bit signed, one launch's tiles (at most, with 16-token
  // tiles) must fit the grid's x extent, and so must the prep kernel's T + N / 8 CTAs.
  return N < ((int64_t)1 << 31) && K < ((int64_t)1 << 31) && T < ((int64_t)1 << 31) &&
         tile_count(N, T, 16) < ((int64_t)1 << 31) &&
         T + (N + kPrepRowsPerCta - 1) / kPrepRowsPerCta < ((int64_t)1 << 31);
}

int tc_launch(const LinearArgs& a, int route) {
  if (!tc_supported(a.N, a.K, a.T)) {
    set_error_detail("tc: shape beyond the tensor-core route's limits");
    return Q4LIN_ERR_INVALID_ARG;
  }
  if (a.fmt != 0 && (route_folds(route) || a.fmt < 1 || a.fmt > 3)) {
    set_error_detail("tc: sibling formats run on the exact tile routes (Q5G64, Q6G64, W8G32)");
    return Q4LIN_ERR_UNSUPPORTED_SHAPE;
  }
  // rows the tile space covers: SwiGLU 2N (64 + 64 per tile), Pair both weights' row tiles
  const int64_t n_plan = a.mode == 1 ? 2 * a.N
                       : a.mode == 2 ? kTileM * ((a.N + kTileM - 1) / kTileM + (a.n_b + kTileM - 1) / kTileM)
                                     : a.N;
  if (a.mode != 0 && (a.fmt != 0 || route_folds(route))) {
    set_error_detail("tc: the fused forms run on the exact Q4 tile route");
    return Q4LIN_ERR_INVALID_ARG;
  }
  const TcPlan pl = tc_plan_current_device(route, n_plan, a.K, a.T, a.fmt);
  const bool fold = route_folds(route);
  auto launch = [&](int splitk, int64_t base, int64_t n) {
    if (a.fmt == 3) {
      switch (pl.bn) {
        case 128: return launch_tile<128, false, 3>(a, splitk, base, n);
        case 64: return launch_tile<64, false, 3>(a, splitk, base, n);
        case 32: return launch_tile<32, false, 3>(a, splitk, base, n);
        case 16: return launch_tile<16, false, 3>(a, splitk, base, n);
        default: set_error_detail("tc: no tile width for this format"); return (int)Q4LIN_ERR_UNSUPPORTED_SHAPE;
      }
    }
    if (a.fmt != 0) {
      const bool q5 = a.fmt == 1;
      switch (pl.bn) {
        case 256: return q5 ? launch_tile<256, false, 1>(a, splitk, base, n) : launch_tile<256, false, 2>(a, splitk, base, n);
        case 128: return q5 ? launch_tile<128, false, 1>(a, splitk, base, n) : launch_tile<128, false, 2>(a, splitk, base, n);
        case 64: return q5 ? launch_tile<64, false, 1>(a, splitk, base, n) : launch_tile<64, false, 2>(a, splitk, base, n);
        case 32: return q5 ? launch_tile<32, false, 1>(a, splitk, base, n) : launch_tile<32, false, 2>(a, splitk, base, n);
        case 16: return q5 ? launch_tile<16, false, 1>(a, splitk, base, n) : launch_tile<16, false, 2>(a, splitk, base, n);
        default: set_error_detail("tc: no tile width for this format"); return (int)Q4LIN_ERR_UNSUPPORTED_SHAPE;
      }
    }
    if (fold) {
      switch (pl.bn) {
        case 256: return launch_tile<256, true>(a, splitk, base, n);
        case 128: return launch_tile<128, true>(a, splitk, base, n);
        case 64: return launch_tile<64, true>(a, splitk, base, n);
        case 32: return launch_tile<32, true>(a, splitk, base, n);
        default: return launch_tile<16, true>(a, splitk, base, n);
      }
    }
    if (a.mode == 1) {
      switch (pl.bn) {
        case 256: return launch_tile<256, false, 0, 1>(a, splitk, base, n);
        case 128: return launch_tile<128, false, 0, 1>(a, splitk, base, n);
        case 64: return launch_tile<64, false, 0, 1>(a, splitk, base, n);
        case 32: return launch_tile<32, false, 0, 1>(a, splitk, base, n);
        default: return launch_tile<16, false, 0, 1>(a, splitk, base, n);
      }
    }
    if (a.mode == 2) {
      switch (pl.bn) {
        case 256: return launch_tile<256, false, 0, 2>(a, splitk, base, n);
        case 128: return launch_tile<128, false, 0, 2>(a, splitk, base, n);
        case 64: return launch_tile<64, false, 0, 2>(a, splitk, base, n);
        case 32: return launch_tile<32, false, 0, 2>(a, splitk, base, n);
        default: return launch_tile<16, false, 0, 2>(a, splitk, base, n);
      }
    }
    switch (pl.bn) {
      case 256: return launch_tile<256, false>(a, splitk, base, n);
      case 128: return launch_tile<128, false>(a, splitk, base, n);
      case 64: return launch_tile<64, false>(a, splitk, base, n);
      case 32: return launch_tile<32, false>(a, splitk, base, n);
      default: return launch_tile<16, false>(a, splitk, base, n);
    }
  };
  const int64_t tiles = tile_count(n_plan, a.T, pl.bn);
  int rc = fold ? launch_prep(a) : Q4LIN_OK;
  if (rc == Q4LIN_OK) rc = launch(pl.splitk, 0, pl.main_tiles);
  if (rc == Q4LIN_OK && pl.main_tiles < tiles) rc = launch(pl.tail_splitk, pl.main_tiles, tiles - pl.main_tiles);
  return rc;
}

// ----------------------------------------------------------------- allocation-free fp16 route
// Some callers cannot allocate device memory per call: code that runs where
// cudaMalloc is off limits (inside a stream capture that must not allocate, or
// under an allocator that owns the whole device and hands out no scratch), or a
// host that links this library without any allocator at all.  For them the fp16
// tile route keeps its operand scratch in this fixed array instead of a caller
// workspace.  Every process that loads the library holds the array on every GPU it
// uses until it exits; all calls share it, and each call's prep kernel rewrites
// every byte the tile kernel reads, so nothing needs clearing between calls.
constexpr size_t kStaticScratchBytes = (size_t)16 << 20;
static __device__ __align__(256) uint8_t g_fp16_scratch[kStaticScratchBytes];

size_t tc_fp16_static_capacity() { return kStaticScratchBytes; }

bool tc_fp16_static_fits(int64_t N, int64_t K, int64_t T) {
  return tc_supported(N, K, T) && fold_ws_bytes(N, K, T) <= kStaticScratchBytes;
}

int tc_fp16_static_launch(const LinearArgs& args) {
  if (!tc_fp16_static_fits(args.N, args.K, args.T)) {
    set_error_detail("fp16 route without allocation: 2*T*K + 4*T + 4*N bytes (each rounded up to 256) "
                     "exceed its 16 MiB static scratch");
    return Q4LIN_ERR_UNSUPPORTED_SHAPE;
  }
  // The array's device address, looked up once per CUDA context with that context
  // current (in host code its name is only a stand-in, not a device address).  The
  // cache is keyed by the context, not the device ordinal: after cudaDeviceReset, or
  // under another context on the same device, the address is looked up again.
  static CUcontext ctx_of[64] = {};
  static void* addr_of[64] = {};
  static int n_ctx = 0;
  static std::mutex mu;
  CUcontext ctx = nullptr;
  if (CtxGetCurrentFn get = ctx_get_current_fn()) {
    if (get(&ctx) != CUDA_SUCCESS) ctx = nullptr;
  }
  if (ctx == nullptr) {
    // make the runtime's primary context current, then ask again
    if (const int rc = cuda_check(cudaFree(nullptr), "cudaFree(nullptr) (context set-up)")) return rc;
    CtxGetCurrentFn get = ctx_get_current_fn();
    if (get == nullptr || get(&ctx) != CUDA_SUCCESS || ctx == nullptr) {
      set_error_detail("fp16 route without allocation: no current CUDA context");
      return Q4LIN_ERR_CUDA;
    }
  }
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n_ctx; ++i)
      if (ctx_of[i] == ctx) scratch = addr_of[i];
    if (scratch == nullptr) {
      void* p = nullptr;
      if (const int rc = cuda_check(cudaGetSymbolAddress(&p, g_fp16_scratch), "cudaGetSymbolAddress(scratch)"))
        return rc;
      // a context seen before whose slot is reused (table full): overwrite round robin
      const int slot = n_ctx < 64 ? n_ctx++ : (int)(reinterpret_cast<uintptr_t>(ctx) % 64);
      ctx_of[slot] = ctx;
      addr_of[slot] = p;
      scratch = p;
    }
  }
  LinearArgs a = args;
  a.workspace = scratch;
  return tc_launch(a, Q4LIN_ROUTE_TC_FP16);
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
