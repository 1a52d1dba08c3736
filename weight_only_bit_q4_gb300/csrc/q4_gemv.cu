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
  const int64_t Kp = (K + 127) / 128 * 128;   // planes are stored for K_pad columns
  const int64_t chunks = (K + 31) >> 5;        // 16-byte chunks (32 weights) holding columns < K
  const int64_t row_bytes = Kp >> 1;
  const int64_t groups = Kp >> 6;

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
        // columns k >= K (a multiple of 8) read as zeros
        const uint4 xv = (c * 32 + i * 8 < K) ? ld_nc_u4(xrow[t] + c * 32 + i * 8) : make_uint4(0, 0, 0, 0);
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
// range of rows (balanced to one row), cut into blocks of RB rows.  Thread 0
// copies x into shared memory (one bulk copy per CTA), then streams every
// block's code bytes and its scales (a block's scales are one contiguous run
// of the scale plane) into a ring of shared-memory slots with 1-D bulk async
// copies, so the CTA's share is in flight from the start and no consumer ever
// waits on a global load.
//
// K is cut into column groups of 32 chunks (a chunk = 16 code bytes = 32
// weights = half a scale group).  A work item is one (block, column group)
// pair; the W consumer warps take the items in block-major order, warp w the
// items w, w + W, w + 2W, ...  Where a multiple of the group count between 12
// and 15 exists, W is that multiple, so a warp keeps one column group and its
// 32 x values per lane in registers for the whole kernel; otherwise W = 15 and
// a warp reloads its x values from shared memory whenever its group changes.
// Per item a lane decodes one conflict-free 16-byte code chunk per row into
// (128 + q) floats with byte permutes, accumulates with packed FP32 FMAs,
// applies (partial - 136 * sum x) * s, and the warp reduces the RB row partials
// with a halving butterfly (each exchange hands half of the remaining rows to
// the partner lane, so 8 rows take 9 shuffles instead of 40).  The
// column-group partials of a row are summed in a fixed order at the end
// (deterministic), then rounded to bf16.
constexpr int kStreamThreads = 512;
constexpr int kStreamConsumers = 15;   // warps 1..15
constexpr int64_t kStreamSmemBudget = 232448 - 1024;
// L2 prefetch of one CTA's codes before the dependency wait, at most.  Enough to
// cover the start of the CTA's stream; prefetching a whole large share competes
// with the ring's own copies (measured: 34816 x 5120 takes 31.8 us with 512 KB,
// 27.7 us with 64 KB; the 6144 x 5120 decode call is 7.8 us either way).
constexpr int64_t kPrefetchCapBytes = 64 * 1024;

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

__device__ __forceinline__ uint2 ld_shared_v2(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t ld_shared_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

// nibbles 0..3 of m (bits 0..15) to the low nibbles of bytes 0..3
__device__ __forceinline__ uint32_t spread_nibbles_to_bytes(uint32_t m) {
  m = (m | (m << 8)) & 0x00FF00FFu;
  return (m | (m << 4)) & 0x0F0F0F0Fu;
}

__device__ __forceinline__ uint16_t ld_shared_u16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

// Weight formats of the streaming GEMV (linear-benchmark.md section 4, format
// table): Q4G64 (the layer's own), and the sibling formats Q5G64 / Q6G64 (the
// Q4 code plane plus a plane of 1 or 2 high bits per weight, in k order from
// each byte's least significant bit; zero points 16 and 32) and W8G32 (signed
// int8 codes, one scale per 32 weights).
enum : int { kFmtQ4 = 0, kFmtQ5 = 1, kFmtQ6 = 2, kFmtW8 = 3 };
__host__ __device__ constexpr int fmt_high_bits(int f) { return f == kFmtQ5 ? 1 : f == kFmtQ6 ? 2 : 0; }
__host__ __device__ constexpr int fmt_group(int f) { return f == kFmtW8 ? 32 : 64; }
// bytes of one stored row (Kp columns) of each plane
__host__ __device__ constexpr int64_t fmt_code_row(int f, int64_t Kp) { return f == kFmtW8 ? Kp : Kp / 2; }
__host__ __device__ constexpr int64_t fmt_high_row(int f, int64_t Kp) { return Kp * fmt_high_bits(f) / 8; }
__host__ __device__ constexpr int64_t fmt_scale_row(int f, int64_t Kp) { return Kp / fmt_group(f) * 2; }

struct StreamLayout {
  uint32_t x_off, part_off, bar_off, code_off, code_stride, high_off, high_stride, sc_off, sc_stride, bytes;
};

// x (bf16, TT rows of K), partial sums [rows_cap][nj][TT] fp32, the x barrier, nfull
// "block landed" barriers and `slots` "slot free" barriers, the code slots
// (128-byte aligned), the high-bit slots (Q5 / Q6 only) and the scale slots
// (16-byte aligned; a block's run of scales plus up to 15 bytes of alignment
// slack on either side).
__host__ __device__ inline StreamLayout stream_layout(int64_t K, int tt, int rb, int64_t rows_cap, int nj, int slots,
                                                      int nfull, int fmt = kFmtQ4) {
  StreamLayout L;
  const int64_t Kp = (K + 127) & ~(int64_t)127;   // the planes' stored width
  L.x_off = 0;
  L.part_off = (uint32_t)(tt * K * 2);
  L.bar_off = (uint32_t)((L.part_off + rows_cap * nj * tt * 4 + 15) / 16 * 16);
  L.code_off = (L.bar_off + 8 + (uint32_t)(nfull + slots) * 8 + 127) / 128 * 128;
  L.code_stride = (uint32_t)((rb * fmt_code_row(fmt, Kp) + 127) / 128 * 128);
  L.high_off = L.code_off + (uint32_t)slots * L.code_stride;
  L.high_stride = (uint32_t)((rb * fmt_high_row(fmt, Kp) + 15) / 16 * 16);
  L.sc_off = L.high_off + (uint32_t)slots * L.high_stride;
  L.sc_stride = (uint32_t)((rb * fmt_scale_row(fmt, Kp) + 32 + 15) / 16 * 16);
  L.bytes = L.sc_off + (uint32_t)slots * L.sc_stride;
  return L;
}

// Queue block b (rows [ra, ra + nr)) into slot s: its code rows, and the
// 16-byte granules of the scale plane that cover its scale run [st, en) (the
// plane starts 16-byte aligned; a granule past the plane's last full one is
// never copied -- the at most 7 scales there are read with plain loads and
// stored before the barrier arrival that publishes them).
__device__ __forceinline__ void stream_issue(const uint8_t* wq, const uint8_t* sc_plane, int64_t plane_bytes,
                                             int64_t row_bytes, int64_t sc_row_bytes, int64_t ra, int nr,
                                             uint32_t code_dst, uint32_t sc_dst, uint32_t full_bar,
                                             const uint8_t* wh = nullptr, int64_t high_row_bytes = 0,
                                             uint32_t high_dst = 0) {
  const uint32_t cbytes = (uint32_t)(nr * row_bytes);
  const uint32_t hbytes = (uint32_t)(nr * high_row_bytes);   // Q5 / Q6 high-bit rows
  const int64_t st = ra * sc_row_bytes, en = (ra + nr) * sc_row_bytes;
  const int64_t a = st & ~(int64_t)15;
  const int64_t e_up = (en + 15) & ~(int64_t)15, e_cap = plane_bytes & ~(int64_t)15;
  const int64_t e = e_up < e_cap ? e_up : e_cap;  // >= a, since st < plane_bytes
  for (int64_t t = (e > st ? e : st); t < en; t += 2)
    st_shared_u16(sc_dst + (uint32_t)(t - a), *reinterpret_cast<const uint16_t*>(sc_plane + t));
  const uint32_t sbytes = (uint32_t)(e - a);
  mbar_expect_tx(full_bar, cbytes + hbytes + sbytes);
  bulk_g2s(code_dst, wq + ra * row_bytes, cbytes, full_bar);
  if (hbytes > 0) bulk_g2s(high_dst, wh + ra * high_row_bytes, hbytes, full_bar);
  if (sbytes > 0) bulk_g2s(sc_dst, sc_plane + a, sbytes, full_bar);
}

// Sum each of the RB per-lane row partials over the warp.  Round r (offset
// 16 >> r) swaps half of the rows still held with lane ^ offset, so afterwards
// a lane holds one row whose index is read from lane bits 4, 3, ... (most
// significant first); the remaining rounds are a plain butterfly.
template <int RB>
__device__ __forceinline__ float reduce_rows(const float (&acc)[RB], int lane, int* row) {
  float a[RB];
#pragma unroll
  for (int i = 0; i < RB; ++i) a[i] = acc[i];
  int r = 0;
#pragma unroll
  for (int n = RB, off = 16; n > 1; n >>= 1, off >>= 1) {
    const bool h = (lane & off) != 0;
#pragma unroll
    for (int q = 0; q < n / 2; ++q) {
      const float send = h ? a[q] : a[q + n / 2];
      const float keep = h ? a[q + n / 2] : a[q];
      a[q] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
    r = 2 * r + (h ? 1 : 0);
  }
#pragma unroll
  for (int off = 16 / RB; off >= 1; off >>= 1) a[0] += __shfl_xor_sync(0xffffffffu, a[0], off);
  *row = r;
  return a[0];
}

template <int RB, int TT, bool kPad, int FMT>
__global__ void __launch_bounds__(kStreamThreads, 1)
q4_gemv_stream_kernel(const uint8_t* __restrict__ wq, const uint16_t* __restrict__ scales,
                      const uint16_t* __restrict__ x, uint16_t* __restrict__ y, int64_t N, int64_t K,
                      int64_t rows_cap, int nj, int nw, int slots, int nfull, const uint8_t* __restrict__ wh) {
  // A lane's chunk: 32 weights for one token, 16 for several, so the x values of
  // every token fit in registers.  Its codes are 16 / 8 bytes (4-bit low plane;
  // W8: 32 / 16 bytes), its high bits 4 / 2 bytes (Q5) or 8 / 4 bytes (Q6).
  constexpr int kCV = TT == 1 ? 32 : 16;          // weights per lane chunk
  constexpr int kCW = FMT == kFmtW8 ? kCV : kCV / 2;   // code bytes per lane chunk
  constexpr int kWords = kCW / 4;                 // 32-bit code words per chunk
  constexpr int kHB = kCV * fmt_high_bits(FMT) / 8;    // high-bit bytes per lane chunk
  constexpr int kGroup = fmt_group(FMT);
  // (128 + q) x summed, minus (128 + zero point) sum x; W8 see the decode below
  constexpr float kBias = FMT == kFmtQ5 ? 144.f : FMT == kFmtQ6 ? 160.f : FMT == kFmtW8 ? 2304.f : 136.f;
  constexpr int kTP = TT == 1 ? 1 : TT == 2 ? 2 : 4;   // tokens padded to a power of two
  static_assert(RB * kTP <= 32, "one butterfly reduces at most 32 partials");
  extern __shared__ __align__(128) uint8_t smem[];
  pdl_launch_dependents();
  const int64_t r0 = (int64_t)blockIdx.x * N / gridDim.x;
  const int64_t r1 = (int64_t)(blockIdx.x + 1) * N / gridDim.x;
  // The planes are stored for K_pad = K rounded up to 128 columns, and lane chunks
  // cover the columns < K.  kPad is false when K is a multiple of 128 (K_pad = K):
  // that instantiation keeps the simpler address arithmetic, which measured a few
  // percent faster.
  const int64_t Kp = kPad ? ((K + 127) & ~(int64_t)127) : K;
  const int64_t row_bytes = fmt_code_row(FMT, Kp), sc_row_bytes = fmt_scale_row(FMT, Kp);
  const int64_t high_row_bytes = fmt_high_row(FMT, Kp);
  const int64_t nchunk = kPad ? (K + kCV - 1) / kCV : K / kCV;
  const int64_t plane_bytes = N * sc_row_bytes;
  const uint8_t* sc_plane = reinterpret_cast<const uint8_t*>(scales);
  if (threadIdx.x == 0) {
    // While the previous kernel finishes, start the head of this CTA's rows on their way
    // into L2: the first kPrefetchCapBytes of its codes, and the 16-byte-aligned interior
    // of those rows' scale run (never past it), 32 KB per prefetch.
    const uint8_t* cb = wq + r0 * row_bytes;
    int64_t len = (r1 - r0) * row_bytes;
    if (len > kPrefetchCapBytes) len = kPrefetchCapBytes;
    for (int64_t off = 0; off < len; off += 32768)
      bulk_prefetch_l2(cb + off, (uint32_t)(len - off < 32768 ? len - off : 32768));
    const int64_t pf_end = r0 + (len + row_bytes - 1) / row_bytes;   // <= r1
    const int64_t a0 = (r0 * sc_row_bytes + 15) & ~(int64_t)15, a1 = (pf_end * sc_row_bytes) & ~(int64_t)15;
    for (int64_t off = a0; off < a1; off += 32768)
      bulk_prefetch_l2(sc_plane + off, (uint32_t)(a1 - off < 32768 ? a1 - off : 32768));
  }
  pdl_wait_previous();  // before any global-memory read that must see the previous kernel's writes
  const StreamLayout L = stream_layout(K, TT, RB, rows_cap, nj, slots, nfull, FMT);
  float* part = reinterpret_cast<float*>(smem + L.part_off);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t xbar = sbase + L.bar_off;
  const uint32_t full0 = xbar + 8, empty0 = full0 + 8u * nfull;
  __shared__ int abort_word;
  volatile int* abort_flag = &abort_word;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nb = (int)((r1 - r0 + RB - 1) / RB);
  const int64_t last_rows = (r1 - r0) - (int64_t)(nb - 1) * RB;   // rows of the last block

  // Barrier setup and the first copies are issued before the CTA-wide barrier,
  // so the loads start while the other warps are still being set up.
  const int first = nb < slots ? nb : slots;
  if (threadIdx.x == 0) {
    mbar_init(xbar, 1);
    for (int f = 0; f < nfull; ++f) mbar_init(full0 + 8u * f, 1);
    for (int s = 0; s < slots; ++s) mbar_init(empty0 + 8u * s, nj);   // one arrival per work item
    abort_word = 0;
    fence_mbar_init();
    // x first (one copy per CTA: every warp reading it from global memory would hammer
    // the same few L2 lines from every SM at once), then the first blocks
    mbar_expect_tx(xbar, (uint32_t)(TT * K * 2));
    bulk_g2s(sbase + L.x_off, x, (uint32_t)(TT * K * 2), xbar);
    for (int b = 0; b < first; ++b)
      stream_issue(wq, sc_plane, plane_bytes, row_bytes, sc_row_bytes, r0 + (int64_t)b * RB,
                   b == nb - 1 ? (int)last_rows : RB, sbase + L.code_off + (uint32_t)b * L.code_stride,
                   sbase + L.sc_off + (uint32_t)b * L.sc_stride, full0 + 8u * b, wh, high_row_bytes,
                   sbase + L.high_off + (uint32_t)b * L.high_stride);
  }
  __syncthreads();

  if (warp == 0) {
    // ---- producer (whole warp runs the loop; lane 0 issues): refill freed slots
    int b = first;
    for (; b < nb; ++b) {
      const int s = b % slots;
      if (!warp_wait(empty0 + 8u * s, ((b / slots) & 1) ^ 1, abort_flag, &g_gemv_status)) break;
      if (lane == 0)
        stream_issue(wq, sc_plane, plane_bytes, row_bytes, sc_row_bytes, r0 + (int64_t)b * RB,
                     b == nb - 1 ? (int)last_rows : RB, sbase + L.code_off + (uint32_t)s * L.code_stride,
                     sbase + L.sc_off + (uint32_t)s * L.sc_stride, full0 + 8u * (b % nfull), wh,
                     high_row_bytes, sbase + L.high_off + (uint32_t)s * L.high_stride);
      __syncwarp();
    }
    if (b < nb && lane == 0) {  // aborted: let the copies already issued land before the CTA exits
      mbar_drain(xbar, 0);
      for (int d = (b - slots > 0 ? b - slots : 0); d < b; ++d)
        mbar_drain(full0 + 8u * (d % nfull), (d / nfull) & 1);
    }
    __syncwarp();
  } else if (warp - 1 < nw) {
    const int w = warp - 1;
    const int items = nb * nj;
    const uint32_t rowb = (uint32_t)row_bytes, scrb = (uint32_t)sc_row_bytes, hrowb = (uint32_t)high_row_bytes;
    // alignment slack of block 0's scale run in its slot; block b's is (d0 + b RB scrb) mod 16
    const uint32_t d0 = (uint32_t)((r0 * sc_row_bytes) & 15);
    float2 xv[TT][kCV / 2];
    float bias[TT];
    int cur_j = -1;
    // item it = w, w + nw, ...: block b = it / nj and group j = it % nj, the block's slot
    // s = b % slots, and its "landed" barrier fb = b % nfull with phase parity
    // fph = (b / nfull) & 1, all advanced incrementally
    int b = w / nj, j = w - (w / nj) * nj;
    const int db = nw / nj, dj = nw - (nw / nj) * nj;
    int s = b % slots, fb = b % nfull, fph = (b / nfull) & 1;
    bool ok = warp_wait(xbar, 0, abort_flag, &g_gemv_status);
    for (int it = w; ok && it < items; it += nw) {
      const uint32_t c = (uint32_t)j * 32u + (uint32_t)lane;     // this lane's chunk
      const bool c_ok = c < (uint32_t)nchunk;
      if (j != cur_j) {
        // this lane's x values of every token and their sums, kept in registers while the
        // group stays; positions k >= K (K a multiple of 8) read as zeros
#pragma unroll
        for (int t = 0; t < TT; ++t) {
#pragma unroll
          for (int q = 0; q < kCV / 8; ++q) {
            const bool v_ok = c_ok && (!kPad || c * (uint32_t)kCV + (uint32_t)q * 8u < (uint32_t)K);
            const uint4 v = v_ok ? ld_shared_v4(sbase + L.x_off + (uint32_t)t * (uint32_t)(K * 2) +
                                                c * (uint32_t)(kCV * 2) + (uint32_t)q * 16u)
                                 : make_uint4(0, 0, 0, 0);
            xv[t][4 * q + 0] = make_float2(bf16lo(v.x), bf16hi(v.x));
            xv[t][4 * q + 1] = make_float2(bf16lo(v.y), bf16hi(v.y));
            xv[t][4 * q + 2] = make_float2(bf16lo(v.z), bf16hi(v.z));
            xv[t][4 * q + 3] = make_float2(bf16lo(v.w), bf16hi(v.w));
          }
          float2 xs2 = xv[t][0];
#pragma unroll
          for (int q = 1; q < kCV / 2; ++q) xs2 = fadd2(xs2, xv[t][q]);
          bias[t] = -kBias * (xs2.x + xs2.y);
        }
        cur_j = j;
      }
      if (!warp_wait(full0 + 8u * fb, fph, abort_flag, &g_gemv_status)) break;
      const int nr = b == nb - 1 ? (int)last_rows : RB;
      const uint32_t crow = sbase + L.code_off + (uint32_t)s * L.code_stride + c * (uint32_t)kCW;
      const uint32_t hrow = sbase + L.high_off + (uint32_t)s * L.high_stride + c * (uint32_t)kHB;
      const uint32_t srow = sbase + L.sc_off + (uint32_t)s * L.sc_stride +
                            ((d0 + (uint32_t)b * (uint32_t)RB * scrb) & 15u) + (c * (uint32_t)kCV / (uint32_t)kGroup) * 2u;
      float acc[RB * kTP];
#pragma unroll
      for (int i = 0; i < RB * kTP; ++i) acc[i] = 0.f;
#pragma unroll
      for (int i = 0; i < RB; ++i) {
        if (i < nr && c_ok) {
          uint32_t words[kWords];
          if constexpr (kWords == 8) {
            const uint4 cw0 = ld_shared_v4(crow + (uint32_t)i * rowb), cw1 = ld_shared_v4(crow + (uint32_t)i * rowb + 16u);
            words[0] = cw0.x; words[1] = cw0.y; words[2] = cw0.z; words[3] = cw0.w;
            words[4] = cw1.x; words[5] = cw1.y; words[6] = cw1.z; words[7] = cw1.w;
          } else if constexpr (kWords == 4) {
            const uint4 cw = ld_shared_v4(crow + (uint32_t)i * rowb);
            words[0] = cw.x; words[1] = cw.y; words[2] = cw.z; words[3] = cw.w;
          } else {
            const uint2 cw = ld_shared_v2(crow + (uint32_t)i * rowb);
            words[0] = cw.x; words[1] = cw.y;
          }
          // Q5 / Q6: this lane's high bits of row i (in k order from bit 0)
          uint32_t hb[kHB >= 8 ? 2 : 1] = {};
          if constexpr (kHB > 0) {
            const uint32_t ha = hrow + (uint32_t)i * hrowb;
            if constexpr (kHB == 8) {
              const uint2 h = ld_shared_v2(ha);
              hb[0] = h.x;
              hb[kHB >= 8 ? 1 : 0] = h.y;
            } else if constexpr (kHB == 4) {
              hb[0] = ld_shared_u32(ha);
            } else {
              hb[0] = ld_shared_u16(ha);
            }
          }
          const float sc = fp16_bits_to_float(ld_shared_u16(srow + (uint32_t)i * scrb));
          float2 p2[TT];
          float2 ph[FMT == kFmtW8 ? TT : 1];   // W8: partials of the high nibbles
#pragma unroll
          for (int t = 0; t < TT; ++t) p2[t] = make_float2(0.f, 0.f);
#pragma unroll
          for (int t = 0; t < (FMT == kFmtW8 ? TT : 1); ++t) ph[t] = make_float2(0.f, 0.f);
#pragma unroll
          for (int wi = 0; wi < kWords; ++wi) {
            if constexpr (FMT == kFmtW8) {
              // 4 signed codes: code = lo + 16 (hs - 8) with lo, hs in 0..15, so
              // sum code x = sum (128 + lo) x + 16 sum (128 + hs) x - 2304 sum x
              const uint32_t lo = words[wi] & 0x0F0F0F0Fu;
              const uint32_t hs = ((words[wi] >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u;
              const float2 l01 = make_float2(f128_plus_byte<0>(lo), f128_plus_byte<1>(lo));
              const float2 l23 = make_float2(f128_plus_byte<2>(lo), f128_plus_byte<3>(lo));
              const float2 h01 = make_float2(f128_plus_byte<0>(hs), f128_plus_byte<1>(hs));
              const float2 h23 = make_float2(f128_plus_byte<2>(hs), f128_plus_byte<3>(hs));
#pragma unroll
              for (int t = 0; t < TT; ++t) {
                p2[t] = ffma2(l01, xv[t][2 * wi + 0], p2[t]);
                p2[t] = ffma2(l23, xv[t][2 * wi + 1], p2[t]);
                ph[t] = ffma2(h01, xv[t][2 * wi + 0], ph[t]);
                ph[t] = ffma2(h23, xv[t][2 * wi + 1], ph[t]);
              }
            } else {
              uint32_t lo = words[wi] & 0x0F0F0F0Fu, hi = (words[wi] >> 4) & 0x0F0F0F0Fu;
              if constexpr (FMT == kFmtQ5) {
                // the word's 8 high bits: even weights' bits to bit 4 of bytes 0..3 of lo,
                // odd weights' to hi (one multiply spreads four bits without carries)
                const uint32_t bits = (hb[0] >> (8 * wi)) & 0xFFu;
                lo |= ((bits & 0x55u) * 0x00410410u) & 0x10101010u;
                hi |= ((bits & 0xAAu) * 0x00208208u) & 0x10101010u;
              } else if constexpr (FMT == kFmtQ6) {
                // the word's 16 high bits (2 per weight): even weights' fields to bits 4..5
                // of bytes 0..3 of lo, odd weights' to hi
                const uint32_t h16 = (hb[wi >> 1] >> (16 * (wi & 1))) & 0xFFFFu;
                lo |= spread_nibbles_to_bytes(h16 & 0x3333u) << 4;
                hi |= spread_nibbles_to_bytes((h16 >> 2) & 0x3333u) << 4;
              }
              const float2 f0 = make_float2(f128_plus_byte<0>(lo), f128_plus_byte<0>(hi));
              const float2 f1 = make_float2(f128_plus_byte<1>(lo), f128_plus_byte<1>(hi));
              const float2 f2 = make_float2(f128_plus_byte<2>(lo), f128_plus_byte<2>(hi));
              const float2 f3 = make_float2(f128_plus_byte<3>(lo), f128_plus_byte<3>(hi));
#pragma unroll
              for (int t = 0; t < TT; ++t) {
                p2[t] = ffma2(f0, xv[t][4 * wi + 0], p2[t]);
                p2[t] = ffma2(f1, xv[t][4 * wi + 1], p2[t]);
                p2[t] = ffma2(f2, xv[t][4 * wi + 2], p2[t]);
                p2[t] = ffma2(f3, xv[t][4 * wi + 3], p2[t]);
              }
            }
          }
          if constexpr (FMT == kFmtW8) {
#pragma unroll
            for (int t = 0; t < TT; ++t) p2[t].x += 16.f * (ph[t].x + ph[t].y);
          }
#pragma unroll
          for (int t = 0; t < TT; ++t) acc[i * kTP + t] = sc * ((p2[t].x + p2[t].y) + bias[t]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8u * s);
      int idx = 0;
      const float v = reduce_rows<RB * kTP>(acc, lane, &idx);
      const int row = idx / kTP, t = idx - (idx / kTP) * kTP;
      if ((lane & (32 / (RB * kTP) - 1)) == 0 && row < nr && t < TT)
        part[((b * RB + row) * nj + j) * TT + t] = v;
      // next item
      int nb_step = db;
      j += dj;
      if (j >= nj) {
        j -= nj;
        ++nb_step;
      }
      b += nb_step;
      s += nb_step;
      while (s >= slots) s -= slots;
      fb += nb_step;
      while (fb >= nfull) {
        fb -= nfull;
        fph ^= 1;
      }
    }
  }

  // ---- final: y[t, row] = bf16(sum over column groups, in order).  Every warp
  // reaches this barrier converged (all role loops are warp-uniform).
  __syncthreads();
  if (*abort_flag) return;
  for (int64_t r = threadIdx.x; r < (r1 - r0) * TT; r += kStreamThreads) {
    const int64_t row = r / TT, t = r - (r / TT) * TT;
    float v = 0.f;
    for (int jj = 0; jj < nj; ++jj) v += part[(row * nj + jj) * TT + t];
    y[t * N + r0 + row] = float_to_bf16_bits(v);
  }
}

}  // namespace

size_t gemv_workspace_bytes(int64_t, int64_t, int64_t) { return 0; }

int gemv_launch_count(int64_t N, int64_t K, int64_t T) {
  return gemv_stream_ok(N, K, T) ? 1 : (int)((T + 3) / 4);
}

struct StreamPlan {
  int64_t grid, rows_cap;
  int tt, rb, nj, nw, slots, nfull, fmt;
  uint32_t bytes;
};

// Tokens 1..4.  Rows per block: 8 if their code rows fit 32 KB, else 4 if they
// fit 40 KB, else 2 (with several tokens, 8-row blocks also halve how often a
// warp reloads x per row decoded: 6144 x 5120 T = 3 takes 13.4 us with them,
// 15.7 us with 4-row blocks); the ring gets as many slots as the shared-memory
// budget holds (at least 2).
static bool stream_plan(int64_t N, int64_t K, int64_t T, int nsm, StreamPlan* p, int fmt = kFmtQ4) {
  if (N < 1 || K < 8 || T < 1 || T > 4) return false;
  p->fmt = fmt;
  p->tt = (int)T;
  const int64_t chunk_w = T == 1 ? 32 : 16;   // weights per lane chunk
  const int64_t nchunk = (K + chunk_w - 1) / chunk_w;
  const int64_t Kp = (K + 127) / 128 * 128;
  p->nj = (int)((nchunk + 31) / 32);
  // consumer warps: a multiple of the group count (no x reloads) unless that idles
  // more than 3 of the 15, then all 15 (a warp reloads x when its group changes)
  const int whole = p->nj <= kStreamConsumers ? (kStreamConsumers / p->nj) * p->nj : 0;
  p->nw = whole >= kStreamConsumers - 3 ? whole : kStreamConsumers;
  const int64_t code_row = fmt_code_row(fmt, Kp);
  p->rb = 8 * code_row <= 32768 ? 8 : 4 * code_row <= 40960 ? 4 : 2;
  p->grid = (N + 3) / 4;  // at least 4 rows per CTA
  if (p->grid > nsm) p->grid = nsm;
  if (p->grid < 1) p->grid = 1;
  p->rows_cap = ((N + p->grid - 1) / p->grid + p->rb - 1) / p->rb * p->rb;
  // A consumer waiting for block b has consumed its previous block, at most `lead`
  // blocks earlier, so every block up to lead + slots before b has landed (the
  // producer refills a slot only after its block was consumed).  With
  // slots + lead "landed" barriers, block b's barrier was last used by a block
  // that has landed, so a parity wait can never match a phase two behind.
  const int lead = p->nw / p->nj + (p->nw % p->nj != 0 ? 1 : 0);
  const int64_t budget = kStreamSmemBudget;
  if (T * K * 2 > budget) return false;
  const StreamLayout L0 = stream_layout(K, p->tt, p->rb, p->rows_cap, p->nj, 0, lead, fmt);
  const int64_t per = (int64_t)L0.code_stride + L0.high_stride + L0.sc_stride + 16;
  if ((int64_t)L0.code_off + 128 > budget) return false;
  int64_t s = (budget - L0.code_off - 128) / per;
  if (s > 32) s = 32;
  if (s < 2) return false;
  p->slots = (int)s;
  p->nfull = p->slots + lead;
  p->bytes = stream_layout(K, p->tt, p->rb, p->rows_cap, p->nj, p->slots, p->nfull, fmt).bytes;
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

template <int RB, int TT, bool kPad, int FMT>
static int gemv_stream_launch_cfg(const LinearArgs& a, const StreamPlan& pl) {
  static bool attr[64] = {};
  int dev = 0;
  if (cuda_check(cudaGetDevice(&dev), "cudaGetDevice")) return Q4LIN_ERR_CUDA;
  if (dev >= 64 || !attr[dev]) {
    if (cuda_check(cudaFuncSetAttribute(q4_gemv_stream_kernel<RB, TT, kPad, FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)kStreamSmemBudget),
                   "gemv: cudaFuncSetAttribute"))
      return Q4LIN_ERR_CUDA;
    if (dev < 64) attr[dev] = true;
  }
  // programmatic dependent launch: the kernel waits for its predecessor before touching memory
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)pl.grid, 1, 1);
  cfg.blockDim = dim3(kStreamThreads, 1, 1);
  cfg.dynamicSmemBytes = pl.bytes;
  cfg.stream = a.stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cuda_check(cudaLaunchKernelEx(&cfg, q4_gemv_stream_kernel<RB, TT, kPad, FMT>, a.wq, a.scales, a.x, a.y, a.N, a.K,
                                       pl.rows_cap, pl.nj, pl.nw, pl.slots, pl.nfull, a.wh),
                    "gemv: streaming kernel launch");
}

template <int TT, bool kPad, int FMT>
static int gemv_stream_launch_pad(const LinearArgs& a, const StreamPlan& pl) {
  if (pl.rb == 8) return gemv_stream_launch_cfg<8, TT, kPad, FMT>(a, pl);
  if (pl.rb == 4) return gemv_stream_launch_cfg<4, TT, kPad, FMT>(a, pl);
  return gemv_stream_launch_cfg<2, TT, kPad, FMT>(a, pl);
}

// Q4 has an instantiation for K a multiple of 128 and one for padded K; the
// sibling formats use the padded form, which is correct for every K.
template <int TT>
static int gemv_stream_launch_tt(const LinearArgs& a, const StreamPlan& pl) {
  switch (pl.fmt) {
    case kFmtQ5: return gemv_stream_launch_pad<TT, true, kFmtQ5>(a, pl);
    case kFmtQ6: return gemv_stream_launch_pad<TT, true, kFmtQ6>(a, pl);
    case kFmtW8: return gemv_stream_launch_pad<TT, true, kFmtW8>(a, pl);
    default:
      return a.K % 128 != 0 ? gemv_stream_launch_pad<TT, true, kFmtQ4>(a, pl)
                            : gemv_stream_launch_pad<TT, false, kFmtQ4>(a, pl);
  }
}

static int gemv_stream_launch(const LinearArgs& a) {
  StreamPlan pl;
  if (!stream_plan(a.N, a.K, a.T, device_sms(), &pl, a.fmt)) return Q4LIN_ERR_INVALID_ARG;
  switch (pl.tt) {
    case 1: return gemv_stream_launch_tt<1>(a, pl);
    case 2: return gemv_stream_launch_tt<2>(a, pl);
    case 3: return gemv_stream_launch_tt<3>(a, pl);
    default: return gemv_stream_launch_tt<4>(a, pl);
  }
}

bool gemv_stream_ok(int64_t N, int64_t K, int64_t T, int fmt) {
  StreamPlan pl;
  return stream_plan(N, K, T, device_sms(), &pl, fmt);   // the plan the launch will make
}

int gemv_launch_fmt(const LinearArgs& a) {
  if (!gemv_stream_ok(a.N, a.K, a.T, a.fmt)) {
    set_error_detail("gemv: no streaming plan for this format and shape (1..4 tokens only)");
    return Q4LIN_ERR_UNSUPPORTED_SHAPE;
  }
  return gemv_stream_launch(a);
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
