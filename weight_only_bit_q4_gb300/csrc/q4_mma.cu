// Streaming warp-MMA route of the Q4_G64_FP16 linear layer (and its sibling formats), for a few tokens.
//
// Below a few dozen tokens the layer is a stream of packed weights: every weight
// is read once from HBM and used T times.  The tile route's per-group pipeline
// (decode team -> tensor memory -> single MMA issuer -> tensor-memory readback)
// costs several instructions per weight there and leaves most of HBM idle, and
// CUDA-core FMAs cost T / 2 instructions per weight.  This route keeps the whole
// inner loop in registers: one AND per weight pair turns the packed nibbles
// straight into fp16 operands, and the warp-level tensor-core MMA
// (mma.sync m16n8k16, fp16 x fp16 -> fp32) does the multiply and the reduction
// along K, so a weight costs about one instruction whatever the token count.
//
// Exactness.  A nibble pair masked out of a code word, w & 0x000F000F, is read as
// two fp16 bit patterns q and q': fp16 subnormals worth q * 2^-24 exactly.  The
// odd nibbles, w & 0x00F000F0, are 16 q * 2^-24, also exact (at most 240 < 2^10),
// and meet x / 16 on the other side.  X is converted to fp16 once per call by a
// prep kernel, each 64-wide group of each token taken at the power of two 2^-e that
// puts the group's largest |x| in [2^14, 2^15) (bf16 -> fp16 is then exact down to
// 2^-38 of that largest value).  Every product q * x-hat is exact in FP32, so the MMA
// of one group gives D = 2^-24 sum q x-hat, and
//     sum_k (q - 8) x  =  2^(24 + e) D - 8 2^e sum_k x-hat  =  F D + Z,
// with F and Z written by the prep kernel per group and token.  The group scale
// multiplies that FP32 partial before the one bf16 rounding.  No product is rounded.
//
// Operand layout.  In one m16n8k16 MMA a thread (g = lane / 4, c = lane % 4) holds
// A elements of rows g and g + 8 at K slots 2c, 2c + 1, 2c + 8, 2c + 9, and B
// elements of token g at the same K slots.  The K order inside an MMA is free as
// long as A and B agree, so thread c takes the 8 code bytes [8c, 8c + 8) of a
// 64-wide group (k = 16c .. 16c + 15) from its two rows and uses the masked
// nibble pairs as they come: (k, k + 4) pairs of one 32-bit code word.  The prep
// kernel writes X in exactly that order ("B fragments"), so a thread loads its
// B operands with two 16-byte shared-memory loads per group and token tile.
// Rows: mma row g is band row 16 m + 2g and row g + 8 is 16 m + 2g + 1, which makes
// the 8-byte code loads of a warp conflict-free in the 128-byte-swizzled stage.
//
// Work split.  One persistent CTA per SM owns a contiguous range of rows
// (balanced to one row), cut into bands of at most 240 rows.  For each band the
// producer warp streams K in chunks: KS code sub-boxes of 256 K values x band
// rows (TMA, 128-byte swizzle), the chunk's B fragments and zero-point terms
// (bulk copies from the prep kernel's buffer), into a ring of stages; the band's
// scale run (contiguous rows of the scale plane) goes into one of two buffers.
// Consumer warp (m, s) handles m-tile m (16 rows) of sub-box s of every chunk and
// keeps its FP32 partial sums in registers across the band; at the end of the
// band the KS partials of each row are summed in a fixed order through shared
// memory (deterministic) and the band's outputs are rounded to bf16 and stored.
//
// Forms.  Q5G64 / Q6G64 stage their high-bit plane beside the code sub-boxes and join
// the high bits to the nibble operands; W8G32 offsets its signed bytes to u = code + 128
// (two MMAs per 32-wide group).  Without a workspace (the fused operations, up to 8
// tokens) the kernel converts X itself into whole-K fragments in shared memory and no
// prep kernel runs; LinearAdd adds its residual in the band epilogue and LinearSwiGLU
// pairs each band of gate rows with the band of up rows it multiplies.
//
// Every mbarrier wait is bounded (kSpinLimit): on expiry the kernel records
// Q4LIN_ERR_TIMEOUT, every role skips its remaining work but still passes the
// band barriers, and the producer drains the copies it issued before exiting.
#include "q4_internal.h"
#include "q4_sm100.cuh"

namespace q4 {

namespace {

__device__ int g_mma_status = 0;

constexpr int kMmaWarps = 16;  // warp 0: producer; warps 1..15: consumers
constexpr int kMmaThreads = 32 * kMmaWarps;
constexpr int kMaxConsumers = kMmaWarps - 1;
constexpr int kMaxBand = 240;  // rows per band: TMA box height <= 256, 15 m-tiles
constexpr uint32_t kMmaSmem = 232448;  // dynamic shared memory per CTA (incl. 1024-byte alignment slack)
constexpr int kRedBar = 1;             // named barrier of the consumer warps
constexpr int kConvBar = 2;            // fused form: named barrier of the warps converting X
// Early launch order: L2 prefetch of one CTA's code rows before the dependency wait, at
// most (the whole share of a 6144-row layer on 152 SMs: 103 KB at K = 5120).
constexpr int64_t kMmaPrefetchCap = 128 * 1024;

struct MmaParams {
  const uint8_t* wq;       // packed codes [N, Kp/2]
  const uint16_t* scales;  // fp16 bits [N, Kp/64]
  const uint8_t* xf;       // B fragments [galloc][NT][2][lanes][16 bytes] (prep kernel's buffer)
  const float* zs;         // per (group, token tile, c): (Z[t], Z[t + 1], F[t], F[t + 1]), t = 2c
  const uint16_t* x;       // fused form: bf16 X [T, K], converted in the kernel
  uint16_t* y;             // bf16 [T, N]
  const uint16_t* r;       // LinearAdd: bf16 residual [T, N], added before the bf16 store (may be y)
  int64_t N, K, Kp, T;
  int t0;       // first token of this pass
  int tp;       // tokens of this pass (<= 8 NT)
  int nk;       // groups holding columns < K
  int br;       // band rows (TMA box height, a multiple of 8)
  int ks;       // code sub-boxes per chunk
  int mt;       // m-tiles per band
  int nchunks;  // chunks per band
  int stages;
  int lanes;    // B-fragment lanes stored per (group, token tile)
  int early;    // launch order: 1 early (launched before the prep kernel's wait), 0 late
  int galloc;   // groups of the B-fragment buffer
  uint32_t hi_off;                        // Q5 / Q6: the high-bit sub-boxes inside a stage
  uint32_t stage_bytes, xf_off, zs_off;  // stage size; B fragments and zero points (inside a stage, or
                                         // the fused form's whole-K buffers)
  uint32_t scl_off, scl_bytes;           // the two band scale buffers
  uint32_t red_off, gate_off, bar_off;
};

// Shared-memory layout of one launch.  Stages hold a chunk's code sub-boxes and (two-kernel
// form) its B fragments and zero-point terms; the fused form keeps the whole K extent of
// both, written by the kernel itself, after the stages (fx_off, fz_off).
struct MmaLayout {
  uint32_t code_bytes, hi_bytes, xf_bytes, zs_bytes, stage_bytes, scl_bytes, red_bytes;
  uint32_t fx_off, fx_bytes, fz_off, fz_bytes;
  uint32_t scl_off, red_off, gate_off, bar_off, total;
};

// fbytes: B-fragment bytes per lane per group and token tile (Q4: 32, four MMAs; W8: 16, two)
__host__ __device__ inline MmaLayout mma_layout(int nt, int br, int ks, int mt, int stages, int lanes, int64_t Kp,
                                                int fbytes = 32, int64_t srb = 0, bool fused = false,
                                                int galloc = 0, bool swiglu = false, int hb = 0) {
  MmaLayout L;
  L.code_bytes = (uint32_t)(ks * br * 128);  // ks sub-boxes of br rows x 128 bytes (128-byte swizzle)
  L.hi_bytes = (uint32_t)(ks * br * 32 * hb);   // Q5 / Q6: ks sub-boxes of br rows x 32 hb bytes
  L.xf_bytes = fused ? 0u : (uint32_t)(4 * ks * nt * lanes * fbytes);
  L.zs_bytes = fused ? 0u : (uint32_t)(4 * ks * nt * 64);
  L.stage_bytes = (L.code_bytes + L.hi_bytes + L.xf_bytes + L.zs_bytes + 1023) / 1024 * 1024;
  L.fx_off = (uint32_t)stages * L.stage_bytes;
  L.fx_bytes = fused ? (uint32_t)galloc * (uint32_t)(nt * lanes * fbytes) : 0u;
  L.fz_off = L.fx_off + L.fx_bytes;
  L.fz_bytes = fused ? (uint32_t)galloc * (uint32_t)(nt * 64) : 0u;
  // a band's scale run: br rows of Kp / 64 scales, plus up to 15 bytes of alignment slack
  // on either side
  if (srb == 0) srb = Kp / 32;  // bytes of a scale row (Q4: Kp / 64 scales)
  L.scl_bytes = (uint32_t)((br * srb + 32 + 15) / 16 * 16);
  L.red_bytes = (uint32_t)(ks * mt * 16 * 8 * nt * 4);
  L.scl_off = L.fz_off + L.fz_bytes;
  L.red_off = L.scl_off + 2 * L.scl_bytes;
  // LinearSwiGLU: a gate band's FP32 sums wait here for the matching up band
  L.gate_off = L.red_off + L.red_bytes;
  const uint32_t gate_bytes = swiglu ? (uint32_t)(mt * 16 * 8 * nt * 4) : 0u;
  L.bar_off = (L.gate_off + gate_bytes + 15) / 16 * 16;
  L.total = L.bar_off + (uint32_t)(2 * stages + 4) * 8 + 16;
  return L;
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// Pull global bytes into L2 (no destination, no completion): a hint that never changes
// what a later load returns.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ uint2 lds_u64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t lds_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint16_t lds_u16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ void sts_u16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

// D = A . B + C, m16n8k16, fp16 operands, fp32 accumulate.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The 16 weights k = 16c .. 16c + 15 of one row of a group (code words w0, w1) as the
// eight A operand registers of the group's four MMAs: p[2i] holds (q, q') of the
// even-position nibbles as fp16 subnormal patterns (q * 2^-24), p[2i + 1] the
// odd-position ones at 16 q * 2^-24.  K order: p[0] = (0, 4), p[1] = (1, 5),
// p[2] = (2, 6), p[3] = (3, 7), p[4..7] the same for k + 8.
__device__ __forceinline__ void decode_q4_pairs(uint32_t w0, uint32_t w1, uint32_t (&p)[8]) {
  const uint32_t v0 = w0 >> 8, v1 = w1 >> 8;
  p[0] = w0 & 0x000F000Fu;
  p[1] = w0 & 0x00F000F0u;
  p[2] = v0 & 0x000F000Fu;
  p[3] = v0 & 0x00F000F0u;
  p[4] = w1 & 0x000F000Fu;
  p[5] = w1 & 0x00F000F0u;
  p[6] = v1 & 0x000F000Fu;
  p[7] = v1 & 0x00F000F0u;
}

// Q5G64 / Q6G64: the high bits of the same 16 weights (hw: Q5 bit j, Q6 bits 2j..2j+1 belong
// to weight k + j) joined to the nibbles of decode_q4_pairs, as 16 h (even registers) and
// 256 h (odd registers, which hold 16 q): q = nibble + 16 h stays below 64, so 16 q <= 1008
// is still an exact fp16 subnormal pattern.  For register j (weights j and j + 4, or 8 + j
// and 12 + j) the spread y = h | h << 12 (Q5) or h | h << 8 (Q6) puts the two weights' bits
// 16 positions apart.
template <int kHB>
__device__ __forceinline__ void add_high_pairs(uint32_t hw, uint32_t (&p)[8]) {
  constexpr uint32_t kMask = kHB == 1 ? 0x00010001u : 0x00030003u;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const uint32_t h = kHB == 1 ? (hw >> (8 * half)) & 0xFFu : (hw >> (16 * half)) & 0xFFFFu;
    const uint32_t y = kHB == 1 ? h | (h << 12) : h | (h << 8);
#pragma unroll
    for (int j = 0; j < 4; ++j) p[4 * half + j] |= ((y >> (kHB * j)) & kMask) << ((j & 1) ? 8 : 4);
  }
}

// FMT: 0 Q4G64 (64-wide groups, four MMAs per group), 1 Q5G64 / 2 Q6G64 (the same, with 1 or
// 2 high bits per weight from the high-bit plane), 3 W8G32 (32-wide groups of signed bytes, two
// MMAs per group; the scale plane has Kp / 32 scales per row).
// W8G32: the 8 signed codes k = 8c .. 8c + 7 of one row of a 32-wide group (words w0, w1) as
// the four A registers of the group's two MMAs: each code offset to u = code + 128 (the sign
// bit flipped) and read as the fp16 subnormal u * 2^-24 (u <= 255).  K order: p[0] = (0, 2),
// p[1] = (1, 3), p[2] = (4, 6), p[3] = (5, 7).
__device__ __forceinline__ void decode_w8_pairs(uint32_t w0, uint32_t w1, uint32_t (&p)[8]) {
  const uint32_t u0 = w0 ^ 0x80808080u, u1 = w1 ^ 0x80808080u;
  p[0] = u0 & 0x00FF00FFu;
  p[1] = (u0 >> 8) & 0x00FF00FFu;
  p[2] = u1 & 0x00FF00FFu;
  p[3] = (u1 >> 8) & 0x00FF00FFu;
  p[4] = p[5] = p[6] = p[7] = 0u;
}

// ----------------------------------------------------------------- operand pass
// One thread per (token slot t of the pass, group G, c): the values of token t in group G
// that thread c of an MMA feeds -- k = 64 G + 16 c .. + 15 (Q4) or 32 G + 8 c .. + 7 (W8)
// -- become its fp16x2 B registers, in the order the decode produces A.  The four c of a
// (t, G) are adjacent lanes: they take the group's largest |x| (compared as bf16 magnitude
// bits) and the power of two 2^-e that puts it in [2^14, 2^15), so every value of the group
// down to 2^-38 of that largest one converts to fp16 exactly, and the group's terms
//     Z = -zero * 2^e * sum x-hat,   F = 2^(24 + e)
// make sum_k (q_k - zero) x_k = F D + Z for the MMA result D = 2^-24 sum q x-hat (zero = 8 for
// Q4, 16 for Q5, 32 for Q6, 128 for W8's offset codes).  No pass over a whole token is needed, so the threads of
// any number of CTAs share the work.  Slots past the pass's tokens write zeros.  Groups holding
// Inf or NaN keep e = 0 so those values propagate.
constexpr int kPrepThreads = 256;

// Operand unit u = (token slot t, group G, c) of a pass whose tokens start at x, in two
// phases so that a thread can keep the loads of several units in flight: the load of its
// X values, then the conversion.  The conversion is called by all 32 lanes of a warp
// together (the four c of a (t, G) are adjacent lanes and exchange their maxima and sums
// by shuffles); act is false for the lanes past the last unit.  xf and zs are the
// B-fragment and zero-point buffers, laid out as the streaming kernel reads them (global
// memory for the prep kernel, shared memory for the fused form).
template <int NT, int FMT>
__device__ __forceinline__ void mma_operand_load(const uint16_t* __restrict__ x, int64_t K, int tp, int galloc,
                                                 int64_t u, bool act, uint4 (&q)[2]) {
  constexpr int kVals = FMT == 3 ? 8 : 16;  // values of one (group, c) unit
  const int c = (int)(u & 3);
  const int64_t tg = u >> 2;
  const int G = (int)(tg % galloc), t = (int)(tg / galloc);
  const bool live = act && t < tp;
  const int64_t k0 = (int64_t)G * (4 * kVals) + kVals * c;
  const uint16_t* xr = x + (int64_t)(live ? t : 0) * K;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    // K is a multiple of 8: each run of 8 columns is either wholly inside or wholly past K
    const bool in = h < kVals / 8 && live && k0 + 8 * h < K;
    q[h] = in ? __ldg(reinterpret_cast<const uint4*>(xr + k0 + 8 * h)) : make_uint4(0u, 0u, 0u, 0u);
  }
}

template <int NT, int FMT>
__device__ __forceinline__ void mma_operand_convert(int tp, int galloc, int lanes, int64_t u, bool act,
                                                    const uint4 (&q)[2], uint8_t* xf, float* zs) {
  constexpr bool kW8 = FMT == 3;
  constexpr int kVals = kW8 ? 8 : 16;  // values of one (group, c) unit
  const int c = (int)(u & 3);
  const int64_t tg = u >> 2;
  const int G = (int)(tg % galloc), t = (int)(tg / galloc);
  const bool live = act && t < tp;
  float v[16];
  uint32_t m2 = 0;
#pragma unroll
  for (int h = 0; h < kVals / 8; ++h) {
    m2 = __vmaxu2(m2, __vmaxu2(__vmaxu2(q[h].x & 0x7FFF7FFFu, q[h].y & 0x7FFF7FFFu),
                               __vmaxu2(q[h].z & 0x7FFF7FFFu, q[h].w & 0x7FFF7FFFu)));
    v[8 * h + 0] = bf16lo(q[h].x); v[8 * h + 1] = bf16hi(q[h].x);
    v[8 * h + 2] = bf16lo(q[h].y); v[8 * h + 3] = bf16hi(q[h].y);
    v[8 * h + 4] = bf16lo(q[h].z); v[8 * h + 5] = bf16hi(q[h].z);
    v[8 * h + 6] = bf16lo(q[h].w); v[8 * h + 7] = bf16hi(q[h].w);
  }
  uint32_t mx = max(m2 & 0xFFFFu, m2 >> 16);
  mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
  mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
  const int E = (int)(mx >> 7);  // bf16 biased exponent of the group's largest |x|
  const int e = (mx == 0 || E == 255) ? 0 : min(max(E - 141, -100), 100);
  const float s1 = exp2i(-e), s16 = exp2i(-e - 4);
  // x-hat = fp16(x 2^-e) (exact in fp16's normal range); the zero-point term sums the same values
  float sum = 0.f;
#pragma unroll
  for (int i = 0; i < kVals; ++i) sum += __half2float(__float2half_rn(v[i] * s1));
  sum += __shfl_xor_sync(0xffffffffu, sum, 1);
  sum += __shfl_xor_sync(0xffffffffu, sum, 2);
  auto pk = [&](int i0, int i1, float sc) -> uint32_t {
    return (uint32_t)__half_as_ushort(__float2half_rn(v[i0] * sc)) |
           ((uint32_t)__half_as_ushort(__float2half_rn(v[i1] * sc)) << 16);
  };
  const int n = t / 8, tl = t % 8;
  if (act && tl * 4 < lanes) {  // this token's B lanes exist in the buffer
    const int L = tl * 4 + c;
    if constexpr (kW8) {
      // registers per MMA kk: (x[k0 + 4kk], x[+2]) then (x[+1], x[+3])
      uint4* dst = reinterpret_cast<uint4*>(xf + (size_t)(G * NT + n) * lanes * 16);
      dst[L] = make_uint4(pk(0, 2, s1), pk(1, 3, s1), pk(4, 6, s1), pk(5, 7, s1));
    } else {
      // registers per MMA kk: (x[k0 + 2kk'], x[+4]) then (x[+1] / 16, x[+5] / 16), kk' = 0, 1, 4, 5
      uint4* dst = reinterpret_cast<uint4*>(xf + ((size_t)(G * NT + n) * 2) * lanes * 16);
      dst[L] = make_uint4(pk(0, 4, s1), pk(1, 5, s16), pk(2, 6, s1), pk(3, 7, s16));
      dst[lanes + L] = make_uint4(pk(8, 12, s1), pk(9, 13, s16), pk(10, 14, s1), pk(11, 15, s16));
    }
  }
  if (act && c == 0) {
    // (Z[t], Z[t + 1], F[t], F[t + 1]) of MMA thread c' = tl / 2 of this group and token tile
    float* zq = zs + ((size_t)(G * NT + n) * 4 + tl / 2) * 4;
    constexpr float kZero = FMT == 3 ? 128.f : FMT == 2 ? 32.f : FMT == 1 ? 16.f : 8.f;
    zq[tl & 1] = live ? -kZero * exp2i(e) * sum : 0.f;
    zq[2 + (tl & 1)] = live ? exp2i(24 + e) : 0.f;
  }
}

template <int NT, int FMT>
__global__ void __launch_bounds__(kPrepThreads)
q4_mma_prep_kernel(const uint16_t* __restrict__ x, uint8_t* __restrict__ xf, float* __restrict__ zs,
                   int64_t K, int tp, int galloc, int lanes, int early) {
  // Wait for the previous kernel (it may write x, or still read these buffers).  The
  // streaming kernel launches after that wait (late order: it copies weight rows as soon
  // as it starts) or before it (early order: it only prefetches them into L2 until its
  // own wait).
  if (early) pdl_launch_dependents();
  pdl_wait_previous();
  if (!early) pdl_launch_dependents();
  const int64_t units = (int64_t)8 * NT * galloc * 4;   // a multiple of 32: whole warps take part
  for (int64_t u = (int64_t)blockIdx.x * kPrepThreads + threadIdx.x; u - (threadIdx.x & 31) < units;
       u += (int64_t)gridDim.x * kPrepThreads)
  {
    uint4 q[2];
    mma_operand_load<NT, FMT>(x, K, tp, galloc, u, u < units, q);
    mma_operand_convert<NT, FMT>(tp, galloc, lanes, u, u < units, q, xf, zs);
  }
}

// ----------------------------------------------------------------- streaming kernel
// kFuse (one token tile, the B fragments of the whole K extent fit in shared memory): the
// consumer warps run the operand pass themselves, every CTA for all groups, into shared
// memory, while the producer streams the weight rows -- one launch, no workspace, and no
// wait for a second kernel's completion.  Always the early launch order.
template <int NT, int FMT, bool kFuse = false, bool kSwi = false>
__global__ void __launch_bounds__(kMmaThreads, 1)
q4_mma_kernel(const __grid_constant__ CUtensorMap tm_codes, const __grid_constant__ CUtensorMap tm_high,
              const MmaParams p) {
  static_assert(!kFuse || NT == 1, "the fused operand pass covers one token tile");
  static_assert(!kSwi || (kFuse && FMT == 0), "LinearSwiGLU: the one-launch Q4 form");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  pdl_launch_dependents();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t r0 = (int64_t)blockIdx.x * p.N / gridDim.x;
  const int64_t r1 = (int64_t)(blockIdx.x + 1) * p.N / gridDim.x;
  const int BR = p.br, KS = p.ks, NS = p.stages, NCH = p.nchunks;
  const int WC = KS * p.mt;
  // Bands of BR rows over the CTA's rows [r0, r1); LinearSwiGLU alternates a band of gate
  // rows [r0, r1) and the band of up rows F + [r0, r1) that pairs with it.
  const int nb1 = (int)((r1 - r0 + BR - 1) / BR);
  const int nbands = kSwi ? 2 * nb1 : nb1;
  auto band_row = [&](int b) -> int64_t {  // first weight row of band b
    return kSwi ? (b & 1 ? p.N : 0) + r0 + (int64_t)(b >> 1) * BR : r0 + (int64_t)b * BR;
  };
  auto band_rows = [&](int b) -> int {
    const int64_t o = r0 + (int64_t)(kSwi ? b >> 1 : b) * BR;
    return (int)((o + BR < r1 ? o + BR : r1) - o);
  };
  constexpr bool kW8 = FMT == 3;
  constexpr int kHB = (FMT == 1 || FMT == 2) ? FMT : 0;  // Q5 / Q6: high bits per weight
  constexpr uint32_t kHRow = 32u * kHB;                // high-plane bytes of one sub-box row (256 weights)
  constexpr int FB = kW8 ? 16 : 32;                   // B-fragment bytes per lane per group and token tile
  const int64_t srb = kW8 ? p.Kp / 16 : p.Kp / 32;    // bytes of one row of the scale plane
  const uint32_t bars = sbase + p.bar_off;
  auto full = [&](int s) { return bars + 8u * (uint32_t)s; };
  auto empty = [&](int s) { return bars + 8u * (uint32_t)(NS + s); };
  const uint32_t sfull0 = bars + 8u * (uint32_t)(2 * NS), sempty0 = sfull0 + 16u;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + p.bar_off + (2 * NS + 4) * 8);
  auto stage = [&](int s) { return sbase + (uint32_t)s * p.stage_bytes; };
  auto scl_buf = [&](int b) { return sbase + p.scl_off + (uint32_t)(b & 1) * p.scl_bytes; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), (uint32_t)WC);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(sfull0 + 8u * b, 1);
      mbar_init(sempty0 + 8u * b, (uint32_t)WC);
    }
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_codes);
    if constexpr (kHB > 0) prefetch_tmap(&tm_high);
  }
  __syncthreads();
  // Launch order (programmatic dependent launch) of the two-kernel form, one of two per
  // call (p.early; the fused form has no prep kernel and always takes the early path):
  //  - late: the prep kernel waits for its own predecessor before it lets this kernel
  //    launch, so every kernel before this call has completed when this one starts, and
  //    the weight planes are streamed at once, while the prep kernel works.  Only what
  //    the prep kernel writes (B fragments, zero points, exponents) waits for
  //    griddepcontrol.wait: the producer before its first fragment copy, the consumers
  //    before the first epilogue.
  //  - early: the prep kernel lets this kernel launch at once, so its CTAs take their SMs
  //    as the previous kernel's CTAs leave.  Until griddepcontrol.wait returns (the prep
  //    kernel, and with it every earlier kernel, has completed) the producer only pulls
  //    the head of the CTA's weight rows into L2 -- the previous kernel may still write
  //    the planes, and an L2 prefetch never changes what a later load returns -- then
  //    streams them from there.

  const uint32_t xf_chunk = (uint32_t)(4 * KS * NT * p.lanes * FB);  // B-fragment bytes per chunk
  const uint32_t zs_chunk = (uint32_t)(4 * KS * NT * 64);
  if (warp == 0) {
    // ------------------------------------------------------------- producer (lane 0 issues)
    if (lane == 0) {
      const uint8_t* sc_plane = reinterpret_cast<const uint8_t*>(p.scales);
      const int64_t plane_bytes = (kSwi ? 2 * p.N : p.N) * srb;
      bool ok = true, waited = false;
      if (kFuse || p.early) {
        // the first kMmaPrefetchCap bytes of the CTA's code rows (contiguous) and the
        // 16-byte-aligned interior of those rows' scale run, 32 KB per prefetch
        // (LinearSwiGLU: half of it for the gate rows, half for the up rows)
        const int64_t code_row = kW8 ? p.Kp : p.Kp / 2;
        for (int sg = 0; sg < (kSwi ? 2 : 1); ++sg) {
          const int64_t q0 = r0 + (sg ? p.N : 0), q1 = r1 + (sg ? p.N : 0);
          const uint8_t* cb = p.wq + q0 * code_row;
          int64_t len = (q1 - q0) * code_row;
          const int64_t cap = kSwi ? kMmaPrefetchCap / 2 : kMmaPrefetchCap;
          if (len > cap) len = cap;
          for (int64_t off = 0; off < len; off += 32768)
            bulk_prefetch_l2(cb + off, (uint32_t)(len - off < 32768 ? len - off : 32768));
          const int64_t pf_end = q0 + (len + code_row - 1) / code_row;  // <= q1
          const int64_t a0 = (q0 * srb + 15) & ~(int64_t)15, a1 = (pf_end * srb) & ~(int64_t)15;
          for (int64_t off = a0; off < a1; off += 32768)
            bulk_prefetch_l2(sc_plane + off, (uint32_t)(a1 - off < 32768 ? a1 - off : 32768));
        }
        pdl_wait_previous();  // before the first copy into shared memory
        waited = true;
      }
      int it = 0, last_it = -1, last_band = -1, frag_next = 0;
      auto issue_frags = [&](int q) {  // the B fragments and zero points of iteration q
        const int gq = (q % NCH) * 4 * KS;
        const uint32_t sq = stage(q % NS);
        bulk_g2s(sq + p.xf_off, p.xf + (size_t)gq * NT * p.lanes * FB, xf_chunk, full(q % NS));
        bulk_g2s(sq + p.zs_off, reinterpret_cast<const uint8_t*>(p.zs) + (size_t)gq * NT * 64, zs_chunk,
                 full(q % NS));
      };
      for (int b = 0; ok && b < nbands; ++b) {
        const int64_t R0 = band_row(b);
        const int64_t Re = R0 + band_rows(b);
        if (b >= 2 && !(ok = mbar_wait(sempty0 + 8u * (b & 1), (uint32_t)(((b - 2) >> 1) & 1), abort_flag,
                                       &g_mma_status)))
          break;
        {
          // the band's scale run [st, en) of the plane: its 16-byte granules by one bulk copy,
          // the at most 7 scales past the plane's last full granule by plain loads
          const int64_t st = R0 * srb, en = Re * srb;
          const int64_t a = st & ~(int64_t)15;
          const int64_t e_up = (en + 15) & ~(int64_t)15, e_cap = plane_bytes & ~(int64_t)15;
          const int64_t e = e_up < e_cap ? e_up : e_cap;
          const uint32_t dst = scl_buf(b);
          for (int64_t t = (e > st ? e : st); t < en; t += 2)
            sts_u16(dst + (uint32_t)(t - a), *reinterpret_cast<const uint16_t*>(sc_plane + t));
          const uint32_t bytes = e > a ? (uint32_t)(e - a) : 0u;
          mbar_expect_tx(sfull0 + 8u * (b & 1), bytes);
          if (bytes > 0) bulk_g2s(dst, sc_plane + a, bytes, sfull0 + 8u * (b & 1));
          last_band = b;
        }
        for (int j = 0; j < NCH; ++j, ++it) {
          const int s = it % NS;
          if (it >= NS && !(ok = mbar_wait(empty(s), (uint32_t)(((it / NS) - 1) & 1), abort_flag, &g_mma_status)))
            break;
          // sub-boxes holding a group < nk (the consumers skip the others)
          const int g0 = j * 4 * KS;
          int nsub = (p.nk - g0 + 3) / 4;
          nsub = nsub < KS ? nsub : KS;
          const uint32_t sb = stage(s);
          mbar_expect_tx(full(s), (uint32_t)(nsub * BR) * (128u + kHRow) + (kFuse ? 0u : xf_chunk + zs_chunk));
          for (int k = 0; k < nsub; ++k)
            tma_load_2d(sb + (uint32_t)(k * BR * 128), &tm_codes, full(s), (j * KS + k) * 128, (int32_t)R0);
          if constexpr (kHB > 0)  // the sub-boxes' high bits: kHRow bytes per row, unswizzled
            for (int k = 0; k < nsub; ++k)
              tma_load_2d(sb + p.hi_off + (uint32_t)(k * BR) * kHRow, &tm_high, full(s), (j * KS + k) * (int)kHRow,
                          (int32_t)R0);
          // late order: band 0's first stages carry their code sub-boxes before the wait;
          // every later wait of the producer (a free stage, a free scale buffer) comes after it
          if (!kFuse && (waited || it == (NS < NCH ? NS : NCH) - 1)) {
            if (!waited) {
              pdl_wait_previous();
              waited = true;
            }
            for (int q = frag_next; q <= it; ++q) issue_frags(q);
            frag_next = it + 1;
          }
          last_it = it;
        }
      }
      if (!ok) {  // aborted: let every copy already issued land before shared memory is released
        if (!waited) pdl_wait_previous();
        if (!kFuse)
          for (int q = frag_next; q <= last_it; ++q) issue_frags(q);  // complete the stages missing fragments
        for (int i = (last_it - NS + 1 > 0 ? last_it - NS + 1 : 0); i <= last_it; ++i)
          mbar_drain(full(i % NS), (uint32_t)((i / NS) & 1));
        for (int q = (last_band - 1 > 0 ? last_band - 1 : 0); q <= last_band; ++q)
          mbar_drain(sfull0 + 8u * (q & 1), (uint32_t)((q >> 1) & 1));
      }
    }
    __syncwarp();
    return;
  }
  if constexpr (kFuse) {
    // the operand pass of the whole K extent into shared memory by every warp but the
    // producer (the warps the band plan leaves idle included), then one barrier of those
    // warps; x may come from the previous kernel
    pdl_wait_previous();
    // kUnits units per thread per round, their loads issued together
    constexpr int kUnits = 3;
    const int64_t units = (int64_t)32 * p.galloc;  // 8 token slots x 4 lanes per group
    const int64_t wstride = (int64_t)kMaxConsumers * 32;
    uint8_t* fx = smem + p.xf_off;
    float* fz = reinterpret_cast<float*>(smem + p.zs_off);
    const uint16_t* xp = p.x + (int64_t)p.t0 * p.K;
    for (int64_t base = (int64_t)(warp - 1) * 32; base < units; base += kUnits * wstride) {
      uint4 q[kUnits][2];
#pragma unroll
      for (int j = 0; j < kUnits; ++j) {
        const int64_t u = base + j * wstride + lane;
        mma_operand_load<NT, FMT>(xp, p.K, p.tp, p.galloc, u, u < units, q[j]);
      }
#pragma unroll
      for (int j = 0; j < kUnits; ++j) {
        const int64_t u = base + j * wstride + lane;
        if (base + j * wstride < units)  // warp-uniform: the shuffles need every lane
          mma_operand_convert<NT, FMT>(p.tp, p.galloc, p.lanes, u, u < units, q[j], fx, fz);
      }
    }
    named_bar_sync(kConvBar, (uint32_t)(kMaxConsumers * 32));
  }
  if (warp - 1 >= WC) return;

  // ------------------------------------------------------------- consumers
  const int wc = warp - 1;
  const int m = wc / KS, sub = wc % KS;
  const int g = lane >> 2, c = lane & 3;
  const int ra = 16 * m + 2 * g, rb = ra + 1;  // band rows of mma rows g and g + 8
  const bool bload = lane < p.lanes;           // this lane's B fragment is stored (the others are zero)
  int it = 0;
  bool ok = true;
  for (int b = 0; b < nbands; ++b) {
    const int64_t R0 = band_row(b);
    const int rows = band_rows(b);
    const bool va = ra < rows, vb = rb < rows;
    ok = ok && warp_wait(sfull0 + 8u * (b & 1), (uint32_t)((b >> 1) & 1), abort_flag, &g_mma_status);
    const uint32_t sc0 = scl_buf(b) + (uint32_t)((R0 * srb) & 15);
    const uint32_t sca = sc0 + (uint32_t)(ra * srb), scb = sc0 + (uint32_t)(rb * srb);
    float acc[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
    for (int j = 0; j < NCH; ++j, ++it) {
      const int s = it % NS;
      ok = ok && warp_wait(full(s), (uint32_t)((it / NS) & 1), abort_flag, &g_mma_status);
      const int gb = j * 4 * KS + 4 * sub;  // first group of this warp's sub-box
      if (ok && gb < p.nk) {
        const uint32_t code = stage(s) + (uint32_t)(sub * BR * 128);
        const uint32_t rowa = code + (uint32_t)(ra * 128), rowb = code + (uint32_t)(rb * 128);
        // B fragments and zero-point terms of the chunk: in its stage, or (fused) at the chunk's
        // first group of the whole-K buffers
        const uint32_t xf_base = kFuse ? sbase + p.xf_off + (uint32_t)(j * 4 * KS * NT * p.lanes * FB) : stage(s) + p.xf_off;
        const uint32_t zs_base = kFuse ? sbase + p.zs_off + (uint32_t)(j * 4 * KS * NT * 64) : stage(s) + p.zs_off;
        const uint32_t xf = xf_base + (uint32_t)(4 * sub * NT * p.lanes * FB) + (uint32_t)lane * 16u;
        const uint32_t zs = zs_base + (uint32_t)(4 * sub * NT * 64) + (uint32_t)c * 16u;
#pragma unroll
        for (int gl = 0; gl < 4; ++gl) {
          const int G = gb + gl;
          if (G >= p.nk) break;
          // 8 code bytes [8c, 8c + 8) of the group in each row: 16-byte chunk (2 gl + c / 2) of the
          // 128-byte row, swizzled by the row; rows past the band (zero-filled or the next CTA's)
          // decode to finite subnormals whose results are never stored
          const uint32_t ch = (uint32_t)(2 * gl + (c >> 1)), cofs = (uint32_t)((c & 1) << 3);
          const uint2 wa = lds_u64(rowa + (((ch ^ (uint32_t)(ra & 7)) << 4) | cofs));
          const uint2 wb = lds_u64(rowb + (((ch ^ (uint32_t)(rb & 7)) << 4) | cofs));
          uint32_t pa[8], pb[8];
          if constexpr (kW8) {
            decode_w8_pairs(wa.x, wa.y, pa);
            decode_w8_pairs(wb.x, wb.y, pb);
          } else {
            decode_q4_pairs(wa.x, wa.y, pa);
            decode_q4_pairs(wb.x, wb.y, pb);
          }
          if constexpr (kHB > 0) {
            // the high bits of the same 16 weights of each row: 2 (Q5) or 4 (Q6) bytes at
            // 8 kHB bytes per group and 2 kHB per thread column c
            const uint32_t hrow = stage(s) + p.hi_off + (uint32_t)(sub * BR) * kHRow + (uint32_t)(gl * 8 * kHB + c * 2 * kHB);
            uint32_t ha, hb;
            if constexpr (kHB == 1) {
              ha = lds_u16(hrow + (uint32_t)ra * kHRow);
              hb = lds_u16(hrow + (uint32_t)rb * kHRow);
            } else {
              ha = lds_u32(hrow + (uint32_t)ra * kHRow);
              hb = lds_u32(hrow + (uint32_t)rb * kHRow);
            }
            add_high_pairs<kHB>(ha, pa);
            add_high_pairs<kHB>(hb, pb);
          }
          const float sa = va ? fp16_bits_to_float(lds_u16(sca + 2u * (uint32_t)G)) : 0.f;
          const float sbv = vb ? fp16_bits_to_float(lds_u16(scb + 2u * (uint32_t)G)) : 0.f;
#pragma unroll
          for (int n = 0; n < NT; ++n) {
            const uint32_t fa = xf + (uint32_t)((gl * NT + n) * p.lanes * FB);
            const uint4 b0 = bload ? ld_shared_v4(fa) : make_uint4(0u, 0u, 0u, 0u);
            float d[4] = {0.f, 0.f, 0.f, 0.f};
            mma_16816(d, pa[0], pb[0], pa[1], pb[1], b0.x, b0.y);
            mma_16816(d, pa[2], pb[2], pa[3], pb[3], b0.z, b0.w);
            if constexpr (!kW8) {
              const uint4 b1 = bload ? ld_shared_v4(fa + (uint32_t)(p.lanes * 16)) : make_uint4(0u, 0u, 0u, 0u);
              mma_16816(d, pa[4], pb[4], pa[5], pb[5], b1.x, b1.y);
              mma_16816(d, pa[6], pb[6], pa[7], pb[7], b1.z, b1.w);
            }
            // (Z, F) of this thread's two tokens: sum (q - zero) x = F D + Z
            const float4 zf = ld_shared_f4(zs + (uint32_t)((gl * NT + n) * 64));
            const float2 z = make_float2(zf.x, zf.y), f = make_float2(zf.z, zf.w);
            const float2 e01 = ffma2(make_float2(d[0], d[1]), f, z);
            const float2 e23 = ffma2(make_float2(d[2], d[3]), f, z);
            const float2 a01 = ffma2(make_float2(sa, sa), e01, make_float2(acc[n][0], acc[n][1]));
            const float2 a23 = ffma2(make_float2(sbv, sbv), e23, make_float2(acc[n][2], acc[n][3]));
            acc[n][0] = a01.x;
            acc[n][1] = a01.y;
            acc[n][2] = a23.x;
            acc[n][3] = a23.y;
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty(s));
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(sempty0 + 8u * (b & 1));  // the band's scales are no longer read

    // ---- band end: partial sums of the KS sub-boxes, summed in a fixed order
    const int TP = 8 * NT, MR = 16 * p.mt;
    float* red = reinterpret_cast<float*>(smem + p.red_off);
    if (ok) {
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        const int t = 8 * n + 2 * c;
        red[((size_t)sub * MR + ra) * TP + t] = acc[n][0];
        red[((size_t)sub * MR + ra) * TP + t + 1] = acc[n][1];
        red[((size_t)sub * MR + rb) * TP + t] = acc[n][2];
        red[((size_t)sub * MR + rb) * TP + t + 1] = acc[n][3];
      }
    }
    named_bar_sync(kRedBar, (uint32_t)(WC * 32));
    if (b == 0) pdl_wait_previous();  // the exponents are the prep kernel's; every earlier kernel is done
    if (ok && !*abort_flag) {
      float* gate = reinterpret_cast<float*>(smem + p.gate_off);
      const int64_t yrow = kSwi ? r0 + (int64_t)(b >> 1) * BR : R0;  // output row of band row 0
      for (int e = wc * 32 + lane; e < rows * p.tp; e += WC * 32) {
        const int t = e / rows, rw = e - (e / rows) * rows;
        float v = 0.f;
        for (int q = 0; q < KS; ++q) v += red[((size_t)q * MR + rw) * TP + t];
        if (kSwi && (b & 1) == 0) {  // gate band: keep g for the up band that follows
          gate[rw * TP + t] = v;
          continue;
        }
        const int64_t gi = (int64_t)(p.t0 + t) * p.N + yrow + rw;
        if constexpr (kSwi) {  // y = silu(g) * u, silu(g) = g / (1 + e^-g), in FP32
          const float g = gate[rw * TP + t];
          v = g / (1.f + expf(-g)) * v;
        }
        if (p.r != nullptr) v += __uint_as_float((uint32_t)p.r[gi] << 16);
        p.y[gi] = float_to_bf16_bits(v);
      }
    }
    named_bar_sync(kRedBar, (uint32_t)(WC * 32));  // the partial-sum buffer is free again
  }
}

// ----------------------------------------------------------------- host side
struct MmaPlan {
  int fmt, nt, grid, br, ks, mt, nchunks, stages, lanes, galloc, nk, fbytes, early;
  int fused;  // one launch: the streaming kernel runs the operand pass itself (no workspace)
  int64_t code_row, srb;  // bytes of one row of the code plane and of the scale plane
  MmaLayout L;
};

// Token tiles per pass: T <= 8, 16, 24 or 32; a call with more tokens runs passes of 32.
int mma_nt(int64_t T) { return T >= 32 ? 4 : (int)((T + 7) / 8); }

// Launch order of a pass.  Early hides the streaming kernel's launch behind the previous
// kernel but copies its weight rows into shared memory only after the prep kernel has
// finished; late streams them while the prep kernel works.  Early pays off while the B
// fragments are small against the weight rows and the CTA's rows fit the L2 prefetch.
// Measured on 6144 x 5120, back-to-back calls (late -> early): Q4 T = 2, 3, 4: 10.54 ->
// 9.83, 10.63 -> 9.90, 10.70 -> 9.96 us; T = 5, 6: 11.02 -> 10.90, 11.07 -> 10.95;
// T = 7 even; T = 8: 10.92 -> 11.24; T = 12: 13.0 -> 13.9; W8G32 T = 5..8 about 1.1 us
// slower early (its code rows are twice as long).
int mma_early_order(int fmt, int lanes, int nt) { return (fmt == 0 && nt == 1 && lanes <= 24) ? 1 : 0; }

// fmt 0: Q4G64; fmt 3: W8G32 (the other formats have no plan here).  fused: the one-launch
// form (at most 8 tokens, the whole-K B fragments in shared memory), for callers without a
// workspace; otherwise the operand pass and its workspace.
bool mma_plan_for(int64_t N, int64_t K, int64_t T, int sms, MmaPlan* pl, int fmt = 0, bool fused = false,
                  bool swiglu = false) {
  if (N < 1 || K < 8 || T < 1 || fmt < 0 || fmt > 3) return false;
  if (fused && (fmt == 1 || fmt == 2)) return false;   // (no fused operation takes Q5 / Q6)
  const int hb = (fmt == 1 || fmt == 2) ? fmt : 0;       // Q5 / Q6 high bits per weight
  if (fused && T > 8) return false;
  if (swiglu && !fused) return false;   // LinearSwiGLU: the one-launch form only
  if (N >= ((int64_t)1 << 31) || K >= ((int64_t)1 << 31)) return false;
  const bool w8 = fmt == 3;
  const int64_t Kp = (K + 127) / 128 * 128;
  pl->fmt = fmt;
  pl->nk = (int)(w8 ? (K + 31) / 32 : (K + 63) / 64);
  pl->fbytes = w8 ? 16 : 32;
  pl->code_row = w8 ? Kp : Kp / 2;
  pl->srb = w8 ? Kp / 16 : Kp / 32;
  const int nk = pl->nk;
  pl->nt = mma_nt(T);
  const int tpass = (int)(T < 8 * pl->nt ? T : 8 * pl->nt);
  pl->lanes = (pl->nt == 1 && tpass < 8) ? 4 * tpass : 32;
  pl->early = mma_early_order(fmt, pl->lanes, pl->nt);
  int64_t grid = (N + 7) / 8;  // at least 8 rows per CTA
  if (grid > sms) grid = sms;
  pl->grid = (int)grid;
  const int64_t rows_max = (N + grid - 1) / grid;
  // band height: at most 240 rows, and low enough that a band's scale run fits a 32 KB
  // buffer (two of them alternate between bands)
  int64_t cap = 32768 / pl->srb;
  cap = cap > kMaxBand ? kMaxBand : cap / 8 * 8;
  if (cap < 8) return false;
  const int64_t nbands = (rows_max + cap - 1) / cap;
  int br = (int)((rows_max + nbands - 1) / nbands);
  br = (br + 7) / 8 * 8;
  pl->br = br;
  pl->mt = (br + 15) / 16;
  if (pl->mt > kMaxConsumers) return false;
  // sub-boxes per chunk: as many as the consumer warps allow, fewer if the stages do not fit
  for (int ks = kMaxConsumers / pl->mt; ks >= 1; --ks) {
    const int chunk_groups = 4 * ks;
    const int nchunks = (nk + chunk_groups - 1) / chunk_groups;
    int stages = 8;
    for (; stages >= 2; --stages) {
      const MmaLayout L = mma_layout(pl->nt, br, ks, pl->mt, stages, pl->lanes, Kp, pl->fbytes, pl->srb, false, 0,
                                     false, hb);
      if (L.total + 1024 <= kMmaSmem) break;
    }
    if (stages < 2) continue;
    pl->ks = ks;
    pl->nchunks = nchunks;
    pl->stages = stages;
    pl->galloc = nchunks * chunk_groups;
    pl->L = mma_layout(pl->nt, br, ks, pl->mt, stages, pl->lanes, Kp, pl->fbytes, pl->srb, false, 0, false, hb);
    pl->fused = 0;
    if (!fused) return true;
    // the whole-K B fragments beside at least two code stages (else fewer sub-boxes per chunk)
    for (int fs = 8; fs >= 2; --fs) {
      const MmaLayout F = mma_layout(pl->nt, br, ks, pl->mt, fs, pl->lanes, Kp, pl->fbytes, pl->srb, true,
                                     pl->galloc, swiglu);
      if (F.total + 1024 <= kMmaSmem) {
        pl->fused = 1;
        pl->early = 1;
        pl->stages = fs;
        pl->L = F;
        return true;
      }
    }
  }
  return false;
}

int mma_sm_count() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (dev < 64 && cached[dev]) return cached[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  if (dev < 64) cached[dev] = n;
  return n;
}

// Workspace of one pass: B fragments, then the zero-point terms and factors (each 256-byte aligned).
size_t mma_ws_xf(const MmaPlan& pl) { return ((size_t)pl.galloc * pl.nt * pl.lanes * pl.fbytes + 255) / 256 * 256; }
size_t mma_ws_zs(const MmaPlan& pl) { return ((size_t)pl.galloc * pl.nt * 64 + 255) / 256 * 256; }
size_t mma_ws_total(const MmaPlan& pl) { return pl.fused ? 0 : mma_ws_xf(pl) + mma_ws_zs(pl); }

// Opt a streaming-kernel instantiation into the large dynamic shared memory, once per device.
template <int NT, int FMT, bool kFuse, bool kSwi = false>
int mma_kernel_attrs() {
  static bool attr[64] = {};
  int dev = 0;
  if (cuda_check(cudaGetDevice(&dev), "cudaGetDevice")) return Q4LIN_ERR_CUDA;
  if (dev >= 64 || !attr[dev]) {
    if (cuda_check(cudaFuncSetAttribute(q4_mma_kernel<NT, FMT, kFuse, kSwi>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)kMmaSmem),
                   "mma: cudaFuncSetAttribute"))
      return Q4LIN_ERR_CUDA;
    if (dev < 64) attr[dev] = true;
  }
  return Q4LIN_OK;
}

template <int NT, int FMT>
int mma_launch_pass(const LinearArgs& a, const MmaPlan& pl, const CUtensorMap& tm, const CUtensorMap& th, int64_t t0,
                    int tp) {
  const bool fused = NT == 1 && pl.fused && (FMT == 0 || FMT == 3);
  const bool swi = FMT == 0 && fused && a.mode == 1;
  int rc0 = Q4LIN_OK;
  if constexpr (FMT == 0 || FMT == 3)
    rc0 = swi ? mma_kernel_attrs<1, 0, true, true>()
              : fused ? mma_kernel_attrs<1, FMT, true>() : mma_kernel_attrs<NT, FMT, false>();
  else
    rc0 = mma_kernel_attrs<NT, FMT, false>();
  if (rc0 != Q4LIN_OK) return rc0;
  uint8_t* xf = nullptr;
  float* zs = nullptr;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  if (!fused) {
    uint8_t* ws = static_cast<uint8_t*>(a.workspace);
    xf = ws;
    zs = reinterpret_cast<float*>(ws + mma_ws_xf(pl));
    cudaLaunchConfig_t cfg = {};
    const int64_t units = (int64_t)8 * NT * pl.galloc * 4;
    int64_t blocks = (units + kPrepThreads - 1) / kPrepThreads;
    if (blocks > 4 * (int64_t)pl.grid) blocks = 4 * (int64_t)pl.grid;
    cfg.gridDim = dim3((unsigned)blocks, 1, 1);
    cfg.blockDim = dim3(kPrepThreads, 1, 1);
    cfg.stream = a.stream;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    if (cuda_check(cudaLaunchKernelEx(&cfg, q4_mma_prep_kernel<NT, FMT>, a.x + t0 * a.K, xf, zs, a.K, tp,
                                      pl.galloc, pl.lanes, pl.early),
                   "mma: prep kernel launch"))
      return Q4LIN_ERR_CUDA;
  }
  MmaParams p{};
  p.wq = a.wq;
  p.scales = a.scales;
  p.xf = xf;
  p.zs = zs;
  p.x = a.x;
  p.y = a.y;
  p.r = a.r;
  p.N = a.N;
  p.K = a.K;
  p.Kp = k_pad(a.K);
  p.T = a.T;
  p.t0 = (int)t0;
  p.tp = tp;
  p.nk = pl.nk;
  p.br = pl.br;
  p.ks = pl.ks;
  p.mt = pl.mt;
  p.nchunks = pl.nchunks;
  p.stages = pl.stages;
  p.lanes = pl.lanes;
  p.early = pl.early;
  p.galloc = pl.galloc;
  p.stage_bytes = pl.L.stage_bytes;
  p.hi_off = pl.L.code_bytes;
  p.xf_off = fused ? pl.L.fx_off : pl.L.code_bytes + pl.L.hi_bytes;
  p.zs_off = fused ? pl.L.fz_off : pl.L.code_bytes + pl.L.hi_bytes + pl.L.xf_bytes;
  p.scl_off = pl.L.scl_off;
  p.scl_bytes = pl.L.scl_bytes;
  p.red_off = pl.L.red_off;
  p.gate_off = pl.L.gate_off;
  p.bar_off = pl.L.bar_off;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)pl.grid, 1, 1);
  cfg.blockDim = dim3(kMmaThreads, 1, 1);
  cfg.dynamicSmemBytes = kMmaSmem;
  cfg.stream = a.stream;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  if constexpr (NT == 1 && (FMT == 0 || FMT == 3)) {
    if (swi) return cuda_check(cudaLaunchKernelEx(&cfg, q4_mma_kernel<1, 0, true, true>, tm, th, p), "mma: kernel launch");
    if (fused) return cuda_check(cudaLaunchKernelEx(&cfg, q4_mma_kernel<1, FMT, true>, tm, th, p), "mma: kernel launch");
  }
  return cuda_check(cudaLaunchKernelEx(&cfg, q4_mma_kernel<NT, FMT, false>, tm, th, p), "mma: kernel launch");
}

template <int FMT>
int mma_launch_fmt(const LinearArgs& a, const MmaPlan& pl, const CUtensorMap& tm, const CUtensorMap& th) {
  // passes of at most 32 tokens (8 NT each), sharing the workspace in stream order
  for (int64_t t0 = 0; t0 < a.T; t0 += 8 * pl.nt) {
    const int tp = (int)((a.T - t0) < 8 * pl.nt ? (a.T - t0) : 8 * pl.nt);
    int rc;
    switch (pl.nt) {
      case 1: rc = mma_launch_pass<1, FMT>(a, pl, tm, th, t0, tp); break;
      case 2: rc = mma_launch_pass<2, FMT>(a, pl, tm, th, t0, tp); break;
      case 3: rc = mma_launch_pass<3, FMT>(a, pl, tm, th, t0, tp); break;
      default: rc = mma_launch_pass<4, FMT>(a, pl, tm, th, t0, tp); break;
    }
    if (rc != Q4LIN_OK) return rc;
  }
  return Q4LIN_OK;
}

}  // namespace

bool mma_supported(int64_t N, int64_t K, int64_t T, int fmt) {
  MmaPlan pl;
  return mma_plan_for(N, K, T, mma_sm_count(), &pl, fmt);
}

size_t mma_workspace_bytes(int64_t N, int64_t K, int64_t T, int fmt) {
  MmaPlan pl;
  if (!mma_plan_for(N, K, T, mma_sm_count(), &pl, fmt)) return 0;
  return mma_ws_total(pl);
}

int mma_launch_count(int64_t, int64_t, int64_t T, int) { return 2 * (int)((T + 31) / 32); }

bool mma_fused_supported(int64_t N, int64_t K, int64_t T, int fmt, bool swiglu) {
  MmaPlan pl;
  return mma_plan_for(N, K, T, mma_sm_count(), &pl, fmt, true, swiglu);
}

int mma_launch(const LinearArgs& a, bool fused) {
  MmaPlan pl;
  const bool swiglu = a.mode == 1;
  if (a.mode == 2 || (swiglu && a.fmt != 0) || !mma_plan_for(a.N, a.K, a.T, mma_sm_count(), &pl, a.fmt, fused, swiglu)) {
    set_error_detail("mma: no shared-memory plan for this format and shape");
    return Q4LIN_ERR_UNSUPPORTED_SHAPE;
  }
  CUtensorMap tm;
  if (!encode_map_2d(&tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.wq, (uint64_t)pl.code_row, (uint64_t)(swiglu ? 2 * a.N : a.N),
                     (uint64_t)pl.code_row, 128, (uint32_t)pl.br, CU_TENSOR_MAP_SWIZZLE_128B)) {
    set_error_detail("mma: cuTensorMapEncodeTiled failed (or is unavailable)");
    return Q4LIN_ERR_CUDA;
  }
  // Q5 / Q6: the high-bit plane, rows of K_pad * hb / 8 bytes, boxes of one sub-box (256 weights,
  // 32 hb bytes) x band rows, unswizzled
  CUtensorMap th = tm;  // unused for Q4 and W8
  if (pl.fmt == 1 || pl.fmt == 2) {
    if (a.wh == nullptr) {
      set_error_detail("mma: Q5 / Q6 without a high-bit plane");
      return Q4LIN_ERR_INVALID_ARG;
    }
    const uint64_t hrow = (uint64_t)(k_pad(a.K) * pl.fmt / 8);
    if (!encode_map_2d(&th, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.wh, hrow, (uint64_t)a.N, hrow, (uint32_t)(32 * pl.fmt),
                       (uint32_t)pl.br, CU_TENSOR_MAP_SWIZZLE_NONE)) {
      set_error_detail("mma: cuTensorMapEncodeTiled failed for the high-bit plane");
      return Q4LIN_ERR_CUDA;
    }
  }
  switch (pl.fmt) {
    case 1: return mma_launch_fmt<1>(a, pl, tm, th);
    case 2: return mma_launch_fmt<2>(a, pl, tm, th);
    case 3: return mma_launch_fmt<3>(a, pl, tm, th);
    default: return mma_launch_fmt<0>(a, pl, tm, th);
  }
}

int mma_status(int* value, bool clear) {
  if (cudaMemcpyFromSymbol(value, g_mma_status, sizeof(int)) != cudaSuccess) return Q4LIN_ERR_CUDA;
  if (clear) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_mma_status, &zero, sizeof(int)) != cudaSuccess) return Q4LIN_ERR_CUDA;
  }
  return Q4LIN_OK;
}

}  // namespace q4
