// Device helpers shared by the q4lin kernels (sm_103a).  Inline PTX wrappers
// for loads, mbarriers, TMA and bf16/fp16 conversions.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>

#include "q4lin.h"

namespace q4 {

// Weights per scale group along K, and the code zero point: w = (q - 8) * s.
constexpr int kGroup = 64;
constexpr int kZeroPoint = 8;

// Bound on every device-side spin wait (iterations of a try_wait loop that
// each suspend for up to ~1 us in hardware); hitting it means a pipeline bug,
// not slowness, and the kernel records Q4LIN_ERR_TIMEOUT instead of hanging.
constexpr uint32_t kSpinLimit = 1u << 22;

__device__ __forceinline__ uint4 ld_stream_u4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

__device__ __forceinline__ uint4 ld_nc_u4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

__device__ __forceinline__ float fp16_bits_to_float(uint16_t b) {
  return __half2float(__ushort_as_half(b));
}

__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// bf16 pair (two bf16 in one 32-bit word, element 0 in the low half) -> floats.
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// fp32 (128 + q) for the nibble held in byte j of `b` (the byte's upper
// nibble must already be clear): bytes {0, 0, q, 0x43} = 2^7 * (1 + q/128).
template <int J>
__device__ __forceinline__ float f128_plus_byte(uint32_t b) {
  return __uint_as_float(__byte_perm(b, 0x43u, 0x4055u | (J << 8)));
}

// Packed fp32x2 fused multiply-add (sm_100 family): d = a * b + c per lane pair.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(d)
      : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)),
        "l"(*reinterpret_cast<uint64_t*>(&c)));
  return *reinterpret_cast<float2*>(&d);
}

__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;"
      : "=l"(d)
      : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)));
  return *reinterpret_cast<float2*>(&d);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace q4
