// Host-buffer staging of q4lin_linear_host: X copied from page-locked host memory
// into the workspace before the layer (the routes read X with bulk and tensor copies;
// they store Y with plain stores, straight into the page-locked output).
//
// The copies are kernels rather than copy-engine transfers: on a host whose memory
// the GPU reaches coherently, SM loads and stores of page-locked memory start within
// a launch, where a small cudaMemcpyAsync pays the copy engine's setup per transfer.
// The staging kernel takes part in the layer's programmatic-dependent-launch chain:
// it lets the next kernel launch at once and waits for the previous one before it
// touches memory the previous kernel may use (the X staging area the previous
// call's kernels read).  With K == 0 the same kernel copies the staged zeros out.
#include "q4_internal.h"
#include "q4_sm100.cuh"

namespace q4 {

namespace {

constexpr int kStageThreads = 256;

// n16 16-byte units, then n2 2-byte elements (the tail of a buffer whose size is not a
// multiple of 16), from src to dst; either side may be page-locked host memory mapped
// into the device's address space.
__global__ void __launch_bounds__(kStageThreads)
q4_stage_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, int64_t n16, int64_t n2) {
  pdl_launch_dependents();
  pdl_wait_previous();
  const int64_t stride = (int64_t)gridDim.x * kStageThreads;
  int64_t i = (int64_t)blockIdx.x * kStageThreads + threadIdx.x;
  // two independent 16-byte loads in flight per thread per step
  for (; i + stride < n16; i += 2 * stride) {
    const uint4 a = src[i], b = src[i + stride];
    dst[i] = a;
    dst[i + stride] = b;
  }
  for (; i < n16; i += stride) dst[i] = src[i];
  const uint16_t* s2 = reinterpret_cast<const uint16_t*>(src + n16);
  uint16_t* d2 = reinterpret_cast<uint16_t*>(dst + n16);
  for (int64_t j = (int64_t)blockIdx.x * kStageThreads + threadIdx.x; j < n2; j += stride) d2[j] = s2[j];
}

}  // namespace

int stage_copy(const void* src, void* dst, size_t bytes, cudaStream_t stream) {
  if (bytes == 0) return 0;
  const int64_t n16 = (int64_t)(bytes / 16), n2 = (int64_t)((bytes % 16) / 2);
  int dev = 0, sms = 0;
  if (cuda_check(cudaGetDevice(&dev), "cudaGetDevice") ||
      cuda_check(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev), "SM count"))
    return 6;
  // one thread per two 16-byte units, at most two CTAs per SM
  int64_t blocks = (n16 / 2 + kStageThreads - 1) / kStageThreads;
  if (blocks < 1) blocks = 1;
  if (blocks > 2 * (int64_t)sms) blocks = 2 * (int64_t)sms;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks, 1, 1);
  cfg.blockDim = dim3(kStageThreads, 1, 1);
  cfg.stream = stream;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cuda_check(cudaLaunchKernelEx(&cfg, q4_stage_kernel, static_cast<const uint4*>(src), static_cast<uint4*>(dst),
                                       n16, n2),
                    "host staging copy");
}

}  // namespace q4
