// Diagnostics of q4lin: an HBM read probe and a bounded-wait expiry check.
//
// Read probe.  The linear-benchmark contract (section 4, theoretical traffic)
// takes a pure-read probe -- 128-bit loads over a 4 GiB buffer -- rather than a
// copy as the ceiling a weight-streaming GEMV can reach.  q4lin_hbm_read_probe is
// that probe: a grid-stride loop of 16-byte non-allocating loads over `bytes`
// bytes, folded with XOR into one word per CTA so the loads cannot be dropped.
//
// Wait expiry.  Every pipeline wait in the q4lin kernels is a bounded poll of an
// mbarrier phase; when the bound runs out the kernel records Q4LIN_ERR_TIMEOUT in
// its device error word, raises the CTA's abort flag and returns instead of
// hanging.  q4lin_diag_wait_expiry runs that same bounded wait (mbar_wait) on an
// mbarrier phase that nothing ever completes, with a caller-chosen short bound, so
// a test can see the timeout reach q4lin_device_status() and the context stay usable.
#include "q4_internal.h"
#include "q4_sm100.cuh"

namespace q4 {

namespace {

__device__ int g_probe_status = 0;

constexpr int kProbeThreads = 512;

__global__ void __launch_bounds__(kProbeThreads)
q4_hbm_read_probe_kernel(const uint4* __restrict__ src, int64_t n16, uint32_t* __restrict__ sink) {
  uint32_t acc = 0;
  const int64_t stride = (int64_t)gridDim.x * kProbeThreads;
  int64_t i = (int64_t)blockIdx.x * kProbeThreads + threadIdx.x;
  // four independent loads in flight per thread per step
  for (; i + 3 * stride < n16; i += 4 * stride) {
    const uint4 a = ld_stream_u4(src + i), b = ld_stream_u4(src + i + stride);
    const uint4 c = ld_stream_u4(src + i + 2 * stride), d = ld_stream_u4(src + i + 3 * stride);
    acc ^= a.x ^ a.y ^ a.z ^ a.w ^ b.x ^ b.y ^ b.z ^ b.w ^ c.x ^ c.y ^ c.z ^ c.w ^ d.x ^ d.y ^ d.z ^ d.w;
  }
  for (; i < n16; i += stride) {
    const uint4 a = ld_stream_u4(src + i);
    acc ^= a.x ^ a.y ^ a.z ^ a.w;
  }
  acc = __reduce_xor_sync(0xffffffffu, acc);
  __shared__ uint32_t red[kProbeThreads / 32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t v = 0;
    for (int w = 0; w < kProbeThreads / 32; ++w) v ^= red[w];
    sink[blockIdx.x] = v;
  }
}

// One warp waits, with the bound `limit`, on phase 0 of an mbarrier that expects one
// arrival which never comes.  Lane 0 polls with the kernels' own bounded wait
// (mbar_wait): on expiry it raises the abort flag the other roles of a real kernel
// would see and records Q4LIN_ERR_TIMEOUT in this unit's device error word.
// out[0] = 1 if the wait succeeded (it cannot) | 2 if the abort flag is up.
__global__ void q4_wait_expiry_bounded_kernel(uint32_t limit, int* __restrict__ out) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_word;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    abort_word = 0;
    fence_mbar_init();
  }
  __syncthreads();
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(b, 0, &abort_word, &g_probe_status, limit);
  ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  if (threadIdx.x == 0) out[0] = (ok ? 1 : 0) | (abort_word ? 2 : 0);
}

}  // namespace

int probe_status(int* value, bool clear) {
  if (cudaMemcpyFromSymbol(value, g_probe_status, sizeof(int)) != cudaSuccess) return Q4LIN_ERR_CUDA;
  if (clear) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_probe_status, &zero, sizeof(int)) != cudaSuccess) return Q4LIN_ERR_CUDA;
  }
  return Q4LIN_OK;
}

int hbm_read_probe(const void* src, size_t bytes, uint32_t* sink, int blocks, cudaStream_t stream) {
  q4_hbm_read_probe_kernel<<<(unsigned)blocks, kProbeThreads, 0, stream>>>(static_cast<const uint4*>(src),
                                                                           (int64_t)(bytes / 16), sink);
  return cuda_check(cudaGetLastError(), "hbm read probe launch");
}

int wait_expiry(uint32_t limit, int* out, cudaStream_t stream) {
  q4_wait_expiry_bounded_kernel<<<1, 32, 0, stream>>>(limit, out);
  return cuda_check(cudaGetLastError(), "wait expiry kernel launch");
}

}  // namespace q4
