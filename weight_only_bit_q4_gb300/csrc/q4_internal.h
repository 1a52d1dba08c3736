// Host-side declarations shared by the q4lin translation units.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace q4 {

struct LinearArgs {
  const uint8_t* wq;
  const uint16_t* scales;
  const uint16_t* x;
  uint16_t* y;
  int64_t N, K, T;
  void* workspace;
  cudaStream_t stream;
};

// CUDA-core GEMV: each weight is decoded once per block of up to 4 tokens.
int gemv_launch(const LinearArgs& a);
size_t gemv_workspace_bytes(int64_t N, int64_t K, int64_t T);
int gemv_launch_count(int64_t N, int64_t K, int64_t T);

// tcgen05 tile route: X converted to fp16 in the workspace, then one CTA per
// 128-row x BN-token output tile with the accumulator in tensor memory.
int tc_launch(const LinearArgs& a);
size_t tc_workspace_bytes(int64_t N, int64_t K, int64_t T);
int tc_launch_count(int64_t N, int64_t K, int64_t T);
bool tc_supported(int64_t N, int64_t K, int64_t T);

// Reads (and optionally clears) the device error word of one translation unit.
int gemv_status(int* value, bool clear);
int tc_status(int* value, bool clear);

}  // namespace q4
