// MUFU exp2 throughput probe: the peak the importance kernel's exp work is
// measured against. Each thread runs 8 independent chains x -> 2^-x, which
// stay inside [0.5, 1] and never hit special values.
#include <cuda_runtime.h>

#include "common.cuh"

namespace tsel {

constexpr int kProbeThreads = 512;

__global__ void __launch_bounds__(kProbeThreads) probe_ex2_kernel(int iters, float* sink) {
  float x[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) x[j] = 0.5f + 0.01f * j + 1e-6f * threadIdx.x;
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int j = 0; j < 8; ++j) asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(x[j]) : "f"(-x[j]));
  }
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) s += x[j];
  sink[blockIdx.x * kProbeThreads + threadIdx.x] = s;
}

cudaError_t launch_probe_ex2(int blocks, int iters, float* sink, cudaStream_t stream) {
  probe_ex2_kernel<<<blocks, kProbeThreads, 0, stream>>>(iters, sink);
  return cudaPeekAtLastError();
}

}  // namespace tsel
