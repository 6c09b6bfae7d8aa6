// MUFU exp2 throughput probe: the peak the importance kernel's exp work is
// measured against. Each thread runs 8 independent chains x -> 2^-x, which
// stay inside [0.5, 1] and never hit special values. The first thread of
// block 0 also times its own run in SM clocks and in nanoseconds, so the
// caller knows the SM clock the peak was taken at.
#include <cuda_runtime.h>

#include "common.cuh"
#include "ptx.cuh"

namespace tsel {

constexpr int kProbeThreads = 512;

__global__ void __launch_bounds__(kProbeThreads) probe_ex2_kernel(int iters, float* sink) {
  const bool timer = blockIdx.x == 0 && threadIdx.x == 0;
  const uint64_t c0 = timer ? clock64() : 0, t0 = timer ? ptx::globaltimer_ns() : 0;
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
  if (timer) {
    const uint64_t c1 = clock64(), t1 = ptx::globaltimer_ns();
    // two 64-bit words after the per-thread floats (8-byte aligned: the
    // floats fill whole 2 KB blocks)
    uint64_t* w = reinterpret_cast<uint64_t*>(sink + size_t(gridDim.x) * kProbeThreads);
    w[0] = c1 - c0;
    w[1] = t1 - t0;
  }
}

cudaError_t launch_probe_ex2(int blocks, int iters, float* sink, cudaStream_t stream) {
  probe_ex2_kernel<<<blocks, kProbeThreads, 0, stream>>>(iters, sink);
  return cudaPeekAtLastError();
}

}  // namespace tsel
