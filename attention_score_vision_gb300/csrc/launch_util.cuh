// Launch helpers shared by every kernel of the library.
//
// Every kernel is launched with programmatic stream serialization (PDL): the
// next kernel on the stream may start its prologue while the previous one
// drains. Each kernel therefore calls pdl_launch_dependents() once all of its
// CTAs are resident (the top-B kernel only after its radix rounds, so the
// compaction's CTAs do not sit on its SMs meanwhile) and pdl_wait() before it
// touches memory that an earlier kernel on the stream writes or reads, so
// stream order holds for data.
//
// Cluster kernels (top-B, dynamic budget) run one thread-block cluster per
// request, sized from the average request length and capped by what the
// device can co-schedule.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace tsel {

constexpr int kMaxClusterCtas = 16;

// Cluster size from the average request size (the host does not see the
// per-request offsets): small requests need no cluster.
inline int cluster_size_for(int total_tokens, int num_req) {
  const int64_t avg = num_req > 0 ? (int64_t(total_tokens) + num_req - 1) / num_req : 0;
  if (avg >= 32768) return 16;
  if (avg >= 16384) return 8;
  if (avg >= 8192) return 4;
  return 1;
}

// Cluster size for num_clusters clusters of `kernel` (threads per CTA, dyn
// bytes of dynamic shared memory): the largest power of two <= want at which
// the device can hold every one of them at once, else 1. A cluster that has
// to wait for another one to finish would double these latency-bound
// kernels' time (at most 7 clusters of 16 top-B CTAs fit on a GB300).
// cache[dev][0] notes that the kernel's attributes are set on that device;
// cache[dev][k] keeps 1 + the number of resident clusters of 2^k CTAs.
template <typename Kernel>
int cluster_size_for_grid(Kernel kernel, int want, int num_clusters, int threads, size_t dyn,
                          int (*cache)[5], cudaError_t* err) {
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return 1;
  const bool cacheable = dev >= 0 && dev < 128;
  int lw = 0;
  while ((1 << (lw + 1)) <= want && lw < 4) ++lw;
  if (!cacheable || cache[dev][0] == 0) {
    *err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(dyn));
    if (*err != cudaSuccess) return 1;
    *err = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (*err != cudaSuccess) return 1;
    if (cacheable) cache[dev][0] = 1;
  }
  for (; lw > 0; --lw) {
    int active = 0;
    if (cacheable && cache[dev][lw] > 0) {
      active = cache[dev][lw] - 1;
    } else {
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 1u << lw;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.gridDim = dim3(1u << lw);
      cfg.blockDim = dim3(unsigned(threads));
      cfg.dynamicSmemBytes = dyn;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&active, kernel, &cfg) != cudaSuccess) {
        active = 0;
        (void)cudaGetLastError();
      }
      if (cacheable) cache[dev][lw] = active + 1;
    }
    if (active >= num_clusters) return 1 << lw;
  }
  return 1;
}

// Launches `kernel` on `stream` with programmatic stream serialization and,
// when cluster_x > 1, clusters of cluster_x CTAs along x.
template <typename Kernel, typename... Args>
cudaError_t launch_kernel(Kernel kernel, dim3 grid, int threads, size_t dyn, cudaStream_t stream,
                          int cluster_x, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(unsigned(threads));
  cfg.dynamicSmemBytes = dyn;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster_x > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = unsigned(cluster_x);
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = unsigned(n);
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
  if (e != cudaSuccess) return e;
  return cudaPeekAtLastError();
}

// Launches `kernel` with one cluster of `csize` CTAs per request.
template <typename Kernel, typename... Args>
cudaError_t launch_clusters(Kernel kernel, int num_req, int csize, int threads, size_t dyn,
                            cudaStream_t stream, Args... args) {
  return launch_kernel(kernel, dim3(unsigned(num_req) * unsigned(csize)), threads, dyn, stream,
                       csize, args...);
}

}  // namespace tsel
