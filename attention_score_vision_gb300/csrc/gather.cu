// Order-preserving compaction of the kept tokens with their metadata.
//
// The dynamic vision-token compression article (section 3.2) requires the
// pruned sequence to keep its input lengths, image boundaries, original
// spatial indices and position ids consistent, so it can flow into prefill
// and the KV cache. keep_idx is ascending, so every output row k is an
// independent copy and the new per-image boundaries are lower bounds of the
// old ones in keep_idx.
//
// Rows are copied with 16-byte vector loads/stores, one warp per row, several
// rows in flight per warp (HBM-bound: the algorithmic bytes are the kept rows
// read once and written once).
#include <cuda_runtime.h>

#include "common.cuh"
#include "launch_util.cuh"

namespace tsel {

constexpr int kGatherThreads = 256;
constexpr int kGatherUnroll = 4;

__device__ __forceinline__ int upper_bound_i32(const int32_t* a, int n, int v) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(a + mid) <= v) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

__device__ __forceinline__ int lower_bound_i32(const int32_t* a, int n, int v) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(a + mid) < v) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

__global__ void __launch_bounds__(kGatherThreads)
    gather_kernel(const uint8_t* __restrict__ hidden, int64_t row_stride_bytes, int row_vecs,
                  const int32_t* __restrict__ pos, int pos_dim,
                  const int32_t* __restrict__ cu_k, int G, int Tk,
                  const int32_t* __restrict__ keep_idx, int K, const int32_t* K_dev,
                  uint8_t* __restrict__ out_hidden, int32_t* __restrict__ out_pos,
                  int32_t* __restrict__ out_img, int32_t* __restrict__ out_cu,
                  uint32_t* status) {
  const int lane = threadIdx.x & 31;
  pdl_launch_dependents();
  pdl_wait();
  if (K_dev != nullptr) {
    // kept count produced on the device; K is the capacity the launch was sized for
    const int kd = __ldg(K_dev);
    if (kd < 0 || kd > K) {
      if (blockIdx.x == 0 && threadIdx.x == 0) set_status(status, TSEL_DEV_KEEP_IDX);
    }
    K = kd < 0 ? 0 : (kd > K ? K : kd);
  }
  const int gwarp = (blockIdx.x * kGatherThreads + threadIdx.x) >> 5;
  const int nwarps = (gridDim.x * kGatherThreads) >> 5;
  const int gtid = blockIdx.x * kGatherThreads + threadIdx.x;

  // New per-image boundaries: kept tokens below each old boundary.
  for (int g = gtid; g <= G; g += gridDim.x * kGatherThreads)
    out_cu[g] = lower_bound_i32(keep_idx, K, __ldg(cu_k + g));

  for (int k = gwarp; k < K; k += nwarps) {
    const int t = __ldg(keep_idx + k);
    const bool ok = t >= 0 && t < Tk && (k == 0 || __ldg(keep_idx + k - 1) < t);
    if (!ok) {
      if (lane == 0) set_status(status, TSEL_DEV_KEEP_IDX);
      continue;
    }
    const uint4* src = reinterpret_cast<const uint4*>(hidden + int64_t(t) * row_stride_bytes);
    uint4* dst = reinterpret_cast<uint4*>(out_hidden + int64_t(k) * row_vecs * 16);
    int v = lane;
    for (; v + 32 * (kGatherUnroll - 1) < row_vecs; v += 32 * kGatherUnroll) {
      uint4 x[kGatherUnroll];
#pragma unroll
      for (int u = 0; u < kGatherUnroll; ++u) x[u] = __ldcs(src + v + 32 * u);
#pragma unroll
      for (int u = 0; u < kGatherUnroll; ++u) __stcs(dst + v + 32 * u, x[u]);
    }
    for (; v < row_vecs; v += 32) __stcs(dst + v, __ldcs(src + v));
    if (lane < pos_dim) out_pos[int64_t(k) * pos_dim + lane] = __ldg(pos + int64_t(t) * pos_dim + lane);
    if (lane == 0) out_img[k] = upper_bound_i32(cu_k, G + 1, t) - 1;
  }
}

cudaError_t launch_gather(const void* hidden, int64_t row_stride_bytes, int row_bytes,
                          const int32_t* pos, int pos_dim, const int32_t* cu_k, int G, int Tk,
                          const int32_t* keep_idx, int K, const int32_t* K_dev,
                          void* out_hidden, int32_t* out_pos, int32_t* out_img, int32_t* out_cu,
                          uint32_t* status, int num_sms, cudaStream_t stream) {
  const int64_t warps_needed = K > G + 1 ? K : G + 1;
  int64_t blocks = (warps_needed * 32 + kGatherThreads - 1) / kGatherThreads;
  const int64_t max_blocks = int64_t(num_sms) * (2048 / kGatherThreads);
  if (blocks > max_blocks) blocks = max_blocks;
  if (blocks < 1) blocks = 1;
  return launch_kernel(gather_kernel, dim3(unsigned(blocks)), kGatherThreads, 0, stream, 1,
                       static_cast<const uint8_t*>(hidden), row_stride_bytes, row_bytes / 16, pos,
                       pos_dim, cu_k, G, Tk, keep_idx, K, K_dev, static_cast<uint8_t*>(out_hidden),
                       out_pos, out_img, out_cu, status);
}

}  // namespace tsel
