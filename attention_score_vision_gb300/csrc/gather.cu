// Order-preserving compaction of the kept tokens with their metadata.
//
// The dynamic vision-token compression article (section 3.2) requires the
// pruned sequence to keep its input lengths, image boundaries, original
// spatial indices and position ids consistent, so it can flow into prefill
// and the KV cache. keep_idx is ascending, so every output row k is an
// independent copy and the new per-image boundaries are lower bounds of the
// old ones in keep_idx.
//
// Rows are copied with 16-byte streaming loads/stores. Each warp takes two
// consecutive kept rows at a time and issues every load of both rows (and
// their positions) before its stores (rows of up to 4 KB stay in registers),
// so each lane keeps up to 16 loads in flight (HBM-bound: the algorithmic
// bytes are the kept rows read once and written once). A few warps at the end
// of the grid find the new image boundaries meanwhile, by 32-ary searches of
// keep_idx (a handful of dependent loads each, which for small requests would
// otherwise be the kernel's longest chain).
#include <cuda_runtime.h>

#include "common.cuh"
#include "launch_util.cuh"

namespace tsel {

constexpr int kGatherThreads = 256;
constexpr int kGatherRows = 2;     // kept rows per warp per step
constexpr int kGatherMaxVpl = 8;   // 16-byte vectors per lane per row held in registers

__device__ __forceinline__ int upper_bound_i32(const int32_t* a, int n, int v) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(a + mid) <= v) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

// First index i in [0, n) with a[i] >= v (n if none) for ascending a: a
// 32-ary search by one warp, so that a search over the kept tokens takes two
// or three dependent loads (n up to 64K) instead of log2(n). Every lane
// returns the index. For input that is not ascending it still returns an
// index in [0, n].
__device__ __forceinline__ int warp_lower_bound(const int32_t* a, int n, int v) {
  const int lane = threadIdx.x & 31;
  int lo = 0, hi = n;   // the index lies in [lo, hi]
  while (hi - lo > 64) {
    const int step = (hi - lo + 31) >> 5;
    const int idx = lo + (lane + 1) * step - 1;   // last element of sub-range `lane`
    const bool below = idx < hi && __ldg(a + idx) < v;
    lo += step * __popc(__ballot_sync(0xffffffffu, below));   // sub-ranges wholly below v
    hi = min(hi, lo + step);
  }
  const int i0 = lo + lane, i1 = lo + 32 + lane;
  const bool b0 = i0 < hi && __ldg(a + i0) < v;
  const bool b1 = i1 < hi && __ldg(a + i1) < v;
  return lo + __popc(__ballot_sync(0xffffffffu, b0)) + __popc(__ballot_sync(0xffffffffu, b1));
}

// VPL = 16-byte vectors per lane per row (rows of up to 32 * VPL vectors in
// registers); VPL = 0 copies rows of any length in a loop.
// Register caps keep the blocks per SM the copy's loads in flight need: 4
// (32 warps) for rows of up to 5 vectors per lane, 3 for 6 or 7.
template <int VPL>
__global__ void __launch_bounds__(kGatherThreads, (VPL >= 1 && VPL <= 5) ? 4 : ((VPL == 6 || VPL == 7) ? 3 : 1))
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
  // The last nb warps find the new per-image boundaries (kept tokens below
  // each old boundary), one boundary per warp at a time, while the others
  // copy rows.
  const int nb = min(G + 1, nwarps / 16 + 1);
  const int row_warps = nwarps - nb;
  if (gwarp >= row_warps) {
    for (int g = gwarp - row_warps; g <= G; g += nb) {
      const int b = warp_lower_bound(keep_idx, K, __ldg(cu_k + g));
      if (lane == 0) out_cu[g] = b;
    }
    return;
  }

  // Image of a token: boundaries <= t, minus one (a ballot when they fit a warp).
  const bool few_images = G < 32;
  const int cu_lane = few_images && lane <= G ? __ldg(cu_k + lane) : 0x7FFFFFFF;

  for (int k0 = kGatherRows * gwarp; k0 < K; k0 += kGatherRows * row_warps) {
    int t[kGatherRows];
    bool ok[kGatherRows];
    int pv[kGatherRows];   // position component `lane` of each row, loaded with the row
#pragma unroll
    for (int r = 0; r < kGatherRows; ++r) {
      const int k = k0 + r;
      t[r] = k < K ? __ldg(keep_idx + k) : -1;
      const int prev = k > 0 && k < K ? __ldg(keep_idx + k - 1) : -1;
      ok[r] = k < K && t[r] >= 0 && t[r] < Tk && prev < t[r];
      if (k < K && !ok[r] && lane == 0) set_status(status, TSEL_DEV_KEEP_IDX);
      pv[r] = ok[r] && lane < pos_dim ? __ldg(pos + int64_t(t[r]) * pos_dim + lane) : 0;
    }
    if (VPL > 0) {
      uint4 x[kGatherRows][VPL > 0 ? VPL : 1];
#pragma unroll
      for (int r = 0; r < kGatherRows; ++r) {
        const uint4* src = reinterpret_cast<const uint4*>(hidden + int64_t(t[r]) * row_stride_bytes);
#pragma unroll
        for (int u = 0; u < VPL; ++u) {
          const int v = lane + 32 * u;
          if (ok[r] && v < row_vecs) x[r][u] = __ldcs(src + v);
        }
      }
#pragma unroll
      for (int r = 0; r < kGatherRows; ++r) {
        uint4* dst = reinterpret_cast<uint4*>(out_hidden + int64_t(k0 + r) * row_vecs * 16);
#pragma unroll
        for (int u = 0; u < VPL; ++u) {
          const int v = lane + 32 * u;
          if (ok[r] && v < row_vecs) __stcs(dst + v, x[r][u]);
        }
      }
    } else {
#pragma unroll
      for (int r = 0; r < kGatherRows; ++r) {
        if (!ok[r]) continue;
        const uint4* src = reinterpret_cast<const uint4*>(hidden + int64_t(t[r]) * row_stride_bytes);
        uint4* dst = reinterpret_cast<uint4*>(out_hidden + int64_t(k0 + r) * row_vecs * 16);
        int v = lane;
        for (; v + 32 * (kGatherMaxVpl - 1) < row_vecs; v += 32 * kGatherMaxVpl) {
          uint4 x[kGatherMaxVpl];
#pragma unroll
          for (int u = 0; u < kGatherMaxVpl; ++u) x[u] = __ldcs(src + v + 32 * u);
#pragma unroll
          for (int u = 0; u < kGatherMaxVpl; ++u) __stcs(dst + v + 32 * u, x[u]);
        }
        for (; v < row_vecs; v += 32) __stcs(dst + v, __ldcs(src + v));
      }
    }
#pragma unroll
    for (int r = 0; r < kGatherRows; ++r) {
      if (!ok[r]) continue;
      const int k = k0 + r;
      if (lane < pos_dim) out_pos[int64_t(k) * pos_dim + lane] = pv[r];
      if (few_images) {
        const int img = __popc(__ballot_sync(0xffffffffu, cu_lane <= t[r])) - 1;
        if (lane == 0) out_img[k] = img;
      } else if (lane == 0) {
        out_img[k] = upper_bound_i32(cu_k, G + 1, t[r]) - 1;
      }
    }
  }
}

template <int VPL>
static cudaError_t launch_gather_vpl(int num_sms, int64_t warps_needed, cudaStream_t stream,
                                     const uint8_t* hidden, int64_t row_stride_bytes, int row_vecs,
                                     const int32_t* pos, int pos_dim, const int32_t* cu_k, int G,
                                     int Tk, const int32_t* keep_idx, int K, const int32_t* K_dev,
                                     uint8_t* out_hidden, int32_t* out_pos, int32_t* out_img,
                                     int32_t* out_cu, uint32_t* status) {
  static int resident[128] = {};   // blocks per SM, per device (0 = not asked yet)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int per_sm = dev >= 0 && dev < 128 ? resident[dev] : 0;
  if (per_sm == 0) {
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gather_kernel<VPL>, kGatherThreads, 0);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    if (dev >= 0 && dev < 128) resident[dev] = per_sm;
  }
  int64_t blocks = (warps_needed * 32 + kGatherThreads - 1) / kGatherThreads;
  const int64_t max_blocks = int64_t(num_sms) * per_sm;
  if (blocks > max_blocks) blocks = max_blocks;
  if (blocks < 1) blocks = 1;
  return launch_kernel(gather_kernel<VPL>, dim3(unsigned(blocks)), kGatherThreads, 0, stream, 1,
                       hidden, row_stride_bytes, row_vecs, pos, pos_dim, cu_k, G, Tk, keep_idx, K,
                       K_dev, out_hidden, out_pos, out_img, out_cu, status);
}

cudaError_t launch_gather(const void* hidden, int64_t row_stride_bytes, int row_bytes,
                          const int32_t* pos, int pos_dim, const int32_t* cu_k, int G, int Tk,
                          const int32_t* keep_idx, int K, const int32_t* K_dev,
                          void* out_hidden, int32_t* out_pos, int32_t* out_img, int32_t* out_cu,
                          uint32_t* status, int num_sms, cudaStream_t stream) {
  const int row_vecs = row_bytes / 16;
  // row warps plus the boundary warps (the kernel keeps min(G + 1, warps / 16 + 1))
  const int64_t row_warps = (int64_t(K) + kGatherRows - 1) / kGatherRows;
  const int64_t warps_needed = row_warps + (G + 1 < 32 ? G + 1 : 32);
  const int vpl = (row_vecs + 31) / 32;
  const auto* h = static_cast<const uint8_t*>(hidden);
  auto* oh = static_cast<uint8_t*>(out_hidden);
#define TSEL_GATHER_CASE(N)                                                                    \
  case N:                                                                                      \
    return launch_gather_vpl<N>(num_sms, warps_needed, stream, h, row_stride_bytes, row_vecs,  \
                                pos, pos_dim, cu_k, G, Tk, keep_idx, K, K_dev, oh, out_pos,    \
                                out_img, out_cu, status);
  switch (vpl) {
    TSEL_GATHER_CASE(1)
    TSEL_GATHER_CASE(2)
    TSEL_GATHER_CASE(3)
    TSEL_GATHER_CASE(4)
    TSEL_GATHER_CASE(5)
    TSEL_GATHER_CASE(6)
    TSEL_GATHER_CASE(7)
    TSEL_GATHER_CASE(8)
    default:
      // no hidden rows (vpl 0) or rows longer than 4 KB
      return launch_gather_vpl<0>(num_sms, warps_needed, stream, h, row_stride_bytes, row_vecs,
                                  pos, pos_dim, cu_k, G, Tk, keep_idx, K, K_dev, oh, out_pos,
                                  out_img, out_cu, status);
  }
#undef TSEL_GATHER_CASE
}

}  // namespace tsel
