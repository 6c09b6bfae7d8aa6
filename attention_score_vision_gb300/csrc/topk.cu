// Pooled global top-B per request.
//
// The dynamic vision-token compression article (sections 3.2 and 3.3) puts
// every image of a request into one candidate pool and keeps the best tokens
// under one global budget; LiteVLM (section 3.2) fixes the budget through the
// keep ratio r.
//
// One CTA per request:
//   1. radix select, 8 bits per pass from the top, finds the key of the B-th
//      largest score (keys are fp32 bits mapped to an order-preserving uint32);
//   2. one pass in index order keeps every token above that key and the
//      lowest-index tokens equal to it, writing indices in ascending order
//      through block-wide prefix sums (deterministic, bit-exact).
#include <cuda_runtime.h>

#include "common.cuh"

namespace tsel {

constexpr int kTopkThreads = 1024;
constexpr int kTopkItems = 4;  // consecutive tokens per thread in the compaction pass

// fp32 bits -> uint32 with the same order; -0 maps to +0.
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ int warp_incl_scan(int x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

// Exclusive scan of one value per thread over the block; `total` gets the sum.
__device__ __forceinline__ int topk_block_scan(int v, int* warp_sums, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int x = warp_incl_scan(v);
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) warp_sums[lane] = warp_incl_scan(warp_sums[lane]);
  __syncthreads();
  const int excl = x - v + (warp > 0 ? warp_sums[warp - 1] : 0);
  total = warp_sums[31];
  __syncthreads();
  return excl;
}

__global__ void __launch_bounds__(kTopkThreads)
    topk_kernel(const float* __restrict__ scores, int total_tokens,
                const int32_t* __restrict__ req_off, int num_req,
                const int32_t* __restrict__ keep, int total_keep, int32_t* __restrict__ keep_idx,
                int32_t* __restrict__ cu_keep, uint32_t* status) {
  __shared__ int hist[256];
  __shared__ int warp_sums[32];
  __shared__ int s_base, s_bad, s_digit, s_above;
  const int r = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // Output offset of this request = sum of the budgets before it.
  int part = 0;
  int neg = 0;
  for (int i = tid; i < r; i += kTopkThreads) {
    const int b = keep[i];
    part += b;
    neg |= b < 0;
  }
  int total;
  (void)topk_block_scan(part, warp_sums, total);
  if (tid == 0) {
    const int lo = req_off[r], hi = req_off[r + 1];
    const int B = keep[r];
    int bad = 0;
    if (lo < 0 || hi < lo || hi > total_tokens || B < 0 || B > hi - lo) bad = 1;
    if (total < 0 || int64_t(total) + B > total_keep) bad = 1;
    if (r == num_req - 1 && int64_t(total) + B != total_keep) bad = 1;
    s_base = total;
    s_bad = bad;
  }
  __syncthreads();
  if (neg) atomicOr(&s_bad, 1);
  __syncthreads();
  if (s_bad) {
    if (tid == 0) set_status(status, TSEL_DEV_REQUESTS);
    return;
  }
  const int lo = req_off[r], hi = req_off[r + 1];
  const int n = hi - lo;
  const int B = keep[r];
  const int base = s_base;
  if (tid == 0) {
    if (r == 0) cu_keep[0] = 0;
    cu_keep[r + 1] = base + B;
  }
  const float* s = scores + lo;
  int32_t* out = keep_idx + base;
  if (B == 0) return;

  // ---- radix select: key of the B-th largest element --------------------
  uint32_t prefix = 0, mask = 0;
  int remaining = B;  // how many still to take among keys matching `prefix`
  int nan_seen = 0;
#pragma unroll 1
  for (int shift = 24; shift >= 0; shift -= 8) {
    if (tid < 256) hist[tid] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += kTopkThreads) {
      const float f = s[i];
      if (shift == 24) nan_seen |= (f != f);
      const uint32_t k = order_key(f);
      if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & 255u], 1);
    }
    __syncthreads();
    if (warp == 0) {
      // lane l owns bins 255-8l ... 248-8l (descending)
      int c[8];
      int sum = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = hist[255 - 8 * lane - j];
        sum += c[j];
      }
      const int incl = warp_incl_scan(sum);
      int above = incl - sum;  // count in bins above this lane's bins
      int found = -1, found_above = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (found < 0 && above < remaining && above + c[j] >= remaining) {
          found = 255 - 8 * lane - j;
          found_above = above;
        }
        above += c[j];
      }
      if (found >= 0) {
        s_digit = found;
        s_above = found_above;
      }
    }
    __syncthreads();
    prefix |= uint32_t(s_digit) << shift;
    mask |= 255u << shift;
    remaining -= s_above;
    __syncthreads();
  }
  if (nan_seen) set_status(status, TSEL_DEV_NAN);
  const uint32_t thr = prefix;
  const int need_eq = remaining;  // tokens equal to the threshold to keep

  // ---- compaction in index order ------------------------------------------
  int written = 0, eq_seen = 0;
  for (int c0 = 0; c0 < n; c0 += kTopkThreads * kTopkItems) {
    const int i0 = c0 + tid * kTopkItems;
    uint32_t k[kTopkItems];
    int n_eq = 0;
#pragma unroll
    for (int j = 0; j < kTopkItems; ++j) {
      k[j] = (i0 + j < n) ? order_key(s[i0 + j]) : 0u;
      n_eq += (i0 + j < n) && k[j] == thr;
    }
    int eq_total;
    int eq_rank = eq_seen + topk_block_scan(n_eq, warp_sums, eq_total);
    bool take[kTopkItems];
    int n_take = 0;
#pragma unroll
    for (int j = 0; j < kTopkItems; ++j) {
      const bool valid = i0 + j < n;
      bool t = valid && k[j] > thr;
      if (valid && k[j] == thr) {
        t = eq_rank < need_eq;
        ++eq_rank;
      }
      take[j] = t;
      n_take += t;
    }
    int take_total;
    int pos = written + topk_block_scan(n_take, warp_sums, take_total);
#pragma unroll
    for (int j = 0; j < kTopkItems; ++j) {
      if (take[j]) out[pos++] = lo + i0 + j;
    }
    written += take_total;
    eq_seen += eq_total;
  }
}

cudaError_t launch_topk(const float* scores, int total_tokens, const int32_t* req_off,
                        int num_req, const int32_t* keep, int total_keep, int32_t* keep_idx,
                        int32_t* cu_keep, uint32_t* status, cudaStream_t stream) {
  topk_kernel<<<num_req, kTopkThreads, 0, stream>>>(scores, total_tokens, req_off, num_req, keep,
                                                    total_keep, keep_idx, cu_keep, status);
  return cudaPeekAtLastError();
}

}  // namespace tsel
