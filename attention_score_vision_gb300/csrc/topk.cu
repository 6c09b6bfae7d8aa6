// Pooled global top-B per request.
//
// The dynamic vision-token compression article (sections 3.2 and 3.3) puts
// every image of a request into one candidate pool and keeps the best tokens
// under one global budget; LiteVLM (section 3.2) fixes the budget through the
// keep ratio r.
//
// One thread-block cluster per request (up to 16 CTAs, one slice of the
// request's tokens each, cached in shared memory):
//   1. radix select, 8 bits per round from the top: every CTA builds
//      warp-private histograms of its slice and adds bin b into CTA
//      (b % cluster size) through distributed shared memory (the merge is
//      spread over the cluster); after one cluster barrier every CTA reads the
//      merged bins and picks the same digit. After four rounds the key of the
//      B-th largest score is known (keys are fp32 bits mapped to an
//      order-preserving uint32);
//   2. each CTA's counts of keys above / equal to that key follow from its
//      own per-round histograms; they are sent to every CTA, and each CTA
//      writes its kept indices in index order through block-wide prefix sums:
//      tokens above the key, and the lowest-index tokens equal to it. The
//      output is deterministic.
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include "launch_util.cuh"
#include "common.cuh"

namespace cg = cooperative_groups;

namespace tsel {

constexpr int kTopkThreads = 512;
static_assert(kTopkThreads >= 256, "one thread per histogram bin");
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kTopkItems = 16;              // consecutive tokens per thread when compacting
constexpr int kTopkMaxCluster = kMaxClusterCtas;
constexpr int kTopkCacheKeys = 16384;       // keys cached in shared memory per CTA

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
  if (warp == 0) {
    const int w = lane < kTopkWarps ? warp_sums[lane] : 0;
    const int s = warp_incl_scan(w);
    if (lane < kTopkWarps) warp_sums[lane] = s;
  }
  __syncthreads();
  const int excl = x - v + (warp > 0 ? warp_sums[warp - 1] : 0);
  total = warp_sums[kTopkWarps - 1];
  __syncthreads();
  return excl;
}

struct TopkShared {
  int whist[kTopkWarps][256];      // warp-private histograms
  int hist[4][256];                // merged histograms (bin b lives in CTA b % csize)
  int cnt_gt[kTopkMaxCluster];     // every CTA's counts above / equal to the threshold
  int cnt_eq[kTopkMaxCluster];
  int warp_sums[32];
  int digit, above, bad, nan_seen;
};

__global__ void __launch_bounds__(kTopkThreads)
    topk_cluster_kernel(const float* __restrict__ scores, int total_tokens,
                        const int32_t* __restrict__ req_off, int num_req,
                        const int32_t* __restrict__ keep, int total_keep,
                        int32_t* __restrict__ keep_idx, int32_t* __restrict__ cu_keep,
                        uint32_t* status) {
  __shared__ TopkShared sh;
  extern __shared__ uint32_t skeys[];  // kTopkCacheKeys
  cg::cluster_group cluster = cg::this_cluster();
  const int crank = int(cluster.block_rank());
  const int csize = int(cluster.num_blocks());
  const int r = int(blockIdx.x) / csize;
  const bool solo = csize == 1;   // one CTA: plain block barriers, no exchange
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_launch_dependents();
  pdl_wait();

  // ---- request checks and output offset (identical in every CTA) --------
  int part = 0, neg = 0;
  for (int i = tid; i < r; i += kTopkThreads) {
    const int b = keep[i];
    part += b;
    neg |= b < 0;
  }
  int before;
  (void)topk_block_scan(part, sh.warp_sums, before);
  const int lo = req_off[r], hi = req_off[r + 1];
  const int B = keep[r];
  if (tid == 0) {
    int bad = neg;
    if (lo < 0 || hi < lo || hi > total_tokens || B < 0 || B > hi - lo) bad = 1;
    if (before < 0) bad = 1;
    if (total_keep >= 0) {
      if (int64_t(before) + B > total_keep) bad = 1;
      if (r == num_req - 1 && int64_t(before) + B != total_keep) bad = 1;
    } else if (int64_t(before) + B > total_tokens) {
      bad = 1;   // budgets from the device: keep_idx has room for total_tokens entries
    }
    sh.bad = bad;
    sh.nan_seen = 0;
  }
  for (int i = tid; i < 4 * 256; i += kTopkThreads) (&sh.hist[0][0])[i] = 0;
  if (tid < kTopkMaxCluster) {
    sh.cnt_gt[tid] = 0;
    sh.cnt_eq[tid] = 0;
  }
  __syncthreads();
  if (sh.bad) {
    // every CTA of the cluster takes this branch together (same request)
    if (tid == 0 && crank == 0) set_status(status, TSEL_DEV_REQUESTS);
    return;
  }
  if (tid == 0 && crank == 0) {
    if (r == 0) cu_keep[0] = 0;
    cu_keep[r + 1] = before + B;
  }
  const int n = hi - lo;
  if (B == 0) return;

  // This CTA's slice of the request.
  const int chunk = (n + csize - 1) / csize;
  const int c0 = min(n, crank * chunk), c1 = min(n, c0 + chunk);
  const int len = c1 - c0;
  const float* s = scores + lo + c0;
  const bool cached = len <= kTopkCacheKeys;
  // Histograms are zeroed everywhere before any remote add: arrive now, wait
  // after the slice is loaded.
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  int nan_local = 0;
  for (int i0 = 0; i0 < len; i0 += kTopkThreads * 8) {
    float f[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {   // eight independent loads in flight per thread
      const int i = i0 + j * kTopkThreads + tid;
      f[j] = i < len ? __ldcg(s + i) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = i0 + j * kTopkThreads + tid;
      nan_local |= (f[j] != f[j]);
      if (cached && i < len) skeys[i] = order_key(f[j]);
    }
  }
  if (nan_local) atomicOr(&sh.nan_seen, 1);
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
  __syncthreads();

  // ---- radix select -------------------------------------------------------
  // Bin b of each round is merged in CTA (b % csize), so the merge spreads
  // over the cluster instead of queueing at one SM. Thread t keeps this
  // CTA's count of bin t, from which the counts above / at the threshold
  // follow without another pass over the keys.
  uint32_t prefix = 0, mask = 0;
  int remaining = B;  // how many still to take among keys matching `prefix`
  int gt_part = 0, eq_part = 0;   // this CTA: keys above / equal to the threshold (bin tid)
#pragma unroll 1
  for (int round = 0; round < 4; ++round) {
    const int shift = 24 - 8 * round;
    for (int i = tid; i < kTopkWarps * 256; i += kTopkThreads) (&sh.whist[0][0])[i] = 0;
    __syncthreads();
    for (int i0 = 0; i0 < len; i0 += kTopkThreads) {
      const int i = i0 + tid;
      const bool in = i < len;
      const uint32_t k = in ? (cached ? skeys[i] : order_key(s[i])) : 0u;
      const bool match = in && (k & mask) == prefix;
      const uint32_t d = (k >> shift) & 255u;
      // aggregate equal digits within the warp: one shared atomic per value
      const uint32_t peers = __match_any_sync(0xffffffffu, match ? d : 0x100u);
      if (match && (__ffs(peers) - 1) == lane) atomicAdd(&sh.whist[warp][d], __popc(peers));
    }
    __syncthreads();
    int v = 0;   // this CTA's count of bin tid (threads >= 256 hold no bin)
    if (tid < 256) {
#pragma unroll
      for (int w = 0; w < kTopkWarps; ++w) v += sh.whist[w][tid];
    }
    if (solo) {
      if (tid < 256) sh.hist[round][tid] = v;
      __syncthreads();
    } else {
      if (v) atomicAdd(cluster.map_shared_rank(&sh.hist[round][tid], tid % csize), v);
      cluster.sync();
    }
    if (warp == 0) {
      // lane l owns bins 255-8l ... 248-8l (descending)
      int c[8];
      int sum = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int b = 255 - 8 * lane - j;
        c[j] = solo ? sh.hist[round][b] : *cluster.map_shared_rank(&sh.hist[round][b], b % csize);
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
        sh.digit = found;
        sh.above = found_above;
      }
    }
    __syncthreads();
    const int digit = sh.digit;
    gt_part += tid > digit ? v : 0;
    if (round == 3) eq_part = tid == digit ? v : 0;
    prefix |= uint32_t(digit) << shift;
    mask |= 255u << shift;
    remaining -= sh.above;
    __syncthreads();
  }
  if (tid == 0 && sh.nan_seen) set_status(status, TSEL_DEV_NAN);   // this CTA's slice
  const uint32_t thr = prefix;
  const int need_eq = remaining;  // tokens equal to the threshold to keep (request-wide)

  // ---- per-CTA counts, sent to every CTA of the cluster ----------------------
  if (!solo) {
    int gt_total, eq_total;
    (void)topk_block_scan(gt_part, sh.warp_sums, gt_total);
    (void)topk_block_scan(eq_part, sh.warp_sums, eq_total);
    if (tid < csize) {
      *cluster.map_shared_rank(&sh.cnt_gt[crank], tid) = gt_total;
      *cluster.map_shared_rank(&sh.cnt_eq[crank], tid) = eq_total;
    }
    cluster.sync();   // no CTA reads another CTA's shared memory after this point
  }
  if (solo) {
    if (tid == 0) {
      sh.above = 0;
      sh.digit = 0;
    }
  } else if (warp == 0) {
    // lane c: CTA c's counts; exclusive prefixes give this CTA's output slot
    const int e = lane < csize ? sh.cnt_eq[lane] : 0;
    const int g = lane < csize ? sh.cnt_gt[lane] : 0;
    const int e_incl = warp_incl_scan(e);
    const int e_before = e_incl - e;
    const int take = max(0, min(e, need_eq - e_before));
    const int t_incl = warp_incl_scan(g + take);
    if (lane == crank) {
      sh.above = t_incl - (g + take);   // output slots of CTAs before this one
      sh.digit = e_before;              // tied tokens in CTAs before this one
    }
  }
  __syncthreads();
  const int out_base = sh.above, eq_before = sh.digit;

  // ---- compaction in index order --------------------------------------------
  // kTopkItems consecutive tokens per thread; one block scan per pass gives
  // both the tied tokens (for their rank) and the tokens above the threshold
  // in front of each thread (16-bit halves: a pass has <= 4096 tokens).
  int32_t* out = keep_idx + before + out_base;
  int written = 0, eq_seen = eq_before;
  for (int i0 = 0; i0 < len; i0 += kTopkThreads * kTopkItems) {
    const int ib = i0 + tid * kTopkItems;
    uint32_t k[kTopkItems];
    if (cached && ib + kTopkItems <= len) {
#pragma unroll
      for (int j = 0; j < kTopkItems; j += 4) {
        const uint4 v = *reinterpret_cast<const uint4*>(skeys + ib + j);
        k[j] = v.x;
        k[j + 1] = v.y;
        k[j + 2] = v.z;
        k[j + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < kTopkItems; ++j) {
        const int i = ib + j;
        k[j] = i < len ? (cached ? skeys[i] : order_key(s[i])) : 0u;
      }
    }
    int n_eq = 0, n_gt = 0;
#pragma unroll
    for (int j = 0; j < kTopkItems; ++j) {
      const bool valid = ib + j < len;
      n_eq += valid && k[j] == thr;
      n_gt += valid && k[j] > thr;
    }
    int tot;
    const int pre = topk_block_scan((n_eq << 16) | n_gt, sh.warp_sums, tot);
    int eq_rank = eq_seen + (pre >> 16);
    int pos = written + (pre & 0xFFFF) + max(0, min(pre >> 16, need_eq - eq_seen));
#pragma unroll
    for (int j = 0; j < kTopkItems; ++j) {
      const bool valid = ib + j < len;
      bool t = valid && k[j] > thr;
      if (valid && k[j] == thr) {
        t = eq_rank < need_eq;
        ++eq_rank;
      }
      if (t) out[pos++] = lo + c0 + ib + j;
    }
    const int tot_eq = tot >> 16, tot_gt = tot & 0xFFFF;
    written += tot_gt + max(0, min(tot_eq, need_eq - eq_seen));
    eq_seen += tot_eq;
  }
}

cudaError_t launch_topk(const float* scores, int total_tokens, const int32_t* req_off,
                        int num_req, const int32_t* keep, int total_keep, int32_t* keep_idx,
                        int32_t* cu_keep, uint32_t* status, cudaStream_t stream) {
  static int cache[128][5] = {};
  const size_t dyn = size_t(kTopkCacheKeys) * sizeof(uint32_t);
  cudaError_t e = cudaSuccess;
  const int csize = usable_cluster_size(topk_cluster_kernel,
                                        cluster_size_for(total_tokens, num_req), kTopkThreads,
                                        dyn, cache, &e);
  if (e != cudaSuccess) return e;
  return launch_clusters(topk_cluster_kernel, num_req, csize, kTopkThreads, dyn, stream, scores,
                         total_tokens, req_off, num_req, keep, total_keep, keep_idx, cu_keep,
                         status);
}

}  // namespace tsel
