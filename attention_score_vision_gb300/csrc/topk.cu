// Pooled global top-B per request.
//
// The dynamic vision-token compression article (sections 3.2 and 3.3) puts
// every image of a request into one candidate pool and keeps the best tokens
// under one global budget; LiteVLM (section 3.2) fixes the budget through the
// keep ratio r.
//
// One thread-block cluster per request (up to 16 CTAs, one slice of the
// request's tokens each, cached in shared memory; keys are fp32 bits mapped
// to an order-preserving uint32):
//   1. radix select in three rounds of 11, 11 and 10 bits from the top. Every
//      CTA counts the digits of its slice's still-matching keys into a
//      2048-bin histogram (shared atomics); group g of four bins is added
//      into CTA (g % cluster size) through distributed shared memory, so the
//      merge spreads over the cluster. After one cluster barrier each thread
//      gathers its four merged bins, and after one block barrier every warp
//      finds the digit holding the B-th largest key on its own (warp totals,
//      then the groups of one warp, then the bins of one group; bins
//      descending). After the last round the key of the B-th largest score
//      and the number of tokens equal to it still to keep are known;
//   2. before the last cluster barrier each CTA publishes, per warp and per
//      bin group of the last round, its counts of keys above the first two
//      rounds' prefix and in higher groups. After the barrier one warp of
//      each CTA reads every CTA's counts at the chosen digit, so the output
//      offset needs no further exchange;
//   3. each CTA writes its kept indices in index order: per pass of 4096
//      tokens one block-wide prefix sum gives every thread's slots (tokens
//      above the key, and the lowest-index tokens equal to it), the indices
//      are staged in shared memory and stored with coalesced writes.
// The output is deterministic and independent of the cluster size.
//
// Histogram-seeded start (fused score + select path): the column pass that
// wrote the scores also counted them per request by their first 11 and first
// 16 key bits. The top-B then reads the 2048 first-digit counts with its
// slice (no first round), and the 32 counts under the chosen digit give the
// threshold's first 16 bits. When at most kTopkCand keys share them, every
// CTA sends those candidates (key, index) and its count of keys above them to
// every CTA of the cluster: one cluster barrier, after which each CTA finds
// the threshold among the candidates alone (two 8-bit rounds in shared
// memory, block barriers only) and knows its output offset. More candidates,
// or counts that do not add up to the request's tokens, fall back to the
// radix rounds above (from the second digit, or from the first). Requests of
// one CTA get no histograms (their rounds need no cluster barrier).
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include "launch_util.cuh"
#include "common.cuh"

namespace cg = cooperative_groups;

namespace tsel {

constexpr int kTopkThreads = 512;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kTopkBins = 2048;                    // 11-bit digits (the last round uses 1024)
constexpr int kTopkGroups = kTopkBins / 4;         // one group of four bins per thread
static_assert(kTopkGroups == kTopkThreads, "one bin group per thread");
constexpr int kTopkItems = 8;                      // consecutive tokens per thread when compacting
constexpr int kTopkPass = kTopkThreads * kTopkItems;   // tokens per compaction pass (<= 65535)
constexpr int kTopkCacheKeys = 16384;              // keys cached in shared memory per CTA
constexpr int kTopkLoad = 8;                       // score loads in flight per thread
constexpr int kTopkCand = 2048;                    // histogram start: candidates exchanged in the cluster
static_assert(2 * kTopkCand <= kTopkPass, "candidates are staged in the compaction stage buffer");

// Digit of round `round` (0, 1, 2): bits 31..21, 20..10, 9..0.
__device__ __forceinline__ int topk_shift(int round) { return round == 0 ? 21 : (round == 1 ? 10 : 0); }
__device__ __forceinline__ uint32_t topk_dmask(int round) { return round == 2 ? 1023u : 2047u; }

__device__ __forceinline__ int warp_incl_scan(int x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

// Sum over this lane and the lanes above it.
__device__ __forceinline__ int warp_suffix_scan(int x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_down_sync(0xffffffffu, x, o);
    if (lane + o < 32) x += y;
  }
  return x;
}

__device__ __forceinline__ int warp_sum(int x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Exclusive scan of one value per thread over the block; `total` gets the
// sum. One block barrier: every warp adds the totals of the warps below it.
// The caller separates two calls by a barrier (warp_sums is rewritten).
__device__ __forceinline__ int topk_block_scan(int v, int* warp_sums, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int x = warp_incl_scan(v);
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  int below = 0, all = 0;
#pragma unroll
  for (int i = 0; i < kTopkWarps; i += 4) {
    const int4 w = *reinterpret_cast<const int4*>(warp_sums + i);
    below += (i < warp ? w.x : 0) + (i + 1 < warp ? w.y : 0) + (i + 2 < warp ? w.z : 0) +
             (i + 3 < warp ? w.w : 0);
    all += w.x + w.y + w.z + w.w;
  }
  total = all;
  return x - v + below;
}

// Sum of w[i] over the warps i > warp (16 per-warp values).
__device__ __forceinline__ int sum_warps_above(const int* w, int warp) {
  int s = 0;
#pragma unroll
  for (int i = 0; i < kTopkWarps; i += 4) {
    const int4 v = *reinterpret_cast<const int4*>(w + i);
    s += (i > warp ? v.x : 0) + (i + 1 > warp ? v.y : 0) + (i + 2 > warp ? v.z : 0) +
         (i + 3 > warp ? v.w : 0);
  }
  return s;
}

struct __align__(16) TopkShared {
  int local[3][kTopkBins];    // this CTA's digit counts per round
  int merged[3][kTopkBins];   // cluster-wide counts; bin group g lives in CTA g % cluster size
  int bins[kTopkBins];        // this round's cluster-wide counts, gathered for the digit search
  int grp_sfx[kTopkGroups];   // last round: this CTA's keys in the groups above g of g's warp
  int stage[kTopkPass];       // kept indices of one compaction pass
  // histogram start: every CTA's candidates (keys sharing the threshold's
  // first 16 bits) and per-CTA counts, written by the CTAs that hold them
  uint32_t cand_key[kTopkCand];
  int cand_idx[kTopkCand];
  int gt16_of[kMaxClusterCtas];   // per CTA: its keys above the candidates' 16-bit prefix
  int cls_gt[kMaxClusterCtas];    // per CTA: its candidates above the threshold
  int cls_eq[kMaxClusterCtas];    // per CTA: its candidates equal to the threshold
  int cbase[kMaxClusterCtas];     // this CTA's first slot in each CTA's candidate list
  int cand_n, loc_n;
  __align__(16) int wtot[kTopkWarps];       // digit search: per-warp bin totals
  __align__(16) int gt_w[kTopkWarps];       // last round: per-warp keys above the rounds 0-1 prefix
  __align__(16) int grp_w[kTopkWarps];      // last round: per-warp totals of this CTA's counts
  __align__(16) int warp_sums[kTopkWarps];  // compaction scan
  __align__(16) long long pre_w[kTopkWarps];  // budgets of earlier requests, per warp
  int neg_w[kTopkWarps];
  int out_base, eq_before;
  int nan_seen;
  int pad_[1];
};
static_assert(sizeof(TopkShared) % 16 == 0, "key cache follows at a 16-byte boundary");

// Finds the bin holding the `remaining`-th largest key, bins descending, in
// every warp at once (no further block barrier): the warp totals give the
// warp whose bin groups hold it, that warp's 32 groups give the group, the
// group's four bins give the bin. Returns the digit; `above` gets the keys
// in higher bins. wtot[w] = sum of the bins of groups 32w .. 32w+31.
__device__ __forceinline__ int find_digit(const int* bins, const int* wtot, int remaining,
                                          int& above) {
  const int lane = threadIdx.x & 31;
  const int v = lane < kTopkWarps ? wtot[lane] : 0;
  const int xs = warp_suffix_scan(v);
  const unsigned hw = __ballot_sync(0xffffffffu, lane < kTopkWarps && xs - v < remaining && xs >= remaining);
  const int w = hw ? __ffs(hw) - 1 : 0;
  const int above_w = __shfl_sync(0xffffffffu, xs - v, w);
  const int4 c = reinterpret_cast<const int4*>(bins)[32 * w + lane];
  const int sum4 = c.x + c.y + c.z + c.w;
  const int xg = warp_suffix_scan(sum4);
  const int a0 = above_w + xg - sum4;   // keys in groups above this lane's
  const unsigned hg = __ballot_sync(0xffffffffu, a0 < remaining && a0 + sum4 >= remaining);
  const int g = hg ? __ffs(hg) - 1 : 0;
  int a = __shfl_sync(0xffffffffu, a0, g);
  const int cw = __shfl_sync(0xffffffffu, c.w, g), cz = __shfl_sync(0xffffffffu, c.z, g);
  const int cy = __shfl_sync(0xffffffffu, c.y, g);
  const int base = 4 * (32 * w + g);
  int digit;
  if (a + cw >= remaining) {
    digit = base + 3;
  } else if ((a += cw) + cz >= remaining) {
    digit = base + 2;
  } else if ((a += cz) + cy >= remaining) {
    digit = base + 1;
  } else {
    a += cy;
    digit = base;
  }
  above = a;
  return digit;
}

// find_digit over 256 bins (the candidates' last two rounds): lane l holds
// bins 8l .. 8l + 7. Every warp finds the same digit.
__device__ __forceinline__ int find_digit256(const int* bins, int remaining, int& above) {
  const int lane = threadIdx.x & 31;
  const int4 lo4 = reinterpret_cast<const int4*>(bins)[2 * lane];
  const int4 hi4 = reinterpret_cast<const int4*>(bins)[2 * lane + 1];
  const int b[8] = {lo4.x, lo4.y, lo4.z, lo4.w, hi4.x, hi4.y, hi4.z, hi4.w};
  const int sum8 = lo4.x + lo4.y + lo4.z + lo4.w + hi4.x + hi4.y + hi4.z + hi4.w;
  const int xs = warp_suffix_scan(sum8);
  const int a0 = xs - sum8;   // keys in the bins of higher lanes
  const unsigned hb = __ballot_sync(0xffffffffu, a0 < remaining && xs >= remaining);
  const int g = hb ? __ffs(hb) - 1 : 0;
  int a = __shfl_sync(0xffffffffu, a0, g);
  int bg[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) bg[j] = __shfl_sync(0xffffffffu, b[j], g);
  int digit = 8 * g;
#pragma unroll
  for (int j = 7; j >= 0; --j) {
    if (a + bg[j] >= remaining) {
      digit = 8 * g + j;
      break;
    }
    a += bg[j];
  }
  above = a;
  return digit;
}

__global__ void __launch_bounds__(kTopkThreads)
    topk_cluster_kernel(const float* __restrict__ scores, int total_tokens,
                        const int32_t* __restrict__ req_off, int num_req,
                        const int32_t* __restrict__ keep, int total_keep,
                        int32_t* __restrict__ keep_idx, int32_t* __restrict__ cu_keep,
                        uint32_t* status, const int32_t* hist, const int32_t* hist_ok,
                        int inputs_final) {
  extern __shared__ __align__(16) unsigned char topk_smem[];
  TopkShared& sh = *reinterpret_cast<TopkShared*>(topk_smem);
  uint32_t* skeys = reinterpret_cast<uint32_t*>(topk_smem + sizeof(TopkShared));  // kTopkCacheKeys
  cg::cluster_group cluster = cg::this_cluster();
  const int crank = int(cluster.block_rank());
  const int csize = int(cluster.num_blocks());
  const int r = int(blockIdx.x) / csize;
  const bool solo = csize == 1;   // one CTA: no distributed shared memory, no cluster barrier
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // Histograms start at zero in every CTA before any remote add (the first
  // cluster barrier below orders the two). `local` and `merged` are adjacent.
  {
    int4* h = reinterpret_cast<int4*>(&sh.local[0][0]);
    for (int i = tid; i < 6 * kTopkBins / 4; i += kTopkThreads) h[i] = make_int4(0, 0, 0, 0);
    if (tid < kMaxClusterCtas) {
      sh.gt16_of[tid] = 0;
      sh.cls_gt[tid] = 0;
      sh.cls_eq[tid] = 0;
    }
    if (tid == 0) {
      sh.nan_seen = 0;
      sh.cand_n = 0;
      sh.loc_n = 0;
      sh.out_base = 0;
      sh.eq_before = 0;
    }
  }
  // The request's offsets and budget: read before the wait for the scores
  // when no kernel still running may write them (the fused score + select
  // call: its schedule kernel released its dependents after the caller's
  // earlier work had completed), else after it.
  int lo_raw = 0, hi_raw = 0, B = 0;
  if (inputs_final) {
    lo_raw = req_off[r];
    hi_raw = req_off[r + 1];
    B = keep[r];
  }
  pdl_wait();
  if (!inputs_final) {
    lo_raw = req_off[r];
    hi_raw = req_off[r + 1];
    B = keep[r];
  }

  // ---- this CTA's slice; its first scores in flight during the checks ------
  const int lo = min(max(lo_raw, 0), total_tokens);
  const int hi = min(max(hi_raw, lo), total_tokens);
  const int n = hi - lo;
  const int chunk = (n + csize - 1) / csize;
  const int c0 = min(n, crank * chunk), c1 = min(n, c0 + chunk);
  const int len = c1 - c0;
  const float* s = scores + lo + c0;
  const bool cached = len <= kTopkCacheKeys;
  float f[kTopkLoad];
#pragma unroll
  for (int j = 0; j < kTopkLoad; ++j) {
    const int i = j * kTopkThreads + tid;
    f[j] = i < len ? __ldcg(s + i) : 0.f;
  }
  // histogram start: this request's first-digit counts (bins 4 tid .. 4 tid + 3)
  const bool use_hist = hist != nullptr && *reinterpret_cast<const volatile int32_t*>(hist_ok) != 0;
  const int32_t* hreq = use_hist ? hist + int64_t(r) * kHistWords : nullptr;
  const int4 hc = use_hist ? __ldcg(reinterpret_cast<const int4*>(hreq) + tid) : make_int4(0, 0, 0, 0);

  // ---- request checks and output offset (every thread, every CTA alike) ----
  long long part = 0;
  int neg = 0;
  for (int i = tid; i < r; i += kTopkThreads) {
    const int b = keep[i];
    part += b;
    neg |= b < 0;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
  neg = __any_sync(0xffffffffu, neg);
  if (lane == 0) {
    sh.pre_w[warp] = part;
    sh.neg_w[warp] = neg;
  }
  __syncthreads();
  long long before64 = 0;
  bool bad = false;
#pragma unroll
  for (int w = 0; w < kTopkWarps; ++w) {
    before64 += sh.pre_w[w];
    bad |= sh.neg_w[w] != 0;
  }
  if (lo_raw < 0 || hi_raw < lo_raw || hi_raw > total_tokens || B < 0 || B > hi_raw - lo_raw)
    bad = true;
  if (total_keep >= 0) {
    if (before64 + B > total_keep) bad = true;
    if (r == num_req - 1 && before64 + B != total_keep) bad = true;
  } else if (before64 + B > total_tokens) {
    bad = true;   // budgets from the device: keep_idx has room for total_tokens entries
  }
  if (bad) {
    // every CTA of the cluster takes this branch together (same request)
    if (tid == 0 && crank == 0) set_status(status, TSEL_DEV_REQUESTS);
    return;
  }
  const int before = int(before64);
  if (tid == 0 && crank == 0) {
    if (r == 0) cu_keep[0] = 0;
    cu_keep[r + 1] = before + B;
  }
  if (B == 0) return;

  // Zeroed histograms are released to the cluster now; the wait comes after
  // the slice is loaded.
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  int nan_local = 0;
  for (int i0 = 0; i0 < len; i0 += kTopkThreads * kTopkLoad) {
    if (i0 > 0) {
#pragma unroll
      for (int j = 0; j < kTopkLoad; ++j) {
        const int i = i0 + j * kTopkThreads + tid;
        f[j] = i < len ? __ldcg(s + i) : 0.f;
      }
    }
#pragma unroll
    for (int j = 0; j < kTopkLoad; ++j) {
      const int i = i0 + j * kTopkThreads + tid;
      nan_local |= (f[j] != f[j]);
      if (cached && i < len) skeys[i] = order_key(f[j]);
    }
  }
  if (nan_local) atomicOr(&sh.nan_seen, 1);
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
  __syncthreads();

  // ---- threshold -----------------------------------------------------------
  uint32_t prefix = 0, mask = 0;
  int remaining = B;   // how many still to take among keys matching `prefix`
  int gt_part = 0;     // this thread's share: this CTA's keys above the prefix
  int digit = 0;
  int round0 = 0;      // first radix round still to run
  bool cand_mode = false;
  uint32_t pfx16 = 0;  // candidates: keys whose first 16 bits are pfx16
  int cnt16 = 0;
  uint32_t thr = 0;
  int need_eq = 0;     // tokens equal to the threshold to keep (request-wide)
  int path = 0;        // 0 radix rounds, 1 histogram + rounds, 2 candidates, 3 candidates rejected
  if (use_hist) {
    reinterpret_cast<int4*>(sh.bins)[tid] = hc;
    const int t = warp_sum(hc.x + hc.y + hc.z + hc.w);
    if (lane == 0) sh.wtot[warp] = t;
    __syncthreads();
    int counted = 0;
#pragma unroll
    for (int w = 0; w < kTopkWarps; w += 4) {
      const int4 v = *reinterpret_cast<const int4*>(sh.wtot + w);
      counted += v.x + v.y + v.z + v.w;
    }
    // Every token of the request counted (else the scores did not all come
    // from the column pass that built the histogram): the same outcome in
    // every CTA of the cluster, which all read the same counts.
    if (counted == n) {
      int above0;
      const int d0 = find_digit(sh.bins, sh.wtot, remaining, above0);
      const int rem0 = remaining - above0;
      // the 32 first-16-bit bins under d0, bins descending = lanes descending
      const int fb = __ldcg(hreq + kHistCoarse + d0 * 32 + lane);
      const int xs = warp_suffix_scan(fb);
      const unsigned hb = __ballot_sync(0xffffffffu, xs - fb < rem0 && xs >= rem0);
      const int d1 = hb ? __ffs(hb) - 1 : 0;
      cnt16 = __shfl_sync(0xffffffffu, fb, d1);
      if (cnt16 <= kTopkCand) {
        cand_mode = true;   // (remaining is set from the exchanged counts)
        path = 2;
        pfx16 = (uint32_t(d0) << 5) | uint32_t(d1);
      } else {
        path = 1;
        // too many candidates: radix rounds from the second digit on
        round0 = 1;
        prefix = uint32_t(d0) << 21;
        mask = 0x7FFu << 21;
        remaining = rem0;
        for (int i = tid; i < len; i += kTopkThreads) {
          const uint32_t kk = cached ? skeys[i] : order_key(s[i]);
          gt_part += (kk >> 21) > uint32_t(d0);
        }
      }
    }
  }

  if (cand_mode) {
    // This CTA's keys above the 16-bit prefix, and its candidates (staged in
    // the compaction buffer: keys, then indices).
    int gt16 = 0;
    for (int i = tid; i < len; i += kTopkThreads) {
      const uint32_t kk = cached ? skeys[i] : order_key(s[i]);
      const uint32_t top = kk >> 16;
      if (top > pfx16) {
        ++gt16;
      } else if (top == pfx16) {
        const int slot = atomicAdd(&sh.loc_n, 1);
        if (slot < kTopkCand) {
          sh.stage[slot] = int(kk);
          sh.stage[kTopkCand + slot] = lo + c0 + i;
        }
      }
    }
    gt16 = warp_sum(gt16);
    if (lane == 0) sh.gt_w[warp] = gt16;
    __syncthreads();
    const int nloc = min(sh.loc_n, kTopkCand);
    if (tid < csize) {
      int gsum = 0;
#pragma unroll
      for (int w = 0; w < kTopkWarps; ++w) gsum += sh.gt_w[w];
      // the full count (a CTA with more candidates than fit stores only the
      // first kTopkCand; the total then exceeds the list and is rejected below)
      int* cn = solo ? &sh.cand_n : cluster.map_shared_rank(&sh.cand_n, tid);
      sh.cbase[tid] = atomicAdd(cn, sh.loc_n);
      int* g16 = solo ? &sh.gt16_of[crank] : cluster.map_shared_rank(&sh.gt16_of[crank], tid);
      *g16 = gsum;
    }
    __syncthreads();
    for (int j = 0; j < csize; ++j) {
      const int base = sh.cbase[j];
      uint32_t* dk = solo ? sh.cand_key : cluster.map_shared_rank(sh.cand_key, j);
      int* di = solo ? sh.cand_idx : cluster.map_shared_rank(sh.cand_idx, j);
      for (int t = tid; t < nloc && base + t < kTopkCand; t += kTopkThreads) {
        dk[base + t] = uint32_t(sh.stage[t]);
        di[base + t] = sh.stage[kTopkCand + t];
      }
    }
    // The one exchange: after it no CTA touches another's shared memory.
    if (!solo) cluster.sync();
    __syncthreads();
    // The threshold lies among the candidates when the keys above their
    // prefix (counted in the slices, not taken from the histograms) number
    // fewer than B and the candidates make up the rest; every CTA holds the
    // same counts, so every CTA takes the same branch.
    int above16 = 0;
    for (int c = 0; c < csize; ++c) above16 += sh.gt16_of[c];
    if (sh.cand_n <= kTopkCand && above16 < B && B <= above16 + sh.cand_n) {
      remaining = B - above16;
      cnt16 = sh.cand_n;
    } else {
      // radix rounds from the start
      cand_mode = false;
      path = 3;
      round0 = 0;
      prefix = 0;
      mask = 0;
      remaining = B;
      gt_part = 0;
    }
  }

  if (tid == 0 && crank == 0) {
    // the status word heads the workspace header: count this request's path
    atomicAdd(&reinterpret_cast<WsHeader*>(status)->sel_paths[path], 1);
  }

  if (cand_mode) {
    // The threshold among the candidates: two 8-bit rounds over their low
    // 16 bits (local[0], local[1]: zeroed at entry, unused on this path).
    const int ncand = cnt16;
    int* binsA = sh.local[0];
    int* binsB = sh.local[1];
    for (int i = tid; i < ncand; i += kTopkThreads) atomicAdd(&binsA[(sh.cand_key[i] >> 8) & 255u], 1);
    __syncthreads();
    int aboveA;
    const int dA = find_digit256(binsA, remaining, aboveA);
    remaining -= aboveA;
    const uint32_t pfx24 = (pfx16 << 8) | uint32_t(dA);
    for (int i = tid; i < ncand; i += kTopkThreads) {
      const uint32_t kk = sh.cand_key[i];
      if ((kk >> 8) == pfx24) atomicAdd(&binsB[kk & 255u], 1);
    }
    __syncthreads();
    int aboveB;
    const int dB = find_digit256(binsB, remaining, aboveB);
    remaining -= aboveB;
    thr = (pfx24 << 8) | uint32_t(dB);
    need_eq = remaining;
    // per CTA (the slice holding the index): candidates above / equal to thr
    for (int i = tid; i < ncand; i += kTopkThreads) {
      const uint32_t kk = sh.cand_key[i];
      if (kk >= thr) {
        const int src = min(csize - 1, (sh.cand_idx[i] - lo) / chunk);
        atomicAdd(kk > thr ? &sh.cls_gt[src] : &sh.cls_eq[src], 1);
      }
    }
    __syncthreads();
    if (tid == 0) {
      int base = 0, eqb = 0;
      for (int c = 0; c < crank; ++c) {
        const int take = max(0, min(sh.cls_eq[c], need_eq - eqb));
        base += sh.gt16_of[c] + sh.cls_gt[c] + take;
        eqb += sh.cls_eq[c];
      }
      sh.out_base = base;     // read after the compaction's first block barrier
      sh.eq_before = eqb;
    }
    if (tid == 0 && sh.nan_seen) set_status(status, TSEL_DEV_NAN);   // this CTA's slice
    pdl_launch_dependents();
  } else {
#pragma unroll 1
  for (int round = round0; round < 3; ++round) {
    const int shift = topk_shift(round);
    const uint32_t dmask = topk_dmask(round);
    int* loc = sh.local[round];
    if (round == 2 && !solo) {
      const int g = warp_sum(gt_part);
      if (lane == 0) sh.gt_w[warp] = g;
    }
    for (int i0 = 0; i0 < len; i0 += kTopkThreads * kTopkLoad) {
      uint32_t kk[kTopkLoad];
#pragma unroll
      for (int j = 0; j < kTopkLoad; ++j) {
        const int i = i0 + j * kTopkThreads + tid;
        kk[j] = i < len ? (cached ? skeys[i] : order_key(s[i])) : 0u;
      }
#pragma unroll
      for (int j = 0; j < kTopkLoad; ++j) {
        const bool match = i0 + j * kTopkThreads + tid < len && (kk[j] & mask) == prefix;
        if (match) atomicAdd(&loc[(kk[j] >> shift) & dmask], 1);
      }
    }
    __syncthreads();
    const int4 lv = reinterpret_cast<const int4*>(loc)[tid];   // bins 4 tid .. 4 tid + 3
    const int* bins = loc;
    if (!solo) {
      int* mrg = sh.merged[round];
      int* dst = cluster.map_shared_rank(mrg + 4 * tid, tid % csize);
      if (lv.x) atomicAdd(dst, lv.x);
      if (lv.y) atomicAdd(dst + 1, lv.y);
      if (lv.z) atomicAdd(dst + 2, lv.z);
      if (lv.w) atomicAdd(dst + 3, lv.w);
      if (round == 2) {
        // published for the other CTAs' output offsets (read after the barrier)
        const int sum4 = lv.x + lv.y + lv.z + lv.w;
        const int x = warp_suffix_scan(sum4);
        sh.grp_sfx[tid] = x - sum4;
        if (lane == 0) sh.grp_w[warp] = x;
      }
      cluster.sync();
      const int4 c = *reinterpret_cast<const int4*>(cluster.map_shared_rank(mrg + 4 * tid, tid % csize));
      reinterpret_cast<int4*>(sh.bins)[tid] = c;
      const int t = warp_sum(c.x + c.y + c.z + c.w);
      if (lane == 0) sh.wtot[warp] = t;
      bins = sh.bins;
    } else {
      const int t = warp_sum(lv.x + lv.y + lv.z + lv.w);
      if (lane == 0) sh.wtot[warp] = t;
    }
    __syncthreads();
    int above;
    digit = find_digit(bins, sh.wtot, remaining, above);
    if (round < 2) {
      const int b0 = 4 * tid;
      gt_part += (b0 > digit ? lv.x : 0) + (b0 + 1 > digit ? lv.y : 0) +
                 (b0 + 2 > digit ? lv.z : 0) + (b0 + 3 > digit ? lv.w : 0);
    }
    prefix |= uint32_t(digit) << shift;
    mask |= dmask << shift;
    remaining -= above;
  }
  if (tid == 0 && sh.nan_seen) set_status(status, TSEL_DEV_NAN);   // this CTA's slice
  // The compaction kernel that follows may launch now: its CTAs would only
  // wait on this request's SMs during the rounds.
  pdl_launch_dependents();
  thr = prefix;
  need_eq = remaining;

  // ---- output offset: the other CTAs' counts at the chosen digit -------------
  if (!solo) {
    if (warp == 0) {
      const int g = digit >> 2, j = digit & 3;
      int gt = 0, eq = 0;
      if (lane < csize) {
        const TopkShared* o = cluster.map_shared_rank(&sh, lane);
        int tot = 0;
#pragma unroll
        for (int w = 0; w < kTopkWarps; w += 4) {
          const int4 a = *reinterpret_cast<const int4*>(o->gt_w + w);
          const int4 b = *reinterpret_cast<const int4*>(o->grp_w + w);
          tot += a.x + a.y + a.z + a.w;
          const int gw = g >> 5;
          tot += (w > gw ? b.x : 0) + (w + 1 > gw ? b.y : 0) + (w + 2 > gw ? b.z : 0) +
                 (w + 3 > gw ? b.w : 0);
        }
        const int4 l = *reinterpret_cast<const int4*>(&o->local[2][4 * g]);
        gt = tot + o->grp_sfx[g] + (j < 3 ? l.w : 0) + (j < 2 ? l.z : 0) + (j < 1 ? l.y : 0);
        eq = j == 3 ? l.w : (j == 2 ? l.z : (j == 1 ? l.y : l.x));
      }
      // lane c: CTA c's counts; exclusive prefixes give this CTA's output slot
      const int e_incl = warp_incl_scan(eq);
      const int e_before = e_incl - eq;
      const int take = max(0, min(eq, need_eq - e_before));
      const int t_incl = warp_incl_scan(gt + take);
      if (lane == crank) {
        sh.out_base = t_incl - (gt + take);   // output slots of CTAs before this one
        sh.eq_before = e_before;              // tied tokens in CTAs before this one
      }
    }
    // This CTA reads no other CTA's shared memory after this point; no CTA
    // leaves before every CTA has arrived here (wait at the end).
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  }
  }

  // ---- compaction in index order --------------------------------------------
  // kTopkItems consecutive tokens per thread; one block scan per pass gives
  // both the tied tokens (for their rank) and the tokens above the threshold
  // in front of each thread (16-bit halves: a pass has <= 4096 tokens). The
  // output offset written by warp 0 above is read after the first scan's
  // barrier.
  int32_t* out = keep_idx + before;
  int written = 0, eq_seen = 0, room = B;
  for (int i0 = 0; i0 < len; i0 += kTopkPass) {
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
    if (i0 == 0) {   // (0 for one CTA on the radix-round path)
      out += sh.out_base;
      room = B - sh.out_base;
      eq_seen = sh.eq_before;
    }
    int eq_rank = eq_seen + (pre >> 16);
    int pos = (pre & 0xFFFF) + max(0, min(pre >> 16, need_eq - eq_seen));
#pragma unroll
    for (int j = 0; j < kTopkItems; ++j) {
      const bool valid = ib + j < len;
      bool t = valid && k[j] > thr;
      if (valid && k[j] == thr) {
        t = eq_rank < need_eq;
        ++eq_rank;
      }
      if (t) sh.stage[pos++] = lo + c0 + ib + j;
    }
    const int tot_eq = tot >> 16, tot_gt = tot & 0xFFFF;
    const int cnt = tot_gt + max(0, min(tot_eq, need_eq - eq_seen));
    __syncthreads();
    // (every thread has read warp_sums and the stage is read here before the
    // next pass's first barrier, so the next pass may rewrite both)
    // (stores stay inside the request's B slots whatever the counts said)
    for (int i = tid; i < cnt && written + i < room; i += kTopkThreads) out[written + i] = sh.stage[i];
    written += cnt;
    eq_seen += tot_eq;
  }
  if (!solo && !cand_mode) asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

// Per-request histograms of given scores (tsel_select_topk_hist), into a
// zeroed region: one warp per 32 consecutive tokens. Every CTA checks the
// request offsets itself (ordered, inside the tokens) and adds nothing when
// they are not; CTA 0 records the outcome for the top-B that follows.
constexpr int kHistThreads = 256;

__global__ void __launch_bounds__(kHistThreads)
    topk_hist_kernel(const float* __restrict__ scores, int total_tokens,
                     const int32_t* __restrict__ req_off, int R, int32_t* hist, int32_t* hist_ok) {
  __shared__ int ok_s;
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (warp == 0) {
    bool ok = R >= 1 && R <= kHistMaxReq;
    for (int r = lane; ok && r <= R; r += 32) {
      const int o = __ldg(req_off + r);
      const int prev = r > 0 ? __ldg(req_off + r - 1) : 0;
      if (o < prev || o > total_tokens) ok = false;
    }
    ok = __all_sync(0xffffffffu, ok);
    if (lane == 0) {
      ok_s = ok ? 1 : 0;
      if (blockIdx.x == 0) *hist_ok = ok_s;
    }
  }
  __syncthreads();
  if (!ok_s) return;
  const int64_t warps = int64_t(gridDim.x) * (kHistThreads / 32);
  for (int64_t w = int64_t(blockIdx.x) * (kHistThreads / 32) + warp; w * 32 < total_tokens; w += warps) {
    const int tok = int(w * 32) + lane;
    const bool valid = tok < total_tokens;
    const float sc = valid ? __ldcg(scores + tok) : 0.f;
    hist_add_warp(hist, req_off, R, tok, sc, valid);
  }
}

cudaError_t launch_topk_hist(const float* scores, int total_tokens, const int32_t* req_off, int R,
                             int32_t* hist, int32_t* hist_ok, int num_sms, cudaStream_t stream) {
  const int64_t warps = (int64_t(total_tokens) + 31) / 32;
  int64_t blocks = (warps + kHistThreads / 32 - 1) / (kHistThreads / 32);
  if (blocks > 4 * int64_t(num_sms)) blocks = 4 * int64_t(num_sms);
  if (blocks < 1) blocks = 1;
  return launch_kernel(topk_hist_kernel, dim3(unsigned(blocks)), kHistThreads, 0, stream, 1, scores,
                       total_tokens, req_off, R, hist, hist_ok);
}

static const size_t kTopkDyn = sizeof(TopkShared) + size_t(kTopkCacheKeys) * sizeof(uint32_t);

// CTAs per request of the top-B launch for these sizes (1: one CTA each,
// for which the radix rounds cost no cluster barrier and the histogram
// start does not pay).
int topk_cluster_size(int total_tokens, int num_req, cudaError_t* e) {
  static int cache[128][5] = {};
  *e = cudaSuccess;
  const int want = cluster_size_for(total_tokens, num_req);
  return cluster_size_for_grid(topk_cluster_kernel, want, num_req, kTopkThreads, kTopkDyn, cache, e);
}

cudaError_t launch_topk(const float* scores, int total_tokens, const int32_t* req_off,
                        int num_req, const int32_t* keep, int total_keep, int32_t* keep_idx,
                        int32_t* cu_keep, uint32_t* status, const int32_t* hist,
                        const int32_t* hist_ok, int inputs_final, cudaStream_t stream) {
  const size_t dyn = kTopkDyn;
  cudaError_t e = cudaSuccess;
  const int csize = topk_cluster_size(total_tokens, num_req, &e);
  if (e != cudaSuccess) return e;
  return launch_clusters(topk_cluster_kernel, num_req, csize, kTopkThreads, dyn, stream, scores,
                         total_tokens, req_off, num_req, keep, total_keep, keep_idx, cu_keep,
                         status, hist, hist_ok, inputs_final);
}

}  // namespace tsel
