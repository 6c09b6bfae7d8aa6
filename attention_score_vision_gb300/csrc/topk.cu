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
//   3. each CTA writes its kept indices in index order: each warp counts its
//      run of the slice's keys above and equal to the threshold, one block
//      barrier and a warp scan of those counts give every warp its output
//      slots and tie ranks, and each warp stores one coalesced word of
//      indices per 32 tokens.
// The output is deterministic and independent of the cluster size.
//
// Histogram-seeded start (fused score + select path): the column pass that
// wrote the scores also counted them per request by their first 11 and first
// 16 key bits. Every CTA reads the 2048 first-digit counts beside its slice,
// and the 32 counts under the chosen digit give the threshold's first 16
// bits, before any cluster barrier. When at most kTopkCand keys share them,
// each CTA lists its own candidates (key, index) and counts its keys above
// them in one pass over its slice; after one cluster barrier every CTA reads
// the other CTAs' counts and lists (distributed shared memory loads) and finds
// the threshold among the candidates alone: by ranking them (up to kTopkRank)
// or in two 8-bit rounds. More candidates, or counts that do not add up to
// the request's tokens, fall back to the radix rounds above (from the second
// digit, or from the first). Requests of one CTA get no histograms (their
// rounds need no cluster barrier).
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
constexpr int kTopkCacheKeys = 16384;              // keys cached in shared memory per CTA
constexpr int kTopkLoad = 8;                       // score loads in flight per thread
constexpr int kTopkCand = 2048;                    // histogram start: candidates exchanged in the cluster
constexpr int kTopkLoc = 1024;                     // histogram start: candidates listed per CTA
constexpr int kTopkRank = 256;                     // up to this many: threshold by ranking the candidates

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

struct __align__(16) TopkShared {
  int local[3][kTopkBins];    // this CTA's digit counts per round
  int merged[3][kTopkBins];   // cluster-wide counts; bin group g lives in CTA g % cluster size
  int bins[kTopkBins];        // this round's cluster-wide counts, gathered for the digit search
  int grp_sfx[kTopkGroups];   // last round: this CTA's keys in the groups above g of g's warp
  // histogram start: this CTA's candidates (keys sharing the threshold's
  // first 16 bits) and counts, read by every CTA of the cluster ...
  uint32_t loc_key[kTopkLoc];
  int loc_idx[kTopkLoc];
  int pub_gt;                     // this CTA's keys above the 16-bit prefix
  int pub_n;                      // this CTA's candidates (all, even past kTopkLoc)
  // ... and every CTA's, merged in CTA order
  __align__(16) uint32_t cand_key[kTopkCand];
  int cand_idx[kTopkCand];
  int n_of[kMaxClusterCtas];      // per CTA: its candidates
  int gt16_of[kMaxClusterCtas];   // per CTA: its keys above the candidates' 16-bit prefix
  int cls_gt[kMaxClusterCtas];    // per CTA: its candidates above the threshold
  int cls_eq[kMaxClusterCtas];    // per CTA: its candidates equal to the threshold
  int cbase[kMaxClusterCtas];     // per CTA: its first entry in the merged list
  uint32_t thr_s;                 // threshold key found by ranking
  int need_s;                     // ... and its ties still to keep
  int loc_n;
  __align__(16) int wtot[kTopkWarps];       // digit search: per-warp bin totals
  __align__(16) int gt_w[kTopkWarps];       // last round: per-warp keys above the rounds 0-1 prefix
  __align__(16) int grp_w[kTopkWarps];      // last round: per-warp totals of this CTA's counts
  int cw_gt[kTopkWarps];                    // compaction: per-warp keys above the threshold
  int cw_eq[kTopkWarps];                    // ... and equal to it
  __align__(16) long long pre_w[kTopkWarps];  // budgets of earlier requests, per warp
  int neg_w[kTopkWarps];
  int out_base, eq_before;
  int nan_seen;
  int pad_[1];
};
static_assert(sizeof(TopkShared) % 16 == 0, "key cache follows at a 16-byte boundary");

// Threshold among ncand candidate keys (ncand <= kTopkThreads, keys 16-byte
// aligned): the key with fewer than `remaining` keys above it and at least
// `remaining` at or above it; its ties all write the same values to thr_s
// and need_s (the ties still to keep). The caller separates this from the
// reads of thr_s / need_s by a block barrier.
__device__ __forceinline__ void rank_threshold(const uint32_t* keys, int ncand, int remaining,
                                               uint32_t* thr_s, int* need_s) {
  const int tid = threadIdx.x;
  if (tid >= ncand) return;
  const uint32_t ki = keys[tid];
  const uint4* ck = reinterpret_cast<const uint4*>(keys);
  int gt = 0, ge = 0;
#pragma unroll 4
  for (int j = 0; j < ncand; j += 4) {
    const uint4 v = ck[j >> 2];
    const int m = ncand - j;   // keys of this load inside the list (>= 1)
    gt += (v.x > ki) + (m > 1 && v.y > ki) + (m > 2 && v.z > ki) + (m > 3 && v.w > ki);
    ge += (v.x >= ki) + (m > 1 && v.y >= ki) + (m > 2 && v.z >= ki) + (m > 3 && v.w >= ki);
  }
  if (gt < remaining && remaining <= ge) {
    *thr_s = ki;
    *need_s = remaining - gt;
  }
}

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
  // histogram start: this request's first-digit counts (bins 4 tid .. 4 tid + 3),
  // loaded beside the flag that says whether they were built (not after it)
  const int32_t* hreq = hist != nullptr ? hist + int64_t(r) * kHistWords : nullptr;
  const int4 hc = hreq != nullptr ? __ldcg(reinterpret_cast<const int4*>(hreq) + tid)
                                  : make_int4(0, 0, 0, 0);
  const bool use_hist = hist != nullptr && *reinterpret_cast<const volatile int32_t*>(hist_ok) != 0;

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
  // the histogram start's first-digit counts are staged under the same barrier
  if (hreq != nullptr) {
    reinterpret_cast<int4*>(sh.bins)[tid] = hc;
    const int t = warp_sum(hc.x + hc.y + hc.z + hc.w);
    if (lane == 0) sh.wtot[warp] = t;
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

  // ---- histogram start: the threshold's first 16 bits from the column
  // pass's counts. Every CTA of the cluster reads the same counts, so all
  // take the same branch, before any cluster barrier. -----------------------
  uint32_t prefix = 0, mask = 0;
  int remaining = B;   // how many still to take among keys matching `prefix`
  int gt_part = 0;     // this thread's share: this CTA's keys above the prefix
  int digit = 0;
  int round0 = 0;      // first radix round still to run
  bool cand_mode = false;
  uint32_t pfx16 = 0;  // candidates: keys whose first 16 bits are pfx16
  int cnt16 = 0;
  int d0 = 0;
  uint32_t thr = 0;
  int need_eq = 0;     // tokens equal to the threshold to keep (request-wide)
  int path = 0;        // 0 radix rounds, 1 histogram + rounds, 2 candidates, 3 candidates rejected
  if (use_hist) {
    int counted = 0;
#pragma unroll
    for (int w = 0; w < kTopkWarps; w += 4) {
      const int4 v = *reinterpret_cast<const int4*>(sh.wtot + w);
      counted += v.x + v.y + v.z + v.w;
    }
    // Every token of the request counted (else the scores did not all come
    // from the column pass that built the histogram).
    if (counted == n) {
      int above0;
      d0 = find_digit(sh.bins, sh.wtot, remaining, above0);
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
        // too many candidates: radix rounds from the second digit on
        path = 1;
        round0 = 1;
        prefix = uint32_t(d0) << 21;
        mask = 0x7FFu << 21;
        remaining = rem0;
      }
    }
  }

  int nan_local = 0;
  if (cand_mode) {
    // One pass over the slice: keys cached, keys above the 16-bit prefix
    // counted, candidates (keys sharing it) listed in this CTA's own list.
    int gt16 = 0;
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
        if (i < len) {
          const uint32_t kk = order_key(f[j]);
          nan_local |= (f[j] != f[j]);
          if (cached) skeys[i] = kk;
          const uint32_t top = kk >> 16;
          if (top > pfx16) {
            ++gt16;
          } else if (top == pfx16) {
            const int slot = atomicAdd(&sh.loc_n, 1);
            if (slot < kTopkLoc) {
              sh.loc_key[slot] = kk;
              sh.loc_idx[slot] = lo + c0 + i;
            }
          }
        }
      }
    }
    if (nan_local) atomicOr(&sh.nan_seen, 1);
    gt16 = warp_sum(gt16);
    if (lane == 0) sh.gt_w[warp] = gt16;
    __syncthreads();
    if (tid == 0) {
      int g = 0;
#pragma unroll
      for (int w = 0; w < kTopkWarps; ++w) g += sh.gt_w[w];
      sh.pub_gt = g;
      sh.pub_n = sh.loc_n;   // the full count (a list that overflowed is rejected below)
    }
    // The one exchange: every CTA publishes its counts and list, then reads
    // the others' (below).
    if (!solo) {
      asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
      asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
    } else {
      __syncthreads();
    }
    // Lane l of every warp reads CTA l's counts; warp c also reads CTA c's
    // first 32 list entries (whatever the count; kept only below it). All in
    // one round trip, so each warp finds the totals and its CTA's place in
    // the merged list without a block barrier.
    int nl = 0, gl = 0;
    if (lane < csize) {
      const TopkShared* o = solo ? &sh : cluster.map_shared_rank(&sh, lane);
      nl = o->pub_n;
      gl = o->pub_gt;
    }
    const TopkShared* src = nullptr;
    uint32_t k_e = 0;
    int i_e = 0;
    if (warp < csize) {
      src = solo ? &sh : cluster.map_shared_rank(&sh, warp);
      k_e = src->loc_key[lane];
      i_e = src->loc_idx[lane];
    }
    const int c_all = warp_sum(nl);
    const int above16 = warp_sum(gl);
    const bool fit = __all_sync(0xffffffffu, nl <= kTopkLoc) && c_all <= kTopkCand;
    const int n_incl = warp_incl_scan(nl);
    if (warp == 0 && lane < kMaxClusterCtas) {
      sh.n_of[lane] = nl;
      sh.gt16_of[lane] = gl;
      sh.cbase[lane] = n_incl - nl;
    }
    if (fit && warp < csize) {
      const int n_c = __shfl_sync(0xffffffffu, nl, warp);
      const int base = __shfl_sync(0xffffffffu, n_incl - nl, warp);
      if (lane < n_c) {
        sh.cand_key[base + lane] = k_e;
        sh.cand_idx[base + lane] = i_e;
      }
      for (int x = 32 + lane; x < n_c; x += 32) {
        sh.cand_key[base + x] = src->loc_key[x];
        sh.cand_idx[base + x] = src->loc_idx[x];
      }
    }
    __syncthreads();
    // The threshold lies among the candidates when the keys above their
    // prefix (counted in the slices, not taken from the histograms) number
    // fewer than B and the candidates make up the rest; every CTA holds the
    // same counts, so every CTA takes the same branch.
    if (fit && above16 < B && B <= above16 + c_all) {
      remaining = B - above16;
      cnt16 = c_all;
      // This CTA reads no other CTA's shared memory after this point (every
      // value read is in its own shared memory, behind the block barrier
      // above, so the arrival orders nothing else); no CTA leaves before
      // every CTA has arrived here (wait at the end).
      if (!solo) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    } else {
      // radix rounds from the start
      cand_mode = false;
      path = 3;
      round0 = 0;
      prefix = 0;
      mask = 0;
      remaining = B;
    }
  }
  if (!cand_mode) {
    // Zeroed histograms are released to the cluster now; the wait comes
    // after the slice is loaded (one CTA: the block barrier below suffices).
    if (!solo) asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    for (int i0 = 0; i0 < len; i0 += kTopkThreads * kTopkLoad) {
      if (i0 > 0 || path == 3) {
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
    if (!solo) asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
    __syncthreads();
    if (path == 1) {
      for (int i = tid; i < len; i += kTopkThreads) {
        const uint32_t kk = cached ? skeys[i] : order_key(s[i]);
        gt_part += (kk >> 21) > uint32_t(d0);
      }
    }
  }

  if (tid == 0 && crank == 0) {
    // the status word heads the workspace header: count this request's path
    atomicAdd(&reinterpret_cast<WsHeader*>(status)->sel_paths[path], 1);
  }

  if (cand_mode) {
    const int ncand = cnt16;
    if (ncand <= kTopkRank) {
      rank_threshold(sh.cand_key, ncand, remaining, &sh.thr_s, &sh.need_s);
      __syncthreads();
      thr = sh.thr_s;
      need_eq = sh.need_s;
    } else {
      // Two 8-bit rounds over the candidates' low 16 bits (local[0],
      // local[1]: zeroed at entry, unused on this path).
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
    }
    // Per CTA (warp c: CTA c's entries of the merged list): its candidates
    // above and equal to the threshold, read after the compaction's barrier.
    if (warp < csize) {
      const int nc = sh.n_of[warp], bc = sh.cbase[warp];
      int g = 0, q = 0;
      for (int x = lane; x < nc; x += 32) {
        const uint32_t kk = sh.cand_key[bc + x];
        g += kk > thr;
        q += kk == thr;
      }
      g = warp_sum(g);
      q = warp_sum(q);
      if (lane == 0) {
        sh.cls_gt[warp] = g;
        sh.cls_eq[warp] = q;
      }
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
  // Warp w takes a run of whole 32-token words of the slice. One pass counts
  // the warp's keys above and equal to the threshold (ballots); after one
  // block barrier every warp scans the warps' counts itself (its output slot,
  // the ties in front of it) and a second pass writes its kept indices, one
  // coalesced store per word. The CTA's output offset and the ties in the
  // CTAs before it are found after that barrier too.
  const int span = ((len + kTopkWarps - 1) / kTopkWarps + 31) & ~31;
  const int w0 = min(len, warp * span), w1 = min(len, w0 + span);
  const unsigned lt = (1u << lane) - 1u;
  int c_gt = 0, c_eq = 0;
#pragma unroll 4
  for (int b = w0; b < w1; b += 32) {
    const int i = b + lane;
    const bool valid = i < w1;
    const uint32_t kk = valid ? (cached ? skeys[i] : order_key(s[i])) : 0u;
    c_gt += __popc(__ballot_sync(0xffffffffu, valid && kk > thr));
    c_eq += __popc(__ballot_sync(0xffffffffu, valid && kk == thr));
  }
  if (lane == 0) {
    sh.cw_gt[warp] = c_gt;
    sh.cw_eq[warp] = c_eq;
  }
  __syncthreads();
  // This CTA's output slot and the ties in the CTAs before it: from warp 0's
  // exchange on the radix path, else from every CTA's candidate counts (lane
  // c: CTA c), scanned by each warp.
  int cta_base = sh.out_base, cta_eq = sh.eq_before;
  if (cand_mode) {
    const int gc = lane < csize ? sh.gt16_of[lane] + sh.cls_gt[lane] : 0;
    const int ec = lane < csize ? sh.cls_eq[lane] : 0;
    const int ec_incl = warp_incl_scan(ec);
    const int tc = max(0, min(ec, need_eq - (ec_incl - ec)));
    const int kc_incl = warp_incl_scan(gc + tc);
    cta_base = __shfl_sync(0xffffffffu, kc_incl - (gc + tc), crank);
    cta_eq = __shfl_sync(0xffffffffu, ec_incl - ec, crank);
  }
  const int gv = lane < kTopkWarps ? sh.cw_gt[lane] : 0;
  const int ev = lane < kTopkWarps ? sh.cw_eq[lane] : 0;
  const int e_incl = warp_incl_scan(ev);
  const int e_before = cta_eq + e_incl - ev;   // ties before warp `lane`'s run
  const int take = max(0, min(ev, need_eq - e_before));
  const int k_incl = warp_incl_scan(gv + take);
  int pos = cta_base + __shfl_sync(0xffffffffu, k_incl - (gv + take), warp);
  int eqb = __shfl_sync(0xffffffffu, e_before, warp);
  int32_t* out = keep_idx + before;
#pragma unroll 2
  for (int b = w0; b < w1; b += 32) {
    const int i = b + lane;
    const bool valid = i < w1;
    const uint32_t kk = valid ? (cached ? skeys[i] : order_key(s[i])) : 0u;
    const bool eq = valid && kk == thr;
    const unsigned em = __ballot_sync(0xffffffffu, eq);
    const bool kept = (valid && kk > thr) || (eq && eqb + __popc(em & lt) < need_eq);
    const unsigned km = __ballot_sync(0xffffffffu, kept);
    const int p = pos + __popc(km & lt);
    // (stores stay inside the request's B slots whatever the counts said)
    if (kept && p < B) out[p] = lo + c0 + i;
    pos += __popc(km);
    eqb += __popc(em);
  }
  if (!solo) asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
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
