// Dynamic keep budget per request from its score distribution.
//
// The dynamic vision-token compression article names a content-dependent
// compression ratio as future work (section 6.2) and notes that images differ
// in how much pruning they tolerate; LiteVLM (section 3.2) fixes one keep
// ratio. Rule used here: keep the fewest top tokens (score descending, lowest
// index first) whose scores hold a fraction tau of the request's total score,
// bounded by a floor and a ceiling ratio. Scores enter as integer quanta
// q = floor(s * 2^(24 - E)), E the binary exponent with the request's largest
// score in [2^(E-1), 2^E): every sum is exact and independent of the order
// in which threads add, so the budget is deterministic.
//
// One thread-block cluster per request (up to 16 CTAs, one slice of the
// request each, its keys cached in shared memory): the slice maxima meet in
// CTA 0 (distributed shared memory) and give E; then four 8-bit radix rounds
// over the order-preserving score keys build (count, quanta) histograms, bin
// b merged in CTA (b % cluster size), from which every CTA picks the same
// digit. The first
// round's histogram also gives the request total M and the target T. After
// the last round the key of the token that crosses T is known exactly; the
// tokens tied on it carry equal quanta, so the number of them needed is one
// division.
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include "launch_util.cuh"
#include "common.cuh"

namespace cg = cooperative_groups;

namespace tsel {

constexpr int kBudgetThreads = 256;
constexpr int kBudgetWarps = kBudgetThreads / 32;
constexpr int kBudgetCacheKeys = 16384;    // keys cached in shared memory per CTA

// Binary exponent E with s in [2^(E-1), 2^E) for a positive fp32 bit pattern.
__device__ __forceinline__ int score_exponent(uint32_t bits) {
  const uint32_t ex = bits >> 23, mant = bits & 0x7FFFFFu;
  if (ex != 0) return int(ex) - 126;
  return (32 - __clz(int(mant))) - 149;   // subnormal
}

// floor(s * 2^(24 - E)) for the bits of a positive fp32 s <= the request max.
__device__ __forceinline__ uint32_t score_quantum(uint32_t bits, int E) {
  const uint32_t ex = bits >> 23, mant = bits & 0x7FFFFFu;
  const uint32_t m = ex != 0 ? (mant | 0x800000u) : mant;   // s = m * 2^e2
  const int e2 = (ex != 0 ? int(ex) : 1) - 150;
  const int sh = e2 + 24 - E;
  if (m == 0) return 0u;
  if (sh >= 0) return sh >= 24 ? 0u : (m << sh);   // the result stays below 2^24
  return sh <= -32 ? 0u : (m >> (-sh));
}

// Quantum of the score behind an order key: NaN, negative and zero count 0.
__device__ __forceinline__ uint32_t quantum_of_key(uint32_t key, int E) {
  if (key <= 0x80000000u) return 0u;                 // negative scores and +-0
  const uint32_t bits = key & 0x7FFFFFFFu;
  if (bits > 0x7F800000u) return 0u;                 // NaN
  return score_quantum(bits, E);
}

struct BudgetShared {
  int cnt[4][256];                   // merged histograms (bin b lives in CTA b % csize)
  unsigned long long mass[4][256];
  int lcnt[256];                     // this CTA's histogram of the current round
  unsigned long long lmass[256];
  uint32_t red[kBudgetWarps];
  uint32_t smax;                     // CTA 0: largest positive score bits of the request
  int bad, nan_seen, digit, cnt_above;
  unsigned long long mass_above, target;
};

__global__ void __launch_bounds__(kBudgetThreads)
    budget_cluster_kernel(const float* __restrict__ scores, int total_tokens,
                          const int32_t* __restrict__ req_off, int mass_pm, int min_pm,
                          int max_pm, int32_t* __restrict__ keep_out, int32_t* total_out,
                          uint32_t* status) {
  __shared__ BudgetShared sh;
  extern __shared__ uint32_t skeys[];   // kBudgetCacheKeys
  cg::cluster_group cluster = cg::this_cluster();
  const int crank = int(cluster.block_rank());
  const int csize = int(cluster.num_blocks());
  const int r = int(blockIdx.x) / csize;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_launch_dependents();
  pdl_wait();

  const int lo = req_off[r], hi = req_off[r + 1];
  if (tid == 0) {
    sh.bad = (lo < 0 || hi < lo || hi > total_tokens) ? 1 : 0;
    sh.nan_seen = 0;
    sh.smax = 0u;
  }
  for (int i = tid; i < 4 * 256; i += kBudgetThreads) {
    (&sh.cnt[0][0])[i] = 0;
    (&sh.mass[0][0])[i] = 0ull;
  }
  __syncthreads();
  if (sh.bad) {
    // every CTA of the cluster takes this branch together (same request)
    if (tid == 0 && crank == 0) {
      set_status(status, TSEL_DEV_REQUESTS);
      keep_out[r] = 0;
    }
    return;
  }
  const int n = hi - lo;
  const int chunk = (n + csize - 1) / csize;
  const int c0 = min(n, crank * chunk), c1 = min(n, c0 + chunk);
  const int len = c1 - c0;
  const float* s = scores + lo + c0;
  const bool cached = len <= kBudgetCacheKeys;
  // CTA 0's histograms and max are zeroed before any remote update: arrive
  // now, wait after the slice is loaded.
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  uint32_t mx = 0;
  int nan_local = 0;
  for (int i0 = 0; i0 < len; i0 += kBudgetThreads * 8) {
    float f[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {   // eight independent loads in flight per thread
      const int i = i0 + j * kBudgetThreads + tid;
      f[j] = i < len ? __ldcg(s + i) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = i0 + j * kBudgetThreads + tid;
      nan_local |= (f[j] != f[j]);
      if (f[j] > 0.f) mx = max(mx, __float_as_uint(f[j]));
      if (cached && i < len) skeys[i] = order_key(f[j]);
    }
  }
  mx = __reduce_max_sync(0xffffffffu, mx);
  if (lane == 0) sh.red[warp] = mx;
  if (nan_local) atomicOr(&sh.nan_seen, 1);
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
  __syncthreads();
  uint32_t* smax0 = cluster.map_shared_rank(&sh.smax, 0);
  if (tid == 0) {
    uint32_t m = 0;
    for (int w = 0; w < kBudgetWarps; ++w) m = max(m, sh.red[w]);
    if (m) atomicMax(smax0, m);
  }
  cluster.sync();
  const uint32_t smax_bits = *smax0;
  const int E = smax_bits != 0 ? score_exponent(smax_bits) : 0;

  // ---- radix rounds on the score key, (count, quanta) histograms ---------
  uint32_t prefix = 0, mask = 0;
  unsigned long long need = 0;   // quanta still to collect among keys matching prefix
  int cnt_above = 0;
  bool done = smax_bits == 0;    // no positive score: nothing to collect
#pragma unroll 1
  for (int round = 0; round < 4 && !done; ++round) {
    const int shift = 24 - 8 * round;
    for (int i = tid; i < 256; i += kBudgetThreads) {
      sh.lcnt[i] = 0;
      sh.lmass[i] = 0ull;
    }
    __syncthreads();
    for (int i0 = 0; i0 < len; i0 += kBudgetThreads) {
      const int i = i0 + tid;
      const bool in = i < len;
      const uint32_t k = in ? (cached ? skeys[i] : order_key(__ldcg(s + i))) : 0u;
      const bool match = in && (k & mask) == prefix;
      const uint32_t d = (k >> shift) & 255u;
      const uint32_t q = match ? quantum_of_key(k, E) : 0u;
      // one shared atomic per distinct digit of the warp; quanta < 2^24, so
      // a group's sum fits 32 bits
      const uint32_t peers = __match_any_sync(0xffffffffu, match ? d : 0x100u);
      const uint32_t gsum = __reduce_add_sync(peers, q);
      if (match && (__ffs(peers) - 1) == lane) {
        atomicAdd(&sh.lcnt[d], __popc(peers));
        atomicAdd(&sh.lmass[d], (unsigned long long)gsum);
      }
    }
    __syncthreads();
    for (int b = tid; b < 256; b += kBudgetThreads) {
      if (sh.lcnt[b]) {   // bin b is merged in CTA b % csize
        atomicAdd(cluster.map_shared_rank(&sh.cnt[round][b], b % csize), sh.lcnt[b]);
        atomicAdd(cluster.map_shared_rank(&sh.mass[round][b], b % csize), sh.lmass[b]);
      }
    }
    cluster.sync();
    if (warp == 0) {
      // lane l owns bins 255-8l ... 248-8l (descending)
      unsigned long long m8[8], msum = 0;
      int c8[8], csum = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int b = 255 - 8 * lane - j;
        m8[j] = *cluster.map_shared_rank(&sh.mass[round][b], b % csize);
        c8[j] = *cluster.map_shared_rank(&sh.cnt[round][b], b % csize);
        msum += m8[j];
        csum += c8[j];
      }
      unsigned long long mi = msum;
      int ci = csum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xffffffffu, mi, o);
        const int yc = __shfl_up_sync(0xffffffffu, ci, o);
        if (lane >= o) {
          mi += y;
          ci += yc;
        }
      }
      if (round == 0) {
        // request total = every bin of the first round; T = ceil(tau * M)
        const unsigned long long M = __shfl_sync(0xffffffffu, mi, 31);
        const unsigned long long a = M / 1000ull, b = M % 1000ull;
        const unsigned long long T = a * (unsigned long long)mass_pm +
                                     (b * (unsigned long long)mass_pm + 999ull) / 1000ull;
        if (lane == 0) sh.target = T;
        need = T;
      }
      unsigned long long m_before = mi - msum;
      int c_before = ci - csum;
      int found = -1;
      unsigned long long f_mass = 0;
      int f_cnt = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (found < 0 && m_before < need && m_before + m8[j] >= need) {
          found = 255 - 8 * lane - j;
          f_mass = m_before;
          f_cnt = c_before;
        }
        m_before += m8[j];
        c_before += c8[j];
      }
      if (found >= 0) {
        sh.digit = found;
        sh.mass_above = f_mass;
        sh.cnt_above = f_cnt;
      }
    }
    __syncthreads();
    if (round == 0) {
      need = sh.target;
      if (need == 0) {
        done = true;
        break;
      }
    }
    prefix |= uint32_t(sh.digit) << shift;
    mask |= 255u << shift;
    need -= sh.mass_above;
    cnt_above += sh.cnt_above;
    __syncthreads();
  }
  if (tid == 0 && sh.nan_seen) set_status(status, TSEL_DEV_NAN);   // this CTA's slice
  if (tid == 0 && crank == 0) {
    long long b_dyn = 0;
    if (!done) {
      // every token left on the threshold key carries the same quantum
      const uint32_t qs = quantum_of_key(prefix, E);
      const unsigned long long k = qs > 0 ? (need + qs - 1) / qs : 0ull;
      b_dyn = (long long)cnt_above + (long long)k;
    }
    const long long floor_b = (long long)n * min_pm / 1000;
    const long long ceil_b = (long long)n * max_pm / 1000;
    if (b_dyn < floor_b) b_dyn = floor_b;
    if (b_dyn > ceil_b) b_dyn = ceil_b;
    keep_out[r] = int32_t(b_dyn);
    if (total_out != nullptr) atomicAdd(total_out, int32_t(b_dyn));
  }
  cluster.sync();   // no CTA's shared memory is read remotely after this point
}

cudaError_t launch_budget(const float* scores, int total_tokens, const int32_t* req_off,
                          int num_req, int mass_pm, int min_pm, int max_pm, int32_t* keep_out,
                          int32_t* total_out, uint32_t* status, cudaStream_t stream) {
  static int cache[128][5] = {};
  if (total_out != nullptr) {
    cudaError_t e = cudaMemsetAsync(total_out, 0, sizeof(int32_t), stream);
    if (e != cudaSuccess) return e;
  }
  const size_t dyn = size_t(kBudgetCacheKeys) * sizeof(uint32_t);
  cudaError_t e = cudaSuccess;
  const int csize = usable_cluster_size(budget_cluster_kernel,
                                        cluster_size_for(total_tokens, num_req), kBudgetThreads,
                                        dyn, cache, &e);
  if (e != cudaSuccess) return e;
  return launch_clusters(budget_cluster_kernel, num_req, csize, kBudgetThreads, dyn, stream,
                         scores, total_tokens, req_off, mass_pm, min_pm, max_pm, keep_out,
                         total_out, status);
}

}  // namespace tsel
