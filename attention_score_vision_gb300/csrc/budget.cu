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
// every CTA through distributed shared memory and give E; then three radix
// rounds of 11, 11 and 10 bits over the order-preserving score keys build
// (count, quanta) histograms of 2048 bins (shared atomics), bin group g
// (four bins) merged in CTA (g % cluster size). After one cluster barrier
// each thread gathers its merged group, and after one block barrier every
// warp finds the digit on its own (warp totals, then the groups of one
// warp, then the bins of one group; bins descending). The first round's
// totals also give the request total M and the target T. After the last
// round the key of the token that crosses T is known exactly; the tokens
// tied on it carry equal quanta, so the number of them needed is one
// division.
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include "launch_util.cuh"
#include "common.cuh"

namespace cg = cooperative_groups;

namespace tsel {


constexpr int kBudgetThreads = 512;
constexpr int kBudgetWarps = kBudgetThreads / 32;
constexpr int kBudgetBins = 2048;                // 11-bit digits (the last round uses 1024)
static_assert(kBudgetBins / 4 == kBudgetThreads, "one bin group per thread");
constexpr int kBudgetCacheKeys = 16384;          // keys cached in shared memory per CTA
constexpr int kBudgetLoad = 8;                   // score loads in flight per thread

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

// Digit of round `round` (0, 1, 2): bits 31..21, 20..10, 9..0 of the key.
__device__ __forceinline__ int budget_shift(int round) { return round == 0 ? 21 : (round == 1 ? 10 : 0); }
__device__ __forceinline__ uint32_t budget_dmask(int round) { return round == 2 ? 1023u : 2047u; }

template <typename T>
__device__ __forceinline__ T budget_warp_sum(T x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Sum over this lane and the lanes above it.
template <typename T>
__device__ __forceinline__ T budget_suffix_scan(T x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const T y = __shfl_down_sync(0xffffffffu, x, o);
    if (lane + o < 32) x += y;
  }
  return x;
}

// Quanta sums are 64-bit but kept as two 32-bit words (low, high): a sum is
// added with a native 32-bit atomic on the low word that returns the old
// value, and the carry it produces goes into the high word. Once every add
// has landed, high * 2^32 + low is the exact sum. Every key adds its own
// count and quantum (no warp grouping: on the seeded scores that was slower
// in every round, and in later rounds, where a warp's digits are mostly
// distinct, it serialised).
__device__ __forceinline__ void add_u64_split(uint32_t* lo, uint32_t* hi, unsigned long long x) {
  const uint32_t xl = uint32_t(x), xh = uint32_t(x >> 32);
  const uint32_t old = atomicAdd(lo, xl);
  const uint32_t up = xh + (old + xl < old ? 1u : 0u);
  if (up) atomicAdd(hi, up);
}

__device__ __forceinline__ unsigned long long join_u64(uint32_t lo, uint32_t hi) {
  return (static_cast<unsigned long long>(hi) << 32) | lo;
}

struct __align__(16) BudgetShared {
  uint32_t lmlo[kBudgetBins];                 // this CTA's quanta per digit (current round)
  uint32_t lmhi[kBudgetBins];
  uint32_t mmlo[3][kBudgetBins];              // merged; bin group g lives in CTA g % csize
  uint32_t mmhi[3][kBudgetBins];
  unsigned long long bmass[kBudgetBins];      // the round's merged quanta, gathered
  int lcnt[kBudgetBins];                      // this CTA's token count per digit
  int mcnt[3][kBudgetBins];
  int bcnt[kBudgetBins];
  unsigned long long wmass[kBudgetWarps];     // per-warp totals of the gathered bins
  int wcnt[kBudgetWarps];
  uint32_t wmax[kBudgetWarps];                // per-warp largest positive score bits
  uint32_t cmax[kMaxClusterCtas];             // every CTA's slice maximum
  int nan_seen;
  int pad_[3];
};
static_assert(sizeof(BudgetShared) % 16 == 0, "key cache follows at a 16-byte boundary");

// Finds, in every warp at once, the bin (descending) where the quanta of the
// higher bins plus its own first reach `need`. Returns the digit; mass_above
// and cnt_above get the quanta and the tokens of the higher bins.
__device__ __forceinline__ int budget_find_digit(const BudgetShared& sh, unsigned long long need,
                                                 unsigned long long& mass_above, int& cnt_above) {
  const int lane = threadIdx.x & 31;
  const unsigned long long vm = lane < kBudgetWarps ? sh.wmass[lane] : 0ull;
  const int vc = lane < kBudgetWarps ? sh.wcnt[lane] : 0;
  const unsigned long long xm = budget_suffix_scan(vm);
  const int xc = budget_suffix_scan(vc);
  const unsigned hw = __ballot_sync(0xffffffffu, lane < kBudgetWarps && xm - vm < need && xm >= need);
  const int w = hw ? __ffs(hw) - 1 : 0;
  const unsigned long long am_w = __shfl_sync(0xffffffffu, xm - vm, w);
  const int ac_w = __shfl_sync(0xffffffffu, xc - vc, w);
  const int grp = 32 * w + lane;
  const int4 c4 = reinterpret_cast<const int4*>(sh.bcnt)[grp];
  const ulonglong2 m01 = reinterpret_cast<const ulonglong2*>(sh.bmass)[2 * grp];
  const ulonglong2 m23 = reinterpret_cast<const ulonglong2*>(sh.bmass)[2 * grp + 1];
  const unsigned long long sm = m01.x + m01.y + m23.x + m23.y;
  const int sc = c4.x + c4.y + c4.z + c4.w;
  const unsigned long long xg = budget_suffix_scan(sm);
  const int xgc = budget_suffix_scan(sc);
  const unsigned long long a0 = am_w + xg - sm;
  const int a0c = ac_w + xgc - sc;
  const unsigned hg = __ballot_sync(0xffffffffu, a0 < need && a0 + sm >= need);
  const int g = hg ? __ffs(hg) - 1 : 0;
  unsigned long long a = __shfl_sync(0xffffffffu, a0, g);
  int ac = __shfl_sync(0xffffffffu, a0c, g);
  const unsigned long long m3 = __shfl_sync(0xffffffffu, m23.y, g);
  const unsigned long long m2 = __shfl_sync(0xffffffffu, m23.x, g);
  const unsigned long long m1 = __shfl_sync(0xffffffffu, m01.y, g);
  const int k3 = __shfl_sync(0xffffffffu, c4.w, g), k2 = __shfl_sync(0xffffffffu, c4.z, g);
  const int k1 = __shfl_sync(0xffffffffu, c4.y, g);
  const int base = 4 * (32 * w + g);
  int digit;
  if (a + m3 >= need) {
    digit = base + 3;
  } else {
    a += m3;
    ac += k3;
    if (a + m2 >= need) {
      digit = base + 2;
    } else {
      a += m2;
      ac += k2;
      if (a + m1 >= need) {
        digit = base + 1;
      } else {
        a += m1;
        ac += k1;
        digit = base;
      }
    }
  }
  mass_above = a;
  cnt_above = ac;
  return digit;
}

__global__ void __launch_bounds__(kBudgetThreads, 1)
    budget_cluster_kernel(const float* __restrict__ scores, int total_tokens,
                          const int32_t* __restrict__ req_off, int mass_pm, int min_pm,
                          int max_pm, int32_t* __restrict__ keep_out, int32_t* total_out,
                          uint32_t* status) {
  extern __shared__ __align__(16) unsigned char budget_smem[];
  BudgetShared& sh = *reinterpret_cast<BudgetShared*>(budget_smem);
  uint32_t* skeys = reinterpret_cast<uint32_t*>(budget_smem + sizeof(BudgetShared));
  cg::cluster_group cluster = cg::this_cluster();
  const int crank = int(cluster.block_rank());
  const int csize = int(cluster.num_blocks());
  const int r = int(blockIdx.x) / csize;
  const bool solo = csize == 1;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // Histograms start at zero before any remote add (ordered by the first
  // cluster barrier below).
  {
    int4* h = reinterpret_cast<int4*>(&sh.lmlo[0]);
    constexpr int n16 = int((offsetof(BudgetShared, wmass)) / 16);
    for (int i = tid; i < n16; i += kBudgetThreads) h[i] = make_int4(0, 0, 0, 0);
    if (tid == 0) sh.nan_seen = 0;
  }
  pdl_wait();

  const int lo = req_off[r], hi = req_off[r + 1];
  if (lo < 0 || hi < lo || hi > total_tokens) {
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
  // Zeroed histograms released to the cluster now; the wait (which also
  // makes sure every CTA runs before any remote access) follows the loads.
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  uint32_t mx = 0;
  int nan_local = 0;
  for (int i0 = 0; i0 < len; i0 += kBudgetThreads * kBudgetLoad) {
    float f[kBudgetLoad];
#pragma unroll
    for (int j = 0; j < kBudgetLoad; ++j) {
      const int i = i0 + j * kBudgetThreads + tid;
      f[j] = i < len ? __ldcg(s + i) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < kBudgetLoad; ++j) {
      const int i = i0 + j * kBudgetThreads + tid;
      nan_local |= (f[j] != f[j]);
      if (f[j] > 0.f) mx = max(mx, __float_as_uint(f[j]));
      if (cached && i < len) skeys[i] = order_key(f[j]);
    }
  }
  mx = __reduce_max_sync(0xffffffffu, mx);
  if (lane == 0) sh.wmax[warp] = mx;
  if (nan_local) atomicOr(&sh.nan_seen, 1);
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
  __syncthreads();
  // this slice's maximum into slot crank of every CTA
  if (warp == 0) {
    uint32_t m = lane < kBudgetWarps ? sh.wmax[lane] : 0u;
    m = __reduce_max_sync(0xffffffffu, m);
    if (lane < csize) *cluster.map_shared_rank(&sh.cmax[crank], lane) = m;
  }
  cluster.sync();
  uint32_t smax_bits = 0;
  for (int c = 0; c < csize; ++c) smax_bits = max(smax_bits, sh.cmax[c]);
  const int E = smax_bits != 0 ? score_exponent(smax_bits) : 0;

  // ---- radix rounds on the score key, (count, quanta) histograms ---------
  uint32_t prefix = 0, mask = 0;
  unsigned long long need = 0;   // quanta still to collect among keys matching prefix
  int cnt_above = 0;
  bool done = smax_bits == 0;    // no positive score: nothing to collect (same in every CTA)
#pragma unroll 1
  for (int round = 0; round < 3 && !done; ++round) {
    const int shift = budget_shift(round);
    const uint32_t dmask = budget_dmask(round);
    for (int i0 = 0; i0 < len; i0 += kBudgetThreads * kBudgetLoad) {
      uint32_t kk[kBudgetLoad];
#pragma unroll
      for (int j = 0; j < kBudgetLoad; ++j) {
        const int i = i0 + j * kBudgetThreads + tid;
        kk[j] = i < len ? (cached ? skeys[i] : order_key(__ldcg(s + i))) : 0u;
      }
#pragma unroll
      for (int j = 0; j < kBudgetLoad; ++j) {
        const bool match = i0 + j * kBudgetThreads + tid < len && (kk[j] & mask) == prefix;
        const uint32_t d = (kk[j] >> shift) & dmask;
        if (match) {
          atomicAdd(&sh.lcnt[d], 1);
          const uint32_t q = quantum_of_key(kk[j], E);
          if (q) add_u64_split(&sh.lmlo[d], &sh.lmhi[d], q);
        }
      }
    }
    __syncthreads();
    // this thread's group: read, re-zero for the next round, merge
    int4 c4 = reinterpret_cast<const int4*>(sh.lcnt)[tid];
    uint4 lo4 = reinterpret_cast<const uint4*>(sh.lmlo)[tid];
    uint4 hi4 = reinterpret_cast<const uint4*>(sh.lmhi)[tid];
    reinterpret_cast<int4*>(sh.lcnt)[tid] = make_int4(0, 0, 0, 0);
    reinterpret_cast<uint4*>(sh.lmlo)[tid] = make_uint4(0u, 0u, 0u, 0u);
    reinterpret_cast<uint4*>(sh.lmhi)[tid] = make_uint4(0u, 0u, 0u, 0u);
    if (!solo) {
      const int owner = tid % csize;
      int* dc = cluster.map_shared_rank(&sh.mcnt[round][4 * tid], owner);
      uint32_t* dlo = cluster.map_shared_rank(&sh.mmlo[round][4 * tid], owner);
      uint32_t* dhi = cluster.map_shared_rank(&sh.mmhi[round][4 * tid], owner);
      if (c4.x) atomicAdd(dc, c4.x);
      if (c4.y) atomicAdd(dc + 1, c4.y);
      if (c4.z) atomicAdd(dc + 2, c4.z);
      if (c4.w) atomicAdd(dc + 3, c4.w);
      const unsigned long long v0 = join_u64(lo4.x, hi4.x), v1 = join_u64(lo4.y, hi4.y);
      const unsigned long long v2 = join_u64(lo4.z, hi4.z), v3 = join_u64(lo4.w, hi4.w);
      if (v0) add_u64_split(dlo, dhi, v0);
      if (v1) add_u64_split(dlo + 1, dhi + 1, v1);
      if (v2) add_u64_split(dlo + 2, dhi + 2, v2);
      if (v3) add_u64_split(dlo + 3, dhi + 3, v3);
      cluster.sync();
      c4 = *reinterpret_cast<const int4*>(dc);
      lo4 = *reinterpret_cast<const uint4*>(dlo);
      hi4 = *reinterpret_cast<const uint4*>(dhi);
    }
    const ulonglong2 m01 = make_ulonglong2(join_u64(lo4.x, hi4.x), join_u64(lo4.y, hi4.y));
    const ulonglong2 m23 = make_ulonglong2(join_u64(lo4.z, hi4.z), join_u64(lo4.w, hi4.w));
    reinterpret_cast<int4*>(sh.bcnt)[tid] = c4;
    reinterpret_cast<ulonglong2*>(sh.bmass)[2 * tid] = m01;
    reinterpret_cast<ulonglong2*>(sh.bmass)[2 * tid + 1] = m23;
    const unsigned long long wm = budget_warp_sum(m01.x + m01.y + m23.x + m23.y);
    const int wc = budget_warp_sum(c4.x + c4.y + c4.z + c4.w);
    if (lane == 0) {
      sh.wmass[warp] = wm;
      sh.wcnt[warp] = wc;
    }
    __syncthreads();
    if (round == 0) {
      // request total = every bin of the first round; T = ceil(tau * M)
      unsigned long long M = 0;
#pragma unroll
      for (int w = 0; w < kBudgetWarps; ++w) M += sh.wmass[w];
      const unsigned long long a = M / 1000ull, b = M % 1000ull;
      need = a * (unsigned long long)mass_pm + (b * (unsigned long long)mass_pm + 999ull) / 1000ull;
      if (need == 0) {
        done = true;
        break;
      }
    }
    unsigned long long mass_above;
    int cnt_r;
    const int digit = budget_find_digit(sh, need, mass_above, cnt_r);
    prefix |= uint32_t(digit) << shift;
    mask |= dmask << shift;
    need -= mass_above;
    cnt_above += cnt_r;
  }
  pdl_launch_dependents();
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
  if (!solo) cluster.sync();   // no CTA's shared memory is read remotely after this point
}

cudaError_t launch_budget(const float* scores, int total_tokens, const int32_t* req_off,
                          int num_req, int mass_pm, int min_pm, int max_pm, int32_t* keep_out,
                          int32_t* total_out, uint32_t* status, cudaStream_t stream) {
  static int cache[128][5] = {};
  if (total_out != nullptr) {
    cudaError_t e = cudaMemsetAsync(total_out, 0, sizeof(int32_t), stream);
    if (e != cudaSuccess) return e;
  }
  const size_t dyn = sizeof(BudgetShared) + size_t(kBudgetCacheKeys) * sizeof(uint32_t);
  cudaError_t e = cudaSuccess;
  const int want = cluster_size_for(total_tokens, num_req);
  const int csize =
      cluster_size_for_grid(budget_cluster_kernel, want, num_req, kBudgetThreads, dyn, cache, &e);
  if (e != cudaSuccess) return e;
  return launch_clusters(budget_cluster_kernel, num_req, csize, kBudgetThreads, dyn, stream,
                         scores, total_tokens, req_off, mass_pm, min_pm, max_pm, keep_out,
                         total_out, status);
}

}  // namespace tsel
