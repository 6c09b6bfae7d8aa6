// One-launch importance for small problems: every segment has at most 256
// query rows and 256 keys (a single image of a 256-token ViT, or a handful of
// them), bf16 or E4M3, at most 16 heads; with the caller's LSE, the column
// sums alone.
//
// Same quantity as the two passes of imp_pass.cuh (LiteVLM review, section
// 3.2; dynamic vision-token compression article, section 3.2: the mean
// attention each key receives, probabilities recovered from the row LSE and
// reduced along columns on chip), with the whole 256 x 256 score block of one
// (segment, head) held in TMEM at once, so one CTA does both passes:
//
//   1. S = Q K^T: two 128-row query tiles x two 128-key tiles, four 128x128
//      tcgen05 accumulators (all 512 TMEM columns), each issued as soon as its
//      two tiles have landed. Each epilogue warpgroup takes one accumulator:
//      per query row a max-referenced exp2 sum over its 128 keys (the
//      reference follows the row max, terms stay below 2^8), and hands the
//      accumulator back once its columns are in registers; the two warpgroups
//      of a query tile merge into the row's LSE (kept as -LSE*log2 e in shared
//      memory, written out as the natural-log LSE).
//   2. S^T = K Q^T into the same columns (each as soon as its columns are
//      handed back), keys on the MMA M dimension: each epilogue thread owns
//      one key and sums exp2(S*c - LSE2) over the query columns in registers;
//      the two warpgroups of a key tile add up.
//   3. The CTAs of one segment form a thread-block cluster, one CTA per head.
//      Each CTA stores every key's sum for its head into the shared memory of
//      the CTA that reduces that key (distributed shared memory); after one
//      cluster barrier each CTA adds its keys' sums in head order (a fixed
//      order: the scores are deterministic) and writes the scores.
//
// There is no schedule kernel (each CTA checks the cu_seqlens itself), no
// second launch and no global counter. The launch is programmatically
// dependent like every kernel of the library; it allocates TMEM before it
// releases the next kernel, and releases it only after its own grid-dependency
// wait (so a kernel that launches early may read the caller's inputs).
//
// CTA: warp 0 TMA producer, warp 1 TMEM allocator + MMA issuer (one thread),
// warps 2-17 four epilogue warpgroups (warp w reads TMEM lanes 32*(w%4)..).
// The dynamic shared memory is padded so that a second CTA never shares an SM
// (each holds all of TMEM until its part of the cluster's work is done).
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include "imp_pass.cuh"

namespace cg = cooperative_groups;

namespace tsel {

namespace {

constexpr int kSmallThreads = 32 * (2 + kEpiWarps);   // 576

template <int D, bool FP8>
struct SmallCfg {
  using C = TileCfg<D, FP8>;
  static constexpr int OFF_Q = 0;                        // two query tiles
  static constexpr int OFF_K = 2 * C::TILE_BYTES;        // two key tiles
  static constexpr int OFF_NL = 4 * C::TILE_BYTES;       // -LSE2 of the 256 query rows
  static constexpr int OFF_CM = OFF_NL + kPair * 4;      // warpgroup exchange [2][128]
  static constexpr int OFF_CL = OFF_CM + kPair * 4;      // warpgroup exchange [2][128]
  static constexpr int OFF_RECV = OFF_CL + kPair * 4;    // per-head sums of this CTA's keys
  static constexpr int OFF_SEL = OFF_RECV + kMaxClusterCtas * kPair * 4;   // top-B scratch [64]
  static constexpr int OFF_RANK = OFF_SEL + 256;         // top-B: 64-bit keys [256], ranks [2][256]
  static constexpr int NUM_BARS = 2 + 2 + 4 + 4 + 4 + 1;   // tiles, S, S freed, S^T, MMAs done
  static constexpr int OFF_BAR = OFF_RANK + 4 * kPair * 4;
  static constexpr int OFF_MISC = OFF_BAR + 8 * NUM_BARS;   // TMEM address, abort flag, check
  static constexpr int USED = OFF_MISC + 64 + 1024;      // + alignment slack
  static constexpr int MIN_ONE_PER_SM = 120 * 1024;      // two of these exceed an SM
  static constexpr int SMEM_BYTES = USED > MIN_ONE_PER_SM ? USED : MIN_ONE_PER_SM;
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

// Hands an accumulator back (`rel`, one arrival per warp) once its last
// columns are in registers, so S^T can be computed into it meanwhile.
__device__ __forceinline__ void release_acc(uint64_t* rel, int lane) {
  tc_fence_before();
  __syncwarp();
  mbar_arrive_lane0(rel, lane);
}

// Row max/sum of one 128-column accumulator piece (phase 1). `valid` columns
// lie inside the segment (> 0); m is the row's reference for S*c, l the sum of
// exp2(S*c - m) before the accumulators acc.
__device__ __forceinline__ void small_row_lse(uint32_t taddr, int valid, float c, float2 c2,
                                              float& m, float& l, float2 (&acc)[2],
                                              uint64_t* rel, int lane) {
  uint32_t r0[32], r1[32];
  tmem_ld32_async(taddr, r0);
  tmem_ld32_async(taddr + 32, r1);
  tmem_wait_ld(r0);
  tmem_wait_ld(r1);
  if (valid <= 64) release_acc(rel, lane);
  mask_cols(r0, valid);
  mask_cols(r1, valid - 32);
  move_reference(fmaxf(cols_max(r0), cols_max(r1)) * c, m, l, acc);
  float2 nm2 = make_float2(-m, -m);
  cols_exp_sum(r0, c2, nm2, acc);
  if (valid > 32) cols_exp_sum(r1, c2, nm2, acc);
  if (valid > 64) {
    tmem_ld32_async(taddr + 64, r0);
    tmem_ld32_async(taddr + 96, r1);
    tmem_wait_ld(r0);
    tmem_wait_ld(r1);
    release_acc(rel, lane);
    mask_cols(r0, valid - 64);
    mask_cols(r1, valid - 96);
    move_reference(fmaxf(cols_max(r0), cols_max(r1)) * c, m, l, acc);
    nm2 = make_float2(-m, -m);
    cols_exp_sum(r0, c2, nm2, acc);
    if (valid > 96) cols_exp_sum(r1, c2, nm2, acc);
  }
}

// Per-key sum of exp2(S*c - LSE2) over the 128 query columns of one
// accumulator (phase 2); nl holds -LSE2 of those columns (-inf past the
// segment), `vq` of them lie inside the segment (> 0).
__device__ __forceinline__ void small_col_sum(uint32_t taddr, int vq, const float4* nl, float2 c2,
                                              float2 (&acc)[2]) {
  uint32_t r0[32], r1[32];
  tmem_ld32_async(taddr, r0);
  tmem_ld32_async(taddr + 32, r1);
  tmem_wait_ld(r0);
  tmem_wait_ld(r1);
  column_sum_chunk(r0, nl, c2, acc);
  if (vq > 32) column_sum_chunk(r1, nl + 8, c2, acc);
  if (vq > 64) {
    tmem_ld32_async(taddr + 64, r0);
    tmem_ld32_async(taddr + 96, r1);
    tmem_wait_ld(r0);
    tmem_wait_ld(r1);
    column_sum_chunk(r0, nl + 16, c2, acc);
    if (vq > 96) column_sum_chunk(r1, nl + 24, c2, acc);
  }
}

// Top-B of the one request of a one-segment problem, in CTA 0 of its cluster
// (the pooled global top-B of the dynamic vision-token compression article,
// section 3.2; one image, so its pool is that image): every key's score from
// the per-head sums (head order); then each key's rank among the request's
// keys under the order (score key descending, token index ascending) — the
// count of larger 64-bit keys (order-preserving score bits, then 255 minus
// the token index), two threads per key, 128 keys each — and the tokens of
// rank below B in token order. The request checks, status bits and outputs
// are those of the top-B kernel (topk.cu) for the same request. sRecv
// [cs][256] per-head sums; sKey [256]; scratch: 64-bit keys [256] + ranks
// [2][256]; sW [64] (sW[8..10]: the request's offsets and budget, read at
// kernel start).
__device__ __forceinline__ void small_select(const ImpSmallParams& p, int cs, int nq, int nk,
                                             float rows, const float* sRecv, uint32_t* sKey,
                                             int* scratch, int* sW) {
  const int t = int(threadIdx.x);
  const int lo = sW[8], hi = sW[9], B = sW[10];
  bool nan_in = false;
  if (t < nk) {   // one segment: token index = key index
    float sum = 0.f;
#pragma unroll
    for (int r = 0; r < kMaxClusterCtas; ++r)
      if (r < cs) sum += sRecv[r * kPair + t];
    const float sc = nq > 0 ? sum / rows : 0.f;
    p.scores[t] = sc;
    sKey[t] = order_key(sc);
    nan_in = sc != sc && t >= lo && t < hi;
  }
  const int any_nan = __syncthreads_or(nan_in);
  bool bad = lo < 0 || hi < lo || hi > p.Tk || B < 0 || B > hi - lo;
  bad = bad || (p.total_keep >= 0 ? B != p.total_keep : B > p.Tk);
  if (bad) {
    if (t == 0) set_status(p.status, TSEL_DEV_REQUESTS);
    return;
  }
  if (B > 0) {
    uint64_t* k64 = reinterpret_cast<uint64_t*>(scratch);   // [256]
    int* rank = scratch + 2 * kPair;                        // [2][256]
    // Keys outside [lo, hi) are 0: no key of the request is below it. (hi <= 256)
    if (t < kPair)
      k64[t] = (t >= lo && t < hi) ? ((uint64_t(sKey[t]) << 8) | uint64_t(255 - t)) : 0ull;
    __syncthreads();
    if (t < 2 * kPair) {
      const int i = t & (kPair - 1), half = t >> 8;
      const uint64_t ki = k64[i];
      const ulonglong2* k2 = reinterpret_cast<const ulonglong2*>(k64) + half * 64;
      int rk = 0;
#pragma unroll 16
      for (int q = 0; q < 64; ++q) {
        const ulonglong2 v = k2[q];
        rk += int(v.x > ki) + int(v.y > ki);
      }
      rank[half * kPair + i] = rk;
    }
    __syncthreads();
    if (t < kPair) {
      // slot = kept tokens of lower index
      const int lane = t & 31, w = t >> 5;
      const bool kept = t >= lo && t < hi && rank[t] + rank[kPair + t] < B;
      const unsigned mk = __ballot_sync(0xffffffffu, kept);
      if (lane == 0) sW[w] = __popc(mk);
      asm volatile("bar.sync 3, %0;" ::"n"(kPair) : "memory");
      int base = 0;
      for (int x = 0; x < w; ++x) base += sW[x];
      if (kept) p.keep_idx[base + __popc(mk & ((1u << lane) - 1u))] = t;
    }
  }
  if (t == 0) {
    p.cu_keep[0] = 0;
    p.cu_keep[1] = B;
    if (B > 0) {
      atomicAdd(&reinterpret_cast<WsHeader*>(p.status)->sel_paths[4], 1);
      if (any_nan) set_status(p.status, TSEL_DEV_NAN);
    }
  }
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

template <int D, bool FP8>
__global__ void __launch_bounds__(kSmallThreads, 1)
    imp_small_kernel(const __grid_constant__ CUtensorMap mapQ64,
                     const __grid_constant__ CUtensorMap mapQ16,
                     const __grid_constant__ CUtensorMap mapK64,
                     const __grid_constant__ CUtensorMap mapK16, const ImpSmallParams p) {
  using C = TileCfg<D, FP8>;
  using S = SmallCfg<D, FP8>;
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = smem_dyn + ((1024u - (smem_u32(smem_dyn) & 1023u)) & 1023u);
  uint8_t* sQ = smem + S::OFF_Q;
  uint8_t* sK = smem + S::OFF_K;
  float* sNl = reinterpret_cast<float*>(smem + S::OFF_NL);
  float* sCm = reinterpret_cast<float*>(smem + S::OFF_CM);
  float* sCl = reinterpret_cast<float*>(smem + S::OFF_CL);
  float* sRecv = reinterpret_cast<float*>(smem + S::OFF_RECV);
  uint64_t* q_full = reinterpret_cast<uint64_t*>(smem + S::OFF_BAR);   // [2] query tiles
  uint64_t* k_full = q_full + 2;       // [2] key tiles
  uint64_t* acc1_full = k_full + 2;    // [4] S accumulators complete
  uint64_t* acc1_free = acc1_full + 4; // [4] S accumulators read out
  uint64_t* acc2_full = acc1_free + 4; // [4] S^T accumulators complete
  uint64_t* mma_done = acc2_full + 4;  // every MMA complete
  static_assert(2 + 2 + 4 + 4 + 4 + 1 == S::NUM_BARS, "barrier region");
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + S::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + S::OFF_MISC + 4);
  int* s_bad = reinterpret_cast<int*>(smem + S::OFF_MISC + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  cg::cluster_group cluster = cg::this_cluster();
  const int cs = int(cluster.num_blocks());   // = the number of heads
  const int h = int(cluster.block_rank());    // this CTA's head
  const int g = int(blockIdx.x) / cs;         // this cluster's segment
  const uint64_t T = p.timeout_ns;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&k_full[i], 1);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(&acc1_full[i], 1);
      mbar_init(&acc1_free[i], 4);   // the four warps of the reading warpgroup
      mbar_init(&acc2_full[i], 1);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&mapQ64);
    prefetch_tensormap(&mapQ16);
    prefetch_tensormap(&mapK64);
    prefetch_tensormap(&mapK16);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();                 // cu_seqlens, Q and K may come from earlier kernels
  pdl_launch_dependents();    // after the TMEM allocation and the wait (see above)

  // Every CTA checks every segment (the same data gives every CTA the same
  // outcome, so a bad input sends all of them out before any cluster barrier).
  if (warp == 0) {
    bool b = false;
    for (int i = lane; i < p.G; i += 32) {
      const int nq = __ldg(p.cu_q + i + 1) - __ldg(p.cu_q + i);
      const int nk = __ldg(p.cu_k + i + 1) - __ldg(p.cu_k + i);
      b = b || nq < 0 || nk < 0 || nq > p.max_q || nk > p.max_k;
    }
    if (lane == 0)
      b = b || __ldg(p.cu_q) != 0 || __ldg(p.cu_k) != 0 || __ldg(p.cu_q + p.G) != p.Tq ||
          __ldg(p.cu_k + p.G) != p.Tk;
    b = __any_sync(0xffffffffu, b);
    if (lane == 0) *s_bad = b ? 1 : 0;
  }
  __syncthreads();
  if (*s_bad) {
    if (blockIdx.x == 0 && threadIdx.x == 0) set_status(p.status, TSEL_DEV_SEQLENS);
    if (warp == 1) tmem_dealloc(tmem, 512);
    return;
  }
  if (p.select && h == 0 && threadIdx.x == 0) {
    int* sW = reinterpret_cast<int*>(smem + S::OFF_SEL);
    sW[8] = __ldg(p.req_off);        // read now: used after the cluster barrier
    sW[9] = __ldg(p.req_off + 1);
    sW[10] = __ldg(p.keep);
  }
  const int q0 = __ldg(p.cu_q + g), nq = __ldg(p.cu_q + g + 1) - q0;
  const int k0 = __ldg(p.cu_k + g), nk = __ldg(p.cu_k + g + 1) - k0;
  const int nA = int(ceil_div(nq, kTile)), nB = int(ceil_div(nk, kTile));
  const bool work = nA > 0 && nB > 0;
  // Accumulator j holds S tile (query tile j>>1, key tile j&1), then S^T tile
  // (key tile j>>1, query tile j&1), in TMEM columns [128 j, 128 j + 128).
  // With the caller's LSE there is no S phase.
  const bool lse_given = p.lse_in != nullptr;
  auto exists1 = [&](int j) { return !lse_given && (j >> 1) < nA && (j & 1) < nB; };
  auto exists2 = [&](int j) { return (j >> 1) < nB && (j & 1) < nA; };
  // Keys [r * per, (r + 1) * per) are summed over the heads by CTA r (all
  // of them by CTA 0 when it also selects the request's top-B).
  const int per = p.select ? kPair : (kPair + cs - 1) / cs;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && work && p.stall == 0) {   // the test hook issues nothing: waits run out
      const int kvh = h / (p.H / p.Hkv);
      // in the order the MMAs need them: Q0, K0, K1, Q1
      mbar_arrive_expect_tx(&q_full[0], uint32_t(C::TILE_BYTES));
      load_tile<D, FP8>(sQ, &mapQ64, &mapQ16, &q_full[0], h, q0);
      mbar_arrive_expect_tx(&k_full[0], uint32_t(C::TILE_BYTES));
      load_tile<D, FP8>(sK, &mapK64, &mapK16, &k_full[0], kvh, k0);
      if (nB > 1) {
        mbar_arrive_expect_tx(&k_full[1], uint32_t(C::TILE_BYTES));
        load_tile<D, FP8>(sK + C::TILE_BYTES, &mapK64, &mapK16, &k_full[1], kvh, k0 + kTile);
      }
      if (nA > 1) {
        mbar_arrive_expect_tx(&q_full[1], uint32_t(C::TILE_BYTES));
        load_tile<D, FP8>(sQ + C::TILE_BYTES, &mapQ64, &mapQ16, &q_full[1], h, q0 + kTile);
      }
      // the copies have landed before the CTA can exit
      wait_drain(&q_full[0], 0, T);
      wait_drain(&k_full[0], 0, T);
      if (nB > 1) wait_drain(&k_full[1], 0, T);
      if (nA > 1) wait_drain(&q_full[1], 0, T);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && work) {
      bool ok = true;
      for (int j = 0; j < 4 && ok; ++j) {
        if (!exists1(j)) continue;
        if (!wait_bounded(&q_full[j >> 1], 0, abort_flag, T) ||
            !wait_bounded(&k_full[j & 1], 0, abort_flag, T)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_tile_mmas<D, FP8>(tmem + uint32_t(j * kTile), sQ + (j >> 1) * C::TILE_BYTES,
                                sK + (j & 1) * C::TILE_BYTES);
        mma_commit(&acc1_full[j]);
      }
      for (int j = 0; j < 4 && ok; ++j) {
        if (!exists2(j)) continue;
        if (lse_given && (!wait_bounded(&q_full[j & 1], 0, abort_flag, T) ||
                          !wait_bounded(&k_full[j >> 1], 0, abort_flag, T))) {
          ok = false;
          break;
        }
        if (exists1(j) && !wait_bounded(&acc1_free[j], 0, abort_flag, T)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_tile_mmas<D, FP8>(tmem + uint32_t(j * kTile), sK + (j >> 1) * C::TILE_BYTES,
                                sQ + (j & 1) * C::TILE_BYTES);
        mma_commit(&acc2_full[j]);
      }
      if (!ok) {
        *abort_flag = 1;
        set_status(p.status, TSEL_DEV_TIMEOUT);
      }
      // every MMA this thread issued has completed before TMEM is freed
      mma_commit(mma_done);
      wait_drain(mma_done, 0, T);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // Warpgroup j reads accumulator j in both phases.
    const int j = (warp - kEpiFirstWarp) >> 2;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t taddr = tmem + (uint32_t(quad * 32) << 16) + uint32_t(j * kTile);
    const float c = p.c;
    const float2 c2 = make_float2(c, c);
    {
      // Phase 1: query tile a x key tile b; the two warpgroups of a query tile merge.
      const int a = j >> 1, b = j & 1;
      float m = kNegInf, l = 0.f;
      float2 acc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      if (exists1(j)) {
        if (warp_wait(&acc1_full[j], 0, abort_flag, T)) {
          tc_fence_after();
          small_row_lse(taddr, nk - b * kTile, c, c2, m, l, acc, &acc1_free[j], lane);
        } else if (lane == 0) {
          *abort_flag = 1;
          set_status(p.status, TSEL_DEV_TIMEOUT);
        }
      }
      const float2 s2 = __fadd2_rn(acc[0], acc[1]);
      const float L = l + (s2.x + s2.y);
      if (b == 1) {
        sCm[a * kTile + row] = m;
        sCl[a * kTile + row] = L;
      }
      asm volatile("bar.sync 1, %0;" ::"n"(32 * kEpiWarps) : "memory");
      if (lse_given) {
        // the caller's natural-log LSE as -LSE2; a row without keys (-inf) or a
        // NaN adds nothing, as in the two-pass path's LSE import
        const int qrow = (warp - kEpiFirstWarp) * 32 + lane;   // 0..511
        if (qrow < kPair) {
          float v = kNegInf;
          if (qrow < nq) {
            v = -__ldg(p.lse_in + int64_t(h) * p.Tq + q0 + qrow) * 1.4426950408889634f;
            if (!(v < __builtin_huge_valf() && v > kNegInf)) v = kNegInf;
          }
          sNl[qrow] = v;
        }
      } else if (b == 0) {
        const float m1 = sCm[a * kTile + row], l1 = sCl[a * kTile + row];
        const float M = fmaxf(m, m1);
        float Ls = 0.f;
        if (M > kNegInf) Ls = __fadd_rn(__fmul_rn(L, ex2(m - M)), __fmul_rn(l1, ex2(m1 - M)));
        const int qrow = a * kTile + row;
        const bool valid = qrow < nq;
        const float lse2 = Ls > 0.f ? M + log2f(Ls) : kNegInf;
        sNl[qrow] = (valid && Ls > 0.f) ? -lse2 : kNegInf;
        if (valid && p.lse_out != nullptr && *abort_flag == 0)
          p.lse_out[int64_t(h) * p.Tq + q0 + qrow] = lse2 * 0.69314718055994531f;
      }
      asm volatile("bar.sync 1, %0;" ::"n"(32 * kEpiWarps) : "memory");   // sNl complete
    }
    {
      // Phase 2: key tile b x query tile a; the two warpgroups of a key tile add up
      // and send each key's sum for this head to the CTA that reduces it.
      const int b = j >> 1, a = j & 1;
      float2 acc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      if (exists2(j)) {
        if (warp_wait(&acc2_full[j], 0, abort_flag, T)) {
          tc_fence_after();
          small_col_sum(taddr, nq - a * kTile, reinterpret_cast<const float4*>(sNl + a * kTile),
                        c2, acc);
        } else if (lane == 0) {
          *abort_flag = 1;
          set_status(p.status, TSEL_DEV_TIMEOUT);
        }
      }
      const float2 s2 = __fadd2_rn(acc[0], acc[1]);
      const float part = s2.x + s2.y;
      if (a == 1) sCm[b * kTile + row] = part;
      asm volatile("bar.sync 1, %0;" ::"n"(32 * kEpiWarps) : "memory");
      const int key = b * kTile + row;
      if (a == 0 && key < nk) {
        const int r = key / per;
        float* dst = sRecv + h * per + (key - r * per);
        if (cs > 1) dst = cluster.map_shared_rank(dst, r);
        *dst = part + sCm[b * kTile + row];
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();   // per-key sums complete, every TMEM read done
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);

  // Head sum in head order: every CTA has sent its sums, CTA h adds those of
  // keys [h * per, (h + 1) * per). No shared memory of another CTA is touched
  // after this barrier.
  if (cs > 1) cluster_sync_all();
  if (*abort_flag != 0) return;
  const float rows = p.sum_norm ? 1.f : float(p.H * nq);
  if (!p.select) {
    if (int(threadIdx.x) < per) {
      const int key = h * per + int(threadIdx.x);
      if (key < nk) {
        float sum = 0.f;
        for (int r = 0; r < cs; ++r) sum += sRecv[r * per + int(threadIdx.x)];
        p.scores[k0 + key] = nq > 0 ? sum / rows : 0.f;
      }
    }
    return;
  }
  if (h == 0)
    small_select(p, cs, nq, nk, rows, sRecv, reinterpret_cast<uint32_t*>(sNl),
                 reinterpret_cast<int*>(smem + S::OFF_RANK), reinterpret_cast<int*>(smem + S::OFF_SEL));
}

template <int D, bool FP8>
cudaError_t launch_small_t(const CUtensorMap* maps, const ImpSmallParams& p, cudaStream_t stream) {
  using S = SmallCfg<D, FP8>;
  auto kern = imp_small_kernel<D, FP8>;
  static bool attr_set[128] = {};   // per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 128 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 128) attr_set[dev] = true;
  }
  return launch_clusters(kern, p.G, p.H, kSmallThreads, size_t(S::SMEM_BYTES), stream, maps[0],
                         maps[1], maps[2], maps[3], p);
}

template <int D, bool FP8>
int small_active_clusters_t(int H, cudaError_t* err) {
  using S = SmallCfg<D, FP8>;
  auto kern = imp_small_kernel<D, FP8>;
  *err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM_BYTES);
  if (*err != cudaSuccess) return 0;
  *err = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (*err != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = unsigned(H);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(unsigned(H));
  cfg.blockDim = dim3(unsigned(kSmallThreads));
  cfg.dynamicSmemBytes = size_t(S::SMEM_BYTES);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int active = 0;
  *err = cudaOccupancyMaxActiveClusters(&active, kern, &cfg);
  return *err == cudaSuccess ? active : 0;
}

}  // namespace

cudaError_t launch_imp_small(int head_dim, bool fp8, const CUtensorMap* maps,
                             const ImpSmallParams& p, cudaStream_t stream) {
#define TSEL_SMALL_CASE(DD)                                                               \
  case DD:                                                                                \
    return fp8 ? launch_small_t<DD, true>(maps, p, stream) : launch_small_t<DD, false>(maps, p, stream);
  switch (head_dim) {
    TSEL_SMALL_CASE(64)
    TSEL_SMALL_CASE(80)
    TSEL_SMALL_CASE(96)
    TSEL_SMALL_CASE(112)
    TSEL_SMALL_CASE(128)
    default:
      return cudaErrorInvalidValue;
  }
#undef TSEL_SMALL_CASE
}

// How many clusters of H CTAs of the one-launch kernel the device holds at
// once (cached per device, input type, head_dim and H; 0 when none fits).
int imp_small_clusters(int head_dim, bool fp8, int H, cudaError_t* err) {
  *err = cudaSuccess;
  if (H < 1 || H > kMaxClusterCtas) return 0;
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return 0;
  static int cache[128][2][5][kMaxClusterCtas + 1] = {};   // 1 + resident clusters (0 unknown)
  const int di = (head_dim - 64) / 16;
  if (di < 0 || di > 4 || (head_dim % 16) != 0) return 0;
  const bool cacheable = dev >= 0 && dev < 128;
  const int fi = fp8 ? 1 : 0;
  if (cacheable && cache[dev][fi][di][H] != 0) return cache[dev][fi][di][H] - 1;
  int active = 0;
#define TSEL_SMALL_OCC(DD)                                                                   \
  case DD:                                                                                   \
    active = fp8 ? small_active_clusters_t<DD, true>(H, err) : small_active_clusters_t<DD, false>(H, err); \
    break;
  switch (head_dim) {
    TSEL_SMALL_OCC(64)
    TSEL_SMALL_OCC(80)
    TSEL_SMALL_OCC(96)
    TSEL_SMALL_OCC(112)
    default:
      active = fp8 ? small_active_clusters_t<128, true>(H, err) : small_active_clusters_t<128, false>(H, err);
      break;
  }
#undef TSEL_SMALL_OCC
  if (*err != cudaSuccess) {
    (void)cudaGetLastError();
    *err = cudaSuccess;   // not a failure of the call: the scheduled path takes the problem
    active = 0;
  }
  if (cacheable) cache[dev][fi][di][H] = active + 1;
  return active;
}

}  // namespace tsel
