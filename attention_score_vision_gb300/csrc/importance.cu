// Importance scores: the schedule kernel, the LSE import of the LSE-provided
// mode, and the dispatch to the pass kernels (imp_pass.cuh, instantiated in
// imp_pass1.cu and imp_pass2.cu so the two passes compile in parallel).
#include <cuda_runtime.h>

#include "imp_pass.cuh"

namespace tsel {

// ---------------------------------------------------------------------------
// Prep kernel
// ---------------------------------------------------------------------------

// Exclusive scan of one value per thread over a 1024-thread block.
__device__ __forceinline__ int block_excl_scan(int v, int* warp_sums, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    warp_sums[lane] = w;
  }
  __syncthreads();
  const int excl = x - v + (warp > 0 ? warp_sums[warp - 1] : 0);
  total = warp_sums[31];
  __syncthreads();
  return excl;
}

// In-place exclusive scan of a[0..n); returns the sum.
__device__ int block_scan_array(int* a, int n, int* warp_sums) {
  int carry = 0;
  for (int base = 0; base < n; base += 1024) {
    const int i = base + threadIdx.x;
    const int v = i < n ? a[i] : 0;
    int total;
    const int e = block_excl_scan(v, warp_sums, total);
    if (i < n) a[i] = carry + e;
    carry += total;
    __syncthreads();
  }
  return carry;
}

// Replaces key[g] (0..1023) by g's position in descending key order.
__device__ void bucket_positions_desc(int* key, int G, int* hist, int* warp_sums) {
  hist[threadIdx.x] = 0;
  __syncthreads();
  for (int g = threadIdx.x; g < G; g += 1024) atomicAdd(&hist[key[g]], 1);
  __syncthreads();
  const int b = 1023 - threadIdx.x;  // bucket 1023 comes first
  const int cnt = hist[b];
  int total;
  const int start = block_excl_scan(cnt, warp_sums, total);
  hist[b] = start;
  __syncthreads();
  for (int g = threadIdx.x; g < G; g += 1024) key[g] = atomicAdd(&hist[key[g]], 1);
  __syncthreads();
}

// Exclusive scan over the 32 lanes of a warp; `total` gets the sum.
__device__ __forceinline__ int warp_excl_scan(int v, int& total) {
  const int lane = threadIdx.x & 31;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  total = __shfl_sync(0xffffffffu, x, 31);
  return x - v;
}

// THREADS = 1024: any number of segments; fewer threads: up to 32 segments.
template <int THREADS>
__global__ void __launch_bounds__(THREADS) imp_prep_kernel(const int32_t* __restrict__ cu_q,
                                                        const int32_t* __restrict__ cu_k, int G,
                                                        int Tq, int Tk, int max_q, int max_k,
                                                        int H, int HG, uint8_t* ws,
                                                        ImpWsLayout L,
                                                        const int32_t* __restrict__ req_off,
                                                        int R) {
  __shared__ int bad;
  __shared__ int totals[2];
  __shared__ int hist[1024];
  __shared__ int warp_sums[32];
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  int32_t* qtile_off = reinterpret_cast<int32_t*>(ws + L.qtile_off);
  int32_t* kpair_off = reinterpret_cast<int32_t*>(ws + L.kpair_off);
  int32_t* grp_ctr = reinterpret_cast<int32_t*>(ws + L.grp_ctr);
  int32_t* pos1 = reinterpret_cast<int32_t*>(ws + L.scratch);
  int32_t* pos2 = pos1 + G;
  int32_t* inv1 = pos2 + G;
  int32_t* inv2 = inv1 + G;
  int32_t* start1 = inv2 + G;
  int32_t* start2 = start1 + G;
  uint2* units1 = reinterpret_cast<uint2*>(ws + L.units1);
  uint2* units2 = reinterpret_cast<uint2*>(ws + L.units2);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_wait();   // cu_seqlens and the workspace belong to earlier kernels until here
  // Released only now: every kernel of this call that launches early may
  // then read the caller's inputs, which no earlier kernel still writes.
  pdl_launch_dependents();

  if (threadIdx.x == 0) {
    bad = 0;
    hdr->num_units[0] = 0;
    hdr->num_units[1] = 0;
    hdr->sched_ctr[0] = 0;
    hdr->sched_ctr[1] = 0;
    hdr->redo_count = 0;
    hdr->fix_ctr = 0;
  }
  if (warp == 1) {
    // Fused score + select (req_off given): the column pass builds per-request
    // score histograms only for requests that cover ordered token ranges
    // (0 <= o[0] <= ... <= o[R] <= Tk) and when both passes run.
    bool ok = req_off != nullptr && R >= 1 && R <= kHistMaxReq && Tq > 0 && Tk > 0 && G > 0;
    if (ok) {
      for (int r = lane; r <= R; r += 32) {
        const int o = req_off[r];
        const int prev = r > 0 ? req_off[r - 1] : 0;
        if (o < prev || o > Tk) ok = false;
      }
    }
    ok = __all_sync(0xffffffffu, ok);
    if (lane == 0) hdr->hist_ok = ok ? 1 : 0;
  }
  for (int64_t i = threadIdx.x; i < L.n_grp; i += THREADS) grp_ctr[i] = 0;
  {
    int32_t* redo_flags = reinterpret_cast<int32_t*>(ws + L.redo_flags);
    for (int64_t i = threadIdx.x; i < int64_t(H) * (L.lse_stride / kTile); i += THREADS) redo_flags[i] = 0;
  }
  if (L.ks > 1) {
    int32_t* lse_ctr = reinterpret_cast<int32_t*>(ws + L.lse_ctr);
    for (int64_t i = threadIdx.x; i < int64_t(H) * (L.lse_stride / 32); i += THREADS) lse_ctr[i] = 0;
  }
  if constexpr (THREADS < 1024) {
    if (G > 32) {   // the launcher sends larger segment counts to the 1024-thread form
      if (threadIdx.x == 0) set_status(&hdr->status, TSEL_DEV_SEQLENS);
      return;
    }
  }
  if (G <= 32) {
    // Few segments: one warp checks, orders and scans them with shuffles.
    if (warp == 0) {
      const bool act = lane < G;
      const int nq = act ? cu_q[lane + 1] - cu_q[lane] : 0;
      const int nk = act ? cu_k[lane + 1] - cu_k[lane] : 0;
      bool b = act && (nq < 0 || nk < 0 || nq > max_q || nk > max_k);
      if (lane == 0) b = b || cu_q[0] != 0 || cu_k[0] != 0 || cu_q[G] != Tq || cu_k[G] != Tk;
      const bool any_bad = __any_sync(0xffffffffu, b);
      if (lane == 0) bad = any_bad ? 1 : 0;
      if (!any_bad) {
        const int nqt = int(ceil_div(nq, kTile)), nkt = int(ceil_div(nk, kTile));
        const int nqp = int(ceil_div(nq, kPair)), nkp = int(ceil_div(nk, kPair));
        const int ksg = segment_key_splits(L.ks, nkt);   // key chunks of this segment
        // rank in descending cost (pass 1: key tiles, pass 2: query tiles),
        // ties by segment index; idle lanes rank last
        const int key1 = act ? nkt : -1, key2 = act ? nqt : -1;
        int r1 = 0, r2 = 0;
#pragma unroll 4
        for (int j = 0; j < 32; ++j) {
          const int k1 = __shfl_sync(0xffffffffu, key1, j);
          const int k2 = __shfl_sync(0xffffffffu, key2, j);
          r1 += (k1 > key1) || (k1 == key1 && j < lane);
          r2 += (k2 > key2) || (k2 == key2 && j < lane);
        }
        hist[r1] = lane;            // hist[0..31]: segment at pass-1 rank
        hist[32 + r2] = lane;       // hist[32..63]: segment at pass-2 rank
        __syncwarp();
        const int g1 = hist[lane], g2 = hist[32 + lane];
        // every lane takes part in the shuffles (a shuffle inside the
        // conditional would leave the idle lanes out of a full-mask exchange)
        const int nqp_g1 = __shfl_sync(0xffffffffu, nqp, g1);
        const int ksg_g1 = __shfl_sync(0xffffffffu, ksg, g1);
        const int nkp_g2 = __shfl_sync(0xffffffffu, nkp, g2);
        const int v1 = act ? H * nqp_g1 * ksg_g1 : 0;
        const int v2 = act ? HG * nkp_g2 : 0;
        int t1, t2, tq, tk;
        const int s1 = warp_excl_scan(v1, t1);
        const int s2 = warp_excl_scan(v2, t2);
        const int oq = warp_excl_scan(nqt, tq);
        const int ok = warp_excl_scan(nkp, tk);
        if (act) {
          inv1[lane] = g1;
          inv2[lane] = g2;
          start1[lane] = s1;
          start2[lane] = s2;
          qtile_off[lane] = oq;
          kpair_off[lane] = ok;
        }
        if (lane == 0) {
          qtile_off[G] = tq;
          kpair_off[G] = tk;
          totals[0] = t1;
          totals[1] = t2;
        }
      }
    }
    __syncthreads();
    if (bad) {
      if (threadIdx.x == 0) set_status(&hdr->status, TSEL_DEV_SEQLENS);
      return;
    }
  } else if constexpr (THREADS == 1024) {
    if (threadIdx.x == 0 &&
        (cu_q[0] != 0 || cu_k[0] != 0 || cu_q[G] != Tq || cu_k[G] != Tk))
      bad = 1;
    __syncthreads();
    for (int g = threadIdx.x; g < G; g += 1024) {
      const int nq = cu_q[g + 1] - cu_q[g];
      const int nk = cu_k[g + 1] - cu_k[g];
      if (nq < 0 || nk < 0 || nq > max_q || nk > max_k) atomicOr(&bad, 1);
    }
    __syncthreads();
    if (bad) {
      if (threadIdx.x == 0) set_status(&hdr->status, TSEL_DEV_SEQLENS);
      return;
    }
    // Cost keys: a pass-1 unit walks all key tiles of its segment, a pass-2
    // unit all query tiles (times the heads).
    for (int g = threadIdx.x; g < G; g += 1024) {
      const int nqt = int(ceil_div(cu_q[g + 1] - cu_q[g], kTile));
      const int nkt = int(ceil_div(cu_k[g + 1] - cu_k[g], kTile));
      pos1[g] = min(nkt, 1023);
      pos2[g] = min(nqt, 1023);
      qtile_off[g] = nqt;
      kpair_off[g] = int(ceil_div(cu_k[g + 1] - cu_k[g], kPair));
    }
    __syncthreads();
    bucket_positions_desc(pos1, G, hist, warp_sums);
    bucket_positions_desc(pos2, G, hist, warp_sums);
    for (int g = threadIdx.x; g < G; g += 1024) {
      const int nqp = int(ceil_div(cu_q[g + 1] - cu_q[g], kPair));
      const int nkp = int(ceil_div(cu_k[g + 1] - cu_k[g], kPair));
      const int ksg = segment_key_splits(L.ks, int(ceil_div(cu_k[g + 1] - cu_k[g], kTile)));
      inv1[pos1[g]] = g;
      inv2[pos2[g]] = g;
      start1[pos1[g]] = H * nqp * ksg;
      start2[pos2[g]] = HG * nkp;
    }
    __syncthreads();
    const int total1 = block_scan_array(start1, G, warp_sums);
    const int total2 = block_scan_array(start2, G, warp_sums);
    const int total_qt = block_scan_array(qtile_off, G, warp_sums);
    const int total_kp = block_scan_array(kpair_off, G, warp_sums);
    if (threadIdx.x == 0) {
      qtile_off[G] = total_qt;
      kpair_off[G] = total_kp;
      totals[0] = total1;
      totals[1] = total2;
    }
    __syncthreads();
    }
  // Unit lists in descending-cost segment order.
  for (int i = warp; i < G; i += THREADS / 32) {
    const int g = inv1[i];
    const int nqp = int(ceil_div(cu_q[g + 1] - cu_q[g], kPair));
    const int ksg = segment_key_splits(L.ks, int(ceil_div(cu_k[g + 1] - cu_k[g], kTile)));
    const int n = H * nqp * ksg;
    const int s = start1[i];
    // the key chunks of one (head, query pair) are adjacent
    for (int j = lane; j < n; j += 32) {
      const int t = j / ksg, kc = j - t * ksg;
      const int h = t / nqp, qp = t - h * nqp;
      units1[s + j] = make_uint2(uint32_t(g), (uint32_t(h) << 24) | (uint32_t(kc) << 20) |
                                                  uint32_t(qp));
    }
    const int g2 = inv2[i];
    const int nkp = int(ceil_div(cu_k[g2 + 1] - cu_k[g2], kPair));
    const int s2 = start2[i];
    // The head groups of one key pair are adjacent, so the last one to finish
    // (which adds up the partial sums) follows the others closely.
    for (int j = lane; j < HG * nkp; j += 32) {
      const int kp = j / HG, hg = j - kp * HG;
      units2[s2 + j] = make_uint2(uint32_t(g2), (uint32_t(hg) << 24) | uint32_t(kp));
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    hdr->num_units[0] = totals[0];
    hdr->num_units[1] = totals[1];
  }
}

// ---------------------------------------------------------------------------
// LSE import (LSE-provided mode)
// ---------------------------------------------------------------------------

// Writes -LSE*log2(e) of a caller-provided natural-log LSE [H, Tq] into the
// padded per-segment layout the column pass reads (pad rows and rows without
// keys get -inf, so they add nothing). One CTA per (128-row tile, head).
__global__ void __launch_bounds__(kTile) imp_lse_import_kernel(
    const float* __restrict__ lse_in, int Tq, const int32_t* __restrict__ cu_q, int G,
    const int32_t* __restrict__ qtile_off, float* __restrict__ nlse2, int64_t lse_stride,
    const uint32_t* status, int32_t* hist, int64_t hist_words) {
  pdl_launch_dependents();
  pdl_wait();
  if (hist != nullptr) {
    // the column pass that follows adds into zeroed histograms
    const int64_t cta = int64_t(blockIdx.y) * gridDim.x + blockIdx.x;
    const int64_t ctas = int64_t(gridDim.x) * gridDim.y;
    int4* h4 = reinterpret_cast<int4*>(hist);
    for (int64_t i = cta * kTile + threadIdx.x; i < hist_words / 4; i += ctas * kTile)
      h4[i] = make_int4(0, 0, 0, 0);
  }
  if (*reinterpret_cast<const volatile uint32_t*>(status) & TSEL_DEV_SEQLENS) return;
  const int t = blockIdx.x, h = blockIdx.y;
  const int total = qtile_off[G];
  if (t >= total) return;
  int lo = 0, hi = G;  // last g with qtile_off[g] <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (qtile_off[mid] <= t) lo = mid;
    else hi = mid - 1;
  }
  const int g = lo;
  const int r = (t - qtile_off[g]) * kTile + int(threadIdx.x);
  const int q0 = cu_q[g], nq = cu_q[g + 1] - q0;
  float v = kNegInf;
  if (r < nq) {
    v = -lse_in[int64_t(h) * Tq + q0 + r] * 1.4426950408889634f;
    if (!(v < __builtin_huge_valf() && v > kNegInf)) v = kNegInf;  // no keys (lse -inf) or NaN
  }
  nlse2[int64_t(h) * lse_stride + int64_t(t) * kTile + threadIdx.x] = v;
}

// ---------------------------------------------------------------------------
// Host-side launch helpers (called from tsel_api.cu)
// ---------------------------------------------------------------------------

cudaError_t launch_imp_prep(const int32_t* cu_q, const int32_t* cu_k, int G, int Tq, int Tk,
                            int max_q, int max_k, int H, int HG, uint8_t* ws,
                            const ImpWsLayout& L, const int32_t* req_off, int R,
                            cudaStream_t stream) {
  // Few segments and few units: a small block (one warp orders the segments,
  // four write the units); otherwise all 32 warps write the unit lists.
  if (G <= 32 && L.u1_max + L.u2_max <= 1024)
    return launch_kernel(imp_prep_kernel<128>, dim3(1), 128, 0, stream, 1, cu_q, cu_k, G, Tq, Tk,
                         max_q, max_k, H, HG, ws, L, req_off, R);
  return launch_kernel(imp_prep_kernel<1024>, dim3(1), 1024, 0, stream, 1, cu_q, cu_k, G, Tq, Tk,
                       max_q, max_k, H, HG, ws, L, req_off, R);
}

cudaError_t launch_lse_import(const float* lse_in, int Tq, const int32_t* cu_q, int G,
                              const int32_t* qtile_off, float* nlse2, int64_t lse_stride,
                              int max_qtiles, int H, const uint32_t* status, int32_t* hist,
                              int64_t hist_words, cudaStream_t stream) {
  if (max_qtiles <= 0) return cudaSuccess;
  return launch_kernel(imp_lse_import_kernel, dim3(unsigned(max_qtiles), unsigned(H)), kTile, 0,
                       stream, 1, lse_in, Tq, cu_q, G, qtile_off, nlse2, lse_stride, status, hist,
                       hist_words);
}

cudaError_t launch_imp_pass1(int head_dim, bool fp8, bool ksplit, const CUtensorMap* maps,
                             const ImpPassParams& p, int grid, cudaStream_t stream);
cudaError_t launch_imp_pass2(int head_dim, bool fp8, const CUtensorMap* maps,
                             const ImpPassParams& p, int grid, cudaStream_t stream);

// maps: A64, A16, B64, B16 (pass 1: A = Q, B = K; pass 2: A = K, B = Q). For
// E4M3 inputs A64 / B64 are the 3-D maps and A16 / B16 are unused.
cudaError_t launch_imp_pass(int pass, int head_dim, bool fp8, const CUtensorMap* maps,
                            const ImpPassParams& p, int grid, cudaStream_t stream) {
  if (pass == 1) return launch_imp_pass1(head_dim, fp8, p.kspl > 1, maps, p, grid, stream);
  return launch_imp_pass2(head_dim, fp8, maps, p, grid, stream);
}

}  // namespace tsel
