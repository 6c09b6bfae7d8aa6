// Shared definitions of libtsel: workspace layout, device status helpers and
// the parameter blocks passed to the kernels.
#pragma once

#include <cstddef>
#include <cstdint>

#include "../../include/tsel.h"

namespace tsel {

constexpr int kTile = 128;          // rows per MMA tile (queries or keys)
constexpr int kWsHeaderBytes = 1024;

// First bytes of every workspace. Counters sit on separate 128-byte lines.
struct WsHeader {
  uint32_t status;        // TSEL_DEV_* bits
  uint32_t pad0[31];
  int32_t sched_ctr[2];   // dynamic unit counters of the two passes
  uint32_t pad1[30];
  int32_t num_units[2];   // units of the two passes (written by the prep kernel)
  uint32_t pad2[30];
  int32_t fix_ctr;        // unit counter of the pass-1 redo launch
  uint32_t pad3[31];
  int32_t redo_count;     // pass-1 units queued for an exact redo
  uint32_t pad4[31];
  int32_t hist_ok;        // 1: the request offsets are valid and the score histograms are built
  uint32_t pad5[31];
  int32_t sel_paths[5];   // top-B requests per threshold path (tsel_select_path_counts)
  uint32_t pad6[27];
};
static_assert(sizeof(WsHeader) <= kWsHeaderBytes, "header too large");

__host__ __device__ constexpr int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
__host__ __device__ constexpr int64_t align_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

// Pass-2 units may split the query heads into up to this many groups; each
// group writes partial column sums that the last group of a 32-key slice adds up.
constexpr int kMaxHeadGroups = 8;
constexpr int kPairRows = 256;   // A rows per unit (two 128-row tiles)

// Pass-1 units may split a segment's key tiles into up to this many chunks,
// when the problem has too few (head, query pair) units to fill the GPU; the
// last chunk to finish a 32-row slice merges the chunks' (max, sum) pairs.
constexpr int kMaxKeySplits = 8;

// Key chunks per pass-1 unit for these sizes: the largest power of two (at
// most kMaxKeySplits) that keeps the units within about one wave of CTAs
// (128); a segment then uses min(chunks, key tiles / 2), so every chunk has
// at least two key tiles. A pure function of the sizes, so the workspace
// size and every launch agree on it.
__host__ __device__ inline int pass1_key_splits(int G, int Tq, int H) {
  const int64_t pairs = (int64_t(Tq) + kPairRows - 1) / kPairRows;
  const int64_t est = int64_t(H) * (pairs > G ? pairs : G);
  int ks = 1;
  while (ks < kMaxKeySplits && est * ks * 2 <= 128) ks *= 2;
  return ks;
}

// Key chunks of one segment with nkt key tiles.
__host__ __device__ inline int segment_key_splits(int ks, int nkt) {
  const int half = nkt / 2;
  return ks < half ? ks : (half > 1 ? half : 1);
}

// Byte offsets of the importance workspace regions.
struct ImpWsLayout {
  int64_t qtile_off;   // int32 [G+1]: per-segment first 128-row tile of the padded LSE rows
  int64_t kpair_off;   // int32 [G+1]: per-segment first 256-key pair (pass-2 slice counters)
  int64_t scratch;     // int32 [8*G]: sort positions, inverses and unit starts (prep kernel)
  int64_t units1;      // uint2 [U1]: pass-1 units (segment, head<<24 | query pair)
  int64_t units2;      // uint2 [U2]: pass-2 units (segment, head group<<24 | key pair)
  int64_t redo_units;  // uint2 [H][lse_stride/128]: (head, query pair)s queued for an exact redo
  int64_t redo_flags;  // int32 [H][lse_stride/128]: pair already queued (index: its first tile)
  int64_t grp_ctr;     // int32 [n_grp]: arrivals per 32-key slice (head-group split)
  int64_t part;        // fp32 [kMaxHeadGroups][Tk]: per-head-group partial column sums
  int64_t part1;       // float2 [ks][H][lse_stride]: per-key-chunk (max, sum) of pass 1 (ks > 1)
  int64_t lse_ctr;     // int32 [H][lse_stride/32]: arrivals per 32-row slice (ks > 1)
  int64_t nlse2;       // fp32 [H][lse_stride]: -LSE*log2(e), 128-row padded per segment
  int64_t lse_stride;  // floats per head (multiple of 128)
  int64_t u1_max, u2_max, n_grp;
  int ks;              // pass-1 key chunks
  int64_t total;
};

__host__ __device__ inline ImpWsLayout imp_ws_layout(int G, int Tq, int Tk, int H) {
  ImpWsLayout L{};
  int64_t off = kWsHeaderBytes;
  L.qtile_off = off;
  off = align_up(off + 4 * (int64_t(G) + 1), 256);
  L.kpair_off = off;
  off = align_up(off + 4 * (int64_t(G) + 1), 256);
  L.scratch = off;
  off = align_up(off + 32 * int64_t(G), 256);
  L.ks = pass1_key_splits(G, Tq, H);
  L.u1_max = int64_t(H) * (ceil_div(Tq, kTile) + G) * L.ks;
  L.u2_max = int64_t(kMaxHeadGroups) * (ceil_div(Tk, kPairRows) + G);
  L.units1 = off;
  off = align_up(off + 8 * L.u1_max, 256);
  L.units2 = off;
  off = align_up(off + 8 * L.u2_max, 256);
  L.lse_stride = int64_t(kTile) * (ceil_div(Tq, kTile) + G);
  L.redo_units = off;
  off = align_up(off + 8 * int64_t(H) * (L.lse_stride / kTile), 256);
  L.redo_flags = off;
  off = align_up(off + 4 * int64_t(H) * (L.lse_stride / kTile), 256);
  L.n_grp = 8 * (ceil_div(Tk, kPairRows) + G);
  L.grp_ctr = off;
  off = align_up(off + 4 * L.n_grp, 256);
  L.part = off;
  off = align_up(off + 4 * int64_t(kMaxHeadGroups) * Tk, 1024);
  L.part1 = off;
  if (L.ks > 1) off = align_up(off + 8 * int64_t(L.ks) * H * L.lse_stride, 256);
  L.lse_ctr = off;
  if (L.ks > 1) off = align_up(off + 4 * int64_t(H) * (L.lse_stride / 32), 1024);
  L.nlse2 = off;
  off = align_up(off + 4 * int64_t(H) * L.lse_stride, 256);
  L.total = off;
  return L;
}

// Per-request score histograms the column pass builds for the top-B (fused
// score + select path): bins of the first 11 bits of the order-preserving
// score key (the top-B's first radix digit) followed by bins of its first 16
// bits, int32 counts.
constexpr int kHistCoarse = 2048;
constexpr int kHistFine = 65536;
constexpr int64_t kHistWords = kHistCoarse + kHistFine;
constexpr int kHistMaxReq = 64;   // more requests: the fused path runs without histograms

// Histogram region of a fused score + select workspace (after the importance
// layout); 0 bytes when the requests get no histograms.
__host__ __device__ inline int64_t sel_hist_offset(const ImpWsLayout& L) {
  return align_up(L.total, 1024);
}
__host__ __device__ inline int64_t sel_hist_bytes(int R) {
  return (R >= 1 && R <= kHistMaxReq) ? int64_t(R) * kHistWords * 4 : 0;
}

// One-launch importance of small problems (imp_small.cu): one cluster of H
// CTAs per segment, both passes per (segment, head) in one CTA.
struct ImpSmallParams {
  const int32_t* cu_q;
  const int32_t* cu_k;
  int G, Tq, Tk;
  int max_q, max_k;      // the caller's bounds (<= 256), checked on the device
  int H, Hkv;
  float c;               // softmax_scale * log2(e)
  float* lse_out;        // natural log [H][Tq] (may be null)
  const float* lse_in;   // the caller's natural-log LSE [H][Tq]: no row-LSE phase (or null)
  float* scores;         // [Tk]
  uint32_t* status;
  uint64_t timeout_ns;
  int stall;             // test hook: no loads are issued, every wait runs out
  int sum_norm;          // 1: total attention received (no division by H*Nq)
  // top-B of a one-segment, one-request problem in the same launch (select = 1)
  int select;
  const int32_t* req_off;   // [2] the request's token range
  const int32_t* keep;      // [1] its budget
  int total_keep;           // or TSEL_KEEP_FROM_DEVICE
  int32_t* keep_idx;
  int32_t* cu_keep;         // [2]
};

struct ImpPassParams {
  const int32_t* cu_q;
  const int32_t* cu_k;
  const uint2* units;
  const int32_t* num_units;
  int32_t* sched_ctr;
  const int32_t* qtile_off;
  float* nlse2;          // pass 1 writes, pass 2 reads
  int64_t lse_stride;
  float* lse_out;        // natural log [H][Tq] (pass 1, may be null)
  float* scores;         // [Tk] (pass 2)
  uint32_t* status;
  int H, Hkv, Tq;
  float c;               // softmax_scale * log2(e)
  uint64_t timeout_ns;
  int stall;             // test hook: publish no work so every wait runs out
  // pass 2, head-group split
  int hgroups;           // kv-head groups per key pair (1 = scores written directly)
  int Tk;
  const int32_t* kpair_off;
  int32_t* grp_ctr;
  float* part;
  int sum_norm;          // 1: scores are total attention received (no division by H*Nq)
  // pass 1, key split
  int kspl;              // key chunks per (head, query pair) (1 = LSE written directly)
  float2* part1;
  int32_t* lse_ctr;
  // pass 1, fixed row reference (exact = 0): a (head, query pair) with a row
  // whose sum overflows is queued; a second launch (redo = 1, exact = 1,
  // units = the queue) redoes it with a moving reference
  int exact;
  int redo;
  uint2* redo_units;
  int32_t* redo_flags;
  int32_t* redo_count;
  // fused score + select: per-request score histograms (pass 1 zeroes them,
  // pass 2 adds every score it writes); null when not requested
  int32_t* hist;
  int64_t hist_words;        // R * kHistWords
  const int32_t* req_off;    // [R+1] request token offsets
  int R;
  const int32_t* hist_ok;    // header word written by the schedule kernel
};

__device__ __forceinline__ void set_status(uint32_t* status, uint32_t bits) {
  atomicOr(status, bits);
}

// Programmatic dependent launch: let the next kernel on the stream launch
// (its CTAs then wait in pdl_wait) ...
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ... and wait until the previous kernel on the stream has completed and its
// memory is visible (returns at once for a kernel launched without PDL).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// fp32 bits -> uint32 with the same order; -0 maps to +0.
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Adds the scores of a warp's tokens to their requests' histograms (coarse:
// first 11 bits of the key, fine: first 16 bits). Lanes holding the same bin
// add once (match_any); lanes with valid == false or tokens outside every
// request add nothing. Every lane of the warp must call it. req_off: the
// R + 1 request offsets, staged in shared memory by the caller.
__device__ __forceinline__ void hist_add_warp(int32_t* hist, const int32_t* req_off, int R,
                                              int tok, float s, bool valid) {
  const int lane = threadIdx.x & 31;
  int r = -1;
  uint32_t key = 0;
  if (valid) {
    int lo = 0, hi = R + 1;   // first i in [0, R] with req_off[i] > tok
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (req_off[mid] <= tok) lo = mid + 1;
      else hi = mid;
    }
    r = lo - 1 < R ? lo - 1 : -1;
    key = order_key(s);
  }
  const bool in = r >= 0;
  const uint32_t tc = in ? (uint32_t(r) << 11) | (key >> 21) : 0xFFFFFFFFu;
  const uint32_t tf = in ? (uint32_t(r) << 16) | (key >> 16) : 0xFFFFFFFFu;
  const unsigned mc = __match_any_sync(0xffffffffu, tc);
  const unsigned mf = __match_any_sync(0xffffffffu, tf);
  if (in) {
    int32_t* h = hist + int64_t(r) * kHistWords;
    if (lane == __ffs(mc) - 1) atomicAdd(h + (key >> 21), __popc(mc));
    if (lane == __ffs(mf) - 1) atomicAdd(h + kHistCoarse + (key >> 16), __popc(mf));
  }
}

// Inverse of order_key (for keys of non-negative scores).
__device__ __forceinline__ float key_to_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

}  // namespace tsel
