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
};
static_assert(sizeof(WsHeader) <= kWsHeaderBytes, "header too large");

__host__ __device__ constexpr int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
__host__ __device__ constexpr int64_t align_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

// Pass-2 units may split the query heads into up to this many groups; each
// group writes partial column sums that the last group of a 32-key slice adds up.
constexpr int kMaxHeadGroups = 8;
constexpr int kPairRows = 256;   // A rows per unit (two 128-row tiles)

// Byte offsets of the importance workspace regions.
struct ImpWsLayout {
  int64_t qtile_off;   // int32 [G+1]: per-segment first 128-row tile of the padded LSE rows
  int64_t kpair_off;   // int32 [G+1]: per-segment first 256-key pair (pass-2 slice counters)
  int64_t scratch;     // int32 [8*G]: sort positions, inverses and unit starts (prep kernel)
  int64_t units1;      // uint2 [U1]: pass-1 units (segment, head<<24 | query pair)
  int64_t units2;      // uint2 [U2]: pass-2 units (segment, head group<<24 | key pair)
  int64_t grp_ctr;     // int32 [n_grp]: arrivals per 32-key slice (head-group split)
  int64_t part;        // fp32 [kMaxHeadGroups][Tk]: per-head-group partial column sums
  int64_t nlse2;       // fp32 [H][lse_stride]: -LSE*log2(e), 128-row padded per segment
  int64_t lse_stride;  // floats per head (multiple of 128)
  int64_t u1_max, u2_max, n_grp;
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
  L.u1_max = int64_t(H) * (ceil_div(Tq, kTile) + G);
  L.u2_max = int64_t(kMaxHeadGroups) * (ceil_div(Tk, kPairRows) + G);
  L.units1 = off;
  off = align_up(off + 8 * L.u1_max, 256);
  L.units2 = off;
  off = align_up(off + 8 * L.u2_max, 256);
  L.n_grp = 8 * (ceil_div(Tk, kPairRows) + G);
  L.grp_ctr = off;
  off = align_up(off + 4 * L.n_grp, 256);
  L.part = off;
  off = align_up(off + 4 * int64_t(kMaxHeadGroups) * Tk, 1024);
  L.lse_stride = int64_t(kTile) * (ceil_div(Tq, kTile) + G);
  L.nlse2 = off;
  off = align_up(off + 4 * int64_t(H) * L.lse_stride, 256);
  L.total = off;
  return L;
}

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

// Inverse of order_key (for keys of non-negative scores).
__device__ __forceinline__ float key_to_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

}  // namespace tsel
