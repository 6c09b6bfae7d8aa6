// Importance passes: mean softmax attention received by every key token.
//
// Follows the LiteVLM review (section 3.2, s_j = Attn(h, v_j)) and the
// dynamic vision-token compression article (section 3.2: mean attention
// received; probabilities recovered block by block from the row LSE and
// reduced along columns; the attention matrix never leaves the chip).
//
// Three launches on one stream:
//   prep   one CTA: checks cu_seqlens, sorts segments by cost (longest first)
//          and writes the unit lists of both passes into the workspace.
//   pass 1 units (segment, head, 256 query rows = two 128-row A tiles):
//          S = Q K^T tile by tile on the tensor cores (tcgen05, accumulators
//          in TMEM), each 128-key B tile multiplied by both A tiles, online
//          max/sum per query row -> row LSE (kept as -LSE*log2 e, padded to
//          128-row tiles per segment). Each row fixes its reference max on
//          its first 64 columns; a (head, query pair) with a row whose sum
//          then overflows fp32 is queued, and a second launch of the same
//          kernel redoes the queue with a reference that follows the row
//          max (nothing is queued unless the logits of a row climb more than
//          ~88 above the maximum of its first 64 keys; the launch then exits
//          at once).
//   pass 2 units (segment, 256 keys, group of query heads): S^T = K Q^T with
//          the keys on the MMA M dimension, so each epilogue thread owns one
//          key and sums exp2(S*c - LSE2) over the query columns in registers:
//          the column reduction needs no shuffles. When the heads are split
//          into groups (so that small requests still fill every SM), each
//          group stores its partial sums and the last group to finish a
//          32-key slice adds them up in group order: the result stays
//          deterministic.
// Two A tiles per unit halve the operand bytes each B tile costs per element
// (the shared-memory feed, not the tensor cores, limited 128-row units).
//
// CTA layout (608 threads, one CTA per SM, persistent, units fetched from a
// global counter in longest-first order):
//   warp 0      TMA producer (A tile pairs, B tiles, LSE slices)
//   warp 1      TMEM allocator + MMA issuer for the B tiles of parity 0 (one
//               thread): per B tile, one 128x128 accumulator for each A tile
//   warp 18     MMA issuer for the B tiles of parity 1. With one issuer for
//               both parities, a warpgroup that released its accumulator
//               late held up the other parity's next tile as well.
//   warps 2-17  four epilogue warpgroups; warpgroup 2*par + a owns TMEM
//               accumulator 2*par + a (A tile a, B tiles of parity par);
//               warp w reads TMEM lanes 32*(w%4).. . Each warp loads its
//               128 columns in 32-column pieces, the next piece in flight
//               while the current one is computed. The math is packed (f32x2
//               FMA/ADD, 3-input max), one MUFU exp2 per element. The two
//               warpgroups of an A tile merge their partials once per unit.
// The issue slots, not only the MUFU, bound the epilogue: each warp walks its
// own parity's tiles directly, full tiles run without column masks, waits
// sleep on the barrier instead of spinning, and arrivals are predicated.
#pragma once

#include <cuda_runtime.h>

#include "common.cuh"
#include "launch_util.cuh"
#include "ptx.cuh"

namespace tsel {

using namespace ptx;

constexpr float kNegInf = -__builtin_huge_valf();
constexpr int kPair = 2 * kTile;    // A rows per unit: two 128-row A tiles
constexpr int kAccBufs = 4;         // TMEM accumulators of 128 columns (512 columns)
constexpr int kLseSlots = 8;        // LSE slices in flight (pass 2)
constexpr int kSchedSlots = 4;      // scheduler ring depth
constexpr int kEpiWarps = 16;       // four warpgroups
constexpr int kEpiFirstWarp = 2;
constexpr int kMma1Warp = kEpiFirstWarp + kEpiWarps;        // second MMA issuer
constexpr int kThreads = 32 * (kEpiFirstWarp + kEpiWarps + 1);  // 608

// Shared-memory tile geometry. bf16 rows are D*2 bytes, split into 64-column
// chunks (128-byte swizzle) and 16-column chunks (32-byte swizzle). E4M3 rows
// are padded to one 128-byte chunk (128 columns; the padding reads as zeros)
// and the MMA runs ceil(D/32) K-steps of 32 over it.
template <int D, bool FP8>
struct TileCfg {
  static_assert(D % 16 == 0 && D >= 64 && D <= 128, "head_dim");
  static constexpr int N64 = FP8 ? 1 : D / 64;           // 128-byte swizzle chunks
  static constexpr int N16 = FP8 ? 0 : (D % 64) / 16;    // 32-byte swizzle chunks
  static constexpr int KSTEPS128 = FP8 ? (D + 31) / 32 : 4;  // MMA K-steps per 128-byte chunk
  static constexpr int ROW_BYTES = FP8 ? 128 : D * 2;
  static constexpr int TILE_BYTES = kTile * ROW_BYTES;   // one 128-row tile
  static constexpr int A_BYTES = 4 * TILE_BYTES;         // 2 slots x 2 A tiles
  static constexpr int STAGES_RAW = (200 * 1024 - A_BYTES - 8192) / TILE_BYTES;
  static constexpr int STAGES = STAGES_RAW > 8 ? 8 : STAGES_RAW;
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = A_BYTES;
  static constexpr int OFF_LSE = OFF_B + STAGES * TILE_BYTES;
  static constexpr int OFF_COMB = OFF_LSE + kLseSlots * kTile * 4;
  static constexpr int OFF_BAR = OFF_COMB + 2 * 2 * 2 * kTile * 4;
  static constexpr int NUM_BARS = 2 + 2 + 2 * STAGES + 2 * kAccBufs + kLseSlots +
                                  2 * kSchedSlots + 4 + 4 + 1;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 256 + 64 + 1024;  // + alignment slack
  static_assert(STAGES >= 2, "at least double-buffered B tiles");
  static_assert(TILE_BYTES % 1024 == 0, "tiles stay 1024-byte aligned");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
  static_assert(SMEM_BYTES > 116 * 1024, "one CTA per SM (TMEM is allocated whole)");
};

// ---------------------------------------------------------------------------
// Pass kernel
// ---------------------------------------------------------------------------

struct Unit {
  int g, h, pair, q0, nq, k0, nk;
  int nA;          // valid 128-row A tiles in this unit's 256-row pair (1 or 2)
  int qtile_base;  // first 128-row tile of the segment in the padded LSE rows
  int h1;          // pass 2: query heads [h, h1) (pass 1: h + 1)
  int hg;          // pass 2: head group of the unit
  int kt0, kt1;    // B tiles [kt0, kt1) of the unit (pass 1: its key chunk)
  int kc, ksg;     // pass 1: key chunk of the unit and chunks of its segment
  int valid;       // 1 for a unit, 0 for the end-of-work marker
};

static_assert(kSchedSlots * sizeof(Unit) <= 256, "scheduler ring fits its shared-memory slot");

template <int PASS, bool KSPLIT>
__device__ __forceinline__ Unit decode_unit(const ImpPassParams& p, uint2 u) {
  Unit r;
  r.g = int(u.x);
  if (PASS == 1) {
    r.pair = int(u.y & 0xFFFFFu);
    r.kc = int((u.y >> 20) & 0xFu);
    r.h = int(u.y >> 24);
    r.h1 = r.h + 1;
    r.hg = 0;
  } else {
    r.pair = int(u.y & 0xFFFFFFu);
    r.kc = 0;
    r.hg = int(u.y >> 24);
    const int per = p.H / p.hgroups;
    r.h = r.hg * per;
    r.h1 = r.h + per;
  }
  r.q0 = __ldg(p.cu_q + r.g);
  r.nq = __ldg(p.cu_q + r.g + 1) - r.q0;
  r.k0 = __ldg(p.cu_k + r.g);
  r.nk = __ldg(p.cu_k + r.g + 1) - r.k0;
  const int rows_left = (PASS == 1 ? r.nq : r.nk) - r.pair * kPair;
  r.nA = rows_left > kTile ? 2 : 1;
  if (PASS == 1) {
    const int nkt = int(ceil_div(r.nk, kTile));
    if (KSPLIT) {
      // balanced split of the segment's key tiles: every chunk is non-empty
      r.ksg = segment_key_splits(p.kspl > 0 ? p.kspl : 1, nkt);
      r.kt0 = int(int64_t(r.kc) * nkt / r.ksg);
      r.kt1 = int(int64_t(r.kc + 1) * nkt / r.ksg);
    } else {
      r.ksg = 1;
      r.kt0 = 0;
      r.kt1 = nkt;
    }
  } else {
    r.ksg = 1;
    r.kt0 = 0;
    r.kt1 = int(ceil_div(r.nq, kTile));
  }
  r.qtile_base = __ldg(p.qtile_off + r.g);
  r.valid = 1;
  return r;
}

// Loads one 128-row tile of head `head` (columns [0, D)) starting at row y.
// bf16: 2-D maps over [rows, heads*D] (x = head*D + column); E4M3: a 3-D map
// over [rows, heads, D] whose 128-column box pads past D with zeros.
template <int D, bool FP8>
__device__ __forceinline__ void load_tile(uint8_t* dst, const CUtensorMap* m64,
                                          const CUtensorMap* m16, uint64_t* bar, int head, int y) {
  using C = TileCfg<D, FP8>;
  if (FP8) {
    tma_load_3d(dst, m64, bar, 0, head, y);
  } else {
    const int x0 = head * D;
#pragma unroll
    for (int c = 0; c < C::N64; ++c) tma_load_2d(dst + c * 16384, m64, bar, x0 + 64 * c, y);
#pragma unroll
    for (int j = 0; j < C::N16; ++j)
      tma_load_2d(dst + C::N64 * 16384 + j * 4096, m16, bar, x0 + 64 * C::N64 + 16 * j, y);
  }
}

// Issues the MMAs of one 128x128 tile: D = A * B^T over the head dimension.
template <int D, bool FP8>
__device__ __forceinline__ void issue_tile_mmas(uint32_t d_tmem, const uint8_t* a,
                                                const uint8_t* b) {
  using C = TileCfg<D, FP8>;
  const uint32_t a0 = smem_u32(a), b0 = smem_u32(b);
  uint32_t acc = 0;
  if (FP8) {
    constexpr uint32_t kIdesc = idesc_e4m3_f32(kTile, kTile);
#pragma unroll
    for (int k = 0; k < C::KSTEPS128; ++k) {
      mma_f8(d_tmem, smem_desc(a0 + k * 32, 2, 1024), smem_desc(b0 + k * 32, 2, 1024), kIdesc,
             acc);
      acc = 1;
    }
    return;
  }
  constexpr uint32_t kIdesc = idesc_bf16_f32(kTile, kTile);
#pragma unroll
  for (int c = 0; c < C::N64; ++c) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t off = c * 16384 + k * 32;
      mma_bf16(d_tmem, smem_desc(a0 + off, 2, 1024), smem_desc(b0 + off, 2, 1024), kIdesc, acc);
      acc = 1;
    }
  }
#pragma unroll
  for (int j = 0; j < C::N16; ++j) {
    const uint32_t off = C::N64 * 16384 + j * 4096;
    mma_bf16(d_tmem, smem_desc(a0 + off, 6, 256), smem_desc(b0 + off, 6, 256), kIdesc, acc);
    acc = 1;
  }
}

// Waits with the time limit only (used to drain copies before exit).
__device__ __forceinline__ bool wait_drain(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
  const int zero = 0;
  return wait_bounded(bar, parity, &zero, timeout_ns);
}

// Epilogue waits: all lanes wait, and the outcome is made warp-uniform so a
// timeout never leaves part of a warp in front of a .sync.aligned TMEM load.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity,
                                          const volatile int* abort_flag, uint64_t timeout_ns) {
  return __all_sync(0xffffffffu, wait_bounded(bar, parity, abort_flag, timeout_ns));
}


// Adds exp2(S*c - LSE2) of 32 query columns into the packed per-key
// accumulators (pass 2). nl holds -LSE2 of those columns (-inf for padding).
__device__ __forceinline__ void column_sum_chunk(const uint32_t (&r)[32], const float4* nl,
                                                 float2 c2, float2 (&acc)[2]) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float4 t = nl[j];
    const float2 x01 = __ffma2_rn(
        make_float2(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1])), c2,
        make_float2(t.x, t.y));
    const float2 x23 = __ffma2_rn(
        make_float2(__uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3])), c2,
        make_float2(t.z, t.w));
    acc[0] = ex2_add2(acc[0], x01);
    acc[1] = ex2_add2(acc[1], x23);
  }
}



// Pass 1 (row LSE), on 32 columns held as raw TMEM words. Per query row, m
// is a reference for S*c and l the sum of exp2(S*c - m) before the current
// accumulators a. First launch (lazy): m is the max of the row's first 64
// columns and stays there — the terms of later columns may exceed 1, and a
// row whose logits climb ~128 (log2) above m overflows to inf, which the
// unit end detects. Redo launch (exact): m moves whenever the max of the
// next 64 columns exceeds it by more than 8 (terms stay below 2^8).
// Columns at or beyond `valid` lie outside the segment and read as -inf.
__device__ __forceinline__ void mask_cols(uint32_t (&r)[32], int valid) {
#pragma unroll
  for (int j = 0; j < 32; ++j) r[j] = j < valid ? r[j] : __float_as_uint(kNegInf);
}

__device__ __forceinline__ float cols_max(const uint32_t (&r)[32]) {
#define V_(j) __uint_as_float(r[j])
  float t0 = fmax3(V_(0), V_(1), V_(2)), t1 = fmax3(V_(3), V_(4), V_(5));
  float t2 = fmax3(V_(6), V_(7), V_(8)), t3 = fmax3(V_(9), V_(10), V_(11));
#pragma unroll
  for (int j = 12; j < 28; j += 8) {
    t0 = fmax3(t0, V_(j), V_(j + 1));
    t1 = fmax3(t1, V_(j + 2), V_(j + 3));
    t2 = fmax3(t2, V_(j + 4), V_(j + 5));
    t3 = fmax3(t3, V_(j + 6), V_(j + 7));
  }
  return fmax3(fmax3(t0, t1, V_(28)), fmax3(t2, t3, V_(29)), fmaxf(V_(30), V_(31)));
#undef V_
}

__device__ __forceinline__ void move_reference(float t, float& m, float& l, float2 (&a)[2]) {
  if (t > m + 8.f) {   // also covers the first columns of a row (m = -inf, l = 0)
    const float s = ex2(m - t);
    const float2 a01 = __fadd2_rn(a[0], a[1]);
    l = (l + (a01.x + a01.y)) * s;
    a[0] = make_float2(0.f, 0.f);
    a[1] = make_float2(0.f, 0.f);
    m = t;
  }
}

__device__ __forceinline__ void cols_exp_sum(const uint32_t (&r)[32], float2 c2, float2 nm2,
                                             float2 (&a)[2]) {
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float2 x = __ffma2_rn(make_float2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1])),
                                c2, nm2);
    a[j & 1] = ex2_add2(a[j & 1], x);
  }
}

// One 128-column accumulator: two 32-column pieces in flight; the
// accumulator is handed back to the MMA once all of it is in registers.
// FULL: all 128 columns lie inside the segment (no masking).
template <int PASS, bool FULL>
__device__ __forceinline__ void epilogue_tile(uint32_t taddr, int valid, const float4* nl,
                                              float c, float2 c2, bool lazy, float& m, float& l,
                                              float2 (&acc)[2], uint64_t* acc_empty, int lane) {
  uint32_t r0[32], r1[32];
  tmem_ld32_async(taddr, r0);
  tmem_ld32_async(taddr + 32, r1);
  tmem_wait_ld(r0);
  tmem_wait_ld(r1);
  if constexpr (PASS == 1) {
    // row max over 64 columns at a time: one reference move per 64 columns
    // and the exps of both 32-column pieces independent of each other
    if (!FULL) {
      mask_cols(r0, valid);
      mask_cols(r1, valid - 32);
    }
    if (!lazy || m == kNegInf) move_reference(fmaxf(cols_max(r0), cols_max(r1)) * c, m, l, acc);
    float2 nm2 = make_float2(-m, -m);
    cols_exp_sum(r0, c2, nm2, acc);
    tmem_ld32_async(taddr + 64, r0);
    if (FULL || valid > 32) cols_exp_sum(r1, c2, nm2, acc);
    tmem_ld32_async(taddr + 96, r1);
    tmem_wait_ld(r0);
    tmem_wait_ld(r1);
    tc_fence_before();
    __syncwarp();
    mbar_arrive_lane0(acc_empty, lane);
    if (FULL || valid > 64) {
      if (!FULL) {
        mask_cols(r0, valid - 64);
        mask_cols(r1, valid - 96);
      }
      if (!lazy) move_reference(fmaxf(cols_max(r0), cols_max(r1)) * c, m, l, acc);
      nm2 = make_float2(-m, -m);
      cols_exp_sum(r0, c2, nm2, acc);
      if (FULL || valid > 96) cols_exp_sum(r1, c2, nm2, acc);
    }
  } else {
    if (FULL || valid > 0) column_sum_chunk(r0, nl, c2, acc);
    tmem_ld32_async(taddr + 64, r0);
    if (FULL || valid > 32) column_sum_chunk(r1, nl + 8, c2, acc);
    tmem_ld32_async(taddr + 96, r1);
    tmem_wait_ld(r0);
    tmem_wait_ld(r1);
    tc_fence_before();
    __syncwarp();
    mbar_arrive_lane0(acc_empty, lane);
    if (FULL || valid > 64) column_sum_chunk(r0, nl + 16, c2, acc);
    if (FULL || valid > 96) column_sum_chunk(r1, nl + 24, c2, acc);
  }
}

// KSPLIT: pass-1 units may cover a key chunk (merged across chunks at the end).
template <int PASS, int D, bool FP8, bool KSPLIT>
__global__ void __launch_bounds__(kThreads, 1)
    imp_pass_kernel(const __grid_constant__ CUtensorMap mapA64,
                    const __grid_constant__ CUtensorMap mapA16,
                    const __grid_constant__ CUtensorMap mapB64,
                    const __grid_constant__ CUtensorMap mapB16, const ImpPassParams p) {
  using C = TileCfg<D, FP8>;
  constexpr int S = C::STAGES;
  extern __shared__ uint8_t smem_dyn[];
  // 128-byte swizzle atoms key off shared-address bits: align the carve-out
  // on the shared-window address itself.
  uint8_t* smem = smem_dyn + ((1024u - (smem_u32(smem_dyn) & 1023u)) & 1023u);
  uint8_t* sA = smem + C::OFF_A;   // [2 slots][2 tiles]
  uint8_t* sB = smem + C::OFF_B;   // [S stages]
  float* sLse = reinterpret_cast<float*>(smem + C::OFF_LSE);
  float* sComb = reinterpret_cast<float*>(smem + C::OFF_COMB);  // [A half][buf][m|l][128]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* a_full = bars;
  uint64_t* a_empty = a_full + 2;
  uint64_t* b_full = a_empty + 2;
  uint64_t* b_empty = b_full + S;
  uint64_t* acc_full = b_empty + S;
  uint64_t* acc_empty = acc_full + kAccBufs;
  // The LSE slice of a B tile lands on that tile's b_full barrier; the
  // epilogue reads it after acc_full, which the MMA thread commits only after
  // it has seen b_full complete. lse_empty returns the slot to the producer.
  uint64_t* lse_empty = acc_empty + kAccBufs;
  uint64_t* sch_full = lse_empty + kLseSlots;
  uint64_t* sch_empty = sch_full + kSchedSlots;
  uint64_t* comb_full = sch_empty + kSchedSlots;  // [A half][buf]
  uint64_t* comb_empty = comb_full + 4;
  uint64_t* mma_done = comb_empty + 4;
  Unit* sched = reinterpret_cast<Unit*>(smem + C::OFF_MISC);   // decoded units in flight
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC + 256);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 260);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t T = p.timeout_ns;

  if (PASS == 1 && p.redo != 0) {
    // Redo launch: the queue is complete once the first launch has finished;
    // it is almost always empty, so leave before any set-up.
    pdl_wait();
    if (*reinterpret_cast<const volatile int*>(p.num_units) == 0) {
      pdl_launch_dependents();
      return;
    }
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&a_full[i], 1);
      mbar_init(&a_empty[i], 2);             // both MMA issuers
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(&comb_full[i], 4);
      mbar_init(&comb_empty[i], 4);
    }
    for (int i = 0; i < S; ++i) {
      mbar_init(&b_full[i], 1);
      mbar_init(&b_empty[i], 1);
    }
    for (int i = 0; i < kAccBufs; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 4);           // the owning warpgroup
    }
    for (int i = 0; i < kLseSlots; ++i) {
      mbar_init(&lse_empty[i], 8);           // both warpgroups of the B-tile parity
    }
    for (int i = 0; i < kSchedSlots; ++i) {
      mbar_init(&sch_full[i], 1);
      mbar_init(&sch_empty[i], 2 + kEpiWarps);
    }
    mbar_init(mma_done, 2);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&mapA64);
    prefetch_tensormap(&mapA16);
    prefetch_tensormap(&mapB64);
    prefetch_tensormap(&mapB16);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Prologue done: the next kernel may launch; wait for the schedule kernel
  // (unit lists) and, in pass 2, the row-LSE pass.
  pdl_launch_dependents();
  pdl_wait();
  const int total_units = *reinterpret_cast<const volatile int*>(p.num_units);
  const int group = p.H / p.Hkv;
  if (PASS == 1 && p.hist != nullptr && warp >= kEpiFirstWarp && warp < kMma1Warp) {
    // Fused score + select: zero the per-request score histograms the column
    // pass adds into (the epilogue warps have nothing to do yet).
    constexpr int kZeroThreads = 32 * kEpiWarps;
    const int t = (warp - kEpiFirstWarp) * 32 + lane;
    int4* h4 = reinterpret_cast<int4*>(p.hist);
    for (int64_t i = int64_t(blockIdx.x) * kZeroThreads + t; i < p.hist_words / 4;
         i += int64_t(gridDim.x) * kZeroThreads)
      h4[i] = make_int4(0, 0, 0, 0);
  }
  const bool add_hist =
      PASS == 2 && p.hist != nullptr && *reinterpret_cast<const volatile int32_t*>(p.hist_ok) != 0;
  // request offsets for the histogram adds, read once per CTA
  __shared__ int32_t s_req_off[kHistMaxReq + 1];
  if (add_hist && warp >= kEpiFirstWarp && warp < kMma1Warp) {
    const int t = (warp - kEpiFirstWarp) * 32 + lane;
    if (t <= p.R) s_req_off[t] = __ldg(p.req_off + t);
    asm volatile("bar.sync 1, %0;" ::"n"(32 * kEpiWarps) : "memory");   // the epilogue warps
  }

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int s_it = 0, a_it = 0, b_it = 0;
      bool ok = p.stall == 0;   // the test hook leaves the consumers waiting for work
      // No more units than CTAs: each CTA takes the unit of its own index
      // (no round trip to the counter for it, nor for the end of the work).
      const bool one_each = total_units <= int(gridDim.x);
      while (ok) {
        const int slot = s_it % kSchedSlots;
        if (!wait_bounded(&sch_empty[slot], ((s_it / kSchedSlots) & 1) ^ 1, abort_flag, T)) {
          ok = false;
          break;
        }
        const int u = one_each ? (s_it == 0 ? int(blockIdx.x) : total_units)
                               : atomicAdd(p.sched_ctr, 1);
        Unit w;
        if (u < total_units) {
          w = decode_unit<PASS, KSPLIT>(p, p.units[u]);
        } else {
          w = Unit{};
          w.valid = 0;
        }
        sched[slot] = w;   // consumers read the decoded unit from shared memory
        mbar_arrive(&sch_full[slot]);
        ++s_it;
        if (!w.valid) break;
        if (w.kt1 == w.kt0) continue;   // no B tiles (a segment without keys / queries)
        // pass 2: one A tile pair per kv head the unit's query heads read
        const int ag0 = PASS == 1 ? 0 : w.h / group;
        const int ag1 = PASS == 1 ? 1 : (w.h1 - 1) / group + 1;
        const int qtile_base = w.qtile_base;
        for (int ag = ag0; ag < ag1 && ok; ++ag) {
          const int as = a_it & 1;
          if (!wait_bounded(&a_empty[as], ((a_it >> 1) & 1) ^ 1, abort_flag, T)) { ok = false; break; }
          mbar_arrive_expect_tx(&a_full[as], uint32_t(w.nA * C::TILE_BYTES));
          const int ahead = PASS == 1 ? w.h : ag;
          const int ay = (PASS == 1 ? w.q0 : w.k0) + w.pair * kPair;
          for (int a = 0; a < w.nA; ++a)
            load_tile<D, FP8>(sA + (as * 2 + a) * C::TILE_BYTES, &mapA64, &mapA16, &a_full[as],
                              ahead, ay + a * kTile);
          ++a_it;
          const int hb0 = PASS == 1 ? w.h : max(w.h, ag * group);
          const int hb1 = PASS == 1 ? w.h + 1 : min(w.h1, (ag + 1) * group);
          for (int h = hb0; h < hb1 && ok; ++h) {
            const int bhead = PASS == 1 ? w.h / group : h;
            for (int bt = w.kt0; bt < w.kt1; ++bt) {
              const int bs = b_it % S;
              if (!wait_bounded(&b_empty[bs], ((b_it / S) & 1) ^ 1, abort_flag, T)) { ok = false; break; }
              const int ls = b_it % kLseSlots;
              if (PASS == 2 &&
                  !wait_bounded(&lse_empty[ls], ((b_it / kLseSlots) & 1) ^ 1, abort_flag, T)) {
                ok = false;
                break;
              }
              mbar_arrive_expect_tx(&b_full[bs], C::TILE_BYTES + (PASS == 2 ? kTile * 4 : 0));
              load_tile<D, FP8>(sB + bs * C::TILE_BYTES, &mapB64, &mapB16, &b_full[bs], bhead,
                                (PASS == 1 ? w.k0 : w.q0) + bt * kTile);
              if (PASS == 2)
                bulk_load(sLse + ls * kTile,
                          p.nlse2 + int64_t(h) * p.lse_stride + int64_t(qtile_base + bt) * kTile,
                          kTile * 4, &b_full[bs]);
              ++b_it;
            }
          }
        }
      }
      if (!ok && p.stall == 0) {
        *abort_flag = 1;
        set_status(p.status, TSEL_DEV_TIMEOUT);
      }
      // Drain: every copy this thread issued has landed before the CTA exits.
      for (int i = 0; i < S && i < b_it; ++i) {
        const int n = b_it - 1 - i;
        wait_drain(&b_full[n % S], (n / S) & 1, T);
      }
      for (int i = 0; i < 2 && i < a_it; ++i) {
        const int n = a_it - 1 - i;
        wait_drain(&a_full[n & 1], (n >> 1) & 1, T);
      }

    }
  } else if (warp == 1 || warp == kMma1Warp) {
    // ------------------------------------------------------------ MMA issuers
    // Each walks every unit and B tile, and issues the tiles of its parity.
    if (lane == 0) {
      const int mypar = warp == 1 ? 0 : 1;
      int s_it = 0, a_it = 0, b_it = 0;
      bool ok = true;
      while (ok) {
        const int slot = s_it % kSchedSlots;
        if (!wait_bounded(&sch_full[slot], (s_it / kSchedSlots) & 1, abort_flag, T)) { ok = false; break; }
        const Unit w = sched[slot];
        mbar_arrive(&sch_empty[slot]);
        ++s_it;
        if (!w.valid) break;
        const int nbt = w.kt1 - w.kt0;
        if (nbt == 0) continue;
        const int ag0 = PASS == 1 ? 0 : w.h / group;
        const int ag1 = PASS == 1 ? 1 : (w.h1 - 1) / group + 1;
        for (int ag = ag0; ag < ag1 && ok; ++ag) {
          const int as = a_it & 1;
          if (!wait_bounded(&a_full[as], (a_it >> 1) & 1, abort_flag, T)) { ok = false; break; }
          tc_fence_after();
          const int n_b = PASS == 1
                              ? nbt
                              : (min(w.h1, (ag + 1) * group) - max(w.h, ag * group)) * nbt;
          for (int bi = 0; bi < n_b; ++bi) {
            if ((b_it & 1) != mypar) {
              ++b_it;
              continue;
            }
            const int bs = b_it % S;
            if (!wait_bounded(&b_full[bs], (b_it / S) & 1, abort_flag, T)) { ok = false; break; }
            const uint32_t use = uint32_t(b_it >> 1) & 1u;
            for (int a = 0; a < 2; ++a) {
              const int k = 2 * (b_it & 1) + a;
              if (!wait_bounded(&acc_empty[k], use ^ 1u, abort_flag, T)) { ok = false; break; }
              tc_fence_after();
              if (a < w.nA)
                issue_tile_mmas<D, FP8>(tmem_base + uint32_t(k * kTile),
                                   sA + (as * 2 + a) * C::TILE_BYTES, sB + bs * C::TILE_BYTES);
              mma_commit(&acc_full[k]);
            }
            if (!ok) break;
            mma_commit(&b_empty[bs]);
            ++b_it;
          }
          mma_commit(&a_empty[as]);
          ++a_it;
        }
      }
      if (!ok) {
        *abort_flag = 1;
        set_status(p.status, TSEL_DEV_TIMEOUT);
      }
      // All MMAs issued by this thread have completed before TMEM is freed.
      mma_commit(mma_done);
      wait_drain(mma_done, 0, T);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // Warpgroup wg = 2*par + a owns TMEM accumulator k = 2*par + a: rows of
    // A tile `a` against the B tiles of parity `par`.
    const int wg = (warp - kEpiFirstWarp) >> 2;
    const int a_half = wg & 1, par = wg >> 1;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const int kbuf = 2 * par + a_half;
    const uint32_t taddr = tmem_base + (uint32_t(quad * 32) << 16) + uint32_t(kbuf * kTile);
    const float c = p.c;
    const float2 c2 = make_float2(c, c);
    const bool lazy = PASS == 1 && p.exact == 0;
    int s_it = 0, b_it = 0, unit_it = 0;
    bool ok = true;
    while (ok) {
      const int slot = s_it % kSchedSlots;
      if (!warp_wait(&sch_full[slot], (s_it / kSchedSlots) & 1, abort_flag, T)) { ok = false; break; }
      // Pass 2 reads its unit from the ring slot and hands the slot back at
      // the end of the unit (fewer registers held across the tile loop); pass
      // 1 keeps a copy and hands the slot back at once.
      Unit w_copy;
      if constexpr (PASS == 1) {
        w_copy = sched[slot];
        __syncwarp();
        mbar_arrive_lane0(&sch_empty[slot], lane);
      }
      const Unit& w = PASS == 1 ? w_copy : sched[slot];
      ++s_it;
      if (!w.valid) {
        if constexpr (PASS == 2) {
          __syncwarp();
          mbar_arrive_lane0(&sch_empty[slot], lane);
        }
        break;
      }
      const bool mine = a_half < w.nA;   // this warpgroup's A tile holds rows of the unit
      // without key chunks pass 1 walks every key tile of the segment
      constexpr bool kWhole = PASS == 1 && !KSPLIT;
      const int nbt = kWhole ? int(ceil_div(w.nk, kTile)) : w.kt1 - w.kt0;
      const int n_b = PASS == 1 ? nbt : (nbt > 0 ? (w.h1 - w.h) * nbt : 0);
      const int vbase = kWhole ? w.nk : (PASS == 1 ? w.nk : w.nq) - w.kt0 * kTile;  // valid cols from kt0
      float m = kNegInf, l = 0.f;           // pass 1
      float2 acc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};  // pass 1: sum since m; pass 2: per-key sum
      // This warpgroup's tiles: global B-tile indices of parity `par`; bt is
      // the tile's column block within its head.
      const int b_end = b_it + n_b;
      int g = b_it + ((par ^ b_it) & 1);
      int bt = g - b_it;
      if (bt >= nbt) bt -= nbt;
      for (; g < b_end; g += 2) {
        const uint32_t use = uint32_t(g >> 1) & 1u;
        if (!warp_wait(&acc_full[kbuf], use, abort_flag, T)) { ok = false; break; }
        const int ls = g & (kLseSlots - 1);

        tc_fence_after();
        if (mine) {
          const int valid = vbase - bt * kTile;
          const float4* nl = reinterpret_cast<const float4*>(sLse + ls * kTile);
          if (valid >= kTile)
            epilogue_tile<PASS, true>(taddr, valid, nl, c, c2, lazy, m, l, acc, &acc_empty[kbuf], lane);
          else
            epilogue_tile<PASS, false>(taddr, valid, nl, c, c2, lazy, m, l, acc, &acc_empty[kbuf], lane);
        } else {
          tc_fence_before();
          __syncwarp();
          mbar_arrive_lane0(&acc_empty[kbuf], lane);
        }
        if (PASS == 2) {
          __syncwarp();
          mbar_arrive_lane0(&lse_empty[ls], lane);
        }
        bt += 2;
        if (bt >= nbt) bt -= nbt;
        if (bt >= nbt) bt -= nbt;
      }
      if (!ok) break;
      b_it = b_end;
      // Merge the two warpgroups of the same A half (B-tile parities 0 and 1).
      const int cb = unit_it & 1;
      const uint32_t cpar = (unit_it >> 1) & 1;
      float* comb = sComb + (a_half * 2 + cb) * 2 * kTile;
      uint64_t* cfull = &comb_full[a_half * 2 + cb];
      uint64_t* cempty = &comb_empty[a_half * 2 + cb];
      const float2 accs = __fadd2_rn(acc[0], acc[1]);
      const float part = accs.x + accs.y;   // pass 1: sum since m; pass 2: per-key sum
      if (par == 1) {
        if (!warp_wait(cempty, cpar ^ 1, abort_flag, T)) { ok = false; break; }
        comb[row] = PASS == 1 ? m : part;
        comb[kTile + row] = PASS == 1 ? l + part : 0.f;
        __syncwarp();
        if (lane == 0) mbar_arrive(cfull);
      } else {
        if (!warp_wait(cfull, cpar, abort_flag, T)) { ok = false; break; }
        const float o0 = comb[row], o1 = comb[kTile + row];
        __syncwarp();
        if (lane == 0) mbar_arrive(cempty);
        if (mine) {
          if (PASS == 1) {
            const float l0 = l + part;
            float M = fmaxf(m, o0);
            float Lsum = 0.f;
            // Which warpgroup holds the even tiles of the unit depends on
            // the CTA's earlier units: the merge is written symmetric (two
            // rounded products, one add; no contraction into an FMA) so the
            // result does not.
            if (M > kNegInf) Lsum = __fadd_rn(__fmul_rn(l0, ex2(m - M)), __fmul_rn(o1, ex2(o0 - M)));
            const int qrow = w.pair * kPair + a_half * kTile + row;
            const bool valid = qrow < w.nq;
            const int qtile = w.qtile_base + w.pair * 2 + a_half;
            const int64_t lrow = int64_t(w.h) * p.lse_stride + int64_t(qtile) * kTile + row;
            bool write = true;
            if (KSPLIT && w.ksg > 1) {
              // (max, sum) of this key chunk; the last chunk of the 32-row
              // slice to finish merges all chunks in chunk order.
              p.part1[int64_t(w.kc) * p.H * p.lse_stride + lrow] = make_float2(M, Lsum);
              __threadfence();
              __syncwarp();
              int old = 0;
              if (lane == 0) {
                const int64_t slice = int64_t(w.h) * (p.lse_stride / 32) + int64_t(qtile) * 4 + quad;
                old = atomicAdd(p.lse_ctr + slice, 1);
                if (old == w.ksg - 1) p.lse_ctr[slice] = 0;   // no other arrival follows
              }
              old = __shfl_sync(0xffffffffu, old, 0);
              write = old == w.ksg - 1;
              if (write) {
                __threadfence();
                M = kNegInf;
                for (int kc = 0; kc < w.ksg; ++kc)
                  M = fmaxf(M, __ldcg(&p.part1[int64_t(kc) * p.H * p.lse_stride + lrow].x));
                Lsum = 0.f;
                if (M > kNegInf) {
                  for (int kc = 0; kc < w.ksg; ++kc) {
                    const float2 ml = __ldcg(&p.part1[int64_t(kc) * p.H * p.lse_stride + lrow]);
                    if (ml.x > kNegInf) Lsum += ml.y * ex2(ml.x - M);
                  }
                }
              }
            }
            if (write) {
              const float lse2 = Lsum > 0.f ? M + log2f(Lsum) : kNegInf;
              p.nlse2[lrow] = (valid && Lsum > 0.f) ? -lse2 : kNegInf;
              if (valid && p.lse_out != nullptr)
                p.lse_out[int64_t(w.h) * p.Tq + w.q0 + qrow] = lse2 * 0.69314718055994531f;
              // A sum past the fp32 range (inf, or NaN from inf * 0) under the
              // fixed reference: queue the (head, query pair) for the redo
              // launch, once (the flag is indexed by the pair's first tile).
              const bool over = lazy && valid && !(Lsum <= 3.402823466e38f);
              if (__any_sync(0xffffffffu, over) && lane == 0) {
                const int64_t fi = int64_t(w.h) * (p.lse_stride / kTile) + w.qtile_base + 2 * w.pair;
                if (atomicExch(p.redo_flags + fi, 1) == 0) {
                  const int slot_r = atomicAdd(p.redo_count, 1);
                  p.redo_units[slot_r] = make_uint2(uint32_t(w.g), (uint32_t(w.h) << 24) | uint32_t(w.pair));
                }
              }
            }
          } else {
            const int krow = w.pair * kPair + a_half * kTile + row;
            const float total = part + o0;
            const float rows = p.sum_norm ? 1.f : float(p.H * w.nq);
            if (p.hgroups == 1) {
              const float sc = w.nq > 0 ? total / rows : 0.f;
              if (krow < w.nk) p.scores[w.k0 + krow] = sc;
              if (add_hist) hist_add_warp(p.hist, s_req_off, p.R, w.k0 + krow, sc, krow < w.nk);
            } else {
              // Partial sums of this head group; the last group of the 32-key
              // slice adds all groups' partials in group order.
              if (krow < w.nk) p.part[int64_t(w.hg) * p.Tk + w.k0 + krow] = total;
              __threadfence();
              __syncwarp();
              int old = 0;
              if (lane == 0) {
                const int slice = (__ldg(p.kpair_off + w.g) + w.pair) * 8 + a_half * 4 + quad;
                old = atomicAdd(p.grp_ctr + slice, 1);
                if (old == p.hgroups - 1) p.grp_ctr[slice] = 0;   // no other arrival follows
              }
              old = __shfl_sync(0xffffffffu, old, 0);
              if (old == p.hgroups - 1) {
                __threadfence();
                float sc = 0.f;
                if (krow < w.nk) {
                  float sum = 0.f;
                  for (int gi = 0; gi < p.hgroups; ++gi)
                    sum += __ldcg(p.part + int64_t(gi) * p.Tk + w.k0 + krow);
                  sc = w.nq > 0 ? sum / rows : 0.f;
                  p.scores[w.k0 + krow] = sc;
                }
                if (add_hist) hist_add_warp(p.hist, s_req_off, p.R, w.k0 + krow, sc, krow < w.nk);
              }
            }
          }
        }
      }
      ++unit_it;
      if constexpr (PASS == 2) {
        __syncwarp();
        mbar_arrive_lane0(&sch_empty[slot], lane);
      }
    }
    if (!ok) {
      *abort_flag = 1;
      set_status(p.status, TSEL_DEV_TIMEOUT);
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, 512);
}


// Launches one pass instance (sets its shared-memory attribute once per device).
template <int PASS, int D, bool FP8, bool KSPLIT>
cudaError_t launch_pass_t(const CUtensorMap* maps, const ImpPassParams& p, int grid,
                          cudaStream_t stream) {
  using C = TileCfg<D, FP8>;
  auto kern = imp_pass_kernel<PASS, D, FP8, KSPLIT>;
  static bool attr_set[128] = {};  // per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 128 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 128) attr_set[dev] = true;
  }
  return launch_kernel(kern, dim3(unsigned(grid)), kThreads, size_t(C::SMEM_BYTES), stream, 1,
                       maps[0], maps[1], maps[2], maps[3], p);
}

}  // namespace tsel
