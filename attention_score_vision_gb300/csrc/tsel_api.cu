// Host side of the C ABI declared in include/tsel.h: argument checks, TMA
// descriptor encoding, workspace carving and kernel launches. Nothing here
// allocates device memory or synchronises, except tsel_read_device_status.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <mutex>
#include <string>

#include "common.cuh"
#include "launch_util.cuh"

namespace tsel {
// Attended-pair bound above which the row-LSE pass fixes its row reference
// (2^28: ~43 us of pass 1; the redo launch costs ~4 us in the chain).
constexpr double kFixedRefMinPairs = 268435456.0;

cudaError_t launch_imp_prep(const int32_t* cu_q, const int32_t* cu_k, int G, int Tq, int Tk,
                            int max_q, int max_k, int H, int HG, uint8_t* ws,
                            const ImpWsLayout& L, const int32_t* req_off, int R,
                            cudaStream_t stream);
cudaError_t launch_imp_pass(int pass, int head_dim, bool fp8, const CUtensorMap* maps,
                            const ImpPassParams& p, int grid, cudaStream_t stream);
cudaError_t launch_imp_small(int head_dim, bool fp8, const CUtensorMap* maps,
                             const ImpSmallParams& p, cudaStream_t stream);
int imp_small_clusters(int head_dim, bool fp8, int H, cudaError_t* err);
cudaError_t launch_lse_import(const float* lse_in, int Tq, const int32_t* cu_q, int G,
                              const int32_t* qtile_off, float* nlse2, int64_t lse_stride,
                              int max_qtiles, int H, const uint32_t* status, int32_t* hist,
                              int64_t hist_words, cudaStream_t stream);
cudaError_t launch_topk(const float* scores, int total_tokens, const int32_t* req_off,
                        int num_req, const int32_t* keep, int total_keep, int32_t* keep_idx,
                        int32_t* cu_keep, uint32_t* status, const int32_t* hist,
                        const int32_t* hist_ok, int inputs_final, cudaStream_t stream);
cudaError_t launch_topk_hist(const float* scores, int total_tokens, const int32_t* req_off, int R,
                             int32_t* hist, int32_t* hist_ok, int num_sms, cudaStream_t stream);
int topk_cluster_size(int total_tokens, int num_req, cudaError_t* e);
cudaError_t launch_gather(const void* hidden, int64_t row_stride_bytes, int row_bytes,
                          const int32_t* pos, int pos_dim, const int32_t* cu_k, int G, int Tk,
                          const int32_t* keep_idx, int K, const int32_t* K_dev,
                          void* out_hidden, int32_t* out_pos, int32_t* out_img, int32_t* out_cu,
                          uint32_t* status, int num_sms, cudaStream_t stream);
cudaError_t launch_budget(const float* scores, int total_tokens, const int32_t* req_off,
                          int num_req, int mass_pm, int min_pm, int max_pm, int32_t* keep_out,
                          int32_t* total_out, uint32_t* status, cudaStream_t stream);
cudaError_t launch_probe_ex2(int blocks, int iters, float* sink, cudaStream_t stream);
}  // namespace tsel

using namespace tsel;

namespace {

thread_local std::string g_last_error;

tsel_status fail(tsel_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
tsel_status fail(tsel_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

tsel_status cuda_fail(cudaError_t e, const char* where) {
  return fail(TSEL_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

int sm_count(int* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return -1;
  static int cache[128] = {0};
  if (dev >= 0 && dev < 128 && cache[dev] > 0) {
    *out = cache[dev];
    return 0;
  }
  int n = 0;
  e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess || n <= 0) return -1;
  if (dev >= 0 && dev < 128) cache[dev] = n;
  *out = n;
  return 0;
}

// Query-head groups per pass-2 key pair: the smallest power of two (dividing
// the head count, at most kMaxHeadGroups) that gives every SM about four
// units, so the last units of the pass do not leave most SMs idle. A pure
// function of the sizes: the stages of one call agree on it.
int pass2_head_groups(int H, int G, int Tk, int sms) {
  const int64_t pairs = ceil_div(Tk, kPairRows) + (G > 0 ? G / 2 : 0);
  int hg = 1;
  while (2 * hg <= kMaxHeadGroups && H % (2 * hg) == 0 && pairs * hg < 4 * int64_t(sms)) hg *= 2;
  return hg;
}

// 2-D bf16 tensor map over `rows` rows of `width` elements (row stride in
// bytes), box of `box_w` x 128 elements.
bool make_map(CUtensorMap* map, const void* base, int64_t width, int64_t rows,
              int64_t row_stride_bytes, int box_w, CUtensorMapSwizzle sw) {
  auto enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[2] = {cuuint64_t(width), cuuint64_t(rows)};
  cuuint64_t strides[1] = {cuuint64_t(row_stride_bytes)};
  cuuint32_t box[2] = {cuuint32_t(box_w), cuuint32_t(kTile)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D uint8 tensor map over [rows, heads, head_dim] bytes, box of 128 columns
// (past head_dim the box reads zeros) x 1 head x 128 rows, 128-byte swizzle.
bool make_map_fp8(CUtensorMap* map, const void* base, int64_t head_dim, int64_t heads, int64_t rows,
                  int64_t row_stride_bytes) {
  auto enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {cuuint64_t(head_dim), cuuint64_t(heads), cuuint64_t(rows)};
  cuuint64_t strides[2] = {cuuint64_t(head_dim), cuuint64_t(row_stride_bytes)};
  cuuint32_t box[3] = {128u, 1u, cuuint32_t(kTile)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

uint64_t wait_timeout_ns() {
  static uint64_t t = [] {
    const char* s = std::getenv("TSEL_WAIT_TIMEOUT_MS");
    long v = s ? std::strtol(s, nullptr, 10) : 0;
    if (v <= 0) v = 1000;
    return uint64_t(v) * 1000000ull;
  }();
  return t;
}

}  // namespace

namespace tsel {
// Lets other translation units of the library report a detailed error.
void record_error(const char* msg) { g_last_error = msg; }
}  // namespace tsel

extern "C" {

const char* tsel_status_string(tsel_status s) {
  switch (s) {
    case TSEL_OK: return "TSEL_OK";
    case TSEL_ERR_INVALID_VALUE: return "TSEL_ERR_INVALID_VALUE";
    case TSEL_ERR_UNSUPPORTED: return "TSEL_ERR_UNSUPPORTED";
    case TSEL_ERR_WORKSPACE: return "TSEL_ERR_WORKSPACE";
    case TSEL_ERR_CUDA: return "TSEL_ERR_CUDA";
    case TSEL_ERR_DEVICE_CHECK: return "TSEL_ERR_DEVICE_CHECK";
  }
  return "TSEL_ERR_UNKNOWN";
}

const char* tsel_last_error(void) { return g_last_error.c_str(); }

int tsel_keep_count(int n_tokens, int keep_permille) {
  if (n_tokens < 0 || keep_permille < 0) return -1;
  return int((int64_t(n_tokens) * int64_t(keep_permille)) / 1000);
}

size_t tsel_importance_workspace_size(int num_seg, int total_q, int total_k, int num_heads) {
  if (num_seg < 0 || total_q < 0 || total_k < 0 || num_heads < 1) return 0;
  return size_t(imp_ws_layout(num_seg, total_q, total_k, num_heads).total);
}

size_t tsel_select_topk_workspace_size(int num_req) {
  (void)num_req;
  return kWsHeaderBytes;
}

size_t tsel_gather_compact_workspace_size(void) { return kWsHeaderBytes; }

}  // extern "C"

namespace {

// Histograms the column pass builds for the top-B of the fused path.
// TMA maps of Q and K: bf16 as 64-column boxes (128-byte swizzle) plus, when
// head_dim is not a multiple of 64, 16-column boxes (32-byte swizzle); E4M3 as
// one 3-D map each.
tsel_status make_qk_maps(const void* q, const void* k, int64_t q_row_stride, int64_t k_row_stride,
                         bool fp8, int head_dim, int64_t hd, int64_t kvd, int num_heads,
                         int num_kv_heads, int total_q, int total_k, CUtensorMap* qm64,
                         CUtensorMap* qm16, CUtensorMap* km64, CUtensorMap* km16) {
  const CUtensorMapSwizzle sw128 = CU_TENSOR_MAP_SWIZZLE_128B, sw32 = CU_TENSOR_MAP_SWIZZLE_32B;
  const bool tail = !fp8 && (head_dim % 64) != 0;
  if (fp8) {
    if (!make_map_fp8(qm64, q, head_dim, num_heads, total_q, q_row_stride) ||
        !make_map_fp8(km64, k, head_dim, num_kv_heads, total_k, k_row_stride))
      return fail(TSEL_ERR_CUDA, "cuTensorMapEncodeTiled failed (E4M3 maps)");
  } else if (!make_map(qm64, q, hd, total_q, q_row_stride * 2, 64, sw128) ||
             !make_map(km64, k, kvd, total_k, k_row_stride * 2, 64, sw128)) {
    return fail(TSEL_ERR_CUDA, "cuTensorMapEncodeTiled failed (64-wide box)");
  }
  if (tail) {
    if (!make_map(qm16, q, hd, total_q, q_row_stride * 2, 16, sw32) ||
        !make_map(km16, k, kvd, total_k, k_row_stride * 2, 16, sw32))
      return fail(TSEL_ERR_CUDA, "cuTensorMapEncodeTiled failed (16-wide box)");
  } else {
    *qm16 = *qm64;
    *km16 = *km64;
  }
  return TSEL_OK;
}

// The one-launch path's shape rule (tsel_importance's header comment).
bool one_launch_eligible(unsigned flags, int num_seg, int total_q, int total_k, int max_q,
                         int max_k, int num_heads, int head_dim, int sms, cudaError_t* err) {
  *err = cudaSuccess;
  const unsigned excl = TSEL_IMP_STAGE_PREP | TSEL_IMP_STAGE_PASS1 | TSEL_IMP_STAGE_PASS2 |
                        TSEL_SEL_STAGE_TOPK | TSEL_IMP_ROWREF_FIXED | TSEL_IMP_ROWREF_MOVING |
                        TSEL_IMP_TWO_PASS;
  if ((flags & excl) != 0 || num_seg < 1 || total_q < 1 || total_k < 1 || max_q > kPairRows ||
      max_k > kPairRows || num_heads < 1 || num_heads > kMaxClusterCtas ||
      int64_t(num_seg) * num_heads > sms)
    return false;
  // every segment's cluster resident at once (a cluster that waits for
  // another would double the latency this path is for)
  return imp_small_clusters(head_dim, (flags & TSEL_IMP_FP8_E4M3) != 0, num_heads, err) >= num_seg;
}

struct SelHist {
  const int32_t* req_off;   // [R+1]
  int R;
  int32_t* hist;            // R * kHistWords int32 (null: no histograms)
  // the top-B arguments, for the one-launch kernel to select a one-segment,
  // one-request problem itself (it then sets *selected)
  const int32_t* keep = nullptr;
  int total_keep = 0;
  int32_t* keep_idx = nullptr;
  int32_t* cu_keep = nullptr;
  bool* selected = nullptr;
};

// Importance: the schedule kernel, the row-LSE pass (or the LSE import) and
// the column pass; with `sel` the column pass also builds the histograms.
tsel_status importance_impl(const void* q, int64_t q_row_stride, const void* k,
                            int64_t k_row_stride, const int32_t* cu_seqlens_q,
                            const int32_t* cu_seqlens_k, int num_seg, int total_q, int total_k,
                            int max_seqlen_q, int max_seqlen_k, int num_heads, int num_kv_heads,
                            int head_dim, float softmax_scale, unsigned flags, float* lse,
                            float* scores, void* workspace, size_t workspace_bytes,
                            size_t workspace_needed, const SelHist& sel, cudaStream_t stream) {
  if (num_seg < 0 || total_q < 0 || total_k < 0 || max_seqlen_q < 0 || max_seqlen_k < 0)
    return fail(TSEL_ERR_INVALID_VALUE, "negative size");
  if (num_heads < 1 || num_heads > 256 || num_kv_heads < 1 || num_heads % num_kv_heads != 0)
    return fail(TSEL_ERR_INVALID_VALUE, "num_heads=%d num_kv_heads=%d", num_heads, num_kv_heads);
  if (!(head_dim == 64 || head_dim == 80 || head_dim == 96 || head_dim == 112 || head_dim == 128))
    return fail(TSEL_ERR_UNSUPPORTED, "head_dim=%d (supported: 64, 80, 96, 112, 128)", head_dim);
  if ((flags & ~(TSEL_IMP_LSE_PROVIDED | TSEL_IMP_FP8_E4M3 | TSEL_IMP_SCORE_SUM |
                 TSEL_IMP_ROWREF_FIXED | TSEL_IMP_ROWREF_MOVING | TSEL_IMP_TWO_PASS |
                 TSEL_IMP_TEST_STALL |
                 TSEL_IMP_STAGE_PREP | TSEL_IMP_STAGE_PASS1 | TSEL_IMP_STAGE_PASS2 |
                 (sel.req_off != nullptr ? TSEL_SEL_STAGE_TOPK : 0u))) != 0)
    return fail(TSEL_ERR_UNSUPPORTED, "flags=0x%x", flags);
  if ((flags & TSEL_IMP_ROWREF_FIXED) && (flags & TSEL_IMP_ROWREF_MOVING))
    return fail(TSEL_ERR_INVALID_VALUE, "TSEL_IMP_ROWREF_FIXED and _MOVING are exclusive");
  const bool lse_provided = (flags & TSEL_IMP_LSE_PROVIDED) != 0;
  if (lse_provided && total_q > 0 && lse == nullptr)
    return fail(TSEL_ERR_INVALID_VALUE, "TSEL_IMP_LSE_PROVIDED needs the lse input");
  if (cu_seqlens_q == nullptr || cu_seqlens_k == nullptr || workspace == nullptr)
    return fail(TSEL_ERR_INVALID_VALUE, "null cu_seqlens or workspace");
  if ((total_k > 0 && (scores == nullptr || k == nullptr)) || (total_q > 0 && q == nullptr))
    return fail(TSEL_ERR_INVALID_VALUE, "null q/k/scores");
  const bool fp8 = (flags & TSEL_IMP_FP8_E4M3) != 0;
  const int elem = fp8 ? 1 : 2;
  if (fp8 && !(softmax_scale > 0.f))
    return fail(TSEL_ERR_INVALID_VALUE, "TSEL_IMP_FP8_E4M3 needs softmax_scale > 0");
  const int64_t hd = int64_t(num_heads) * head_dim, kvd = int64_t(num_kv_heads) * head_dim;
  if (q_row_stride == 0) q_row_stride = hd;
  if (k_row_stride == 0) k_row_stride = kvd;
  if (q_row_stride < hd || k_row_stride < kvd || (q_row_stride * elem) % 16 != 0 ||
      (k_row_stride * elem) % 16 != 0)
    return fail(TSEL_ERR_INVALID_VALUE, "row strides %lld/%lld", (long long)q_row_stride,
                (long long)k_row_stride);
  if ((q && !aligned16(q)) || (k && !aligned16(k)))
    return fail(TSEL_ERR_INVALID_VALUE, "q/k must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(TSEL_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  const ImpWsLayout L = imp_ws_layout(num_seg, total_q, total_k, num_heads);
  if (workspace_bytes < workspace_needed)
    return fail(TSEL_ERR_WORKSPACE, "workspace %zu < %zu bytes", workspace_bytes,
                workspace_needed);
  const unsigned stage_bits = TSEL_IMP_STAGE_PREP | TSEL_IMP_STAGE_PASS1 | TSEL_IMP_STAGE_PASS2 |
                              TSEL_SEL_STAGE_TOPK;
  const unsigned stages = (flags & stage_bits) ? (flags & stage_bits) : stage_bits;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  cudaError_t e;
  int sms = 0;
  if (sm_count(&sms) != 0) return fail(TSEL_ERR_CUDA, "cannot query the SM count");
  const int hgroups = pass2_head_groups(num_heads, num_seg, total_k, sms);

  // Small problems: both passes in one launch (imp_small.cu), no schedule.
  if (sel.hist == nullptr) {
    cudaError_t fe = cudaSuccess;
    if (one_launch_eligible(flags, num_seg, total_q, total_k, max_seqlen_q, max_seqlen_k,
                            num_heads, head_dim, sms, &fe)) {
      CUtensorMap m[4];
      const tsel_status ms = make_qk_maps(q, k, q_row_stride, k_row_stride, fp8, head_dim, hd,
                                          kvd, num_heads, num_kv_heads, total_q, total_k, &m[0],
                                          &m[1], &m[2], &m[3]);
      if (ms != TSEL_OK) return ms;
      ImpSmallParams sp{};
      sp.cu_q = cu_seqlens_q;
      sp.cu_k = cu_seqlens_k;
      sp.G = num_seg;
      sp.Tq = total_q;
      sp.Tk = total_k;
      sp.max_q = max_seqlen_q;
      sp.max_k = max_seqlen_k;
      sp.H = num_heads;
      sp.Hkv = num_kv_heads;
      const float sc = softmax_scale > 0.f ? softmax_scale : 1.0f / std::sqrt(float(head_dim));
      sp.c = sc * 1.4426950408889634f;
      sp.lse_out = lse_provided ? nullptr : lse;
      sp.lse_in = lse_provided ? lse : nullptr;
      sp.scores = scores;
      sp.status = &hdr->status;
      sp.timeout_ns = (flags & TSEL_IMP_TEST_STALL) ? 50ull * 1000000ull : wait_timeout_ns();
      sp.stall = (flags & TSEL_IMP_TEST_STALL) ? 1 : 0;
      sp.sum_norm = (flags & TSEL_IMP_SCORE_SUM) ? 1 : 0;
      if (sel.selected != nullptr && sel.R == 1 && num_seg == 1) {
        sp.select = 1;
        sp.req_off = sel.req_off;
        sp.keep = sel.keep;
        sp.total_keep = sel.total_keep;
        sp.keep_idx = sel.keep_idx;
        sp.cu_keep = sel.cu_keep;
        *sel.selected = true;
      }
      e = launch_imp_small(head_dim, fp8, m, sp, stream);
      return e == cudaSuccess ? TSEL_OK : cuda_fail(e, "one-launch importance");
    }
  }

  if (stages & TSEL_IMP_STAGE_PREP) {
    e = launch_imp_prep(cu_seqlens_q, cu_seqlens_k, num_seg, total_q, total_k, max_seqlen_q,
                        max_seqlen_k, num_heads, hgroups, ws, L, sel.hist ? sel.req_off : nullptr,
                        sel.R, stream);
    if (e != cudaSuccess) return cuda_fail(e, "prep launch");
  }
  if (total_k == 0 || num_seg == 0) return TSEL_OK;
  if (total_q == 0) {
    // No query rows anywhere: every score is 0 (mean over zero rows).
    if (stages & TSEL_IMP_STAGE_PASS2) {
      e = cudaMemsetAsync(scores, 0, sizeof(float) * size_t(total_k), stream);
      if (e != cudaSuccess) return cuda_fail(e, "memset scores");
    }
    return TSEL_OK;
  }
  if (!(stages & (TSEL_IMP_STAGE_PASS1 | TSEL_IMP_STAGE_PASS2))) return TSEL_OK;

  CUtensorMap qm64, qm16, km64, km16;
  {
    const tsel_status ms = make_qk_maps(q, k, q_row_stride, k_row_stride, fp8, head_dim, hd, kvd,
                                        num_heads, num_kv_heads, total_q, total_k, &qm64, &qm16,
                                        &km64, &km16);
    if (ms != TSEL_OK) return ms;
  }
  ImpPassParams p{};
  p.cu_q = cu_seqlens_q;
  p.cu_k = cu_seqlens_k;
  p.qtile_off = reinterpret_cast<const int32_t*>(ws + L.qtile_off);
  p.nlse2 = reinterpret_cast<float*>(ws + L.nlse2);
  p.lse_stride = L.lse_stride;
  p.lse_out = lse;
  p.scores = scores;
  p.status = &hdr->status;
  p.H = num_heads;
  p.Hkv = num_kv_heads;
  p.Tq = total_q;
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / std::sqrt(float(head_dim));
  p.c = scale * 1.4426950408889634f;
  p.timeout_ns = wait_timeout_ns();
  p.stall = (flags & TSEL_IMP_TEST_STALL) ? 1 : 0;
  p.sum_norm = (flags & TSEL_IMP_SCORE_SUM) ? 1 : 0;
  if (p.stall) p.timeout_ns = 50ull * 1000000ull;
  p.hist = sel.hist;
  p.hist_words = sel.hist ? int64_t(sel.R) * kHistWords : 0;
  p.req_off = sel.req_off;
  p.R = sel.R;
  p.hist_ok = &hdr->hist_ok;

  if ((stages & TSEL_IMP_STAGE_PASS1) && lse_provided) {
    // The caller's LSE replaces the row-LSE pass.
    e = launch_lse_import(lse, total_q, cu_seqlens_q, num_seg, p.qtile_off, p.nlse2, L.lse_stride,
                          int(ceil_div(total_q, kTile) + num_seg), num_heads, &hdr->status,
                          p.hist, p.hist_words, stream);
    if (e != cudaSuccess) return cuda_fail(e, "LSE import launch");
  } else if (stages & TSEL_IMP_STAGE_PASS1) {
    const CUtensorMap maps[4] = {qm64, qm16, km64, km16};
    ImpPassParams p1 = p;
    p1.units = reinterpret_cast<const uint2*>(ws + L.units1);
    p1.num_units = &hdr->num_units[0];
    p1.sched_ctr = &hdr->sched_ctr[0];
    p1.kspl = L.ks;
    p1.part1 = reinterpret_cast<float2*>(ws + L.part1);
    p1.lse_ctr = reinterpret_cast<int32_t*>(ws + L.lse_ctr);
    p1.redo_units = reinterpret_cast<uint2*>(ws + L.redo_units);
    p1.redo_flags = reinterpret_cast<int32_t*>(ws + L.redo_flags);
    p1.redo_count = &hdr->redo_count;
    const int grid = int(L.u1_max < sms ? L.u1_max : sms);
    // Fixed row reference (and its redo launch) only where the pass is long
    // enough for the saved max to outweigh one more launch in the chain; the
    // bound is H * total_q * max_seqlen_k attended pairs, about 40 us of
    // pass 1 at the GB300 exp2 rate.
    const bool fixed_ref =
        (flags & TSEL_IMP_ROWREF_FIXED) ||
        (!(flags & TSEL_IMP_ROWREF_MOVING) &&
         double(num_heads) * double(total_q) * double(max_seqlen_k) >= kFixedRefMinPairs);
    p1.exact = fixed_ref ? 0 : 1;
    e = launch_imp_pass(1, head_dim, fp8, maps, p1, grid, stream);
    if (e != cudaSuccess) return cuda_fail(e, "pass-1 launch");
    // The redo launch: (head, query pair)s whose rows overflowed under the
    // fixed reference, whole (no key chunks), with a moving reference.
    ImpPassParams pr = p1;
    pr.exact = 1;
    pr.redo = 1;
    pr.stall = 0;
    pr.kspl = 1;
    pr.units = p1.redo_units;
    pr.hist = nullptr;   // the histograms were zeroed by the first launch
    pr.num_units = &hdr->redo_count;
    pr.sched_ctr = &hdr->fix_ctr;
    const int64_t redo_max = int64_t(num_heads) * (L.lse_stride / kTile);
    const int grid_r = int(redo_max < sms ? redo_max : sms);
    if (fixed_ref) {
      e = launch_imp_pass(1, head_dim, fp8, maps, pr, grid_r, stream);
      if (e != cudaSuccess) return cuda_fail(e, "pass-1 redo launch");
    }
  }
  if (stages & TSEL_IMP_STAGE_PASS2) {
    const CUtensorMap maps[4] = {km64, km16, qm64, qm16};
    ImpPassParams p2 = p;
    p2.units = reinterpret_cast<const uint2*>(ws + L.units2);
    p2.num_units = &hdr->num_units[1];
    p2.sched_ctr = &hdr->sched_ctr[1];
    p2.hgroups = hgroups;
    p2.Tk = total_k;
    p2.kpair_off = reinterpret_cast<const int32_t*>(ws + L.kpair_off);
    p2.grp_ctr = reinterpret_cast<int32_t*>(ws + L.grp_ctr);
    p2.part = reinterpret_cast<float*>(ws + L.part);
    const int grid = int(L.u2_max < sms ? L.u2_max : sms);
    e = launch_imp_pass(2, head_dim, fp8, maps, p2, grid, stream);
    if (e != cudaSuccess) return cuda_fail(e, "pass-2 launch");
  }
  return TSEL_OK;
}

// Host checks of the top-B arguments (tsel_select_topk and the fused path).
tsel_status check_select_args(const float* scores, int total_tokens, const int32_t* req_tok_offsets,
                              int num_req, const int32_t* keep_per_req, int total_keep,
                              int32_t* keep_idx, int32_t* cu_keep) {
  if (num_req < 0 || total_tokens < 0 || (total_keep < 0 && total_keep != TSEL_KEEP_FROM_DEVICE))
    return fail(TSEL_ERR_INVALID_VALUE, "negative size");
  const int capacity = total_keep == TSEL_KEEP_FROM_DEVICE ? total_tokens : total_keep;
  if (req_tok_offsets == nullptr || keep_per_req == nullptr || cu_keep == nullptr ||
      (total_tokens > 0 && scores == nullptr) || (capacity > 0 && keep_idx == nullptr))
    return fail(TSEL_ERR_INVALID_VALUE, "null pointer");
  return TSEL_OK;
}

}  // namespace

extern "C" {

tsel_status tsel_importance(const void* q, int64_t q_row_stride, const void* k,
                            int64_t k_row_stride, const int32_t* cu_seqlens_q,
                            const int32_t* cu_seqlens_k, int num_seg, int total_q, int total_k,
                            int max_seqlen_q, int max_seqlen_k, int num_heads, int num_kv_heads,
                            int head_dim, float softmax_scale, unsigned flags, float* lse,
                            float* scores, void* workspace, size_t workspace_bytes,
                            void* stream_) {
  if (num_seg < 0 || total_q < 0 || total_k < 0 || num_heads < 1)
    return fail(TSEL_ERR_INVALID_VALUE, "negative size or no heads");
  const SelHist none{nullptr, 0, nullptr};
  const size_t need = size_t(imp_ws_layout(num_seg, total_q, total_k, num_heads).total);
  return importance_impl(q, q_row_stride, k, k_row_stride, cu_seqlens_q, cu_seqlens_k, num_seg,
                         total_q, total_k, max_seqlen_q, max_seqlen_k, num_heads, num_kv_heads,
                         head_dim, softmax_scale, flags, lse, scores, workspace, workspace_bytes,
                         need, none, static_cast<cudaStream_t>(stream_));
}

int tsel_importance_one_launch(int num_seg, int total_q, int total_k, int max_seqlen_q,
                               int max_seqlen_k, int num_heads, int head_dim, unsigned flags) {
  if (!(head_dim == 64 || head_dim == 80 || head_dim == 96 || head_dim == 112 || head_dim == 128))
    return 0;
  int sms = 0;
  if (sm_count(&sms) != 0) return -1;
  cudaError_t e = cudaSuccess;
  const bool one = one_launch_eligible(flags, num_seg, total_q, total_k, max_seqlen_q, max_seqlen_k,
                                       num_heads, head_dim, sms, &e);
  return e != cudaSuccess ? -1 : (one ? 1 : 0);
}

size_t tsel_score_select_workspace_size(int num_seg, int total_q, int total_k, int num_heads,
                                        int num_req) {
  if (num_seg < 0 || total_q < 0 || total_k < 0 || num_heads < 1 || num_req < 0) return 0;
  const ImpWsLayout L = imp_ws_layout(num_seg, total_q, total_k, num_heads);
  return size_t(sel_hist_offset(L) + sel_hist_bytes(num_req));
}

tsel_status tsel_score_select(const void* q, int64_t q_row_stride, const void* k,
                              int64_t k_row_stride, const int32_t* cu_seqlens_q,
                              const int32_t* cu_seqlens_k, int num_seg, int total_q, int total_k,
                              int max_seqlen_q, int max_seqlen_k, int num_heads,
                              int num_kv_heads, int head_dim, float softmax_scale, unsigned flags,
                              float* lse, float* scores, const int32_t* req_tok_offsets,
                              int num_req, const int32_t* keep_per_req, int total_keep,
                              int32_t* keep_idx, int32_t* cu_keep, void* workspace,
                              size_t workspace_bytes, void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  if (num_seg < 0 || total_q < 0 || total_k < 0 || num_heads < 1)
    return fail(TSEL_ERR_INVALID_VALUE, "negative size or no heads");
  tsel_status st = check_select_args(scores, total_k, req_tok_offsets, num_req, keep_per_req,
                                     total_keep, keep_idx, cu_keep);
  if (st != TSEL_OK) return st;
  const ImpWsLayout L = imp_ws_layout(num_seg, total_q, total_k, num_heads);
  const int64_t hbytes = sel_hist_bytes(num_req);
  SelHist sel{req_tok_offsets, num_req, nullptr};
  bool selected = false;
  sel.keep = keep_per_req;
  sel.total_keep = total_keep;
  sel.keep_idx = keep_idx;
  sel.cu_keep = cu_keep;
  sel.selected = &selected;
  // Histograms only for requests the top-B splits over a cluster of CTAs
  // (one CTA per request runs its radix rounds without cluster barriers).
  cudaError_t ce = cudaSuccess;
  const bool clustered = num_req > 0 && topk_cluster_size(total_k, num_req, &ce) > 1;
  if (ce != cudaSuccess) return cuda_fail(ce, "top-B cluster size");
  if (hbytes > 0 && workspace != nullptr && clustered)
    sel.hist = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) + sel_hist_offset(L));
  const size_t need = size_t(sel_hist_offset(L) + hbytes);
  st = importance_impl(q, q_row_stride, k, k_row_stride, cu_seqlens_q, cu_seqlens_k, num_seg,
                       total_q, total_k, max_seqlen_q, max_seqlen_k, num_heads, num_kv_heads,
                       head_dim, softmax_scale, flags, lse, scores, workspace, workspace_bytes,
                       need, sel, stream);
  if (st != TSEL_OK) return st;
  if (selected) return TSEL_OK;   // the one-launch importance kernel also took the top-B
  const unsigned stage_bits = TSEL_IMP_STAGE_PREP | TSEL_IMP_STAGE_PASS1 | TSEL_IMP_STAGE_PASS2 |
                              TSEL_SEL_STAGE_TOPK;
  if ((flags & stage_bits) && !(flags & TSEL_SEL_STAGE_TOPK)) return TSEL_OK;
  WsHeader* hdr = static_cast<WsHeader*>(workspace);
  cudaError_t e;
  if (num_req == 0) {
    e = cudaMemsetAsync(cu_keep, 0, sizeof(int32_t), stream);
    return e == cudaSuccess ? TSEL_OK : cuda_fail(e, "memset cu_keep");
  }
  // After the schedule stage of this call the caller's inputs are final
  // (its launch releases the later kernels only after its own wait).
  const bool chained = (flags & stage_bits) == 0;
  e = launch_topk(scores, total_k, req_tok_offsets, num_req, keep_per_req, total_keep, keep_idx,
                  cu_keep, &hdr->status, sel.hist, &hdr->hist_ok, chained ? 1 : 0, stream);
  return e == cudaSuccess ? TSEL_OK : cuda_fail(e, "top-k launch");
}

tsel_status tsel_select_topk(const float* scores, int total_tokens,
                             const int32_t* req_tok_offsets, int num_req,
                             const int32_t* keep_per_req, int total_keep, int32_t* keep_idx,
                             int32_t* cu_keep, void* workspace, size_t workspace_bytes,
                             void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  tsel_status st = check_select_args(scores, total_tokens, req_tok_offsets, num_req, keep_per_req,
                                     total_keep, keep_idx, cu_keep);
  if (st != TSEL_OK) return st;
  if (workspace == nullptr) return fail(TSEL_ERR_INVALID_VALUE, "null workspace");
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < kWsHeaderBytes)
    return fail(TSEL_ERR_WORKSPACE, "workspace must be >= %d bytes, 256-byte aligned",
                kWsHeaderBytes);
  if (num_req == 0) {
    cudaError_t e = cudaMemsetAsync(cu_keep, 0, sizeof(int32_t), stream);
    return e == cudaSuccess ? TSEL_OK : cuda_fail(e, "memset cu_keep");
  }
  WsHeader* hdr = static_cast<WsHeader*>(workspace);
  cudaError_t e = launch_topk(scores, total_tokens, req_tok_offsets, num_req, keep_per_req,
                              total_keep, keep_idx, cu_keep, &hdr->status, nullptr, nullptr, 0,
                              stream);
  return e == cudaSuccess ? TSEL_OK : cuda_fail(e, "top-k launch");
}

size_t tsel_select_topk_hist_workspace_size(int num_req) {
  if (num_req < 0) return 0;
  return size_t(kWsHeaderBytes + sel_hist_bytes(num_req));
}

tsel_status tsel_select_topk_hist(const float* scores, int total_tokens,
                                  const int32_t* req_tok_offsets, int num_req,
                                  const int32_t* keep_per_req, int total_keep, int32_t* keep_idx,
                                  int32_t* cu_keep, void* workspace, size_t workspace_bytes,
                                  void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  tsel_status st = check_select_args(scores, total_tokens, req_tok_offsets, num_req, keep_per_req,
                                     total_keep, keep_idx, cu_keep);
  if (st != TSEL_OK) return st;
  if (workspace == nullptr) return fail(TSEL_ERR_INVALID_VALUE, "null workspace");
  const int64_t hbytes = sel_hist_bytes(num_req);
  const size_t need = size_t(kWsHeaderBytes + hbytes);
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < need)
    return fail(TSEL_ERR_WORKSPACE, "workspace must be >= %zu bytes, 256-byte aligned", need);
  if (num_req == 0) {
    cudaError_t e = cudaMemsetAsync(cu_keep, 0, sizeof(int32_t), stream);
    return e == cudaSuccess ? TSEL_OK : cuda_fail(e, "memset cu_keep");
  }
  WsHeader* hdr = static_cast<WsHeader*>(workspace);
  int32_t* hist = nullptr;
  cudaError_t e = cudaSuccess;
  const bool clustered = topk_cluster_size(total_tokens, num_req, &e) > 1;
  if (e != cudaSuccess) return cuda_fail(e, "top-B cluster size");
  if (hbytes > 0 && total_tokens > 0 && clustered) {
    int sms = 0;
    if (sm_count(&sms) != 0) return fail(TSEL_ERR_CUDA, "cannot query the SM count");
    hist = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) + kWsHeaderBytes);
    e = cudaMemsetAsync(hist, 0, size_t(hbytes), stream);
    if (e != cudaSuccess) return cuda_fail(e, "memset histograms");
    e = launch_topk_hist(scores, total_tokens, req_tok_offsets, num_req, hist, &hdr->hist_ok, sms,
                         stream);
    if (e != cudaSuccess) return cuda_fail(e, "histogram launch");
  }
  e = launch_topk(scores, total_tokens, req_tok_offsets, num_req, keep_per_req, total_keep,
                  keep_idx, cu_keep, &hdr->status, hist, hist ? &hdr->hist_ok : nullptr, 0, stream);
  return e == cudaSuccess ? TSEL_OK : cuda_fail(e, "top-k launch");
}

namespace {

tsel_status gather_impl(const void* hidden, int64_t hidden_row_stride, int hidden_dim,
                        int elem_bytes, const int32_t* pos, int pos_dim,
                        const int32_t* cu_seqlens_k, int num_seg, int total_k,
                        const int32_t* keep_idx, int total_keep, const int32_t* num_kept,
                        void* out_hidden, int32_t* out_pos, int32_t* out_img_id,
                        int32_t* out_cu_seqlens, void* workspace, size_t workspace_bytes,
                        cudaStream_t stream) {
  if (num_seg < 0 || total_k < 0 || total_keep < 0 || hidden_dim < 0 || pos_dim < 0 ||
      pos_dim > 8 || !(elem_bytes == 1 || elem_bytes == 2 || elem_bytes == 4 || elem_bytes == 8))
    return fail(TSEL_ERR_INVALID_VALUE, "bad size argument");
  if (hidden_row_stride == 0) hidden_row_stride = hidden_dim;
  const int64_t row_bytes = int64_t(hidden_dim) * elem_bytes;
  const int64_t stride_bytes = hidden_row_stride * elem_bytes;
  if (row_bytes % 16 != 0 || stride_bytes % 16 != 0 || hidden_row_stride < hidden_dim ||
      row_bytes > (int64_t(1) << 30))
    return fail(TSEL_ERR_INVALID_VALUE, "row bytes %lld / stride %lld not multiples of 16",
                (long long)row_bytes, (long long)stride_bytes);
  if (cu_seqlens_k == nullptr || out_cu_seqlens == nullptr || workspace == nullptr)
    return fail(TSEL_ERR_INVALID_VALUE, "null pointer");
  if (total_keep > 0 && (keep_idx == nullptr || out_img_id == nullptr ||
                         (row_bytes > 0 && (hidden == nullptr || out_hidden == nullptr)) ||
                         (pos_dim > 0 && (pos == nullptr || out_pos == nullptr))))
    return fail(TSEL_ERR_INVALID_VALUE, "null pointer");
  if ((hidden && !aligned16(hidden)) || (out_hidden && !aligned16(out_hidden)))
    return fail(TSEL_ERR_INVALID_VALUE, "hidden buffers must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < kWsHeaderBytes)
    return fail(TSEL_ERR_WORKSPACE, "workspace must be >= %d bytes, 256-byte aligned",
                kWsHeaderBytes);
  int sms = 0;
  if (sm_count(&sms) != 0) return fail(TSEL_ERR_CUDA, "cannot query the SM count");
  WsHeader* hdr = static_cast<WsHeader*>(workspace);
  cudaError_t e = launch_gather(hidden, stride_bytes, int(row_bytes), pos, pos_dim, cu_seqlens_k,
                                num_seg, total_k, keep_idx, total_keep, num_kept, out_hidden,
                                out_pos, out_img_id, out_cu_seqlens, &hdr->status, sms, stream);
  return e == cudaSuccess ? TSEL_OK : cuda_fail(e, "gather launch");
}

}  // namespace

tsel_status tsel_gather_compact(const void* hidden, int64_t hidden_row_stride, int hidden_dim,
                                int elem_bytes, const int32_t* pos, int pos_dim,
                                const int32_t* cu_seqlens_k, int num_seg, int total_k,
                                const int32_t* keep_idx, int total_keep, void* out_hidden,
                                int32_t* out_pos, int32_t* out_img_id, int32_t* out_cu_seqlens,
                                void* workspace, size_t workspace_bytes, void* stream_) {
  return gather_impl(hidden, hidden_row_stride, hidden_dim, elem_bytes, pos, pos_dim,
                     cu_seqlens_k, num_seg, total_k, keep_idx, total_keep, nullptr, out_hidden,
                     out_pos, out_img_id, out_cu_seqlens, workspace, workspace_bytes,
                     static_cast<cudaStream_t>(stream_));
}

tsel_status tsel_gather_compact_counted(const void* hidden, int64_t hidden_row_stride,
                                        int hidden_dim, int elem_bytes, const int32_t* pos,
                                        int pos_dim, const int32_t* cu_seqlens_k, int num_seg,
                                        int total_k, const int32_t* keep_idx,
                                        const int32_t* num_kept, int max_kept, void* out_hidden,
                                        int32_t* out_pos, int32_t* out_img_id,
                                        int32_t* out_cu_seqlens, void* workspace,
                                        size_t workspace_bytes, void* stream_) {
  if (num_kept == nullptr) return fail(TSEL_ERR_INVALID_VALUE, "null num_kept");
  return gather_impl(hidden, hidden_row_stride, hidden_dim, elem_bytes, pos, pos_dim,
                     cu_seqlens_k, num_seg, total_k, keep_idx, max_kept, num_kept, out_hidden,
                     out_pos, out_img_id, out_cu_seqlens, workspace, workspace_bytes,
                     static_cast<cudaStream_t>(stream_));
}

tsel_status tsel_dynamic_budget(const float* scores, int total_tokens,
                                const int32_t* req_tok_offsets, int num_req, int mass_permille,
                                int min_permille, int max_permille, int32_t* keep_per_req,
                                int32_t* total_keep, void* workspace, size_t workspace_bytes,
                                void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  if (num_req < 0 || total_tokens < 0) return fail(TSEL_ERR_INVALID_VALUE, "negative size");
  if (mass_permille < 0 || mass_permille > 1000 || min_permille < 0 ||
      max_permille > 1000 || min_permille > max_permille)
    return fail(TSEL_ERR_INVALID_VALUE, "permille arguments %d/%d/%d", mass_permille,
                min_permille, max_permille);
  if (req_tok_offsets == nullptr || workspace == nullptr ||
      (num_req > 0 && keep_per_req == nullptr) || (total_tokens > 0 && scores == nullptr))
    return fail(TSEL_ERR_INVALID_VALUE, "null pointer");
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < kWsHeaderBytes)
    return fail(TSEL_ERR_WORKSPACE, "workspace must be >= %d bytes, 256-byte aligned",
                kWsHeaderBytes);
  if (num_req == 0) {
    if (total_keep == nullptr) return TSEL_OK;
    cudaError_t e = cudaMemsetAsync(total_keep, 0, sizeof(int32_t), stream);
    return e == cudaSuccess ? TSEL_OK : cuda_fail(e, "memset total_keep");
  }
  WsHeader* hdr = static_cast<WsHeader*>(workspace);
  cudaError_t e = launch_budget(scores, total_tokens, req_tok_offsets, num_req, mass_permille,
                                min_permille, max_permille, keep_per_req, total_keep,
                                &hdr->status, stream);
  return e == cudaSuccess ? TSEL_OK : cuda_fail(e, "budget launch");
}

tsel_status tsel_read_device_status(const void* workspace, uint32_t* bits, void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  if (workspace == nullptr) return fail(TSEL_ERR_INVALID_VALUE, "null workspace");
  uint32_t word = 0;
  cudaError_t e = cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "read status");
  if (bits) *bits = word;
  return word == 0 ? TSEL_OK : fail(TSEL_ERR_DEVICE_CHECK, "device status 0x%x", word);
}

tsel_status tsel_importance_redo_pairs(const void* workspace, int32_t* pairs, void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  if (workspace == nullptr || pairs == nullptr) return fail(TSEL_ERR_INVALID_VALUE, "null argument");
  const auto* hdr = static_cast<const WsHeader*>(workspace);
  cudaError_t e = cudaMemcpyAsync(pairs, &hdr->redo_count, sizeof(int32_t), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  return e == cudaSuccess ? TSEL_OK : cuda_fail(e, "read redo count");
}

tsel_status tsel_select_path_counts(const void* workspace, int32_t* counts, void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  if (workspace == nullptr || counts == nullptr) return fail(TSEL_ERR_INVALID_VALUE, "null argument");
  const auto* hdr = static_cast<const WsHeader*>(workspace);
  cudaError_t e = cudaMemcpyAsync(counts, hdr->sel_paths, sizeof(hdr->sel_paths),
                                  cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  return e == cudaSuccess ? TSEL_OK : cuda_fail(e, "read path counts");
}

tsel_status tsel_clear_device_status(void* workspace, void* stream_) {
  if (workspace == nullptr) return fail(TSEL_ERR_INVALID_VALUE, "null workspace");
  cudaError_t e = cudaMemsetAsync(workspace, 0, sizeof(uint32_t), static_cast<cudaStream_t>(stream_));
  return e == cudaSuccess ? TSEL_OK : cuda_fail(e, "clear status");
}

tsel_status tsel_probe_ex2(int blocks, int iters, float* sink, void* stream_) {
  if (blocks < 1 || iters < 1 || sink == nullptr) return fail(TSEL_ERR_INVALID_VALUE, "bad probe args");
  if ((reinterpret_cast<uintptr_t>(sink) & 7u) != 0)
    return fail(TSEL_ERR_INVALID_VALUE, "probe sink must be 8-byte aligned");
  cudaError_t e = launch_probe_ex2(blocks, iters, sink, static_cast<cudaStream_t>(stream_));
  return e == cudaSuccess ? TSEL_OK : cuda_fail(e, "probe launch");
}

}  // extern "C"
