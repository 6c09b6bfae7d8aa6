/*
 * tsel.h — C ABI of libtsel: attention-score vision-token pruning on one
 * NVIDIA GB300 (sm_103a).
 *
 * The library scores every visual token by the mean softmax attention it
 * receives, keeps the global top-B tokens of each request's pooled candidate
 * set, and compacts the kept rows with their original indices. It follows:
 *
 *   [LiteVLM]  "LiteVLM: A Low-Latency Vision-Language Model Inference
 *              Pipeline for Resource-Constrained Environments" (paper
 *              review), section 3.2 "Token Selection Module" and the core
 *              formula s_j = Attn(h_dec, v_j); keep ratio r.
 *   [VTC]      The dynamic vision-token compression / SERE article (REDtech),
 *              section 3.1 (VisionZip: dominant tokens found by attention
 *              score), section 3.2 (mean attention received per visual token
 *              at a ViT layer; one candidate pool and one global budget per
 *              request; blockwise probability recovery from the softmax LSE
 *              with a column reduction, only per-token scores leave the
 *              kernel; lengths, image boundaries, original indices and
 *              positions updated after pruning), section 3.3 (unified top-k).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All tensor arguments are DEVICE pointers owned by the caller; the library
 *   allocates no device memory and keeps no pointer after a call returns.
 *   Scratch space is the caller's `workspace` (size from the matching
 *   *_workspace_size function, 256-byte aligned). One workspace serves one
 *   call in flight at a time.
 * - Every call enqueues its kernels on `stream` (a cudaStream_t; NULL is the
 *   legacy default stream) and returns without synchronising.
 * - Host-side checks (null pointers, sizes, alignment, supported shapes) fail
 *   synchronously with TSEL_ERR_INVALID_VALUE or TSEL_ERR_UNSUPPORTED before
 *   anything is enqueued. A failed launch returns TSEL_ERR_CUDA.
 * - Checks that need device data (cu_seqlens, offsets, keep counts, keep
 *   indices) run inside the kernels: a violation sets a bit of the device
 *   status word held in the first bytes of the workspace (TSEL_DEV_* below),
 *   and the affected work is skipped without touching memory out of range.
 *   tsel_read_device_status() returns that word; a fresh workspace must have
 *   it cleared first (tsel_clear_device_status, or zero-filled memory), since
 *   calls only ever set bits. Device waits are bounded:
 *   a wait that runs out sets TSEL_DEV_TIMEOUT and the kernel returns.
 * - No C++ exception crosses this ABI. There is no CPU fallback.
 * - Token index arrays are int32; bf16 tensors are row-major with the
 *   head dimension innermost.
 */
#ifndef TSEL_H_
#define TSEL_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define TSEL_API __attribute__((visibility("default")))
#else
#define TSEL_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum tsel_status {
  TSEL_OK = 0,
  TSEL_ERR_INVALID_VALUE = 1, /* bad pointer, size, stride or alignment */
  TSEL_ERR_UNSUPPORTED = 2,   /* valid request this library does not handle */
  TSEL_ERR_WORKSPACE = 3,     /* workspace missing, too small or misaligned */
  TSEL_ERR_CUDA = 4,          /* CUDA runtime/driver error (launch, device) */
  TSEL_ERR_DEVICE_CHECK = 5   /* a device-side check fired (see status word) */
} tsel_status;

/* Bits of the device status word (tsel_read_device_status). */
#define TSEL_DEV_SEQLENS   0x1u  /* cu_seqlens not monotone / wrong ends / > max_seqlen */
#define TSEL_DEV_REQUESTS  0x2u  /* request offsets or keep counts out of range */
#define TSEL_DEV_KEEP_IDX  0x4u  /* keep_idx out of range or not strictly ascending */
#define TSEL_DEV_TIMEOUT   0x8u  /* a bounded device wait gave up */
#define TSEL_DEV_NAN       0x10u /* NaN score given to the top-B selection or budget */

/* total_keep value of tsel_select_topk when the budgets were computed on the
 * device (tsel_dynamic_budget): keep_idx then has room for total_tokens. */
#define TSEL_KEEP_FROM_DEVICE (-1)

/* tsel_importance flags */
#define TSEL_IMP_LSE_PROVIDED 0x1u   /* lse is an INPUT (natural log [H, Tq], e.g. the softmax
                                        LSE FlashAttention returned): the row-LSE pass is
                                        replaced by importing it */
#define TSEL_IMP_FP8_E4M3     0x2u   /* q and k hold FP8 E4M3 bytes (row strides in bytes);
                                        fold their dequantisation scales into
                                        softmax_scale ([LiteVLM] FP8 deployment) */
#define TSEL_IMP_SCORE_SUM    0x4u   /* scores are the total attention received,
                                        sum_h sum_i P, not divided by H * Nq_g */
#define TSEL_IMP_ROWREF_FIXED  0x8u  /* row-LSE pass: fixed row reference + redo launch, */
#define TSEL_IMP_ROWREF_MOVING 0x20u /*   or moving reference, one launch; neither = chosen
                                        by size (fixed from 2^28 = H*total_q*max_seqlen_k
                                        attended pairs). Same results up to fp32 rounding. */
#define TSEL_IMP_TWO_PASS     0x40u  /* always the scheduled two-pass launches, also for the
                                        small problems the one-launch path would take */
#define TSEL_IMP_TEST_STALL   0x10000u /* test hook for failure detection: the pass kernels'
                                          scheduler publishes no work, every bounded wait
                                          runs out after ~50 ms and TSEL_DEV_TIMEOUT is set
                                          (the one-launch path issues no loads instead);
                                          no copy or MMA is in flight, the context stays
                                          usable. Scores are not written. */
#define TSEL_IMP_STAGE_PREP   0x100u /* run only the listed stages (none listed = all): */
#define TSEL_IMP_STAGE_PASS1  0x200u /*   schedule/validation, row-LSE pass, column pass. */
#define TSEL_IMP_STAGE_PASS2  0x400u /*   Stages run in order on one stream/workspace; each
                                          pass needs a schedule stage after the previous
                                          run of that pass (it resets the pass's counters). */
#define TSEL_SEL_STAGE_TOPK   0x800u /* tsel_score_select only: the top-B stage (listed with
                                        the TSEL_IMP_STAGE_* bits to time the stages apart) */

/* ------------------------------------------------------------------------ */
/* Importance scores                                                        */
/* ------------------------------------------------------------------------ */

/* Bytes of workspace tsel_importance needs for these sizes. */
TSEL_API size_t tsel_importance_workspace_size(int num_seg, int total_q, int total_k, int num_heads);

/*
 * Mean attention probability each key token receives ([LiteVLM] section 3.2,
 * s_j = Attn(h, v_j); [VTC] section 3.2, mean attention received, computed
 * blockwise from the softmax LSE with a column reduction so the attention
 * matrix never reaches memory).
 *
 * For segment g, queries Q[cu_seqlens_q[g] : cu_seqlens_q[g+1]] attend to
 * keys K[cu_seqlens_k[g] : cu_seqlens_k[g+1]] (block-diagonal varlen
 * attention, no causal mask). With s = softmax_scale and kvh(h) = h / (H/Hkv):
 *   P[h,i,j] = exp(s * q_{i,h} . k_{j,kvh(h)} - lse[h,i]),
 *   lse[h,i] = log sum_j exp(s * q_{i,h} . k_{j,kvh(h)})     (natural log)
 *   scores[j] = (1 / (H * Nq_g)) * sum_h sum_i P[h,i,j]
 * so each segment's scores sum to 1. Keys of a segment with no queries get 0;
 * query rows of a segment with no keys get lse = -inf.
 *
 * q            bf16 [total_q, num_heads, head_dim]; row r starts at
 *              q + r*q_row_stride elements (0 = dense, num_heads*head_dim).
 *              16-byte aligned; q_row_stride*2 a multiple of 16.
 * k            bf16 [total_k, num_kv_heads, head_dim]; same rules.
 * cu_seqlens_q int32 [num_seg+1] device; cu_seqlens_k int32 [num_seg+1].
 *              Checked on the device: start 0, monotone, end at total_q /
 *              total_k, lengths <= max_seqlen_q / max_seqlen_k.
 * num_heads    H in [1, 256]; num_kv_heads divides it.
 * head_dim     64, 80, 96, 112 or 128 (else TSEL_ERR_UNSUPPORTED).
 * softmax_scale  <= 0 selects 1/sqrt(head_dim).
 * flags        0, TSEL_IMP_LSE_PROVIDED, TSEL_IMP_FP8_E4M3, TSEL_IMP_SCORE_SUM,
 *              TSEL_IMP_TWO_PASS and/or TSEL_IMP_STAGE_* bits.
 *              With TSEL_IMP_FP8_E4M3, q and k are E4M3 [rows, heads, head_dim] (one byte
 *              per element, row strides in bytes, multiples of 16) and softmax_scale is
 *              the full factor applied to the fp8 dot products (scale x q_scale x
 *              k_scale; must be > 0).
 * lse          fp32 [num_heads, total_q], natural log: an output (may be NULL), or
 *              with TSEL_IMP_LSE_PROVIDED an input that must not be NULL — the
 *              [VTC] section 3.2 design, which reuses the LSE the attention kernel
 *              already produced and runs only the column pass.
 * scores       out fp32 [total_k].
 * workspace    >= tsel_importance_workspace_size(num_seg, total_q, total_k,
 *              num_heads) bytes; holds the status word and the schedule.
 *
 * Kernels, in order on `stream` (no host synchronisation; capturable): the
 * schedule kernel, the row-LSE pass, its redo launch (large problems only),
 * the column pass. Small problems take one launch instead: when every
 * segment has at most 256 query rows and 256 keys (max_seqlen_q and
 * max_seqlen_k <= 256), num_heads <= 16, num_seg * num_heads no more than the
 * GPU's SMs with every segment's cluster of CTAs resident at once, no ROWREF or
 * STAGE bits and not TSEL_IMP_TWO_PASS (bf16 or E4M3 inputs), one CTA per
 * (segment, head) computes both passes from TMEM (each row's reference follows
 * its max; with TSEL_IMP_LSE_PROVIDED only the column sums, from the caller's
 * LSE) and the heads of a segment add their per-key sums over a thread-block
 * cluster in head order. Both forms give the same scores up to fp32 rounding,
 * each deterministically (tsel_importance_one_launch tells which a call takes).
 * On large problems (or with TSEL_IMP_ROWREF_FIXED) the
 * row-LSE pass fixes each row's reference max on its first 64 keys; a query
 * pair with a row whose sum then leaves the fp32 range (logits more than ~88
 * above that maximum) is redone by the redo launch with a moving reference,
 * which otherwise exits at once. Results do not depend on which rows took
 * the redo beyond fp32 rounding.
 */
TSEL_API tsel_status tsel_importance(const void* q, int64_t q_row_stride,
                            const void* k, int64_t k_row_stride,
                            const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                            int num_seg, int total_q, int total_k,
                            int max_seqlen_q, int max_seqlen_k,
                            int num_heads, int num_kv_heads, int head_dim,
                            float softmax_scale, unsigned flags,
                            float* lse, float* scores,
                            void* workspace, size_t workspace_bytes, void* stream);

/*
 * Whether tsel_importance with these sizes and flags takes the one-launch path
 * for small problems (1) or the scheduled two-pass launches (0); -1 on a CUDA
 * error (queried on the current device). Host-side only: enqueues nothing.
 */
TSEL_API int tsel_importance_one_launch(int num_seg, int total_q, int total_k,
                                        int max_seqlen_q, int max_seqlen_k, int num_heads,
                                        int head_dim, unsigned flags);

/*
 * Same scores as tsel_importance, for callers that cannot allocate device
 * memory and have no workspace to pass: plugins of an inference engine whose
 * memory pool already owns all of HBM, or embedded/automotive stacks that
 * forbid allocation after start-up. None of the pages has a counterpart of
 * this entry point; it is a deployment convenience.
 *
 * Scratch comes from one static device array of 16 MiB inside the library
 * (held by every GPU that loads the library until the process exits). A
 * problem whose tsel_importance_workspace_size() exceeds 16 MiB is rejected
 * with TSEL_ERR_WORKSPACE. The call allocates nothing (no cudaMalloc, no
 * library allocator). The first call on each device looks up the array's
 * device address (cudaGetSymbolAddress) with that device current; make that
 * first call before any stream capture. Every call on a device shares the
 * array: its status word is cleared at the start of each call, and calls that
 * overlap on the GPU race on the array, so serialise them.
 *
 * Arguments are those of tsel_importance (flags fixed to 0). device_status,
 * if not NULL, is a device uint32 that receives this call's TSEL_DEV_* bits.
 * The array used is the one of the calling thread's current device, so
 * `stream` must belong to that device (else TSEL_ERR_INVALID_VALUE).
 */
TSEL_API tsel_status tsel_importance_noalloc(const void* q, int64_t q_row_stride,
                                             const void* k, int64_t k_row_stride,
                                             const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                             int num_seg, int total_q, int total_k,
                                             int max_seqlen_q, int max_seqlen_k,
                                             int num_heads, int num_kv_heads, int head_dim,
                                             float softmax_scale, float* lse, float* scores,
                                             uint32_t* device_status, void* stream);

/* ------------------------------------------------------------------------ */
/* Importance and pooled top-B in one call                                  */
/* ------------------------------------------------------------------------ */

/* Bytes of workspace tsel_score_select needs: the importance workspace plus,
 * for 1 to 64 requests, 270,336 bytes of score histograms per request. */
TSEL_API size_t tsel_score_select_workspace_size(int num_seg, int total_q, int total_k,
                                                 int num_heads, int num_req);

/*
 * tsel_importance followed by tsel_select_topk on its scores, with the same
 * results (scores and LSE bit for bit, keep_idx and cu_keep identical), and
 * the selection started from histograms built while the scores are written:
 * the column pass also counts every request's scores by the first 11 and the
 * first 16 bits of their order-preserving keys, so the top-B needs no radix
 * round over the request's scores for those bits, and usually resolves the
 * rest with one exchange among its CTAs. [VTC] section 3.2 (one global budget
 * per request, decided from the per-token importance scores the reduction
 * kernel writes) and section 4 (fusing the steps of one decision into one
 * kernel flow); [LiteVLM] section 3.2 (keep ratio r).
 *
 * Arguments: those of tsel_importance (q ... scores, flags) followed by those
 * of tsel_select_topk (req_tok_offsets ... cu_keep) for the key tokens
 * (total_tokens = total_k), and the workspace. flags may also list
 * TSEL_SEL_STAGE_TOPK with the TSEL_IMP_STAGE_* bits to run the stages
 * separately (in order, on one workspace). Requests whose offsets are not
 * ordered, more than 64 requests, or scores not all written by this call's
 * column pass make the top-B run its plain radix rounds (same results). One
 * segment and one request on tsel_importance's one-launch path (a single
 * image of at most 256 tokens): the importance launch ranks the request's
 * keys itself (keys above, then equal keys at lower token indices) and writes
 * keep_idx and cu_keep; no top-B kernel is launched (same results).
 * workspace: >= tsel_score_select_workspace_size(...) bytes, 256-byte aligned;
 * its status word collects the device checks of both steps.
 */
TSEL_API tsel_status tsel_score_select(const void* q, int64_t q_row_stride,
                                       const void* k, int64_t k_row_stride,
                                       const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                       int num_seg, int total_q, int total_k,
                                       int max_seqlen_q, int max_seqlen_k,
                                       int num_heads, int num_kv_heads, int head_dim,
                                       float softmax_scale, unsigned flags,
                                       float* lse, float* scores,
                                       const int32_t* req_tok_offsets, int num_req,
                                       const int32_t* keep_per_req, int total_keep,
                                       int32_t* keep_idx, int32_t* cu_keep,
                                       void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------ */
/* Pooled global top-B                                                      */
/* ------------------------------------------------------------------------ */

TSEL_API size_t tsel_select_topk_workspace_size(int num_req);

/*
 * Per request r, keep the keep_per_req[r] tokens with the largest scores
 * among tokens [req_tok_offsets[r], req_tok_offsets[r+1]) — every image of
 * the request in one candidate pool under one budget ([VTC] sections 3.2 and
 * 3.3; keep ratio r of [LiteVLM] section 3.2 gives B = floor(r*N), see
 * tsel_keep_count). Order: score descending, ties to the lowest token index
 * (-0 is treated as +0). Kept token indices are written in ascending order,
 * requests concatenated; cu_keep[r] is the first output slot of request r.
 *
 * scores          fp32 [total_tokens] device (NaN sets TSEL_DEV_NAN; its
 *                 rank is then unspecified).
 * req_tok_offsets int32 [num_req+1] device: 0 <= o[r] <= o[r+1] <= total_tokens.
 * keep_per_req    int32 [num_req] device: 0 <= B_r <= o[r+1]-o[r];
 *                 sum must equal total_keep (host value, sizes keep_idx).
 *                 total_keep = TSEL_KEEP_FROM_DEVICE drops that check (budgets
 *                 written by tsel_dynamic_budget, not known on the host):
 *                 keep_idx then needs room for total_tokens entries and
 *                 cu_keep[num_req] holds the kept count.
 * keep_idx        out int32 [total_keep]; cu_keep out int32 [num_req+1].
 * A request that fails its checks sets TSEL_DEV_REQUESTS and writes nothing.
 */
TSEL_API tsel_status tsel_select_topk(const float* scores, int total_tokens,
                             const int32_t* req_tok_offsets, int num_req,
                             const int32_t* keep_per_req, int total_keep,
                             int32_t* keep_idx, int32_t* cu_keep,
                             void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of workspace tsel_select_topk_hist needs: 1 KB plus, for 1 to 64
 * requests, 270,336 bytes of histograms per request. */
TSEL_API size_t tsel_select_topk_hist_workspace_size(int num_req);

/*
 * tsel_select_topk (same arguments, same results) for scores that did not come
 * from tsel_score_select, e.g. from another scoring kernel: one launch counts
 * the scores into per-request histograms of their first 11 and 16 key bits
 * (after a memset of that region), then the top-B starts from them as in
 * tsel_score_select. More than 64 requests: the plain top-B.
 * workspace: >= tsel_select_topk_hist_workspace_size(num_req) bytes.
 */
TSEL_API tsel_status tsel_select_topk_hist(const float* scores, int total_tokens,
                                           const int32_t* req_tok_offsets, int num_req,
                                           const int32_t* keep_per_req, int total_keep,
                                           int32_t* keep_idx, int32_t* cu_keep,
                                           void* workspace, size_t workspace_bytes, void* stream);

/*
 * Dynamic keep budget per request from its scores ([VTC] section 6.2 leaves a
 * content-dependent compression ratio as future work and gives no rule; this
 * is the rule the library uses). For request r with tokens
 * [req_tok_offsets[r], req_tok_offsets[r+1]) (n_r of them):
 *   q_j  = floor(s_j * 2^(24 - E)), E the binary exponent with the request's
 *          largest score in [2^(E-1), 2^E) (integer quanta; NaN, negative
 *          and zero scores count 0);
 *   M    = sum_j q_j, T = ceil(mass_permille * M / 1000);
 *   B_r  = the fewest tokens, taken in top-B order (score descending, lowest
 *          index first), whose quanta reach T (0 when T = 0), then bounded to
 *          [floor(n_r*min_permille/1000), floor(n_r*max_permille/1000)].
 * Integer sums make B_r exact and deterministic. Feed keep_per_req to
 * tsel_select_topk with total_keep = TSEL_KEEP_FROM_DEVICE.
 *
 * scores          fp32 [total_tokens] device (NaN sets TSEL_DEV_NAN).
 * req_tok_offsets int32 [num_req+1] device (bad ranges set TSEL_DEV_REQUESTS
 *                 and give B_r = 0).
 * mass_permille   in [0, 1000]; 0 <= min_permille <= max_permille <= 1000.
 * keep_per_req    out int32 [num_req] device.
 * total_keep      out int32 device scalar = sum_r B_r (may be NULL).
 * workspace       >= tsel_select_topk_workspace_size(num_req) bytes (status).
 * Requests of up to 2^31 - 1 tokens; one thread-block cluster (up to 16 CTAs)
 * per request.
 */
TSEL_API tsel_status tsel_dynamic_budget(const float* scores, int total_tokens,
                                         const int32_t* req_tok_offsets, int num_req,
                                         int mass_permille, int min_permille, int max_permille,
                                         int32_t* keep_per_req, int32_t* total_keep,
                                         void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------ */
/* Order-preserving compaction with metadata                                */
/* ------------------------------------------------------------------------ */

TSEL_API size_t tsel_gather_compact_workspace_size(void);

/*
 * Compact the kept tokens and rebuild their metadata ([VTC] section 3.2:
 * after pruning, input lengths, image boundaries, original spatial indices
 * and position ids must stay consistent for prefill and the KV cache).
 *
 * For k in [0, total_keep), t = keep_idx[k]:
 *   out_hidden[k, :] = hidden[t, :]          (bytes copied unchanged)
 *   out_pos[k, :]    = pos[t, :]
 *   out_img_id[k]    = g with cu_seqlens_k[g] <= t < cu_seqlens_k[g+1]
 * and out_cu_seqlens[g] = number of kept tokens below cu_seqlens_k[g]
 * (the kept per-image lengths, prefix-summed). keep_idx itself is the
 * original-index output.
 *
 * hidden         [total_k rows], row t at hidden + t*hidden_row_stride
 *                elements of elem_bytes each; hidden_dim*elem_bytes and
 *                hidden_row_stride*elem_bytes multiples of 16; 16-byte aligned.
 * pos            int32 [total_k, pos_dim] dense (pos_dim in [0, 8]; NULL
 *                allowed when pos_dim == 0).
 * cu_seqlens_k   int32 [num_seg+1] device.
 * keep_idx       int32 [total_keep] device, strictly ascending, in
 *                [0, total_k) (else TSEL_DEV_KEEP_IDX and the row is skipped).
 * out_hidden     [total_keep, hidden_dim] dense, 16-byte aligned.
 * out_pos        int32 [total_keep, pos_dim] (NULL when pos_dim == 0).
 * out_img_id     int32 [total_keep]; out_cu_seqlens int32 [num_seg+1].
 */
TSEL_API tsel_status tsel_gather_compact(const void* hidden, int64_t hidden_row_stride,
                                int hidden_dim, int elem_bytes,
                                const int32_t* pos, int pos_dim,
                                const int32_t* cu_seqlens_k, int num_seg, int total_k,
                                const int32_t* keep_idx, int total_keep,
                                void* out_hidden, int32_t* out_pos,
                                int32_t* out_img_id, int32_t* out_cu_seqlens,
                                void* workspace, size_t workspace_bytes, void* stream);

/*
 * tsel_gather_compact with the kept count read on the device (e.g.
 * cu_keep + num_req from tsel_select_topk with device budgets), so no host
 * round trip is needed between the calls. K = *num_kept rows are compacted;
 * max_kept (host) sizes the launch and bounds K: outputs need room for
 * max_kept rows, and *num_kept outside [0, max_kept] sets TSEL_DEV_KEEP_IDX
 * (K is then clamped). Other arguments as in tsel_gather_compact.
 */
TSEL_API tsel_status tsel_gather_compact_counted(const void* hidden, int64_t hidden_row_stride,
                                int hidden_dim, int elem_bytes,
                                const int32_t* pos, int pos_dim,
                                const int32_t* cu_seqlens_k, int num_seg, int total_k,
                                const int32_t* keep_idx, const int32_t* num_kept, int max_kept,
                                void* out_hidden, int32_t* out_pos,
                                int32_t* out_img_id, int32_t* out_cu_seqlens,
                                void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------ */
/* Host helpers                                                             */
/* ------------------------------------------------------------------------ */

/* Budget at keep ratio keep_permille/1000: floor(n_tokens*keep_permille/1000)
 * in 64-bit integer arithmetic ([LiteVLM] section 3.2 and its results table:
 * r = 0.8 of 896 visual tokens keeps 716, so 716 + 142 text = 858 tokens).
 * Returns -1 for negative arguments. */
TSEL_API int tsel_keep_count(int n_tokens, int keep_permille);

/* Reads the device status word of `workspace` after synchronising `stream`.
 * *bits receives the TSEL_DEV_* bits (may be NULL). Returns TSEL_OK when the
 * word is zero, TSEL_ERR_DEVICE_CHECK when any bit is set, TSEL_ERR_CUDA on a
 * CUDA error. */
TSEL_API tsel_status tsel_read_device_status(const void* workspace, uint32_t* bits, void* stream);

/* Reads, after synchronising `stream`, how many (head, 256-query-row pair)s
 * the last tsel_importance call on `workspace` sent to its redo launch (rows
 * whose sum overflowed the fixed reference; see tsel_importance). 0 for
 * nearly every input; a diagnostic, not needed for correct results. */
TSEL_API tsel_status tsel_importance_redo_pairs(const void* workspace, int32_t* pairs, void* stream);

/* Reads, after synchronising `stream`, how many requests the top-B calls on
 * `workspace` resolved by each threshold path since the workspace was zeroed,
 * into counts[5]: counts[0] radix rounds over the scores (no histograms),
 * counts[1] first digit from the histograms then radix rounds, counts[2]
 * histograms and one candidate exchange, counts[3] candidate exchange rejected
 * (its counts did not bracket the budget), radix rounds from the start,
 * counts[4] ranked inside the one-launch importance kernel (tsel_score_select
 * of one segment and one request on the one-launch path). Requests with B = 0
 * are not counted. A diagnostic. */
TSEL_API tsel_status tsel_select_path_counts(const void* workspace, int32_t* counts, void* stream);

/* Enqueues a reset of the device status word to zero. */
TSEL_API tsel_status tsel_clear_device_status(void* workspace, void* stream);

TSEL_API const char* tsel_status_string(tsel_status s);

/* Detail of the last non-OK status returned on this host thread. */
TSEL_API const char* tsel_last_error(void);

/* Measurement probe: enqueues a kernel of `blocks` x 512 threads, each thread
 * issuing `iters` x 8 dependent-chain ex2.approx.f32 operations (a MUFU
 * throughput probe; the count of exp2 per launch is blocks*512*iters*8).
 * `sink` (device, 8-byte aligned, blocks*512 + 4 floats) receives one float
 * per thread so nothing is optimised away, then two uint64 words: the SM
 * clock cycles and the nanoseconds (%globaltimer) that block 0's first thread
 * took, so the SM clock during the probe is cycles / ns. */
TSEL_API tsel_status tsel_probe_ex2(int blocks, int iters, float* sink, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TSEL_H_ */
