/*
 * fa_decode.h - C ABI of libfadecode.so: batched decode attention over a
 * paged KV cache for ragged batches, on one GB300 (sm_103a).
 *
 * The calls follow the plan/run statement of the problem on the page
 * "FlashDecoding + FlashInfer - the decode-time attention story", section
 * "The API you actually use (Python)": plan() is called once per batch shape
 * and amortised, run() is the hot path.  The merge of partial softmax states
 * is the rule of section "FlashDecoding - the split-KV trick" on that page.
 *
 * Conventions shared by every entry point
 *  - Plain C types only.  Pointers are "host" or "device" as stated per
 *    argument; device pointers must come from the CUDA device that is current
 *    on the calling thread.  The caller owns every buffer, including the
 *    workspace; the library owns only the opaque plan handle.
 *  - A stream argument is a cudaStream_t passed as void* (NULL = the legacy
 *    default stream).  All device work of a call is enqueued on it.
 *  - Return value: FA_OK (0) or a negative fa_status.  On error nothing has
 *    been launched and no output has been written.
 *  - Supported shapes: page_size 16; head_dim 64 or 128;
 *    num_qo_heads / num_kv_heads in {1, 2, 4, 8}; (q, kv) element types
 *    (F32, F32), (BF16, BF16), (F16, F16), (BF16, E4M3), (F16, E4M3).
 *    Anything else returns FA_ERR_UNSUPPORTED.
 *  - Layouts (row-major, innermost last):
 *      q          [batch, num_qo_heads, head_dim]                 q dtype
 *      paged_kv   [num_pages, 2, page_size, num_kv_heads, head_dim] kv dtype
 *                 (index 0 = K, 1 = V; "NHD": tokens, then heads, then dim)
 *      o          [batch, num_qo_heads, head_dim]                 q dtype
 *      lse        [batch, num_qo_heads]                           float32
 *    Query head h reads kv head h / (num_qo_heads / num_kv_heads).
 *    lse is the natural-log log-sum-exp of the scaled logits
 *    sm_scale * q . k over the request's context.
 */
#ifndef FA_DECODE_H_
#define FA_DECODE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element types.  E4M3 is the OCP FP8 E4M3 "FN" encoding (finite, max 448). */
typedef enum {
  FA_DTYPE_F32 = 0,
  FA_DTYPE_BF16 = 1,
  FA_DTYPE_F16 = 2,
  FA_DTYPE_E4M3 = 3
} fa_dtype;

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = -1,         /* malformed arguments (shapes, indptr, NULL) */
  FA_ERR_UNSUPPORTED = -2,         /* valid but not built (dtype, head_dim, group) */
  FA_ERR_WORKSPACE_TOO_SMALL = -3, /* workspace_bytes below what the plan needs */
  FA_ERR_CUDA = -4,                /* a CUDA runtime call failed */
  FA_ERR_DEVICE_CHECK = -5         /* a kernel recorded a device-side check */
} fa_status;

/* Opaque plan handle, created by fa_decode_plan, freed by
 * fa_decode_plan_destroy.  Not thread-safe: one thread uses a plan at a time. */
typedef struct fa_decode_plan_s* fa_decode_plan_t;

/* Human-readable name of a status code.  Static storage, never NULL. */
const char* fa_status_string(int status);

/* Upper bound, in bytes, of the device workspace that fa_decode_plan needs
 * for a batch of `batch` requests with these head counts and head_dim on the
 * current CUDA device (it depends on the device's SM count).  The bound is
 * independent of the context lengths.  Returns 0 for invalid arguments. */
size_t fa_decode_workspace_size(int batch, int num_qo_heads, int num_kv_heads,
                                int head_dim);

/* plan: build the work list of one decode batch (page "FlashDecoding +
 * FlashInfer", sections "The API you actually use" and "What FlashInfer is",
 * item 3: load-balance across CTAs so that the longest sequence does not stall
 * the batch).
 *
 *  indptr_host         [batch+1] int32, host.  Request i owns page positions
 *                      indptr[i] .. indptr[i+1]-1 of indices_dev.
 *                      indptr[0] = 0, non-decreasing.
 *  indices_dev         [indptr[batch]] int32, device.  Physical page ids.  Kept
 *                      by pointer and read by every fa_decode_run of this plan:
 *                      it must stay valid and unchanged while the plan is used.
 *                      Ids may repeat across requests (shared prefixes).  May
 *                      also be page-locked host memory (cudaHostAlloc or
 *                      cudaHostRegister), which the kernels then read over
 *                      the CPU-GPU link (on a GB300 node, NVLink-C2C: about 2 %
 *                      slower than device memory, and no upload).
 *  last_page_len_host  [batch] int32, host.  Valid slots in each request's last
 *                      page, in [1, page_size]; ignored for a request with no
 *                      pages (its output is o = 0, lse = -inf).
 *  workspace_dev,      device scratch owned by the caller, at least
 *  workspace_bytes     fa_decode_workspace_size(...) bytes, 256-byte aligned.
 *                      It holds the work list and the fp32 partial states; it
 *                      must not be shared by two plans used concurrently.
 *  cuda_stream         the work list is copied into the workspace on this stream.
 *  out_plan            receives the new handle.
 *
 * Per request, len = (pages - 1) * page_size + last_page_len.  Every
 * (request, kv head, page) is assigned to exactly one chunk of the work list;
 * fa_decode_plan_get_work exposes that list for inspection.  The grid is
 * planned in groups of num_kv_heads CTAs that take equal shares of the page
 * stream, one kv head each (fa_plan_work_host_heads shows the same plan on
 * the host); FADECODE_PLAN=stream in the environment selects the plan of
 * fa_plan_work_host instead.
 * Errors: FA_ERR_INVALID_ARG for a malformed indptr or last_page_len, NULL
 * pointers or non-positive sizes; FA_ERR_UNSUPPORTED for shapes or types that
 * are not built; FA_ERR_WORKSPACE_TOO_SMALL; FA_ERR_CUDA. */
int fa_decode_plan(const int32_t* indptr_host, const int32_t* indices_dev,
                   const int32_t* last_page_len_host, int batch,
                   int num_qo_heads, int num_kv_heads, int head_dim,
                   int page_size, fa_dtype q_dtype, fa_dtype kv_dtype,
                   void* workspace_dev, size_t workspace_bytes,
                   void* cuda_stream, fa_decode_plan_t* out_plan);

/* plan for multi-token decode (speculative verification): every request
 * carries q_len query tokens - the draft tokens of speculative decoding, "a
 * handful with speculative decoding" in the page "FlashDecoding + FlashInfer"
 * (section "FlashDecoding + FlashInfer") - whose own K and V are already the
 * last q_len positions of its cache.  Query token i (0-based) attends to
 * positions 0 .. len - q_len + i: the context and the draft tokens up to
 * itself.  A later fa_decode_run of this plan takes
 *      q    [batch, q_len, num_qo_heads, head_dim]
 *      o    [batch, q_len, num_qo_heads, head_dim]
 *      lse  [batch, q_len, num_qo_heads]
 * Arguments otherwise as fa_decode_plan; every request needs len >= q_len
 * (FA_ERR_INVALID_ARG otherwise).  The workspace bound is
 * fa_decode_workspace_size(batch, num_qo_heads * q_len, num_kv_heads,
 * head_dim) for (num_qo_heads / num_kv_heads) * q_len <= 8, else
 * fa_decode_workspace_size_ragged_q.  Built for head_dim 128, (q, kv) =
 * (BF16, BF16) or (BF16, E4M3): with group x q_len <= 8 for q_len 2, 4, 8 at
 * group 1, 2, 4 at group 2 and 2 at group 4; with more columns, the kernels
 * of fa_decode_plan_ragged_q (every request holding q_len rows), up to
 * group x q_len = 32.  Other combinations return FA_ERR_UNSUPPORTED.
 * q_len = 1 is fa_decode_plan. */
int fa_decode_plan_multi_token(const int32_t* indptr_host,
                               const int32_t* indices_dev,
                               const int32_t* last_page_len_host, int batch,
                               int q_len, int num_qo_heads, int num_kv_heads,
                               int head_dim, int page_size, fa_dtype q_dtype,
                               fa_dtype kv_dtype, void* workspace_dev,
                               size_t workspace_bytes, void* cuda_stream,
                               fa_decode_plan_t* out_plan);

/* plan for decode with a different number of query tokens per request:
 * request i owns rows qo_indptr[i] .. qo_indptr[i+1] of q and o - the
 * ragged (indptr) layout of section "Ragged attention - variable-length
 * batching" of the page "FlashDecoding + FlashInfer", applied to the
 * queries, e.g. speculative verification with a draft length of its own per
 * request.  Its n_i query tokens are the last n_i positions of the request's
 * cache and query token j (0-based) attends to positions 0 .. len_i - n_i + j.
 * A later fa_decode_run of this plan takes
 *      q    [qo_indptr[batch], num_qo_heads, head_dim]
 *      o    [qo_indptr[batch], num_qo_heads, head_dim]
 *      lse  [qo_indptr[batch], num_qo_heads]
 *  qo_indptr_host  [batch + 1] int32, host, read during the call: 0 first,
 *                  non-decreasing, n_i <= len_i (n_i = 0 allowed: the
 *                  request contributes no rows; its pages are still read).
 * Arguments otherwise as fa_decode_plan; the workspace bound is
 * fa_decode_workspace_size_ragged_q.  Built for head_dim 128, (q, kv) =
 * (BF16, BF16) or (BF16, E4M3), groups 1, 2, 4, 8 with
 * group x max_i n_i <= 32 (group 8: up to 4 query tokens per request).
 * Up to 8 columns (group x n) the consumer warps split a segment's pages; with
 * more, each warp owns 8 columns and reads every page, on a kernel of as
 * many warps as the batch's widest request has 8-column tiles
 * (t = ceil(group x n_i / 8): 2, 3 or 4).  With E4M3 KV the requests of one
 * tile take a launch of their own on the 8-column kernel when they hold
 * enough work; fa_decode_run then makes both launches, one after the other
 * (fa_plan_info num_buckets, bucket_first_cta, bucket_q_len; in the
 * environment FADECODE_BUCKETS=0 plans one launch of the max_q kernel,
 * FADECODE_BUCKETS=all a launch for every tile count present).
 * Errors as fa_decode_plan; FA_ERR_UNSUPPORTED for shapes beyond those. */
int fa_decode_plan_ragged_q(const int32_t* indptr_host, const int32_t* indices_dev,
                            const int32_t* last_page_len_host,
                            const int32_t* qo_indptr_host, int batch,
                            int num_qo_heads, int num_kv_heads, int head_dim,
                            int page_size, fa_dtype q_dtype, fa_dtype kv_dtype,
                            void* workspace_dev, size_t workspace_bytes,
                            void* cuda_stream, fa_decode_plan_t* out_plan);

/* Workspace bound of any ragged-q plan of this batch and shape (the widest
 * kernel's partial states, 32 columns), current device. */
size_t fa_decode_workspace_size_ragged_q(int batch, int num_qo_heads,
                                         int num_kv_heads, int head_dim);

/* run: decode attention for one query token per request (page "FlashDecoding
 * + FlashInfer", section "FlashDecoding - the split-KV trick": every chunk of
 * the KV axis yields a partial (m, d, o), and a small reduction combines the
 * partials with the merge rule).
 *
 *  q          [batch, num_qo_heads, head_dim], plan's q dtype, device or
 *             page-locked host memory (read by the kernels over the CPU-GPU
 *             link; on a GB300 node this costs the kernel no time, and no
 *             host-to-device copy is needed), 16-byte aligned.
 *  paged_kv   [num_pages, 2, page_size, num_kv_heads, head_dim], plan's kv
 *             dtype, device, 16-byte aligned.
 *  num_pages  leading extent of paged_kv.  A page id outside [0, num_pages)
 *             reads zeros and sets the device-check word (see
 *             fa_decode_check); it never reads outside paged_kv.
 *  sm_scale   logit scale; <= 0 selects 1/sqrt(head_dim).
 *  k_scale,   per-tensor dequantisation scales of an E4M3 cache (stored code
 *  v_scale    times scale = value); use 1 for other kv types.
 *  o          [batch, num_qo_heads, head_dim], q dtype, device or page-locked
 *             host memory (written by the kernels directly), caller-allocated.
 *  lse        [batch, num_qo_heads] float32, device or page-locked host
 *             memory, or NULL to skip it.
 *
 * No allocation and no host synchronisation: the call only enqueues kernels
 * on cuda_stream, so it can be issued repeatedly between plans.  Results are
 * bitwise reproducible for a fixed plan.
 * Errors: FA_ERR_INVALID_ARG (NULL plan/q/paged_kv/o, num_pages <= 0,
 * misaligned paged_kv), FA_ERR_CUDA (encoding the TMA descriptor or a launch
 * failed). */
int fa_decode_run(fa_decode_plan_t plan, const void* q, const void* paged_kv,
                  int64_t num_pages, float sm_scale, float k_scale,
                  float v_scale, void* o, float* lse, void* cuda_stream);

/* run with per-token FP8 scales: like fa_decode_run for a plan whose kv
 * dtype is E4M3, but every stored K and V element is dequantised with the
 * scale of its own token and kv head instead of one scale per tensor - the
 * row-wise dynamic scaling that the page "FlashInfer vs FlashAttention-3"
 * (section "Production War Story: The FP8 Precision Underflow Failure")
 * names as the fix for static-scale underflow over long contexts.
 *
 *  k_scales, v_scales  [num_pages, num_kv_heads, page_size] float32, device,
 *                      16-byte aligned: the K (V) element at page p, slot t,
 *                      kv head h has the value code * scales[(p*Hkv + h)*P + t].
 * Other arguments as fa_decode_run (sm_scale <= 0 selects 1/sqrt(head_dim)).
 * Built for head_dim 128 and groups 2, 4, 8 (the tensor-core consumer); other
 * plans return FA_ERR_UNSUPPORTED, as do plans whose kv dtype is not E4M3. */
int fa_decode_run_token_scales(fa_decode_plan_t plan, const void* q,
                               const void* paged_kv, int64_t num_pages,
                               float sm_scale, const float* k_scales,
                               const float* v_scales, void* o, float* lse,
                               void* cuda_stream);

/* run with one FP8 scale per kv head: like fa_decode_run for a plan whose
 * kv dtype is E4M3, but the K (V) elements of kv head h are dequantised with
 * k_head_scales[h] (v_head_scales[h]) - scales finer than one per tensor,
 * coarser than fa_decode_run_token_scales' per token ("FlashInfer vs
 * FlashAttention-3", section "Production War Story: The FP8 Precision
 * Underflow Failure").
 *
 *  k_head_scales, v_head_scales  [num_kv_heads] float32, device, 4-byte
 *                      aligned, caller-owned: the K (V) element of kv head h
 *                      has the value code * scales[h].
 * Other arguments as fa_decode_run (sm_scale <= 0 selects 1/sqrt(head_dim)).
 * Every plan kind (plain, multi-token, ragged query rows) and kernel takes
 * it; plans whose kv dtype is not E4M3 return FA_ERR_UNSUPPORTED, NULL
 * scales FA_ERR_INVALID_ARG. */
int fa_decode_run_head_scales(fa_decode_plan_t plan, const void* q, const void* paged_kv,
                              int64_t num_pages, float sm_scale, const float* k_head_scales,
                              const float* v_head_scales, void* o, float* lse,
                              void* cuda_stream);

/* run with a unified max (page "FlashDecoding + FlashInfer", section
 * "FlashDecoding++", item 1 "Async-softmax with unified max"): instead of a
 * running maximum per query head, every weight is exp(s - max_bound) for a
 * bound on the logits s = sm_scale * k_scale * (q . k) known before the run,
 * so no page of the KV stream has to wait on a reduction of the maximum.  The
 * result is the same softmax (up to rounding); where a head's true maximum
 * lies more than 16 / log2(e) above max_bound (weights could overflow) or
 * more than 64 / log2(e) below it (weights could underflow), the kernel
 * re-centres that head on its true maximum (an exact rescale) and counts a
 * fallback (see fa_decode_unified_max_fallbacks).
 *
 *  max_bound  the static bound, natural-log units of the logits, finite.
 *             Any finite value gives a correct result; a bound near the true
 *             maxima avoids fallbacks.  One that needs no look at the scores
 *             is sm_scale * k_scale * max|q| * max|k| (Cauchy-Schwarz).
 * Other arguments as fa_decode_run.  Built for q and kv both BF16 (the
 * weights keep fp32's exponent range), groups 2, 4 and 8, head_dim 64 and
 * 128, one query token; other plans return FA_ERR_UNSUPPORTED.
 * Errors: as fa_decode_run; FA_ERR_INVALID_ARG for a non-finite bound. */
int fa_decode_run_unified_max(fa_decode_plan_t plan, const void* q,
                              const void* paged_kv, int64_t num_pages,
                              float sm_scale, float k_scale, float v_scale,
                              float max_bound, void* o, float* lse,
                              void* cuda_stream);

/* Wait for cuda_stream, then read and clear the plan's count of unified-max
 * fallbacks: (work item, consumer warp) pairs that re-centred at least one
 * head since the last read.  Synchronises; keep it off the hot path.
 * Errors: FA_ERR_INVALID_ARG (NULL plan or count), FA_ERR_CUDA. */
int fa_decode_unified_max_fallbacks(fa_decode_plan_t plan, void* cuda_stream,
                                    int* count);

/* merge_states: combine two sets of partial attention states with the merge
 * rule (page "FlashDecoding + FlashInfer", section "FlashDecoding - the
 * split-KV trick").  A state is a normalised output o_x with its natural-log
 * lse_x, i.e. (m = lse_x, d = 1, o = o_x) in the rule's notation; the result is
 * normalised again.  Two states with lse = -inf merge to o = 0, lse = -inf.
 *
 *  o_a, o_b, o_out        [n, num_heads, head_dim], `dtype` (F32, BF16, F16), device
 *  lse_a, lse_b, lse_out  [n, num_heads] float32, device
 * o_out/lse_out may alias o_a/lse_a element for element.
 * Errors: FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED (dtype E4M3 or head_dim not
 * a multiple of 4 up to 1024), FA_ERR_CUDA. */
int fa_merge_states(const void* o_a, const float* lse_a, const void* o_b,
                    const float* lse_b, void* o_out, float* lse_out, int n,
                    int num_heads, int head_dim, fa_dtype dtype,
                    void* cuda_stream);

/* Free a plan handle (host memory only; the workspace stays the caller's).
 * NULL is accepted. */
int fa_decode_plan_destroy(fa_decode_plan_t plan);

/* Summary of a plan, for logging and tests. */
typedef struct {
  int batch, num_qo_heads, num_kv_heads, head_dim, page_size;
  int num_ctas;          /* persistent decode grid */
  int ctas_per_sm;       /* occupancy the grid was sized for */
  int num_sms;
  int num_segments;      /* work items (request, kv head, page range) */
  int num_merge_units;   /* (request, kv head) pairs split over several CTAs */
  int num_partial_slots; /* fp32 partial states written by split work items */
  int threads_per_cta;
  int smem_bytes_per_cta;
  int stages;            /* depth of the shared-memory page ring */
  int64_t total_pages;   /* sum of pages over requests */
  int64_t total_tokens;  /* sum of len over requests */
  size_t workspace_bytes_used;
  size_t plan_upload_bytes;   /* bytes fa_decode_plan copies host -> device */
  int tensor_cores;           /* 1: per-page products on mma.sync, 0: CUDA cores */
  int fused_merge;            /* 1: split requests merged inside the decode kernel */
  int q_len;                  /* query tokens per request (ragged plans: the most the
                                 kernel chosen holds) */
  int unified_max;            /* 1: fa_decode_run_unified_max is built for this plan */
  int num_pool_segments;      /* segments claimed at run time (0: static quotas only) */
  int64_t pool_pages;         /* (page, kv head) pairs in those segments */
  int ragged_q;               /* 1: query rows per request from qo_indptr */
  int64_t total_q_rows;       /* query rows of q / o (batch * q_len unless ragged) */
  int num_buckets;            /* decode launches per run: 1, or more for a ragged plan in
                                 buckets by 8-column tiles (fa_decode_plan_ragged_q) */
  int bucket_first_cta[4];    /* launch b runs CTAs bucket_first_cta[b] up to the next
                                 launch's first (num_ctas for the last); -1 unused */
  int bucket_q_len[4];        /* query tokens per request launch b's kernel holds
                                 (group x bucket_q_len[b] columns); 0 unused */
} fa_plan_info;

int fa_decode_plan_get_info(fa_decode_plan_t plan, fa_plan_info* info);

/* Work list of a plan, host copy owned by the plan (valid until destroy).
 *  cta_offsets  [num_ctas+1]: CTA c runs segments cta_offsets[c] .. [c+1]-1,
 *               then claims pool segments cta_offsets[num_ctas] ..
 *               num_segments-1 one at a time, in order, until none is left
 *               (the pool is the last part of the page stream, cut into
 *               chunks that shrink towards its end; it evens out CTAs that
 *               stream pages at different rates)
 *  segments     [num_segments * FA_SEGMENT_INTS] int32, each
 *               {request, kv_head, page_begin, page_end, last_valid,
 *                out_slot, merge_unit, to_end}; page_begin/page_end index
 *               the indices array, last_valid = valid slots of the
 *               segment's final page, out_slot = -1 when the segment covers
 *               its whole request, else the partial-state slot it writes,
 *               merge_unit = its row of the merge table (-1 when unsplit),
 *               to_end = tokens from the segment's first token to the end
 *               of its request.
 *  merge        [num_merge_units * FA_MERGE_INTS] int32, each
 *               {request, kv_head, first_slot, num_slots}. */
#define FA_SEGMENT_INTS 8
#define FA_MERGE_INTS 4
int fa_decode_plan_get_work(fa_decode_plan_t plan, const int32_t** cta_offsets,
                            const int32_t** segments, const int32_t** merge);

/* Host-only planning step, no CUDA call: the work-list builder that
 * fa_decode_plan uses, exposed so it can be checked without a GPU.  Output
 * buffers are caller-owned host arrays of the stated capacities; counts are
 * written to *n_ctas, *n_segments, *n_merge, *n_slots.
 * pool_fraction in [0, 1): share of the page stream left to the run-time
 * pool (fa_decode_plan uses none unless FADECODE_POOL in the environment
 * sets a fraction up to 0.5; a pool smaller than 4 pages per CTA is not
 * made).
 * With C = max_ctas * 7 + 1 (the most cuts a plan makes), capacities needed:
 * cta_offsets max_ctas+1, segments (batch*num_kv_heads + C) *
 * FA_SEGMENT_INTS, merge C * FA_MERGE_INTS.  Errors: FA_ERR_INVALID_ARG. */
int fa_plan_work_host(const int32_t* indptr, const int32_t* last_page_len,
                      int batch, int num_kv_heads, int page_size, int max_ctas,
                      int min_pages_per_cta, double pool_fraction,
                      int32_t* cta_offsets,
                      int32_t* segments, int32_t* merge, int* n_ctas,
                      int* n_segments, int* n_merge, int* n_slots);

/* The buckets fa_decode_plan_ragged_q makes of a batch whose widest
 * request takes the column split, on the host (no CUDA call).  Request i
 * of group G with n_i = qo_indptr[i+1] - qo_indptr[i] query rows needs
 * t_i = max(1, ceil(G x n_i / 8)) 8-column tiles, at most widest_tiles (the
 * tiles of the batch's one-launch kernel, 2..4).  Every request goes to the
 * bucket of the widest tile count present, except the one-tile requests
 * when flags bit 0 is set (E4M3 KV) and they hold at least min_own_units
 * (page, kv head) pairs, or every tile count when flags bit 1 is set.  One
 * head-grouped work list per bucket (as fa_plan_work_host_heads, with
 * max_ctas_by_tiles[t-1] CTAs at most for the kernel of t tiles),
 * concatenated widest bucket first: a later bucket's CTAs, segments and
 * merge units follow the earlier ones' (request ids and page positions are
 * the batch's); its partial slots start after the columns the earlier
 * buckets' slots take, in units of its own slot of 8t columns
 * (*slot_columns: the total).
 *  qo_indptr        [batch + 1] int32, host, 0 first, non-decreasing.
 *  max_ctas_by_tiles[4]: grid bound of the kernel of 1..4 tiles.
 *  Outputs as fa_plan_work_host, with capacities for the sum of the grids
 *  (C = sum over t of max_ctas_by_tiles[t-1] * 7 + 1), plus *n_buckets (0:
 *  the batch stays one launch of the widest kernel, nothing else written
 *  but zero counts), bucket_tiles[4] and bucket_first_cta[4] (0 / -1 past
 *  *n_buckets).
 * Errors: FA_ERR_INVALID_ARG (malformed input, a tile count above
 * widest_tiles, a bucket whose grid bound is 0). */
int fa_plan_work_host_buckets(const int32_t* indptr, const int32_t* last_page_len,
                              const int32_t* qo_indptr, int batch, int group,
                              int num_kv_heads, int page_size, int widest_tiles,
                              const int* max_ctas_by_tiles, int flags,
                              int64_t min_own_units, int32_t* cta_offsets,
                              int32_t* segments, int32_t* merge, int* n_ctas,
                              int* n_segments, int* n_merge, int* n_buckets,
                              int* bucket_tiles, int* bucket_first_cta,
                              int64_t* slot_columns);

/* The plan fa_decode_plan makes by default, on the host: the grid in
 * groups of num_kv_heads CTAs, group g taking the g-th equal share of the
 * batch's page stream (request by request, a fixed cost of 2 pages before
 * each non-empty request) for every kv head, CTA g * num_kv_heads + h the
 * head-h part, so that a group's CTAs read the same pages' kv-head rows side
 * by side.  A request a group boundary falls inside is split there for
 * every head, and its pieces are merged as in fa_plan_work_host's plans.
 * fa_plan_work_host gives the other plan, the stream of (request, kv head)
 * units cut into equal quotas, which fa_decode_plan uses with a run-time
 * pool or with FADECODE_PLAN=stream in the environment, and whenever the
 * grid has fewer CTAs than kv heads.  Arguments, capacities and errors as
 * fa_plan_work_host (no pool). */
int fa_plan_work_host_heads(const int32_t* indptr, const int32_t* last_page_len, int batch,
                            int num_kv_heads, int page_size, int max_ctas,
                            int min_pages_per_cta, int32_t* cta_offsets, int32_t* segments,
                            int32_t* merge, int* n_ctas, int* n_segments, int* n_merge,
                            int* n_slots);

/* Wait for cuda_stream, then read and clear the plan's device-check word.
 * Returns FA_OK, FA_ERR_DEVICE_CHECK with *flags set (bit 0: page id outside
 * [0, num_pages); bit 1: a pipeline wait timed out), or FA_ERR_CUDA.
 * This is the one call that synchronises; keep it off the hot path. */
int fa_decode_check(fa_decode_plan_t plan, void* cuda_stream, int* flags);

/* Optional timing hook: when both events are non-NULL, later fa_decode_run
 * calls record ev_before on the stream just before the split-KV decode kernel
 * and ev_after just after it (both launches of a ragged plan in two buckets
 * lie between them; events are cudaEvent_t passed as void*, created by the
 * caller).  Pass NULLs to turn the hook off. */
int fa_decode_set_timing_events(fa_decode_plan_t plan, void* ev_before,
                                void* ev_after);

/* Decode one batch without allocating anything.
 *
 * The pages describe no counterpart to this call; it exists for callers that
 * cannot allocate: code handed only input and output pointers by a host
 * framework that owns every device buffer through its own pool, allocator or
 * out-of-memory callbacks, and latency-critical loops where cudaMalloc (which
 * may synchronise the whole device) or a page-locked host allocation is not
 * acceptable.  It does what fa_decode_plan followed by fa_decode_run does,
 * with the workspace replaced by a fixed array of FA_STATIC_SCRATCH_BYTES
 * that the library keeps on every GPU that loads it, for the life of the
 * process, and gives bitwise the same o and lse (same kernels, same grid,
 * same work list).
 *
 * Arguments are those of fa_decode_plan (page table, shapes, dtypes) and of
 * fa_decode_run (q, paged_kv, num_pages, scales, o, lse, stream), with the
 * same layouts and ownership; indices_dev must stay valid until the work
 * enqueued on cuda_stream has finished.  No plan handle is returned: every
 * call plans again on the host, into fixed host arrays (no run-time pool).
 *
 *  - Nothing is allocated on any call: no device memory, no page-locked host
 *    memory, no events, no heap objects.  The work list goes to the GPU with
 *    one cudaMemcpyAsync from a library-owned pageable host buffer, which
 *    the driver stages before the call returns (the call may wait for that
 *    staging, never for the stream's other work).
 *  - The first call on a device looks up the array's device address with
 *    that device current (cudaGetSymbolAddress) and caches the kernels'
 *    occupancy; make that first call outside any stream capture.
 *  - It must not be called while cuda_stream is being captured into a CUDA
 *    graph: a capture cannot record a copy from pageable memory.  Such a
 *    call returns FA_ERR_UNSUPPORTED and enqueues nothing.
 *  - Every call on a device shares the one array: calls whose GPU work
 *    overlaps (different streams, or host threads without ordering) race on
 *    it and give wrong results.  Calls in one stream are ordered and safe.
 *    The host side of calls is serialised by a lock.
 *  - The work list, including the device-check word, is rewritten by each
 *    call, so nothing left by an earlier call is read.  To see whether a
 *    call hit a bad page id or a timed-out wait, call fa_decode_static_check
 *    after it and before the next call.
 *  - A batch whose plan needs more than FA_STATIC_SCRATCH_BYTES (about
 *    (batch * num_kv_heads + CTAs) * 32 bytes of work list plus up to
 *    2 * CTAs * (num_qo_heads / num_kv_heads) * (head_dim + 1) * 4 bytes of
 *    partial states) is refused with FA_ERR_WORKSPACE_TOO_SMALL before
 *    anything is enqueued; use fa_decode_plan with a larger workspace then.
 * Errors: those of fa_decode_plan and fa_decode_run, and FA_ERR_UNSUPPORTED
 * during a stream capture. */
#define FA_STATIC_SCRATCH_BYTES (16u * 1024u * 1024u)
int fa_decode_static(const int32_t* indptr_host, const int32_t* indices_dev,
                     const int32_t* last_page_len_host, int batch,
                     int num_qo_heads, int num_kv_heads, int head_dim,
                     int page_size, fa_dtype q_dtype, fa_dtype kv_dtype,
                     const void* q, const void* paged_kv, int64_t num_pages,
                     float sm_scale, float k_scale, float v_scale, void* o,
                     float* lse, void* cuda_stream);

/* The device-check word of the last fa_decode_static call on the current
 * device: waits for cuda_stream, reads the word from the library's array and
 * clears it.  Returns FA_OK, FA_ERR_DEVICE_CHECK with *flags set (bit 0: a
 * page id outside [0, num_pages); bit 1: a pipeline wait timed out), or
 * FA_ERR_CUDA.  Allocates nothing.  Like fa_decode_check, it synchronises:
 * keep it off the hot path. */
int fa_decode_static_check(void* cuda_stream, int* flags);

/* Counters of the library's own host-side resources since it was loaded:
 * page-locked staging buffers allocated for plan uploads (count and bytes)
 * and uploads made through them.  fa_decode_plan may allocate a staging
 * buffer on its first calls or when a work list outgrows one;
 * fa_decode_static never touches them. */
typedef struct {
  int64_t pinned_host_allocations;
  int64_t pinned_host_bytes;
  int64_t staged_uploads;
} fa_library_stats;
int fa_library_get_stats(fa_library_stats* stats);

/* ---- cascade decode (shared prefix) ------------------------------------
 *
 * A batch whose requests all begin with the same shared prefix (whole pages,
 * e.g. a system prompt or a retrieved document) followed by pages of their
 * own.  Page "GitHub Spotlight: FlashInfer" (sections "Core Superpowers" and
 * "Scenario A") describes cascade attention: the shared prefix is attended
 * once for all requests and combined with each request's own part; the
 * combination is the merge rule of page "FlashDecoding + FlashInfer",
 * section "FlashDecoding - the split-KV trick".  The result equals
 * fa_decode_run over each request's full page list (prefix pages, then its
 * own), but the prefix is read from HBM once per kv head (per two blocks of
 * 128 query rows) instead of once per request: the prefix pass is a dense
 * contraction on the tcgen05 tensor cores (FADECODE_CASCADE=mma at plan time
 * selects the earlier warp-level mma.sync kernel). */
typedef struct fa_cascade_plan_s* fa_cascade_plan_t;

/* Upper bound of the workspace fa_cascade_plan needs (current device). */
size_t fa_cascade_workspace_size(int batch, int num_qo_heads, int num_kv_heads,
                                 int head_dim);

/*  prefix_indices_dev  [num_prefix_pages] int32, device: the shared pages, in
 *                      order, all full (num_prefix_pages * page_size tokens).
 *  indptr_host, indices_dev, last_page_len_host: each request's own pages
 *                      after the prefix, as in fa_decode_plan (a request may
 *                      have none).
 * Both index arrays are kept by pointer for the plan's lifetime.  Supported:
 * page_size 16 and (q, kv, head_dim) in (BF16, BF16, 64 or 128),
 * (F16, F16, 64 or 128), (BF16, E4M3, 128), (F16, E4M3, 128); otherwise
 * FA_ERR_UNSUPPORTED.  The prefix pass runs on the tcgen05 tensor cores for
 * 16-bit KV at head_dim 128, on warp-level MMAs otherwise (an E4M3 cache is
 * widened to f16 in registers).  Errors as fa_decode_plan. */
int fa_cascade_plan(const int32_t* prefix_indices_dev, int num_prefix_pages,
                    const int32_t* indptr_host, const int32_t* indices_dev,
                    const int32_t* last_page_len_host, int batch,
                    int num_qo_heads, int num_kv_heads, int head_dim,
                    int page_size, fa_dtype q_dtype, fa_dtype kv_dtype,
                    void* workspace_dev, size_t workspace_bytes,
                    void* cuda_stream, fa_cascade_plan_t* out_plan);

/* q [batch, num_qo_heads, head_dim], o likewise, lse [batch, num_qo_heads]
 * (may be NULL); paged_kv and num_pages as fa_decode_run.  Enqueues the
 * suffix decode, the prefix kernel and the combine kernel on cuda_stream;
 * the prefix kernel goes on a stream of the library's (one per device,
 * shared by all plans), forked from cuda_stream before the suffix decode
 * and joined before the combine, so that it runs alongside the decode (FADECODE_CASCADE_OVERLAP=0 at plan
 * time, or timing events set, keep all three in order on cuda_stream).  The
 * call is capturable into a CUDA graph either way. */
int fa_cascade_run(fa_cascade_plan_t plan, const void* q, const void* paged_kv,
                   int64_t num_pages, float sm_scale, void* o, float* lse,
                   void* cuda_stream);

/* fa_cascade_run over an E4M3 cache with its per-tensor scales (value =
 * code x scale, as fa_decode_run): k_scale folds into the logit scale of
 * both passes, v_scale into their outputs.  A 16-bit cache takes 1 and 1
 * only (FA_ERR_INVALID_ARG otherwise). */
int fa_cascade_run_scaled(fa_cascade_plan_t plan, const void* q, const void* paged_kv,
                          int64_t num_pages, float sm_scale, float k_scale,
                          float v_scale, void* o, float* lse, void* cuda_stream);

int fa_cascade_plan_destroy(fa_cascade_plan_t plan);

/* As fa_decode_check, for both passes of a cascade plan. */
int fa_cascade_check(fa_cascade_plan_t plan, void* cuda_stream, int* flags);

/* As fa_decode_set_timing_events, around the prefix kernel of later
 * fa_cascade_run calls (the events are recorded on their stream, and those
 * calls run the prefix kernel alone, after the suffix decode). */
int fa_cascade_set_timing_events(fa_cascade_plan_t plan, void* ev_before,
                                 void* ev_after);

#ifdef __cplusplus
}
#endif

#endif /* FA_DECODE_H_ */
