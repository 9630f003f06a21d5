/*
 * verify_attn.h -- C ABI of the GB300 (sm_103a) paged-KV GQA/MQA verify
 * attention library (libverify_attn.so).
 *
 * One step of speculative-decoding verification: each request b holds L_b
 * query tokens (a draft chain under a causal mask, or a draft tree under a
 * bit-packed ancestor mask; L_b = 1 is plain decode, and a request with no
 * cached prefix and a causal mask is ordinary varlen causal prefill).  They
 * attend to the request's cached keys / values -- the prefix plus the drafts
 * themselves, appended first -- reached through a paged KV cache, and the
 * library returns out = softmax(Q K^T * sm_scale * k_scale + M) V * v_scale
 * and the natural-log LSE of every (token, query head) row.
 *
 * Sources (by page and section):
 *  - flashmap 0.1.0, flashmap/sglang/verify_attention.py: the split-KV verify
 *    design (one program per request, KV head, row block and split holding
 *    all G query heads of the KV head; an LSE merge of the splits; k_scale on
 *    the logits and v_scale on the values; a host plan that reads only
 *    shapes so that the run is graph-capturable).
 *  - FlashInfer PR #286 "Separate Q and KV dtypes for decode": the paged
 *    table (indptr, indices, last_page_len, page_size), the plan / run split
 *    (begin_forward caches auxiliary data for many forward calls), the
 *    validation in BeginForward (int32 index arrays, num_qo_heads divisible
 *    by num_kv_heads), a caller-owned workspace, status-code errors, and a
 *    query dtype separate from the (possibly fp8) KV dtype.
 *  - FlashInfer issue #152 "How to implement a tree attention": custom tree
 *    masks; a triu -inf mask is the causal mask.
 *  - vLLM PR #1679 "cached multi-query attention towards speculative
 *    decoding": write every draft's K/V into the cache, then attend.
 *  - vLLM PR #2401 "Support MQA/GQA in prefill stage": GQA as MHA over K/V
 *    shared by G query heads (query head qh uses KV head qh / G).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  Status: every function returns VA_OK (0) or a negative VA_ERR_* code; no
 *  function throws, aborts or exits.  verify_attn_status_string() names a code.
 *
 *  Ownership: the caller owns every buffer, host and device, including the
 *  device workspace and the host plan buffer.  Nothing is allocated on the
 *  device by any entry point, and verify_attn_run / paged_kv_append read no
 *  device memory on the host, so both may be captured into a CUDA graph.
 *
 *  Streams: `stream` is a cudaStream_t passed as void* (NULL = the legacy
 *  default stream).  Device work is enqueued asynchronously on it.
 *
 *  Layouts (all contiguous, row-major):
 *   q, out         [total_qo, num_qo_heads, head_dim]   bf16
 *   lse            [total_qo, num_qo_heads]             fp32, natural log
 *   k_cache/v_cache[num_pages, num_kv_heads, page_size, head_dim]  ("HND", the
 *                  default) or [num_pages, page_size, num_kv_heads, head_dim]
 *                  ("NHD", plan option kv_layout); bf16 or fp8-e4m3 (the KV dtype)
 *   k_new / v_new  [total_new, num_kv_heads, head_dim]  KV dtype
 *   kv_indptr      [batch+1] int32: request b's pages are
 *                  kv_indices[kv_indptr[b] .. kv_indptr[b+1])
 *   kv_indices     [kv_indptr[batch]] int32 page ids in [0, num_pages)
 *   last_page_len  [batch] int32 in [1, page_size] (any value when the
 *                  request has no page); kv_len_b = (pages_b - 1) *
 *                  page_size + last_page_len_b, or 0 with no page
 *   qo_indptr      [batch+1] int32: request b's query tokens are rows
 *                  qo_indptr[b] .. qo_indptr[b+1] of q / out; L_b >= 0
 *   mask           bit-packed uint8, LSB first (element e is bit e & 7 of
 *                  byte e >> 3); request b's L_b x L_b row-major block starts
 *                  at BIT offset mask_indptr[b]; bit (t, u) = 1 means draft
 *                  token t may attend to draft token u.  NULL = causal
 *                  (u <= t).  Prefix keys are always visible.
 *   mask_indptr    [batch+1] int32 bit offsets, mask_indptr[b+1] -
 *                  mask_indptr[b] = L_b * L_b.  (The plan option
 *                  mask_layout = VA_MASK_FULL selects flashmap's full layout
 *                  instead: L_b rows of kv_len_b bits, prefix included.)
 *  The drafts are the LAST L_b positions of each request's kv range, so the
 *  prefix length is kv_len_b - L_b (kv_len_b >= L_b is required).
 *
 *  Supported: head_dim 64 or 128; page_size a power of two in [1, 256];
 *  num_qo_heads a multiple of num_kv_heads (any group G = num_qo_heads /
 *  num_kv_heads; a request's G * L_b rows are cut into row blocks); q / out
 *  bf16; KV bf16 or fp8-e4m3 (OCP "fn": no infinities).  Device pointers
 *  must be 16-byte aligned.
 *  RoPE (LLaMA rotate-half) at caller-given positions: new keys rotated by
 *  paged_kv_append_ex, queries by verify_attn_run_ex.
 *  Unsupported requests (other head dims, page sizes, dtypes; logit caps,
 *  sinks, sliding windows) return VA_ERR_UNSUPPORTED -- there is no
 *  fallback path.
 */
#ifndef VERIFY_ATTN_H
#define VERIFY_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define VA_OK 0
#define VA_ERR_INVALID_ARGUMENT (-1)   /* null pointer, bad size, inconsistent tables */
#define VA_ERR_UNSUPPORTED (-2)        /* a valid request this library does not serve */
#define VA_ERR_WORKSPACE_TOO_SMALL (-3)
#define VA_ERR_PLAN_MISMATCH (-4)      /* plan built for other shapes / dtypes */
#define VA_ERR_CUDA (-5)               /* a CUDA runtime call failed */
#define VA_ERR_DEVICE_CHECK (-6)       /* a kernel's bounds check fired (see device_status) */
#define VA_ERR_PLAN_BUFFER_TOO_SMALL (-7)
#define VA_ERR_STATIC_SCRATCH_TOO_SMALL (-8) /* plan needs more than VA_STATIC_SCRATCH_BYTES */

/* Element types (FlashInfer PR #286: the query dtype and the KV-cache dtype
 * are separate arguments of begin_forward; the cache may be fp8). */
typedef enum { VA_BF16 = 0, VA_FP8_E4M3 = 1, VA_F32 = 2 } va_dtype;
#define VA_DTYPE_BF16 VA_BF16
#define VA_DTYPE_FP8_E4M3 VA_FP8_E4M3

/* Device-side check bits reported by verify_attn_device_status(). */
#define VA_DEV_BAD_PAGE 1        /* a page id outside [0, num_pages): read as zeros / skipped */
#define VA_DEV_BAD_TABLE 2       /* device tables disagree with the plan: item skipped */
#define VA_DEV_BAD_APPEND 4      /* append position outside the request's pages: skipped */
#define VA_DEV_TIMEOUT 8         /* a bounded wait gave up */

/* KV-cache layouts (FlashInfer PR #286's kv_layout argument):
 *   HND  [num_pages, num_kv_heads, page_size, head_dim]  (the default)
 *   NHD  [num_pages, page_size, num_kv_heads, head_dim] */
typedef enum { VA_LAYOUT_HND = 0, VA_LAYOUT_NHD = 1 } va_kv_layout;

/* Custom-mask layouts.  QLEN: request b's L_b x L_b draft block (prefix keys
 * always visible).  FULL (flashmap's full custom mask): L_b rows of kv_len_b
 * bits, one per key of the request, prefix included, row t starting at bit
 * mask_indptr[b] + t * kv_len_b; mask_indptr[b+1] - mask_indptr[b] =
 * L_b * kv_len_b. */
#define VA_MASK_QLEN 0
#define VA_MASK_FULL 1

/* Optional planner knobs and call features (pass NULL for the defaults). */
typedef struct {
    int max_splits;      /* upper bound on kv splits per (request, KV head, row block);
                            0 = planner's choice, 1 = never split */
    int min_chunk;       /* smallest kv chunk (keys) a split may hold; 0 = default */
    int target_ctas;     /* CTAs the plan aims to fill; 0 = derived from the SM count */
    int kernel;          /* force a kernel variant (VA_KERNEL_*); 0 = automatic */
    int mask_layout;     /* VA_MASK_QLEN (default) or VA_MASK_FULL */
    int kv_layout;       /* va_kv_layout of k_cache / v_cache: VA_LAYOUT_HND (default) or NHD */
    int rope;            /* 1: rotate each query row by RoPE at its token's position
                            (verify_attn_run_ex's q_position) before Q K^T; the cache holds
                            keys already rotated at their own positions (paged_kv_append_ex
                            with positions) */
    int q_fp8;           /* 1 (fp8-e4m3 caches, tcgen05 variants): run the MMAs on e4m3
                            operands (kind::f8f6f4): each query row quantised to e4m3 with
                            its own scale amax|q| / 448, P rounded to e4m3, K / V as
                            stored -- twice the tensor rate of the default, which widens
                            K / V to f16, at coarser precision (3 mantissa bits on q and
                            P).  Against attention over the quantised query rows the LSE
                            keeps the fp32 error; each output element moves by at most
                            sum_j e_j |v_j| / sum_j p_j, p_j the key's probability over
                            the row maximum, e_j = 2^-4 p_j + min(p_j, 2^-9).  Requires
                            an fp8 cache and a tcgen05 variant (else
                            VA_ERR_UNSUPPORTED) */
    int draft_items;     /* tcgen05 variants: 1 = a split request's drafts (keys prefix ..
                            kv_len) form a work item of their own, -1 = never, 0 = the
                            planner's choice (on when the split units are few next to the
                            CTAs and the drafts fit one key tile).  verify_attn_append_run
                            with a plain copy append reads such an item's keys and values
                            from k_new / v_new instead of the pages, so it does not wait
                            for the append. */
    int head_dim_v;      /* elements of a value row (sglang's value head size: v_cache rows
                            and out rows), 64 or 128; 0 means head_dim.  A value width
                            other than head_dim is served by the warp-level variants
                            (VA_KERNEL_MMA_64 / _128; a tcgen05 kernel asked for returns
                            VA_ERR_UNSUPPORTED).  out is then [total_qo, num_qo_heads,
                            head_dim_v] and the calls take head_dim (the key's) as before. */
} va_plan_options_t;

#define VA_KERNEL_AUTO 0
#define VA_KERNEL_MMA_64 1      /* warp-level tensor cores, 64-row blocks, 4 warps */
#define VA_KERNEL_MMA_128 2     /* warp-level tensor cores, 128-row blocks, 8 warps */
#define VA_KERNEL_TC_128 3      /* tcgen05 tensor cores + TMA, 128-row blocks; needs head_dim
                                   128, page_size a multiple of 16, 128 % G == 0; with fp8 KV
                                   the MMAs run on f16, so |q| must stay below 65504 */
#define VA_KERNEL_TC_256 4      /* as VA_KERNEL_TC_128 with two 128-row Q tiles per CTA sharing
                                   every K/V tile (256-row blocks, one CTA per SM) */

/* Name of a status code (static string).  FlashInfer PR #286's BeginForward
 * turns a failed check into an error message; here every check returns a
 * code, and this names it. */
const char* verify_attn_status_string(int status);

/* Number of SMs of the current CUDA device (or an error). */
int verify_attn_num_sms(int* num_sms);

/*
 * Upper bounds, for a batch with at most `batch` requests and `total_qo`
 * query tokens, of the host plan buffer and the device workspace any
 * verify_attn_plan() call can need (e.g. to size buffers once before
 * graph capture).  num_sms <= 0 queries the current device.
 */
int verify_attn_plan_bounds(int batch, int64_t total_qo, int num_qo_heads, int num_kv_heads,
                            int head_dim, int num_sms, size_t* plan_bytes,
                            size_t* workspace_bytes);

/*
 * Device workspace that suffices for every plan of a batch of at most
 * `batch` requests with at most `max_qo_len` query tokens each (FlashInfer
 * PR #286: the caller allocates the workspace once and hands it to
 * begin_forward).  Equals verify_attn_plan_bounds' workspace bound for
 * total_qo = batch * max_qo_len.  num_sms <= 0 queries the current device.
 * Errors: VA_ERR_INVALID_ARGUMENT (negative sizes, heads that do not divide,
 * null `bytes`), VA_ERR_CUDA (device query).
 */
int verify_attn_workspace_size(int batch, int num_qo_heads, int num_kv_heads, int head_dim,
                               int max_qo_len, int num_sms, size_t* bytes);

/*
 * Host half of the plan (flashmap's split planner and FlashInfer's
 * begin_forward): from HOST copies of the index arrays, cut the work into
 * items (request b, KV head h, row block, kv chunk [lo, hi)) that fill the
 * GPU, and record it in the caller's host buffer `plan_h` (plan_bytes long).
 * Performs no CUDA call.  mask_indptr_h may be NULL when has_mask = 0.
 * num_sms <= 0 queries the current device (that query is the one CUDA call).
 * On success *workspace_bytes receives the device workspace this plan needs.
 * Errors: VA_ERR_INVALID_ARGUMENT (inconsistent tables, null pointers),
 * VA_ERR_UNSUPPORTED, VA_ERR_PLAN_BUFFER_TOO_SMALL (*workspace_bytes then
 * holds the plan bytes needed).
 */
int verify_attn_plan_host(const int32_t* kv_indptr_h, const int32_t* qo_indptr_h,
                          const int32_t* last_page_len_h, const int32_t* mask_indptr_h,
                          int batch, int num_qo_heads, int num_kv_heads, int head_dim,
                          int page_size, va_dtype q_dtype, va_dtype kv_dtype, int has_mask,
                          int num_sms,
                          const va_plan_options_t* options, void* plan_h, size_t plan_bytes,
                          size_t* workspace_bytes);

/*
 * FlashInfer PR #286's begin_forward: plan once from host copies of the
 * index arrays, then run many times.  verify_attn_plan_host() followed by an
 * asynchronous upload of the plan's work list into the device workspace on
 * `stream`.  The workspace must hold
 * at least the bytes verify_attn_plan_host reports (else
 * VA_ERR_WORKSPACE_TOO_SMALL).  It also clears the workspace's device status
 * word.  If plan_h is pinned host memory it must not change until the
 * upload has run on `stream`.  Pointers into the workspace stay valid until
 * the next plan into the same workspace.
 */
int verify_attn_plan(const int32_t* kv_indptr_h, const int32_t* qo_indptr_h,
                     const int32_t* last_page_len_h, const int32_t* mask_indptr_h, int batch,
                     int num_qo_heads, int num_kv_heads, int head_dim, int page_size,
                     va_dtype q_dtype, va_dtype kv_dtype, int has_mask, int num_sms,
                     const va_plan_options_t* options, void* plan_h, size_t plan_bytes,
                     void* workspace_d, size_t workspace_bytes, void* stream);

/*
 * Verify attention (flashmap's partial kernel followed by its LSE merge).
 * All array arguments are DEVICE pointers with the layouts above; the index
 * arrays must hold the same values the plan was built from (a kernel that
 * finds otherwise skips the item and raises VA_DEV_BAD_TABLE).  The
 * workspace must hold this plan's work list (the last plan uploaded into
 * it); an item of another plan that names a request, KV head or partial row
 * outside this plan is skipped and raises VA_DEV_BAD_TABLE, so a mismatched
 * workspace never makes a kernel read or write outside the call's arrays or
 * the workspace.  mask /
 * mask_indptr are NULL iff the plan was made with has_mask = 0.
 * sm_scale <= 0 selects head_dim^-1/2.  k_scale / v_scale multiply the
 * stored keys / values (1 for bf16 caches); both must be finite and > 0.
 * lse may be NULL.  num_pages bounds every page id (a page id outside the
 * pool is read as zeros and raises VA_DEV_BAD_PAGE).  plan_h is the host plan
 * buffer; it is read on the host during the call only.
 * Errors: VA_ERR_INVALID_ARGUMENT, VA_ERR_PLAN_MISMATCH,
 * VA_ERR_WORKSPACE_TOO_SMALL, VA_ERR_CUDA (launch failure).
 */
int verify_attn_run(const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* kv_indptr, const int32_t* kv_indices,
                    const int32_t* last_page_len, const int32_t* qo_indptr, const uint8_t* mask,
                    const int32_t* mask_indptr, int num_qo_heads, int num_kv_heads, int head_dim,
                    int page_size, float sm_scale, float k_scale, float v_scale, void* out,
                    float* lse, int num_pages, const void* plan_h, void* workspace_d,
                    size_t workspace_bytes, void* stream);

/* Per-call arguments of verify_attn_run_ex / verify_attn_partial_ex. */
typedef struct {
    const int32_t* q_position; /* device [total_qo]: with a plan made with rope = 1, the
                                  position of each query token (for a draft tree: prefix +
                                  the draft's depth, the position its key was appended at);
                                  must be NULL otherwise */
    float rope_theta;          /* RoPE base (> 0, finite) when q_position is given */
    float rope_scale;          /* linear position scaling (> 0, finite); 0 means 1 */
    int early_reads;           /* 1: the call's inputs -- q, the index tables, the mask,
                                  q_position, and for verify_attn_append_run k_new / v_new and
                                  the append positions -- are complete before the kernel
                                  preceding this call in the stream starts (host copies, or
                                  kernels launched before it), and that kernel writes none of
                                  them nor a prefix slot of the cache; the library's kernels may
                                  then read them, and the prefix slots, while it still runs
                                  (programmatic dependent launch).  Writes still wait for it.
                                  0: no kernel reads anything before its predecessor has
                                  completed (verify_attn_append_run's attention still overlaps
                                  its own append). */
    int reserved[3];           /* must be zero */
} va_run_options_t;

/*
 * verify_attn_run with per-call options (RoPE positions of the queries).
 * With a plan made for RoPE, each query row is rotated at q_position[token]
 * (LLaMA rotate-half, angle position / rope_scale * rope_theta^(-2i /
 * head_dim); FlashInfer PR #286's ROPE_LLAMA at the tree positions of
 * FlashInfer issue #152) in fp32 and rounded to the MMA operand type (bf16,
 * or f16 with an fp8 cache) before Q K^T.  NULL options = verify_attn_run.
 * Errors: as verify_attn_run; VA_ERR_PLAN_MISMATCH when q_position is given
 * without a RoPE plan or missing with one.
 */
int verify_attn_run_ex(const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* kv_indptr, const int32_t* kv_indices,
                       const int32_t* last_page_len, const int32_t* qo_indptr,
                       const uint8_t* mask, const int32_t* mask_indptr, int num_qo_heads,
                       int num_kv_heads, int head_dim, int page_size, float sm_scale,
                       float k_scale, float v_scale, void* out, float* lse, int num_pages,
                       const void* plan_h, void* workspace_d, size_t workspace_bytes,
                       const va_run_options_t* options, void* stream);
int verify_attn_partial_ex(const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* kv_indptr, const int32_t* kv_indices,
                           const int32_t* last_page_len, const int32_t* qo_indptr,
                           const uint8_t* mask, const int32_t* mask_indptr, int num_qo_heads,
                           int num_kv_heads, int head_dim, int page_size, float sm_scale,
                           float k_scale, float v_scale, void* out, float* lse, int num_pages,
                           const void* plan_h, void* workspace_d, size_t workspace_bytes,
                           const va_run_options_t* options, void* stream);

/*
 * The two halves of verify_attn_run, for callers that time or schedule them
 * apart: the split attention kernel (it writes the final out / lse of every
 * unsplit item and the fp32 partials of split items into the workspace), and
 * the LSE merge of those partials (a no-op when the plan has no split).
 * verify_attn_merge must follow verify_attn_partial of the same plan on the
 * same stream, with the same out / lse.
 */
int verify_attn_partial(const void* q, const void* k_cache, const void* v_cache,
                        const int32_t* kv_indptr, const int32_t* kv_indices,
                        const int32_t* last_page_len, const int32_t* qo_indptr,
                        const uint8_t* mask, const int32_t* mask_indptr, int num_qo_heads,
                        int num_kv_heads, int head_dim, int page_size, float sm_scale,
                        float k_scale, float v_scale, void* out, float* lse, int num_pages,
                        const void* plan_h, void* workspace_d, size_t workspace_bytes,
                        void* stream);
int verify_attn_merge(const int32_t* qo_indptr, int num_qo_heads, int num_kv_heads, int head_dim,
                      void* out, float* lse, const void* plan_h, void* workspace_d,
                      size_t workspace_bytes, void* stream);

/*
 * The device half of verify_attn_plan for a plan made by
 * verify_attn_plan_host: asynchronously copy its work list into the device
 * workspace on `stream` and clear the workspace's device status word, so a
 * caller can size the workspace from the plan it already has (plan once,
 * allocate exactly, upload).  Same contract for plan_h and the workspace as
 * verify_attn_plan.  Errors: VA_ERR_INVALID_ARGUMENT (no valid plan, a
 * misaligned workspace), VA_ERR_WORKSPACE_TOO_SMALL, VA_ERR_CUDA.
 */
int verify_attn_plan_upload(const void* plan_h, void* workspace_d, size_t workspace_bytes,
                            void* stream);

/* Number of kernel launches verify_attn_run makes for this plan (1 or 2; 0
 * when the batch has no query token). */
int verify_attn_plan_launches(const void* plan_h, int* launches);

/*
 * Read and clear the workspace's device status word (an OR of VA_DEV_* bits
 * raised by kernels since the last plan / read).  Synchronises `stream`.
 * Returns VA_ERR_DEVICE_CHECK when any bit was set, else VA_OK.
 */
int verify_attn_device_status(void* workspace_d, int* bits, void* stream);

/*
 * Paged append (vLLM PR #1679: cache every draft's K/V before attention):
 * for request b and new token i < n_b = append_indptr[b+1] - append_indptr[b]
 * (host-known total_new = append_indptr[batch]), position pos = kv_len_b -
 * n_b + i; copy k_new[append_indptr[b] + i, h, :] bit for bit to
 * k_cache[kv_indices[kv_indptr[b] + pos / page_size], h, pos % page_size, :],
 * and likewise v.  The page table must already cover the new tokens
 * (kv_len_b counts them).  k_new / v_new are in the cache dtype (a pure
 * copy).  Device pointers; status_d (nullable, device int) receives
 * VA_DEV_BAD_APPEND / VA_DEV_BAD_PAGE bits (OR-ed) for skipped tokens.
 * Errors: VA_ERR_INVALID_ARGUMENT, VA_ERR_UNSUPPORTED, VA_ERR_CUDA.
 */
int paged_kv_append(const void* k_new, const void* v_new, const int32_t* append_indptr,
                    const int32_t* kv_indptr, const int32_t* kv_indices,
                    const int32_t* last_page_len, void* k_cache, void* v_cache, int batch,
                    int num_kv_heads, int head_dim, int page_size, int num_pages,
                    va_dtype kv_dtype, int64_t total_new, int* status_d, void* stream);

/* Options of paged_kv_append_ex (all-zero = a plain bit copy into an HND
 * cache, as paged_kv_append). */
typedef struct {
    int quantize;            /* 1: k_new / v_new are bf16 and the cache is fp8-e4m3; each
                                element x is stored as e4m3(x / scale): the correctly rounded
                                binary32 quotient, rounded to nearest even, finite overflow
                                saturated to +-448 (FlashInfer PR #286's fp8 cache with a
                                per-tensor scale: dequantised value = stored * scale) */
    float k_scale, v_scale;  /* the per-tensor scales of the quantising append (> 0, finite) */
    va_kv_layout kv_layout;
    const int32_t* positions; /* device [total_new], or NULL: rotate each new K row by RoPE at
                                this position before storing it (LLaMA's rotate-half pairing
                                of elements i and i + head_dim/2 at angle position /
                                rope_scale * rope_theta^(-2i / head_dim); FlashInfer PR #286's
                                ROPE_LLAMA, applied at the draft's own -- tree -- position as
                                FlashInfer issue #152 asks).  V rows are not rotated. */
    float rope_theta;        /* RoPE base (> 0, finite; e.g. 1e4, Llama-3: 5e5) */
    float rope_scale;        /* linear position scaling (> 0, finite); 0 means 1 */
    int head_dim_v;          /* elements of a V row (v_new and v_cache), sglang's value head
                                size, which may differ from head_dim (64 or 128); 0 means
                                head_dim */
    int reserved[3];         /* must be zero */
} va_append_options_t;

/*
 * paged_kv_append with options: a quantising append into an fp8 cache, RoPE
 * at given positions for the new keys, and the NHD layout.  The page walk,
 * the checks and the status bits are those of paged_kv_append; k_new / v_new
 * are bf16 when options->quantize, else in the cache dtype.  Rotated or
 * quantised rows are computed in fp32 and rounded once to the cache dtype
 * (round to nearest even; e4m3 saturating).  NULL options = paged_kv_append.
 * Errors: VA_ERR_INVALID_ARGUMENT (bad scales, theta, layout, non-zero
 * reserved fields, quantize without an fp8 cache), VA_ERR_UNSUPPORTED,
 * VA_ERR_CUDA.
 */
int paged_kv_append_ex(const void* k_new, const void* v_new, const int32_t* append_indptr,
                       const int32_t* kv_indptr, const int32_t* kv_indices,
                       const int32_t* last_page_len, void* k_cache, void* v_cache, int batch,
                       int num_kv_heads, int head_dim, int page_size, int num_pages,
                       va_dtype kv_dtype, int64_t total_new, const va_append_options_t* options,
                       int* status_d, void* stream);

/*
 * One verification step in one call (vLLM PR #1679: cache the drafts, then
 * attend): paged_kv_append_ex of the drafts' K/V -- k_new / v_new hold the
 * L_b new tokens of each request in qo_indptr order, placed at the request's
 * last L_b positions; append_options as for paged_kv_append_ex (NULL = a bit
 * copy into an HND cache; its kv_layout must be the plan's) -- followed by
 * verify_attn_run_ex over the cache it has just written.  Same arguments,
 * contract and errors as those two; the append's device check bits go to
 * the workspace's status word (verify_attn_device_status reads them).
 *
 * Ordering: the append waits for the kernel before it in the stream to
 * complete and then releases the attention kernels at once, so they read q,
 * the tables and the cache's prefix slots while the append still runs and
 * wait for it only before reading a draft's slot.  With run_options->
 * early_reads the append releases them at its start and reads its tables
 * before its own wait as well (see va_run_options_t for what the caller
 * then guarantees).  k_cache / v_cache are written, so they are not const.
 */
int verify_attn_append_run(const void* k_new, const void* v_new,
                           const va_append_options_t* append_options, const void* q, void* k_cache,
                           void* v_cache, const int32_t* kv_indptr, const int32_t* kv_indices,
                           const int32_t* last_page_len, const int32_t* qo_indptr,
                           const uint8_t* mask, const int32_t* mask_indptr, int num_qo_heads,
                           int num_kv_heads, int head_dim, int page_size, float sm_scale,
                           float k_scale, float v_scale, void* out, float* lse, int num_pages,
                           const void* plan_h, void* workspace_d, size_t workspace_bytes,
                           const va_run_options_t* run_options, void* stream);

/*
 * One verification step from HOST buffers, in one call: the plan / run split
 * of FlashInfer PR #286 (begin_forward plans from host copies of the index
 * arrays) and vLLM PR #1679's step (cache the drafts, then attend), with the
 * step's inputs and its result crossing between host and device inside the
 * call.
 *
 * staging_h (host, pinned for an asynchronous copy) holds the step's inputs,
 * each at its byte offset in `offsets`, with the layouts above: q, k_new,
 * v_new (one row per query token, qo_indptr order), kv_indptr, kv_indices,
 * last_page_len, qo_indptr, and mask / mask_indptr (offsets -1: no mask,
 * the causal case).  staging_d (device, staging_bytes long) receives all of
 * it in one host-to-device copy, and the kernels read the device copies at
 * the same offsets, so every offset must keep the device pointer 16-byte
 * aligned (multiples of 256 are simplest).  The plan is made on the host
 * from the tables in staging_h first (verify_attn_plan_host into plan_h);
 * then the inputs are copied and the plan's work list is uploaded into
 * workspace_d (verify_attn_plan_upload).  Then
 * verify_attn_append_run writes the drafts into k_cache / v_cache and
 * computes out_d / lse_d (lse_d may be NULL).  Last, out_d (total_qo x
 * num_qo_heads x value width, bf16) is copied into result_h at byte 0 and,
 * with lse_d, the LSE (fp32) at byte offset round_up(out bytes, 256): one
 * copy when lse_d sits at that offset from out_d, else two.  result_bytes
 * must hold what is copied.  With synchronize != 0 the call returns after
 * the stream has drained (result_h is then filled); otherwise result_h,
 * staging_h and plan_h must stay untouched until the stream's work is done.
 *
 * q_dtype is bf16; the KV dtype, plan options, append options and run
 * options are those of verify_attn_plan / verify_attn_append_run (the
 * options' device pointers -- positions, q_position -- stay device
 * pointers).  k_new / v_new are bf16 for a quantising append, else the KV
 * dtype.  The host tables are checked against staging_bytes before they are
 * read, and every array the tables size must lie inside it.
 * Errors: those of verify_attn_plan and verify_attn_append_run;
 * VA_ERR_INVALID_ARGUMENT for an offset or array outside staging_bytes or a
 * short result_bytes; VA_ERR_CUDA for a failed copy or synchronisation.
 * The step's own checks and the plan's come before anything is enqueued;
 * a check of verify_attn_append_run that fails leaves the input copy and
 * the plan upload enqueued (nothing else).
 */
typedef struct {
  int64_t q, k_new, v_new;                                /* byte offsets into the staging buffers */
  int64_t kv_indptr, kv_indices, last_page_len, qo_indptr;
  int64_t mask, mask_indptr;                              /* -1 with no mask */
} va_step_offsets_t;

int verify_attn_step_host(const void* staging_h, void* staging_d, size_t staging_bytes,
                          const va_step_offsets_t* offsets, int batch, int num_qo_heads,
                          int num_kv_heads, int head_dim, int page_size, va_dtype kv_dtype,
                          int num_sms, const va_plan_options_t* plan_options, void* plan_h,
                          size_t plan_bytes, void* workspace_d, size_t workspace_bytes,
                          const va_append_options_t* append_options, void* k_cache, void* v_cache,
                          int num_pages, float sm_scale, float k_scale, float v_scale, void* out_d,
                          float* lse_d, void* result_h, size_t result_bytes,
                          const va_run_options_t* run_options, int synchronize, void* stream);

/*
 * Greedy acceptance of draft trees: the step after verification, on the
 * target model's logits (FlashInfer issue #152: Medusa / EAGLE trees are
 * verified against the target model's outputs; its logits come from an LM
 * head outside this library).
 *
 * Request b's nodes are rows qo_indptr[b] .. qo_indptr[b+1] of `logits`
 * ([total_qo, vocab] rows, row_stride elements apart, bf16 or fp32, not
 * NaN).  Node 0 of a request is its root (the last accepted token,
 * parents = -1); every other node i has parents[i] in [0, i) (local
 * indices) and proposes draft_tokens[i].  The root is accepted; node i is
 * accepted iff its parent is accepted and the argmax of the parent's row --
 * the first index among equal maxima -- equals draft_tokens[i].  For each
 * request: accept_len[b] = the number of nodes on the root path of the
 * deepest accepted node (the smallest node index among equally deep ones),
 * that path's local node ids at accepted_nodes[qo_indptr[b] ..], and
 * bonus_token[b] = the argmax of its last node's row (the token the target
 * model emits next).  An empty request gives accept_len 0 and bonus -1; a
 * request whose parents break the rule gives the same and raises
 * VA_DEV_BAD_TABLE in status_d (nullable).  argmax_out (nullable) receives
 * every row's argmax.  Device pointers; the workspace (caller-owned, at
 * least verify_accept_workspace_size bytes, 16-byte aligned) holds per-row
 * scratch.  Errors: VA_ERR_INVALID_ARGUMENT, VA_ERR_UNSUPPORTED (logits
 * dtype), VA_ERR_WORKSPACE_TOO_SMALL, VA_ERR_CUDA.
 */
int verify_accept_workspace_size(int64_t total_qo, int vocab, int num_sms, size_t* bytes);
int verify_accept_greedy(const void* logits, va_dtype logits_dtype, int64_t total_qo, int vocab,
                         int64_t row_stride, const int32_t* qo_indptr, int batch,
                         const int32_t* draft_tokens, const int32_t* parents,
                         int32_t* accept_len, int32_t* accepted_nodes, int32_t* bonus_token,
                         int32_t* argmax_out, int* status_d, int num_sms, void* workspace_d,
                         size_t workspace_bytes, void* stream);

/*
 * verify_attn_run for callers that cannot allocate device memory.
 *
 * No page describes this entry point; it exists for callers that may not
 * call cudaMalloc (or any allocating routine) at all -- e.g. code running
 * inside a memory pool or graph-building framework that owns every device
 * allocation, or a plugin host that forbids allocation on its hot path -- and
 * so cannot hand verify_attn_run a workspace.  It computes exactly what
 * verify_attn_run computes (same kernels, same plan), but its scratch (the
 * work list, the fp32 split partials and the device status word) lives in one
 * file-scope __device__ array of VA_STATIC_SCRATCH_BYTES inside this library.
 *
 *  - Allocates nothing: no cudaMalloc / cudaFree and no allocating library
 *    call.  The caller still owns and passes every input and output; plan_h is
 *    a plan from verify_attn_plan_host (the workspace arguments of
 *    verify_attn_plan are not needed).
 *  - Limit: a plan whose workspace exceeds VA_STATIC_SCRATCH_BYTES is refused
 *    with VA_ERR_STATIC_SCRATCH_TOO_SMALL before anything is enqueued.
 *  - Memory: every GPU that loads the library holds the array until the
 *    process exits.
 *  - Set-up: the first call in each CUDA context (normally: on each device,
 *    with that device current) looks up the array's device address with
 *    cudaGetSymbolAddress and keeps it for that context.  A context created
 *    later (after cudaDeviceReset, or a driver context the caller makes
 *    current) gets its own look-up.
 *  - Every call copies the plan's work list from plan_h into the array and
 *    clears its status word on `stream` with asynchronous copies (so plan_h,
 *    if pinned, must stay unchanged until the copy has run), then launches the
 *    kernels.  All calls share the one array, which keeps the last call's
 *    contents: calls that can overlap on the GPU (different streams, or
 *    devices sharing the array's context) race and must be serialised by the
 *    caller.  Device-side check bits stay in the array's status word until
 *    the next call clears it: verify_attn_static_scratch_status reads them.
 * Errors: as verify_attn_run, plus VA_ERR_STATIC_SCRATCH_TOO_SMALL, and
 * VA_ERR_CUDA if the address look-up or an enqueue fails.
 */
#define VA_STATIC_SCRATCH_BYTES ((size_t)32 << 20)
/*
 * The device-side check bits (VA_DEV_*) of the last
 * verify_attn_run_static_scratch call in the current context, as
 * verify_attn_device_status reads a workspace's: copied out on `stream`
 * (which is synchronised) and cleared; allocates nothing.  Returns VA_OK with
 * *bits = 0, VA_ERR_DEVICE_CHECK with the bits set, VA_ERR_INVALID_ARGUMENT
 * (bits NULL) or VA_ERR_CUDA.
 */
int verify_attn_static_scratch_status(int* bits, void* stream);
int verify_attn_run_static_scratch(const void* q, const void* k_cache, const void* v_cache,
                                   const int32_t* kv_indptr, const int32_t* kv_indices,
                                   const int32_t* last_page_len, const int32_t* qo_indptr,
                                   const uint8_t* mask, const int32_t* mask_indptr,
                                   int num_qo_heads, int num_kv_heads, int head_dim,
                                   int page_size, float sm_scale, float k_scale, float v_scale,
                                   void* out, float* lse, int num_pages, const void* plan_h,
                                   void* stream);

#ifdef __cplusplus
}
#endif

#endif /* VERIFY_ATTN_H */
