/*
 * pkv.h -- C ABI of the paged KV-cache attention library for GB300 (sm_103a).
 *
 * The operations follow the problem statement of the pages this library is
 * built from:
 *  - "mini-infer系统实战-06 True PagedAttention" (smarter.xin), sections 1
 *    and 3: one call writes the new token's K/V in place into the page slot
 *    that block_table and cache_seqlens select, then attends directly over
 *    the physical pages (no dense gather) and returns the output.  Cache
 *    tensors are [num_blocks, block_size, num_kv_heads, head_dim];
 *    block_table is int32 [batch, max_blocks]; cache_seqlens is int32
 *    [batch], the current length of every request.
 *  - "flex_attention + paged KV + CUDA graphs vs vLLM", "Why this works" and
 *    "What broke correctness": physical page 0 is a reserved null page and
 *    padded rows must yield finite output; decode runs under CUDA-graph
 *    capture, so no call syncs the host or allocates.
 *  - "[flashinfer] H100 D256 paged attention cuDNN auto-dispatch", code
 *    analysis part 1: ragged causal prefill over HND pages
 *    [num_pages, num_kv_heads, page_size, head_dim], end aligned (query i of
 *    q queries over kv keys sees kv - q + i + 1 keys), with host-resident
 *    lengths never read back from the device.
 *
 * Conventions shared by every entry point:
 *  - All tensors are dense, row major, in the shapes stated; "bf16" is the
 *    bfloat16 bit layout.  Device pointers must be 16-byte aligned.
 *  - The caller owns every buffer.  The library never allocates or frees
 *    device memory and never synchronises the host inside a device call, so
 *    every device call can be captured in a CUDA graph.  `stream` is a
 *    cudaStream_t (NULL = the legacy default stream).
 *  - GQA: query head h reads kv head h / (num_q_heads / num_kv_heads).
 *  - cache_seqlens[b] is the length BEFORE the append.  A negative value
 *    marks an inactive (padding) row: nothing is appended, its output is 0
 *    and its lse is -inf, and no error is raised.
 *  - Argument errors (shapes, alignment, unsupported sizes, too small a
 *    workspace) are returned synchronously as a pkv_status and nothing is
 *    launched.
 *  - Data errors are found on the device: a block_table entry a row needs
 *    that is outside [1, num_pages), or a row whose tokens do not fit in
 *    max_blocks * page_size.  The row's appends are dropped, its output is
 *    0 with lse -inf, and the matching PKV_ERR_* bit is OR-ed into
 *    *err_flag (when err_flag is not NULL).  No address outside the buffers
 *    is ever formed.  The host reads err_flag whenever it chooses.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PKV_NHD = 0, /* [num_pages, page_size, num_kv_heads, head_dim] */
    PKV_HND = 1  /* [num_pages, num_kv_heads, page_size, head_dim] */
} pkv_layout;

typedef enum {
    PKV_OK = 0,
    PKV_EINVAL = 1,       /* bad argument (NULL, shape, alignment, range) */
    PKV_EUNSUPPORTED = 2, /* valid but not built (head_dim, page size, group) */
    PKV_ECUDA = 3,        /* a CUDA runtime / driver call failed */
    PKV_ENOPAGES = 4,     /* page pool exhausted; nothing was taken */
    PKV_EWORKSPACE = 5,   /* workspace NULL or smaller than required */
    PKV_ETOOBIG = 6       /* problem needs more than the built-in scratch of
                             pkv_decode_attn_noalloc */
} pkv_status;

/* Device-side error bits OR-ed into *err_flag. */
#define PKV_ERR_PAGE 1     /* a needed block_table entry is outside [1, num_pages) */
#define PKV_ERR_OVERFLOW 2 /* a row's tokens exceed max_blocks * page_size */
#define PKV_ERR_TIMEOUT 4  /* an on-chip pipeline wait ran out of time: the call's outputs are
                              unspecified and its workspace must be zero-filled again */
#define PKV_ERR_QLEN 8     /* prefill / mixed step: a request with more queries than keys (or
                              than max_qlen), a query range outside [0, total_q), or a
                              decreasing qo_indptr */
#define PKV_ERR_PLAN 16    /* decode with PKV_DECODE_USE_PLAN: the workspace held no plan for
                              this call's sizes (the call planned for itself; outputs are
                              valid), or the plan's lengths differ from cache_seqlens (a stale
                              plan: outputs and appends are unspecified) */

/* Geometry of one K or V page pool (both share it).  page_size is a power of
 * two in [1, 256]; head_dim is 64, 128 or 256; num_pages >= 2 (page 0 is the
 * null page and is never read or written for a live token). */
typedef struct {
    int32_t num_pages;
    int32_t page_size;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t layout; /* pkv_layout */
} pkv_cache_desc;

/* Opaque host-side page pool (see pkv_pool_create). */
typedef struct pkv_pool pkv_pool;

/*
 * pkv_append -- write new tokens' K/V into their page slots (bit copy).
 * Source: "mini-infer系统实战-06 True PagedAttention", section 1 (step 1 of
 * the fused call: k_new/v_new written in place into the right block slot).
 *
 *  k_cache, v_cache  device bf16 pools described by `desc` (modified).
 *  k_new, v_new      device bf16 [T, num_kv_heads, head_dim].
 *  num_tokens        T (must equal batch when append_indptr is NULL).
 *  append_indptr     device int32 [batch + 1] (row b appends tokens
 *                    append_indptr[b] .. append_indptr[b+1]-1 of k_new at
 *                    positions cache_seqlens[b], cache_seqlens[b]+1, ...),
 *                    or NULL for exactly one token per row (T = batch).  A
 *                    row whose range is reversed or leaves [0, T) appends
 *                    nothing (no error bit).
 *  block_table       device int32 [batch, max_blocks].
 *  cache_seqlens     device int32 [batch]; not modified (the caller advances
 *                    it).
 *  err_flag          device int32, or NULL.  Only the pages that receive a
 *                    token are checked; a failing row appends nothing.
 * Returns PKV_OK once the kernel is enqueued on `stream`.
 */
PKV_API pkv_status pkv_append(const pkv_cache_desc *desc, void *k_cache, void *v_cache, const void *k_new,
                      const void *v_new, int32_t num_tokens, const int32_t *append_indptr,
                      const int32_t *block_table, int32_t max_blocks, const int32_t *cache_seqlens,
                      int32_t batch, int32_t *err_flag, void *stream);

/*
 * pkv_decode_workspace_size -- bytes of device workspace pkv_decode_attn
 * needs for these sizes (0 on invalid arguments).  The workspace holds the
 * split-KV partial results, one combine ticket per (row, kv head) and room
 * for one step plan (see PKV_DECODE_MAKE_PLAN; the plan needs no zeroing).  It
 * must be zero-filled once before its first use (e.g. cudaMemsetAsync);
 * every completed call leaves the tickets at zero again, so it can be reused
 * by later calls with the same or smaller sizes.  After a call that raised
 * PKV_ERR_TIMEOUT, zero it again.  Calls that share a workspace must not run
 * concurrently.
 */
PKV_API size_t pkv_decode_workspace_size(int32_t batch, int32_t max_blocks, int32_t num_q_heads,
                                 const pkv_cache_desc *desc);

/*
 * pkv_decode_attn -- fused append + single-token GQA decode attention
 * straight over the paged cache, with split-KV partitioning planned on the
 * device and a log-sum-exp combine of the partial results.
 * Source: "mini-infer系统实战-06 True PagedAttention", sections 1, 3 and 6
 * (flash_attn_with_kvcache with block_table / cache_seqlens; the split-KV
 * decode kernel behind it); "flex_attention + paged KV + CUDA graphs vs
 * vLLM", "Best config" (q pre-scaled by the softmax scale).
 *
 *  q                 device bf16 [batch, num_q_heads, head_dim].
 *  k_new, v_new      device bf16 [batch, num_kv_heads, head_dim], or both
 *                    NULL (attend only).  When given, row b's token is
 *                    written at position cache_seqlens[b] and the row attends
 *                    cache_seqlens[b] + 1 keys; otherwise cache_seqlens[b].
 *  softmax_scale     scale applied to q.k (finite).
 *  out               device bf16 [batch, num_q_heads, head_dim]
 *                    (round to nearest even from fp32).
 *  lse               device fp32 [batch, num_q_heads] natural-log
 *                    log-sum-exp of the scaled scores, or NULL.
 *  workspace         device buffer of at least pkv_decode_workspace_size
 *                    bytes (see there).
 *  batch             0 .. 1024.
 * Rows that see no key (inactive, or attend-only with length 0) give out = 0
 * and lse = -inf.
 */
PKV_API pkv_status pkv_decode_attn(const pkv_cache_desc *desc, void *k_cache, void *v_cache, const void *q,
                           const void *k_new, const void *v_new, const int32_t *block_table,
                           int32_t max_blocks, const int32_t *cache_seqlens, int32_t batch,
                           int32_t num_q_heads, float softmax_scale, void *out, float *lse,
                           void *workspace, size_t workspace_bytes, int32_t *err_flag,
                           void *stream);

/* Flags of pkv_decode_attn_ex. */
#define PKV_DECODE_OVERLAP_PROLOGUE 1u
/* Launch with programmatic dependent launch: the kernel may start while the
 * preceding kernel in the stream is still finishing, and reads cache_seqlens
 * and block_table (only those) before that kernel has completed; every other
 * input is read, and every output written, only after it has completed.
 * Use it when the immediately preceding kernel does not write cache_seqlens
 * or block_table (for instance the layers of one decode step, which share
 * them).  Capturable in CUDA graphs. */

#define PKV_DECODE_EARLY_KV 2u
/* Only together with PKV_DECODE_OVERLAP_PROLOGUE: the kernel also streams the
 * cached K/V (the tokens below cache_seqlens) before the preceding kernel has
 * completed, so a layer's cache reads overlap the end of the previous kernel.
 * q, k_new, v_new and every output (out, lse, the appended token, err_flag)
 * still wait for it.  Use it when the immediately preceding kernel in the
 * stream does not write this call's cache pages -- for instance the
 * projection producing q / k_new / v_new, or the attention of another layer.
 * Capturable in CUDA graphs. */

#define PKV_DECODE_MAKE_PLAN 4u
/* Step plans.  The work split of a decode call (which CTA streams which
 * tokens of which row, and its first page ids) depends only on
 * cache_seqlens, block_table and the sizes, so every layer of one decode
 * step shares it.  With PKV_DECODE_MAKE_PLAN the call also writes its plan
 * into the workspace: a small plan kernel runs before the decode kernel
 * (an ordinary launch, so everything earlier in the stream has completed
 * when it reads cache_seqlens and block_table).  The decode kernel itself
 * plans as without the flag.  Source: "flex_attention + paged KV + CUDA
 * graphs vs vLLM", "Why this works" (the per-step metadata is built once
 * and every layer of the step replays against it). */

#define PKV_DECODE_USE_PLAN 8u
/* The call takes its plan from the workspace instead of deriving it, so its
 * CTAs reach their first K/V load one dependent memory round trip after they
 * start.  The workspace must hold the plan of an earlier PKV_DECODE_MAKE_PLAN
 * call on the same stream, made with the same desc, batch, max_blocks,
 * num_q_heads and (non-)NULL k_new, and with cache_seqlens and block_table
 * holding the same values then as now (the layers of one decode step).
 * Every decode kernel signals its dependents only after the kernel before
 * it has completed, so the plan kernel has completed before any later
 * launch starts.  A plan made for other sizes (or none) is not used: the
 * call plans for itself and sets PKV_ERR_PLAN.  A plan whose lengths differ
 * from cache_seqlens sets PKV_ERR_PLAN too; then the outputs and appended
 * tokens are unspecified (every address stays inside the pools and the
 * workspace).  Not together with PKV_DECODE_MAKE_PLAN. */

/*
 * pkv_decode_attn_ex -- pkv_decode_attn with launch flags (PKV_DECODE_*).
 * flags = 0 behaves exactly like pkv_decode_attn.
 */
PKV_API pkv_status pkv_decode_attn_ex(const pkv_cache_desc *desc, void *k_cache, void *v_cache,
                                      const void *q, const void *k_new, const void *v_new,
                                      const int32_t *block_table, int32_t max_blocks,
                                      const int32_t *cache_seqlens, int32_t batch,
                                      int32_t num_q_heads, float softmax_scale, void *out,
                                      float *lse, void *workspace, size_t workspace_bytes,
                                      int32_t *err_flag, void *stream, uint32_t flags);

/*
 * pkv_decode_attn_noalloc -- pkv_decode_attn without a caller workspace.
 * The paper has no counterpart: this is a convenience of this library.
 *
 * For callers that cannot allocate device memory at all, such as code running
 * inside a host framework that owns every byte of device memory and forbids
 * its plug-ins to allocate, or a real-time serving loop that must not touch
 * the allocator after start-up.  It computes exactly what pkv_decode_attn
 * computes (same arguments minus the workspace, same outputs, same errors)
 * and allocates nothing: the split-KV scratch is a 16 MiB array compiled into
 * the library, which every GPU that loads the library holds until the process
 * exits.
 *  - Limit: problems whose pkv_decode_workspace_size is at most 16 MiB (for
 *    instance head_dim 128 with up to 4 query heads per kv head and up to
 *    1024 rows); larger ones return PKV_ETOOBIG and launch nothing.
 *  - The first call on each device looks up the array's device address (a
 *    one-time set-up); make that first call before any stream capture.
 *  - Every call on a device shares the one array and its contents persist
 *    between calls; each call clears what must start at zero (on its own
 *    stream) first.  Calls that can overlap on the GPU (different streams,
 *    or different host threads) race on it: serialise them.
 */
PKV_API pkv_status pkv_decode_attn_noalloc(const pkv_cache_desc *desc, void *k_cache, void *v_cache,
                                           const void *q, const void *k_new, const void *v_new,
                                           const int32_t *block_table, int32_t max_blocks,
                                           const int32_t *cache_seqlens, int32_t batch,
                                           int32_t num_q_heads, float softmax_scale, void *out,
                                           float *lse, int32_t *err_flag, void *stream);

/* ---------------------------------------------------------------------
 * A whole decode step captured as a CUDA graph.
 * Source: "flex_attention + paged KV + CUDA graphs vs vLLM", "Why this works"
 * (one CUDA graph per batch bucket replays the step's launches; padding rows
 * take a reserved null slot so that one graph serves every batch up to the
 * bucket).  Here a padding row is inactive: cache_seqlens[b] < 0 (nothing is
 * read or appended for it, its output is 0).
 * --------------------------------------------------------------------- */

/* Opaque captured decode step. */
typedef struct pkv_decode_step pkv_decode_step;

/* The bucket (graph batch size) serving `batch` rows: the smallest power of
 * two that is >= max(batch, 8); 0 if batch is outside [1, 1024]. */
PKV_API int32_t pkv_decode_bucket(int32_t batch);

/*
 * pkv_decode_step_create -- captures the pkv_decode_attn_ex calls of one
 * decode step, layer l = 0 .. num_layers-1 in order, into a CUDA graph.  The
 * layers share desc, block_table, cache_seqlens, batch (the bucket),
 * num_q_heads, softmax_scale, workspace, err_flag and flags; each has its own
 * k_caches[l], v_caches[l], q[l], k_new[l] / v_new[l] (both arrays NULL for
 * attend-only), out[l] and lse[l] (lse NULL, or an array whose entries may be
 * NULL).  All pointer arrays are host arrays of device pointers.
 *  - The pointers are baked into the graph: every launch reads what the
 *    buffers hold at launch time (write the step's q / k_new / v_new and
 *    cache_seqlens there, then launch).
 *  - Every argument error of the layer calls is returned before any CUDA
 *    work; nothing is launched by this call.
 *  - With PKV_DECODE_OVERLAP_PROLOGUE (and PKV_DECODE_EARLY_KV) the layers
 *    overlap inside the graph as described for pkv_decode_attn_ex.
 *  - With PKV_DECODE_USE_PLAN the first layer is captured with
 *    PKV_DECODE_MAKE_PLAN instead and every later layer reuses its plan.
 * On success *step_out owns the graph; free it with pkv_decode_step_destroy.
 */
PKV_API pkv_status pkv_decode_step_create(const pkv_cache_desc *desc, int32_t num_layers, void *const *k_caches,
                                          void *const *v_caches, const void *const *q, const void *const *k_new,
                                          const void *const *v_new, const int32_t *block_table,
                                          int32_t max_blocks, const int32_t *cache_seqlens, int32_t batch,
                                          int32_t num_q_heads, float softmax_scale, void *const *out,
                                          float *const *lse, void *workspace, size_t workspace_bytes,
                                          int32_t *err_flag, uint32_t flags, pkv_decode_step **step_out);

/* Launches the captured step on `stream` (cudaStream_t). */
PKV_API pkv_status pkv_decode_step_launch(pkv_decode_step *step, void *stream);

/* Frees a captured step (NULL is allowed). */
PKV_API void pkv_decode_step_destroy(pkv_decode_step *step);

/*
 * pkv_prefill_workspace_size -- bytes of device workspace pkv_prefill_attn
 * needs (0 on invalid or unsupported arguments).  The workspace holds the
 * call's work plan; it needs no initialisation and is fully rewritten by every
 * call.  Calls that share a workspace must not run concurrently.
 */
PKV_API size_t pkv_prefill_workspace_size(int32_t batch, int32_t total_q, int32_t num_q_heads,
                                          const pkv_cache_desc *desc);

/*
 * pkv_prefill_attn -- ragged end-aligned causal prefill attention straight
 * over the paged cache (no append: fill the cache first, e.g. with
 * pkv_append and an append_indptr).
 * Source: "[flashinfer] H100 D256 paged attention cuDNN auto-dispatch", code
 * analysis part 1 (ragged batch over HND pages; request b with q_b queries
 * over kv_b keys, q_b <= kv_b; its query i sees keys 0 .. kv_b - q_b + i).
 *
 *  k_cache, v_cache  device bf16 pools described by `desc` (read only);
 *                    page_size must be at least 8.
 *  q                 device bf16 [total_q, num_q_heads, head_dim]; request
 *                    b owns rows qo_indptr[b] .. qo_indptr[b+1]-1.
 *  qo_indptr         device int32 [batch + 1], non-decreasing, with
 *                    qo_indptr[b+1] <= total_q.
 *  kv_lens           device int32 [batch]: keys of request b (its cache
 *                    length, the queries' own tokens included).
 *  block_table       device int32 [batch, max_blocks].
 *  num_q_heads       a power-of-two multiple (at most 128) of num_kv_heads.
 *  softmax_scale     scale applied to q.k (finite).
 *  out               device bf16 [total_q, num_q_heads, head_dim] (round to
 *                    nearest even from fp32); rows no request owns are not
 *                    written.
 *  lse               device fp32 [total_q, num_q_heads], natural log, or NULL.
 *  workspace         device buffer of pkv_prefill_workspace_size bytes.
 *  batch             0 .. 1024.
 * A request with q_b = 0 does nothing.  A request whose query range or
 * length is malformed (PKV_ERR_QLEN), whose keys exceed max_blocks *
 * page_size (PKV_ERR_OVERFLOW) or whose block_table holds a page outside
 * [1, num_pages) among its first ceil(kv_b / page_size) entries
 * (PKV_ERR_PAGE) gets out = 0 and lse = -inf on its query rows (those inside
 * [0, total_q)) and sets the bit in *err_flag.
 * Launches two kernels on `stream`: a one-CTA plan (an ordinary launch) and
 * the attention kernel, a programmatic dependent of the plan that waits for
 * it before reading anything the plan or earlier work wrote.
 */
PKV_API pkv_status pkv_prefill_attn(const pkv_cache_desc *desc, const void *k_cache, const void *v_cache,
                                    const void *q, const int32_t *qo_indptr, const int32_t *kv_lens,
                                    const int32_t *block_table, int32_t max_blocks, int32_t batch,
                                    int32_t num_q_heads, int32_t total_q, float softmax_scale, void *out,
                                    float *lse, void *workspace, size_t workspace_bytes, int32_t *err_flag,
                                    void *stream);

/* ---------------------------------------------------------------------
 * One step of a mixed batch: chunked prefill, multi-token (speculative)
 * decode and single-token decode rows in one call.
 * Source: "flex_attention + paged KV + CUDA graphs vs vLLM", "What's left on
 * the table" (vLLM interleaves prefill chunks and decode tokens within one
 * step, where flex ran a separate prefill pass); the end-aligned causal rule
 * of "[flashinfer] H100 D256 paged attention cuDNN auto-dispatch", code
 * analysis part 1; the append of "mini-infer系统实战-06 True PagedAttention",
 * section 1.
 * --------------------------------------------------------------------- */

/*
 * pkv_mixed_workspace_size -- bytes of device workspace pkv_mixed_attn needs
 * for these sizes (0 on invalid or unsupported arguments).  Like the decode
 * workspace it must be zero-filled once before its first use; every
 * completed call leaves it ready for the next (zero it again after
 * PKV_ERR_TIMEOUT).  Calls that share a workspace must not run concurrently.
 */
PKV_API size_t pkv_mixed_workspace_size(int32_t batch, int32_t total_q, int32_t max_blocks, int32_t num_q_heads,
                                        int32_t max_qlen, int32_t decode_max_qlen, const pkv_cache_desc *desc);

/*
 * pkv_mixed_attn -- append every row's new tokens, then attend: row b brings
 * q_b = qo_indptr[b+1] - qo_indptr[b] tokens on top of L_b =
 * cache_seqlens[b] cached ones (L_b is the length BEFORE this call; the
 * caller advances it).
 *
 *  q                 device bf16 [total_q, num_q_heads, head_dim]; row b's
 *                    queries are rows qo_indptr[b] .. qo_indptr[b+1]-1.
 *  k_new, v_new      device bf16 [total_q, num_kv_heads, head_dim], or both
 *                    NULL.  When given, row b's tokens are written at
 *                    positions L_b .. L_b + q_b - 1 (as pkv_append: a row
 *                    whose written pages or length fail appends nothing) and
 *                    the row holds kv_b = L_b + q_b keys; otherwise the
 *                    caller appended already and kv_b = L_b.
 *  qo_indptr         device int32 [batch + 1].
 *  max_qlen          longest q_b accepted (>= 1): a longer row appends
 *                    nothing and gets PKV_ERR_QLEN with out = 0, lse = -inf.
 *  decode_max_qlen   rows with 1 <= q_b <= decode_max_qlen run on the
 *                    split-KV decode kernel (every K/V tile serves up to 16
 *                    (query, head) pairs of a kv head); longer rows on the
 *                    tensor-core prefill kernel, which needs page_size >= 8
 *                    (PKV_EUNSUPPORTED if max_qlen > decode_max_qlen with
 *                    smaller pages).  When max_qlen <= decode_max_qlen the
 *                    prefill kernel is not launched at all.
 *  out               device bf16 [total_q, num_q_heads, head_dim] (round to
 *                    nearest even); lse fp32 [total_q, num_q_heads] natural
 *                    log, or NULL.
 *  workspace         pkv_mixed_workspace_size bytes (see there).
 *  batch             0 .. 1024; total_q * num_q_heads < 2^31.
 * Query i of row b attends keys 0 .. kv_b - q_b + i of its kv head (end
 * aligned).  Row fates: q_b = 0 writes nothing; an inactive row (L_b < 0)
 * appends nothing and gets out = 0, lse = -inf, no error; a query range that
 * is reversed or leaves [0, total_q) sets PKV_ERR_QLEN and writes nothing for
 * the row (with a decreasing qo_indptr the rows' outputs are unspecified);
 * kv_b < q_b (attend only) gives PKV_ERR_QLEN; a row whose keys exceed
 * max_blocks * page_size (PKV_ERR_OVERFLOW) or whose first
 * ceil(kv_b / page_size) block_table entries hold a page outside
 * [1, num_pages) (PKV_ERR_PAGE) gets out = 0 and lse = -inf.
 * Launches up to four kernels on `stream` (the prefill plan when a row may
 * be longer than decode_max_qlen, the append, the decode kernel, the prefill
 * kernel), chained by programmatic dependent launch; the first one is an
 * ordinary launch, so everything earlier in the stream is complete before
 * any of them reads its inputs.  No host sync, no allocation, capturable in
 * a CUDA graph.
 */
PKV_API pkv_status pkv_mixed_attn(const pkv_cache_desc *desc, void *k_cache, void *v_cache, const void *q,
                                  const void *k_new, const void *v_new, const int32_t *qo_indptr,
                                  const int32_t *block_table, int32_t max_blocks, const int32_t *cache_seqlens,
                                  int32_t batch, int32_t num_q_heads, int32_t total_q, int32_t max_qlen,
                                  int32_t decode_max_qlen, float softmax_scale, void *out, float *lse,
                                  void *workspace, size_t workspace_bytes, int32_t *err_flag, void *stream);

/* ---------------------------------------------------------------------
 * Host page-pool and block-table helpers (no device memory involved).
 * Source: "flex_attention + paged KV + CUDA graphs vs vLLM", "What each
 * option did" (PageTable.reserve hands out pages sequentially on a fresh
 * batch) and "Why this works" (page 0 reserved as a no-op slot).
 * --------------------------------------------------------------------- */

/* A pool of pages 1 .. num_pages-1 (page 0 is never handed out), handed out
 * lowest-numbered first.  Returns NULL if num_pages < 2 or on allocation
 * failure.  Not thread safe. */
PKV_API pkv_pool *pkv_pool_create(int32_t num_pages);
PKV_API void pkv_pool_destroy(pkv_pool *pool);

/* Takes n free pages into pages_out[0..n-1].  PKV_ENOPAGES if fewer than n
 * are free (then nothing is taken). */
PKV_API pkv_status pkv_pool_alloc(pkv_pool *pool, int32_t n, int32_t *pages_out);

/* Returns n pages.  PKV_EINVAL if a page is 0, out of range or already free
 * (then nothing is returned). */
PKV_API pkv_status pkv_pool_free(pkv_pool *pool, const int32_t *pages, int32_t n);

PKV_API int32_t pkv_pool_num_free(const pkv_pool *pool);

/* Mixes the free list with a seeded permutation (splitmix64-driven
 * Fisher-Yates), so later allocations are scattered over the pool. */
PKV_API pkv_status pkv_pool_shuffle(pkv_pool *pool, uint64_t seed);

/* Makes a host block_table row cover new_len tokens when it covers cur_len:
 * fills entries [ceil(cur_len/P), ceil(new_len/P)) from the pool.
 * PKV_EINVAL if new_len < cur_len or the row would exceed max_blocks;
 * PKV_ENOPAGES if the pool is short (then the row is unchanged). */
PKV_API pkv_status pkv_table_reserve(pkv_pool *pool, int32_t *block_table_row, int32_t max_blocks,
                             int32_t page_size, int32_t cur_len, int32_t new_len);

/* Returns the pages of a row covering len tokens to the pool and zeroes the
 * row's entries. */
PKV_API pkv_status pkv_table_release(pkv_pool *pool, int32_t *block_table_row, int32_t max_blocks,
                             int32_t page_size, int32_t len);

/* Host-side check of block_table / cache_seqlens (host copies) for a decode
 * or append of extra_tokens per row: returns PKV_EINVAL with *bad_row set to
 * the first failing row, else PKV_OK.  For tests and debugging. */
PKV_API pkv_status pkv_validate_host(const pkv_cache_desc *desc, const int32_t *block_table_host,
                             int32_t max_blocks, const int32_t *seqlens_host, int32_t batch,
                             int32_t extra_tokens, int32_t *bad_row);

/* Bytes of one K or V pool for `desc` (num_pages * page_size * num_kv_heads
 * * head_dim * 2), 0 on invalid arguments. */
PKV_API uint64_t pkv_pool_bytes(const pkv_cache_desc *desc);

/* Static description of a status code. */
PKV_API const char *pkv_status_str(pkv_status status);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
