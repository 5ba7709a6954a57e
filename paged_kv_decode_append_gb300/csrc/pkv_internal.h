// pkv_internal.h -- host-side plumbing shared by the C-ABI front end and the
// kernel launchers.  Not part of the public interface.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "pkv.h"

namespace pkv {

// Largest batch one decode call plans for (the per-CTA plan lives in shared
// memory: two int32 per row).
constexpr int kMaxDecodeBatch = 1024;
// Tokens per pipeline tile of the decode kernel.
constexpr int kDecodeTile = 32;
// Smallest split-KV chunk, in tokens.
constexpr int kDecodeChunkMin = 64;
// A chunk never spans more than this many pages (its page ids are staged in
// shared memory).
constexpr int kDecodeChunkMaxPages = 256;

// Static split of the decode problem: which heads one CTA owns and how the
// workspace is carved.  Computed identically by the workspace-size query and
// by the launch.
struct DecodeShape {
    int group;          // num_q_heads / num_kv_heads
    int heads_per_cta;  // q heads of one kv head handled by one CTA
    int n_sub;          // group / heads_per_cta
    int units_per_row;  // num_kv_heads * n_sub
    int chunk_max;      // largest chunk in tokens (multiple of kDecodeTile)
    int64_t cap_items;  // partial-result slots in the workspace
    size_t off_ml, off_o;
    size_t off_plan;    // step plan (PKV_DECODE_MAKE_PLAN / USE_PLAN); 0: no room for one
    size_t bytes;
};

// Bytes of the step plan a workspace holds for `batch` rows (a header, the
// per-row prefix arrays and one record per CTA of the persistent grid).
size_t decode_plan_bytes(int batch);

// Fills `s`; returns false for unsupported combinations.
bool decode_shape(int batch, int max_blocks, int num_q_heads, const pkv_cache_desc &d, DecodeShape *s);

// The same for multi-query rows of up to max_qlen queries each: a unit holds
// up to 8 (query, head) columns of one kv head.
bool decode_mq_shape(int batch, int max_blocks, int num_q_heads, int max_qlen, const pkv_cache_desc &d,
                     DecodeShape *s);

// Number of split-KV work items a call aims for on this device (a few per
// resident CTA slot).
int decode_target_items(int device, int head_dim, int heads_per_cta, bool multi_query = false);

struct DecodeArgs {
    pkv_cache_desc desc;
    int page_shift;
    int batch, num_q_heads, max_blocks;
    float q_scale; // softmax_scale * log2(e)
    const int32_t *block_table;
    const int32_t *cache_seqlens;
    const void *q;
    const void *k_new;
    const void *v_new;
    void *k_cache;
    void *v_cache;
    void *out;
    float *lse;
    void *workspace;
    int32_t *err_flag;
    DecodeShape shape;
    int target_items;
    int grid;
    uint32_t flags; // PKV_DECODE_*
    // Multi-query rows (shape from decode_mq_shape; q / out / lse are
    // [total_q, Hq, ...]); qo_indptr nullptr: one query per row.
    const int32_t *qo_indptr = nullptr;
    int total_q = 0;
    int mq_hi = 0;       // rows with 1 <= q_len <= mq_hi are served
    int mq_max = 0;      // q_len > mq_max: PKV_ERR_QLEN ...
    int mq_own_long = 0; // ... and zeroed by this kernel
    int mq_kv_add = 0;   // 1: kv = L + q_len (new tokens cached); 0: kv = L
};

// TMA descriptors of one decode call: K and V pools with full boxes
// (decode_box_tokens rows) and with 8-row boxes for the ragged end of a slice
// -- token-group maps (encode_group_map) for pages of 8 tokens or more,
// unswizzled 64-column boxes (encode_pool_map, no 8-row maps) below that.
struct DecodeMaps {
    CUtensorMap k, v, k8, v8;
};

constexpr int kDecodeSmallBox = 8;

cudaError_t launch_decode(const DecodeArgs &a, const DecodeMaps &maps, cudaStream_t stream);

// K / V tensor maps of one decode call over these pools (false if encoding failed).
bool encode_decode_maps(const pkv_cache_desc &desc, void *k_cache, void *v_cache, DecodeMaps *maps);

// Every argument check of pkv_decode_attn_ex (no device access, no launch);
// fills `shape` when the sizes are supported.
pkv_status decode_check(const pkv_cache_desc *desc, const void *k_cache, const void *v_cache, const void *q,
                        const void *k_new, const void *v_new, const int32_t *block_table, int32_t max_blocks,
                        const int32_t *cache_seqlens, int32_t batch, int32_t num_q_heads, float softmax_scale,
                        const void *out, const void *workspace, size_t workspace_bytes, uint32_t flags,
                        DecodeShape *shape);

struct AppendArgs {
    pkv_cache_desc desc;
    int page_shift;
    void *k_cache;
    void *v_cache;
    const void *k_new;
    const void *v_new;
    int num_tokens;
    const int32_t *append_indptr;
    const int32_t *block_table;
    int max_blocks;
    const int32_t *cache_seqlens;
    int batch;
    int32_t *err_flag;
    int max_count = 0x7fffffff; // rows appending more tokens than this append nothing
    // Launch as a programmatic dependent of the preceding kernel: the two may
    // run side by side, so that kernel must not write what the append reads
    // or writes (k_new, v_new, the cache, indptr, cache_seqlens, block_table);
    // the append grid still completes only after it.
    bool overlap_prior = false;
};

cudaError_t launch_append(const AppendArgs &a, cudaStream_t stream);

// Decode TMA geometry: tokens per box and whether boxes are 128B-swizzled.
int decode_box_tokens(int page_size);
int decode_swizzle(int page_size);

// Tensor map over one K or V pool whose boxes are `box_tokens` consecutive
// tokens of one kv head and `box_dim` of its head_dim values
// ([box_tokens][box_dim] in shared memory), optionally 128-byte swizzled.
CUresult encode_pool_map(CUtensorMap *map, const pkv_cache_desc &d, void *base, int box_tokens, int box_dim,
                         int swizzle);

// Tensor map over one K or V pool whose boxes are `box_tokens` (a multiple
// of 8, within one page) consecutive tokens of one kv head with all head_dim
// values, landing in shared memory as [box_tokens / 8][head_dim / 64][8][64]:
// groups of 8 token rows (128 bytes each, 128-byte swizzle) for every 64-column
// block.  Consecutive 8-row groups of one column block are then head_dim * 16
// bytes apart whichever page they come from.  5-D: (64 columns, 8 tokens,
// column blocks, token groups, page-heads) over HND, (64 columns, 8 tokens,
// column blocks, token groups across pages, heads) over NHD.
// box_blocks: 64-column blocks per box (0: all of head_dim).
CUresult encode_group_map(CUtensorMap *map, const pkv_cache_desc &d, void *base, int box_tokens, int box_blocks = 0);

int sm_count(int device);

// ---------------------------------------------------------------- prefill

// Largest batch one prefill call plans for (the plan lives in shared memory).
constexpr int kMaxPrefillBatch = 1024;

// Static shape of a prefill call: the query tile and the workspace size.
struct PrefillShape {
    int group;       // num_q_heads / num_kv_heads (a power of two <= 128)
    int group_shift; // log2(group)
    int q_tile;      // queries per work unit: 128 / group
    int64_t cap_pairs; // upper bound on (request, query tile) pairs
    size_t bytes;    // workspace bytes
};

// Fills `s`; returns false for unsupported combinations.
bool prefill_shape(int batch, int total_q, int num_q_heads, const pkv_cache_desc &d, PrefillShape *s);

struct PrefillArgs {
    pkv_cache_desc desc;
    int batch, num_q_heads, total_q, max_blocks;
    float q_scale; // softmax_scale * log2(e)
    const int32_t *qo_indptr;
    const int32_t *kv_lens;
    const int32_t *block_table;
    const void *q;
    void *out;
    float *lse;
    void *workspace;
    int32_t *err_flag;
    PrefillShape shape;
    // Mixed step: kv_lens unused; request b holds cache_seqlens[b] cached
    // tokens and cache_seqlens[b] + kv_add * q keys; only requests with more
    // than q_lo queries are served, more than q_max is malformed.
    const int32_t *cache_seqlens = nullptr;
    int q_lo = 0;
    int q_max = 0x7fffffff;
    int kv_add = 0;
    // Launches: kPrefillAll = the plan kernel then the attention kernel;
    // kPrefillPlan / kPrefillMain one of them (the same arguments for both).
    int phase = 0;
    // kPrefillMain only: the preceding kernel in the stream is one of this
    // library's that waits (transitively) for the plan, so the attention
    // kernel may start its set-up before that kernel ends.
    bool overlap_prior = false;
};

constexpr int kPrefillAll = 0, kPrefillPlan = 1, kPrefillMain = 2;

// TMA descriptors of one prefill call: token-group boxes (encode_group_map)
// of min(page_size, 64) tokens of the K and V pools.
struct PrefillMaps {
    CUtensorMap k, v;
};

cudaError_t launch_prefill(const PrefillArgs &a, const PrefillMaps &maps, cudaStream_t stream);

int prefill_box_tokens(int page_size);

// The K and V tensor maps the prefill kernel for this head_dim reads.
bool encode_prefill_maps(const pkv_cache_desc &d, const void *k_cache, const void *v_cache, PrefillMaps *maps);


} // namespace pkv
