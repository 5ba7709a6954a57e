// pkv_api.cu -- C ABI front end: argument validation (no device reads, no
// host sync), workspace sizing, TMA tensor-map encoding and kernel launches.
#include <cudaTypedefs.h>
#include <math.h>
#include <mutex>

#include "pkv_internal.h"

namespace pkv {

namespace {

bool aligned16(const void *p)
{
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

int log2_exact(int x)
{
    if (x <= 0 || (x & (x - 1)) != 0)
        return -1;
    int s = 0;
    while ((1 << s) < x)
        ++s;
    return s;
}

// Geometry checks shared by every entry point.
pkv_status check_desc(const pkv_cache_desc *d)
{
    if (d == nullptr)
        return PKV_EINVAL;
    if (d->num_pages < 2 || d->num_kv_heads < 1 || d->page_size < 1 || d->head_dim < 1)
        return PKV_EINVAL;
    if (d->layout != PKV_NHD && d->layout != PKV_HND)
        return PKV_EINVAL;
    if (log2_exact(d->page_size) < 0 || d->page_size > 256)
        return PKV_EUNSUPPORTED;
    if (d->head_dim != 64 && d->head_dim != 128 && d->head_dim != 256)
        return PKV_EUNSUPPORTED;
    // TMA coordinates are int32: the token (NHD) or page-head (HND) axis must fit.
    const int64_t rows = d->layout == PKV_NHD ? (int64_t)d->num_pages * d->page_size
                                              : (int64_t)d->num_pages * d->num_kv_heads;
    if (rows > INT32_MAX)
        return PKV_EUNSUPPORTED;
    return PKV_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

int current_device()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return -1;
    return dev;
}

constexpr int kMaxDevices = 64;

} // namespace

int sm_count(int device)
{
    static int cache[kMaxDevices] = {0};
    if (device < 0 || device >= kMaxDevices)
        return 1;
    if (cache[device] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || n < 1)
            n = 1;
        cache[device] = n;
    }
    return cache[device];
}

CUresult encode_pool_map(CUtensorMap *map, const pkv_cache_desc &d, void *base, int box_tokens, int box_dim,
                         int swizzle)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (enc == nullptr)
        return CUDA_ERROR_NOT_FOUND;
    const cuuint64_t D = (cuuint64_t)d.head_dim;
    cuuint64_t dims[3];
    cuuint64_t strides[2]; // bytes, for dims 1 and 2
    cuuint32_t box[3];
    if (d.layout == PKV_NHD) { // [pages*P, Hkv, D]
        dims[0] = D;
        dims[1] = (cuuint64_t)d.num_kv_heads;
        dims[2] = (cuuint64_t)d.num_pages * d.page_size;
        strides[0] = D * 2;
        strides[1] = D * 2 * d.num_kv_heads;
        box[0] = (cuuint32_t)box_dim;
        box[1] = 1;
        box[2] = (cuuint32_t)box_tokens;
    } else { // [pages*Hkv, P, D]
        dims[0] = D;
        dims[1] = (cuuint64_t)d.page_size;
        dims[2] = (cuuint64_t)d.num_pages * d.num_kv_heads;
        strides[0] = D * 2;
        strides[1] = D * 2 * d.page_size;
        box[0] = (cuuint32_t)box_dim;
        box[1] = (cuuint32_t)box_tokens;
        box[2] = 1;
    }
    const cuuint32_t elem_strides[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, elem_strides,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}



CUresult encode_group_map(CUtensorMap *map, const pkv_cache_desc &d, void *base, int box_tokens, int box_blocks)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (enc == nullptr)
        return CUDA_ERROR_NOT_FOUND;
    const cuuint64_t D = (cuuint64_t)d.head_dim, P = (cuuint64_t)d.page_size, H = (cuuint64_t)d.num_kv_heads;
    const cuuint32_t blocks = box_blocks > 0 ? (cuuint32_t)box_blocks : (cuuint32_t)(D / 64);
    const cuuint32_t box[5] = {64, 8, blocks, (cuuint32_t)(box_tokens / 8), 1};
    const cuuint32_t elem_strides[5] = {1, 1, 1, 1, 1};
    cuuint64_t dims[5], strides[4];
    if (d.layout == PKV_HND) { // [pages * Hkv][P][D]
        const cuuint64_t v_dims[5] = {64, 8, D / 64, P / 8, (cuuint64_t)d.num_pages * H};
        const cuuint64_t v_strides[4] = {D * 2, 128, 8 * D * 2, P * D * 2};
        for (int i = 0; i < 5; ++i)
            dims[i] = v_dims[i];
        for (int i = 0; i < 4; ++i)
            strides[i] = v_strides[i];
    } else { // [pages * P][Hkv][D]: token groups run across pages
        const cuuint64_t v_dims[5] = {64, 8, D / 64, (cuuint64_t)d.num_pages * P / 8, H};
        const cuuint64_t v_strides[4] = {H * D * 2, 128, 8 * H * D * 2, D * 2};
        for (int i = 0; i < 5; ++i)
            dims[i] = v_dims[i];
        for (int i = 0; i < 4; ++i)
            strides[i] = v_strides[i];
    }
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, base, dims, strides, box, elem_strides,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

bool encode_decode_maps(const pkv_cache_desc &desc, void *k_cache, void *v_cache, DecodeMaps *maps)
{
    const int box = decode_box_tokens(desc.page_size);
    if (decode_swizzle(desc.page_size)) { // pages of 8+ tokens: token-group boxes
        return encode_group_map(&maps->k, desc, k_cache, box) == CUDA_SUCCESS &&
               encode_group_map(&maps->v, desc, v_cache, box) == CUDA_SUCCESS &&
               encode_group_map(&maps->k8, desc, k_cache, kDecodeSmallBox) == CUDA_SUCCESS &&
               encode_group_map(&maps->v8, desc, v_cache, kDecodeSmallBox) == CUDA_SUCCESS;
    }
    // pages of 1, 2 or 4 tokens: unswizzled 64-column boxes
    if (encode_pool_map(&maps->k, desc, k_cache, box, 64, 0) != CUDA_SUCCESS ||
        encode_pool_map(&maps->v, desc, v_cache, box, 64, 0) != CUDA_SUCCESS)
        return false;
    maps->k8 = maps->k;
    maps->v8 = maps->v;
    return true;
}

// Static split of a mixed step: the decode kernel's multi-query shape, and
// whether (and where in the workspace) the prefill kernel runs.
struct MixedShape {
    int dq;            // longest query range the decode kernel serves
    bool prefill;      // rows longer than dq exist: the prefill kernel runs
    DecodeShape dshape;
    PrefillShape pshape;
    size_t off_prefill; // prefill plan in the workspace
    size_t bytes;
};

pkv_status mixed_shape(const pkv_cache_desc *desc, int32_t batch, int32_t total_q, int32_t max_blocks,
                       int32_t num_q_heads, int32_t max_qlen, int32_t decode_max_qlen, MixedShape *m)
{
    const pkv_status st = check_desc(desc);
    if (st != PKV_OK)
        return st;
    if (batch < 0 || total_q < 0 || max_blocks < 1 || num_q_heads < 1 || max_qlen < 1 || decode_max_qlen < 1)
        return PKV_EINVAL;
    if (num_q_heads % desc->num_kv_heads != 0)
        return PKV_EINVAL;
    if (batch > kMaxDecodeBatch || batch > kMaxPrefillBatch)
        return PKV_EUNSUPPORTED;
    // output rows (one per query and head) are numbered in int32
    if ((int64_t)total_q * num_q_heads >= ((int64_t)1 << 31))
        return PKV_EUNSUPPORTED;
    m->dq = decode_max_qlen < max_qlen ? decode_max_qlen : max_qlen;
    m->prefill = max_qlen > m->dq;
    if (!decode_mq_shape(batch, max_blocks, num_q_heads, m->dq, *desc, &m->dshape))
        return PKV_EUNSUPPORTED;
    m->off_prefill = (m->dshape.bytes + 255) & ~size_t(255);
    m->bytes = m->off_prefill;
    if (m->prefill) {
        if (!prefill_shape(batch, total_q, num_q_heads, *desc, &m->pshape))
            return PKV_EUNSUPPORTED; // e.g. pages of fewer than 8 tokens
        m->bytes += m->pshape.bytes;
    }
    return PKV_OK;
}

pkv_status decode_check(const pkv_cache_desc *desc, const void *k_cache, const void *v_cache, const void *q,
                        const void *k_new, const void *v_new, const int32_t *block_table, int32_t max_blocks,
                        const int32_t *cache_seqlens, int32_t batch, int32_t num_q_heads, float softmax_scale,
                        const void *out, const void *workspace, size_t workspace_bytes, uint32_t flags,
                        DecodeShape *shape)
{
    if ((flags & ~(PKV_DECODE_OVERLAP_PROLOGUE | PKV_DECODE_EARLY_KV | PKV_DECODE_MAKE_PLAN |
                   PKV_DECODE_USE_PLAN)) != 0)
        return PKV_EINVAL;
    if ((flags & PKV_DECODE_EARLY_KV) && !(flags & PKV_DECODE_OVERLAP_PROLOGUE))
        return PKV_EINVAL;
    if ((flags & PKV_DECODE_MAKE_PLAN) && (flags & PKV_DECODE_USE_PLAN))
        return PKV_EINVAL;
    const pkv_status st = check_desc(desc);
    if (st != PKV_OK)
        return st;
    if (batch < 0 || max_blocks < 1 || num_q_heads < 1 || !isfinite(softmax_scale))
        return PKV_EINVAL;
    if (batch > kMaxDecodeBatch)
        return PKV_EUNSUPPORTED;
    if ((k_new == nullptr) != (v_new == nullptr))
        return PKV_EINVAL;
    if (num_q_heads % desc->num_kv_heads != 0)
        return PKV_EINVAL;
    if (!decode_shape(batch, max_blocks, num_q_heads, *desc, shape))
        return PKV_EUNSUPPORTED;
    if (batch == 0)
        return PKV_OK;
    if (k_cache == nullptr || v_cache == nullptr || q == nullptr || out == nullptr || block_table == nullptr ||
        cache_seqlens == nullptr)
        return PKV_EINVAL;
    if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(q) || !aligned16(out) ||
        (k_new != nullptr && (!aligned16(k_new) || !aligned16(v_new))))
        return PKV_EINVAL;
    if (workspace == nullptr || workspace_bytes < shape->bytes || !aligned16(workspace))
        return PKV_EWORKSPACE;
    return PKV_OK;
}
} // namespace pkv

using namespace pkv;

extern "C" {

const char *pkv_status_str(pkv_status status)
{
    switch (status) {
    case PKV_OK:
        return "ok";
    case PKV_EINVAL:
        return "invalid argument";
    case PKV_EUNSUPPORTED:
        return "unsupported size or layout";
    case PKV_ECUDA:
        return "CUDA call failed";
    case PKV_ENOPAGES:
        return "page pool exhausted";
    case PKV_EWORKSPACE:
        return "workspace missing or too small";
    case PKV_ETOOBIG:
        return "problem larger than the built-in scratch (use pkv_decode_attn with a workspace)";
    }
    return "unknown status";
}

uint64_t pkv_pool_bytes(const pkv_cache_desc *desc)
{
    if (desc == nullptr || desc->num_pages < 0 || desc->page_size < 0 || desc->num_kv_heads < 0 ||
        desc->head_dim < 0)
        return 0;
    return (uint64_t)desc->num_pages * (uint64_t)desc->page_size * (uint64_t)desc->num_kv_heads *
           (uint64_t)desc->head_dim * 2u;
}

pkv_status pkv_append(const pkv_cache_desc *desc, void *k_cache, void *v_cache, const void *k_new,
                      const void *v_new, int32_t num_tokens, const int32_t *append_indptr,
                      const int32_t *block_table, int32_t max_blocks, const int32_t *cache_seqlens, int32_t batch,
                      int32_t *err_flag, void *stream)
{
    const pkv_status st = check_desc(desc);
    if (st != PKV_OK)
        return st;
    if (batch < 0 || num_tokens < 0 || max_blocks < 1)
        return PKV_EINVAL;
    if (append_indptr == nullptr && num_tokens != batch)
        return PKV_EINVAL;
    if (batch == 0 || num_tokens == 0)
        return PKV_OK;
    if (k_cache == nullptr || v_cache == nullptr || k_new == nullptr || v_new == nullptr ||
        block_table == nullptr || cache_seqlens == nullptr)
        return PKV_EINVAL;
    if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_new) || !aligned16(v_new))
        return PKV_EINVAL;
    AppendArgs a;
    a.desc = *desc;
    a.page_shift = log2_exact(desc->page_size);
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.k_new = k_new;
    a.v_new = v_new;
    a.num_tokens = num_tokens;
    a.append_indptr = append_indptr;
    a.block_table = block_table;
    a.max_blocks = max_blocks;
    a.cache_seqlens = cache_seqlens;
    a.batch = batch;
    a.err_flag = err_flag;
    return launch_append(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

size_t pkv_decode_workspace_size(int32_t batch, int32_t max_blocks, int32_t num_q_heads, const pkv_cache_desc *desc)
{
    if (check_desc(desc) != PKV_OK || batch < 0 || batch > kMaxDecodeBatch || max_blocks < 1 || num_q_heads < 1)
        return 0;
    DecodeShape s;
    if (!decode_shape(batch, max_blocks, num_q_heads, *desc, &s))
        return 0;
    return s.bytes;
}

pkv_status pkv_decode_attn(const pkv_cache_desc *desc, void *k_cache, void *v_cache, const void *q,
                           const void *k_new, const void *v_new, const int32_t *block_table, int32_t max_blocks,
                           const int32_t *cache_seqlens, int32_t batch, int32_t num_q_heads, float softmax_scale,
                           void *out, float *lse, void *workspace, size_t workspace_bytes, int32_t *err_flag,
                           void *stream)
{
    return pkv_decode_attn_ex(desc, k_cache, v_cache, q, k_new, v_new, block_table, max_blocks, cache_seqlens, batch,
                              num_q_heads, softmax_scale, out, lse, workspace, workspace_bytes, err_flag, stream, 0u);
}

pkv_status pkv_decode_attn_ex(const pkv_cache_desc *desc, void *k_cache, void *v_cache, const void *q,
                              const void *k_new, const void *v_new, const int32_t *block_table, int32_t max_blocks,
                              const int32_t *cache_seqlens, int32_t batch, int32_t num_q_heads, float softmax_scale,
                              void *out, float *lse, void *workspace, size_t workspace_bytes, int32_t *err_flag,
                              void *stream, uint32_t flags)
{
    DecodeShape shape;
    const pkv_status st = decode_check(desc, k_cache, v_cache, q, k_new, v_new, block_table, max_blocks, cache_seqlens,
                                       batch, num_q_heads, softmax_scale, out, workspace, workspace_bytes, flags,
                                       &shape);
    if (st != PKV_OK || batch == 0)
        return st;

    const int dev = current_device();
    if (dev < 0)
        return PKV_ECUDA;
    DecodeArgs a;
    a.desc = *desc;
    a.page_shift = log2_exact(desc->page_size);
    a.batch = batch;
    a.num_q_heads = num_q_heads;
    a.max_blocks = max_blocks;
    a.q_scale = softmax_scale * 1.4426950408889634f;
    a.block_table = block_table;
    a.cache_seqlens = cache_seqlens;
    a.q = q;
    a.k_new = k_new;
    a.v_new = v_new;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.out = out;
    a.lse = lse;
    a.workspace = workspace;
    a.err_flag = err_flag;
    a.shape = shape;
    // persistent grid: every CTA that fits on the device at once
    a.target_items = 0;
    a.grid = decode_target_items(dev, desc->head_dim, shape.heads_per_cta);
    a.flags = flags;

    DecodeMaps maps;
    if (!encode_decode_maps(*desc, k_cache, v_cache, &maps))
        return PKV_ECUDA;
    return launch_decode(a, maps, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

size_t pkv_prefill_workspace_size(int32_t batch, int32_t total_q, int32_t num_q_heads, const pkv_cache_desc *desc)
{
    if (check_desc(desc) != PKV_OK || batch < 0 || batch > kMaxPrefillBatch || total_q < 0 || num_q_heads < 1)
        return 0;
    PrefillShape s;
    if (!prefill_shape(batch, total_q, num_q_heads, *desc, &s))
        return 0;
    return s.bytes;
}

pkv_status pkv_prefill_attn(const pkv_cache_desc *desc, const void *k_cache, const void *v_cache, const void *q,
                            const int32_t *qo_indptr, const int32_t *kv_lens, const int32_t *block_table,
                            int32_t max_blocks, int32_t batch, int32_t num_q_heads, int32_t total_q,
                            float softmax_scale, void *out, float *lse, void *workspace, size_t workspace_bytes,
                            int32_t *err_flag, void *stream)
{
    const pkv_status st = check_desc(desc);
    if (st != PKV_OK)
        return st;
    if (batch < 0 || total_q < 0 || max_blocks < 1 || num_q_heads < 1 || !isfinite(softmax_scale))
        return PKV_EINVAL;
    if (num_q_heads % desc->num_kv_heads != 0)
        return PKV_EINVAL;
    if (batch > kMaxPrefillBatch)
        return PKV_EUNSUPPORTED;
    PrefillShape shape;
    if (!prefill_shape(batch, total_q, num_q_heads, *desc, &shape))
        return PKV_EUNSUPPORTED;
    if (batch == 0 || total_q == 0)
        return PKV_OK;
    if (k_cache == nullptr || v_cache == nullptr || q == nullptr || out == nullptr || qo_indptr == nullptr ||
        kv_lens == nullptr || block_table == nullptr)
        return PKV_EINVAL;
    if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(q) || !aligned16(out))
        return PKV_EINVAL;
    if (workspace == nullptr || workspace_bytes < shape.bytes || !aligned16(workspace))
        return PKV_EWORKSPACE;

    PrefillArgs a;
    a.desc = *desc;
    a.batch = batch;
    a.num_q_heads = num_q_heads;
    a.total_q = total_q;
    a.max_blocks = max_blocks;
    a.q_scale = softmax_scale * 1.4426950408889634f;
    a.qo_indptr = qo_indptr;
    a.kv_lens = kv_lens;
    a.block_table = block_table;
    a.q = q;
    a.out = out;
    a.lse = lse;
    a.workspace = workspace;
    a.err_flag = err_flag;
    a.shape = shape;
    PrefillMaps maps;
    if (!encode_prefill_maps(*desc, k_cache, v_cache, &maps))
        return PKV_ECUDA;
    return launch_prefill(a, maps, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

size_t pkv_mixed_workspace_size(int32_t batch, int32_t total_q, int32_t max_blocks, int32_t num_q_heads,
                                int32_t max_qlen, int32_t decode_max_qlen, const pkv_cache_desc *desc)
{
    MixedShape m;
    if (mixed_shape(desc, batch, total_q, max_blocks, num_q_heads, max_qlen, decode_max_qlen, &m) != PKV_OK)
        return 0;
    return m.bytes;
}

pkv_status pkv_mixed_attn(const pkv_cache_desc *desc, void *k_cache, void *v_cache, const void *q, const void *k_new,
                          const void *v_new, const int32_t *qo_indptr, const int32_t *block_table, int32_t max_blocks,
                          const int32_t *cache_seqlens, int32_t batch, int32_t num_q_heads, int32_t total_q,
                          int32_t max_qlen, int32_t decode_max_qlen, float softmax_scale, void *out, float *lse,
                          void *workspace, size_t workspace_bytes, int32_t *err_flag, void *stream)
{
    MixedShape m;
    pkv_status st = mixed_shape(desc, batch, total_q, max_blocks, num_q_heads, max_qlen, decode_max_qlen, &m);
    if (st != PKV_OK)
        return st;
    if (!isfinite(softmax_scale) || (k_new == nullptr) != (v_new == nullptr))
        return PKV_EINVAL;
    if (batch == 0)
        return PKV_OK;
    if (k_cache == nullptr || v_cache == nullptr || qo_indptr == nullptr || block_table == nullptr ||
        cache_seqlens == nullptr || (total_q > 0 && (q == nullptr || out == nullptr)))
        return PKV_EINVAL;
    if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(q) || !aligned16(out) ||
        (k_new != nullptr && (!aligned16(k_new) || !aligned16(v_new))))
        return PKV_EINVAL;
    if (workspace == nullptr || workspace_bytes < m.bytes || !aligned16(workspace))
        return PKV_EWORKSPACE;
    const int dev = current_device();
    if (dev < 0)
        return PKV_ECUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const float q_scale = softmax_scale * 1.4426950408889634f;

    // Launch order: the prefill plan (when longer rows exist; it reads only
    // the row arrays and the table), the append (a programmatic dependent of
    // the plan: the two run side by side, and the append completes after the
    // plan), the decode kernel (a programmatic dependent of the append: its
    // plan and page-id prefetch overlap the append), then the prefill kernel.
    PrefillArgs pa;
    PrefillMaps pmaps;
    if (m.prefill) {
        pa.desc = *desc;
        pa.batch = batch;
        pa.num_q_heads = num_q_heads;
        pa.total_q = total_q;
        pa.max_blocks = max_blocks;
        pa.q_scale = q_scale;
        pa.qo_indptr = qo_indptr;
        pa.kv_lens = nullptr;
        pa.block_table = block_table;
        pa.q = q;
        pa.out = out;
        pa.lse = lse;
        pa.workspace = static_cast<unsigned char *>(workspace) + m.off_prefill;
        pa.err_flag = err_flag;
        pa.shape = m.pshape;
        pa.cache_seqlens = cache_seqlens;
        pa.q_lo = m.dq;
        pa.q_max = max_qlen;
        pa.kv_add = k_new != nullptr ? 1 : 0;
        if (!encode_prefill_maps(*desc, k_cache, v_cache, &pmaps))
            return PKV_ECUDA;
        pa.phase = kPrefillPlan;
        if (launch_prefill(pa, pmaps, s) != cudaSuccess)
            return PKV_ECUDA;
    }

    // 1. the new tokens of every row into the cache (rows longer than max_qlen append nothing)
    const bool appended = k_new != nullptr && total_q > 0;
    if (appended) {
        AppendArgs a;
        a.desc = *desc;
        a.page_shift = log2_exact(desc->page_size);
        a.k_cache = k_cache;
        a.v_cache = v_cache;
        a.k_new = k_new;
        a.v_new = v_new;
        a.num_tokens = total_q;
        a.append_indptr = qo_indptr;
        a.block_table = block_table;
        a.max_blocks = max_blocks;
        a.cache_seqlens = cache_seqlens;
        a.batch = batch;
        a.err_flag = err_flag;
        a.max_count = max_qlen;
        a.overlap_prior = m.prefill;
        if (launch_append(a, s) != cudaSuccess)
            return PKV_ECUDA;
    }

    // 2. rows of 1 .. dq queries: the split-KV decode kernel, (query, head) columns
    {
        DecodeArgs a;
        a.desc = *desc;
        a.page_shift = log2_exact(desc->page_size);
        a.batch = batch;
        a.num_q_heads = num_q_heads;
        a.max_blocks = max_blocks;
        a.q_scale = q_scale;
        a.block_table = block_table;
        a.cache_seqlens = cache_seqlens;
        a.q = q;
        a.k_new = nullptr;
        a.v_new = nullptr;
        a.k_cache = k_cache;
        a.v_cache = v_cache;
        a.out = out;
        a.lse = lse;
        a.workspace = workspace;
        a.err_flag = err_flag;
        a.shape = m.dshape;
        a.target_items = 0;
        a.grid = decode_target_items(dev, desc->head_dim, m.dshape.heads_per_cta, true);
        // after the append only: the user's kernel before this call may write
        // the row arrays, which the overlapped prologue reads
        a.flags = appended ? PKV_DECODE_OVERLAP_PROLOGUE : 0u;
        a.qo_indptr = qo_indptr;
        a.total_q = total_q;
        a.mq_hi = m.dq;
        a.mq_max = max_qlen;
        a.mq_own_long = m.prefill ? 0 : 1;
        a.mq_kv_add = k_new != nullptr ? 1 : 0;
        DecodeMaps maps;
        if (!encode_decode_maps(*desc, k_cache, v_cache, &maps))
            return PKV_ECUDA;
        if (launch_decode(a, maps, s) != cudaSuccess)
            return PKV_ECUDA;
    }

    // 3. longer rows (prefill chunks): the tcgen05 prefill kernel over kv = L + q keys
    if (m.prefill) {
        pa.phase = kPrefillMain;
        pa.overlap_prior = true; // the decode kernel waited for the append, which waited for the plan
        if (launch_prefill(pa, pmaps, s) != cudaSuccess)
            return PKV_ECUDA;
    }
    return PKV_OK;
}

} // extern "C"
