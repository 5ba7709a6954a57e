// pkv_append.cu -- standalone append of new tokens' K/V into their page
// slots ("mini-infer系统实战-06 True PagedAttention", section 1: the new K/V
// are written in place into the block slot selected by block_table and
// cache_seqlens).  A bit copy: 16-byte vector loads from k_new/v_new, 16-byte
// stores into the pool.  All-or-nothing per row: if any destination page of a
// row is outside [1, num_pages) or the row would overflow its table, the row
// writes nothing and an error bit is raised.
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kAppendThreads = 128;

struct AParams {
    __nv_bfloat16 *k_cache;
    __nv_bfloat16 *v_cache;
    const __nv_bfloat16 *k_new;
    const __nv_bfloat16 *v_new;
    const int32_t *indptr;
    const int32_t *block_table;
    const int32_t *seqlens;
    int32_t *err_flag;
    int num_tokens, batch, max_blocks, page_size, page_shift, num_pages, num_kv_heads, head_dim, layout;
    int max_count; // rows appending more tokens than this append nothing
    int pdl_wait;  // launched as a programmatic dependent: wait for the preceding grid before exiting
};

// One CTA per new token.
__device__ __forceinline__ void append_token(const AParams &p)
{
    __shared__ int s_row, s_first, s_count;
    const int t = blockIdx.x;
    if (threadIdx.x == 0) {
        int b = t, first = t, count = 1;
        if (p.indptr != nullptr) { // row owning token t: last b with indptr[b] <= t
            int lo = 0, hi = p.batch - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (p.indptr[mid] <= t)
                    lo = mid;
                else
                    hi = mid - 1;
            }
            b = lo;
            first = p.indptr[b];
            count = p.indptr[b + 1] - first;
        }
        s_row = b;
        s_first = first;
        s_count = count;
    }
    __syncthreads();
    const int b = s_row, count = s_count;
    const int L = p.seqlens[b];
    // inactive row; a token outside its row's range (a malformed indptr); a
    // row whose range leaves [0, num_tokens) or that is longer than allowed
    if (L < 0 || t < s_first || t - s_first >= count || s_first < 0 || count > p.num_tokens - s_first ||
        count > p.max_count)
        return;
    // validate the row's destination range [L, L + count)
    const int32_t *bt_row = p.block_table + (int64_t)b * p.max_blocks;
    int err = 0;
    if ((int64_t)L + count > (int64_t)p.max_blocks * p.page_size) {
        err = PKV_ERR_OVERFLOW;
    } else {
        const int blk0 = L >> p.page_shift, blk1 = (L + count - 1) >> p.page_shift;
        int bad = 0;
        for (int k = blk0 + threadIdx.x; k <= blk1; k += kAppendThreads) {
            const int page = bt_row[k];
            bad |= page < 1 || page >= p.num_pages;
        }
        if (__syncthreads_or(bad))
            err = PKV_ERR_PAGE;
    }
    if (err) {
        if (threadIdx.x == 0)
            set_error(p.err_flag, err);
        return;
    }
    const int pos = L + (t - s_first);
    const int page = bt_row[pos >> p.page_shift];
    const int slot = pos & (p.page_size - 1);
    const int D = p.head_dim, H = p.num_kv_heads;
    const int vec_per_head = D / 8;
    const int n_vec = H * vec_per_head;
    const uint4 *ksrc = reinterpret_cast<const uint4 *>(p.k_new + (int64_t)t * H * D);
    const uint4 *vsrc = reinterpret_cast<const uint4 *>(p.v_new + (int64_t)t * H * D);
    for (int c = threadIdx.x; c < n_vec; c += kAppendThreads) {
        const int h = c / vec_per_head, v = c - h * vec_per_head;
        const int64_t dst = p.layout == PKV_NHD ? (((int64_t)page * p.page_size + slot) * H + h) * D
                                                : (((int64_t)page * H + h) * p.page_size + slot) * D;
        reinterpret_cast<uint4 *>(p.k_cache + dst)[v] = ksrc[c];
        reinterpret_cast<uint4 *>(p.v_cache + dst)[v] = vsrc[c];
    }
}

// The next kernel in the stream may start as soon as every CTA has begun (it
// waits for this grid's completion before touching what this grid writes).
// With pdl_wait the grid itself overlaps the preceding kernel, which shares
// no buffer with it, and completes only after that kernel, so that a kernel
// waiting on this grid also waits on the one before.
__global__ void __launch_bounds__(kAppendThreads) append_kernel(const __grid_constant__ AParams p)
{
    if (threadIdx.x == 0)
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    append_token(p);
    if (p.pdl_wait)
        asm volatile("griddepcontrol.wait;" ::: "memory");
}

} // namespace

cudaError_t launch_append(const AppendArgs &a, cudaStream_t stream)
{
    if (a.num_tokens == 0)
        return cudaSuccess;
    AParams p;
    p.k_cache = static_cast<__nv_bfloat16 *>(a.k_cache);
    p.v_cache = static_cast<__nv_bfloat16 *>(a.v_cache);
    p.k_new = static_cast<const __nv_bfloat16 *>(a.k_new);
    p.v_new = static_cast<const __nv_bfloat16 *>(a.v_new);
    p.indptr = a.append_indptr;
    p.block_table = a.block_table;
    p.seqlens = a.cache_seqlens;
    p.err_flag = a.err_flag;
    p.num_tokens = a.num_tokens;
    p.batch = a.batch;
    p.max_blocks = a.max_blocks;
    p.page_size = a.desc.page_size;
    p.page_shift = a.page_shift;
    p.num_pages = a.desc.num_pages;
    p.num_kv_heads = a.desc.num_kv_heads;
    p.head_dim = a.desc.head_dim;
    p.layout = a.desc.layout;
    p.max_count = a.max_count;
    p.pdl_wait = a.overlap_prior ? 1 : 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.num_tokens);
    cfg.blockDim = dim3(kAppendThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (a.overlap_prior) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    void *args[] = {&p};
    return cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(&append_kernel), args);
}

} // namespace pkv
