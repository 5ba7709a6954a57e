// pkv_static.cu -- decode for callers that cannot allocate device memory.
//
// pkv_decode_attn needs a caller-provided workspace for its split-KV partial
// results.  Some callers cannot provide one: code running inside a host
// framework that owns every byte of device memory and forbids its plug-ins
// to allocate (an inference engine's custom-op or plug-in interface, for
// example), or a hard real-time serving loop that must not call the
// allocator after start-up.  pkv_decode_attn_noalloc gives them the same
// computation with the workspace taken from a fixed array compiled into this
// library instead.
#include <mutex>

#include "pkv_internal.h"

namespace pkv {
namespace {

// Built-in scratch: enough for every problem whose pkv_decode_workspace_size
// is at most this.  Each GPU that loads the library holds it until exit.
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_scratch_addr[kMaxDevices]; // device address of the array, per device

// Device address of the array on the current device (the symbol's host name
// is only a stand-in).  Looked up once per device, on its first use.
cudaError_t scratch_address(void **addr)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess)
            return e;
        g_scratch_addr[dev] = p;
    }
    *addr = g_scratch_addr[dev];
    return cudaSuccess;
}

} // namespace
} // namespace pkv

using namespace pkv;

extern "C" PKV_API pkv_status pkv_decode_attn_noalloc(const pkv_cache_desc *desc, void *k_cache, void *v_cache,
                                                      const void *q, const void *k_new, const void *v_new,
                                                      const int32_t *block_table, int32_t max_blocks,
                                                      const int32_t *cache_seqlens, int32_t batch,
                                                      int32_t num_q_heads, float softmax_scale, void *out, float *lse,
                                                      int32_t *err_flag, void *stream)
{
    // Every argument check of pkv_decode_attn first, with a placeholder for
    // the workspace (an aligned non-null address and no size limit), so an
    // invalid call gets the same status it would get there and touches
    // nothing: not the shared array, not the stream.
    DecodeShape shape;
    const pkv_status st = decode_check(desc, k_cache, v_cache, q, k_new, v_new, block_table, max_blocks,
                                       cache_seqlens, batch, num_q_heads, softmax_scale, out,
                                       reinterpret_cast<const void *>(uintptr_t(256)), ~size_t(0), 0u, &shape);
    if (st != PKV_OK || batch == 0)
        return st;
    if (shape.bytes > kNoAllocScratchBytes)
        return PKV_ETOOBIG;
    void *scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess)
        return PKV_ECUDA;
    // The combine tickets at the front of the workspace must start at zero;
    // every call shares the array, so clear them on the call's stream.
    if (cudaMemsetAsync(scratch, 0, shape.off_ml, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return PKV_ECUDA;
    return pkv_decode_attn_ex(desc, k_cache, v_cache, q, k_new, v_new, block_table, max_blocks, cache_seqlens, batch,
                              num_q_heads, softmax_scale, out, lse, scratch, kNoAllocScratchBytes, err_flag, stream,
                              0u);
}
