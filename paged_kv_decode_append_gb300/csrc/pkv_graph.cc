// pkv_graph.cc -- a whole decode step (every layer's fused append + decode)
// captured once into a CUDA graph and replayed step after step.
//
// Source: "flex_attention + paged KV + CUDA graphs vs vLLM", "Why this works":
// one CUDA graph per batch bucket replays the step's launches; padding rows
// take the reserved null slot so that one graph serves every batch up to the
// bucket.  Here padding rows are inactive (cache_seqlens < 0), which the decode
// kernel skips at no cost.
#include <cuda_runtime.h>

#include <new>

#include "pkv_internal.h"

struct pkv_decode_step {
    cudaGraphExec_t exec;
    int32_t layers;
};

namespace {

bool all_set(const void *const *p, int32_t n)
{
    if (p == nullptr)
        return false;
    for (int32_t i = 0; i < n; ++i)
        if (p[i] == nullptr)
            return false;
    return true;
}

} // namespace

extern "C" {

int32_t pkv_decode_bucket(int32_t batch)
{
    if (batch < 1 || batch > 1024)
        return 0;
    int32_t b = 8;
    while (b < batch)
        b <<= 1;
    return b;
}

pkv_status pkv_decode_step_create(const pkv_cache_desc *desc, int32_t num_layers, void *const *k_caches,
                                  void *const *v_caches, const void *const *q, const void *const *k_new,
                                  const void *const *v_new, const int32_t *block_table, int32_t max_blocks,
                                  const int32_t *cache_seqlens, int32_t batch, int32_t num_q_heads,
                                  float softmax_scale, void *const *out, float *const *lse, void *workspace,
                                  size_t workspace_bytes, int32_t *err_flag, uint32_t flags,
                                  pkv_decode_step **step_out)
{
    if (step_out == nullptr)
        return PKV_EINVAL;
    *step_out = nullptr;
    if (num_layers < 1 || batch < 1)
        return PKV_EINVAL;
    if (!all_set(reinterpret_cast<const void *const *>(k_caches), num_layers) ||
        !all_set(reinterpret_cast<const void *const *>(v_caches), num_layers) || !all_set(q, num_layers) ||
        !all_set(reinterpret_cast<const void *const *>(out), num_layers))
        return PKV_EINVAL;
    if ((k_new == nullptr) != (v_new == nullptr))
        return PKV_EINVAL;
    if (flags & PKV_DECODE_MAKE_PLAN)
        return PKV_EINVAL; // the step makes its plan itself (PKV_DECODE_USE_PLAN)
    if (k_new != nullptr && (!all_set(k_new, num_layers) || !all_set(v_new, num_layers)))
        return PKV_EINVAL;
    // Every argument check of the layer calls, before any CUDA work.
    for (int32_t l = 0; l < num_layers; ++l) {
        pkv::DecodeShape shape;
        const pkv_status st = pkv::decode_check(desc, k_caches[l], v_caches[l], q[l], k_new ? k_new[l] : nullptr,
                                                v_new ? v_new[l] : nullptr, block_table, max_blocks, cache_seqlens,
                                                batch, num_q_heads, softmax_scale, out[l], workspace, workspace_bytes,
                                                flags, &shape);
        if (st != PKV_OK)
            return st;
    }

    cudaStream_t cap = nullptr;
    if (cudaStreamCreateWithFlags(&cap, cudaStreamNonBlocking) != cudaSuccess)
        return PKV_ECUDA;
    pkv_status st = PKV_OK;
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    if (cudaStreamBeginCapture(cap, cudaStreamCaptureModeRelaxed) != cudaSuccess) {
        cudaStreamDestroy(cap);
        return PKV_ECUDA;
    }
    // With PKV_DECODE_USE_PLAN the first layer makes the step plan that the
    // others reuse (all layers share cache_seqlens and block_table).
    for (int32_t l = 0; l < num_layers && st == PKV_OK; ++l) {
        uint32_t f = flags;
        if (l == 0 && (flags & PKV_DECODE_USE_PLAN))
            f = (flags & ~PKV_DECODE_USE_PLAN) | PKV_DECODE_MAKE_PLAN;
        st = pkv_decode_attn_ex(desc, k_caches[l], v_caches[l], q[l], k_new ? k_new[l] : nullptr,
                                v_new ? v_new[l] : nullptr, block_table, max_blocks, cache_seqlens, batch,
                                num_q_heads, softmax_scale, out[l], lse ? lse[l] : nullptr, workspace,
                                workspace_bytes, err_flag, cap, f);
    }
    const cudaError_t end = cudaStreamEndCapture(cap, &graph);
    if (st == PKV_OK && end != cudaSuccess)
        st = PKV_ECUDA;
    if (st == PKV_OK && cudaGraphInstantiate(&exec, graph, 0) != cudaSuccess)
        st = PKV_ECUDA;
    if (graph != nullptr)
        cudaGraphDestroy(graph);
    cudaStreamDestroy(cap);
    if (st != PKV_OK) {
        if (exec != nullptr)
            cudaGraphExecDestroy(exec);
        return st;
    }
    pkv_decode_step *step = new (std::nothrow) pkv_decode_step;
    if (step == nullptr) {
        cudaGraphExecDestroy(exec);
        return PKV_ECUDA;
    }
    step->exec = exec;
    step->layers = num_layers;
    *step_out = step;
    return PKV_OK;
}

pkv_status pkv_decode_step_launch(pkv_decode_step *step, void *stream)
{
    if (step == nullptr)
        return PKV_EINVAL;
    return cudaGraphLaunch(step->exec, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

void pkv_decode_step_destroy(pkv_decode_step *step)
{
    if (step == nullptr)
        return;
    cudaGraphExecDestroy(step->exec);
    delete step;
}

} // extern "C"
