// pkv_decode.cu -- fused append + single-token GQA decode attention over a
// paged KV cache, with device-side split-KV planning and a log-sum-exp
// combine of the partial results.
//
// What it computes ("mini-infer系统实战-06 True PagedAttention", sections 1,
// 3 and 6): for each request b with L = cache_seqlens[b] >= 0, the new
// token's K/V go to logical position L (page block_table[b][L / P], slot
// L % P), and every query head h attends keys 0..L of kv head
// h / (Hq / Hkv) read straight from their physical pages.  The split-KV
// structure (work split along the key axis, partial results merged by their
// log-sum-exp) is the one the page's profile names (flash_fwd_splitkv_kernel).
//
// GB300 design:
//  * One CTA = 1 producer warp + 4 consumer warps.  The producer streams
//    32-token tiles of K and V for one kv head through a 3-6 stage
//    shared-memory ring with TMA (cp.async.bulk.tensor, one box per page
//    piece, L2 evict-first), completion tracked by mbarriers.
//  * Consumers hold the pre-scaled queries of up to 4 heads (q * scale *
//    log2 e, the pages' PRESCALE_QK lesson) in fp32 registers; 8 lanes
//    share one key row (16 B vector reads from shared memory), QK and PV run
//    as packed fp32x2 FMAs, online softmax in base 2 with a warp-uniform
//    running max, reductions by warp shuffles.
//  * Work items are (row, kv head, head group, key chunk).  Every CTA
//    rebuilds the same plan from cache_seqlens (no host readback): the
//    chunk size is the smallest multiple of the tile that yields about
//    `target_items` items, so one long row is split over many SMs.
//  * A chunk's CTA writes an fp32 partial (o, m, l); the last CTA of a unit
//    to finish (atomic ticket, never a spin) merges them, folds in the new
//    token (scores it from registers rather than re-reading the cache),
//    performs the append and writes bf16 output and lse.
//  * Every block_table entry is range-checked before an address is formed.
#include <math.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kWarps = 4;                      // consumer warps
constexpr int kThreads = (kWarps + 1) * 32;    // + one producer warp
constexpr int kConsumerThreads = kWarps * 32;
constexpr int kTile = kDecodeTile;             // tokens per pipeline tile
constexpr int kTokPerWarp = kTile / kWarps;    // 8 tokens per warp per tile
constexpr int kSteps = kTokPerWarp / 4;        // 4 tokens (one per 8-lane group) per step
constexpr int kTargetItemsMax = 2048;
constexpr int kBarConsumers = 1;               // named barrier id for consumer warps
constexpr float kNegInf = -INFINITY;

enum RowStatus { ROW_OK = 0, ROW_INACTIVE = 1, ROW_OVERFLOW = 2 };

struct KParams {
    const int32_t *block_table;
    const int32_t *seqlens;
    const __nv_bfloat16 *q;
    const __nv_bfloat16 *k_new;
    const __nv_bfloat16 *v_new;
    __nv_bfloat16 *k_cache;
    __nv_bfloat16 *v_cache;
    __nv_bfloat16 *out;
    float *lse;
    int32_t *tickets;
    float2 *part_ml;
    float *part_o;
    int32_t *err_flag;
    int batch, num_q_heads, num_kv_heads, group, n_sub, units, max_blocks;
    int page_size, page_shift, num_pages, layout, box_tokens;
    int target_items, chunk_max, with_new;
    float q_scale;
};

template <int D>
constexpr int stages_for()
{
    return D == 256 ? 3 : (D == 128 ? 4 : 6);
}

template <int D, int GC>
struct Smem {
    static constexpr int kStages = stages_for<D>();
    __nv_bfloat16 kv[kStages][2][kTile * D]; // [stage][K|V][token][dim]
    float red_o[kWarps][GC][D];
    float fin_o[GC][D];
    float red_m[kWarps][GC], red_l[kWarps][GC];
    float fin_m[GC], fin_l[GC], s_new[GC];
    uint64_t full[kStages], empty[kStages];
    int32_t stage_bad[kStages];
    int32_t len[kMaxDecodeBatch];
    int32_t prefix[kMaxDecodeBatch + 1];
    int32_t pages[kDecodeChunkMaxPages];
    int32_t chunk;
    int32_t flag;
    int32_t bad;
    int32_t abort;
    int32_t stop;
};

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ int row_status(const KParams &p, int L)
{
    if (L < 0)
        return ROW_INACTIVE;
    if ((int64_t)L + p.with_new > (int64_t)p.max_blocks * p.page_size)
        return ROW_OVERFLOW;
    return ROW_OK;
}

__device__ __forceinline__ int row_chunks(const KParams &p, int L, int C)
{
    return (row_status(p, L) == ROW_OK && L > 0) ? (L + C - 1) / C : 1;
}

// Mbarrier wait that also gives up when another warp of the CTA aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, volatile int32_t *abort)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t start = globaltimer_ns();
    for (;;) {
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity))
                return true;
        if (*abort)
            return false;
        if (globaltimer_ns() - start > kWaitLimitNs) {
            *abort = 1;
            return false;
        }
    }
}

// Every CTA derives the same split plan from cache_seqlens: chunk size C and
// the first work item of every row (prefix[b]; prefix[batch] = item count).
template <int D, int GC>
__device__ void build_plan(const KParams &p, Smem<D, GC> &sm)
{
    for (int i = threadIdx.x; i < p.batch; i += kThreads)
        sm.len[i] = p.seqlens[i];
    __syncthreads();
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        long long work = 0;
        for (int i = lane; i < p.batch; i += 32) {
            const int L = sm.len[i];
            if (row_status(p, L) == ROW_OK)
                work += L;
        }
        for (int o = 16; o > 0; o >>= 1)
            work += __shfl_xor_sync(0xffffffffu, work, o);
        work *= p.units;
        long long c = (work + p.target_items - 1) / p.target_items;
        c = (c + kTile - 1) / kTile * kTile;
        if (c < kDecodeChunkMin)
            c = kDecodeChunkMin;
        if (c > p.chunk_max)
            c = p.chunk_max;
        const int C = (int)c;
        int run = 0;
        for (int base = 0; base < p.batch; base += 32) {
            const int i = base + lane;
            const int items = i < p.batch ? row_chunks(p, sm.len[i], C) * p.units : 0;
            int incl = items;
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o)
                    incl += v;
            }
            if (i < p.batch)
                sm.prefix[i] = run + incl - items;
            run += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) {
            sm.prefix[p.batch] = run;
            sm.chunk = C;
        }
    }
    __syncthreads();
}

struct Item {
    int b, unit, kvh, sub, chunk, nchunks, base, L, status, tok0, tok1;
};

template <int D, int GC>
__device__ __forceinline__ Item decode_item(const KParams &p, const Smem<D, GC> &sm, int it)
{
    int lo = 0, hi = p.batch - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (sm.prefix[mid] <= it)
            lo = mid;
        else
            hi = mid - 1;
    }
    Item I;
    I.b = lo;
    I.L = sm.len[lo];
    I.status = row_status(p, I.L);
    const int C = sm.chunk;
    I.nchunks = row_chunks(p, I.L, C);
    const int r = it - sm.prefix[lo];
    const int unit_in_row = r / I.nchunks;
    I.chunk = r - unit_in_row * I.nchunks;
    I.base = it - I.chunk;
    I.kvh = unit_in_row / p.n_sub;
    I.sub = unit_in_row - I.kvh * p.n_sub;
    I.unit = lo * p.units + unit_in_row;
    const int ncache = I.status == ROW_OK ? I.L : 0;
    I.tok0 = min(I.chunk * C, ncache);
    I.tok1 = min(I.tok0 + C, ncache);
    return I;
}

// ---------------------------------------------------------------- producer
template <int D, int GC>
__device__ void producer(const KParams &p, Smem<D, GC> &sm, const CUtensorMap *tm_k, const CUtensorMap *tm_v)
{
    constexpr int S = Smem<D, GC>::kStages;
    const int lane = threadIdx.x & 31;
    const int n_items = sm.prefix[p.batch];
    const uint64_t policy = l2_evict_first_policy();
    const int box = p.box_tokens;
    const uint32_t box_bytes = (uint32_t)box * D * 2u;
    uint32_t g_tile = 0;
    volatile int32_t *abort = &sm.abort;

    for (int it = blockIdx.x; it < n_items && !*abort; it += gridDim.x) {
        const Item I = decode_item(p, sm, it);
        if (I.tok1 <= I.tok0)
            continue;
        const int first_blk = I.tok0 >> p.page_shift;
        const int nblk = ((I.tok1 - 1) >> p.page_shift) - first_blk + 1;
        __syncwarp();
        const int32_t *bt_row = p.block_table + (int64_t)I.b * p.max_blocks;
        for (int i = lane; i < nblk; i += 32)
            sm.pages[i] = bt_row[first_blk + i];
        __syncwarp();
        const int n_tiles = (I.tok1 - I.tok0 + kTile - 1) / kTile;
        for (int t = 0; t < n_tiles; ++t, ++g_tile) {
            const int s = g_tile % S;
            const uint32_t use = g_tile / S;
            if (use > 0 && !wait_or_abort(&sm.empty[s], (use - 1) & 1u, abort))
                break;
            if (lane == 0) {
                const int tile0 = I.tok0 + t * kTile;
                const int nv = min(kTile, I.tok1 - tile0);
                const int nbox = (nv + box - 1) / box;
                int bad = 0;
                uint32_t bytes = 0;
                for (int bx = 0; bx < nbox; ++bx) {
                    const int page = sm.pages[((tile0 + bx * box) >> p.page_shift) - first_blk];
                    if (page < 1 || page >= p.num_pages)
                        bad = 1;
                    else
                        bytes += 2u * box_bytes;
                }
                sm.stage_bad[s] = bad;
                mbar_arrive_expect_tx(&sm.full[s], bytes);
                for (int bx = 0; bx < nbox; ++bx) {
                    const int tok = tile0 + bx * box;
                    const int page = sm.pages[(tok >> p.page_shift) - first_blk];
                    if (page < 1 || page >= p.num_pages)
                        continue;
                    const int slot = tok & (p.page_size - 1);
                    int y, z;
                    if (p.layout == PKV_NHD) {
                        y = I.kvh;
                        z = page * p.page_size + slot;
                    } else {
                        y = slot;
                        z = page * p.num_kv_heads + I.kvh;
                    }
                    __nv_bfloat16 *dst_k = sm.kv[s][0] + bx * box * D;
                    __nv_bfloat16 *dst_v = sm.kv[s][1] + bx * box * D;
                    tma_load_3d(dst_k, tm_k, 0, y, z, &sm.full[s], policy);
                    tma_load_3d(dst_v, tm_v, 0, y, z, &sm.full[s], policy);
                }
                if (bad)
                    set_error(p.err_flag, PKV_ERR_PAGE);
            }
            __syncwarp();
        }
    }
    // After an abort, let copies already issued land before the CTA exits.
    if (*abort && lane == 0) {
        const uint32_t first = g_tile > (uint32_t)S ? g_tile - S : 0;
        for (uint32_t g = first; g < g_tile; ++g)
            (void)mbar_wait(&sm.full[g % S], (g / S) & 1u);
    }
}

// ---------------------------------------------------------------- consumers
template <int D, int GC, bool MASKED>
__device__ __forceinline__ void consume_tile(const __nv_bfloat16 *Ks, const __nv_bfloat16 *Vs, int nv, int warp,
                                             int lane, const float2 (&qf)[GC][D / 64][4],
                                             float2 (&acc)[GC][D / 64][4], float (&m_run)[GC],
                                             float (&l_run)[GC])
{
    constexpr int VPL = D / 64;
    const int grp = lane >> 3, j = lane & 7;
#pragma unroll
    for (int step = 0; step < kSteps; ++step) {
        const int row = warp * kTokPerWarp + step * 4 + grp;
        const bool valid = !MASKED || row < nv;
        const uint4 *krow = reinterpret_cast<const uint4 *>(Ks + row * D);
        float s[GC];
        {
            float2 sacc[GC];
#pragma unroll
            for (int g = 0; g < GC; ++g)
                sacc[g] = make_float2(0.f, 0.f);
#pragma unroll
            for (int i = 0; i < VPL; ++i) {
                const uint4 kw = krow[j + 8 * i];
                const uint32_t w4[4] = {kw.x, kw.y, kw.z, kw.w};
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const float2 kf = bf16x2_to_float2(w4[w]);
#pragma unroll
                    for (int g = 0; g < GC; ++g)
                        sacc[g] = ffma2(qf[g][i][w], kf, sacc[g]);
                }
            }
#pragma unroll
            for (int g = 0; g < GC; ++g)
                s[g] = sacc[g].x + sacc[g].y;
        }
#pragma unroll
        for (int g = 0; g < GC; ++g) {
            s[g] += __shfl_xor_sync(0xffffffffu, s[g], 1);
            s[g] += __shfl_xor_sync(0xffffffffu, s[g], 2);
            s[g] += __shfl_xor_sync(0xffffffffu, s[g], 4);
            if (MASKED && !valid)
                s[g] = kNegInf;
        }
        bool grow = false;
        float m_new[GC];
#pragma unroll
        for (int g = 0; g < GC; ++g) {
            float mt = fmaxf(s[g], __shfl_xor_sync(0xffffffffu, s[g], 8));
            mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 16));
            m_new[g] = fmaxf(m_run[g], mt);
            grow |= m_new[g] > m_run[g];
        }
        if (grow) { // warp-uniform: m_run and m_new are identical in all lanes
#pragma unroll
            for (int g = 0; g < GC; ++g) {
                const float a = ex2(m_run[g] - m_new[g]); // m_run = -inf -> 0
                l_run[g] *= a;
                const float2 a2 = make_float2(a, a);
#pragma unroll
                for (int i = 0; i < VPL; ++i)
#pragma unroll
                    for (int w = 0; w < 4; ++w)
                        acc[g][i][w] = fmul2(acc[g][i][w], a2);
                m_run[g] = m_new[g];
            }
        }
        float pr[GC];
#pragma unroll
        for (int g = 0; g < GC; ++g) {
            pr[g] = valid ? ex2(s[g] - m_run[g]) : 0.f;
            l_run[g] += pr[g];
        }
        if (valid) {
            const uint4 *vrow = reinterpret_cast<const uint4 *>(Vs + row * D);
#pragma unroll
            for (int i = 0; i < VPL; ++i) {
                const uint4 vw = vrow[j + 8 * i];
                const uint32_t w4[4] = {vw.x, vw.y, vw.z, vw.w};
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const float2 vf = bf16x2_to_float2(w4[w]);
#pragma unroll
                    for (int g = 0; g < GC; ++g)
                        acc[g][i][w] = ffma2(make_float2(pr[g], pr[g]), vf, acc[g][i][w]);
                }
            }
        }
    }
}

// Merges the split-KV partials of one unit (written by its nchunks CTAs)
// into fin_*; returns nonzero if any chunk met a bad page.
template <int D, int GC>
__device__ int combine_partials(const KParams &p, Smem<D, GC> &sm, const Item &I)
{
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const float2 *ml = p.part_ml + (int64_t)I.base * GC;
    if (tid == 0)
        sm.bad = 0;
    named_sync(kBarConsumers, kConsumerThreads);
    for (int g = warp; g < GC; g += kWarps) {
        float M = kNegInf;
        int bad = 0;
        for (int i = lane; i < I.nchunks; i += 32) {
            const float2 v = __ldcg(ml + (int64_t)i * GC + g);
            M = fmaxf(M, v.x);
            bad |= v.y < 0.f;
        }
        for (int o = 16; o > 0; o >>= 1)
            M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        bad = __any_sync(0xffffffffu, bad);
        float l = 0.f;
        for (int i = lane; i < I.nchunks; i += 32) {
            const float2 v = __ldcg(ml + (int64_t)i * GC + g);
            l += v.x == kNegInf ? 0.f : ex2(v.x - M) * v.y;
        }
        for (int o = 16; o > 0; o >>= 1)
            l += __shfl_xor_sync(0xffffffffu, l, o);
        if (lane == 0) {
            sm.fin_m[g] = M;
            sm.fin_l[g] = l;
            if (bad)
                sm.bad = 1;
        }
    }
    named_sync(kBarConsumers, kConsumerThreads);
    const float *po = p.part_o + (int64_t)I.base * GC * D;
    for (int e = tid; e < GC * D; e += kConsumerThreads) {
        const int g = e / D;
        const float M = sm.fin_m[g];
        float o = 0.f;
        for (int i = 0; i < I.nchunks; ++i) {
            const float m = __ldcg(&ml[(int64_t)i * GC + g].x);
            if (m != kNegInf)
                o += ex2(m - M) * __ldcg(po + (int64_t)i * GC * D + e);
        }
        (&sm.fin_o[0][0])[e] = o;
    }
    named_sync(kBarConsumers, kConsumerThreads);
    return sm.bad;
}

// Writes the unit's output: zeros for inactive / failed rows, otherwise
// merges the new token (when given), performs the append and normalises.
template <int D, int GC>
__device__ void finalize(const KParams &p, Smem<D, GC> &sm, const Item &I, int bad)
{
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h0 = I.kvh * p.group + I.sub * GC;
    int err = 0;
    if (I.status == ROW_OVERFLOW)
        err = PKV_ERR_OVERFLOW;
    else if (I.status == ROW_OK && bad)
        err = PKV_ERR_PAGE;
    int64_t dst = -1; // element offset of the appended token for this kv head
    if (I.status == ROW_OK && !err && p.with_new) {
        const int page = p.block_table[(int64_t)I.b * p.max_blocks + (I.L >> p.page_shift)];
        if (page < 1 || page >= p.num_pages) {
            err = PKV_ERR_PAGE;
        } else {
            const int slot = I.L & (p.page_size - 1);
            dst = p.layout == PKV_NHD
                      ? (((int64_t)page * p.page_size + slot) * p.num_kv_heads + I.kvh) * D
                      : (((int64_t)page * p.num_kv_heads + I.kvh) * p.page_size + slot) * D;
        }
    }
    const bool live = I.status == ROW_OK && !err;
    if (tid == 0 && err)
        set_error(p.err_flag, err);

    const __nv_bfloat16 *kn = p.k_new + ((int64_t)I.b * p.num_kv_heads + I.kvh) * D;
    const __nv_bfloat16 *vn = p.v_new + ((int64_t)I.b * p.num_kv_heads + I.kvh) * D;
    if (live && p.with_new) {
        // score of the new token for each head: (q * scale * log2 e) . k_new
        for (int g = warp; g < GC; g += kWarps) {
            const __nv_bfloat16 *qh = p.q + ((int64_t)I.b * p.num_q_heads + h0 + g) * D;
            float s = 0.f;
            for (int d = lane; d < D; d += 32)
                s = fmaf(__bfloat162float(qh[d]) * p.q_scale, __bfloat162float(kn[d]), s);
            for (int o = 16; o > 0; o >>= 1)
                s += __shfl_xor_sync(0xffffffffu, s, o);
            if (lane == 0)
                sm.s_new[g] = s;
        }
        named_sync(kBarConsumers, kConsumerThreads);
        if (I.sub == 0) { // the append: one bit copy per kv head
            constexpr int kVec = D / 8;
            for (int c = tid; c < 2 * kVec; c += kConsumerThreads) {
                const bool is_v = c >= kVec;
                const int v = is_v ? c - kVec : c;
                const uint4 val = reinterpret_cast<const uint4 *>(is_v ? vn : kn)[v];
                reinterpret_cast<uint4 *>((is_v ? p.v_cache : p.k_cache) + dst)[v] = val;
            }
        }
    }
    for (int e = tid; e < GC * D; e += kConsumerThreads) {
        const int g = e / D, d = e - g * D;
        const int64_t oidx = ((int64_t)I.b * p.num_q_heads + h0 + g) * D + d;
        float o = 0.f, M = kNegInf, l = 0.f;
        if (live) {
            o = sm.fin_o[g][d];
            M = sm.fin_m[g];
            l = sm.fin_l[g];
            if (p.with_new) {
                const float sn = sm.s_new[g];
                const float Mn = fmaxf(M, sn);
                const float a = ex2(M - Mn); // M = -inf (no cached key) -> 0
                const float c = ex2(sn - Mn);
                o = fmaf(o, a, c * __bfloat162float(vn[d]));
                l = fmaf(l, a, c);
                M = Mn;
            }
        }
        const bool any = l > 0.f;
        p.out[oidx] = __float2bfloat16_rn(any ? o / l : 0.f);
        if (p.lse != nullptr && d == 0)
            p.lse[(int64_t)I.b * p.num_q_heads + h0 + g] = any ? (M + log2f(l)) * 0.69314718055994531f : kNegInf;
    }
}

template <int D, int GC>
__device__ void consumers(const KParams &p, Smem<D, GC> &sm)
{
    constexpr int S = Smem<D, GC>::kStages;
    constexpr int VPL = D / 64;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int j = lane & 7;
    const int n_items = sm.prefix[p.batch];
    volatile int32_t *abort = &sm.abort;
    uint32_t g_tile = 0;

    for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
        const Item I = decode_item(p, sm, it);
        const int h0 = I.kvh * p.group + I.sub * GC;
        float2 qf[GC][VPL][4];
        float2 acc[GC][VPL][4];
        float m_run[GC], l_run[GC];
#pragma unroll
        for (int g = 0; g < GC; ++g) {
            const uint4 *qrow = reinterpret_cast<const uint4 *>(p.q + ((int64_t)I.b * p.num_q_heads + h0 + g) * D);
#pragma unroll
            for (int i = 0; i < VPL; ++i) {
                const uint4 qw = __ldg(qrow + j + 8 * i);
                const uint32_t w4[4] = {qw.x, qw.y, qw.z, qw.w};
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const float2 f = bf16x2_to_float2(w4[w]);
                    qf[g][i][w] = make_float2(f.x * p.q_scale, f.y * p.q_scale);
                    acc[g][i][w] = make_float2(0.f, 0.f);
                }
            }
            m_run[g] = kNegInf;
            l_run[g] = 0.f;
        }
        int bad = 0;
        const int n_tiles = (I.tok1 - I.tok0 + kTile - 1) / kTile;
        for (int t = 0; t < n_tiles; ++t, ++g_tile) {
            const int s = g_tile % S;
            if (!wait_or_abort(&sm.full[s], (g_tile / S) & 1u, abort))
                break;
            bad |= ((volatile int32_t *)sm.stage_bad)[s];
            const int nv = min(kTile, I.tok1 - (I.tok0 + t * kTile));
            if (nv == kTile)
                consume_tile<D, GC, false>(sm.kv[s][0], sm.kv[s][1], nv, warp, lane, qf, acc, m_run, l_run);
            else
                consume_tile<D, GC, true>(sm.kv[s][0], sm.kv[s][1], nv, warp, lane, qf, acc, m_run, l_run);
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&sm.empty[s]);
        }
        // warp: sum the four 8-lane groups (they share m_run)
#pragma unroll
        for (int g = 0; g < GC; ++g) {
#pragma unroll
            for (int i = 0; i < VPL; ++i)
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    float2 v = acc[g][i][w];
                    v.x += __shfl_xor_sync(0xffffffffu, v.x, 8);
                    v.y += __shfl_xor_sync(0xffffffffu, v.y, 8);
                    v.x += __shfl_xor_sync(0xffffffffu, v.x, 16);
                    v.y += __shfl_xor_sync(0xffffffffu, v.y, 16);
                    acc[g][i][w] = v;
                }
            l_run[g] += __shfl_xor_sync(0xffffffffu, l_run[g], 8);
            l_run[g] += __shfl_xor_sync(0xffffffffu, l_run[g], 16);
        }
        if (lane < 8) {
#pragma unroll
            for (int g = 0; g < GC; ++g) {
#pragma unroll
                for (int i = 0; i < VPL; ++i)
#pragma unroll
                    for (int w = 0; w < 4; ++w)
                        *reinterpret_cast<float2 *>(&sm.red_o[warp][g][8 * (j + 8 * i) + 2 * w]) = acc[g][i][w];
                if (lane == 0) {
                    sm.red_m[warp][g] = m_run[g];
                    sm.red_l[warp][g] = l_run[g];
                }
            }
        }
        named_sync(kBarConsumers, kConsumerThreads);
        // CTA: merge the warps' partial softmax states
        for (int e = tid; e < GC * D; e += kConsumerThreads) {
            const int g = e / D, d = e - g * D;
            float M = kNegInf;
#pragma unroll
            for (int w = 0; w < kWarps; ++w)
                M = fmaxf(M, sm.red_m[w][g]);
            float o = 0.f, l = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float m = sm.red_m[w][g];
                const float a = m == kNegInf ? 0.f : ex2(m - M);
                o = fmaf(a, sm.red_o[w][g][d], o);
                l = fmaf(a, sm.red_l[w][g], l);
            }
            sm.fin_o[g][d] = o;
            if (d == 0) {
                sm.fin_m[g] = M;
                sm.fin_l[g] = l;
            }
        }
        // One thread decides whether the CTA stopped, so that every consumer
        // thread takes the same path through the barriers below.
        if (tid == 0)
            sm.stop = *abort;
        named_sync(kBarConsumers, kConsumerThreads);
        const bool aborted = sm.stop != 0;
        if (!aborted) {
            if (I.nchunks == 1) {
                finalize(p, sm, I, bad);
            } else {
                float *po = p.part_o + (int64_t)it * GC * D;
                for (int e = tid; e < GC * D; e += kConsumerThreads)
                    po[e] = (&sm.fin_o[0][0])[e];
                if (tid < GC)
                    p.part_ml[(int64_t)it * GC + tid] = make_float2(sm.fin_m[tid], bad ? -1.f : sm.fin_l[tid]);
                __threadfence();
                named_sync(kBarConsumers, kConsumerThreads);
                if (tid == 0)
                    sm.flag = atomicAdd(&p.tickets[I.unit], 1) == I.nchunks - 1;
                named_sync(kBarConsumers, kConsumerThreads);
                if (sm.flag) {
                    __threadfence();
                    const int any_bad = combine_partials(p, sm, I);
                    finalize(p, sm, I, any_bad);
                    if (tid == 0)
                        p.tickets[I.unit] = 0; // ready for the next call
                }
            }
        }
        named_sync(kBarConsumers, kConsumerThreads);
        if (aborted)
            break;
    }
    if (*abort && tid == 0)
        set_error(p.err_flag, PKV_ERR_TIMEOUT);
}

template <int D, int GC>
__global__ void __maxnreg__(200) decode_kernel(const __grid_constant__ KParams p,
                                                          const __grid_constant__ CUtensorMap tm_k,
                                                          const __grid_constant__ CUtensorMap tm_v)
{
    extern __shared__ unsigned char smem_raw[];
    Smem<D, GC> &sm = *reinterpret_cast<Smem<D, GC> *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    constexpr int S = Smem<D, GC>::kStages;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], kWarps);
        }
        sm.abort = 0;
        mbar_init_fence();
    }
    if (threadIdx.x == kWarps * 32) {
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
    }
    build_plan(p, sm); // ends with __syncthreads()
    if (threadIdx.x >= kWarps * 32)
        producer(p, sm, &tm_k, &tm_v);
    else
        consumers(p, sm);
}

template <int D, int GC>
size_t smem_bytes()
{
    return sizeof(Smem<D, GC>) + 128;
}

struct KernelEntry {
    int D, GC;
    const void *fn;
    size_t smem;
};

template <int D, int GC>
KernelEntry entry()
{
    return KernelEntry{D, GC, reinterpret_cast<const void *>(&decode_kernel<D, GC>), smem_bytes<D, GC>()};
}

const KernelEntry kTable[] = {
    entry<64, 1>(),  entry<64, 2>(),  entry<64, 4>(),  entry<64, 8>(),  entry<128, 1>(),
        entry<128, 2>(), entry<128, 4>(), entry<256, 1>(), entry<256, 2>(),
};

const KernelEntry *find_kernel(int D, int GC)
{
    for (const KernelEntry &e : kTable)
        if (e.D == D && e.GC == GC)
            return &e;
    return nullptr;
}

int kernel_index(const KernelEntry *e)
{
    return static_cast<int>(e - kTable);
}

int heads_per_cta(int group, int D)
{
    int gc = 1;
    while (gc * 2 <= group && group % (gc * 2) == 0 && gc * 2 * D <= 512)
        gc *= 2;
    return gc;
}

} // namespace

bool decode_shape(int batch, int max_blocks, int num_q_heads, const pkv_cache_desc &d, DecodeShape *s)
{
    if (d.num_kv_heads <= 0 || num_q_heads % d.num_kv_heads != 0)
        return false;
    s->group = num_q_heads / d.num_kv_heads;
    if (s->group & (s->group - 1))
        return false; // power-of-two groups only
    s->heads_per_cta = heads_per_cta(s->group, d.head_dim);
    if (find_kernel(d.head_dim, s->heads_per_cta) == nullptr)
        return false;
    s->n_sub = s->group / s->heads_per_cta;
    s->units_per_row = d.num_kv_heads * s->n_sub;
    int cmax = kDecodeChunkMaxPages * d.page_size;
    if (cmax > 8192)
        cmax = 8192;
    if (cmax < kDecodeChunkMin)
        cmax = kDecodeChunkMin;
    s->chunk_max = cmax / kDecodeTile * kDecodeTile;
    const int64_t units = (int64_t)batch * s->units_per_row;
    const int64_t max_tokens = (int64_t)max_blocks * d.page_size;
    int64_t per_unit = (max_tokens + s->chunk_max - 1) / s->chunk_max;
    if (per_unit < 1)
        per_unit = 1;
    // The launch aims for at most kTargetItemsMax items when the chunk size is
    // not capped (then items <= target + units); a capped chunk bounds the
    // items of a unit by per_unit.  The layout does not depend on the device.
    int64_t cap = kTargetItemsMax + units;
    if (units * per_unit > cap)
        cap = units * per_unit;
    s->cap_items = cap;
    auto align = [](size_t x) { return (x + 255) & ~size_t(255); };
    const size_t tickets = align(sizeof(int32_t) * (size_t)units);
    s->off_ml = tickets;
    s->off_o = s->off_ml + align(sizeof(float2) * (size_t)cap * s->heads_per_cta);
    s->bytes = s->off_o + align(sizeof(float) * (size_t)cap * s->heads_per_cta * d.head_dim);
    return true;
}

int decode_target_items(int device, int head_dim, int heads_per_cta)
{
    // Per device and kernel: opt in to the kernel's shared memory once and
    // size the plan for two items per resident CTA slot.
    constexpr int kDevices = 64, kKernels = 16;
    static int cache[kDevices][kKernels] = {};
    const KernelEntry *e = find_kernel(head_dim, heads_per_cta);
    if (e == nullptr || device < 0 || device >= kDevices)
        return kTargetItemsMax;
    int &slot = cache[device][kernel_index(e)];
    if (slot == 0) {
        int occ = 1;
        if (cudaFuncSetAttribute(e->fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)e->smem) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, e->fn, kThreads, e->smem) != cudaSuccess || occ < 1)
            occ = 1;
        const int t = 2 * sm_count(device) * occ;
        slot = t > kTargetItemsMax ? kTargetItemsMax : t;
    }
    return slot;
}

cudaError_t launch_decode(const DecodeArgs &a, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                          cudaStream_t stream)
{
    const KernelEntry *e = find_kernel(a.desc.head_dim, a.shape.heads_per_cta);
    if (e == nullptr)
        return cudaErrorInvalidValue;
    KParams p;
    p.block_table = a.block_table;
    p.seqlens = a.cache_seqlens;
    p.q = static_cast<const __nv_bfloat16 *>(a.q);
    p.k_new = static_cast<const __nv_bfloat16 *>(a.k_new);
    p.v_new = static_cast<const __nv_bfloat16 *>(a.v_new);
    p.k_cache = static_cast<__nv_bfloat16 *>(a.k_cache);
    p.v_cache = static_cast<__nv_bfloat16 *>(a.v_cache);
    p.out = static_cast<__nv_bfloat16 *>(a.out);
    p.lse = a.lse;
    unsigned char *ws = static_cast<unsigned char *>(a.workspace);
    p.tickets = reinterpret_cast<int32_t *>(ws);
    p.part_ml = reinterpret_cast<float2 *>(ws + a.shape.off_ml);
    p.part_o = reinterpret_cast<float *>(ws + a.shape.off_o);
    p.err_flag = a.err_flag;
    p.batch = a.batch;
    p.num_q_heads = a.num_q_heads;
    p.num_kv_heads = a.desc.num_kv_heads;
    p.group = a.shape.group;
    p.n_sub = a.shape.n_sub;
    p.units = a.shape.units_per_row;
    p.max_blocks = a.max_blocks;
    p.page_size = a.desc.page_size;
    p.page_shift = a.page_shift;
    p.num_pages = a.desc.num_pages;
    p.layout = a.desc.layout;
    p.box_tokens = a.desc.page_size < kDecodeTile ? a.desc.page_size : kDecodeTile;
    p.target_items = a.target_items;
    p.chunk_max = a.shape.chunk_max;
    p.with_new = (a.k_new != nullptr) ? 1 : 0;
    p.q_scale = a.q_scale;
    void *args[] = {&p, const_cast<CUtensorMap *>(&tm_k), const_cast<CUtensorMap *>(&tm_v)};
    return cudaLaunchKernel(e->fn, dim3(a.grid), dim3(kThreads), args, e->smem, stream);
}

} // namespace pkv
