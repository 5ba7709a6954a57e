// pkv_prefill.cu -- ragged end-aligned causal prefill attention over a paged
// KV cache on the 5th-generation tensor cores (tcgen05, TMEM accumulators).
//
// What it computes.  Source: "[flashinfer] H100 D256 paged attention cuDNN
// auto-dispatch", code analysis part 1: request b has q_b query tokens and
// kv_b cached keys (q_b <= kv_b) in a paged cache (the HND layout there), and
// its query i (0-based) attends keys 0 .. kv_b - q_b + i: the causal mask is
// aligned to the end of the sequence.  Query head h reads kv head
// h / (Hq / Hkv); softmax scale, output rounding and the error rules are
// those of include/pkv.h.
//
// How (one persistent CTA per SM):
//  - Work unit = (request, kv head, tile of 128/G queries).  The G query
//    heads sharing a kv head times 128/G consecutive queries form the M = 128
//    rows of every MMA (row r = query r/G, head r%G), so every K/V tile read
//    from the pages serves all G heads.
//  - A one-CTA plan kernel validates every request, lists the query tiles and
//    orders them by their number of 64-token kv tiles, longest first; the
//    persistent CTAs take units in that order, snaking over the grid.
//  - Warp roles: warp 0 loads Q once per unit and the unit's K and V tiles,
//    64 tokens x head_dim each, with TMA into a ring of shared-memory stages
//    (in the order the MMAs consume them); warp 1 owns TMEM and one of its
//    threads issues the MMAs; warps 2-5 (one per TMEM lane quarter) run the
//    online softmax and the epilogue, one row per thread.
//  - TMEM: the O [128 x D] fp32 accumulator at columns 0..D-1 and two
//    S [128 x 64] fp32 buffers after it, so S of tile j+1 is computed while
//    the softmax of tile j runs.
//  - S = Q K^T (K-major Q and K); the softmax writes P into shared memory in
//    the K-major swizzled layout as two bf16 parts, p = hi + lo (about 16
//    significant bits: a single bf16 P alone, 8 bits, leaves errors near
//    2^-9 of the row's scale, well above 1e-2 of the small outputs that
//    cancellation produces); O += P_hi V + P_lo V with V as an MN-major
//    operand (its rows are tokens, its columns head_dim).
//  - Online softmax in base 2 on scores scaled by softmax_scale * log2(e).
//    A row's O and running sum are rescaled only when its maximum grows by
//    more than 8: until then the exponentials use the older maximum, which is
//    exact in real arithmetic and keeps every p below 2^8.
#include <cuda_bf16.h>
#include <math.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"
#include "pkv_tcgen05.cuh"

namespace pkv {
namespace {

constexpr int kPfThreads = 192;
constexpr int kPfProducerWarp = 0;
constexpr int kPfMmaWarp = 1;
constexpr int kPfRows = 128;    // M of every MMA
constexpr int kPfTile = 64;     // kv tokens per tile
constexpr int kPfBuckets = 4096; // plan: units are ordered by min(kv tiles, 4095)
constexpr int kPlanThreads = 1024;
constexpr float kRescaleLog2 = 8.0f;
constexpr float kLn2 = 0.693147180559945309f;

template <int D> struct PfCfg {
    static constexpr int kChunks = D / 64;                     // 128-byte column blocks of a row
    static constexpr int kStages = D == 256 ? 3 : 6;           // K / V tiles in flight
    static constexpr uint32_t kQBytes = kPfRows * D * 2;       // [chunk][128 rows][128 B]
    static constexpr uint32_t kStageBytes = kPfTile * D * 2;   // [chunk][64 tokens][128 B]
    static constexpr uint32_t kPHalf = kPfRows * kPfTile * 2;  // [128 rows][128 B]
    static constexpr uint32_t kPBytes = 2 * kPHalf;            // P = hi + lo halves
    static constexpr uint32_t kOffQ = 0;
    static constexpr uint32_t kOffStage = kQBytes;
    static constexpr uint32_t kOffP = kOffStage + kStages * kStageBytes;
    static constexpr uint32_t kOffBar = kOffP + 2 * kPBytes;
    static constexpr uint32_t kSmem = kOffBar + 256 + 1024; // + barriers + alignment slack
    static constexpr uint32_t kTmemCols = D == 256 ? 512 : 256;
    static constexpr uint32_t kColO = 0;
    static constexpr uint32_t kColS = D;
};
static_assert(PfCfg<256>::kSmem <= 232448, "prefill shared memory over the per-CTA limit");

struct PfBars {
    uint64_t q_full, q_empty;
    uint64_t full[6], empty[6];
    uint64_t s_full[2], p_full[2], o_done[2];
    uint64_t o_free;
    uint64_t drain;
    uint32_t tmem_base;
    int32_t abort;
};
static_assert(sizeof(PfBars) <= 256, "barrier block");

// One query tile of one request (all kv heads share it).
struct PfUnit {
    int32_t b, t, q_start, q_len, kv_len, n_tiles, pad0, pad1;
};
static_assert(sizeof(PfUnit) == 32, "unit record");

struct PfParams {
    const int32_t *block_table;
    const PfUnit *units;
    const int32_t *n_pairs;
    __nv_bfloat16 *out;
    float *lse;
    int32_t *err_flag;
    int max_blocks, num_q_heads, num_kv_heads;
    int group_shift, q_tile, page_shift, box_shift, layout;
    float q_scale;
};

struct PfMapsDev {
    CUtensorMap q, k, v;
};

struct PfPlanParams {
    const int32_t *qo_indptr;
    const int32_t *kv_lens;
    const int32_t *block_table;
    PfUnit *units;
    int32_t *n_pairs;
    __nv_bfloat16 *out;
    float *lse;
    int32_t *err_flag;
    int batch, max_blocks, num_pages, page_shift, total_q, q_tile, num_q_heads, head_dim;
    int64_t cap_pairs;
};

// kv tiles a query tile needs: its last query sees kv - q + min(qt(t+1), q) keys.
__host__ __device__ inline int64_t pf_tiles(int64_t kv, int64_t q, int64_t t, int64_t qt)
{
    const int64_t last = (qt * (t + 1) < q ? qt * (t + 1) : q);
    return (kv - q + last + kPfTile - 1) / kPfTile;
}

// Position in the consumption order (K0, K1, V0, K2, V1, ..., V_{nt-1}) of a
// unit's K and V tiles; the producer loads them in this order.
__device__ __forceinline__ int pf_item_k(int j)
{
    return j == 0 ? 0 : 2 * j - 1;
}
__device__ __forceinline__ int pf_item_v(int j, int nt)
{
    return j == nt - 1 ? 2 * nt - 1 : 2 * j + 2;
}

// k-th unit of this CTA: rounds of gridDim.x units, alternating direction.
__device__ __forceinline__ int pf_unit_at(int k)
{
    const int g = (int)gridDim.x, c = (int)blockIdx.x;
    return k * g + ((k & 1) ? g - 1 - c : c);
}

// Bounded barrier wait that also gives up when another role has aborted.
__device__ __noinline__ bool pf_wait(uint64_t *bar, uint32_t parity, PfBars &bars, int32_t *err_flag)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t start = globaltimer_ns();
    volatile int32_t *abort = &bars.abort;
    for (;;) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity))
                return true;
        if (*abort != 0)
            return false;
        if (globaltimer_ns() - start > kWaitLimitNs) {
            *abort = 1;
            set_error(err_flag, PKV_ERR_TIMEOUT);
            return false;
        }
    }
}

// pf_wait for a whole warp: every lane gets the same answer, so warp-collective
// instructions after it are reached by all lanes or none.
__device__ __forceinline__ bool pf_wait_all(uint64_t *bar, uint32_t parity, PfBars &bars, int32_t *err_flag)
{
    const bool ok = pf_wait(bar, parity, bars, err_flag);
    return __all_sync(0xffffffffu, ok);
}

// ---------------------------------------------------------------- producer

template <int D>
__device__ void pf_producer(const PfParams &p, const PfMapsDev &maps, uint8_t *smem, PfBars &bars, int n_units,
                            int lane)
{
    using C = PfCfg<D>;
    const int Hkv = p.num_kv_heads;
    const int G = 1 << p.group_shift;
    const int P = 1 << p.page_shift;
    const int BT = 1 << p.box_shift;             // tokens per box: min(page_size, 64)
    const int boxes = kPfTile >> p.box_shift;     // boxes per full tile
    const uint32_t box_bytes = (uint32_t)BT * 128u;
    int ib = 0, issued = 0;
    uint32_t uc = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
        const int u = pf_unit_at(k);
        if (u >= n_units)
            break;
        const int pair = u / Hkv, g = u - pair * Hkv;
        const PfUnit un = p.units[pair];
        const int32_t *bt_row = p.block_table + (int64_t)un.b * p.max_blocks;
        const int nt = un.n_tiles, kv = un.kv_len;

        if (uc > 0 && !pf_wait_all(&bars.q_empty, (uc - 1) & 1, bars, p.err_flag))
            break;
        if (lane == 0) {
            mbar_arrive_expect_tx(&bars.q_full, C::kQBytes);
            const int z = un.q_start + un.t * p.q_tile;
            for (int c = 0; c < C::kChunks; ++c)
                tma_load_3d_plain(smem + C::kOffQ + c * (kPfRows * 128), &maps.q, 64 * c, g * G, z, &bars.q_full);
        }
        // Lane i holds the page of box i of a tile (boxes <= 8 <= 32 lanes).
        auto page_ids = [&](int j) {
            const int tok = j * kPfTile + lane * BT;
            int id = 0;
            if (lane < boxes && j < nt && tok < kv)
                id = __ldg(bt_row + (tok >> p.page_shift));
            return id;
        };
        int ids_prev = 0, ids_cur = page_ids(0), ids_next = page_ids(1);
        for (int j = 0; j <= nt && ok; ++j) {
            for (int kind = 0; kind < 2; ++kind) { // K_j, then V_{j-1}
                const int jj = kind == 0 ? j : j - 1;
                if (kind == 0 ? (j >= nt) : (j < 1))
                    continue;
                const int itg = ib + (kind == 0 ? pf_item_k(jj) : pf_item_v(jj, nt));
                const int stage = itg % C::kStages;
                const int n = itg / C::kStages;
                if (n > 0 && !pf_wait_all(&bars.empty[stage], (n - 1) & 1, bars, p.err_flag)) {
                    ok = false;
                    break;
                }
                const int tok0 = jj * kPfTile;
                const int ntok = min(kPfTile, kv - tok0);
                const int nbox = (ntok + BT - 1) >> p.box_shift;
                uint8_t *dst = smem + C::kOffStage + stage * C::kStageBytes;
                const CUtensorMap *map = kind == 0 ? &maps.k : &maps.v;
                const int ids = kind == 0 ? ids_cur : ids_prev;
                if (lane == 0)
                    mbar_arrive_expect_tx(&bars.full[stage], (uint32_t)nbox * C::kChunks * box_bytes);
                for (int bx = 0; bx < nbox; ++bx) {
                    const int page = __shfl_sync(0xffffffffu, ids, bx);
                    if (lane == 0) {
                        const int slot = (tok0 + bx * BT) & (P - 1);
                        int y, z;
                        if (p.layout == PKV_NHD) {
                            y = g;
                            z = page * P + slot;
                        } else {
                            y = slot;
                            z = page * Hkv + g;
                        }
                        for (int c = 0; c < C::kChunks; ++c)
                            tma_load_3d_plain(dst + c * (kPfTile * 128) + bx * box_bytes, map, 64 * c, y, z,
                                              &bars.full[stage]);
                    }
                }
                issued = itg + 1;
            }
            ids_prev = ids_cur;
            ids_cur = ids_next;
            ids_next = page_ids(j + 2);
        }
        ib += 2 * nt;
        ++uc;
    }
    // Own copies still in flight (none unless a wait above gave up).
    for (int itg = issued > C::kStages ? issued - C::kStages : 0; itg < issued; ++itg)
        mbar_wait(&bars.full[itg % C::kStages], (itg / C::kStages) & 1);
}

// ---------------------------------------------------------------- MMA issuer

template <int D>
__device__ void pf_mma(const PfParams &p, uint8_t *smem, PfBars &bars, uint32_t tmem, int n_units)
{
    using C = PfCfg<D>;
    constexpr uint32_t kIdescS = tc_idesc_bf16(kPfRows, kPfTile, false, false);
    constexpr uint32_t kIdescO = tc_idesc_bf16(kPfRows, D, false, true);
    const uint32_t q_base = smem_addr(smem + C::kOffQ);
    const uint32_t st_base = smem_addr(smem + C::kOffStage);
    const uint32_t p_base = smem_addr(smem + C::kOffP);
    int ib = 0, gt0 = 0;
    uint32_t uc = 0;
    bool issued = false;
    for (int k = 0;; ++k) {
        const int u = pf_unit_at(k);
        if (u >= n_units)
            break;
        const int nt = p.units[u / p.num_kv_heads].n_tiles;
        if (!pf_wait(&bars.q_full, uc & 1, bars, p.err_flag))
            goto done;
        for (int j = 0; j <= nt; ++j) {
            if (j < nt) { // S[j & 1] = Q K_j^T
                const int gt = gt0 + j;
                const int itg = ib + pf_item_k(j);
                const int stage = itg % C::kStages;
                if (!pf_wait(&bars.full[stage], (itg / C::kStages) & 1, bars, p.err_flag))
                    goto done;
                tc_fence_after();
                issued = true;
                const uint32_t d = tmem + C::kColS + (uint32_t)(gt & 1) * kPfTile;
                const uint32_t kb = st_base + stage * C::kStageBytes;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t a = tc_sw128_desc(q_base + (kk >> 2) * (kPfRows * 128) + (kk & 3) * 32, 16, 1024);
                    const uint64_t b = tc_sw128_desc(kb + (kk >> 2) * (kPfTile * 128) + (kk & 3) * 32, 16, 1024);
                    tc_mma_bf16(d, a, b, kIdescS, kk > 0 ? 1u : 0u);
                }
                tc_commit(&bars.s_full[gt & 1]);
                tc_commit(&bars.empty[stage]);
                if (j == nt - 1)
                    tc_commit(&bars.q_empty);
            }
            if (j >= 1) { // O += P_{j-1} V_{j-1}
                const int jv = j - 1, gt = gt0 + jv;
                if (!pf_wait(&bars.p_full[gt & 1], (gt >> 1) & 1, bars, p.err_flag))
                    goto done;
                if (jv == 0 && uc > 0 && !pf_wait(&bars.o_free, (uc - 1) & 1, bars, p.err_flag))
                    goto done;
                const int itg = ib + pf_item_v(jv, nt);
                const int stage = itg % C::kStages;
                if (!pf_wait(&bars.full[stage], (itg / C::kStages) & 1, bars, p.err_flag))
                    goto done;
                tc_fence_after();
                const uint32_t vb = st_base + stage * C::kStageBytes;
                const uint32_t pb = p_base + (uint32_t)(gt & 1) * C::kPBytes;
#pragma unroll
                for (int kk = 0; kk < 2 * (kPfTile / 16); ++kk) { // hi part, then lo part
                    const int k4 = kk & (kPfTile / 16 - 1);
                    const uint64_t a = tc_sw128_desc(pb + (kk >> 2) * C::kPHalf + k4 * 32, 16, 1024);
                    const uint64_t b = tc_sw128_desc(vb + k4 * (16 * 128), kPfTile * 128, 1024);
                    tc_mma_bf16(tmem + C::kColO, a, b, kIdescO, (jv > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit(&bars.o_done[gt & 1]);
                tc_commit(&bars.empty[stage]);
            }
        }
        gt0 += nt;
        ib += 2 * nt;
        ++uc;
    }
done:
    // Every MMA issued above has completed once this arrives.
    if (issued) {
        tc_commit(&bars.drain);
        mbar_wait(&bars.drain, 0);
    }
}

// ---------------------------------------------------------------- softmax + epilogue

template <int D>
__device__ void pf_softmax(const PfParams &p, uint8_t *smem, PfBars &bars, uint32_t tmem, int n_units, int warp,
                           int lane)
{
    using C = PfCfg<D>;
    const int quarter = warp & 3;         // TMEM lanes this warp may access
    const int r = quarter * 32 + lane;    // tile row = TMEM lane
    const uint32_t t_row = tmem + ((uint32_t)(quarter * 32) << 16);
    const int G = 1 << p.group_shift;
    const int q_in_tile = r >> p.group_shift;
    const int h_in_group = r & (G - 1);
    const float qs = p.q_scale;
    int ib = 0, gt0 = 0;
    for (int k = 0;; ++k) {
        const int u = pf_unit_at(k);
        if (u >= n_units)
            break;
        const int pair = u / p.num_kv_heads, g = u - pair * p.num_kv_heads;
        const PfUnit un = p.units[pair];
        const int nt = un.n_tiles, kv = un.kv_len;
        const int qi = un.t * p.q_tile + q_in_tile; // query index within the request
        const bool valid = qi < un.q_len;
        const int limit = min(kv - un.q_len + qi, kv - 1);            // last key this row sees
        const int limit_min = kv - un.q_len + un.t * p.q_tile;        // smallest limit of the tile
        float m_used = -INFINITY, l = 0.f;
        for (int j = 0; j < nt; ++j) {
            const int gt = gt0 + j;
            if (!pf_wait_all(&bars.s_full[gt & 1], (gt >> 1) & 1, bars, p.err_flag))
                return;
            tc_fence_after();
            float x[kPfTile];
            {
                uint32_t rr[32];
                const uint32_t sa = t_row + C::kColS + (uint32_t)(gt & 1) * kPfTile;
                tmem_ld32(sa, rr);
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    x[i] = __uint_as_float(rr[i]) * qs;
                tmem_ld32(sa + 32, rr);
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    x[32 + i] = __uint_as_float(rr[i]) * qs;
            }
            const int tok0 = j * kPfTile;
            if (tok0 + kPfTile - 1 > limit_min) {
#pragma unroll
                for (int i = 0; i < kPfTile; ++i)
                    x[i] = (tok0 + i <= limit) ? x[i] : -INFINITY;
            }
            float mt = x[0];
#pragma unroll
            for (int i = 1; i < kPfTile; ++i)
                mt = fmaxf(mt, x[i]);
            const bool grow = mt > m_used + kRescaleLog2;
            float alpha = 1.f;
            if (grow) {
                alpha = ex2_approx(m_used - mt); // 0 on the first tile
                l *= alpha;
                m_used = mt;
            }
            // O holds this unit's sum only after its first PV.
            const bool rescale_o = grow && j > 0;
            if (__any_sync(0xffffffffu, rescale_o)) {
                const int gp = gt - 1;
                if (!pf_wait_all(&bars.o_done[gp & 1], (gp >> 1) & 1, bars, p.err_flag))
                    return;
                tc_fence_after();
                const float a = rescale_o ? alpha : 1.f;
                for (int c = 0; c < D; c += 32) {
                    uint32_t rr[32];
                    tmem_ld32(t_row + C::kColO + c, rr);
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        rr[i] = __float_as_uint(__uint_as_float(rr[i]) * a);
                    tmem_st32(t_row + C::kColO + c, rr);
                }
            }
            // This P buffer was last read by the PV MMA of global tile gt - 2.
            if (gt >= 2) {
                const int gp = gt - 2;
                if (!pf_wait_all(&bars.o_done[gp & 1], (gp >> 1) & 1, bars, p.err_flag))
                    return;
            }
            uint8_t *prow = smem + C::kOffP + (gt & 1) * C::kPBytes + r * 128;
            const float m_ref = m_used == -INFINITY ? 0.f : m_used; // a row that has seen no key yet
            float sum = 0.f;
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) {
                uint32_t whi[4], wlo[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float p0 = ex2_approx(x[c8 * 8 + 2 * e] - m_ref);
                    const float p1 = ex2_approx(x[c8 * 8 + 2 * e + 1] - m_ref);
                    sum += p0 + p1;
                    const __nv_bfloat162 hi = __floats2bfloat162_rn(p0, p1);
                    const float2 hf = __bfloat1622float2(hi);
                    const __nv_bfloat162 lo = __floats2bfloat162_rn(p0 - hf.x, p1 - hf.y);
                    whi[e] = *reinterpret_cast<const uint32_t *>(&hi);
                    wlo[e] = *reinterpret_cast<const uint32_t *>(&lo);
                }
                // 128-byte swizzle: 16-byte piece c8 of row r sits at piece c8 ^ (r % 8)
                const int off = (c8 ^ (r & 7)) << 4;
                *reinterpret_cast<uint4 *>(prow + off) = make_uint4(whi[0], whi[1], whi[2], whi[3]);
                *reinterpret_cast<uint4 *>(prow + C::kPHalf + off) = make_uint4(wlo[0], wlo[1], wlo[2], wlo[3]);
            }
            l += sum;
            // V rows at and past kv in the last tile hold another token's or no
            // data: zero them so that p = 0 there contributes exactly 0.
            if (tok0 + kPfTile > kv) {
                const int itg = ib + pf_item_v(j, nt);
                const int stage = itg % C::kStages;
                if (!pf_wait_all(&bars.full[stage], (itg / C::kStages) & 1, bars, p.err_flag))
                    return;
                const int r0 = kv - tok0;
                uint8_t *vb = smem + C::kOffStage + stage * C::kStageBytes + r0 * 128;
                const int per_chunk = (kPfTile - r0) * 8; // 16-byte pieces
                for (int i = r; i < per_chunk * C::kChunks; i += kPfRows) {
                    const int c = i / per_chunk;
                    *reinterpret_cast<uint4 *>(vb + c * (kPfTile * 128) + (i - c * per_chunk) * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&bars.p_full[gt & 1]);
        }
        { // epilogue: O / l -> bf16, lse
            const int gl = gt0 + nt - 1;
            if (!pf_wait_all(&bars.o_done[gl & 1], (gl >> 1) & 1, bars, p.err_flag))
                return;
            tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const int64_t row = (int64_t)(un.q_start + qi) * p.num_q_heads + g * G + h_in_group;
            __nv_bfloat16 *orow = p.out + row * D;
            for (int c = 0; c < D; c += 32) {
                uint32_t rr[32];
                tmem_ld32(t_row + C::kColO + c, rr);
                uint32_t w[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(rr[2 * e]) * inv,
                                                                   __uint_as_float(rr[2 * e + 1]) * inv);
                    w[e] = *reinterpret_cast<const uint32_t *>(&h);
                }
                if (valid) {
                    uint4 *dst = reinterpret_cast<uint4 *>(orow + c);
                    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
                    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
                    dst[2] = make_uint4(w[8], w[9], w[10], w[11]);
                    dst[3] = make_uint4(w[12], w[13], w[14], w[15]);
                }
            }
            tc_fence_before();
            mbar_arrive(&bars.o_free);
            if (valid && p.lse != nullptr)
                p.lse[row] = (m_used + log2f(l)) * kLn2;
        }
        gt0 += nt;
        ib += 2 * nt;
    }
}

template <int D>
__global__ void __launch_bounds__(kPfThreads, 1)
    prefill_kernel(const __grid_constant__ PfParams p, const __grid_constant__ PfMapsDev maps)
{
    using C = PfCfg<D>;
    extern __shared__ unsigned char pf_smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(pf_smem_raw) + 1023) & ~uintptr_t(1023));
    PfBars &bars = *reinterpret_cast<PfBars *>(smem + C::kOffBar);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(&bars.q_full, 1);
        mbar_init(&bars.q_empty, 1);
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&bars.full[s], 1);
            mbar_init(&bars.empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars.s_full[i], 1);
            mbar_init(&bars.p_full[i], kPfRows);
            mbar_init(&bars.o_done[i], 1);
        }
        mbar_init(&bars.o_free, kPfRows);
        mbar_init(&bars.drain, 1);
        bars.abort = 0;
        mbar_init_fence();
    }
    if (warp == kPfProducerWarp && lane == 0) {
        prefetch_tensormap(&maps.q);
        prefetch_tensormap(&maps.k);
        prefetch_tensormap(&maps.v);
    }
    if (warp == kPfMmaWarp) {
        tmem_alloc(&bars.tmem_base, C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars.tmem_base;
    const int n_units = *p.n_pairs * p.num_kv_heads;

    if (warp == kPfProducerWarp)
        pf_producer<D>(p, maps, smem, bars, n_units, lane);
    else if (warp == kPfMmaWarp) {
        if (lane == 0)
            pf_mma<D>(p, smem, bars, tmem, n_units);
        __syncwarp();
    } else
        pf_softmax<D>(p, smem, bars, tmem, n_units, warp, lane);

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kPfMmaWarp)
        tmem_dealloc(tmem, C::kTmemCols);
}

// ---------------------------------------------------------------- plan

// Exclusive prefix sum over the 1024 threads of the block; *total gets the sum.
__device__ int block_exclusive_scan(int v, int *s_warp, int *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o)
            x += y;
    }
    if (lane == 31)
        s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = s_warp[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o)
                w += y;
        }
        s_warp[lane] = w;
    }
    __syncthreads();
    const int ex = (warp > 0 ? s_warp[warp - 1] : 0) + x - v;
    *total = s_warp[31];
    __syncthreads();
    return ex;
}

__global__ void __launch_bounds__(kPlanThreads) prefill_plan_kernel(const PfPlanParams pp)
{
    __shared__ int s_start[kMaxPrefillBatch], s_end[kMaxPrefillBatch], s_kv[kMaxPrefillBatch];
    __shared__ int s_bad[kMaxPrefillBatch], s_scan[kMaxPrefillBatch + 1];
    __shared__ int s_hist[kPfBuckets];
    __shared__ int s_warp[32];
    __shared__ int s_decreasing;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int P = 1 << pp.page_shift;
    if (tid == 0)
        s_decreasing = 0;
    for (int i = tid; i < kPfBuckets; i += kPlanThreads)
        s_hist[i] = 0;
    __syncthreads();

    // 1. Validate every request (one warp per request).
    for (int b = warp; b < pp.batch; b += kPlanThreads / 32) {
        const int s = pp.qo_indptr[b], e = pp.qo_indptr[b + 1], kv = pp.kv_lens[b];
        const int64_t q = (int64_t)e - s;
        int bad = 0;
        if (q != 0) {
            if (s < 0 || e > pp.total_q || q < 0 || kv < q)
                bad = PKV_ERR_QLEN;
            else if ((int64_t)kv > ((int64_t)pp.max_blocks << pp.page_shift))
                bad = PKV_ERR_OVERFLOW;
            else {
                const int nblk = (int)(((int64_t)kv + P - 1) >> pp.page_shift);
                const int32_t *row = pp.block_table + (int64_t)b * pp.max_blocks;
                bool badp = false;
                for (int i = lane; i < nblk; i += 32) {
                    const int id = row[i];
                    badp |= (id < 1 || id >= pp.num_pages);
                }
                if (__any_sync(0xffffffffu, badp))
                    bad = PKV_ERR_PAGE;
            }
        }
        if (lane == 0) {
            s_start[b] = s;
            s_end[b] = e;
            s_kv[b] = kv;
            s_bad[b] = bad;
            if (q < 0)
                s_decreasing = 1;
        }
    }
    __syncthreads();
    // A decreasing qo_indptr makes the query ranges overlap: no request runs.
    if (s_decreasing != 0) {
        for (int b = tid; b < pp.batch; b += kPlanThreads)
            if (s_end[b] != s_start[b])
                s_bad[b] = PKV_ERR_QLEN;
        __syncthreads();
    }

    // 2. Query tiles per request, prefix sum.
    int v = 0;
    if (tid < pp.batch && s_bad[tid] == 0 && s_end[tid] > s_start[tid])
        v = (s_end[tid] - s_start[tid] + pp.q_tile - 1) / pp.q_tile;
    int n_pairs = 0;
    const int ex = block_exclusive_scan(v, s_warp, &n_pairs);
    if (tid < pp.batch)
        s_scan[tid] = ex;
    if (tid == 0)
        s_scan[pp.batch] = n_pairs;
    __syncthreads();

    auto locate = [&](int pi, int *b_out, int *t_out) {
        int lo = 0, hi = pp.batch - 1; // last b with s_scan[b] <= pi
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_scan[mid] <= pi)
                lo = mid;
            else
                hi = mid - 1;
        }
        *b_out = lo;
        *t_out = pi - s_scan[lo];
    };
    auto bucket_of = [&](int b, int t) {
        const int64_t c = pf_tiles(s_kv[b], s_end[b] - s_start[b], t, pp.q_tile);
        return (int)(c < kPfBuckets - 1 ? c : kPfBuckets - 1);
    };

    // 3. Counting sort of the query tiles by kv tiles, longest first.
    for (int pi = tid; pi < n_pairs; pi += kPlanThreads) {
        int b, t;
        locate(pi, &b, &t);
        atomicAdd(&s_hist[bucket_of(b, t)], 1);
    }
    __syncthreads();
    {
        constexpr int kPer = kPfBuckets / kPlanThreads;
        const int grp = kPlanThreads - 1 - tid; // thread 0 owns the longest buckets
        int h[kPer], sum = 0;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            h[i] = s_hist[grp * kPer + i];
            sum += h[i];
        }
        int unused = 0;
        int off = block_exclusive_scan(sum, s_warp, &unused);
#pragma unroll
        for (int i = kPer - 1; i >= 0; --i) {
            s_hist[grp * kPer + i] = off;
            off += h[i];
        }
    }
    __syncthreads();
    for (int pi = tid; pi < n_pairs; pi += kPlanThreads) {
        int b, t;
        locate(pi, &b, &t);
        const int pos = atomicAdd(&s_hist[bucket_of(b, t)], 1);
        if (pos < pp.cap_pairs) {
            PfUnit un;
            un.b = b;
            un.t = t;
            un.q_start = s_start[b];
            un.q_len = s_end[b] - s_start[b];
            un.kv_len = s_kv[b];
            un.n_tiles = (int)pf_tiles(un.kv_len, un.q_len, t, pp.q_tile);
            un.pad0 = un.pad1 = 0;
            pp.units[pos] = un;
        }
    }
    if (tid == 0)
        *pp.n_pairs = n_pairs < pp.cap_pairs ? n_pairs : (int)pp.cap_pairs;

    // 4. Failing requests: error bit, zero output, lse = -inf.
    const int64_t row_elems = (int64_t)pp.num_q_heads * pp.head_dim;
    for (int b = 0; b < pp.batch; ++b) {
        if (s_bad[b] == 0)
            continue;
        if (tid == 0)
            set_error(pp.err_flag, s_bad[b]);
        const int64_t lo = s_start[b] > 0 ? s_start[b] : 0;
        const int64_t hi = s_end[b] < pp.total_q ? s_end[b] : pp.total_q;
        if (hi <= lo)
            continue;
        uint4 *o = reinterpret_cast<uint4 *>(pp.out + lo * row_elems);
        const int64_t pieces = (hi - lo) * row_elems / 8;
        for (int64_t i = tid; i < pieces; i += kPlanThreads)
            o[i] = make_uint4(0u, 0u, 0u, 0u);
        if (pp.lse != nullptr)
            for (int64_t i = tid; i < (hi - lo) * pp.num_q_heads; i += kPlanThreads)
                pp.lse[lo * pp.num_q_heads + i] = -INFINITY;
    }
}

// ---------------------------------------------------------------- host side

struct PfKernelEntry {
    int D;
    const void *fn;
    uint32_t smem;
};

const PfKernelEntry kPfTable[] = {
    {64, reinterpret_cast<const void *>(&prefill_kernel<64>), PfCfg<64>::kSmem},
    {128, reinterpret_cast<const void *>(&prefill_kernel<128>), PfCfg<128>::kSmem},
    {256, reinterpret_cast<const void *>(&prefill_kernel<256>), PfCfg<256>::kSmem},
};

const PfKernelEntry *pf_find(int D)
{
    for (const PfKernelEntry &e : kPfTable)
        if (e.D == D)
            return &e;
    return nullptr;
}

// Persistent grid size: resident CTAs on all SMs (set up once per device).
int pf_grid(int device, const PfKernelEntry *e)
{
    constexpr int kDevices = 64;
    static int cache[kDevices][3] = {};
    if (device < 0 || device >= kDevices)
        return 1;
    int &slot = cache[device][e - kPfTable];
    if (slot == 0) {
        int occ = 1;
        if (cudaFuncSetAttribute(e->fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)e->smem) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, e->fn, kPfThreads, e->smem) != cudaSuccess ||
            occ < 1)
            occ = 1;
        slot = sm_count(device) * occ;
    }
    return slot;
}

} // namespace

bool prefill_shape(int batch, int total_q, int num_q_heads, const pkv_cache_desc &d, PrefillShape *s)
{
    if (d.num_kv_heads <= 0 || num_q_heads % d.num_kv_heads != 0 || batch < 0 || total_q < 0)
        return false;
    const int group = num_q_heads / d.num_kv_heads;
    if ((group & (group - 1)) != 0 || group > kPfRows)
        return false;
    if (d.page_size < 8 || pf_find(d.head_dim) == nullptr)
        return false;
    int gs = 0;
    while ((1 << gs) < group)
        ++gs;
    s->group = group;
    s->group_shift = gs;
    s->q_tile = kPfRows / group;
    s->cap_pairs = ((int64_t)total_q + s->q_tile - 1) / s->q_tile + batch;
    if (s->cap_pairs * d.num_kv_heads >= ((int64_t)1 << 31))
        return false;
    s->bytes = 256 + (((size_t)s->cap_pairs * sizeof(PfUnit) + 255) & ~size_t(255));
    return true;
}

cudaError_t launch_prefill(const PrefillArgs &a, const PrefillMaps &maps, cudaStream_t stream)
{
    const PfKernelEntry *e = pf_find(a.desc.head_dim);
    if (e == nullptr)
        return cudaErrorInvalidValue;
    unsigned char *ws = static_cast<unsigned char *>(a.workspace);
    int32_t *n_pairs = reinterpret_cast<int32_t *>(ws);
    PfUnit *units = reinterpret_cast<PfUnit *>(ws + 256);
    int page_shift = 0;
    while ((1 << page_shift) < a.desc.page_size)
        ++page_shift;

    PfPlanParams pp;
    pp.qo_indptr = a.qo_indptr;
    pp.kv_lens = a.kv_lens;
    pp.block_table = a.block_table;
    pp.units = units;
    pp.n_pairs = n_pairs;
    pp.out = static_cast<__nv_bfloat16 *>(a.out);
    pp.lse = a.lse;
    pp.err_flag = a.err_flag;
    pp.batch = a.batch;
    pp.max_blocks = a.max_blocks;
    pp.num_pages = a.desc.num_pages;
    pp.page_shift = page_shift;
    pp.total_q = a.total_q;
    pp.q_tile = a.shape.q_tile;
    pp.num_q_heads = a.num_q_heads;
    pp.head_dim = a.desc.head_dim;
    pp.cap_pairs = a.shape.cap_pairs;
    prefill_plan_kernel<<<1, kPlanThreads, 0, stream>>>(pp);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess)
        return err;

    PfParams p;
    p.block_table = a.block_table;
    p.units = units;
    p.n_pairs = n_pairs;
    p.out = static_cast<__nv_bfloat16 *>(a.out);
    p.lse = a.lse;
    p.err_flag = a.err_flag;
    p.max_blocks = a.max_blocks;
    p.num_q_heads = a.num_q_heads;
    p.num_kv_heads = a.desc.num_kv_heads;
    p.group_shift = a.shape.group_shift;
    p.q_tile = a.shape.q_tile;
    p.page_shift = page_shift;
    p.box_shift = page_shift < 6 ? page_shift : 6;
    p.layout = a.desc.layout;
    p.q_scale = a.q_scale;
    PfMapsDev m;
    m.q = maps.q;
    m.k = maps.k;
    m.v = maps.v;

    int dev = 0;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess)
        return err;
    int grid = pf_grid(dev, e);
    const int64_t max_units = a.shape.cap_pairs * a.desc.num_kv_heads;
    if (grid > max_units)
        grid = (int)max_units;
    if (grid < 1)
        grid = 1;
    void *args[] = {&p, &m};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kPfThreads);
    cfg.dynamicSmemBytes = e->smem;
    cfg.stream = stream;
    return cudaLaunchKernelExC(&cfg, e->fn, args);
}

int prefill_box_tokens(int page_size)
{
    return page_size < kPfTile ? page_size : kPfTile;
}

} // namespace pkv
