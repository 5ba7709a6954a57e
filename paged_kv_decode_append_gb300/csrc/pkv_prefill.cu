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
//  - Work unit = (request, kv head, one query tile of 128/G queries per CTA
//    of the cluster: two for a CTA pair).
//    The G query heads sharing a kv head times 128/G consecutive queries form
//    a CTA's 128 MMA rows (row r = query r/G, head r%G), so every K/V tile
//    read from the pages serves all G heads.
//  - A one-CTA plan kernel validates every request, lists the units and
//    orders them by their number of 64-token kv tiles, longest first; the
//    persistent clusters (or single CTAs) take units in that order, snaking
//    over the grid.
//  - head_dim 128 and 256 (prefill2_kernel): the cluster is a CTA pair
//    whose MMAs (tcgen05.mma.cta_group::2, M = 256) cover both query tiles,
//    issued by one thread of the even CTA.  Keys go in steps of 128.  For
//    S = Q K^T (N = 128) the even CTA holds the step's first 64-key K tile
//    and the odd CTA the second; for O += P V (N = head_dim) each CTA holds
//    all 128 keys of its half of head_dim -- each SM stages half of every
//    operand, and one instruction does twice the work of a single-CTA MMA
//    with N = 64 (issuing one costs about the same whatever its shape).
//    TMEM: O [128 x D] fp32 and two S [128 x 128] buffers (S of step t+1 is
//    computed while the softmax of step t runs); Q [128 x D] in shared
//    memory, K-major and swizzled.
//  - head_dim 64 (prefill_kernel): one query tile per CTA (clusters of
//    one), 64-key tiles, each CTA loading its own K / V tiles, Q in TMEM.
//  - Warp roles: warp 0 loads this CTA's K and V with TMA into a ring of
//    shared-memory stages (head_dim 64, in the order the MMAs consume them;
//    CTA pairs: warp 0 the K ring, warp 10 the V ring); warp 1 owns TMEM and
//    one of its threads issues the MMAs (the odd CTA of a pair: relays its
//    stage completions to it); warps 2-9 (two per TMEM lane quarter) run the
//    online softmax and the epilogue, each thread on half of its row's
//    columns.
//  - The softmax writes P back over the S columns it has just read, as two
//    bf16 parts, p = hi + lo (about 16 significant bits: a single bf16 P
//    alone, 8 bits, leaves errors near 2^-9 of the row's scale, well above
//    1e-2 of the small outputs that cancellation produces); O += P_hi V +
//    P_lo V with P from TMEM and V as an MN-major operand (its rows are
//    tokens, its columns head_dim).
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

constexpr int kPfSoftmaxWarps = 8; // two per TMEM lane quarter, each on half of a row's columns
constexpr int kPfSoftmaxThreads = kPfSoftmaxWarps * 32;
constexpr int kPfThreads = 64 + kPfSoftmaxThreads;
// CTA-pair kernel: one more warp, a second producer (V items; warp 0 loads K)
constexpr int kPf2VWarp = kPfThreads / 32;
constexpr int kPf2Threads = kPfThreads + 32;
constexpr int kPfProducerWarp = 0;
constexpr int kPfMmaWarp = 1;
constexpr int kPfRows = 128;    // M of every MMA
constexpr int kPfTile = 64;     // kv tokens per tile
constexpr int kPfBuckets = 4096; // plan: units are ordered by min(kv tiles, 4095)
constexpr int kPlanThreads = 1024;
constexpr int kPfZeroOnly = 0x100; // plan: a request whose output is zeroed without an error bit
constexpr float kRescaleLog2 = 8.0f;
constexpr float kLn2 = 0.693147180559945309f;

constexpr int kPfMaxStages = 12;

template <int D> struct PfCfg {
    static constexpr bool kPair = false;
    static constexpr int kChunks = D / 64;                                      // 128-byte column blocks of a row
    static constexpr int kStages = D == 256 ? 6 : kPfMaxStages; // K / V tiles in flight
    // A K or V stage is [8-token group][64-column block][8 rows][128 B]: for
    // one column block, consecutive 8-row groups are kGroupStride apart.
    static constexpr uint32_t kStageBytes = kPfTile * D * 2;
    static constexpr uint32_t kGroupStride = 8 * D * 2;
    static constexpr uint32_t kOffStage = 0;
    static constexpr uint32_t kOffBar = kOffStage + kStages * kStageBytes;
    static constexpr uint32_t kOffXchg = kOffBar + 512;     // softmax half-row exchange
    static constexpr uint32_t kSmem = kOffXchg + 3 * 1024 + 1024; // + alignment slack
    static constexpr uint32_t kColO = 0;
    // Two 64-column S buffers; the softmax overwrites S of a tile with its P
    // (bf16 pairs: P_hi in the first 32 columns, P_lo in the last 32), which
    // the PV MMA reads as its A operand.
    static constexpr uint32_t kColS = D;
    static constexpr uint32_t kColQ = D + 2 * kPfTile;     // D / 2 columns of bf16 pairs
    static constexpr uint32_t kTmemCols = (kColQ + D / 2) <= 256 ? 256 : 512;
    // a V tile in a stage: all of head_dim (the same layout as K)
    static constexpr uint32_t kItemBytes = kStageBytes;
    static constexpr uint32_t kVGroupStride = kGroupStride;
    static constexpr int kVChunks = kChunks;
};

// CTA pairs (head_dim 128 and 256), in steps of 128 keys (two 64-key tiles).
// The pair's MMAs have M = 256 (one query tile per CTA) and read each operand
// half from one CTA: for S = Q K^T (N = 128 keys) the even CTA holds the
// step's first K tile and the odd CTA its second, all of head_dim; for
// O += P V (N = head_dim) each CTA holds all 128 keys of its half of
// head_dim.  Q sits in shared memory (TMEM holds O and two 128-column S
// buffers).  An item is a step's K tile or its V half; both are
// 64 * head_dim * 2 bytes.
constexpr int kPfPairMaxStages = 12;
constexpr int kPfStep = 2 * kPfTile; // keys per step
template <int D> struct Pf2Cfg {
    static_assert(D == 128 || D == 256, "pairs split head_dim into 64-column blocks");
    static constexpr uint32_t kItemBytes = kPfTile * D * 2;
    static constexpr int kStages = 4;                              // items in flight
    // K items (one per step) and V items (one per step) have rings of their
    // own, each filled by its own producer warp: the step's index gs picks
    // the slot, K in [0, kKStages), V in [kKStages, kStages).
    static constexpr int kKStages = kStages / 2;
    static constexpr int kVStages = kStages - kKStages;
    static __device__ __forceinline__ int k_slot(int gs) { return gs % kKStages; }
    static __device__ __forceinline__ uint32_t k_par(int gs) { return (uint32_t)(gs / kKStages) & 1u; }
    static __device__ __forceinline__ int v_slot(int gs) { return kKStages + gs % kVStages; }
    static __device__ __forceinline__ uint32_t v_par(int gs) { return (uint32_t)(gs / kVStages) & 1u; }
    // Rings of two slots: the item of step gs - 2 is the slot's previous one,
    // and the step's own completion barrier (s_full / o_done of parity gs & 1,
    // phase gs >> 1) releases it -- no separate commit to an empty barrier.
    static_assert(kKStages == 2 && kVStages == 2, "slots are released by the step barriers");
    static constexpr uint32_t kGroupStride = 8 * D * 2;            // K and Q: 8 rows x head_dim
    static constexpr uint32_t kVGroupStride = 8 * (D / 2) * 2;     // V half: 8 keys x half of head_dim
    static constexpr int kVChunks = D / 128;                       // 64-column blocks of a V half
    static constexpr uint32_t kOffStage = 0;
    static constexpr uint32_t kOffQ = kOffStage + kStages * kItemBytes;  // Q [128 rows][head_dim], K-major, swizzled
    static constexpr uint32_t kOffBar = kOffQ + kPfRows * D * 2;
    static constexpr uint32_t kOffXchg = kOffBar + 1024;
    // epilogue staging: per softmax warp 32 rows x 32 bf16 columns (2 KB), so
    // that the global stores of out are row-contiguous 64-byte pieces
    static constexpr uint32_t kOffOut = kOffXchg + 3 * 1024;
    static constexpr uint32_t kSmem = kOffOut + kPfSoftmaxWarps * 2048 + 1024;
    static constexpr uint32_t kColO = 0;
    static constexpr uint32_t kColS = D;                           // two S buffers of kPfStep columns
    static constexpr uint32_t kTmemCols = 512;
};
static_assert(Pf2Cfg<256>::kSmem <= 232448 && Pf2Cfg<128>::kSmem <= 232448, "pair prefill shared memory");
static_assert(Pf2Cfg<256>::kColS + 2 * kPfStep <= 512, "pair prefill TMEM columns");

template <int S>
struct PfBarsT {
    uint64_t q_full, q_empty;
    uint64_t full[S], empty[S];
    uint64_t peer_full[S]; // CTA pairs: the odd CTA's half of a stage has landed (relayed)
    uint64_t s_full[2], p_full[2], o_done[2];
    uint64_t o_free;
    uint64_t drain;
    uint64_t pair[4]; // the two softmax warps of each TMEM lane quarter
    uint32_t tmem_base;
    int32_t abort;
};
using PfBars = PfBarsT<kPfMaxStages>;
using Pf2Bars = PfBarsT<kPfPairMaxStages>;
static_assert(sizeof(PfBars) <= 512, "barrier block");
static_assert(sizeof(Pf2Bars) <= 1024, "pair barrier block");

// `cluster` consecutive query tiles of one request (all kv heads share it):
// CTA rank r of a cluster takes query tile t * cluster + r.
struct PfUnit {
    int32_t b, t, q_start, q_len, kv_len, n_tiles, pad0, pad1;
};
static_assert(sizeof(PfUnit) == 32, "unit record");

struct PfParams {
    const __nv_bfloat16 *q;
    const int32_t *block_table;
    const PfUnit *units;
    const int32_t *n_pairs;
    __nv_bfloat16 *out;
    float *lse;
    int32_t *err_flag;
    int max_blocks, num_q_heads, num_kv_heads, total_q;
    int group_shift, q_tile, page_shift, box_shift, layout;
    int cluster; // CTAs per cluster: 2 for a CTA pair, 1 for the single-CTA kernel
    float q_scale;
    int pdl; // launched as a programmatic dependent: set up, then wait for the preceding grid
};

struct PfMapsDev {
    CUtensorMap k, v; // token-group boxes (encode_group_map)
};

struct PfPlanParams {
    const int32_t *qo_indptr;
    const int32_t *kv_lens;
    // Mixed step (kv_lens unused): request b holds cache_seqlens[b] cached
    // tokens (< 0: inactive), kv = cache_seqlens[b] + kv_add * q keys; only
    // requests with q_lo < q are this kernel's, q > q_max is malformed.
    const int32_t *cache_seqlens;
    int q_lo, q_max, kv_add;
    const int32_t *block_table;
    PfUnit *units;
    int32_t *n_pairs;
    __nv_bfloat16 *out;
    float *lse;
    int32_t *err_flag;
    int batch, max_blocks, num_pages, page_shift, total_q, q_tile, num_q_heads, head_dim, cluster;
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

// k-th unit of this CTA's cluster (every CTA of a cluster works on the same
// unit): rounds of one unit per cluster, alternating direction.
__device__ __forceinline__ int pf_unit_at(int k, int cluster)
{
    const int g = (int)gridDim.x / cluster, c = (int)blockIdx.x / cluster;
    return k * g + ((k & 1) ? g - 1 - c : c);
}

// Bounded barrier wait that also gives up when another role has aborted:
// the first test inline, the polling loop out of line.  The waits are
// CTA-scoped, like those of every mbarrier that TMA, tcgen05.commit or a
// peer CTA's remote arrive completes here (the data those signal is written
// by the async proxy, or by tcgen05.st before the signalling fence).
template <class Bars>
__device__ __noinline__ bool pf_wait_slow(uint64_t *bar, uint32_t parity, Bars &bars, int32_t *err_flag)
{
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

// CL: the barrier is also arrived on from the other CTA of a pair (kept for
// the call sites' documentation; the wait is the same).
template <bool CL, class Bars>
__device__ __forceinline__ bool pf_wait(uint64_t *bar, uint32_t parity, Bars &bars, int32_t *err_flag)
{
    if (mbar_try_wait(bar, parity))
        return true;
    return pf_wait_slow(bar, parity, bars, err_flag);
}
__device__ __forceinline__ bool pf_wait(uint64_t *bar, uint32_t parity, PfBars &bars, int32_t *err_flag)
{
    return pf_wait<false>(bar, parity, bars, err_flag);
}

// pf_wait for a whole warp: every lane gets the same answer, so warp-collective
// instructions after it are reached by all lanes or none.
template <bool CL = false, class Bars>
__device__ __forceinline__ bool pf_wait_all(uint64_t *bar, uint32_t parity, Bars &bars, int32_t *err_flag)
{
    const bool ok = pf_wait<CL>(bar, parity, bars, err_flag);
    return __all_sync(0xffffffffu, ok);
}

// ---------------------------------------------------------------- producer

template <int D>
__device__ void pf_producer(const PfParams &p, const PfMapsDev &maps, uint8_t *smem, PfBars &bars, int n_units,
                            int lane)
{
    using C = PfCfg<D>;
    const int Hkv = p.num_kv_heads;
    const int P = 1 << p.page_shift;
    const int BT = 1 << p.box_shift;             // tokens per box: min(page_size, 64)
    const int boxes = kPfTile >> p.box_shift;     // boxes per full tile
    const uint32_t box_bytes = (uint32_t)BT * D * 2; // BT tokens x all of head_dim
    const bool nhd = p.layout == PKV_NHD;
    int ib = 0, issued = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
        const int u = pf_unit_at(k, p.cluster);
        if (u >= n_units)
            break;
        const int grp = u / Hkv, g = u - grp * Hkv;
        const PfUnit un = p.units[grp];
        const int32_t *bt_row = p.block_table + (int64_t)un.b * p.max_blocks;
        const int nt = un.n_tiles, kv = un.kv_len;
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
                // The stage is free once the MMAs that read it have completed.
                if (n > 0 && !pf_wait_all(&bars.empty[stage], (n - 1) & 1, bars, p.err_flag)) {
                    ok = false;
                    break;
                }
                const int tok0 = jj * kPfTile;
                const int ntok = min(kPfTile, kv - tok0);
                const int nbox = (ntok + BT - 1) >> p.box_shift;
                uint8_t *dst = smem + C::kOffStage + stage * C::kStageBytes;
                const int ids = kind == 0 ? ids_cur : ids_prev;
                if (lane == 0)
                    mbar_arrive_expect_tx(&bars.full[stage], (uint32_t)nbox * box_bytes);
                // Sub-boxes: K (and V when a box is a whole tile) in 64-column
                // boxes, [block][64 tokens][128 B], so the S MMA sees evenly
                // spaced rows; V otherwise in page boxes, [box][block][BT][128 B].
                const CUtensorMap *map = kind == 0 ? &maps.k : &maps.v;
                for (int bx = 0; bx < nbox; ++bx) {
                    const int page = __shfl_sync(0xffffffffu, ids, bx);
                    if (lane != 0)
                        continue;
                    const int slot = (tok0 + bx * BT) & (P - 1);
                    if (nhd)
                        tma_load_5d_plain(dst + bx * box_bytes, map, 0, 0, 0, (page * P + slot) >> 3, g,
                                          &bars.full[stage]);
                    else
                        tma_load_5d_plain(dst + bx * box_bytes, map, 0, 0, 0, slot >> 3, page * Hkv + g,
                                          &bars.full[stage]);
                }
                issued = itg + 1;
            }
            ids_prev = ids_cur;
            ids_cur = ids_next;
            ids_next = page_ids(j + 2);
        }
        ib += 2 * nt;
    }
    // Copies still in flight into this CTA: once they have landed nothing
    // writes into its shared memory any more.  Immediate unless a wait gave up.
    for (int itg = issued > C::kStages ? issued - C::kStages : 0; itg < issued; ++itg)
        pf_wait(&bars.full[itg % C::kStages], (itg / C::kStages) & 1, bars, p.err_flag);
}

// ---------------------------------------------------------------- MMA issuer

template <int D>
__device__ void pf_mma(const PfParams &p, uint8_t *smem, PfBars &bars, uint32_t tmem, int n_units)
{
    using C = PfCfg<D>;
    constexpr uint32_t kIdescS = tc_idesc_bf16(kPfRows, kPfTile, false, false);
    constexpr uint32_t kIdescO = tc_idesc_bf16(kPfRows, D, false, true);
    const uint32_t st_base = smem_addr(smem + C::kOffStage);
    int ib = 0, gt0 = 0;
    uint32_t uc = 0;
    bool issued = false;
    for (int k = 0;; ++k) {
        const int u = pf_unit_at(k, p.cluster);
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
                const uint64_t kd = tc_sw128_desc(st_base + stage * C::kStageBytes, 16, C::kGroupStride);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    tc_mma_bf16_ts(d, tmem + C::kColQ + kk * 8, kd + (uint64_t)(((kk >> 2) * 1024 + (kk & 3) * 32) >> 4),
                                   kIdescS, kk > 0 ? 1u : 0u);
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
                const uint32_t pt = tmem + C::kColS + (uint32_t)(gt & 1) * kPfTile; // P of tile gt
                // V rows 16*k4 .. +15: two 8-row groups; N spans the column blocks (1024 B apart)
                const uint64_t vd = tc_sw128_desc(st_base + stage * C::kStageBytes, 1024, C::kGroupStride);
#pragma unroll
                for (int kk = 0; kk < 2 * (kPfTile / 16); ++kk) { // hi part, then lo part
                    const int k4 = kk & (kPfTile / 16 - 1);      // 16-token K step
                    tc_mma_bf16_ts(tmem + C::kColO, pt + (kk >> 2) * (kPfTile / 2) + k4 * 8,
                                   vd + (uint64_t)((2 * k4 * C::kGroupStride) >> 4), kIdescO,
                                   (jv > 0 || kk > 0) ? 1u : 0u);
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

// Writes this thread's half of its row of a unit's Q tile (query r / G, head
// r % G of the group; head_dim columns [half * D/2, (half+1) * D/2)) into TMEM
// columns kColQ + half * D/4 .. as bf16 pairs; rows past total_q get 0.
template <int D, class C>
__device__ __forceinline__ void pf_load_q(const PfParams &p, const PfUnit &un, int g, int r, int half,
                                          uint32_t t_row, int cl_rank)
{
    const int tok = un.q_start + (un.t * p.cluster + cl_rank) * p.q_tile + (r >> p.group_shift);
    const int head = g * (1 << p.group_shift) + (r & ((1 << p.group_shift) - 1));
    const bool in = tok < p.total_q;
    const uint4 *src =
        reinterpret_cast<const uint4 *>(p.q + ((int64_t)(in ? tok : 0) * p.num_q_heads + head) * D + half * (D / 2));
    constexpr int kLoads = D / 16; // 16-byte loads of half a row (at most 16)
    uint4 v[kLoads];
#pragma unroll
    for (int i = 0; i < kLoads; ++i)
        v[i] = in ? __ldg(src + i) : make_uint4(0u, 0u, 0u, 0u);
    if constexpr (kLoads >= 8) {
#pragma unroll
        for (int c = 0; c < kLoads / 8; ++c) {
            uint32_t w[32];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                w[4 * i] = v[8 * c + i].x;
                w[4 * i + 1] = v[8 * c + i].y;
                w[4 * i + 2] = v[8 * c + i].z;
                w[4 * i + 3] = v[8 * c + i].w;
            }
            tmem_st32(t_row + C::kColQ + half * (D / 4) + c * 32, w);
        }
    } else { // head_dim 64: half a row is 16 columns
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            w[4 * i] = v[i].x;
            w[4 * i + 1] = v[i].y;
            w[4 * i + 2] = v[i].z;
            w[4 * i + 3] = v[i].w;
        }
        tmem_st16(t_row + C::kColQ + half * (D / 4), w);
    }
}

// Synchronises the two warps that share a TMEM lane quarter (their `phase`-th
// meeting); bounded like every wait, false if it gave up.
template <class Bars>
__device__ __forceinline__ bool pf_pair_sync(Bars &bars, int quarter, uint32_t &phase, int32_t *err_flag)
{
    mbar_arrive(&bars.pair[quarter]);
    return pf_wait_all(&bars.pair[quarter], (phase++) & 1, bars, err_flag);
}

// A softmax thread's arrival on a barrier the MMA thread waits on: every
// thread arrives (one CTA), or -- CTA pairs -- each warp arrives once on the
// barrier of its pair's even CTA (rank & ~1), whose MMA thread issues for
// both: locally there, remotely from the odd CTA.  The thread's tcgen05 /
// shared-memory writes are fenced before the call.
template <bool PAIR>
__device__ __forceinline__ void pf_arrive_mma(uint64_t *bar, int lane, int rank)
{
    if constexpr (PAIR) {
        __syncwarp();
        if (lane == 0) {
            if ((rank & 1) == 0)
                mbar_arrive(bar);
            else
                mbar_arrive_remote(bar, (uint32_t)(rank & ~1));
        }
    } else {
        mbar_arrive(bar);
    }
}

template <int D, class C, class Bars>
__device__ void pf_softmax(const PfParams &p, uint8_t *smem, Bars &bars, uint32_t tmem, int n_units, int warp,
                           int lane, int cl_rank)
{
    constexpr bool PAIR = C::kPair;
    constexpr int kCols = kPfTile / 2;    // S columns of this thread
    const int quarter = warp & 3;         // TMEM lanes this warp may access
    const int half = (warp - 2) >> 2;     // which half of the row's columns
    const int r = quarter * 32 + lane;    // tile row = TMEM lane
    const int st = half * kPfRows + r;    // index among the softmax threads
    const uint32_t t_row = tmem + ((uint32_t)(quarter * 32) << 16);
    float *xchg = reinterpret_cast<float *>(smem + C::kOffXchg); // [2 parities][2 halves][128 rows] + [2][128] sums
    const int G = 1 << p.group_shift;
    const int q_in_tile = r >> p.group_shift;
    const int h_in_group = r & (G - 1);
    const float qs = p.q_scale;
    int ib = 0, gt0 = 0;
    uint32_t pair_phase = 0;

    int u = pf_unit_at(0, p.cluster);
    if (u >= n_units)
        return;
    {
        const int grp = u / p.num_kv_heads;
        pf_load_q<D, C>(p, p.units[grp], u - grp * p.num_kv_heads, r, half, t_row, cl_rank);
        tc_fence_before();
        pf_arrive_mma<PAIR>(&bars.q_full, lane, cl_rank);
    }
    for (int k = 0;; ++k) {
        u = pf_unit_at(k, p.cluster);
        if (u >= n_units)
            break;
        const int grp = u / p.num_kv_heads, g = u - grp * p.num_kv_heads;
        const PfUnit un = p.units[grp];
        const int nt = un.n_tiles, kv = un.kv_len;
        const int t = un.t * p.cluster + cl_rank;   // this CTA's query tile
        const int qi = t * p.q_tile + q_in_tile;    // query index within the request
        const bool valid = qi < un.q_len;           // a tile past the request's end computes nothing kept
        const int limit = min(kv - un.q_len + qi, kv - 1);                      // last key this row sees
        const int limit_min = min(kv - un.q_len + t * p.q_tile, kv - 1);       // smallest limit of the tile
        const int u_next = pf_unit_at(k + 1, p.cluster);
        float m_used = -INFINITY, l = 0.f; // l: this half's part of the row sum
        for (int j = 0; j < nt; ++j) {
            const int gt = gt0 + j;
            if (!pf_wait_all<PAIR>(&bars.s_full[gt & 1], (gt >> 1) & 1, bars, p.err_flag))
                return;
            tc_fence_after();
            // Raw scores of this half; a non-positive scale is applied here, a
            // positive one is folded into the exponent.
            float x[kCols];
            {
                uint32_t rr[32];
                tmem_ld32(t_row + C::kColS + (uint32_t)(gt & 1) * kPfTile + half * kCols, rr);
#pragma unroll
                for (int i = 0; i < kCols; ++i)
                    x[i] = __uint_as_float(rr[i]);
            }
            if (!(qs > 0.f)) {
#pragma unroll
                for (int i = 0; i < kCols; ++i)
                    x[i] *= qs;
            }
            const float qse = qs > 0.f ? qs : 1.f;
            const int tok0 = j * kPfTile + half * kCols;
            if (j * kPfTile + kPfTile - 1 > limit_min) {
#pragma unroll
                for (int i = 0; i < kCols; ++i)
                    x[i] = (tok0 + i <= limit) ? x[i] : -INFINITY;
            }
            float mx = x[0];
#pragma unroll
            for (int i = 1; i < kCols; ++i)
                mx = fmaxf(mx, x[i]);
            // row maximum over both halves
            float *xm = xchg + (gt & 1) * (2 * kPfRows);
            xm[half * kPfRows + r] = mx;
            if (!pf_pair_sync(bars, quarter, pair_phase, p.err_flag))
                return;
            mx = fmaxf(mx, xm[(1 - half) * kPfRows + r]);
            const float mt = mx * qse; // tile maximum in log2 units
            const bool grow = mt > m_used + kRescaleLog2;
            float alpha = 1.f;
            if (grow) {
                alpha = ex2_approx(m_used - mt); // 0 on the first tile
                l *= alpha;
                m_used = mt;
            }
            const float m_ref = m_used == -INFINITY ? 0.f : m_used; // a row that has seen no key yet
            // p = 2^(x*qse - m_ref) = hi + lo, both bf16, packed in pairs
            uint32_t whi[kCols / 2], wlo[kCols / 2];
            float2 sum2 = make_float2(0.f, 0.f);
            const float2 q2 = make_float2(qse, qse), nm2 = make_float2(-m_ref, -m_ref);
#pragma unroll
            for (int e = 0; e < kCols / 2; ++e) {
                const float2 a = ffma2(make_float2(x[2 * e], x[2 * e + 1]), q2, nm2);
                const float2 pp = make_float2(ex2_approx(a.x), ex2_approx(a.y));
                sum2 = __fadd2_rn(sum2, pp);
                const __nv_bfloat162 hi = __floats2bfloat162_rn(pp.x, pp.y);
                const float2 hf = __bfloat1622float2(hi);
                const float2 d = __fadd2_rn(pp, make_float2(-hf.x, -hf.y));
                const __nv_bfloat162 lo = __floats2bfloat162_rn(d.x, d.y);
                whi[e] = *reinterpret_cast<const uint32_t *>(&hi);
                wlo[e] = *reinterpret_cast<const uint32_t *>(&lo);
            }
            l += sum2.x + sum2.y;
            // O holds this unit's sum only after its first PV; rescale this
            // half's columns once the PV of tile gt - 1 is done.
            const bool rescale_o = grow && j > 0;
            if (__any_sync(0xffffffffu, rescale_o)) {
                const int gp = gt - 1;
                if (!pf_wait_all<PAIR>(&bars.o_done[gp & 1], (gp >> 1) & 1, bars, p.err_flag))
                    return;
                tc_fence_after();
                const float a = rescale_o ? alpha : 1.f;
                for (int c = half * (D / 2); c < (half + 1) * (D / 2); c += 32) {
                    uint32_t rr[32];
                    tmem_ld32(t_row + C::kColO + c, rr);
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        rr[i] = __float_as_uint(__uint_as_float(rr[i]) * a);
                    tmem_st32(t_row + C::kColO + c, rr);
                }
            }
            // P over S in TMEM (both halves of the row have read S: the pair
            // sync above): hi pairs at columns [16 half, +16), lo at 32 + that.
            {
                const uint32_t pcol = t_row + C::kColS + (uint32_t)(gt & 1) * kPfTile + half * (kCols / 2);
                tmem_st16(pcol, whi);
                tmem_st16(pcol + kPfTile / 2, wlo);
            }
            // V rows at and past kv in the last tile hold another token's or no
            // data: zero them so that p = 0 there contributes exactly 0.
            if (j * kPfTile + kPfTile > kv) {
                const int itg = ib + pf_item_v(j, nt);
                const int stage = itg % C::kStages;
                if (!pf_wait_all<PAIR>(&bars.full[stage], (itg / C::kStages) & 1, bars, p.err_flag))
                    return;
                const int r0 = kv - j * kPfTile;
                uint8_t *vb = smem + C::kOffStage + stage * C::kItemBytes;
                // 16-byte pieces of rows r0..63, every 64-column block of the stage
                for (int i = st; i < (kPfTile - r0) * C::kVChunks * 8; i += kPfSoftmaxThreads) {
                    const int piece = i & 7, rest = i >> 3;
                    const int c = rest % C::kVChunks, tt = r0 + rest / C::kVChunks;
                    *reinterpret_cast<uint4 *>(vb + (tt >> 3) * C::kVGroupStride + c * 1024 + (tt & 7) * 128 +
                                               piece * 16) = make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem(); // the zeros before the PV MMA's (async proxy) read
            }
            tc_fence_before();
            pf_arrive_mma<PAIR>(&bars.p_full[gt & 1], lane, cl_rank);
        }
        // The next unit's Q, once this unit's S MMAs have read theirs; the MMA
        // thread meanwhile runs this unit's last PV.
        if (u_next < n_units) {
            if (!pf_wait_all<PAIR>(&bars.q_empty, k & 1, bars, p.err_flag))
                return;
            tc_fence_after();
            const int pn = u_next / p.num_kv_heads;
            pf_load_q<D, C>(p, p.units[pn], u_next - pn * p.num_kv_heads, r, half, t_row, cl_rank);
            tc_fence_before();
            pf_arrive_mma<PAIR>(&bars.q_full, lane, cl_rank);
        }
        { // epilogue: O / l -> bf16 (this half's columns), lse
            float *xl = xchg + 4 * kPfRows;
            xl[half * kPfRows + r] = l;
            if (!pf_pair_sync(bars, quarter, pair_phase, p.err_flag))
                return;
            const float lt = l + xl[(1 - half) * kPfRows + r];
            if (!pf_pair_sync(bars, quarter, pair_phase, p.err_flag)) // both read before the next unit's sums overwrite
                return;
            const int gl = gt0 + nt - 1;
            if (!pf_wait_all<PAIR>(&bars.o_done[gl & 1], (gl >> 1) & 1, bars, p.err_flag))
                return;
            tc_fence_after();
            const float inv = lt > 0.f ? 1.f / lt : 0.f;
            const int64_t row = (int64_t)(un.q_start + qi) * p.num_q_heads + g * G + h_in_group;
            __nv_bfloat16 *orow = p.out + row * D;
            for (int c = half * (D / 2); c < (half + 1) * (D / 2); c += 32) {
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
            pf_arrive_mma<PAIR>(&bars.o_free, lane, cl_rank);
            if (half == 0 && valid && p.lse != nullptr)
                p.lse[row] = (m_used + log2f(lt)) * kLn2;
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
        mbar_init(&bars.q_full, kPfSoftmaxThreads);
        mbar_init(&bars.q_empty, 1);
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&bars.full[s], 1);
            mbar_init(&bars.empty[s], 1); // released by this CTA's MMAs
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars.s_full[i], 1);
            mbar_init(&bars.p_full[i], kPfSoftmaxThreads);
            mbar_init(&bars.o_done[i], 1);
        }
        mbar_init(&bars.o_free, kPfSoftmaxThreads);
        for (int i = 0; i < 4; ++i)
            mbar_init(&bars.pair[i], 64);
        mbar_init(&bars.drain, 1);
        bars.abort = 0;
        mbar_init_fence();
    }
    if (warp == kPfProducerWarp && lane == 0) {
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
    if (p.pdl) // the plan (and, in a mixed step, the append) wrote what follows
        asm volatile("griddepcontrol.wait;" ::: "memory");
    const uint32_t tmem = bars.tmem_base;
    const int n_units = *p.n_pairs * p.num_kv_heads;

    if (warp == kPfProducerWarp)
        pf_producer<D>(p, maps, smem, bars, n_units, lane);
    else if (warp == kPfMmaWarp) {
        if (lane == 0)
            pf_mma<D>(p, smem, bars, tmem, n_units);
        __syncwarp();
    } else
        pf_softmax<D, PfCfg<D>, PfBars>(p, smem, bars, tmem, n_units, warp, lane, 0);

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kPfMmaWarp)
        tmem_dealloc(tmem, C::kTmemCols);
}

// ---------------------------------------------------------------- CTA pairs

// Producers of one CTA of a pair, step by step (128 keys): warp `which` = 0
// loads the K items, warp 1 the V items, each into a ring of its own.  Item
// K_t is the step's tile 2t + r (r = the CTA's rank in its pair), 64 keys
// with all of head_dim; item V_t is all 128 keys of the step with columns
// [r D/2, (r+1) D/2).  Boxes of min(page, 64) tokens, one lane per box.  A
// slot is refilled once the pair's MMAs that read it have completed.
template <int D>
__device__ void pf2_producer(const PfParams &p, const PfMapsDev &maps, uint8_t *smem, Pf2Bars &bars, int n_units,
                             int lane, int rank, int which)
{
    using C = Pf2Cfg<D>;
    const int Hkv = p.num_kv_heads;
    const int P = 1 << p.page_shift;
    const int bsh = p.box_shift; // min(P, 64) tokens per box
    const int BT = 1 << bsh;
    const bool is_k = which == 0;
    const uint32_t box = is_k ? (uint32_t)BT * D * 2 : (uint32_t)BT * (D / 2) * 2;
    const CUtensorMap *map = is_k ? &maps.k : &maps.v;
    const int ring = is_k ? C::kKStages : C::kVStages;
    const bool nhd = p.layout == PKV_NHD;
    const int r2 = rank & 1;                                   // rank in the pair
    const int c2 = is_k ? 0 : r2 * (D / 128);                 // V: this CTA's 64-column blocks
    const int span = is_k ? kPfTile : kPfStep;                // tokens of an item
    const int lane0 = is_k ? (r2 * kPfTile) >> bsh : 0;       // page lane of the item's first box
    // barrier (and parity) that completes once the pair's MMAs have read the item of step j
    auto released = [&](int j) { return is_k ? &bars.s_full[j & 1] : &bars.o_done[j & 1]; };
    auto released_par = [&](int j) { return (uint32_t)(j >> 1) & 1u; };
    int gs = 0; // items issued so far (one per step)
    bool ok = true;
    for (int k = 0; ok; ++k) {
        const int u = pf_unit_at(k, p.cluster);
        if (u >= n_units)
            break;
        const int grp = u / Hkv, g = u - grp * Hkv;
        const PfUnit un = p.units[grp];
        const int32_t *bt_row = p.block_table + (int64_t)un.b * p.max_blocks;
        const int ns = (un.n_tiles + 1) >> 1, kv = un.kv_len;
        // lane i holds the page of tokens 128t + i*BT .. (i < 128 / BT <= 16)
        auto page_ids = [&](int t) {
            const int tok = t * kPfStep + (lane << bsh);
            int id = 0;
            if ((lane << bsh) < kPfStep && t < ns && tok < kv)
                id = __ldg(bt_row + (tok >> p.page_shift));
            return id;
        };
        int ids_cur = page_ids(0), ids_next = page_ids(1);
        for (int t = 0; t < ns; ++t, ++gs) {
            const int slot = is_k ? C::k_slot(gs) : C::v_slot(gs);
            if (gs >= ring && !pf_wait_all<true>(released(gs - ring), released_par(gs - ring), bars, p.err_flag)) {
                ok = false;
                break;
            }
            uint8_t *dst = smem + C::kOffStage + slot * C::kItemBytes;
            const int t0 = t * kPfStep + (is_k ? r2 * kPfTile : 0);
            const int ntok = max(0, min(span, kv - t0));
            const int nbox = (ntok + BT - 1) >> bsh;
            if (lane == 0) // the whole item; an empty K tile completes with none
                mbar_arrive_expect_tx(&bars.full[slot], (uint32_t)nbox * box);
            // lane bx issues box bx (up to 16 per item), all in one warp instruction
            const int page = __shfl_sync(0xffffffffu, ids_cur, (lane0 + lane) & 31);
            const int bx = lane;
            if (bx < nbox) {
                const int tslot = (t0 + (bx << bsh)) & (P - 1);
                const int c3 = nhd ? (page * P + tslot) >> 3 : tslot >> 3;
                const int c4 = nhd ? g : page * Hkv + g;
                uint8_t *bdst = dst + bx * box;
                tma_load_5d_local(bdst, map, c2, c3, c4, &bars.full[slot]);
            }
            ids_cur = ids_next;
            ids_next = page_ids(t + 2);
        }
    }
    // Copies still in flight into this ring, and the pair MMAs still reading it.
    for (int j = gs > ring ? gs - ring : 0; j < gs; ++j) {
        const int slot = is_k ? C::k_slot(j) : C::v_slot(j);
        const uint32_t par = is_k ? C::k_par(j) : C::v_par(j);
        pf_wait<true>(&bars.full[slot], par, bars, p.err_flag);
        pf_wait<true>(released(j), released_par(j), bars, p.err_flag);
    }
}

// The odd CTA's MMA warp (one thread): tells the even CTA's MMA thread, item
// by item in the order the MMAs read them (K_0, K_1, V_0, K_2, V_1, ...),
// that this CTA's part of the slot has landed.
template <int D>
__device__ void pf2_relay(const PfParams &p, Pf2Bars &bars, int n_units)
{
    using C = Pf2Cfg<D>;
    const uint32_t leader = (uint32_t)(cluster_ctarank() & ~1u);
    int gs0 = 0;
    for (int k = 0;; ++k) {
        const int u = pf_unit_at(k, p.cluster);
        if (u >= n_units)
            break;
        const int ns = (p.units[u / p.num_kv_heads].n_tiles + 1) >> 1;
        for (int t = 0; t <= ns; ++t) {
            if (t < ns) {
                const int gs = gs0 + t;
                if (!pf_wait<true>(&bars.full[C::k_slot(gs)], C::k_par(gs), bars, p.err_flag))
                    return;
                mbar_arrive_remote(&bars.peer_full[C::k_slot(gs)], leader);
            }
            if (t >= 1) {
                const int gs = gs0 + t - 1;
                if (!pf_wait<true>(&bars.full[C::v_slot(gs)], C::v_par(gs), bars, p.err_flag))
                    return;
                mbar_arrive_remote(&bars.peer_full[C::v_slot(gs)], leader);
            }
        }
        gs0 += ns;
    }
}

// The even CTA's MMA thread: per step, S = Q K^T (M = 256, N = 128, Q from
// both CTAs' shared memory) into S buffer (step & 1), then O += P V for the
// previous step (P from both CTAs' TMEM as hi and lo parts).  A stage is read
// once both CTAs' parts have landed; every completion goes to both CTAs.
template <int D>
__device__ void pf2_mma(const PfParams &p, uint8_t *smem, Pf2Bars &bars, uint32_t tmem, int n_units)
{
    using C = Pf2Cfg<D>;
    constexpr uint32_t kIdescS = tc_idesc_bf16(2 * kPfRows, kPfStep, false, false);
    constexpr uint32_t kIdescO = tc_idesc_bf16(2 * kPfRows, D, false, true);
    const uint16_t kBoth = (uint16_t)(3u << (cluster_ctarank() & ~1u)); // this pair
    const uint32_t st_base = smem_addr(smem + C::kOffStage);
    const uint64_t qd = tc_sw128_desc(smem_addr(smem + C::kOffQ), 16, C::kGroupStride);
    int gs0 = 0;
    uint32_t uc = 0;
    bool issued = false;
    auto slot_ready = [&](int slot, uint32_t par) {
        return pf_wait<true>(&bars.full[slot], par, bars, p.err_flag) &&
               pf_wait<true>(&bars.peer_full[slot], par, bars, p.err_flag);
    };
    for (int k = 0;; ++k) {
        const int u = pf_unit_at(k, p.cluster);
        if (u >= n_units)
            break;
        const int ns = (p.units[u / p.num_kv_heads].n_tiles + 1) >> 1;
        if (!pf_wait<true>(&bars.q_full, uc & 1, bars, p.err_flag))
            goto done;
        for (int t = 0; t <= ns; ++t) {
            if (t < ns) { // S[gs & 1] = Q K_t^T
                const int gs = gs0 + t;
                const int stage = C::k_slot(gs);
                if (!slot_ready(stage, C::k_par(gs)))
                    goto done;
                tc_fence_after();
                issued = true;
                const uint32_t d = tmem + C::kColS + (uint32_t)(gs & 1) * kPfStep;
                const uint64_t kd = tc_sw128_desc(st_base + stage * C::kItemBytes, 16, C::kGroupStride);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t off = (uint64_t)(((kk >> 2) * 1024 + (kk & 3) * 32) >> 4);
                    tc_mma_bf16_ss_pair(d, qd + off, kd + off, kIdescS, kk > 0 ? 1u : 0u);
                }
                tc_commit_pair_mc(&bars.s_full[gs & 1], kBoth); // the last one also frees Q
            }
            if (t >= 1) { // O += P_{t-1} V_{t-1}
                const int tv = t - 1, gs = gs0 + tv;
                if (!pf_wait<true>(&bars.p_full[gs & 1], (gs >> 1) & 1, bars, p.err_flag))
                    goto done;
                if (tv == 0 && uc > 0 && !pf_wait<true>(&bars.o_free, (uc - 1) & 1, bars, p.err_flag))
                    goto done;
                const int stage = C::v_slot(gs);
                if (!slot_ready(stage, C::v_par(gs)))
                    goto done;
                tc_fence_after();
                const uint32_t pt = tmem + C::kColS + (uint32_t)(gs & 1) * kPfStep; // P of step gs
                const uint64_t vd = tc_sw128_desc(st_base + stage * C::kItemBytes, 1024, C::kVGroupStride);
#pragma unroll
                for (int kk = 0; kk < 2 * (kPfStep / 16); ++kk) { // hi part, then lo part
                    const int k8 = kk & (kPfStep / 16 - 1);      // 16-key step: keys 16 k8 .. +15
                    // P layout (see pf2_softmax): key 16 k8 is in thread half k8 >> 2, chunk (k8 >> 1) & 1
                    const uint32_t a = pt + 64 * (k8 >> 2) + 32 * ((k8 >> 1) & 1) + 8 * (k8 & 1) + 16 * (kk >> 3);
                    tc_mma_bf16_ts_pair(tmem + C::kColO, a, vd + (uint64_t)((2 * k8 * C::kVGroupStride) >> 4),
                                        kIdescO, (tv > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit_pair_mc(&bars.o_done[gs & 1], kBoth);
            }
        }
        gs0 += ns;
        ++uc;
    }
done:
    if (issued) {
        tc_commit_pair(&bars.drain);
        mbar_wait(&bars.drain, 0);
    }
}

// A unit's Q tile into the shared-memory Q operand (K-major, 128-byte
// swizzled, the layout a TMA box of 8-row groups writes): row r = query r / G,
// head r % G; rows past total_q are zeros.  Asynchronous copies (cp.async,
// completed by cp_async_wait_all): each softmax warp fetches its TMEM lane
// quarter's 32 rows, its half of head_dim, with consecutive lanes on
// consecutive 16-byte pieces of one row (32 / (D / 16) rows per instruction).
template <int D>
__device__ __forceinline__ void pf2_load_q_async(const PfParams &p, const PfUnit &un, int g, int quarter, int lane,
                                                 int half, uint8_t *q_smem, int rank)
{
    using C = Pf2Cfg<D>;
    constexpr int kPieces = D / 16;           // 16-byte pieces of half a row
    constexpr int kRows = 32 / kPieces;       // rows per instruction
    const int pc = lane % kPieces;
    const int c = half * kPieces + pc;        // 16-byte chunk of the row: block c / 8, column c % 8
#pragma unroll
    for (int s = 0; s < 32 / kRows; ++s) {
        const int r = quarter * 32 + kRows * s + lane / kPieces; // tile row
        const int tok = un.q_start + (un.t * p.cluster + rank) * p.q_tile + (r >> p.group_shift);
        const int head = g * (1 << p.group_shift) + (r & ((1 << p.group_shift) - 1));
        const bool in = tok < p.total_q;
        const uint4 *src = reinterpret_cast<const uint4 *>(p.q + ((int64_t)(in ? tok : 0) * p.num_q_heads + head) * D +
                                                           half * (D / 2)) + pc;
        uint8_t *dst = q_smem + (r >> 3) * C::kGroupStride + (r & 7) * 128 + (c >> 3) * 1024 + (((c & 7) ^ (r & 7)) << 4);
        cp_async16(dst, src, in ? 16u : 0u);
    }
}

// Softmax warps of one CTA of a pair, step by step: the same online softmax
// as pf_softmax over 128-column S buffers.  Thread half h owns S columns
// [64 h, 64 h + 64) in two 32-column chunks; chunk c's P is written over its
// own columns, hi parts at 64 h + 32 c .. +15 and lo parts at .. +16 .. +31,
// so the other half's S columns are never overwritten before they are read.
template <int D>
__device__ void pf2_softmax(const PfParams &p, uint8_t *smem, Pf2Bars &bars, uint32_t tmem, int n_units, int warp,
                            int lane, int rank)
{
    using C = Pf2Cfg<D>;
    constexpr int kChunk = 32;
    const int quarter = warp & 3;         // TMEM lanes this warp may access
    const int half = (warp - 2) >> 2;     // which half of the step's columns
    const int r = quarter * 32 + lane;    // tile row = TMEM lane
    const int st = half * kPfRows + r;    // index among the softmax threads
    const uint32_t t_row = tmem + ((uint32_t)(quarter * 32) << 16);
    float *xchg = reinterpret_cast<float *>(smem + C::kOffXchg);
    uint8_t *q_smem = smem + C::kOffQ;
    const int G = 1 << p.group_shift;
    const int q_in_tile = r >> p.group_shift;
    const int h_in_group = r & (G - 1);
    const float qs = p.q_scale;
    const float qse = qs > 0.f ? qs : 1.f;
    int gs0 = 0;
    uint32_t pair_phase = 0;

    int u = pf_unit_at(0, p.cluster);
    if (u >= n_units)
        return;
    {
        const int grp = u / p.num_kv_heads;
        pf2_load_q_async<D>(p, p.units[grp], u - grp * p.num_kv_heads, quarter, lane, half, q_smem, rank);
        cp_async_wait_all();
        fence_proxy_async_smem();
        pf_arrive_mma<true>(&bars.q_full, lane, rank);
    }
    for (int k = 0;; ++k) {
        u = pf_unit_at(k, p.cluster);
        if (u >= n_units)
            break;
        const int grp = u / p.num_kv_heads, g = u - grp * p.num_kv_heads;
        const PfUnit un = p.units[grp];
        const int ns = (un.n_tiles + 1) >> 1, kv = un.kv_len;
        const int t = un.t * p.cluster + rank;
        const int qi = t * p.q_tile + q_in_tile;
        const bool valid = qi < un.q_len;
        const int limit = min(kv - un.q_len + qi, kv - 1);
        const int limit_min = min(kv - un.q_len + t * p.q_tile, kv - 1);
        const int u_next = pf_unit_at(k + 1, p.cluster);
        float m_used = -INFINITY, l = 0.f;
        for (int j = 0; j < ns; ++j) {
            const int gs = gs0 + j;
            if (!pf_wait_all<true>(&bars.s_full[gs & 1], (gs >> 1) & 1, bars, p.err_flag))
                return;
            tc_fence_after();
            if (j == ns - 1 && u_next < n_units) {
                // this step's S MMAs were the unit's last reads of Q: fetch the next unit's
                const int pn = u_next / p.num_kv_heads;
                pf2_load_q_async<D>(p, p.units[pn], u_next - pn * p.num_kv_heads, quarter, lane, half, q_smem, rank);
            }
            const uint32_t s_col = C::kColS + (uint32_t)(gs & 1) * kPfStep + half * (kPfStep / 2);
            const bool masked = j * kPfStep + kPfStep - 1 > limit_min;
            // raw scores of chunk c (a non-positive scale applied here, a positive one in the exponent)
            auto load_chunk = [&](int c, float (&x)[kChunk]) {
                uint32_t rr[32];
                tmem_ld32(t_row + s_col + c * kChunk, rr);
#pragma unroll
                for (int i = 0; i < kChunk; ++i)
                    x[i] = __uint_as_float(rr[i]);
                if (!(qs > 0.f)) {
#pragma unroll
                    for (int i = 0; i < kChunk; ++i)
                        x[i] *= qs;
                }
                if (masked) {
                    const int tok0 = j * kPfStep + half * (kPfStep / 2) + c * kChunk;
#pragma unroll
                    for (int i = 0; i < kChunk; ++i)
                        x[i] = (tok0 + i <= limit) ? x[i] : -INFINITY;
                }
            };
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                float x[kChunk];
                load_chunk(c, x);
#pragma unroll
                for (int i = 0; i < kChunk; ++i)
                    mx = fmaxf(mx, x[i]);
            }
            float *xm = xchg + (gs & 1) * (2 * kPfRows);
            xm[half * kPfRows + r] = mx;
            if (!pf_pair_sync(bars, quarter, pair_phase, p.err_flag))
                return;
            mx = fmaxf(mx, xm[(1 - half) * kPfRows + r]);
            const float mt = mx * qse;
            const bool grow = mt > m_used + kRescaleLog2;
            float alpha = 1.f;
            if (grow) {
                alpha = ex2_approx(m_used - mt);
                l *= alpha;
                m_used = mt;
            }
            const float m_ref = m_used == -INFINITY ? 0.f : m_used;
            const float2 q2 = make_float2(qse, qse), nm2 = make_float2(-m_ref, -m_ref);
            float2 sum2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                float x[kChunk];
                load_chunk(c, x);
                uint32_t whi[kChunk / 2], wlo[kChunk / 2];
#pragma unroll
                for (int e = 0; e < kChunk / 2; ++e) {
                    const float2 a = ffma2(make_float2(x[2 * e], x[2 * e + 1]), q2, nm2);
                    const float2 pp = make_float2(ex2_approx(a.x), ex2_approx(a.y));
                    sum2 = __fadd2_rn(sum2, pp);
                    const __nv_bfloat162 hi = __floats2bfloat162_rn(pp.x, pp.y);
                    const float2 hf = __bfloat1622float2(hi);
                    const float2 d = __fadd2_rn(pp, make_float2(-hf.x, -hf.y));
                    const __nv_bfloat162 lo = __floats2bfloat162_rn(d.x, d.y);
                    whi[e] = *reinterpret_cast<const uint32_t *>(&hi);
                    wlo[e] = *reinterpret_cast<const uint32_t *>(&lo);
                }
                tmem_st16(t_row + s_col + c * kChunk, whi);
                tmem_st16(t_row + s_col + c * kChunk + kChunk / 2, wlo);
            }
            l += sum2.x + sum2.y;
            const bool rescale_o = grow && j > 0;
            if (__any_sync(0xffffffffu, rescale_o)) {
                const int gp = gs - 1;
                if (!pf_wait_all<true>(&bars.o_done[gp & 1], (gp >> 1) & 1, bars, p.err_flag))
                    return;
                tc_fence_after();
                const float a = rescale_o ? alpha : 1.f;
                for (int c = half * (D / 2); c < (half + 1) * (D / 2); c += 32) {
                    uint32_t rr[32];
                    tmem_ld32(t_row + C::kColO + c, rr);
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        rr[i] = __float_as_uint(__uint_as_float(rr[i]) * a);
                    tmem_st32(t_row + C::kColO + c, rr);
                }
            }
            // V rows at and past kv in the step hold another token's or no data: zero them
            if (j * kPfStep + kPfStep > kv) {
                const int stage = C::v_slot(gs);
                if (!pf_wait_all<true>(&bars.full[stage], C::v_par(gs), bars, p.err_flag))
                    return;
                const int r0 = kv - j * kPfStep;
                uint8_t *vb = smem + C::kOffStage + stage * C::kItemBytes;
                for (int i = st; i < (kPfStep - r0) * C::kVChunks * 8; i += kPfSoftmaxThreads) {
                    const int piece = i & 7, rest = i >> 3;
                    const int c = rest % C::kVChunks, tt = r0 + rest / C::kVChunks;
                    *reinterpret_cast<uint4 *>(vb + (tt >> 3) * C::kVGroupStride + c * 1024 + (tt & 7) * 128 +
                                               piece * 16) = make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
            }
            tc_fence_before();
            pf_arrive_mma<true>(&bars.p_full[gs & 1], lane, rank);
        }
        // The next unit's Q (copies issued at the last step) has landed.
        if (u_next < n_units) {
            cp_async_wait_all();
            fence_proxy_async_smem();
            pf_arrive_mma<true>(&bars.q_full, lane, rank);
        }
        { // epilogue: O / l -> bf16 (this half's columns), lse
            float *xl = xchg + 4 * kPfRows;
            xl[half * kPfRows + r] = l;
            if (!pf_pair_sync(bars, quarter, pair_phase, p.err_flag))
                return;
            const float lt = l + xl[(1 - half) * kPfRows + r];
            if (!pf_pair_sync(bars, quarter, pair_phase, p.err_flag))
                return;
            const int gl = gs0 + ns - 1;
            if (!pf_wait_all<true>(&bars.o_done[gl & 1], (gl >> 1) & 1, bars, p.err_flag))
                return;
            tc_fence_after();
            const float inv = lt > 0.f ? 1.f / lt : 0.f;
            const int64_t row = (int64_t)(un.q_start + qi) * p.num_q_heads + g * G + h_in_group;
            // Chunk by chunk (32 columns): every thread's 64 bytes of its row into
            // the warp's staging block (16-byte pieces XOR-swizzled by row), then
            // 4 store rounds in which lanes 4 i .. 4 i + 3 write row 8 s + i's 64
            // contiguous bytes -- 8 full 64-byte pieces per instruction instead
            // of 32 scattered 16-byte ones.
            uint8_t *stg = smem + C::kOffOut + (warp - 2) * 2048;
            const int pc = lane & 3;
            for (int c = half * (D / 2); c < (half + 1) * (D / 2); c += 32) {
                uint32_t rr[32];
                tmem_ld32(t_row + C::kColO + c, rr);
                uint32_t w[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(rr[2 * e]) * inv,
                                                                   __uint_as_float(rr[2 * e + 1]) * inv);
                    w[e] = *reinterpret_cast<const uint32_t *>(&h);
                }
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    *reinterpret_cast<uint4 *>(stg + lane * 64 + ((j ^ (lane & 3)) << 4)) =
                        make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
                __syncwarp();
#pragma unroll
                for (int sr = 0; sr < 4; ++sr) {
                    const int rw = 8 * sr + (lane >> 2);          // row of the warp's 32
                    const int r2 = quarter * 32 + rw;             // tile row
                    const int qi2 = t * p.q_tile + (r2 >> p.group_shift);
                    const uint4 v = *reinterpret_cast<const uint4 *>(stg + rw * 64 + ((pc ^ (rw & 3)) << 4));
                    if (qi2 < un.q_len) {
                        const int64_t row2 = (int64_t)(un.q_start + qi2) * p.num_q_heads + g * G + (r2 & (G - 1));
                        *reinterpret_cast<uint4 *>(p.out + row2 * D + c + pc * 8) = v;
                    }
                }
                __syncwarp(); // the block is rewritten by the next chunk
            }
            tc_fence_before();
            pf_arrive_mma<true>(&bars.o_free, lane, rank);
            if (half == 0 && valid && p.lse != nullptr)
                p.lse[row] = (m_used + log2f(lt)) * kLn2;
        }
        gs0 += ns;
    }
}

template <int D>
__global__ void __launch_bounds__(kPf2Threads, 1)
    prefill2_kernel(const __grid_constant__ PfParams p, const __grid_constant__ PfMapsDev maps)
{
    using C = Pf2Cfg<D>;
    extern __shared__ unsigned char pf_smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(pf_smem_raw) + 1023) & ~uintptr_t(1023));
    Pf2Bars &bars = *reinterpret_cast<Pf2Bars *>(smem + C::kOffBar);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rank = (int)cluster_ctarank(); // 0: the even CTA of the pair, 1: the odd one
    constexpr int kWarpArrivals = 2 * kPfSoftmaxWarps; // per-warp arrivals of both CTAs' softmax warps

    if (threadIdx.x == 0) {
        mbar_init(&bars.q_full, kWarpArrivals);
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&bars.full[s], 1);
            mbar_init(&bars.peer_full[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars.s_full[i], 1);
            mbar_init(&bars.p_full[i], kWarpArrivals);
            mbar_init(&bars.o_done[i], 1);
        }
        mbar_init(&bars.o_free, kWarpArrivals);
        for (int i = 0; i < 4; ++i)
            mbar_init(&bars.pair[i], 64);
        mbar_init(&bars.drain, 1);
        bars.abort = 0;
        mbar_init_fence();
    }
    if (warp == kPfProducerWarp && lane == 0) {
        prefetch_tensormap(&maps.k);
        prefetch_tensormap(&maps.v);
    }
    if (warp == kPfMmaWarp) { // collective over the pair: both CTAs get the same columns
        tmem_alloc_pair(&bars.tmem_base, C::kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync(); // both CTAs' barriers and TMEM are ready before anything crosses over
    tc_fence_after();
    if (p.pdl) // the plan (and, in a mixed step, the append) wrote what follows
        asm volatile("griddepcontrol.wait;" ::: "memory");
    const uint32_t tmem = bars.tmem_base;
    const int n_units = *p.n_pairs * p.num_kv_heads;

    if (warp == kPfProducerWarp || warp == kPf2VWarp)
        pf2_producer<D>(p, maps, smem, bars, n_units, lane, rank, warp == kPfProducerWarp ? 0 : 1);
    else if (warp == kPfMmaWarp) {
        if (lane == 0) {
            if ((rank & 1) == 0)
                pf2_mma<D>(p, smem, bars, tmem, n_units);
            else
                pf2_relay<D>(p, bars, n_units);
        }
        __syncwarp();
    } else {
        pf2_softmax<D>(p, smem, bars, tmem, n_units, warp, lane, rank);
        cp_async_wait_all(); // a Q prefetch left in flight by an aborted unit
    }

    tc_fence_before();
    cluster_sync(); // the pair's last MMAs (on both CTAs' smem and TMEM) are complete
    tc_fence_after();
    if (warp == kPfMmaWarp)
        tmem_dealloc_pair(tmem, C::kTmemCols);
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
    if (tid == 0) {
        // a programmatic dependent (the mixed step's append) may start now
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        s_decreasing = 0;
    }
    for (int i = tid; i < kPfBuckets; i += kPlanThreads)
        s_hist[i] = 0;
    __syncthreads();

    // 1. Validate every request (one warp per request).
    const bool mixed = pp.cache_seqlens != nullptr;
    for (int b = warp; b < pp.batch; b += kPlanThreads / 32) {
        int s = pp.qo_indptr[b], e = pp.qo_indptr[b + 1], kv = 0;
        int64_t q = (int64_t)e - s;
        int bad = 0;
        if (mixed) {
            // rows of the decode kernel, or with a range it reports, are not ours
            if (s < 0 || e > pp.total_q || q <= pp.q_lo) {
                s = e = 0;
                q = 0;
            } else if (q > pp.q_max) {
                bad = PKV_ERR_QLEN;
            } else {
                const int L = pp.cache_seqlens[b];
                const int64_t keys = (int64_t)L + (pp.kv_add ? q : 0);
                if (L < 0)
                    bad = kPfZeroOnly; // inactive: zero output, no error
                else if (keys < q)
                    bad = PKV_ERR_QLEN;
                else if (keys > ((int64_t)pp.max_blocks << pp.page_shift))
                    bad = PKV_ERR_OVERFLOW;
                else
                    kv = (int)keys;
            }
        } else {
            kv = pp.kv_lens[b];
        }
        if (q != 0 && bad == 0) {
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
            if (q < 0 && !mixed)
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

    // 2. Groups of `cluster` query tiles per request, prefix sum.
    int v = 0;
    if (tid < pp.batch && s_bad[tid] == 0 && s_end[tid] > s_start[tid])
        v = ((s_end[tid] - s_start[tid] + pp.q_tile - 1) / pp.q_tile + pp.cluster - 1) / pp.cluster;
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
    // kv tiles of a group: those its last query tile needs
    auto tiles_of = [&](int b, int t) {
        const int q = s_end[b] - s_start[b];
        const int last = min(t * pp.cluster + pp.cluster - 1, (q + pp.q_tile - 1) / pp.q_tile - 1);
        return pf_tiles(s_kv[b], q, last, pp.q_tile);
    };
    auto bucket_of = [&](int b, int t) {
        const int64_t c = tiles_of(b, t);
        return (int)(c < kPfBuckets - 1 ? c : kPfBuckets - 1);
    };

    // 3. Counting sort of the groups by kv tiles, longest first.
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
            un.n_tiles = (int)tiles_of(b, t);
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
            set_error(pp.err_flag, s_bad[b] & ~kPfZeroOnly);
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
    bool pair;   // CTA-pair kernel (cta_group::2): half-tile TMA maps
    int cluster; // CTAs per cluster (one query tile each)
    const void *fn;
    uint32_t smem;
    int threads;
};

// head_dim 64 cannot be split into 64-column halves: one CTA per query tile,
// each loading its own K / V tiles.  128 and 256: CTA pairs.
const PfKernelEntry kPfTable[] = {
    {64, false, 1, reinterpret_cast<const void *>(&prefill_kernel<64>), PfCfg<64>::kSmem, kPfThreads},
    {128, true, 2, reinterpret_cast<const void *>(&prefill2_kernel<128>), Pf2Cfg<128>::kSmem, kPf2Threads},
    {256, true, 2, reinterpret_cast<const void *>(&prefill2_kernel<256>), Pf2Cfg<256>::kSmem, kPf2Threads},
};

const PfKernelEntry *pf_find(int D)
{
    for (const PfKernelEntry &e : kPfTable)
        if (e.D == D)
            return &e;
    return nullptr;
}

// Persistent grid size for clusters of `cl` CTAs: every cluster that can be
// resident at once, in CTAs (set up once per device).
int pf_grid(int device, const PfKernelEntry *e, int cl)
{
    constexpr int kDevices = 64;
    static int cache[kDevices][3][5] = {};
    if (device < 0 || device >= kDevices || cl < 1 || cl > 4)
        return cl;
    int &slot = cache[device][e - kPfTable][cl];
    if (slot == 0) {
        int n = 0;
        if (cudaFuncSetAttribute(e->fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)e->smem) == cudaSuccess) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(sm_count(device));
            cfg.blockDim = dim3(e->threads);
            cfg.dynamicSmemBytes = e->smem;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = cl;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int clusters = 0;
            if (cudaOccupancyMaxActiveClusters(&clusters, e->fn, &cfg) == cudaSuccess && clusters > 0)
                n = clusters * cl;
        }
        slot = n > 0 ? n : cl;
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
    pp.cache_seqlens = a.cache_seqlens;
    pp.q_lo = a.q_lo;
    pp.q_max = a.q_max;
    pp.kv_add = a.kv_add;
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
    pp.cluster = e->cluster;
    pp.cap_pairs = a.shape.cap_pairs;
    cudaError_t err = cudaSuccess;
    if (a.phase != kPrefillMain) {
        prefill_plan_kernel<<<1, kPlanThreads, 0, stream>>>(pp);
        if ((err = cudaGetLastError()) != cudaSuccess || a.phase == kPrefillPlan)
            return err;
    }

    PfParams p;
    p.q = static_cast<const __nv_bfloat16 *>(a.q);
    p.total_q = a.total_q;
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
    p.cluster = e->cluster;
    p.q_scale = a.q_scale;
    // after this call's own plan kernel, or after a kernel of ours that
    // waits for it (the mixed step's decode): set-up overlaps its end
    p.pdl = (a.phase == kPrefillAll || a.overlap_prior) ? 1 : 0;
    PfMapsDev m;
    m.k = maps.k;
    m.v = maps.v;

    int dev = 0;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess)
        return err;
    const int cl = e->cluster;
    int grid = pf_grid(dev, e, cl);
    const int64_t max_ctas = a.shape.cap_pairs * a.desc.num_kv_heads * cl; // one unit per cluster at least
    if (grid > max_ctas)
        grid = (int)max_ctas;
    grid = grid / cl * cl;
    if (grid < cl)
        grid = cl;
    void *args[] = {&p, &m};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(e->threads);
    cfg.dynamicSmemBytes = e->smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (p.pdl) {
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.numAttrs = 2;
    }
    return cudaLaunchKernelExC(&cfg, e->fn, args);
}

int prefill_box_tokens(int page_size)
{
    return page_size < kPfTile ? page_size : kPfTile;
}

bool encode_prefill_maps(const pkv_cache_desc &d, const void *k_cache, const void *v_cache, PrefillMaps *maps)
{
    const PfKernelEntry *e = pf_find(d.head_dim);
    if (e == nullptr)
        return false;
    void *k = const_cast<void *>(k_cache), *v = const_cast<void *>(v_cache);
    const int box = prefill_box_tokens(d.page_size);
    if (!e->pair)
        return encode_group_map(&maps->k, d, k, box) == CUDA_SUCCESS &&
               encode_group_map(&maps->v, d, v, box) == CUDA_SUCCESS;
    // K: min(P, 64) keys with all of head_dim; V: min(P, 64) keys with half of head_dim
    return encode_group_map(&maps->k, d, k, box) == CUDA_SUCCESS &&
           encode_group_map(&maps->v, d, v, box, d.head_dim / 128) == CUDA_SUCCESS;
}

} // namespace pkv
