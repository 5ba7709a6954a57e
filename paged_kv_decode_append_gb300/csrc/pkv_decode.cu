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
// GB300 design (one persistent CTA per resident slot, five warps):
//  * producer warp: streams 32-token tiles of K and V of one kv head through
//    a shared-memory ring with TMA (one box per page piece with all of
//    head_dim, landing as 8-token groups, 128-byte swizzle, L2 evict-first;
//    the lanes issue a tile's boxes together, one box each);
//    page ids are prefetched 32 at a time into registers, one window (and one
//    slice) ahead.
//  * two consumer warps: 16 token rows of every tile each, on tensor-core
//    tiles (mma.sync m16n8k16, bf16 in, fp32 accumulate) with an online
//    softmax in base 2; see consume_tile.  At the end of a slice they hand
//    their softmax state to an epilogue warp through a double-buffered
//    shared-memory slot and go straight on to the next slice.
//  * two epilogue warps (alternate slices): merge the two consumer warps'
//    states and finish the slice off the streaming path, with every global
//    input of the finish loaded before the state arrives: a unit cut into
//    n slices writes n fp32 partials;
//    the last slice to arrive (atomic ticket, never a spin) merges them by
//    log-sum-exp, folds in the new token (scored from k_new, not re-read from
//    the cache), performs the append and writes bf16 output and lse.
//  * Stream-K split: the (row, kv head, head group) units are laid end to end
//    as one list of key tokens and every CTA takes an equal contiguous slice
//    (boundaries rounded down to 32 tokens inside a unit), so one long
//    request is spread over many SMs and all CTAs finish together.  The plan
//    is rebuilt by every CTA from cache_seqlens; nothing is read back by the
//    host.  A unit slice is always the first or the last slice of its CTA,
//    so two workspace slots per CTA hold every partial.
//  * Every block_table entry is range-checked before an address is formed.
//
// Multi-query rows (the decode rows of a mixed step, pkv_mixed_attn): row b
// owns query rows qo_indptr[b] .. qo_indptr[b+1]-1 whose new tokens are
// already in the cache, so it holds kv = L + q keys and its query i sees keys
// 0 .. kv - q + i (the end-aligned causal rule of "[flashinfer] H100 D256
// paged attention cuDNN auto-dispatch", code analysis part 1).  A unit's
// columns are then (query, head) pairs, query-major, GC of them per unit:
// every K/V tile read serves all of a kv head's heads for GC / G queries, and
// the tiles past kv - q + 1 mask each column at its own limit.  Up to 16
// columns share one pass over the K/V tiles: a unit of more than 8 columns
// gives each consumer warp 8 of them over all 32 rows of a tile (one MMA
// n-tile each); both epilogue warps then finish it, 8 columns each, with a
// combine ticket per half.
#include <math.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kWarps = 2;                    // consumer warps of units up to 8 columns, 16 token rows each
constexpr int kProducerWarp = kWarps;        // warp 2
constexpr int kEpilogueWarp = kWarps + 1;    // warps 3 and 4
constexpr int kThreads = (kWarps + 3) * 32;

// Warp roles of one instantiation: two consumer warps (units of up to 8
// columns: one per 16-row half of every tile; 16-column units: one per
// 8-column half, over all 32 rows), the producer warp and two epilogue warps.
template <int GC>
struct Roles {
    static constexpr int kCons = 2;
    static constexpr int kProducer = kCons;
    static constexpr int kEpi = kCons + 1;
    static constexpr int kThreads = (kCons + 3) * 32;
};
constexpr int kTile = kDecodeTile; // tokens per pipeline tile
constexpr int kMaxGrid = 2048;     // persistent CTAs at most (workspace sizing)
constexpr int kSliceStartCost = 64; // work positions charged per unit for starting a slice
constexpr int kMinSlice = 192;      // work positions per CTA at least (> kSliceStartCost + kTile)
constexpr int kSlots = 2;          // consumer -> epilogue hand-off buffers
constexpr float kNegInf = -INFINITY;
// Growth of a score over the running maximum (base 2) that moves the maximum.
constexpr float kLazyMax = 8.f;

static_assert(kTile == 16 * kWarps, "each consumer warp owns 16 rows of a tile");

// ROW_QLEN: a malformed query length (multi-query rows): zero output.
// ROW_NONE: no output of this kernel (no query, or a row another kernel of
// the mixed step serves, or a query range outside [0, total_q)).
enum RowStatus { ROW_OK = 0, ROW_INACTIVE = 1, ROW_OVERFLOW = 2, ROW_QLEN = 3, ROW_NONE = 4 };

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
    int with_new, swizzle;
    int pdl;      // launched with programmatic dependent launch
    int early_kv; // ... and the K/V cache may be read before the preceding grid completes
    float q_scale;
    // Multi-query rows: q / out / lse are [total_q, Hq, ...] and row b owns
    // rows qo_indptr[b] .. qo_indptr[b+1]-1 (nullptr: one query per row).
    const int32_t *qo_indptr;
    int total_q, group_shift;
    int mq_hi;       // rows with 1 <= q_len <= mq_hi are this kernel's
    int mq_max;      // q_len > mq_max is malformed (PKV_ERR_QLEN) ...
    int mq_own_long; // ... and zeroed here when no other kernel serves long rows
    int mq_kv_add;   // 1: the row's new tokens are cached (kv = L + q_len); 0: kv = L
    // Step plans (plain rows only): the plan region of the workspace this
    // launch reads its plan from (PKV_DECODE_USE_PLAN), or the one the plan
    // kernel writes (PKV_DECODE_MAKE_PLAN); nullptr otherwise.
    const unsigned char *plan_in;
    unsigned char *plan_out;
};

// K/V stages in flight per CTA, as many as keep two CTAs on an SM (head_dim
// 128 with up to 4 heads per CTA: 5 stages, about 107 KB).
template <int D, int GC>
constexpr int stages_for()
{
    return D == 256 ? 3 : (D == 128 ? (GC <= 4 ? 5 : 4) : 6);
}

// Columns of one consumer warp's softmax state: 8 at most (one MMA n-tile).
template <int GC>
constexpr int warp_cols()
{
    return GC > 8 ? 8 : GC;
}

template <int D, int GC, bool MQ>
struct Smem {
    static constexpr int kGC = GC;
    static constexpr bool kMQ = MQ;
    static constexpr int kStages = stages_for<D, GC>();
    static constexpr int RC = warp_cols<GC>();
    // [stage][K|V] tiles laid out [kTile/8][D/64][8][64]: 8-token groups of
    // 128-byte rows (TMA SWIZZLE_128B when the page size allows 8-row boxes)
    __nv_bfloat16 kv[kStages][2][kTile * D];
    // per-warp softmax states of a finished slice: o (unnormalised), m, l
    static constexpr int CW = Roles<GC>::kCons;
    float red_o[kSlots][CW][RC][D];
    float red_m[kSlots][CW][RC], red_l[kSlots][CW][RC];
    int32_t red_bad[kSlots][CW];
    uint64_t full[kStages], empty[kStages];
    uint64_t epi_full[kSlots], epi_empty[kSlots];
    int32_t stage_bad[kStages];
    int32_t len[kMaxDecodeBatch];
    int32_t qlen[MQ ? kMaxDecodeBatch : 1]; // multi-query rows: q_len (-1: range outside [0, total_q))
    int32_t rowtok[kMaxDecodeBatch + 1]; // prefix of cache tokens per row
    long long rowbase[kMaxDecodeBatch + 1]; // first work position of every row
    long long work;                      // units * rowtok[batch]
    long long slice;                     // work positions per CTA
    int32_t geff;                        // CTAs that own a token slice
    int32_t n_empty;                     // rows with output units but no cached token
    int32_t abort;
    int32_t plan_state;                  // 0: planned here, 1: step plan used, 2: step plan rejected
};

// Programmatic dependent launch: wait for the preceding grid (and its memory)
// before the first access that is not cache_seqlens / block_table.
__device__ __forceinline__ void wait_prior_grid(const KParams &p)
{
    if (p.pdl)
        asm volatile("griddepcontrol.wait;" ::: "memory");
}

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

// Status of a multi-query row with L cached tokens and qn queries (qn < 0:
// a query range outside [0, total_q)); *kv gets the keys it holds.
__device__ __forceinline__ int mq_row_status(const KParams &p, int L, int qn, int *kv)
{
    *kv = 0;
    if (qn <= 0 || (qn > p.mq_hi && qn <= p.mq_max) || (qn > p.mq_max && !p.mq_own_long))
        return ROW_NONE;
    if (qn > p.mq_max)
        return ROW_QLEN;
    if (L < 0)
        return ROW_INACTIVE;
    const int64_t keys = (int64_t)L + (p.mq_kv_add ? qn : 0);
    if (keys < qn)
        return ROW_QLEN;
    if (keys > (int64_t)p.max_blocks * p.page_size)
        return ROW_OVERFLOW;
    *kv = (int)keys;
    return ROW_OK;
}

// Output units of a multi-query row: GC (query, head) columns per unit.
template <int GC>
__device__ __forceinline__ int mq_units(const KParams &p, int status, int qn)
{
    if (status == ROW_NONE)
        return 0;
    return p.num_kv_heads * (int)(((int64_t)qn * p.group + GC - 1) / GC);
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

// ------------------------------------------------------------------ plan
// Every CTA derives the same plan from cache_seqlens.  Work is laid out as a
// line: every (row, kv head, head group) unit with n > 0 cached tokens takes
// kSliceStartCost virtual positions followed by its n token positions, units
// in row-major order (multi-query rows: as many units per kv head as their
// (query, head) columns need).  CTA k takes positions [k * slice, (k+1) * slice),
// moved to token positions (see boundary), so the per-unit cost of starting
// a slice (page ids, queries, a hand-off to the epilogue) is balanced along
// with the tokens.
template <class SM>
__device__ void build_plan_rows(const KParams &p, SM &sm, int grid)
{
    for (int i = threadIdx.x; i < p.batch; i += blockDim.x)
        sm.len[i] = p.seqlens[i];
    __syncthreads();
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        int run = 0, nonempty = 0;
        for (int base = 0; base < p.batch; base += 32) {
            const int i = base + lane;
            int n = 0;
            if (i < p.batch) {
                const int L = sm.len[i];
                n = row_status(p, L) == ROW_OK ? L : 0;
            }
            const unsigned ne = __ballot_sync(0xffffffffu, n > 0);
            const int ne_before = nonempty + __popc(ne & ((1u << lane) - 1u));
            nonempty += __popc(ne);
            int incl = n;
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o)
                    incl += v;
            }
            if (i < p.batch) {
                sm.rowtok[i] = run + incl - n;
                sm.rowbase[i] = (long long)p.units * ((long long)(run + incl - n) + (long long)kSliceStartCost * ne_before);
            }
            run += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) {
            sm.rowtok[p.batch] = run;
            sm.rowbase[p.batch] = (long long)p.units * ((long long)run + (long long)kSliceStartCost * nonempty);
            const long long work = (long long)p.units * ((long long)run + (long long)kSliceStartCost * nonempty);
            long long g = work / kMinSlice;
            if (g > grid)
                g = grid;
            if (g < 1)
                g = 1;
            const long long slice = work > 0 ? (work + g - 1) / g : 1;
            sm.work = work;
            sm.slice = slice;
            sm.n_empty = p.batch - nonempty;
            sm.geff = work > 0 ? (int)((work + slice - 1) / slice) : 1;
        }
    }
    __syncthreads();
}

// Multi-query rows: units per row differ, so the work positions are summed directly.
template <class SM>
__device__ void build_plan_mq(const KParams &p, SM &sm, int grid)
{
    constexpr int GC = SM::kGC;
    for (int i = threadIdx.x; i < p.batch; i += blockDim.x) {
        sm.len[i] = p.seqlens[i];
        const int s = p.qo_indptr[i], e = p.qo_indptr[i + 1];
        sm.qlen[i] = (s < 0 || e > p.total_q || e < s) ? -1 : e - s;
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        int run = 0, empty = 0;
        long long wrun = 0;
        for (int base = 0; base < p.batch; base += 32) {
            const int i = base + lane;
            int n = 0, u = 0; // cached tokens read, output units
            if (i < p.batch) {
                int kv;
                const int st = mq_row_status(p, sm.len[i], sm.qlen[i], &kv);
                n = kv;
                u = mq_units<GC>(p, st, sm.qlen[i]);
            }
            // work positions of the row: every unit costs the slice start plus its tokens
            const long long w = n > 0 ? (long long)u * (n + kSliceStartCost) : 0;
            empty += __popc(__ballot_sync(0xffffffffu, n == 0 && u > 0));
            int incl = n;
            long long wincl = w;
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, o);
                const long long wv = __shfl_up_sync(0xffffffffu, wincl, o);
                if (lane >= o) {
                    incl += v;
                    wincl += wv;
                }
            }
            if (i < p.batch) {
                sm.rowtok[i] = run + incl - n;
                sm.rowbase[i] = wrun + wincl - w;
            }
            run += __shfl_sync(0xffffffffu, incl, 31);
            wrun += __shfl_sync(0xffffffffu, wincl, 31);
        }
        if (lane == 0) {
            sm.rowtok[p.batch] = run;
            sm.rowbase[p.batch] = wrun;
            const long long work = wrun;
            long long g = work / kMinSlice;
            if (g > grid)
                g = grid;
            if (g < 1)
                g = 1;
            const long long slice = work > 0 ? (work + g - 1) / g : 1;
            sm.work = work;
            sm.slice = slice;
            sm.n_empty = empty;
            sm.geff = work > 0 ? (int)((work + slice - 1) / slice) : 1;
        }
    }
    __syncthreads();
}

// grid: the CTAs of the decode launch the plan is for.
template <class SM>
__device__ __forceinline__ void build_plan(const KParams &p, SM &sm, int grid)
{
    if constexpr (SM::kMQ)
        build_plan_mq(p, sm, grid);
    else
        build_plan_rows(p, sm, grid);
}

// Unit containing work position x (x < work): row b, unit r in the row and
// the offset rel inside the unit's kSliceStartCost + n positions; returns the
// unit's first token position.  units * (row tokens + cost) < 2^31 (checked
// on the host), so in-row math is 32-bit.
template <class SM>
__device__ __forceinline__ long long locate(const KParams &p, const SM &sm, long long x, int &b, int &r, int &rel)
{
    int lo = 0, hi = p.batch - 1; // largest row starting at or before x (never an empty row)
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (sm.rowbase[mid] <= x)
            lo = mid;
        else
            hi = mid - 1;
    }
    b = lo;
    const long long base = sm.rowbase[lo];
    const int w = sm.rowtok[lo + 1] - sm.rowtok[lo] + kSliceStartCost;
    const int d = (int)(x - base);
    r = d / w;
    rel = d - r * w;
    return base + (long long)r * w + kSliceStartCost;
}

// First position of CTA k's range (k in [0, geff]): k * slice moved to a
// token position -- the unit's first token if it falls on the unit's virtual
// positions, else rounded down to a multiple of the tile inside the unit.
template <class SM>
__device__ __forceinline__ long long boundary(const KParams &p, const SM &sm, int k)
{
    const long long x = (long long)k * sm.slice;
    if (x >= sm.work)
        return sm.work;
    int b, r, rel;
    const long long t0 = locate(p, sm, x, b, r, rel);
    const int t = rel - kSliceStartCost;
    return t0 + (t < 0 ? 0 : (t & ~(kTile - 1)));
}

// CTA whose range holds token position x (x < work): close to x / slice, the
// boundaries being at most kTile below or kSliceStartCost above k * slice.
template <class SM>
__device__ __forceinline__ int owner_of(const KParams &p, const SM &sm, long long x)
{
    int k = (int)(x / sm.slice);
    if (k > sm.geff - 1)
        k = sm.geff - 1;
    while (k + 1 < sm.geff && boundary(p, sm, k + 1) <= x)
        ++k;
    while (k > 0 && boundary(p, sm, k) > x)
        --k;
    return k;
}

struct Seg {
    int b, r, kvh, sub, unit, L, status, tok0, tok1;
    long long u0; // unit's first token position
    int n;        // unit's cache tokens
    int qn, qs;   // multi-query rows: queries and the first query row (else 1, b)
    int mask_from; // first token some column of the unit may not see (n: none)
};

// Row-level fields of unit r of row b (everything but the token range).
template <class SM>
__device__ __forceinline__ void seg_unit(const KParams &p, const SM &sm, Seg &s, int b, int r)
{
    constexpr int GC = SM::kGC;
    constexpr bool MQ = SM::kMQ;
    s.b = b;
    s.r = r;
    s.unit = b * p.units + r;
    s.L = sm.len[b];
    if constexpr (MQ) {
        int kv;
        s.qn = sm.qlen[b];
        s.status = mq_row_status(p, s.L, s.qn, &kv);
        const int n_sub = max(1, (int)(((int64_t)s.qn * p.group + GC - 1) / GC));
        s.kvh = r / n_sub;
        s.sub = r - s.kvh * n_sub;
        s.qs = s.status == ROW_NONE ? 0 : p.qo_indptr[b];
        // column c of the unit is query (sub * GC + c) >> group_shift, which sees kv - qn + query + 1 keys
        s.mask_from = kv - s.qn + ((s.sub * GC) >> p.group_shift) + 1;
    } else {
        s.qn = 1;
        s.qs = b;
        s.status = row_status(p, s.L);
        s.kvh = r / p.n_sub;
        s.sub = r - s.kvh * p.n_sub;
        s.mask_from = 0x7fffffff;
    }
}

// Walks the slices of one CTA's range [pos0, end), one unit each.  The two
// boundary slices come first (the range's first and last unit, the only ones
// that can be shared with a neighbouring CTA), then the whole units between
// them, so the partial-merging work of shared units is not left for the end.
struct SegIter {
    long long pos0, end, f_end, mid_pos, mid_end;
    long long t0_f, t0_l;
    int b_f, r_f, b_l, r_l;
    int stage; // 0: first slice, 1: last slice, 2: middle units, 3: done
    template <class SM>
    __device__ __forceinline__ void init(const KParams &p, const SM &sm, int k)
    {
        stage = 3;
        if (k >= sm.geff)
            return;
        const long long x = (long long)k * sm.slice;
        if (x >= sm.work)
            return;
        int rel;
        t0_f = locate(p, sm, x, b_f, r_f, rel); // the unit of this range's first token
        const int t = rel - kSliceStartCost;
        pos0 = t0_f + (t < 0 ? 0 : (t & ~(kTile - 1)));
        end = boundary(p, sm, k + 1);
        if (pos0 >= end)
            return;
        f_end = min(end, t0_f + (sm.rowtok[b_f + 1] - sm.rowtok[b_f]));
        stage = 0;
    }
    template <class SM>
    __device__ __forceinline__ void fill(const KParams &p, const SM &sm, Seg &s, int b, int r, long long t0,
                                         long long from, long long to)
    {
        seg_unit(p, sm, s, b, r);
        s.u0 = t0;
        s.n = sm.rowtok[b + 1] - sm.rowtok[b];
        s.tok0 = (int)(from - t0);
        s.tok1 = (int)(to - t0);
    }
    template <class SM>
    __device__ __forceinline__ bool next(const KParams &p, const SM &sm, Seg &s)
    {
        if (stage == 0) {
            fill(p, sm, s, b_f, r_f, t0_f, pos0, f_end);
            stage = 3;
            if (f_end < end) {
                int rel;
                t0_l = locate(p, sm, end - 1, b_l, r_l, rel);
                mid_pos = f_end; // virtual start of the next unit
                if (end > t0_l) { // the range ends inside a unit's tokens
                    mid_end = t0_l - kSliceStartCost;
                    stage = 1;
                } else {
                    mid_end = end;
                    stage = 2;
                }
            }
            return true;
        }
        if (stage == 1) {
            fill(p, sm, s, b_l, r_l, t0_l, t0_l, end);
            stage = 2;
            return true;
        }
        if (stage == 2 && mid_pos < mid_end) {
            int b, r, rel;
            const long long t0 = locate(p, sm, mid_pos, b, r, rel); // rel == 0: a unit's virtual start
            if (t0 < mid_end) {
                const long long e = t0 + (sm.rowtok[b + 1] - sm.rowtok[b]);
                fill(p, sm, s, b, r, t0, t0, e);
                mid_pos = e;
                return true;
            }
        }
        stage = 3;
        return false;
    }
};

// ---------------------------------------------------------------- step plans
// A step plan (PKV_DECODE_MAKE_PLAN) is the shared-memory plan above written
// to the workspace, plus one record per CTA of the decode launch: its
// SegIter after the first slice was taken, that slice, and the page ids of
// the slice's first window.  A later launch of the same step
// (PKV_DECODE_USE_PLAN) copies the plan instead of deriving it, and its
// producer issues the first tile straight from the record.
constexpr uint32_t kPlanMagic = 0x31564b50u; // "PKV1"
constexpr int kPlanRecBytes = 256;

struct PlanHeader {
    uint32_t magic;
    int32_t batch, units, grid, max_blocks, page_size, with_new, num_kv_heads;
    long long work, slice;
    int32_t geff, n_empty;
};

struct PlanRec {
    SegIter si; // after the first next()
    int32_t have, b, kvh, tok0, tok1;
    int32_t pages[32];
};
static_assert(sizeof(PlanRec) <= kPlanRecBytes, "plan record");

// A CTA's record as its producer warp holds it (win: page id `lane` of the
// first window).
struct RecRegs {
    SegIter si;
    int have, b, kvh, tok0, tok1, win;
};
static_assert(sizeof(PlanHeader) <= 256, "plan header");

// Offsets (bytes, from the plan region's start) of a plan for `batch` rows.
struct PlanLayout {
    size_t len, rowtok, rowbase, recs, bytes;
};

__host__ __device__ inline PlanLayout plan_layout(int batch)
{
    auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
    PlanLayout l;
    l.len = 256;
    l.rowtok = l.len + al(4 * (size_t)batch);
    l.rowbase = l.rowtok + al(4 * ((size_t)batch + 1));
    l.recs = l.rowbase + al(8 * ((size_t)batch + 1));
    l.bytes = l.recs + (size_t)kMaxGrid * kPlanRecBytes;
    return l;
}

// The plan's header matches this launch (every thread takes the same decision).
__device__ __forceinline__ bool plan_matches(const KParams &p, const PlanHeader *h)
{
    return __ldcg(&h->magic) == kPlanMagic && __ldcg(&h->batch) == p.batch && __ldcg(&h->units) == p.units &&
           __ldcg(&h->grid) == (int)gridDim.x && __ldcg(&h->max_blocks) == p.max_blocks &&
           __ldcg(&h->page_size) == p.page_size && __ldcg(&h->with_new) == p.with_new &&
           __ldcg(&h->num_kv_heads) == p.num_kv_heads;
}

// Copy of a plain-old-data record from global memory, bypassing L1 (the plan
// of an earlier kernel).
template <class T>
__device__ __forceinline__ T ldcg_pod(const T *src)
{
    static_assert(sizeof(T) % 4 == 0, "whole words");
    T v;
    const int *s = reinterpret_cast<const int *>(src);
    int *d = reinterpret_cast<int *>(&v);
#pragma unroll
    for (int i = 0; i < (int)(sizeof(T) / 4); ++i)
        d[i] = __ldcg(s + i);
    return v;
}

// ---------------------------------------------------------------- producer
// Page ids of 32 consecutive blocks of a row, one per lane (0 past `last`).
__device__ __forceinline__ int load_window(const int32_t *bt_row, int first, int last, int lane)
{
    return first + lane <= last ? bt_row[first + lane] : 0;
}

// rec: this CTA's record of a step plan (its SegIter, first slice and first
// page ids), loaded into registers before the shared-memory plan is ready.
// The first tile is then issued at once; the producer meets the other warps
// at named barrier 2 (the plan written to shared memory) right after it.
template <int D, int GC, bool MQ>
__device__ void producer(const KParams &p, Smem<D, GC, MQ> &sm, const DecodeMaps *maps, const RecRegs *rec)
{
    constexpr int S = Smem<D, GC, MQ>::kStages;
    const int lane = threadIdx.x & 31;
    const uint64_t policy = l2_evict_first_policy();
    const int box = p.box_tokens;
    // a partly used box is fetched in 8-row pieces (rows past the slice are not read)
    const bool split_tail = box > kDecodeSmallBox;
    uint32_t g_tile = 0;
    volatile int32_t *abort = &sm.abort;
    SegIter si;
    Seg sg, nx;
    bool have;
    int win; // first window of the current slice, prefetched one slice ahead
    if (rec != nullptr) {
        si = rec->si;
        have = rec->have != 0;
        sg.b = rec->b;
        sg.kvh = rec->kvh;
        sg.tok0 = rec->tok0;
        sg.tok1 = rec->tok1;
        win = rec->win;
        // the record is only trusted as far as its addresses go: one that
        // names no valid row, kv head or token range stops the CTA (the other
        // warps' bounded waits then end, PKV_ERR_TIMEOUT), never forms an address
        if (have && (sg.b < 0 || sg.b >= p.batch || sg.kvh < 0 || sg.kvh >= p.num_kv_heads || sg.tok0 < 0 ||
                     sg.tok1 <= sg.tok0 || sg.tok1 > p.max_blocks * p.page_size)) {
            have = false;
            if (lane == 0)
                sm.abort = 1;
        }
    } else {
        si.init(p, sm, blockIdx.x);
        have = si.next(p, sm, sg);
        win = have ? load_window(p.block_table + (int64_t)sg.b * p.max_blocks, sg.tok0 >> p.page_shift,
                                 (sg.tok1 - 1) >> p.page_shift, lane)
                   : 0;
    }
    bool met = rec == nullptr; // met the other warps at named barrier 2
    // live page ids of the record's window, checked against it after the first slice
    int live0 = 0;
    const int rec0 = win;
    const int32_t *rec_row = rec != nullptr && have ? p.block_table + (int64_t)sg.b * p.max_blocks : nullptr;
    const int rec_first = have ? sg.tok0 >> p.page_shift : 0, rec_last = have ? (sg.tok1 - 1) >> p.page_shift : -1;
    // Page ids are loading.  K/V come after the preceding grid unless the
    // caller declared that it does not write this call's cache; the error
    // flag always does (below).
    if (!p.early_kv)
        wait_prior_grid(p);
    while (have && !*abort) {
        const int32_t *bt_row = p.block_table + (int64_t)sg.b * p.max_blocks;
        const int last_pg = (sg.tok1 - 1) >> p.page_shift;
        int wbase = sg.tok0 >> p.page_shift;
        int nxt = load_window(bt_row, wbase + 32, last_pg, lane);
        bool more = false;
        int nwin = 0;
        const int n_tiles = (sg.tok1 - sg.tok0 + kTile - 1) / kTile;
        for (int t = 0; t < n_tiles; ++t, ++g_tile) {
            const int s = g_tile % S;
            const uint32_t use = g_tile / S;
            if (use > 0 && !wait_or_abort(&sm.empty[s], (use - 1) & 1u, abort))
                break;
            const int tile0 = sg.tok0 + t * kTile;
            const int nv = min(kTile, sg.tok1 - tile0);
            const int nbox = (nv + box - 1) / box;
            const int nfull = split_tail ? nv / box : nbox;
            const int tail_rows = split_tail ? ((nv - nfull * box + kDecodeSmallBox - 1) & ~(kDecodeSmallBox - 1)) : 0;
            if ((tile0 >> p.page_shift) >= wbase + 32) { // tiles never straddle a window
                wbase += 32;
                win = nxt;
                nxt = load_window(bt_row, wbase + 32, last_pg, lane);
            }
            // page of box `lane` (lanes >= nbox carry junk and are not used)
            const int mine = __shfl_sync(0xffffffffu, win, (((tile0 + lane * box) >> p.page_shift) - wbase) & 31);
            const bool ok = lane < nbox && mine >= 1 && mine < p.num_pages;
            const unsigned okmask = __ballot_sync(0xffffffffu, ok);
            const int bad = __popc(okmask) != nbox;
            if (lane == 0) {
                const unsigned fullmask = nfull >= 32 ? 0xffffffffu : ((1u << nfull) - 1u);
                const uint32_t rows = (uint32_t)box * __popc(okmask & fullmask) +
                                      (nfull < nbox && ((okmask >> nfull) & 1u) ? (uint32_t)tail_rows : 0u);
                sm.stage_bad[s] = bad;
                mbar_arrive_expect_tx(&sm.full[s], 2u * rows * D * 2u);
            }
            __syncwarp();
            // one lane per box (after lane 0's expect_tx, ordered by the __syncwarp above)
            {
                const int bx = lane, page = mine;
                if (bx < nbox && ((okmask >> bx) & 1u)) {
                    const int slot = (tile0 + bx * box) & (p.page_size - 1);
                    int y, z;
                    if (p.layout == PKV_NHD) {
                        y = sg.kvh;
                        z = page * p.page_size + slot;
                    } else {
                        y = slot;
                        z = page * p.num_kv_heads + sg.kvh;
                    }
                    // A stage is [kTile / 8 token groups][D / 64 column blocks][8 rows][64]
                    // (group_off: element offset of token row `row`'s group).
                    auto group_off = [](int row) { return (row >> 3) * (8 * D); };
                    if (p.swizzle) { // token-group boxes: all of head_dim for box (or 8) tokens at once
                        if (bx < nfull) {
                            const int off = group_off(bx * box);
                            const int c3 = p.layout == PKV_NHD ? (page * p.page_size + slot) >> 3 : slot >> 3;
                            const int c4 = p.layout == PKV_NHD ? sg.kvh : page * p.num_kv_heads + sg.kvh;
                            tma_load_5d(sm.kv[s][0] + off, &maps->k, 0, 0, 0, c3, c4, &sm.full[s], policy);
                            tma_load_5d(sm.kv[s][1] + off, &maps->v, 0, 0, 0, c3, c4, &sm.full[s], policy);
                        } else { // the slice ends inside this box: 8-token groups up to its end
                            for (int r = 0; r < tail_rows; r += kDecodeSmallBox) {
                                const int off = group_off(bx * box + r);
                                const int c3 = p.layout == PKV_NHD ? (page * p.page_size + slot + r) >> 3
                                                                   : (slot + r) >> 3;
                                const int c4 = p.layout == PKV_NHD ? sg.kvh : page * p.num_kv_heads + sg.kvh;
                                tma_load_5d(sm.kv[s][0] + off, &maps->k8, 0, 0, 0, c3, c4, &sm.full[s], policy);
                                tma_load_5d(sm.kv[s][1] + off, &maps->v8, 0, 0, 0, c3, c4, &sm.full[s], policy);
                            }
                        }
                    } else { // pages of 1, 2 or 4 tokens: 64-column boxes inside one token group
                        const int row = bx * box;
#pragma unroll
                        for (int h = 0; h < D / 64; ++h) {
                            const int off = group_off(row) + h * 512 + (row & 7) * 64;
                            tma_load_3d(sm.kv[s][0] + off, &maps->k, 64 * h, y, z, &sm.full[s], policy);
                            tma_load_3d(sm.kv[s][1] + off, &maps->v, 64 * h, y, z, &sm.full[s], policy);
                        }
                    }
                }
            }
            if (lane == 0 && bad) {
                wait_prior_grid(p);
                set_error(p.err_flag, PKV_ERR_PAGE);
            }
            __syncwarp();
            if (t == 0) { // next slice and its first page window, off the first tile's critical path
                if (!met) {
                    named_sync(2, Roles<GC>::kThreads); // the shared-memory plan is written
                    met = true;
                }
                if (rec_row != nullptr)
                    live0 = load_window(rec_row, rec_first, rec_last, lane);
                more = si.next(p, sm, nx);
                nwin = more ? load_window(p.block_table + (int64_t)nx.b * p.max_blocks, nx.tok0 >> p.page_shift,
                                          (nx.tok1 - 1) >> p.page_shift, lane)
                            : 0;
            }
        }
        if (rec_row != nullptr) { // the record's window against the live table
            if (__any_sync(0xffffffffu, live0 != rec0) && lane == 0) {
                wait_prior_grid(p);
                set_error(p.err_flag, PKV_ERR_PLAN);
            }
            rec_row = nullptr;
        }
        have = more;
        sg = nx;
        win = nwin;
    }
    if (!met)
        named_sync(2, Roles<GC>::kThreads); // no tile issued: still meet the other warps
    // After an abort, let copies already issued land before the CTA exits.
    if (*abort && lane == 0) {
        const uint32_t first = g_tile > (uint32_t)S ? g_tile - S : 0;
        for (uint32_t g = first; g < g_tile; ++g)
            (void)mbar_wait(&sm.full[g % S], (g / S) & 1u);
    }
}

// ---------------------------------------------------------------- consumers
// Each consumer warp owns 16 of a tile's 32 token rows.  Tensor-core tiles
// (mma.sync m16n8k16, bf16 in, fp32 accumulate) put the tokens on the M side
// so only the 8-wide head side is padded (GC <= 8 heads share one kv head):
//   S^T[16 tok][8 heads] = K[16 tok][D] . Q^T[D][8 heads]
//   O^T[D][8 heads]     += V^T[D][16 tok] . P^T[16 tok][8 heads]
// P^T moves from the accumulator layout to the B-operand layout with
// movmatrix (an in-register 8x8 transpose).  P is split into bf16 high and
// low parts (two MMAs) so the weights carry ~16 significant bits.

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a)
{
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ float2 unpack_bf16(uint32_t w)
{
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// Shared-memory byte address of the 16-byte chunk `chunk` (0..D/8-1) of token
// row `row` in a [kTile/8][D/64][8][64] tile (8-token groups, each 8 rows of
// every 64-column block); with swz = 7 the 128-byte rows are stored TMA
// SWIZZLE_128B style (chunk index XOR row % 8).
template <int D>
__device__ __forceinline__ uint32_t tile_addr(uint32_t base, int row, int chunk, int swz)
{
    const int blk = chunk >> 3, c = chunk & 7;
    return base + (uint32_t)((((row >> 3) * (D / 64) + blk) * 8 + (row & 7)) * 128 + ((c ^ (row & swz)) << 4));
}

// MASKED: token rows >= nv hold no token, and column 2c + j (c = lane & 3)
// sees only the tile's rows below lim[j] (multi-query rows; else lim >= nv).
// half: the 16-row half of the tile this warp takes.  Warps that share a half
// (16-column units) zero the same masked V rows, each before its own reads.
template <int D, bool MASKED, bool MQ>
__device__ __forceinline__ void consume_tile(const __nv_bfloat16 *Kt, __nv_bfloat16 *Vt, int nv, int lim0, int lim1,
                                             int half, int lane, int swz, float scale,
                                             const uint32_t (&qf)[D / 16][2], float (&acc)[D / 16][4],
                                             float (&m_run)[2], float (&l_run)[2])
{
    constexpr int KS = D / 16;
    const int row0 = half * 16;
    const int g = lane >> 2;
    const uint32_t kbase = smem_addr(Kt), vbase = smem_addr(Vt);
    if (MASKED && nv < row0 + 16) {
        // zero V rows of masked tokens: P is 0 there, but 0 * NaN would not be
        const int first = nv > row0 ? nv : row0;
        for (int i = lane; i < (row0 + 16 - first) * (D / 8); i += 32) {
            const int r = first + i / (D / 8), chunk = i % (D / 8);
            *reinterpret_cast<uint4 *>(Vt + (((r >> 3) * (D / 64) + (chunk >> 3)) * 8 + (r & 7)) * 64 +
                                       (chunk & 7) * 8) = make_uint4(0u, 0u, 0u, 0u);
        }
        __syncwarp();
    }
    // ---- S^T = K Q^T, two accumulators for two independent MMA chains
    float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
    const int krow = row0 + (lane & 15);
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
        uint32_t a[4];
        ldsm_x4(tile_addr<D>(kbase, krow, 2 * ks + (lane >> 4), swz), a);
        if (ks & 1)
            mma_16816(sb, a, qf[ks][0], qf[ks][1]);
        else
            mma_16816(sa, a, qf[ks][0], qf[ks][1]);
    }
    float v[4]; // rows g (v[0], v[1]) and g+8 (v[2], v[3]); heads 2c, 2c+1
#pragma unroll
    for (int i = 0; i < 4; ++i)
        v[i] = (sa[i] + sb[i]) * scale;
    if constexpr (MASKED && MQ) {
        const int e0 = min(nv, lim0), e1 = min(nv, lim1);
        if (row0 + g >= e0)
            v[0] = kNegInf;
        if (row0 + g >= e1)
            v[1] = kNegInf;
        if (row0 + g + 8 >= e0)
            v[2] = kNegInf;
        if (row0 + g + 8 >= e1)
            v[3] = kNegInf;
    } else if constexpr (MASKED) {
        if (row0 + g >= nv)
            v[0] = v[1] = kNegInf;
        if (row0 + g + 8 >= nv)
            v[2] = v[3] = kNegInf;
    }
    // ---- online softmax per head column.  Lazy maximum: the running maximum
    // moves (a reduction over the 8 row groups, then a rescale) only when a
    // score exceeds it by more than kLazyMax; until then the exponentials use
    // the older maximum, which is exact in real arithmetic and keeps every
    // p below 2^kLazyMax.
    bool grow = false;
#pragma unroll
    for (int j = 0; j < 2; ++j)
        grow |= fmaxf(v[j], v[2 + j]) > m_run[j] + kLazyMax;
    if (__any_sync(0xffffffffu, grow)) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            float mt = fmaxf(v[j], v[2 + j]);
            mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 4));
            mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 8));
            mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 16));
            const float m_new = fmaxf(m_run[j], mt);
            const float a = m_new == kNegInf ? 1.f : ex2(m_run[j] - m_new);
            l_run[j] *= a;
#pragma unroll
            for (int mt2 = 0; mt2 < KS; ++mt2) {
                acc[mt2][j] *= a;
                acc[mt2][2 + j] *= a;
            }
            m_run[j] = m_new;
        }
    }
    float pr[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float m = m_run[i & 1];
        pr[i] = ex2(v[i] - (m == kNegInf ? 0.f : m)); // masked: ex2(-inf) = 0
    }
    l_run[0] += pr[0] + pr[2];
    l_run[1] += pr[1] + pr[3];
    // ---- P^T as B fragments: high and low bf16 parts, transposed in registers
    const uint32_t h01 = pack_bf16(pr[0], pr[1]), h23 = pack_bf16(pr[2], pr[3]);
    const float2 f01 = unpack_bf16(h01), f23 = unpack_bf16(h23);
    const uint32_t l01 = pack_bf16(pr[0] - f01.x, pr[1] - f01.y), l23 = pack_bf16(pr[2] - f23.x, pr[3] - f23.y);
    const uint32_t bh0 = movmatrix_trans(h01), bh1 = movmatrix_trans(h23);
    const uint32_t bl0 = movmatrix_trans(l01), bl1 = movmatrix_trans(l23);
    // ---- O^T += V^T P^T
    const int vrow = row0 + (lane & 7) + ((lane >> 4) << 3);
    const int vchunk = (lane >> 3) & 1;
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
        uint32_t a[4];
        ldsm_x4_trans(tile_addr<D>(vbase, vrow, 2 * mt + vchunk, swz), a);
        mma_16816(acc[mt], a, bh0, bh1);
        mma_16816(acc[mt], a, bl0, bl1);
    }
}

// A 16-column unit's tile for one consumer warp: its 8 columns over all 32
// token rows, as two 16-row halves that share one online-softmax update.
// MASKED as in consume_tile; both warps zero the masked V rows they read
// (the same zeros, written before either warp's own reads).
template <int D, bool MASKED>
__device__ __forceinline__ void consume_tile_wide(const __nv_bfloat16 *Kt, __nv_bfloat16 *Vt, int nv, int lim0,
                                                  int lim1, int lane, int swz, float scale,
                                                  const uint32_t (&qf)[D / 16][2], float (&acc)[D / 16][4],
                                                  float (&m_run)[2], float (&l_run)[2])
{
    constexpr int KS = D / 16;
    const int g = lane >> 2;
    const uint32_t kbase = smem_addr(Kt), vbase = smem_addr(Vt);
    if (MASKED && nv < kTile) {
        for (int i = lane; i < (kTile - nv) * (D / 8); i += 32) {
            const int r = nv + i / (D / 8), chunk = i % (D / 8);
            *reinterpret_cast<uint4 *>(Vt + (((r >> 3) * (D / 64) + (chunk >> 3)) * 8 + (r & 7)) * 64 +
                                       (chunk & 7) * 8) = make_uint4(0u, 0u, 0u, 0u);
        }
        __syncwarp();
    }
    // ---- S^T = K Q^T for rows 16h .. 16h + 15
    float v[2][4];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
        const int krow = 16 * h + (lane & 15);
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            uint32_t a[4];
            ldsm_x4(tile_addr<D>(kbase, krow, 2 * ks + (lane >> 4), swz), a);
            if (ks & 1)
                mma_16816(sb, a, qf[ks][0], qf[ks][1]);
            else
                mma_16816(sa, a, qf[ks][0], qf[ks][1]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
            v[h][i] = (sa[i] + sb[i]) * scale;
        if constexpr (MASKED) {
            const int e0 = min(nv, lim0), e1 = min(nv, lim1), r = 16 * h + g;
            if (r >= e0)
                v[h][0] = kNegInf;
            if (r >= e1)
                v[h][1] = kNegInf;
            if (r + 8 >= e0)
                v[h][2] = kNegInf;
            if (r + 8 >= e1)
                v[h][3] = kNegInf;
        }
    }
    // ---- online softmax per column over both halves (lazy maximum, as in
    // consume_tile)
    bool grow = false;
#pragma unroll
    for (int j = 0; j < 2; ++j)
        grow |= fmaxf(fmaxf(v[0][j], v[0][2 + j]), fmaxf(v[1][j], v[1][2 + j])) > m_run[j] + kLazyMax;
    if (__any_sync(0xffffffffu, grow)) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            float mt = fmaxf(fmaxf(v[0][j], v[0][2 + j]), fmaxf(v[1][j], v[1][2 + j]));
            mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 4));
            mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 8));
            mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 16));
            const float m_new = fmaxf(m_run[j], mt);
            const float a = m_new == kNegInf ? 1.f : ex2(m_run[j] - m_new);
            l_run[j] *= a;
#pragma unroll
            for (int mt2 = 0; mt2 < KS; ++mt2) {
                acc[mt2][j] *= a;
                acc[mt2][2 + j] *= a;
            }
            m_run[j] = m_new;
        }
    }
    uint32_t bh[2][2], bl[2][2]; // P^T B fragments of each half: high and low bf16 parts
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        float pr[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float m = m_run[i & 1];
            pr[i] = ex2(v[h][i] - (m == kNegInf ? 0.f : m));
        }
        l_run[0] += pr[0] + pr[2];
        l_run[1] += pr[1] + pr[3];
        const uint32_t h01 = pack_bf16(pr[0], pr[1]), h23 = pack_bf16(pr[2], pr[3]);
        const float2 f01 = unpack_bf16(h01), f23 = unpack_bf16(h23);
        const uint32_t l01 = pack_bf16(pr[0] - f01.x, pr[1] - f01.y), l23 = pack_bf16(pr[2] - f23.x, pr[3] - f23.y);
        bh[h][0] = movmatrix_trans(h01);
        bh[h][1] = movmatrix_trans(h23);
        bl[h][0] = movmatrix_trans(l01);
        bl[h][1] = movmatrix_trans(l23);
    }
    // ---- O^T += V^T P^T over both halves
    const int vchunk = (lane >> 3) & 1;
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t a[4];
            ldsm_x4_trans(tile_addr<D>(vbase, 16 * h + (lane & 7) + ((lane >> 4) << 3), 2 * mt + vchunk, swz), a);
            mma_16816(acc[mt], a, bh[h][0], bh[h][1]);
            mma_16816(acc[mt], a, bl[h][0], bl[h][1]);
        }
    }
}

// Workspace slot of slice j of a unit whose first slice belongs to CTA kf:
// slice 0 is CTA kf's last slice (slot 2kf+1), slice j >= 1 is CTA kf+j's
// first slice (slot 2(kf+j)).
__device__ __forceinline__ int slot_of(int kf, int j)
{
    return j == 0 ? 2 * kf + 1 : 2 * (kf + j);
}

// Row of q / out / lse (one row per (query, head)) of column c of a unit, or
// -1 for a column past the unit's (query, head) pairs.  Rows number fewer
// than 2^31 (checked on the host).
template <int GC, bool MQ>
__device__ __forceinline__ int column_row(const KParams &p, const Seg &sg, int c)
{
    if constexpr (!MQ)
        return sg.b * p.num_q_heads + sg.kvh * p.group + sg.sub * GC + c;
    const int col = sg.sub * GC + c;
    if (c >= GC || col >= sg.qn * p.group)
        return -1;
    return (sg.qs + (col >> p.group_shift)) * p.num_q_heads + sg.kvh * p.group + (col & (p.group - 1));
}

// Keys column c of a unit sees (multi-query rows; else all of them).
template <int GC, bool MQ>
__device__ __forceinline__ int column_keys(const KParams &p, const Seg &sg, int c)
{
    if constexpr (!MQ)
        return 0x7fffffff;
    return sg.mask_from + ((sg.sub * GC + c) >> p.group_shift) - ((sg.sub * GC) >> p.group_shift);
}

// (query, head) columns of a multi-query unit (GC > 8 kernels only).
template <int GC>
__device__ __forceinline__ int unit_cols(const KParams &p, const Seg &sg)
{
    return min(GC, sg.qn * p.group - sg.sub * GC);
}

// B fragments of Q^T for one slice: column cb + g of the unit (zero beyond
// its columns), dims 16ks + 2c (+8).
template <int D, int GC, bool MQ>
__device__ __forceinline__ void load_q(const KParams &p, const Seg &sg, int lane, uint32_t (&qf)[D / 16][2],
                                       int cb = 0)
{
    const int g = lane >> 2, c = lane & 3;
    const int row = g < GC ? column_row<GC, MQ>(p, sg, cb + g) : -1;
    const uint32_t *qrow = reinterpret_cast<const uint32_t *>(p.q + (int64_t)(row < 0 ? 0 : row) * D);
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
        qf[ks][0] = row >= 0 ? __ldg(qrow + 8 * ks + c) : 0u;
        qf[ks][1] = row >= 0 ? __ldg(qrow + 8 * ks + 4 + c) : 0u;
    }
}

// Consumer warp: runs the tile loop of every slice of this CTA and hands each
// slice's softmax state (o, m, l per head) to an epilogue warp.
template <int D, int GC, bool MQ>
__device__ void consumers(const KParams &p, Smem<D, GC, MQ> &sm)
{
    constexpr int S = Smem<D, GC, MQ>::kStages;
    constexpr int KS = D / 16;
    constexpr int RC = Smem<D, GC, MQ>::RC;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const int swz = p.swizzle ? 7 : 0;
    volatile int32_t *abort = &sm.abort;
    SegIter si;
    si.init(p, sm, blockIdx.x);
    Seg sg, nx;
    bool have = si.next(p, sm, sg);
    uint32_t qf[KS][2];
    wait_prior_grid(p);
    // Dependents may start only now that the grid before this one has
    // completed: a later launch that reads a step plan before its own wait
    // then finds the plan kernel (two or more launches back) complete.
    if (p.pdl && threadIdx.x == 0)
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // a unit of more than 8 columns (GC = 16 only) splits its columns between
    // the warps: this warp's first column is cb
    bool wide = false;
    int cb = 0;
    if constexpr (GC > 8) {
        wide = have && unit_cols<GC>(p, sg) > 8;
        cb = wide ? 8 * warp : 0;
    }
    if (have)
        load_q<D, GC, MQ>(p, sg, lane, qf, cb);
    int lim0 = have ? column_keys<GC, MQ>(p, sg, cb + 2 * c) : 0;
    int lim1 = have ? column_keys<GC, MQ>(p, sg, cb + 2 * c + 1) : 0;
    uint32_t g_tile = 0;
    int seg_i = 0;
    while (have) {
        bool more = false;
        uint32_t qn[KS][2]; // next slice's queries, loading while this slice streams
        float acc[KS][4];
#pragma unroll
        for (int mt = 0; mt < KS; ++mt)
            acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
        float m_run[2] = {kNegInf, kNegInf}, l_run[2] = {0.f, 0.f};
        int bad = 0;
        bool ok = true;
        const int n_tiles = (sg.tok1 - sg.tok0 + kTile - 1) / kTile;
        for (int t = 0; t < n_tiles; ++t, ++g_tile) {
            const int s = g_tile % S;
            if (!wait_or_abort(&sm.full[s], (g_tile / S) & 1u, abort)) {
                ok = false;
                break;
            }
            bad |= ((volatile int32_t *)sm.stage_bad)[s];
            const int tstart = sg.tok0 + t * kTile;
            const int nv = min(kTile, sg.tok1 - tstart);
            bool done = false;
            if constexpr (GC > 8) {
                if (wide) {
                    if (nv == kTile && tstart + kTile <= sg.mask_from) {
                        consume_tile_wide<D, false>(sm.kv[s][0], sm.kv[s][1], nv, 0, 0, lane, swz, p.q_scale, qf, acc,
                                                    m_run, l_run);
                    } else {
                        consume_tile_wide<D, true>(sm.kv[s][0], sm.kv[s][1], nv, lim0 - tstart, lim1 - tstart, lane,
                                                   swz, p.q_scale, qf, acc, m_run, l_run);
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    }
                    done = true;
                }
            }
            if (done) {
            } else if (nv == kTile && (!MQ || tstart + kTile <= sg.mask_from)) {
                consume_tile<D, false, MQ>(sm.kv[s][0], sm.kv[s][1], nv, 0, 0, warp, lane, swz, p.q_scale, qf, acc,
                                       m_run, l_run);
            } else {
                consume_tile<D, true, MQ>(sm.kv[s][0], sm.kv[s][1], nv, lim0 - tstart, lim1 - tstart, warp, lane, swz,
                                      p.q_scale, qf, acc, m_run, l_run);
                // the zeroed V rows were written by the generic proxy; order
                // them before the TMA that refills this stage
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&sm.empty[s]);
            if (t == 0) {
                more = si.next(p, sm, nx);
                if (more) {
                    int ncb = 0;
                    if constexpr (GC > 8)
                        ncb = unit_cols<GC>(p, nx) > 8 ? 8 * warp : 0;
                    load_q<D, GC, MQ>(p, nx, lane, qn, ncb);
                }
            }
        }
        if (!ok)
            break;
        // l over the 8 row groups
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            l_run[j] += __shfl_xor_sync(0xffffffffu, l_run[j], 4);
            l_run[j] += __shfl_xor_sync(0xffffffffu, l_run[j], 8);
            l_run[j] += __shfl_xor_sync(0xffffffffu, l_run[j], 16);
        }
        const int slot = seg_i & 1;
        if (seg_i >= kSlots && !wait_or_abort(&sm.epi_empty[slot], ((seg_i >> 1) - 1) & 1u, abort))
            break;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int h = 2 * c + j;
            if (h < RC) {
#pragma unroll
                for (int mt = 0; mt < KS; ++mt) {
                    sm.red_o[slot][warp][h][16 * mt + g] = acc[mt][j];
                    sm.red_o[slot][warp][h][16 * mt + g + 8] = acc[mt][2 + j];
                }
                if (g == 0) {
                    sm.red_m[slot][warp][h] = m_run[j];
                    sm.red_l[slot][warp][h] = l_run[j];
                }
            }
        }
        if (lane == 0)
            sm.red_bad[slot][warp] = bad;
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&sm.epi_full[slot]);
        ++seg_i;
        have = more;
        sg = nx;
        if (have) {
            if constexpr (GC > 8) {
                wide = unit_cols<GC>(p, sg) > 8;
                cb = wide ? 8 * warp : 0;
            }
            lim0 = column_keys<GC, MQ>(p, sg, cb + 2 * c);
            lim1 = column_keys<GC, MQ>(p, sg, cb + 2 * c + 1);
        }
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            qf[ks][0] = qn[ks][0];
            qf[ks][1] = qn[ks][1];
        }
    }
}

// ---------------------------------------------------------------- epilogue
// Two epilogue warps; warp w finishes the slices with index parity w.  Lane l
// holds element pairs e = 2 l + 64 i (i < EPT2) of the unit's [GC][D]
// output, i.e. head e / D, dims e % D and e % D + 1.
template <int D, int GC>
struct EpiState {
    static constexpr int EPT2 = GC * D / 64;
    float2 o[EPT2];
    float M[GC], L[GC];
};

template <int D>
__device__ __forceinline__ int pair_elem(int lane, int i)
{
    return 2 * lane + 64 * i;
}

// Everything a unit's finish reads from global memory besides the partials,
// loaded into registers before the slice's softmax state arrives, and the new
// token's scores computed from them meanwhile.
template <int D, int GC>
struct EpiInputs {
    static constexpr int KP = D / 64;                // bf16 pairs of one row per lane
    static constexpr int CH = (2 * D / 8 + 31) / 32; // 16-byte append chunks per lane
    uint32_t v2[KP];
    uint4 chunk[CH];
    int page;
    float sn[GC]; // (q . k_new) * scale * log2 e of every head
};

// Loads issued where they stand: the volatile asm keeps them ahead of the
// barrier wait that follows, so their latency overlaps it.
__device__ __forceinline__ uint32_t ld_pinned(const void *ptr)
{
    uint32_t v;
    asm volatile("ld.global.nc.b32 %0, [%1];" : "=r"(v) : "l"(ptr));
    return v;
}

__device__ __forceinline__ uint4 ld_pinned4(const void *ptr)
{
    uint4 v;
    asm volatile("ld.global.nc.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(ptr));
    return v;
}

template <int D, int GC, bool MQ>
__device__ __forceinline__ void load_epi_inputs(const KParams &p, const Seg &sg, int lane, EpiInputs<D, GC> &in)
{
    constexpr int KP = EpiInputs<D, GC>::KP;
    in.page = 0;
    if constexpr (MQ)
        return; // multi-query rows were appended by the caller: no new token here
    if (sg.status != ROW_OK || !p.with_new)
        return;
    const int h0 = sg.kvh * p.group + sg.sub * GC;
    const __nv_bfloat16 *kn = p.k_new + ((int64_t)sg.b * p.num_kv_heads + sg.kvh) * D;
    const __nv_bfloat16 *vn = p.v_new + ((int64_t)sg.b * p.num_kv_heads + sg.kvh) * D;
    uint32_t q2[GC][KP], k2[KP];
#pragma unroll
    for (int j = 0; j < KP; ++j) {
        k2[j] = ld_pinned(reinterpret_cast<const uint32_t *>(kn) + lane + 32 * j);
        in.v2[j] = ld_pinned(reinterpret_cast<const uint32_t *>(vn) + lane + 32 * j);
#pragma unroll
        for (int g = 0; g < GC; ++g)
            q2[g][j] = ld_pinned(reinterpret_cast<const uint32_t *>(p.q + ((int64_t)sg.b * p.num_q_heads + h0 + g) * D) +
                                 lane + 32 * j);
    }
    constexpr int kVec = D / 8;
#pragma unroll
    for (int ci = 0; ci < EpiInputs<D, GC>::CH; ++ci) {
        const int cix = lane + 32 * ci;
        in.chunk[ci] = make_uint4(0u, 0u, 0u, 0u);
        if (cix < 2 * kVec)
            in.chunk[ci] = ld_pinned4(cix < kVec ? reinterpret_cast<const uint4 *>(kn) + cix
                                                 : reinterpret_cast<const uint4 *>(vn) + (cix - kVec));
    }
    in.page = (int)ld_pinned(p.block_table + (int64_t)sg.b * p.max_blocks + (sg.L >> p.page_shift));
    // the new token's scores, off the path that follows the state's arrival
#pragma unroll
    for (int g = 0; g < GC; ++g) {
        float s = 0.f;
#pragma unroll
        for (int j = 0; j < KP; ++j) {
            const float2 qv = unpack_bf16(q2[g][j]), kv = unpack_bf16(k2[j]);
            s = fmaf(qv.x, kv.x, fmaf(qv.y, kv.y, s));
        }
        for (int o = 16; o > 0; o >>= 1)
            s += __shfl_xor_sync(0xffffffffu, s, o);
        in.sn[g] = s * p.q_scale;
    }
}

// Writes one unit's output: zeros for inactive / failed rows, otherwise
// merges the new token (when given), performs the append and normalises.
// Multi-query units of UGC columns are written GC columns at a time, from
// column col0.
template <int D, int GC, bool MQ, int UGC = GC>
__device__ void finalize_warp(const KParams &p, const Seg &sg, EpiState<D, GC> &st, const EpiInputs<D, GC> &in,
                              int bad, int lane, int col0 = 0)
{
    constexpr int EPT2 = EpiState<D, GC>::EPT2;
    constexpr int KP = EpiInputs<D, GC>::KP;
    int err = 0;
    if (sg.status == ROW_OVERFLOW)
        err = PKV_ERR_OVERFLOW;
    else if (sg.status == ROW_QLEN)
        err = PKV_ERR_QLEN;
    else if (sg.status == ROW_OK && bad)
        err = PKV_ERR_PAGE;
    if (sg.status == ROW_OK && !err && p.with_new && (in.page < 1 || in.page >= p.num_pages))
        err = PKV_ERR_PAGE;
    const bool live = sg.status == ROW_OK && !err;
    if (lane == 0 && err)
        set_error(p.err_flag, err);
    if (live && p.with_new) {
        const float *sn = in.sn; // (q . k_new) * scale * log2 e
        if (sg.sub == 0) { // the append: one bit copy per kv head
            constexpr int kVec = D / 8;
            const int slot = sg.L & (p.page_size - 1);
            const int64_t dst = p.layout == PKV_NHD
                                    ? (((int64_t)in.page * p.page_size + slot) * p.num_kv_heads + sg.kvh) * D
                                    : (((int64_t)in.page * p.num_kv_heads + sg.kvh) * p.page_size + slot) * D;
#pragma unroll
            for (int ci = 0; ci < EpiInputs<D, GC>::CH; ++ci) {
                const int cix = lane + 32 * ci;
                if (cix < 2 * kVec) {
                    const bool is_v = cix >= kVec;
                    reinterpret_cast<uint4 *>((is_v ? p.v_cache : p.k_cache) + dst)[is_v ? cix - kVec : cix] =
                        in.chunk[ci];
                }
            }
        }
        float a[GC], cn[GC];
#pragma unroll
        for (int g = 0; g < GC; ++g) {
            const float Mn = fmaxf(st.M[g], sn[g]);
            a[g] = ex2(st.M[g] - Mn); // M = -inf (no cached key) -> 0
            cn[g] = ex2(sn[g] - Mn);
            st.L[g] = fmaf(st.L[g], a[g], cn[g]);
            st.M[g] = Mn;
        }
#pragma unroll
        for (int i = 0; i < EPT2; ++i) {
            const int g = pair_elem<D>(lane, i) / D;
            const float2 v = unpack_bf16(in.v2[i % KP]);
            st.o[i].x = fmaf(st.o[i].x, a[g], cn[g] * v.x);
            st.o[i].y = fmaf(st.o[i].y, a[g], cn[g] * v.y);
        }
    }
    // rows without a visible key (or failed rows) give exact zeros: select,
    // never multiply, since their state may hold NaN from unread slots
    float inv[GC];
    bool any[GC];
#pragma unroll
    for (int g = 0; g < GC; ++g) {
        any[g] = live && st.L[g] > 0.f;
        inv[g] = any[g] ? 1.f / st.L[g] : 0.f;
    }
    if constexpr (!MQ) {
        const int h0 = sg.kvh * p.group + sg.sub * GC;
        uint32_t *out = reinterpret_cast<uint32_t *>(p.out + ((int64_t)sg.b * p.num_q_heads + h0) * D);
#pragma unroll
        for (int i = 0; i < EPT2; ++i) {
            const int e = pair_elem<D>(lane, i), g = e / D;
            out[e >> 1] = any[g] ? pack_bf16(st.o[i].x * inv[g], st.o[i].y * inv[g]) : 0u;
        }
        if (p.lse != nullptr && lane < GC) {
            float M = kNegInf, L = 0.f;
#pragma unroll
            for (int g = 0; g < GC; ++g)
                if (g == lane) {
                    M = st.M[g];
                    L = st.L[g];
                }
            const bool any = live && L > 0.f;
            p.lse[(int64_t)sg.b * p.num_q_heads + h0 + lane] =
                any ? (M + log2f(L)) * 0.69314718055994531f : kNegInf;
        }
        return;
    }
    // multi-query rows: output row of every column (-1: a column past the unit's (query, head) pairs)
    int orow[GC];
#pragma unroll
    for (int g = 0; g < GC; ++g)
        orow[g] = column_row<UGC, MQ>(p, sg, col0 + g);
    uint32_t *out = reinterpret_cast<uint32_t *>(p.out);
#pragma unroll
    for (int i = 0; i < EPT2; ++i) {
        const int e = pair_elem<D>(lane, i), g = e / D;
        if (orow[g] >= 0)
            out[((int64_t)orow[g] * D + e % D) >> 1] =
                any[g] ? pack_bf16(st.o[i].x * inv[g], st.o[i].y * inv[g]) : 0u;
    }
    if (p.lse != nullptr && lane < GC) {
        float M = kNegInf, L = 0.f;
        int row = -1;
#pragma unroll
        for (int g = 0; g < GC; ++g)
            if (g == lane) {
                M = st.M[g];
                L = st.L[g];
                row = orow[g];
            }
        const bool any = live && L > 0.f;
        if (row >= 0)
            p.lse[row] = any ? (M + log2f(L)) * 0.69314718055994531f : kNegInf;
    }
}

// One log-sum-exp step: st (the running merge) takes in a partial with
// (m, l) pairs `ml` (l < 0: a slice that met a bad page) and outputs `ov`.
// Every merge of partials goes through this one expression, so that equal
// operands in equal roles give equal bits.  Returns nonzero for a bad slice.
template <int D, int GC>
__device__ __forceinline__ int lse_step(EpiState<D, GC> &st, const float2 (&ml)[GC],
                                        const float2 (&ov)[EpiState<D, GC>::EPT2], int lane)
{
    constexpr int EPT2 = EpiState<D, GC>::EPT2;
    int bad = 0;
    float a[GC], b[GC];
#pragma unroll
    for (int g = 0; g < GC; ++g) {
        bad |= ml[g].y < 0.f;
        const float l = fmaxf(ml[g].y, 0.f);
        const float Mn = fmaxf(st.M[g], ml[g].x);
        a[g] = st.M[g] == kNegInf ? 0.f : ex2(st.M[g] - Mn);
        b[g] = ml[g].x == kNegInf ? 0.f : ex2(ml[g].x - Mn);
        st.L[g] = st.L[g] * a[g] + l * b[g];
        st.M[g] = Mn;
    }
#pragma unroll
    for (int i = 0; i < EPT2; ++i) {
        const int g = pair_elem<D>(lane, i) / D;
        st.o[i].x = st.o[i].x * a[g] + ov[i].x * b[g];
        st.o[i].y = st.o[i].y * a[g] + ov[i].y * b[g];
    }
    return bad;
}

// Merges the n slice partials of one unit into st (columns col0 .. col0 +
// GC - 1 of partials `stride` columns wide), all but slice `skip` (-1: none);
// returns nonzero if any merged slice met a bad page.  The loads of all
// slices are issued before the math.
template <int D, int GC, int kBatchMax = 4>
__device__ int combine_warp(const KParams &p, EpiState<D, GC> &st, int kf, int n, int lane, int stride = GC,
                           int col0 = 0, int skip = -1)
{
    constexpr int EPT2 = EpiState<D, GC>::EPT2;
    // slices whose loads are in flight together
    constexpr int kBatch0 = EPT2 >= 16 ? 1 : (EPT2 >= 8 ? 2 : 4);
    constexpr int kBatch = kBatch0 < kBatchMax ? kBatch0 : kBatchMax;
    int bad = 0;
#pragma unroll
    for (int g = 0; g < GC; ++g) {
        st.M[g] = kNegInf;
        st.L[g] = 0.f;
    }
#pragma unroll
    for (int i = 0; i < EPT2; ++i)
        st.o[i] = make_float2(0.f, 0.f);
    for (int j0 = 0; j0 < n; j0 += kBatch) {
        float2 ml[kBatch][GC];
        float2 ov[kBatch][EPT2];
#pragma unroll
        for (int jj = 0; jj < kBatch; ++jj) {
            if (j0 + jj < n && j0 + jj != skip) {
                const int slot = slot_of(kf, j0 + jj);
#pragma unroll
                for (int g = 0; g < GC; ++g)
                    ml[jj][g] = __ldcg(p.part_ml + (int64_t)slot * stride + col0 + g);
                const float2 *po = reinterpret_cast<const float2 *>(p.part_o + ((int64_t)slot * stride + col0) * D);
#pragma unroll
                for (int i = 0; i < EPT2; ++i)
                    ov[jj][i] = __ldcg(po + (pair_elem<D>(lane, i) >> 1));
            }
        }
#pragma unroll
        for (int jj = 0; jj < kBatch; ++jj) {
            if (j0 + jj >= n)
                break;
            if (j0 + jj == skip)
                continue;
            bad |= lse_step<D, GC>(st, ml[jj], ov[jj], lane);
        }
    }
    return bad;
}

// Epilogue warps that read one hand-off slot before it is refilled: both in
// kernels with 16-column units (a wide unit's two 8-column halves are
// finished side by side), else the one that owns the slice.
template <int GC>
__host__ __device__ constexpr int kEpiReaders()
{
    return GC > 8 ? 2 : 1;
}

// A slice's softmax state from hand-off slot `slot`: the two consumer warps'
// row halves merged, or (wide units) warp h's columns as they are.
template <int D, int GC, bool MQ>
__device__ __forceinline__ void slot_state(const Smem<D, GC, MQ> &sm, int slot, bool wide, int h, int lane,
                                           EpiState<D, Smem<D, GC, MQ>::RC> &st)
{
    constexpr int RC = Smem<D, GC, MQ>::RC;
    constexpr int EPT2 = EpiState<D, RC>::EPT2;
    if (wide) {
#pragma unroll
        for (int g = 0; g < RC; ++g) {
            st.M[g] = sm.red_m[slot][h][g];
            st.L[g] = sm.red_l[slot][h][g];
        }
#pragma unroll
        for (int i = 0; i < EPT2; ++i)
            st.o[i] = *reinterpret_cast<const float2 *>(&(&sm.red_o[slot][h][0][0])[pair_elem<D>(lane, i)]);
        return;
    }
    float w0[RC], w1[RC];
#pragma unroll
    for (int g = 0; g < RC; ++g) {
        const float m0 = sm.red_m[slot][0][g], m1 = sm.red_m[slot][1][g];
        const float M = fmaxf(m0, m1);
        w0[g] = m0 == kNegInf ? 0.f : ex2(m0 - M);
        w1[g] = m1 == kNegInf ? 0.f : ex2(m1 - M);
        st.M[g] = M;
        st.L[g] = w0[g] * sm.red_l[slot][0][g] + w1[g] * sm.red_l[slot][1][g];
    }
#pragma unroll
    for (int i = 0; i < EPT2; ++i) {
        const int e = pair_elem<D>(lane, i), g = e / D;
        const float2 r0 = *reinterpret_cast<const float2 *>(&(&sm.red_o[slot][0][0][0])[e]);
        const float2 r1 = *reinterpret_cast<const float2 *>(&(&sm.red_o[slot][1][0][0])[e]);
        st.o[i] = make_float2(w0[g] * r0.x + w1[g] * r1.x, w0[g] * r0.y + w1[g] * r1.y);
    }
}

// Writes a slice's state as split-KV partial `wslot` (columns col0 .. col0 +
// GC - 1 of a partial `stride` columns wide); l = -1 marks a bad page.
template <int D, int GC>
__device__ __forceinline__ void write_partial(const KParams &p, const EpiState<D, GC> &st, int wslot, int stride,
                                              int col0, int bad, int lane)
{
    constexpr int EPT2 = EpiState<D, GC>::EPT2;
    float2 *po = reinterpret_cast<float2 *>(p.part_o + ((int64_t)wslot * stride + col0) * D);
#pragma unroll
    for (int i = 0; i < EPT2; ++i)
        po[pair_elem<D>(lane, i) >> 1] = st.o[i];
    if (lane < GC) {
        float M = 0.f, L = 0.f;
#pragma unroll
        for (int g = 0; g < GC; ++g)
            if (g == lane) {
                M = st.M[g];
                L = st.L[g];
            }
        p.part_ml[(int64_t)wslot * stride + col0 + lane] = make_float2(M, bad ? -1.f : L);
    }
}

// acc takes in the state inc (of the same columns) as combine_warp would take
// in inc's partial: the same lse_step, so the bits equal that merge's.
template <int D, int GC>
__device__ __forceinline__ void merge_in(EpiState<D, GC> &acc, const EpiState<D, GC> &inc, int lane)
{
    float2 ml[GC];
#pragma unroll
    for (int g = 0; g < GC; ++g)
        ml[g] = make_float2(inc.M[g], inc.L[g]);
    (void)lse_step<D, GC>(acc, ml, inc.o, lane);
}

// A split unit's ticket: release orders this warp's partial stores (all lanes,
// joined by the __syncwarp before it) ahead of the increment; acquire orders
// the last arriver's reads of the other partials (after the __syncwarp that
// follows) behind it.  One atomic in place of a sequentially consistent fence
// on each side.
__device__ __forceinline__ int atom_add_acq_rel(int32_t *ptr, int v)
{
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(ptr), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ int ld_acquire(const int32_t *ptr)
{
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
    return v;
}

// The merge ahead of wait_slice, one slice's loads at a time (it runs while
// the slice streams; kept out of line so the waiting loop stays small).
template <int D, int GC>
__device__ __noinline__ int merge_ahead(const KParams &p, EpiState<D, GC> &pre, int kf, int n, int lane, int stride,
                                        int col0, int skip)
{
    return combine_warp<D, GC, 1>(p, pre, kf, n, lane, stride, col0, skip);
}

// Waits for hand-off slot `slot` (parity `par`) like wait_or_abort.  For a
// slice of a split unit it watches the unit's ticket meanwhile: once every
// other slice has arrived (ticket == n - 1), this slice is the last one, and
// the others' partials are merged into `pre` while this one still streams.
template <int D, int GC>
__device__ __forceinline__ bool wait_slice(const KParams &p, uint64_t *bar, uint32_t par, volatile int32_t *abort,
                                           const int32_t *ticket, int kf, int n, int jown, int lane, int stride,
                                           int col0, EpiState<D, GC> &pre, bool &have_pre, int &pre_bad)
{
    // the merge order stays the slot order: the other slice of a pair, or
    // all the others when this slice is the unit's last
    const bool watch = n == 2 || (n > 2 && jown == n - 1);
    if (!watch && mbar_try_wait(bar, par))
        return true;
    const uint64_t start = globaltimer_ns();
    for (;;) {
        if (watch && !have_pre) {
            // the ticket load is in flight while the barrier is tested
            // without suspending
            const int t = ld_acquire(ticket);
            for (int i = 0; i < 16; ++i)
                if (mbar_test_wait(bar, par))
                    return true;
            if (t == n - 1) {
                pre_bad = merge_ahead<D, GC>(p, pre, kf, n, lane, stride, col0, jown);
                have_pre = true;
            }
        } else {
            for (int i = 0; i < 32; ++i)
                if (mbar_try_wait(bar, par))
                    return true;
        }
        if (*abort)
            return false;
        if (globaltimer_ns() - start > kWaitLimitNs) {
            *abort = 1;
            return false;
        }
    }
}

template <int D, int GC, bool MQ>
__device__ void epilogue(const KParams &p, Smem<D, GC, MQ> &sm, int ew)
{
    constexpr int RC = Smem<D, GC, MQ>::RC; // columns per pass: a 16-column unit takes two passes
    constexpr int EPT2 = EpiState<D, RC>::EPT2;
    const int lane = threadIdx.x & 31;
    const int k = (int)blockIdx.x;
    volatile int32_t *abort = &sm.abort;
    SegIter si;
    si.init(p, sm, k);
    Seg sg;
    int seg_i = 0;
    bool stopped = false;
    wait_prior_grid(p);
    if (k == 0 && ew == 0) { // a step plan that was rejected, or whose lengths are stale
        int bad = sm.plan_state == 2;
        if (sm.plan_state == 1)
            for (int i = lane; i < p.batch; i += 32)
                bad |= p.seqlens[i] != sm.len[i];
        if (__any_sync(0xffffffffu, bad) && lane == 0)
            set_error(p.err_flag, PKV_ERR_PLAN);
    }
    while (si.next(p, sm, sg)) {
        const int mine = seg_i;
        ++seg_i;
        // a wide unit (more than 8 columns) is finished by both warps, warp
        // ew taking columns 8 ew .. 8 ew + 7; other slices by one warp
        bool wide = false;
        if constexpr (GC > 8)
            wide = unit_cols<GC>(p, sg) > 8;
        if (!wide && (mine & 1) != ew)
            continue;
        const int slot = mine & 1;
        const int h = wide ? ew : 0; // this warp's 8-column pass
        EpiInputs<D, RC> in;
        load_epi_inputs<D, RC, MQ>(p, sg, lane, in);
        // slices of this unit: kf .. kf + n - 1 (a slice from the unit's first
        // to its last token is the whole unit)
        int kf = k, n = 1;
        if (sg.tok0 != 0 || sg.tok1 != sg.n) {
            kf = sg.tok0 == 0 ? k : owner_of(p, sm, sg.u0);
            const int kl = sg.tok1 == sg.n ? k : owner_of(p, sm, sg.u0 + sg.n - 1);
            n = kl - kf + 1;
        }
        // this warp's ticket and partial columns of the unit
        int32_t *ticket = GC > 8 ? p.tickets + 2 * sg.unit + h : p.tickets + sg.unit;
        const int col0 = GC > 8 ? RC * h : 0;
        EpiState<D, RC> pre; // the other slices, merged ahead when they arrive first
        bool have_pre = false;
        int pre_bad = 0;
        if (!wait_slice<D, RC>(p, &sm.epi_full[slot], (mine >> 1) & 1u, abort, ticket, kf, n, k - kf, lane, GC, col0,
                               pre, have_pre, pre_bad)) {
            stopped = true;
            break;
        }
        EpiState<D, RC> st;
        slot_state(sm, slot, wide, h, lane, st);
        int bad = sm.red_bad[slot][0] | sm.red_bad[slot][1];
        __syncwarp();
        if (lane == 0) { // consumers may refill this slot once every reader is done
            if constexpr (kEpiReaders<GC>() == 1)
                mbar_arrive(&sm.epi_empty[slot]);
            else
                mbar_arrive_cnt(&sm.epi_empty[slot], wide ? 1u : (uint32_t)kEpiReaders<GC>());
        }
        if (have_pre) { // every other slice is in: the last merge, no ticket
            // in slot order, the lower slot taking in the higher one
            if (k - kf == 0) {
                merge_in(st, pre, lane);
            } else {
                merge_in(pre, st, lane);
                st = pre;
            }
            if constexpr (GC > 8)
                finalize_warp<D, RC, MQ, GC>(p, sg, st, in, bad | pre_bad, lane, RC * h);
            else
                finalize_warp<D, GC, MQ>(p, sg, st, in, bad | pre_bad, lane);
            __syncwarp();
            if (lane == 0)
                *ticket = 0; // ready for the next call
            continue;
        }
        if constexpr (GC > 8) {
            if (n == 1) {
                finalize_warp<D, RC, MQ, GC>(p, sg, st, in, bad, lane, RC * h);
                continue;
            }
            write_partial<D, RC>(p, st, slot_of(kf, k - kf), GC, RC * h, bad, lane);
            __syncwarp();
            int32_t *ticket = p.tickets + 2 * sg.unit + h;
            int last = 0;
            if (lane == 0)
                last = atom_add_acq_rel(ticket, 1) == n - 1;
            __syncwarp();
            last = __shfl_sync(0xffffffffu, last, 0);
            if (last) {
                bad = combine_warp<D, RC>(p, st, kf, n, lane, GC, RC * h);
                finalize_warp<D, RC, MQ, GC>(p, sg, st, in, bad, lane, RC * h);
                if (lane == 0)
                    *ticket = 0; // ready for the next call
            }
        } else {
            if (n == 1) {
                finalize_warp<D, GC, MQ>(p, sg, st, in, bad, lane);
                continue;
            }
            write_partial<D, GC>(p, st, slot_of(kf, k - kf), GC, 0, bad, lane);
            __syncwarp();
            int last = 0;
            if (lane == 0)
                last = atom_add_acq_rel(&p.tickets[sg.unit], 1) == n - 1;
            __syncwarp();
            last = __shfl_sync(0xffffffffu, last, 0);
            if (last) {
                bad = combine_warp<D, GC>(p, st, kf, n, lane);
                finalize_warp<D, GC, MQ>(p, sg, st, in, bad, lane);
                if (lane == 0)
                    p.tickets[sg.unit] = 0; // ready for the next call
            }
        }
    }
    // Units with no cached token (inactive, overflowing or empty rows, and
    // malformed multi-query rows) get their output (zeros, or the new token
    // alone) here: empty unit e goes to CTA e % gridDim.x, epilogue warp
    // (e / gridDim.x) % 2.
    if (!stopped && !*abort && sm.n_empty > 0) {
        const int G = (int)gridDim.x;
        long long e0 = 0; // empty units before row b
        for (int b = 0; b < p.batch; ++b) {
            if (sm.rowtok[b + 1] != sm.rowtok[b])
                continue;
            int units = p.units;
            if constexpr (MQ) {
                int kv;
                units = mq_units<GC>(p, mq_row_status(p, sm.len[b], sm.qlen[b], &kv), sm.qlen[b]);
            }
            for (int r = (int)(((long long)k - e0 % G + G) % G); r < units; r += G) {
                if (((e0 + r) / G & 1) != ew)
                    continue;
                Seg es;
                seg_unit(p, sm, es, b, r);
                es.tok0 = es.tok1 = 0;
                es.u0 = 0;
                es.n = 0;
                EpiInputs<D, RC> in;
                load_epi_inputs<D, RC, MQ>(p, es, lane, in);
                int npass_e = 1;
                if constexpr (GC > 8)
                    npass_e = unit_cols<GC>(p, es) > 8 ? 2 : 1;
                for (int h = 0; h < npass_e; ++h) {
                    EpiState<D, RC> st;
#pragma unroll
                    for (int g = 0; g < RC; ++g) {
                        st.M[g] = kNegInf;
                        st.L[g] = 0.f;
                    }
#pragma unroll
                    for (int i = 0; i < EPT2; ++i)
                        st.o[i] = make_float2(0.f, 0.f);
                    finalize_warp<D, RC, MQ, GC>(p, es, st, in, 0, lane, RC * h);
                }
            }
            e0 += units;
        }
    }
    // multi-query rows whose query range lies outside [0, total_q): no output, one error bit
    if (MQ && k == 0 && ew == 0 && lane == 0)
        for (int b = 0; b < p.batch; ++b)
            if (sm.qlen[b] < 0) {
                set_error(p.err_flag, PKV_ERR_QLEN);
                break;
            }
    if (*abort && lane == 0)
        set_error(p.err_flag, PKV_ERR_TIMEOUT);
}

template <int D, int GC, bool MQ>
__device__ __forceinline__ void init_barriers(Smem<D, GC, MQ> &sm)
{
    constexpr int S = Smem<D, GC, MQ>::kStages;
    for (int s = 0; s < S; ++s) {
        mbar_init(&sm.full[s], 1);
        mbar_init(&sm.empty[s], Roles<GC>::kCons);
    }
    for (int s = 0; s < kSlots; ++s) {
        mbar_init(&sm.epi_full[s], Roles<GC>::kCons);
        mbar_init(&sm.epi_empty[s], kEpiReaders<GC>());
    }
    sm.abort = 0;
    mbar_init_fence();
}

// PLAN: the instantiation that can start from a step plan (PKV_DECODE_USE_PLAN);
// the plain one carries no code of that path, which keeps the start of a
// lone launch (whose instructions come from memory) short.
template <int D, int GC, bool MQ, bool PLAN>
__device__ __forceinline__ void decode_body(const KParams &p, const DecodeMaps &maps)
{
    extern __shared__ unsigned char smem_raw[];
    Smem<D, GC, MQ> &sm = *reinterpret_cast<Smem<D, GC, MQ> *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    using R = Roles<GC>;
    if constexpr (!MQ && PLAN) {
        if (p.plan_in != nullptr) {
            // A step plan.  The producer warp alone decides whether it matches
            // this launch, from the header it loads together with its CTA's
            // record, publishes the decision (named barrier 1, without
            // waiting) and, if taken, issues its first tile at once.  The
            // other warps load the plan's arrays into registers meanwhile and
            // write them to shared memory once the plan is taken (named
            // barrier 2, which the producer joins after that first tile).
            // Every thread passes barrier 1 once, and barrier 2 once when the
            // plan is taken; a rejected plan is replaced by planning here.
            const PlanLayout lay = plan_layout(p.batch);
            const PlanHeader *h = reinterpret_cast<const PlanHeader *>(p.plan_in);
            if (warp == R::kProducer) {
                if (lane == 0) {
                    init_barriers(sm);
                    prefetch_tensormap(&maps.k);
                    prefetch_tensormap(&maps.v);
                    prefetch_tensormap(&maps.k8);
                    prefetch_tensormap(&maps.v8);
                }
                const PlanRec *rp = reinterpret_cast<const PlanRec *>(p.plan_in + lay.recs) + blockIdx.x;
                RecRegs rec;
                rec.si = ldcg_pod(&rp->si);
                rec.have = __ldcg(&rp->have);
                rec.b = __ldcg(&rp->b);
                rec.kvh = __ldcg(&rp->kvh);
                rec.tok0 = __ldcg(&rp->tok0);
                rec.tok1 = __ldcg(&rp->tok1);
                rec.win = __ldcg(&rp->pages[lane]);
                const bool ok = __shfl_sync(0xffffffffu, plan_matches(p, h), 0);
                if (lane == 0)
                    sm.plan_state = ok ? 1 : 2;
                __syncwarp();
                named_arrive(1, R::kThreads);
                if (ok) {
                    producer(p, sm, &maps, &rec);
                    return;
                }
            } else {
                // this thread's share of the arrays, at most kMaxDecodeBatch + 1 rows
                constexpr int kCopy = R::kThreads - 32;
                constexpr int kPer = (kMaxDecodeBatch + 1 + kCopy - 1) / kCopy;
                const int t = threadIdx.x < R::kProducer * 32 ? threadIdx.x : threadIdx.x - 32; // 0 .. kCopy - 1
                const int32_t *len = reinterpret_cast<const int32_t *>(p.plan_in + lay.len);
                const int32_t *rowtok = reinterpret_cast<const int32_t *>(p.plan_in + lay.rowtok);
                const long long *rowbase = reinterpret_cast<const long long *>(p.plan_in + lay.rowbase);
                int r_len[kPer], r_tok[kPer];
                long long r_base[kPer];
#pragma unroll
                for (int j = 0; j < kPer; ++j) {
                    const int i = t + j * kCopy;
                    r_len[j] = i < p.batch ? __ldcg(len + i) : 0;
                    r_tok[j] = i <= p.batch ? __ldcg(rowtok + i) : 0;
                    r_base[j] = i <= p.batch ? __ldcg(rowbase + i) : 0;
                }
                long long work = 0, slice = 0;
                int geff = 0, n_empty = 0;
                if (t == 0) {
                    work = __ldcg(&h->work);
                    slice = __ldcg(&h->slice);
                    geff = __ldcg(&h->geff);
                    n_empty = __ldcg(&h->n_empty);
                }
                named_sync(1, R::kThreads); // the producer's decision
                if (sm.plan_state == 1) {
#pragma unroll
                    for (int j = 0; j < kPer; ++j) {
                        const int i = t + j * kCopy;
                        if (i < p.batch)
                            sm.len[i] = r_len[j];
                        if (i <= p.batch) {
                            sm.rowtok[i] = r_tok[j];
                            sm.rowbase[i] = r_base[j];
                        }
                    }
                    if (t == 0) {
                        sm.work = work;
                        sm.slice = slice;
                        sm.geff = geff;
                        sm.n_empty = n_empty;
                    }
                    named_sync(2, R::kThreads); // the plan is in shared memory
                    if (warp < R::kCons)
                        consumers(p, sm);
                    else
                        epilogue(p, sm, warp - R::kEpi);
                    return;
                }
            }
            // rejected: plan here, as without a step plan (barriers are initialised)
            build_plan(p, sm, (int)gridDim.x); // ends with __syncthreads()
            if (warp < R::kCons)
                consumers(p, sm);
            else if (warp == R::kProducer)
                producer(p, sm, &maps, nullptr);
            else
                epilogue(p, sm, warp - R::kEpi);
            return;
        }
    }
    if (threadIdx.x == 0) {
        init_barriers(sm);
        sm.plan_state = 0;
    }
    if (threadIdx.x == R::kProducer * 32) {
        prefetch_tensormap(&maps.k);
        prefetch_tensormap(&maps.v);
        prefetch_tensormap(&maps.k8);
        prefetch_tensormap(&maps.v8);
    }
    build_plan(p, sm, (int)gridDim.x); // ends with __syncthreads()
    if (warp < R::kCons)
        consumers(p, sm);
    else if (warp == R::kProducer)
        producer(p, sm, &maps, nullptr);
    else
        epilogue(p, sm, warp - R::kEpi);
}

// The plan kernel of PKV_DECODE_MAKE_PLAN: builds the plan of a decode launch
// of `grid` CTAs (as every CTA of that launch would) and writes it to
// p.plan_out, one record per CTA (one warp per record).  An ordinary launch;
// it lets the decode kernel after it start at once (that kernel plans for
// itself and does not read this plan).
template <int D, int GC>
__global__ void __launch_bounds__(kThreads) decode_plan_kernel(const __grid_constant__ KParams p, int grid)
{
    extern __shared__ unsigned char smem_raw[];
    Smem<D, GC, false> &sm = *reinterpret_cast<Smem<D, GC, false> *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    if (threadIdx.x == 0)
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    build_plan(p, sm, grid); // ends with __syncthreads()
    const PlanLayout lay = plan_layout(p.batch);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int kWarpsAll = kThreads / 32;
    PlanRec *recs = reinterpret_cast<PlanRec *>(p.plan_out + lay.recs);
    for (int k = blockIdx.x * kWarpsAll + warp; k < grid; k += gridDim.x * kWarpsAll) {
        SegIter si;
        si.init(p, sm, k);
        Seg sg;
        const bool have = si.next(p, sm, sg);
        const int win = have ? load_window(p.block_table + (int64_t)sg.b * p.max_blocks, sg.tok0 >> p.page_shift,
                                           (sg.tok1 - 1) >> p.page_shift, lane)
                             : 0;
        PlanRec *r = recs + k;
        r->pages[lane] = win;
        if (lane == 0) {
            r->si = si;
            r->have = have ? 1 : 0;
            r->b = have ? sg.b : 0;
            r->kvh = have ? sg.kvh : 0;
            r->tok0 = have ? sg.tok0 : 0;
            r->tok1 = have ? sg.tok1 : 0;
        }
    }
    if (blockIdx.x != 0)
        return;
    int32_t *len = reinterpret_cast<int32_t *>(p.plan_out + lay.len);
    int32_t *rowtok = reinterpret_cast<int32_t *>(p.plan_out + lay.rowtok);
    long long *rowbase = reinterpret_cast<long long *>(p.plan_out + lay.rowbase);
    for (int i = threadIdx.x; i < p.batch; i += kThreads)
        len[i] = sm.len[i];
    for (int i = threadIdx.x; i <= p.batch; i += kThreads) {
        rowtok[i] = sm.rowtok[i];
        rowbase[i] = sm.rowbase[i];
    }
    if (threadIdx.x == 0) {
        PlanHeader *h = reinterpret_cast<PlanHeader *>(p.plan_out);
        h->magic = kPlanMagic;
        h->batch = p.batch;
        h->units = p.units;
        h->grid = grid;
        h->max_blocks = p.max_blocks;
        h->page_size = p.page_size;
        h->with_new = p.with_new;
        h->num_kv_heads = p.num_kv_heads;
        h->work = sm.work;
        h->slice = sm.slice;
        h->geff = sm.geff;
        h->n_empty = sm.n_empty;
    }
}

template <int D, int GC, bool MQ, bool PLAN>
__global__ void __launch_bounds__(kThreads) decode_kernel(const __grid_constant__ KParams p,
                                                          const __grid_constant__ DecodeMaps maps)
{
    decode_body<D, GC, MQ, PLAN>(p, maps);
}

// 16-column multi-query units: the register bound keeps two CTAs on an SM
// at head_dim <= 128 (the other instantiations fit two without it, or never
// do at head_dim 256).
template <int D, int GC, bool MQ>
__global__ void __launch_bounds__(Roles<GC>::kThreads, D <= 128 ? 2 : 1)
    decode_kernel_wide(const __grid_constant__ KParams p, const __grid_constant__ DecodeMaps maps)
{
    decode_body<D, GC, MQ, false>(p, maps);
}

template <int D, int GC, bool MQ>
size_t smem_bytes()
{
    return sizeof(Smem<D, GC, MQ>) + 1024;
}

// Two CTAs per SM: 228 KB of shared memory per SM, 1 KB of it reserved per CTA.
static_assert(sizeof(Smem<128, 4, true>) + 1024 + 1024 <= 228 * 1024 / 2, "decode<128,4> must fit twice on an SM");
static_assert(sizeof(Smem<128, 8, true>) + 1024 + 1024 <= 228 * 1024 / 2, "decode<128,8> must fit twice on an SM");
static_assert(sizeof(Smem<128, 16, true>) + 1024 + 1024 <= 228 * 1024 / 2, "decode<128,16> must fit twice on an SM");

struct KernelEntry {
    int D, GC;
    bool mq; // multi-query rows
    const void *fn;      // the decode kernel
    size_t smem;
    const void *plan_fn; // its step-plan kernel (plain rows), same shared memory
    const void *use_fn;  // the decode kernel that starts from a step plan (plain rows)
    int threads;         // block size of the decode kernels
};

template <int D, int GC, bool MQ>
KernelEntry entry()
{
    const void *fn;
    const void *plan_fn = nullptr, *use_fn = nullptr;
    if constexpr (GC > 8)
        fn = reinterpret_cast<const void *>(&decode_kernel_wide<D, GC, MQ>);
    else
        fn = reinterpret_cast<const void *>(&decode_kernel<D, GC, MQ, false>);
    if constexpr (!MQ) {
        plan_fn = reinterpret_cast<const void *>(&decode_plan_kernel<D, GC>);
        use_fn = reinterpret_cast<const void *>(&decode_kernel<D, GC, MQ, true>);
    }
    return KernelEntry{D, GC, MQ, fn, smem_bytes<D, GC, MQ>(), plan_fn, use_fn, Roles<GC>::kThreads};
}

const KernelEntry kTable[] = {
    entry<64, 1, false>(),  entry<64, 2, false>(),  entry<64, 4, false>(),  entry<64, 8, false>(),
    entry<128, 1, false>(), entry<128, 2, false>(), entry<128, 4, false>(), entry<128, 8, false>(),
    entry<256, 1, false>(), entry<256, 2, false>(), entry<256, 4, false>(), entry<256, 8, false>(),
    entry<64, 1, true>(),   entry<64, 2, true>(),   entry<64, 4, true>(),   entry<64, 8, true>(),
    entry<128, 1, true>(),  entry<128, 2, true>(),  entry<128, 4, true>(),  entry<128, 8, true>(),
    entry<256, 1, true>(),  entry<256, 2, true>(),  entry<256, 4, true>(),  entry<256, 8, true>(),
    entry<64, 16, true>(),  entry<128, 16, true>(), entry<256, 16, true>(),
};

const KernelEntry *find_kernel(int D, int GC, bool mq = false)
{
    for (const KernelEntry &e : kTable)
        if (e.D == D && e.GC == GC && e.mq == mq)
            return &e;
    return nullptr;
}

int kernel_index(const KernelEntry *e)
{
    return static_cast<int>(e - kTable);
}

// Heads of one kv head that share a CTA: the MMA's N side holds 8.
int heads_per_cta(int group)
{
    return group < 8 ? group : 8;
}

} // namespace

int decode_box_tokens(int page_size)
{
    return page_size < kDecodeTile ? page_size : kDecodeTile;
}

int decode_swizzle(int page_size)
{
    // 128-byte swizzle needs every box to start on a 1024-byte (8-row) boundary
    return page_size >= 8 ? 1 : 0;
}

namespace {

// Shared tail of decode_shape / decode_mq_shape once the columns per unit
// (heads_per_cta) and units per row are set.  Plain rows get room for a step
// plan after the partials.
bool finish_shape(int batch, int max_blocks, const pkv_cache_desc &d, bool multi_query, DecodeShape *s)
{
    if (find_kernel(d.head_dim, s->heads_per_cta, multi_query) == nullptr)
        return false;
    // the plan counts tokens of all rows, and work positions inside a row, in int32
    const int64_t row_tokens = (int64_t)max_blocks * d.page_size;
    if ((int64_t)batch * row_tokens >= ((int64_t)1 << 31) ||
        (int64_t)s->units_per_row * (row_tokens + kSliceStartCost) >= ((int64_t)1 << 31))
        return false;
    s->chunk_max = 0;
    s->cap_items = 2 * (int64_t)kMaxGrid; // two partial slots per persistent CTA
    const int64_t units = (int64_t)batch * s->units_per_row;
    auto align = [](size_t x) { return (x + 255) & ~size_t(255); };
    // one combine ticket per unit (16-column units: one per 8-column half)
    const size_t tickets = align(sizeof(int32_t) * (size_t)units * (s->heads_per_cta > 8 ? 2 : 1));
    s->off_ml = tickets;
    s->off_o = s->off_ml + align(sizeof(float2) * (size_t)s->cap_items * s->heads_per_cta);
    s->bytes = s->off_o + align(sizeof(float) * (size_t)s->cap_items * s->heads_per_cta * d.head_dim);
    s->off_plan = 0;
    if (!multi_query) {
        s->off_plan = s->bytes;
        s->bytes += align(plan_layout(batch).bytes);
    }
    return true;
}

} // namespace

size_t decode_plan_bytes(int batch)
{
    return plan_layout(batch).bytes;
}

bool decode_shape(int batch, int max_blocks, int num_q_heads, const pkv_cache_desc &d, DecodeShape *s)
{
    if (d.num_kv_heads <= 0 || num_q_heads % d.num_kv_heads != 0)
        return false;
    s->group = num_q_heads / d.num_kv_heads;
    if (s->group & (s->group - 1))
        return false; // power-of-two groups only
    s->heads_per_cta = heads_per_cta(s->group);
    s->n_sub = s->group / s->heads_per_cta;
    s->units_per_row = d.num_kv_heads * s->n_sub;
    return finish_shape(batch, max_blocks, d, false, s);
}

bool decode_mq_shape(int batch, int max_blocks, int num_q_heads, int max_qlen, const pkv_cache_desc &d,
                     DecodeShape *s)
{
    if (d.num_kv_heads <= 0 || num_q_heads % d.num_kv_heads != 0 || max_qlen < 1)
        return false;
    s->group = num_q_heads / d.num_kv_heads;
    if (s->group & (s->group - 1))
        return false;
    // (query, head) columns of one kv head; a unit takes up to 16 (two 8-wide
    // MMA n-tiles, one per consumer warp, over one pass of the K/V tiles)
    const int64_t cols = (int64_t)s->group * max_qlen;
    int gc = 1;
    while (gc < cols && gc < 16)
        gc <<= 1;
    s->heads_per_cta = gc;
    const int64_t n_sub = (cols + gc - 1) / gc;
    if (n_sub * d.num_kv_heads >= ((int64_t)1 << 24))
        return false;
    s->n_sub = (int)n_sub;
    s->units_per_row = d.num_kv_heads * s->n_sub;
    return finish_shape(batch, max_blocks, d, true, s);
}

int decode_target_items(int device, int head_dim, int heads_per_cta, bool multi_query)
{
    // Per device and kernel: opt in to the kernel's shared memory once and
    // size the persistent grid to the CTAs that fit on all SMs.
    constexpr int kDevices = 64, kKernels = 32;
    static_assert(sizeof(kTable) / sizeof(kTable[0]) <= kKernels, "grid cache too small");
    static int cache[kDevices][kKernels] = {};
    const KernelEntry *e = find_kernel(head_dim, heads_per_cta, multi_query);
    if (e == nullptr || device < 0 || device >= kDevices)
        return 1;
    int &slot = cache[device][kernel_index(e)];
    if (slot == 0) {
        // The plain and the plan-using kernels take the same grid (a plan is
        // made for, and checked against, the grid): the CTAs both fit.
        auto fits = [&](const void *fn) {
            int occ = 1;
            if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)e->smem) != cudaSuccess ||
                cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared) != cudaSuccess ||
                cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, e->threads, e->smem) != cudaSuccess || occ < 1)
                occ = 1;
            return occ;
        };
        int occ = fits(e->fn);
        if (e->use_fn != nullptr) {
            const int o2 = fits(e->use_fn);
            occ = o2 < occ ? o2 : occ;
        }
        if (e->plan_fn != nullptr)
            (void)cudaFuncSetAttribute(e->plan_fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)e->smem);
        const int t = sm_count(device) * occ;
        slot = t > kMaxGrid ? kMaxGrid : t;
    }
    return slot;
}

cudaError_t launch_decode(const DecodeArgs &a, const DecodeMaps &maps, cudaStream_t stream)
{
    const KernelEntry *e = find_kernel(a.desc.head_dim, a.shape.heads_per_cta, a.qo_indptr != nullptr);
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
    p.box_tokens = decode_box_tokens(a.desc.page_size);
    p.with_new = (a.k_new != nullptr) ? 1 : 0;
    p.swizzle = decode_swizzle(a.desc.page_size);
    p.pdl = (a.flags & PKV_DECODE_OVERLAP_PROLOGUE) ? 1 : 0;
    p.early_kv = (a.flags & PKV_DECODE_EARLY_KV) ? 1 : 0;
    p.q_scale = a.q_scale;
    p.qo_indptr = a.qo_indptr;
    p.total_q = a.total_q;
    p.group_shift = 0;
    while ((1 << p.group_shift) < a.shape.group)
        ++p.group_shift;
    p.mq_hi = a.mq_hi;
    p.mq_max = a.mq_max;
    p.mq_own_long = a.mq_own_long;
    p.mq_kv_add = a.mq_kv_add;
    unsigned char *plan = a.shape.off_plan != 0 ? ws + a.shape.off_plan : nullptr;
    p.plan_in = (a.flags & PKV_DECODE_USE_PLAN) ? plan : nullptr;
    p.plan_out = nullptr;
    if ((a.flags & PKV_DECODE_MAKE_PLAN) && plan != nullptr && e->plan_fn != nullptr) {
        // the step plan first: an ordinary launch, one warp per record
        KParams pp = p;
        pp.plan_out = plan;
        int grid = a.grid;
        void *pargs[] = {&pp, &grid};
        const int per_cta = kThreads / 32;
        const cudaError_t err = cudaLaunchKernel(e->plan_fn, dim3((a.grid + per_cta - 1) / per_cta), dim3(kThreads),
                                                 pargs, e->smem, stream);
        if (err != cudaSuccess)
            return err;
    }
    void *args[] = {&p, const_cast<DecodeMaps *>(&maps)};
    const void *fn = p.plan_in != nullptr && e->use_fn != nullptr ? e->use_fn : e->fn;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.grid);
    cfg.blockDim = dim3(e->threads);
    cfg.dynamicSmemBytes = e->smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (p.pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelExC(&cfg, fn, args);
}

} // namespace pkv
