// pkv_tcgen05.cuh -- sm_103a 5th-generation tensor-core helpers: tensor
// memory (TMEM) allocation, tcgen05.mma issue and completion, TMEM <-> register
// moves, and the shared-memory matrix / instruction descriptors the MMA reads.
//
// Conventions used by every caller in this library:
//  - one CTA (cta_group::1); the MMA is issued by one thread;
//  - operands are bf16, staged in shared memory in the 128-byte-swizzled
//    layout a TMA load with CU_TENSOR_MAP_SWIZZLE_128B writes: rows of 128
//    bytes (64 bf16), 8-row atoms of 1024 bytes aligned to 1024;
//  - accumulators are fp32 in TMEM: row i of an M = 128 tile lives in TMEM
//    lane i, column n in TMEM column (base + n).
#pragma once

#include "pkv_device.cuh"

namespace pkv {

// --- tensor memory -------------------------------------------------------

// Allocates `ncols` TMEM columns (a power of two >= 32) for this CTA and writes
// their base address to shared memory.  Executed by one whole warp.
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

// Declares that this CTA allocates no more TMEM (lets other CTAs' allocations
// proceed).  One whole warp.
__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

// Frees what tmem_alloc took.  One whole warp, the same one that allocated.
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Orders this thread's earlier tcgen05 operations before a following
// thread synchronisation (mbarrier arrive, bar.sync).
__device__ __forceinline__ void tc_fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

// Orders later tcgen05 operations after a preceding thread synchronisation.
__device__ __forceinline__ void tc_fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// --- MMA -----------------------------------------------------------------

// Instruction descriptor of kind::f16 with bf16 A and B and an fp32
// accumulator: bits 4-5 D format (1 = f32), 7-9 A format (1 = bf16), 10-12 B
// format (1 = bf16), 15 / 16 A / B major-ness (0 = K-major, 1 = MN-major),
// 17-22 N >> 3, 24-28 M >> 4.
__host__ __device__ constexpr uint32_t tc_idesc_bf16(int M, int N, bool a_mn_major, bool b_mn_major)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(a_mn_major) << 15) | (uint32_t(b_mn_major) << 16) |
           (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

// Shared-memory matrix descriptor for a 128-byte-swizzled operand: bits 0-13
// start address >> 4, 16-29 leading-dimension byte offset >> 4, 32-45
// stride-dimension byte offset >> 4, 46-47 descriptor version (1), 61-63
// layout (2 = 128-byte swizzle).  For a K-major operand the stride offset is
// the distance between 8-row groups and the leading offset is unused; for an
// MN-major operand the leading offset is the distance between 64-element
// column blocks and the stride offset the distance between 8-row K groups.
__device__ __forceinline__ uint64_t tc_sw128_desc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes)
{
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// D[tmem] (+)= A[smem] * B[smem]; `accumulate` = 0 overwrites D.
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "setp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
                 "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
                 : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem].  A (M = 128) sits in TMEM lanes 0..127, one
// row per lane, two bf16 per 32-bit column (lower K index in the low half):
// K = 16 spans 8 columns from `a_tmem`.
__device__ __forceinline__ void tc_mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                               uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "setp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
                 "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
                 : "memory");
}

// Arrives once on `bar` when every tcgen05.mma this thread issued before has
// completed (its shared-memory reads and TMEM writes included).
__device__ __forceinline__ void tc_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_addr(bar))
                 : "memory");
}

// --- TMEM <-> registers (warp-collective; warp w reaches lanes 32*(w%4)..+31)

#define PKV_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), "=r"(r[i + 4]), "=r"(r[i + 5]), \
                  "=r"(r[i + 6]), "=r"(r[i + 7])
#define PKV_W8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), "r"(r[i + 4]), "r"(r[i + 5]), \
                  "r"(r[i + 6]), "r"(r[i + 7])

// 32 consecutive columns of this thread's lane, waited for before returning.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 "
                 "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
                 "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
                 "tcgen05.wait::ld.sync.aligned;"
                 : PKV_R8(0), PKV_R8(8), PKV_R8(16), PKV_R8(24)
                 : "r"(taddr)
                 : "memory");
}

// Writes 32 consecutive columns of this thread's lane and waits for the write.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
                 "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
                 "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};\n\t"
                 "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
                 PKV_W8(0), PKV_W8(8), PKV_W8(16), PKV_W8(24)
                 : "memory");
}

// Writes 16 consecutive columns of this thread's lane and waits for the write.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
                 "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};\n\t"
                 "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
                 PKV_W8(0), PKV_W8(8)
                 : "memory");
}

#undef PKV_R8
#undef PKV_W8

// Makes this thread's generic-proxy shared-memory writes visible to the async
// proxy (TMA, tcgen05.mma operand reads) after a following synchronisation.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 16-byte asynchronous copy global -> shared memory; src_bytes 0 writes zeros.
__device__ __forceinline__ void cp_async16(void *dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all()
{
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// 3-D tiled TMA load with the default L2 policy.
__device__ __forceinline__ void tma_load_3d_plain(void *dst, const CUtensorMap *map, int x, int y, int z,
                                                  uint64_t *bar)
{
    asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
                 "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
                 : "memory");
}

// 4-D and 5-D tiled TMA loads with the default L2 policy.
__device__ __forceinline__ void tma_load_4d_plain(void *dst, const CUtensorMap *map, int c0, int c1, int c2, int c3,
                                                  uint64_t *bar)
{
    asm volatile("cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_addr(dst)),
                 "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void tma_load_5d_plain(void *dst, const CUtensorMap *map, int c0, int c1, int c2, int c3,
                                                  int c4, uint64_t *bar)
{
    asm volatile("cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(smem_addr(dst)),
                 "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4),
                 "r"(smem_addr(bar))
                 : "memory");
}

// --- thread-block clusters ----------------------------------------------

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Barrier over every thread of every CTA of the cluster, with release /
// acquire ordering of shared-memory accesses (mbarrier initialisation
// included) across the cluster.
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// --- CTA pairs (cta_group::2) ---------------------------------------------
// A pair is CTA ranks 2i and 2i+1 of a cluster.  One thread of the even CTA
// issues MMAs with M = 256: rows 0..127 of A and D live in the even CTA
// (its smem / TMEM), rows 128..255 in the odd one at the same addresses, and
// B is split along N -- columns 0..N/2-1 come from the even CTA's smem, the
// rest from the odd CTA's, through the same descriptor.  Every tcgen05
// allocation, MMA and commit of a kernel that pairs CTAs uses cta_group::2.

// Collective over the pair: one warp of each CTA executes it; both receive
// the same TMEM base address.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t *dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// D (+)= A[tmem] * B[smem] over the pair (M = 256).
__device__ __forceinline__ void tc_mma_bf16_ts_pair(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                                    uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "setp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
                 "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
                 : "memory");
}
// D (+)= A[smem] * B[smem] over the pair (M = 256; A rows 0..127 from the
// even CTA's smem, 128..255 from the odd CTA's, through the same descriptor).
__device__ __forceinline__ void tc_mma_bf16_ss_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                    uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "setp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
                 "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
                 : "memory");
}
// Arrives once on the barrier at the same offset in every CTA of `cta_mask`
// when the pair MMAs this thread issued before have completed.
__device__ __forceinline__ void tc_commit_pair_mc(uint64_t *bar, uint16_t cta_mask)
{
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::
                     "r"(smem_addr(bar)),
                 "h"(cta_mask)
                 : "memory");
}
// The same on this CTA's barrier only.
__device__ __forceinline__ void tc_commit_pair(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}
// Arrives on the barrier at the address of `bar` in CTA `rank` of the
// cluster (default semantics: release, the barrier's CTA scope).  Writes the
// barrier's waiter reads through tcgen05 (TMEM, or shared memory an MMA
// reads) are ordered by the tcgen05 / proxy fences before the call.
__device__ __forceinline__ void mbar_arrive_remote(uint64_t *bar, uint32_t rank)
{
    asm volatile("{\n\t.reg .b32 ra;\n\t"
                 "mapa.shared::cluster.u32 ra, %0, %1;\n\t"
                 "mbarrier.arrive.shared::cluster.b64 _, [ra];\n\t}" ::"r"(smem_addr(bar)),
                 "r"(rank)
                 : "memory");
}
// 5-D tiled TMA load into this CTA's shared memory (default L2 policy); c2
// selects the first 64-column block.
__device__ __forceinline__ void tma_load_5d_local(void *dst, const CUtensorMap *map, int c2, int c3, int c4,
                                                  uint64_t *bar)
{
    asm volatile("cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(smem_addr(dst)),
                 "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(0), "r"(c2), "r"(c3), "r"(c4), "r"(smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

} // namespace pkv
