// tcgen05 (5th-generation tensor core) helpers for sm_103a: tensor-memory
// allocation, shared-memory matrix descriptors, MMA issue and commit, TMEM
// loads/stores, mbarriers with bounded waits, and named barriers.
//
// Operand layout used throughout (no swizzle): a "core matrix" is 8 rows of
// 16 contiguous bytes (128 B). For both K-major and MN-major operands the
// descriptor's leading byte offset (LBO) is the distance between core
// matrices adjacent along K and the stride byte offset (SBO) the distance
// between core matrices adjacent along M (or N). For M = 64 the accumulator
// row r lives in TMEM lane (r % 16) + 32 * (r / 16); for M = 128 in lane r.
// (These conventions were checked on GB300 against torch matmuls of every
// combination of K-/MN-major A and B, bf16 and E4M3, M = 64 and 128.)
#pragma once

#include <cstdint>

namespace smla {
namespace umma {

// Shared-memory matrix descriptor (no swizzle).
__device__ __forceinline__ uint64_t desc(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}

// Shared-memory matrix descriptor for the 128-byte swizzled layout (the
// layout a TMA copy with CU_TENSOR_MAP_SWIZZLE_128B writes): rows of 128 B in
// atoms of 8 rows (1 KB), the 16-byte chunk index XORed with the row index in
// the atom; the atom base must be 1024-byte aligned. K-major: SBO = distance
// between 8-row atoms, LBO unused, a K step inside the 128-byte row moves the
// start address. MN-major: LBO = distance between atoms along M/N (the next
// 64 bf16 elements), SBO = distance between atoms along K (the next 8 rows).
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    return desc(saddr, lbo, sbo) | (2ull << 61);
}

// Instruction descriptor: fp32 accumulate; fmt 0/1 = f16/bf16 (kind::f16) or
// 0 = e4m3 (kind::f8f6f4); major 0 = K-major, 1 = MN-major.
__host__ __device__ constexpr uint32_t idesc(int M, int N, int afmt, int bfmt, int amaj, int bmaj)
{
    return (1u << 4) | ((uint32_t)afmt << 7) | ((uint32_t)bfmt << 10) | ((uint32_t)amaj << 15) |
           ((uint32_t)bmaj << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate)
{
    asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
                 "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate)
{
    asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
                 "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
                 "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

// D (tensor memory) (+)= A (tensor memory) . B (shared memory), kind::f16.
// A [M x K] sits in lanes 0..M-1 (row = lane), two consecutive K elements
// per 32-bit column (the even one in the low half).
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                           uint32_t accumulate)
{
    asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
                 "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate));
}

// Arrive once on the mbarrier at shared-memory offset `mbar` of every CTA of
// the cluster in `cta_mask` when every tcgen05 op issued so far by this
// thread is done.
__device__ __forceinline__ void commit_multicast(uint32_t mbar, uint16_t cta_mask)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n" ::"r"(mbar),
                 "h"(cta_mask)
                 : "memory");
}

// Arrive once on `mbar` when every tcgen05 op issued so far by this thread is done.
__device__ __forceinline__ void commit(uint32_t mbar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(mbar)
                 : "memory");
}

__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }
// Make this thread's generic-proxy shared-memory writes visible to the tensor core.
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }

__device__ __forceinline__ void alloc(uint32_t dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(dst_smem), "r"(ncols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
}

__device__ __forceinline__ void dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols));
}

// 32 lanes x 16 consecutive 32-bit columns (warp-wide; lane base = 32 * (warp % 4)).
__device__ __forceinline__ void ld16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                   "=r"(r[15])
                 : "r"(taddr));
}

// 32 lanes x 32 consecutive 32-bit columns (warp-wide).
__device__ __forceinline__ void ld32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                   "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
                   "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
                   "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr));
}

// 32 lanes x 8 consecutive 32-bit columns (warp-wide).
__device__ __forceinline__ void ld8(uint32_t taddr, uint32_t (&r)[8])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
}

__device__ __forceinline__ void st8(uint32_t taddr, const uint32_t (&r)[8])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};\n" ::"r"(taddr), "r"(r[0]),
                 "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}

__device__ __forceinline__ void st16(uint32_t taddr, const uint32_t (&r)[16])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
                 "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
                 : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns (warp-wide).
__device__ __forceinline__ void st32(uint32_t taddr, const uint32_t (&r)[32])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
                 "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
                 "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
                 "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
                 "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
                 : "memory");
}

// 16 lanes x 4 repetitions of 8 consecutive 32-bit columns (warp-wide; the
// lane base is 32 * (warp % 4) or 16 more). Thread T's registers 4i..4i+3 go
// to repetition i as (lane T/4, column 2(T%4)), (lane T/4, column 2(T%4)+1),
// (lane T/4+8, column 2(T%4)), (lane T/4+8, column 2(T%4)+1).
__device__ __forceinline__ void st16x256b_x4(uint32_t taddr, const uint32_t (&r)[16])
{
    asm volatile("tcgen05.st.sync.aligned.16x256b.x4.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
                 "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
                 : "memory");
}

__device__ __forceinline__ void wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }
__device__ __forceinline__ void wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }

__device__ __forceinline__ void mbar_init(uint32_t mbar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(mbar), "r"(count));
}

__device__ __forceinline__ void mbar_init_fence() { asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory"); }

// Arrive once and add `bytes` to the transaction count of the current phase.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t mbar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(mbar), "r"(bytes) : "memory");
}

// TMA row gather: rows r0..r3, columns [x, x + box width) of a 2-D tensor map
// into shared memory at dst (4 rows of the box, in the map's swizzle), bytes
// counted on mbar. Rows outside the tensor are filled with zeros.
__device__ __forceinline__ void tma_gather4(uint32_t dst, const void *tmap, int x, int r0, int r1, int r2, int r3,
                                            uint32_t mbar)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];\n" ::"r"(dst),
                 "l"(tmap), "r"(x), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(mbar)
                 : "memory");
}

// tma_gather4 delivered to the same shared-memory offset (dst) in every CTA
// of the cluster in `cta_mask`; each destination CTA counts the bytes on its
// own mbarrier at offset `mbar`.
__device__ __forceinline__ void tma_gather4_multicast(uint32_t dst, const void *tmap, int x, int r0, int r1, int r2,
                                                      int r3, uint32_t mbar, uint16_t cta_mask)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes.multicast::cluster"
                 " [%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;\n" ::"r"(dst),
                 "l"(tmap), "r"(x), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(mbar), "h"(cta_mask)
                 : "memory");
}

// TMA tile load of the box at (x, y) of a 2-D tensor map into shared memory at
// dst (in the map's swizzle), bytes counted on mbar; out-of-range parts of the
// box are filled with zeros.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *tmap, int x, int y, uint32_t mbar)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%2, %3}], [%4];\n" ::"r"(dst),
                 "l"(tmap), "r"(x), "r"(y), "r"(mbar)
                 : "memory");
}

// Bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned)
// from global to shared memory, bytes counted on mbar.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t mbar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(mbar)
                 : "memory");
}

// Prefetch of `bytes` (a multiple of 16, 16-byte aligned) of global memory
// into L2, without waiting.
__device__ __forceinline__ void prefetch_l2(const void *src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(src), "r"(bytes) : "memory");
}

// Bulk copy of `bytes` (a multiple of 16; 16-byte aligned offsets) from this
// CTA's shared memory at src to the same-numbered shared-memory offset dst of
// cluster CTA `rank`, counted on that CTA's mbarrier at offset `mbar`.
__device__ __forceinline__ void bulk_copy_s2peer(uint32_t dst, uint32_t src, uint32_t bytes, uint32_t mbar,
                                                 uint32_t rank)
{
    uint32_t rdst, rbar;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(rdst) : "r"(dst), "r"(rank));
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(rbar) : "r"(mbar), "r"(rank));
    asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(rdst),
                 "r"(src), "r"(bytes), "r"(rbar)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t mbar)
{
    asm volatile("{\n.reg .b64 st;\nmbarrier.arrive.shared::cta.b64 st, [%0];\n}\n" ::"r"(mbar) : "memory");
}

// Arrive once, with release semantics at cluster scope, on the mbarrier at
// shared-memory offset `mbar` of cluster CTA `rank` (which may be this CTA).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t mbar, uint32_t rank)
{
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(remote) : "r"(mbar), "r"(rank));
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];\n" ::"r"(remote) : "memory");
}

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
    return r;
}

// Barrier over every thread of every CTA of the cluster (release / acquire).
__device__ __forceinline__ void cluster_barrier()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

__device__ __forceinline__ uint64_t globaltimer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;\n" : "=l"(t));
    return t;
}

// Wait for phase `parity` of `mbar` to complete, for at most 2^32 SM cycles
// (about 2 s at 2 GHz). Returns false on timeout (the caller records the
// error and stops waiting). The bound is kept on the SM's cycle counter,
// which is read in a few cycles, so a phase that completes is seen at once.
__device__ __forceinline__ bool mbar_wait(uint32_t mbar, uint32_t parity)
{
    uint32_t done = 0;
    asm volatile("{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
                 : "=r"(done)
                 : "r"(mbar), "r"(parity)
                 : "memory");
    if (done)
        return true;
    const long long c0 = clock64();
    while (true) {
        asm volatile("{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
                     : "=r"(done)
                     : "r"(mbar), "r"(parity)
                     : "memory");
        if (done)
            return true;
        if (clock64() - c0 > (1ll << 32))
            return false;
    }
}

// Programmatic dependent launch: allow the next kernel in the stream to be
// scheduled now (it still waits in its own grid_wait), and wait until the
// previous kernel has completed and its memory operations are visible.
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }
__device__ __forceinline__ void grid_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }

// Named barrier over `count` threads (ids 1..15; 0 is __syncthreads).
__device__ __forceinline__ void named_bar(int id, int count)
{
    asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(count) : "memory");
}

} // namespace umma
} // namespace smla
