// tc05.cuh -- thin inline-PTX wrappers for the sm_100-family tensor-core path:
// tcgen05 (TMEM allocation, MMA, commit, TMEM loads), mbarrier, and the bulk
// asynchronous copy engine.  Written from the public PTX ISA description of
// these instructions; nothing here is generated.
//
// Conventions used by every kernel in this library:
//   * All MMA operands are bf16, K-major, in the 128-byte swizzled layout:
//     rows of 128 bytes (64 bf16 along K), 8-row atoms of 1024 bytes, the
//     16-byte chunk c of row r stored at chunk position c ^ (r & 7).  Atom
//     bases are 1024-byte aligned.  Operands wider than 64 along K are split
//     into 64-wide "halves", each a separate run of atoms.
//   * Accumulators are fp32 in TMEM, M = 128 (lane i = row i).
#pragma once
#include <cstdint>

namespace gdn {

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Byte offset of element (row, col) in a K-major 128B-swizzled tile whose rows
// hold 64 bf16 (col < 64).
__device__ __forceinline__ uint32_t sw128_offset(uint32_t row, uint32_t col)
{
    return row * 128u + ((((col >> 3) ^ row) & 7u) << 4) + ((col & 7u) << 1);
}
// Byte offset of 16-byte chunk `chunk` (0..7) of row `row`.
__device__ __forceinline__ uint32_t sw128_chunk_offset(uint32_t row, uint32_t chunk)
{
    return row * 128u + (((chunk ^ row) & 7u) << 4);
}

// ---------------------------------------------------------------------------
// Shared-memory matrix descriptor (tcgen05 format):
//   [0,14)  start address >> 4      [16,30) leading byte offset >> 4
//   [32,46) stride byte offset >> 4 [46,48) version = 1
//   [49,52) base offset = 0          [52]    LBO mode = 0
//   [61,64) layout: 2 = 128-byte swizzle
// For K-major swizzled operands the leading offset is unused (set to 1) and
// the stride offset is the distance between 8-row atoms (1024 bytes).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t make_sw128_desc(uint32_t saddr)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)1u << 16;              // LBO (ignored for swizzled K-major)
    d |= (uint64_t)(1024u >> 4) << 32;    // SBO = 1024 bytes
    d |= (uint64_t)1u << 46;              // version
    d |= (uint64_t)2u << 61;              // SWIZZLE_128B
    return d;
}

// Instruction descriptor for kind::f16 with bf16 A/B, fp32 D, both K-major.
__host__ __device__ constexpr uint32_t make_idesc_bf16(uint32_t M, uint32_t N)
{
    return (1u << 4)            // D format: f32
         | (1u << 7)            // A format: bf16
         | (1u << 10)           // B format: bf16
         | ((N >> 3) << 17)     // N / 8
         | ((M >> 4) << 24);    // M / 16
}

// ---------------------------------------------------------------------------
// TMEM allocation (one full warp executes these).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t *slot_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(slot_smem)), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                 :: "r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Make generic-proxy shared-memory writes visible to the async proxy (MMA
// operand reads, bulk copies).
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem]; issued by a single thread.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "setp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                 :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
                 : "memory");
}

// The mbarrier gets one arrival when every tcgen05 op this thread issued so
// far has completed.
__device__ __forceinline__ void mma_commit(uint64_t *mbar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(smem_u32(mbar)) : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane (warp w may only
// touch lanes 32*(w%4) .. 32*(w%4)+31; taddr carries that lane base).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&r)[32])
{
    uint32_t u[32];
    // The load and its wait sit in one asm block so that no use of the
    // registers can be scheduled between them.
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
                 "tcgen05.wait::ld.sync.aligned;"
                 : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]),
                   "=r"(u[6]), "=r"(u[7]), "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]),
                   "=r"(u[12]), "=r"(u[13]), "=r"(u[14]), "=r"(u[15]), "=r"(u[16]),
                   "=r"(u[17]), "=r"(u[18]), "=r"(u[19]), "=r"(u[20]), "=r"(u[21]),
                   "=r"(u[22]), "=r"(u[23]), "=r"(u[24]), "=r"(u[25]), "=r"(u[26]),
                   "=r"(u[27]), "=r"(u[28]), "=r"(u[29]), "=r"(u[30]), "=r"(u[31])
                 : "r"(taddr) : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i)
        r[i] = __uint_as_float(u[i]);
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *mbar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(mbar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *mbar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(smem_u32(mbar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *mbar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(smem_u32(mbar)), "r"(parity) : "memory");
    return ok != 0;
}

// Bounded wait: gives up after ~2^22 polls (each poll may itself suspend for
// a short hardware-defined time), returning false.  Callers turn a false into
// a device status bit and leave the kernel without touching more data.
constexpr uint32_t kWaitPolls = 1u << 22;
__device__ __forceinline__ bool mbar_wait(uint64_t *mbar, uint32_t parity)
{
    for (uint32_t i = 0; i < kWaitPolls; ++i)
        if (mbar_try_wait(mbar, parity))
            return true;
    return false;
}

// Bulk asynchronous global -> shared copy (size a multiple of 16, both
// addresses 16-byte aligned), completing bytes on `mbar`.
__device__ __forceinline__ void bulk_g2s(void *dst_smem, const void *src_gmem, uint32_t bytes,
                                         uint64_t *mbar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
                 "[%0], [%1], %2, [%3];"
                 :: "r"(smem_u32(dst_smem)), "l"(src_gmem), "r"(bytes), "r"(smem_u32(mbar))
                 : "memory");
}

}  // namespace gdn
