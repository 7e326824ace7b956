// tc05.cuh -- thin inline-PTX wrappers for the sm_100-family tensor-core path:
// tcgen05 (TMEM allocation, MMA, commit, TMEM loads), mbarrier, and the bulk
// asynchronous copy engine.  Written from the public PTX ISA description of
// these instructions; nothing here is generated.
//
// Conventions used by every kernel in this library:
//   * MMA operands are 16-bit (bf16 or fp16) in swizzled shared-memory
//     layouts: K-major or MN-major with 128-byte rows (64 elements; 8-row
//     atoms of 1024 bytes, 16-byte chunk c of row r at position c ^ (r & 7)),
//     or MN-major with 64-byte rows (32 elements; 8-row atoms of 512 bytes,
//     chunk c of row r at c ^ ((r >> 1) & 3)).  Atom bases are aligned to the
//     atom size.  Extents wider than one row are split into "halves", each a
//     separate run of atoms.
//   * Accumulators are fp32 in TMEM, M = 128 (lane i = row i).
#pragma once
#include <cstdint>

namespace gdn {

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` in a K-major
// 128B-swizzled tile whose rows hold 64 16-bit elements.
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

// General form: layout 2 = 128-byte swizzle, 4 = 64-byte swizzle.
//   K-major 128B:  rows of 64 K elements, SBO = 1024 between 8-row atoms.
//   MN-major 128B: rows of 64 MN elements, one row per K index; SBO = 1024
//                  between groups of 8 K rows, LBO = distance between
//                  successive 64-wide MN blocks.
//   MN-major 64B:  rows of 32 MN elements (64 bytes), one per K index;
//                  SBO = 512 between groups of 8 K rows (atoms of 512 bytes).
__device__ __forceinline__ uint64_t make_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                              uint32_t layout)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1u << 46;
    d |= (uint64_t)layout << 61;
    return d;
}
constexpr uint32_t kSw128 = 2, kSw64 = 4;

// Byte offset of 16-byte chunk `chunk` (0..3) of row `row` in a 64-byte-row
// swizzled tile (atoms of 8 rows x 64 bytes, 512-byte aligned).
__device__ __forceinline__ uint32_t sw64_chunk_offset(uint32_t row, uint32_t chunk)
{
    return row * 64u + (((chunk ^ (row >> 1)) & 3u) << 4);
}

// Instruction descriptors for kind::f16 with fp32 D; both operands share one
// type (bf16, or fp16).  a_mn / b_mn select MN-major (transposed) operands;
// the default is K-major.
__host__ __device__ constexpr uint32_t make_idesc_f16(uint32_t M, uint32_t N, bool a_mn = false,
                                                      bool b_mn = false)
{
    return (1u << 4)            // D format: f32
         | (0u << 7)            // A format: f16
         | (0u << 10)           // B format: f16
         | ((a_mn ? 1u : 0u) << 15)
         | ((b_mn ? 1u : 0u) << 16)
         | ((N >> 3) << 17)     // N / 8
         | ((M >> 4) << 24);    // M / 16
}
__host__ __device__ constexpr uint32_t make_idesc_bf16(uint32_t M, uint32_t N, bool a_mn = false,
                                                       bool b_mn = false)
{
    return (1u << 4)            // D format: f32
         | (1u << 7)            // A format: bf16
         | (1u << 10)           // B format: bf16
         | ((a_mn ? 1u : 0u) << 15)
         | ((b_mn ? 1u : 0u) << 16)
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

// D[tmem] (+)= A[smem] * B[smem] (tcgen05 kind::f16: bf16 or fp16 operands,
// the type given by the instruction descriptor); issued by a single thread.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
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

// Two 32-column loads (addresses ta, tb) in flight together, one wait.
__device__ __forceinline__ void tmem_ld32x2(uint32_t ta, uint32_t tb, float (&a)[32], float (&b)[32])
{
    uint32_t u[32], v[32];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n\t"
                 "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
                 "{%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
                 "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];\n\t"
                 "tcgen05.wait::ld.sync.aligned;"
                 : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]),
                   "=r"(u[6]), "=r"(u[7]), "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]),
                   "=r"(u[12]), "=r"(u[13]), "=r"(u[14]), "=r"(u[15]), "=r"(u[16]),
                   "=r"(u[17]), "=r"(u[18]), "=r"(u[19]), "=r"(u[20]), "=r"(u[21]),
                   "=r"(u[22]), "=r"(u[23]), "=r"(u[24]), "=r"(u[25]), "=r"(u[26]),
                   "=r"(u[27]), "=r"(u[28]), "=r"(u[29]), "=r"(u[30]), "=r"(u[31]),
                   "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]),
                   "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]),
                   "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]),
                   "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]),
                   "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]),
                   "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
                 : "r"(ta), "r"(tb) : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        a[i] = __uint_as_float(u[i]);
        b[i] = __uint_as_float(v[i]);
    }
}

// The sum of two 16-column TMEM loads (addresses ta, tb): both in flight
// together, one wait.
__device__ __forceinline__ void tmem_ld16_sum2(uint32_t ta, uint32_t tb, float (&r)[16])
{
    uint32_t u[16], v[16];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%32];\n\t"
                 "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
                 "{%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%33];\n\t"
                 "tcgen05.wait::ld.sync.aligned;"
                 : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]),
                   "=r"(u[6]), "=r"(u[7]), "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]),
                   "=r"(u[12]), "=r"(u[13]), "=r"(u[14]), "=r"(u[15]),
                   "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]),
                   "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]),
                   "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
                 : "r"(ta), "r"(tb) : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i)
        r[i] = __uint_as_float(u[i]) + __uint_as_float(v[i]);
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
// try_wait suspends the thread until the phase completes or about
// kSuspendNs nanoseconds pass, so waiting threads leave the issue slots to the
// others instead of polling.
constexpr uint32_t kSuspendNs = 20000;
__device__ __forceinline__ bool mbar_try_wait(uint64_t *mbar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(smem_u32(mbar)), "r"(parity), "n"(kSuspendNs) : "memory");
    return ok != 0;
}

// Plain arrive (release, CTA scope) on a local mbarrier.
__device__ __forceinline__ void mbar_arrive(uint64_t *mbar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_u32(mbar)) : "memory");
}

// Non-blocking test of a phase (unlike try_wait it never suspends the thread).
__device__ __forceinline__ bool mbar_test(uint64_t *mbar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(smem_u32(mbar)), "r"(parity) : "memory");
    return ok != 0;
}

// Named CTA barriers: producers arrive without waiting, the consumer syncs.
// The non-.aligned forms, which do not require the warp to arrive converged
// (the .aligned bar.arrive / bar.sync leave a split warp undefined); callers
// still reconverge after one-lane branches with __syncwarp().
__device__ __forceinline__ void named_arrive(uint32_t id, uint32_t nthreads)
{
    asm volatile("barrier.cta.arrive %0, %1;" :: "r"(id), "r"(nthreads) : "memory");
}
__device__ __forceinline__ void named_sync(uint32_t id, uint32_t nthreads)
{
    asm volatile("barrier.cta.sync %0, %1;" :: "r"(id), "r"(nthreads) : "memory");
}

// Bounded wait: gives up after kWaitPolls suspended polls (~2 s), returning
// false.  Callers turn a false into a device status bit and leave the kernel
// without touching more data.
constexpr uint32_t kWaitPolls = 100000;
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

// Bulk prefetch of a global range into L2 (address 16-byte aligned, size a
// multiple of 16); nothing waits for it.
__device__ __forceinline__ void bulk_prefetch_l2(const void *src_gmem, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(src_gmem), "r"(bytes) : "memory");
}

// Bulk shared -> global copy, committed as its own bulk group of the issuing
// thread (both addresses 16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_s2g(void *dst_gmem, const void *src_smem, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                 :: "l"(dst_gmem), "r"(smem_u32(src_smem)), "r"(bytes) : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until at most N of this thread's bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read()
{
    asm volatile("cp.async.bulk.wait_group.read %0;" :: "n"(N) : "memory");
}
// Wait until every bulk group of this thread has completed (writes visible).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Tiled 3-D tensor copy global -> shared through a tensor map (a CUtensorMap
// kernel parameter), completing bytes on `mbar`.  c0 is the innermost
// coordinate; c0 * element size must be a multiple of 16 bytes.  Boxes that
// reach past the tensor are filled with zeros and still count in full.
__device__ __forceinline__ void tma_load_3d(void *dst_smem, const void *tmap, int c0, int c1, int c2,
                                            uint64_t *mbar)
{
    asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
                 "[%0], [%1, {%2, %3, %4}], [%5];"
                 :: "r"(smem_u32(dst_smem)), "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(mbar))
                 : "memory");
}

// Tiled 3-D tensor copy shared -> global through a tensor map, committed as a
// bulk group of the issuing thread.  Only the part of the box inside the
// tensor is written.
__device__ __forceinline__ void tma_store_3d(const void *tmap, int c0, int c1, int c2, const void *src_smem)
{
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];"
                 :: "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(src_smem)) : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start before the previous kernel in the stream ends;
// grid_dep_wait() blocks until that kernel has completed and its memory
// operations are visible.  grid_dep_launch() lets the next such kernel
// start launching once every CTA of this grid has called it or exited.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------------------
// Warp-level 16x16 fp16 products for block algebra that is too small for a
// tcgen05 tile (16 x 16 x 16 blocks, latency-bound).  ldmatrix.x4 loads four
// 8x8 b16 matrices whose rows are addressed by lanes 0-7, 8-15, 16-23, 24-31.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr) : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr) : "memory");
}
// d = a * b + d for one m16n8k16 tile, fp16 operands, fp32 accumulate.
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
                 "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

}  // namespace gdn
