// gdn_prefill_out.cu -- chunk outputs of the chunked GDN prefill and the
// optional gated RMSNorm epilogue (JevAny page "Add opt-in fused Qwen3.5
// inference kernels", Summary: chunked kernel followed by a fused gated
// RMSNorm o * rsqrt(mean(o^2) + eps) * w * silu(z)).
//
// All (chunk, value head) units are independent: with S the fp16 state
// entering the chunk (written by the scan kernel) and the chunk's maps from
// the prep kernel,
//   o = scale [Qc | Fc] [S; V]          tcgen05, M = 128, N = 128, K = 192
// The record stores Qc's two K halves and Fc back to back, so a 128-row
// operand starting at any of them has it as rows 0-63 (rows 64-127 are the
// next image and are ignored): the outputs land in TMEM lanes 0-63, one token
// row per lane, and the norm over Dv needs only the two threads that share a
// row.
//
// A persistent grid (one CTA per SM) walks the units with a pipeline, so the
// copies for the next units overlap this unit's products and epilogue.  TMEM
// lanes 32q .. 32q+31 are readable only by warps w with w % 4 == q, so a
// unit's 64 output rows would reach only half of the SM's schedulers; units
// therefore alternate between lane halves: the odd ones read their A operand
// 64 rows (8 KB) earlier in shared memory, which puts their rows in lanes
// 64-127, and two epilogue groups run side by side:
//   warps w % 4 in {0, 1}   epilogue of the even units (lanes 0-63)
//   warps w % 4 in {2, 3}   epilogue of the odd units (lanes 64-127)
//     each: token row 32 (w % 2) + lane, value columns 32 (w / 4) .. + 31;
//     scale, gated RMSNorm, bf16 outputs written over the unit's z tile,
//     tensor-map store
//   warp 16   loads a unit's [Qc | Fc | V | S] run into one of two stages once
//             the products of the unit two before have read that stage
//   warp 17   loads the z tiles into four slots (two per epilogue group),
//             starting before the dependency wait (z is a call input): a
//             group's slot is refilled as soon as the store of the unit that
//             last used it has read it
//   warp 18   issues the 12 MMAs of a unit into one of four accumulators
//             (512 TMEM columns), so a unit's products wait only for the
//             epilogue four units before
// The CTA's unit list (first token and rows of each unit) and the norm
// weights are read before the dependency wait too: cu_seqlens and the weights
// are call inputs, and the chunk index is final before the scan starts.  So is
// the prep kernel's part of the first two record runs ([Qc | Fc | V]): prep
// finished before the scan passed its own wait, and this grid launches only
// after that; the S part of those runs waits.
#include <atomic>

#include "chunks.cuh"
#include "common.cuh"
#include "kernels.h"
#include "tc05.cuh"

namespace gdn {
namespace {

constexpr int kEpiWarps = 16;
constexpr int kLoadWarp = kEpiWarps, kZWarp = kEpiWarps + 1, kMmaWarp = kEpiWarps + 2;
constexpr int kThreads = (kEpiWarps + 3) * 32;
// Run stage: the record's [Qc | Fc | V | S] run (72 KB) as copied.
constexpr uint32_t kOffQc0 = 0, kOffQc1 = 8192, kOffFc = 16384, kOffV = 24576, kOffS = 40960;
constexpr uint32_t kRunBytes = 73728;
constexpr int kRunStages = 2;
// Tile slots: a unit's 64 x 128 bf16 z tile (tensor-map copy, dk halves of
// 8 KB, 128-byte swizzle), overwritten in place by its outputs, which a
// tensor-map store then copies out.  Slots 2g and 2g + 1 belong to group g.
constexpr uint32_t kOffTile = kRunStages * kRunBytes;
constexpr uint32_t kTileBytes = 16384;
constexpr int kSlots = 4;
constexpr uint32_t kOffSmall = kOffTile + kSlots * kTileBytes;
constexpr int kAccs = 4;                     // 128-column accumulators
constexpr uint32_t kTmemCols = 512;
constexpr int kTab = 256;                    // units listed ahead (more are located on the way)
constexpr uint32_t kBarEpi = 1, kCntEpi = 256;   // barrier 1 + g: the eight warps of epilogue group g
constexpr float kScale = 0.088388347648318440550f;  // 1/sqrt(128)

struct Small {
    float red[2][4][64];       // per epilogue group: row sums of squares of each 32-column quarter
    int2 tab[kTab];            // unit j of this CTA: (first token, valid rows); rows 0 past the last chunk
    uint4 nw[kD / 8];          // the gated norm's weights (bf16)
    uint64_t full[kRunStages]; // run landed
    uint64_t rfree[kRunStages];// run read by the products
    uint64_t zfull[kSlots];    // z tile landed
    uint64_t zfree[kSlots];    // slot's outputs read by their store: the slot may be refilled
    uint64_t afull[kAccs];     // accumulator written
    uint64_t efree[kAccs];     // accumulator read by the epilogue
    uint32_t tmem_base;
    int fail;
};
constexpr uint32_t kSmemBytes = kOffSmall + ((sizeof(Small) + 127) / 128) * 128 + 1024;
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

// Global chunk gc of the packed sequences: first token and valid rows.
__device__ __forceinline__ bool locate_chunk(const PrefillArgs &p, int gc, int &tok0, int &L)
{
    int n;
    bool bad;
    return find_chunk(p, gc, n, tok0, L, bad);
}

__device__ __forceinline__ bool wait_bar(Small *s, uint64_t *bar, uint32_t parity, uint32_t *status)
{
    if (*reinterpret_cast<volatile int *>(&s->fail))
        return false;
    if (!mbar_wait(bar, parity)) {
        s->fail = 1;
        set_status(status, kStatusWaitTimeout);
        return false;
    }
    return true;
}

template <bool kNorm>
__global__ void __launch_bounds__(kThreads, 1)
out_kernel(PrefillArgs p, const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_o)
{
    const int hv = p.hv, units = p.max_chunks * hv;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // this CTA's units: u = blockIdx.x + j * gridDim.x, j < nj; the live ones
    // (chunks that exist) come first, since the chunk grows with u
    const int nj = (units - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;

    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Small *s = reinterpret_cast<Small *>(sm + kOffSmall);
    const uint32_t sbase = smem_u32(sm);

    if (tid == 0) {
        for (int i = 0; i < kRunStages; ++i) {
            mbar_init(&s->full[i], 1);
            mbar_init(&s->rfree[i], 1);
        }
        for (int i = 0; i < kSlots; ++i) {
            mbar_init(&s->zfull[i], 1);
            mbar_init(&s->zfree[i], 1);
        }
        for (int i = 0; i < kAccs; ++i) {
            mbar_init(&s->afull[i], 1);
            mbar_init(&s->efree[i], 1);
        }
        mbar_fence_init();
        s->fail = 0;
    }
    if (warp == 0) {
        tmem_alloc(&s->tmem_base, kTmemCols);
        tmem_relinquish();
        tc_fence_before();
    }
    if (warp == kLoadWarp) {
        const int nt = nj < kTab ? nj : kTab;
        for (int j = lane; j < nt; j += 32) {
            int tok0 = 0, L = 0;
            const int gc = ((int)blockIdx.x + j * (int)gridDim.x) / hv;
            s->tab[j] = locate_chunk(p, gc, tok0, L) ? make_int2(tok0, L) : make_int2(0, 0);
        }
    }
    if (kNorm && tid < kD / 8)
        s->nw[tid] = reinterpret_cast<const uint4 *>(p.norm_w)[tid];
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = s->tmem_base;
    // Unit j: head, first token and valid rows; false past the last chunk.
    auto unit_at = [&](int j, int &h, int &tok0, int &L) -> bool {
        const int u = (int)blockIdx.x + j * (int)gridDim.x, gc = u / hv;
        h = u - gc * hv;
        if (j < kTab) {
            const int2 e = s->tab[j];
            tok0 = e.x;
            L = e.y;
            return L > 0;
        }
        return locate_chunk(p, gc, tok0, L);
    };

    if (warp == kZWarp) {
        if (kNorm && lane == 0) {
            // ------------------------------------------------------ z loader
            // z is a call input: no dependency wait
            int issued[kSlots] = {0, 0, 0, 0};
            for (int j = 0; j < nj; ++j) {
                int h, tok0, L;
                if (!unit_at(j, h, tok0, L))
                    break;
                const int g = j & 1, i = j >> 1, zid = 2 * g + (i & 1);
                // the group's unit before last used this slot: its store must have read it
                if (i >= 2 && !wait_bar(s, &s->zfree[zid], (uint32_t)((i >> 1) - 1) & 1, p.status))
                    break;
                unsigned char *tile = sm + kOffTile + zid * kTileBytes;
                mbar_arrive_expect_tx(&s->zfull[zid], kTileBytes);
                tma_load_3d(tile, &tm_z, 0, h, tok0, &s->zfull[zid]);
                tma_load_3d(tile + 8192, &tm_z, 64, h, tok0, &s->zfull[zid]);
                ++issued[zid];
            }
            // no copy may still be landing in shared memory when the CTA exits
            if (*reinterpret_cast<volatile int *>(&s->fail)) {
                for (int i = 0; i < kSlots; ++i)
                    if (issued[i] > 0)
                        mbar_wait(&s->zfull[i], (uint32_t)(issued[i] - 1) & 1);
            }
        }
        __syncwarp();
    } else {
        // Launched early behind the scan kernel, whose S records are read
        // below.  The prep kernel's part of the first two runs ([Qc | Fc | V],
        // 40 KB of 72) is requested before the dependency wait: prep finished
        // before the scan passed its own wait, and this grid launches after
        // that.  Only the S part waits.
        constexpr uint32_t kPrepPart = (uint32_t)(kWsS - kWsQc0);
        int early = 0;   // runs whose prep part is in flight (loader lane)
        if (warp == kLoadWarp && lane == 0) {
            for (; early < kRunStages && early < nj; ++early) {
                int h, tok0, L;
                if (!unit_at(early, h, tok0, L))
                    break;
                const unsigned char *rec = p.workspace + (size_t)((int)blockIdx.x + early * (int)gridDim.x) * kPerVHead;
                mbar_arrive_expect_tx(&s->full[early], kRunBytes);
                bulk_g2s(sm + early * kRunBytes, rec + kWsQc0, kPrepPart, &s->full[early]);
            }
        }
        grid_dep_wait();
        if (warp == kLoadWarp) {
            if (lane == 0) {
                // ---------------------------------------------------- loader
                int issued[kRunStages] = {0, 0};
                for (int j = 0; j < nj; ++j) {
                    int h, tok0, L;
                    if (!unit_at(j, h, tok0, L))
                        break;
                    const int rs = j & 1;
                    // the unit two before used this stage: its products must have read it
                    if (j >= kRunStages && !wait_bar(s, &s->rfree[rs], (uint32_t)((j >> 1) - 1) & 1, p.status))
                        break;
                    unsigned char *stage = sm + rs * kRunBytes;
                    const unsigned char *rec = p.workspace + (size_t)((int)blockIdx.x + j * (int)gridDim.x) * kPerVHead;
                    if (j < early) {   // the S part of a run whose prep part is on its way
                        bulk_g2s(stage + kPrepPart, rec + kWsS, kRunBytes - kPrepPart, &s->full[rs]);
                    } else {
                        mbar_arrive_expect_tx(&s->full[rs], kRunBytes);
#pragma unroll
                        for (int q = 0; q < 3; ++q)
                            bulk_g2s(stage + q * 24576, rec + kWsQc0 + q * 24576, 24576, &s->full[rs]);
                    }
                    ++issued[rs];
                }
                if (*reinterpret_cast<volatile int *>(&s->fail)) {
                    for (int i = 0; i < kRunStages; ++i)
                        if (issued[i] > 0)
                            mbar_wait(&s->full[i], (uint32_t)(issued[i] - 1) & 1);
                }
            }
            __syncwarp();
        } else if (warp == kMmaWarp) {
            if (lane == 0) {
                // ---------------------------------------------------- issuer
                constexpr uint32_t idesc = make_idesc_f16(128, 128, false, true);
                for (int j = 0; j < nj; ++j) {
                    int h, tok0, L;
                    if (!unit_at(j, h, tok0, L))
                        break;
                    const int rs = j & 1, a = j & (kAccs - 1);
                    // odd units: A starts 64 rows (8 KB) early, so the unit's rows
                    // are rows 64-127 (the rows before are whatever precedes them
                    // in shared memory, and their accumulator lanes are not read)
                    const uint32_t stb = sbase + rs * kRunBytes, stg = stb - (rs ? 8192u : 0u);
                    const uint32_t d = tbase + a * 128;
                    bool ok = wait_bar(s, &s->full[rs], (uint32_t)(j >> 1) & 1, p.status);
                    if (ok && j >= kAccs)   // accumulator a read by the epilogue four units ago
                        ok = wait_bar(s, &s->efree[a], (uint32_t)((j >> 2) - 1) & 1, p.status);
                    if (ok) {
                        tc_fence_after();
                        const uint64_t bv = make_desc(stb + kOffV, 4096, 512, kSw64);
                        const uint64_t bs = make_desc(stb + kOffS, 8192, 512, kSw64);
                        const uint64_t af = make_desc(stg + kOffFc, 16, 1024, kSw128);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)   // Fc V over the chunk's 64 tokens
                            mma_f16(d, af + (uint64_t)(kk * 2), bv + (uint64_t)(kk * 64), idesc, kk != 0);
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) {  // Qc S over the 128 state rows
                            const uint64_t aq = make_desc(stg + (kk < 4 ? kOffQc0 : kOffQc1), 16, 1024, kSw128);
                            mma_f16(d, aq + (uint64_t)((kk & 3) * 2), bs + (uint64_t)(kk * 64), idesc, 1u);
                        }
                    }
                    mma_commit(&s->afull[a]);
                    mma_commit(&s->rfree[rs]);
                }
            }
            __syncwarp();
        } else {
            // -------------------------------------------------------- epilogue
            const int qd = warp & 3, g = qd >> 1, cq = warp >> 2;   // lane quadrant, group, column quarter
            const int row = 32 * (qd & 1) + lane;                    // token row of the unit
            const bool lead = lane == 0 && warp == 2 * g;            // the group's store thread
            const uint32_t bar = kBarEpi + g;
            const int c0 = (cq & 1) * 4;   // this thread's 16-byte chunks 4 (cq & 1) .. of dk half cq / 2
            int i = 0;                     // the group's own unit count
            for (int j = g; j < nj; j += 2) {
                int h, tok0, L;
                if (!unit_at(j, h, tok0, L))
                    break;
                const int a = j & (kAccs - 1), zid = 2 * g + (i & 1);
                unsigned char *tile = sm + kOffTile + zid * kTileBytes;
                unsigned char *yt = tile + (cq >> 1) * 8192;
                if (lead) {
                    // the group's earlier stores have read their tiles: this
                    // unit's slot may be written, and the last unit's refilled
                    bulk_wait_read<0>();
                    if (i >= 1)
                        mbar_arrive(&s->zfree[2 * g + ((i - 1) & 1)]);
                }
                if (kNorm)
                    wait_bar(s, &s->zfull[zid], (uint32_t)(i >> 1) & 1, p.status);   // z tile visible
                wait_bar(s, &s->afull[a], (uint32_t)(j >> 2) & 1, p.status);
                __syncwarp();   // converged (after the lead's wait) for the .aligned TMEM load
                tc_fence_after();
                float o[32];
                tmem_ld32(tbase + a * 128 + ((uint32_t)(32 * qd) << 16) + cq * 32, o);
#pragma unroll
                for (int q = 0; q < 32; ++q) o[q] *= kScale;
                if (kNorm) {
                    float ss = 0.f;
#pragma unroll
                    for (int q = 0; q < 32; ++q) ss = fmaf(o[q], o[q], ss);
                    s->red[g][cq][row] = ss;
                    named_sync(bar, kCntEpi);
                    const float rn = rsqrtf((s->red[g][0][row] + s->red[g][1][row] + s->red[g][2][row]
                                             + s->red[g][3][row]) * (1.f / kD) + p.eps);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        float zf[8], wf[8];
                        unpack8(*reinterpret_cast<const uint4 *>(yt + sw128_chunk_offset(row, c0 + q)), zf);
                        unpack8(s->nw[cq * 4 + q], wf);
#pragma unroll
                        for (int e = 0; e < 8; ++e)   // silu(z) = z / (1 + e^-z)
                            o[8 * q + e] = o[8 * q + e] * rn * wf[e] * __fdividef(zf[e], 1.f + __expf(-zf[e]));
                    }
                } else {
                    named_sync(bar, kCntEpi);   // the lead's wait for the slot
                }
                if (L == kC) {
                    // whole chunk: bf16 outputs over this thread's own z chunks,
                    // then one tensor-map store per dk half
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        float v[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) v[e] = o[8 * q + e];
                        *reinterpret_cast<uint4 *>(yt + sw128_chunk_offset(row, c0 + q)) = pack8(v);
                    }
                } else if (row < L) {
                    // a sequence's ragged last chunk: the rows past it belong to the
                    // next sequence, so each valid row is stored on its own
                    uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(p.out)
                                                           + ((size_t)(tok0 + row) * hv + h) * kD + cq * 32);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        float v[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) v[e] = o[8 * q + e];
                        dst[q] = pack8(v);
                    }
                }
                // one proxy fence for both directions: the tile's generic
                // writes before the tensor-map store reads it, and the
                // generic reads of z before the z loader's TMA refills it
                fence_async_smem();
                tc_fence_before();
                named_sync(bar, kCntEpi);   // accumulator and z read, tile complete, red consumed
                if (lead) {
                    mbar_arrive(&s->efree[a]);   // the accumulator is free
                    if (L == kC) {
                        tma_store_3d(&tm_o, 0, h, tok0, tile);
                        tma_store_3d(&tm_o, 64, h, tok0, tile + 8192);
                        bulk_commit();
                    }
                }
                ++i;
            }
            if (lead)
                bulk_wait_all();   // every output tile copy complete before exit
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tbase, kTmemCols);
    }
}

}  // namespace

cudaError_t launch_prefill_out(const PrefillArgs &p, cudaStream_t stream)
{
    // the shared-memory attribute and the SM count, once per device (a repeat
    // from a racing host thread stores the same values)
    static std::atomic<int> sm_count[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    int sms = sm_count[dev].load(std::memory_order_relaxed);
    if (!sms) {
        cudaError_t e = cudaFuncSetAttribute(out_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(out_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e == cudaSuccess)
            e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess)
            return e;
        sm_count[dev].store(sms, std::memory_order_relaxed);
    }
    CUtensorMap tz, to;
    if (!encode_tile_map(&to, p.out, p.hv, p.total_tokens, (int64_t)p.hv * kD, kD))
        return cudaErrorInvalidValue;
    if (p.z) {
        if (!encode_tile_map(&tz, p.z, p.hv, p.total_tokens, p.in.z.t, p.in.z.h))
            return cudaErrorInvalidValue;
    } else {
        tz = to;   // unused without the epilogue
    }
    const int units = p.max_chunks * p.hv;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(units < sms ? units : sms);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = p.z ? cudaLaunchKernelEx(&cfg, out_kernel<true>, p, tz, to)
                        : cudaLaunchKernelEx(&cfg, out_kernel<false>, p, tz, to);
    if (e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

}  // namespace gdn
