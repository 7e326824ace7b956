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
// A persistent grid (one CTA per SM) walks the units with a two-stage
// pipeline, so the copies for the next units overlap this unit's products and
// epilogue.  TMEM lanes 32q .. 32q+31 are readable only by warps w with
// w % 4 == q, so a unit's 64 output rows would reach only half of the SM's
// schedulers; units therefore alternate between lane halves: the odd ones
// read their A operand 64 rows (8 KB) earlier in shared memory, which puts
// their rows in lanes 64-127 of the second accumulator, and two epilogue
// groups run side by side:
//   warps w % 4 in {0, 1}   epilogue of the even units (lanes 0-63)
//   warps w % 4 in {2, 3}   epilogue of the odd units (lanes 64-127)
//     each: token row 32 (w % 2) + lane, value columns 32 (w / 4) .. + 31;
//     scale, gated RMSNorm, bf16 output tile, tensor-map store
//   warp 16   lane 0 loads a unit's [Qc | Fc | V | S] run into its stage once
//             the products of the unit two before are done with it; lane 1
//             loads its z tile once the epilogue two units before has read
//             that stage's tile; lane 2 issues the 12 MMAs into the unit's
//             accumulator
// The run (72 KB) is released by the products and the z tile (16 KB) by the
// epilogue, so the next-but-one unit's run is in flight during an epilogue.
#include "chunks.cuh"
#include "common.cuh"
#include "kernels.h"
#include "tc05.cuh"

namespace gdn {
namespace {

constexpr int kEpiWarps = 16;
constexpr int kRoleWarp = kEpiWarps;            // lanes 0, 1, 2: loader, z loader, issuer
constexpr int kThreads = (kEpiWarps + 1) * 32;
// Stage: the record's [Qc | Fc | V | S] run (72 KB) as copied, then the unit's
// 64 x 128 bf16 tile of z (tensor-map copy, dk halves of 8 KB, 128-byte
// swizzle), which the epilogue overwrites with the outputs.
constexpr uint32_t kOffQc0 = 0, kOffQc1 = 8192, kOffFc = 16384, kOffV = 24576, kOffS = 40960;
constexpr uint32_t kRunBytes = 73728;
constexpr uint32_t kOffY = kRunBytes;
constexpr uint32_t kStageBytes = kRunBytes + 16384;
constexpr int kStages = 2;
// Two output tiles of 64 x 128 bf16 (dk halves of 8 KB, 128-byte swizzle),
// used in turn: a unit's stage is released as soon as its z tile and
// accumulator are read, and its output tile only has to be read by the
// tensor-map store before the unit after next writes it again.
constexpr uint32_t kOffOut = kStages * kStageBytes;
constexpr uint32_t kOffSmall = kOffOut + 2 * 16384;
constexpr uint32_t kTmemCols = 256;          // two 128-column accumulators
constexpr uint32_t kBarEpi = 1, kCntEpi = 256;   // barrier 1 + g: the eight warps of epilogue group g
constexpr float kScale = 0.088388347648318440550f;  // 1/sqrt(128)

struct Small {
    float red[2][4][64];       // per epilogue group: row sums of squares of each 32-column quarter
    uint64_t full[kStages];    // record run landed
    uint64_t zfull[kStages];   // z tile landed
    uint64_t mfull[kStages];   // accumulator written (the record run is free again)
    uint64_t efree[kStages];   // epilogue done: accumulator and z tile read
    uint32_t tmem_base;
    int fail;
};
constexpr uint32_t kSmemBytes = kOffSmall + ((sizeof(Small) + 127) / 128) * 128 + 1024;

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

    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Small *s = reinterpret_cast<Small *>(sm + kOffSmall);
    const uint32_t sbase = smem_u32(sm);

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&s->full[i], 1);
            mbar_init(&s->zfull[i], 1);
            mbar_init(&s->mfull[i], 1);
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
    __syncthreads();
    tc_fence_after();
    // launched early behind the scan kernel: its S copies are read below
    grid_dep_wait();
    const uint32_t tbase = s->tmem_base;
    // Every role walks the same units (u = chunk * Hv + head, strided by the
    // grid) and counts only the live ones, so stage k % 2 and barrier phases
    // agree across roles.

    if (warp == kRoleWarp) {
        if (lane == 0) {
            // -------------------------------------------------------- loader
            int k = 0, issued[kStages] = {0, 0};
            for (int u = blockIdx.x; u < units; u += gridDim.x) {
                const int gc = u / hv, h = u - gc * hv;
                int tok0 = 0, L = 0;
                if (!locate_chunk(p, gc, tok0, L))
                    continue;
                const int st = k & 1;
                // the unit two before used this stage's run: its products must be done
                if (k >= kStages && !wait_bar(s, &s->mfull[st], ((uint32_t)(k >> 1) & 1) ^ 1, p.status))
                    break;
                unsigned char *stage = sm + st * kStageBytes;
                const unsigned char *rec = p.workspace + ((size_t)gc * hv + h) * kPerVHead;
                mbar_arrive_expect_tx(&s->full[st], kRunBytes);
#pragma unroll
                for (int j = 0; j < 3; ++j)
                    bulk_g2s(stage + j * 24576, rec + kWsQc0 + j * 24576, 24576, &s->full[st]);
                ++issued[st];
                ++k;
            }
            // no copy may still be landing in shared memory when the CTA exits
            if (*reinterpret_cast<volatile int *>(&s->fail)) {
                for (int i = 0; i < kStages; ++i)
                    if (issued[i] > 0)
                        mbar_wait(&s->full[i], (uint32_t)(issued[i] - 1) & 1);
            }
        } else if (lane == 1 && kNorm) {
            // ------------------------------------------------------ z loader
            int k = 0, issued[kStages] = {0, 0};
            for (int u = blockIdx.x; u < units; u += gridDim.x) {
                const int gc = u / hv, h = u - gc * hv;
                int tok0 = 0, L = 0;
                if (!locate_chunk(p, gc, tok0, L))
                    continue;
                const int st = k & 1;
                // the unit two before read this stage's z tile in its epilogue
                if (k >= kStages && !wait_bar(s, &s->efree[st], ((uint32_t)(k >> 1) & 1) ^ 1, p.status))
                    break;
                unsigned char *stage = sm + st * kStageBytes;
                mbar_arrive_expect_tx(&s->zfull[st], 16384u);
                tma_load_3d(stage + kOffY, &tm_z, 0, h, tok0, &s->zfull[st]);
                tma_load_3d(stage + kOffY + 8192, &tm_z, 64, h, tok0, &s->zfull[st]);
                ++issued[st];
                ++k;
            }
            if (*reinterpret_cast<volatile int *>(&s->fail)) {
                for (int i = 0; i < kStages; ++i)
                    if (issued[i] > 0)
                        mbar_wait(&s->zfull[i], (uint32_t)(issued[i] - 1) & 1);
            }
        } else if (lane == 2) {
            // -------------------------------------------------------- issuer
            constexpr uint32_t idesc = make_idesc_f16(128, 128, false, true);
            int k = 0;
            for (int u = blockIdx.x; u < units; u += gridDim.x) {
                int tok0 = 0, L = 0;
                if (!locate_chunk(p, u / hv, tok0, L))
                    continue;
                const int st = k & 1;
                // odd units: A starts 64 rows (8 KB) early, so the unit's rows
                // are rows 64-127 (the rows before are whatever precedes them
                // in shared memory, and their accumulator lanes are not read)
                const uint32_t stg = sbase + st * kStageBytes - (st ? 8192u : 0u), d = tbase + st * 128;
                const uint32_t stb = sbase + st * kStageBytes;
                bool ok = wait_bar(s, &s->full[st], (uint32_t)(k >> 1) & 1, p.status);
                if (ok && k >= kStages)   // accumulator st read by the epilogue two units ago
                    ok = wait_bar(s, &s->efree[st], ((uint32_t)(k >> 1) & 1) ^ 1, p.status);
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
                mma_commit(&s->mfull[st]);
                ++k;
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int qd = warp & 3, g = qd >> 1, cq = warp >> 2;   // lane quadrant, group, column quarter
        const int row = 32 * (qd & 1) + lane;                    // token row of the unit
        const bool lead = lane == 0 && warp == 2 * g;            // the group's store thread
        const uint32_t bar = kBarEpi + g;
        int k = 0;
        for (int u = blockIdx.x; u < units; u += gridDim.x) {
            const int gc = u / hv, h = u - gc * hv;
            int tok0 = 0, L = 0;
            if (!locate_chunk(p, gc, tok0, L))
                continue;
            const int st = k & 1;
            ++k;
            if (st != g)
                continue;
            // this thread's 32 columns: 16-byte chunks 4 (cq & 1) .. of dk half cq / 2
            unsigned char *yt = sm + st * kStageBytes + kOffY + (cq >> 1) * 8192;
            unsigned char *ot = sm + kOffOut + g * 16384 + (cq >> 1) * 8192;
            const int c0 = (cq & 1) * 4;
            const uint32_t ph = (uint32_t)((k - 1) >> 1) & 1;
            // the group's output tile was last stored two units ago: that
            // store must have read it before the tile is written again
            if (lead)
                bulk_wait_read<0>();
            if (kNorm)
                wait_bar(s, &s->zfull[st], ph, p.status);   // z tile visible
            wait_bar(s, &s->mfull[st], ph, p.status);
            __syncwarp();   // converged (after the lead's wait) for the .aligned TMEM load
            tc_fence_after();
            float o[32];
            tmem_ld32(tbase + st * 128 + ((uint32_t)(32 * qd) << 16) + cq * 32, o);
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] *= kScale;
            if (kNorm) {
                float ss = 0.f;
#pragma unroll
                for (int j = 0; j < 32; ++j) ss = fmaf(o[j], o[j], ss);
                s->red[g][cq][row] = ss;
                named_sync(bar, kCntEpi);
                const float rn = rsqrtf((s->red[g][0][row] + s->red[g][1][row] + s->red[g][2][row]
                                         + s->red[g][3][row]) * (1.f / kD) + p.eps);
                const __nv_bfloat16 *wg = reinterpret_cast<const __nv_bfloat16 *>(p.norm_w) + cq * 32;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float zf[8], wf[8];
                    unpack8(*reinterpret_cast<const uint4 *>(yt + sw128_chunk_offset(row, c0 + j)), zf);
                    unpack8(reinterpret_cast<const uint4 *>(wg)[j], wf);
#pragma unroll
                    for (int e = 0; e < 8; ++e)   // silu(z) = z / (1 + e^-z)
                        o[8 * j + e] = o[8 * j + e] * rn * wf[e] * __fdividef(zf[e], 1.f + __expf(-zf[e]));
                }
            } else {
                named_sync(bar, kCntEpi);   // the lead's wait for the output tile
            }
            if (L == kC) {
                // whole chunk: bf16 outputs into the tile, one tensor-map store per dk half
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float v[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) v[e] = o[8 * j + e];
                    *reinterpret_cast<uint4 *>(ot + sw128_chunk_offset(row, c0 + j)) = pack8(v);
                }
            } else if (row < L) {
                // a sequence's ragged last chunk: the rows past it belong to the
                // next sequence, so each valid row is stored on its own
                uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(p.out)
                                                       + ((size_t)(tok0 + row) * hv + h) * kD + cq * 32);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float v[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) v[e] = o[8 * j + e];
                    dst[j] = pack8(v);
                }
            }
            // one proxy fence for both directions: the output tile's generic
            // writes before the tensor-map store reads it, and the generic
            // reads of the z tile before the z loader's TMA refills it
            fence_async_smem();
            tc_fence_before();
            named_sync(bar, kCntEpi);   // accumulator and z read, tile complete, red consumed
            if (lead) {
                mbar_arrive(&s->efree[st]);   // the stage's z tile and the accumulator are free
                if (L == kC) {
                    unsigned char *tile = sm + kOffOut + g * 16384;
                    tma_store_3d(&tm_o, 0, h, tok0, tile);
                    tma_store_3d(&tm_o, 64, h, tok0, tile + 8192);
                    bulk_commit();
                }
            }
        }
        if (lead)
            bulk_wait_all();   // every output tile copy complete before exit
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
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(out_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(out_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e != cudaSuccess)
            return e;
        configured = true;
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
    static int sm_count[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return cudaErrorInvalidDevice;
    if (!sm_count[dev]) {
        cudaError_t e = cudaDeviceGetAttribute(&sm_count[dev], cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess)
            return e;
    }
    const int units = p.max_chunks * p.hv;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(units < sm_count[dev] ? units : sm_count[dev]);
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
