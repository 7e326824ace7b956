// gdn_prefill_out.cu -- chunk outputs of the chunked GDN prefill and the
// optional gated RMSNorm epilogue (JevAny page "Add opt-in fused Qwen3.5
// inference kernels", Summary: chunked kernel followed by a fused gated
// RMSNorm o * rsqrt(mean(o^2) + eps) * w * silu(z)).
//
// One CTA per (64-token chunk, value head), all chunks at once: with S the
// fp16 state entering the chunk (written by the scan kernel) and the chunk's
// maps from the prep kernel,
//   o = scale [Qc | Fc] [S; V]          tcgen05, M = 128, N = 128, K = 192
// The record stores Qc's two K halves and Fc back to back, so a 128-row
// operand starting at any of them has it as rows 0-63 (rows 64-127 are the
// next image and are ignored): the outputs land in TMEM lanes 0-63, one token
// row per lane, and the norm over Dv needs only the two threads that share a
// row.
#include "common.cuh"
#include "kernels.h"
#include "tc05.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 256;
// Shared memory: the record's [Qc | Fc | V | S] run (72 KB) as copied.
constexpr uint32_t kOffQc0 = 0, kOffQc1 = 8192, kOffFc = 16384, kOffV = 24576, kOffS = 40960;
constexpr uint32_t kRunBytes = 73728;
constexpr uint32_t kOffSmall = kRunBytes;
constexpr uint32_t kTmemCols = 128;
constexpr float kScale = 0.088388347648318440550f;  // 1/sqrt(128)

struct Small {
    float red[2][64];   // row sums of squares of each 64-column half
    uint64_t mbar_ld, mbar_mma;
    uint32_t tmem_base;
    int fail;
};
constexpr uint32_t kSmemBytes = kOffSmall + ((sizeof(Small) + 127) / 128) * 128 + 1024;

__device__ bool locate_chunk(const PrefillArgs &p, int gc, int &tok0, int &L)
{
    int c = 0;
    for (int n = 0; n < p.num_seqs; ++n) {
        const int s = p.cu_seqlens[n], e = p.cu_seqlens[n + 1];
        if (s < 0 || e < s || e > p.total_tokens)
            continue;
        const int nc = (e - s + kC - 1) / kC;
        if (gc < c + nc) {
            tok0 = s + (gc - c) * kC;
            L = min(kC, e - tok0);
            return true;
        }
        c += nc;
    }
    return false;
}

__device__ __forceinline__ void wait_bar(Small *s, uint64_t *bar, uint32_t parity, uint32_t *status)
{
    if (*reinterpret_cast<volatile int *>(&s->fail))
        return;
    if (!mbar_wait(bar, parity)) {
        s->fail = 1;
        set_status(status, kStatusWaitTimeout);
    }
}

template <bool kNorm>
__global__ void __launch_bounds__(kThreads, 2)
out_kernel(PrefillArgs p)
{
    const int gc = blockIdx.x, h = blockIdx.y, hv = p.hv;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int tok0 = 0, L = 0;
    if (!locate_chunk(p, gc, tok0, L))
        return;

    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Small *s = reinterpret_cast<Small *>(sm + kOffSmall);
    const uint32_t sbase = smem_u32(sm);
    const unsigned char *rec = p.workspace + ((size_t)gc * hv + h) * kPerVHead;

    if (tid == 0) {
        mbar_init(&s->mbar_ld, 1);
        mbar_init(&s->mbar_mma, 1);
        mbar_fence_init();
        s->fail = 0;
        mbar_arrive_expect_tx(&s->mbar_ld, kRunBytes);
#pragma unroll
        for (int k = 0; k < 3; ++k)
            bulk_g2s(sm + k * 24576, rec + kWsQc0 + k * 24576, 24576, &s->mbar_ld);
    }
    if (warp == 0) {
        tmem_alloc(&s->tmem_base, kTmemCols);
        tmem_relinquish();
        tc_fence_before();
    }
    // warps 0-1 and 4-5: token row 32 (w % 4) + lane, value columns 64 (w / 4) ..
    const int q = warp & 3, ch = warp >> 2;
    const int row = 32 * q + lane;
    const bool outw = q < 2;
    const size_t oidx = ((size_t)(tok0 + row) * hv + h) * kD + ch * 64;
    uint4 zr[8];
    if (kNorm && outw && row < L) {   // z of this row, loaded under the copy and the MMA
        const uint4 *zs = reinterpret_cast<const uint4 *>(reinterpret_cast<const __nv_bfloat16 *>(p.z) + oidx);
#pragma unroll
        for (int j = 0; j < 8; ++j) zr[j] = zs[j];
    }
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        if (lane == 0) {
            wait_bar(s, &s->mbar_ld, 0, p.status);
            if (!*reinterpret_cast<volatile int *>(&s->fail)) {
                constexpr uint32_t idesc = make_idesc_f16(128, 128, false, true);
                const uint64_t bv = make_desc(sbase + kOffV, 4096, 512, kSw64);
                const uint64_t bs = make_desc(sbase + kOffS, 8192, 512, kSw64);
                const uint64_t af = make_desc(sbase + kOffFc, 16, 1024, kSw128);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)   // Fc V over the chunk's 64 tokens
                    mma_f16(s->tmem_base, af + (uint64_t)(kk * 2), bv + (uint64_t)(kk * 64), idesc, kk != 0);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {  // Qc S over the 128 state rows
                    const uint64_t aq = make_desc(sbase + (kk < 4 ? kOffQc0 : kOffQc1), 16, 1024, kSw128);
                    mma_f16(s->tmem_base, aq + (uint64_t)((kk & 3) * 2), bs + (uint64_t)(kk * 64), idesc, 1u);
                }
            }
            mma_commit(&s->mbar_mma);
        }
        __syncwarp();
    }
    if (outw) {
        wait_bar(s, &s->mbar_mma, 0, p.status);
        tc_fence_after();
        float o[64];
        {
            float d[32];
            tmem_ld32(s->tmem_base + ((uint32_t)(32 * q) << 16) + ch * 64, d);
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = d[j] * kScale;
            tmem_ld32(s->tmem_base + ((uint32_t)(32 * q) << 16) + ch * 64 + 32, d);
#pragma unroll
            for (int j = 0; j < 32; ++j) o[32 + j] = d[j] * kScale;
        }
        if (kNorm) {
            float ss = 0.f;
#pragma unroll
            for (int j = 0; j < 64; ++j) ss = fmaf(o[j], o[j], ss);
            s->red[ch][row] = ss;
            named_sync(1, 128);   // the four output warps
            const float rn = rsqrtf((s->red[0][row] + s->red[1][row]) * (1.f / kD) + p.eps);
            const __nv_bfloat16 *wg = reinterpret_cast<const __nv_bfloat16 *>(p.norm_w) + ch * 64;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                float zf[8], wf[8];
                unpack8(zr[j], zf);
                unpack8(reinterpret_cast<const uint4 *>(wg)[j], wf);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    o[8 * j + e] = o[8 * j + e] * rn * wf[e] * (zf[e] * sigmoid_f(zf[e]));
            }
        }
        if (row < L) {
            uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(p.out) + oidx);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                float v[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) v[e] = o[8 * j + e];
                dst[j] = pack8(v);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(s->tmem_base, kTmemCols);
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
    dim3 grid(p.max_chunks, p.hv);
    if (p.z)
        out_kernel<true><<<grid, kThreads, kSmemBytes, stream>>>(p);
    else
        out_kernel<false><<<grid, kThreads, kSmemBytes, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace gdn
