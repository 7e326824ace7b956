// gdn_prefill_scan.cu -- serial half of the chunked GDN prefill: the fp32
// inter-chunk state scan (JevAny page "Add opt-in fused Qwen3.5 inference
// kernels", Summary: chunked kernel; pegainfer page "feat(qwen35): add SM120
// FlashInfer GDN prefill candidate", Correctness: chunked vs unchunked
// prefill, initial/final states).
//
// One CTA per (sequence, value head, 32-column slice of Dv).  The recurrence
// is independent per value column, so the four slices of a head run in
// parallel with no communication.
//
// The prep kernel turns each chunk into an affine map of the state (tcgen05,
// M = 128, fp16 operands; S is the fp32 slice, 128 x 32):
//   S' = e^{G_last} S + [Mc | Ec] [S; V]
// Ec V does not depend on S and is issued ahead, so the serial chain per
// chunk is S (fp16 operand) -> 8 MMAs -> TMEM -> S' in registers.  Each
// chunk's fp16 S operand is also copied to the workspace, where the output
// kernel, fully parallel over chunks, turns it into the chunk's outputs.
//
// Roles (10 warps):
//   warps 0-7   state: warp w holds TMEM lane quadrant w % 4 = state rows
//               32 (w % 4) .. +31 and value columns 16 (w / 4) .. +15
//   warp 8      issues every MMA and the copies of S to the workspace
//   warp 9      issues the operand copies (three stages of 52 KB)
#include "common.cuh"
#include "kernels.h"
#include "tc05.cuh"

namespace gdn {


namespace {

constexpr int kThreads = 10 * 32;
constexpr int kStateWarps = 8;
constexpr int kIssuerWarp = 8;
constexpr int kLoaderWarp = 9;
// Named barrier (id, participating threads): state warps arrive, the issuer syncs.
constexpr uint32_t kBarS = 1, kCntS = kStateWarps * 32 + 32;   // S operand written
constexpr int kNv = 32;                 // value columns per CTA
constexpr int kTiles = kD / kNv;        // 4 CTAs per (sequence, head)
constexpr int kCols = 16;               // value columns per thread

// Stage: the chunk's Mc and Ec (one contiguous run of the record) and this
// CTA's V slice.
constexpr uint32_t kStEc = (uint32_t)kWsEc;
constexpr uint32_t kStV = 49152;
constexpr uint32_t kStageBytes = 53248;
constexpr int kStages = 3;
constexpr uint32_t kLoadBytes = 49152 + 4096;

constexpr uint32_t kOffS = kStages * kStageBytes;   // two S operands [dk][32] fp16, MN-major, 8 KB each
constexpr uint32_t kOffSmall = kOffS + 16384;

// TMEM columns: chain accumulators at 0 / 32.
constexpr uint32_t kTmemCols = 64;

struct Small {
    uint64_t full[kStages];     // stage landed (one arrival + bytes)
    uint64_t sfree[kStages];    // every MMA reading the stage has completed
    uint64_t bar_chain;
    uint32_t tmem_base;
    int fail;
};
constexpr uint32_t kSmemBytes = kOffSmall + ((sizeof(Small) + 127) / 128) * 128 + 1024;

__device__ __forceinline__ bool failed(Small *s) { return *reinterpret_cast<volatile int *>(&s->fail) != 0; }

__device__ __forceinline__ bool wait_bar(Small *s, uint64_t *bar, uint32_t parity, uint32_t *status)
{
    if (failed(s))
        return false;
    if (!mbar_wait(bar, parity)) {
        s->fail = 1;
        set_status(status, kStatusWaitTimeout);
        return false;
    }
    return true;
}

// Chunks that precede sequence n, with the same treatment of malformed
// cu_seqlens as the prep kernel (a malformed sequence owns no chunks).
__device__ int chunk_base_of(const PrefillArgs &p, int n, int &tok0, int &len)
{
    int c = 0;
    for (int m = 0; m < p.num_seqs; ++m) {
        const int s = p.cu_seqlens[m], e = p.cu_seqlens[m + 1];
        const bool ok = !(s < 0 || e < s || e > p.total_tokens);
        if (m == n) {
            tok0 = ok ? s : 0;
            len = ok ? e - s : 0;
            return c;
        }
        if (ok)
            c += (e - s + kC - 1) / kC;
    }
    tok0 = 0;
    len = 0;
    return c;
}

// Descriptors of the stage operands (shared-memory byte address `st`).
__device__ __forceinline__ uint64_t desc_k128(uint32_t addr) { return make_desc(addr, 16, 1024, kSw128); }

// D = Ec V: four K steps over the chunk's 64 tokens.
__device__ __forceinline__ void issue_ecv(uint32_t d, uint32_t st, uint32_t idesc)
{
    const uint64_t a = desc_k128(st + kStEc), b = make_desc(st + kStV, 512, 512, kSw64);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
        mma_f16(d, a + (uint64_t)(kk * 2), b + (uint64_t)(kk * 64), idesc, kk != 0 ? 1u : 0u);
}
// D += Mc S over the two 64-wide K halves of the state.
__device__ __forceinline__ void issue_mcs(uint32_t d, uint32_t st, uint64_t ds, uint32_t idesc)
{
    const uint64_t a0 = desc_k128(st + (uint32_t)kWsMc0), a1 = desc_k128(st + (uint32_t)kWsMc1);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
        mma_f16(d, (kk < 4 ? a0 : a1) + (uint64_t)((kk & 3) * 2), ds + (uint64_t)(kk * 64), idesc, 1u);
}

__global__ void __launch_bounds__(kThreads, 1)
scan_kernel(PrefillArgs p)
{
    const int r = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
    const int hv = p.hv;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Small *s = reinterpret_cast<Small *>(sm + kOffSmall);
    const uint32_t sbase = smem_u32(sm);

    int tok0 = 0, len = 0;
    const int cbase = chunk_base_of(p, n, tok0, len);
    const int nck = (len + kC - 1) / kC;
    auto record = [&](int c) { return p.workspace + ((size_t)(cbase + c) * hv + h) * kPerVHead; };

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&s->full[i], 1);
            mbar_init(&s->sfree[i], 1);
        }
        mbar_init(&s->bar_chain, 1);
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
    const uint32_t tbase = s->tmem_base;
    const uint32_t idesc = make_idesc_f16(128, kNv, false, true);

    if (warp == kIssuerWarp) {
        // ------------------------------------------------------------ issuer
        bool pre = false;   // Ec V of the current chunk already issued
        for (int c = 0; c < nck; ++c) {
            const int b = c & 1, st = c % kStages;   // S operand and accumulator buffer; stage
            const uint32_t sst = sbase + st * kStageBytes;
            const uint32_t dS = tbase + b * kNv;
            if (lane == 0 && !pre && wait_bar(s, &s->full[st], (uint32_t)(c / kStages) & 1, p.status)) {
                tc_fence_after();
                issue_ecv(dS, sst, idesc);
            }
            __syncwarp();
            named_sync(kBarS, kCntS);            // S(c) operand written
            if (lane == 0) {
                if (!failed(s)) {
                    tc_fence_after();
                    issue_mcs(dS, sst, make_desc(sbase + kOffS + b * 8192, 512, 512, kSw64), idesc);
                }
                // the S(c) operand -> workspace, for the output kernel; the copy
                // of S(c-1) must have finished reading its buffer before the
                // state warps (released by this chunk's chain) overwrite it
                bulk_s2g(record(c) + kWsS + r * 8192, sm + kOffS + b * 8192, 8192);
                bulk_wait_read<1>();
                mma_commit(&s->bar_chain);
                mma_commit(&s->sfree[st]);
                pre = false;
                const int ns = (c + 1) % kStages;
                if (c + 1 < nck && !failed(s) && mbar_test(&s->full[ns], (uint32_t)((c + 1) / kStages) & 1)) {
                    tc_fence_after();
                    issue_ecv(tbase + (b ^ 1) * kNv, sbase + ns * kStageBytes, idesc);
                    pre = true;
                }
            }
            __syncwarp();
        }
        if (lane == 0)
            bulk_wait_all();   // every S copy complete before exit
        __syncwarp();
    } else if (warp == kLoaderWarp) {
        // ------------------------------------------------------------ loader
        int issued[kStages] = {0, 0, 0};
        if (lane == 0) {
            for (int c = 0; c < nck; ++c) {
                const int st = c % kStages;
                // chunk c goes into the stage chunk c-3 used, once every MMA
                // that read it has completed
                if (c >= kStages && !wait_bar(s, &s->sfree[st], (uint32_t)(c / kStages - 1) & 1, p.status))
                    break;
                unsigned char *stage = sm + st * kStageBytes;
                const unsigned char *rec = record(c);
                mbar_arrive_expect_tx(&s->full[st], kLoadBytes);
                bulk_g2s(stage, rec, 24576, &s->full[st]);
                bulk_g2s(stage + 24576, rec + 24576, 24576, &s->full[st]);
                bulk_g2s(stage + kStV, rec + kWsV + r * 4096, 4096, &s->full[st]);
                ++issued[st];
            }
            // no copy may still be landing in shared memory when the CTA exits
            if (failed(s)) {
                for (int qq = 0; qq < kStages; ++qq)
                    if (issued[qq] > 0)
                        mbar_wait(&s->full[qq], (uint32_t)(issued[qq] - 1) & 1);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ state
        const int q = warp & 3, cg = warp >> 2;
        const int row = 32 * q + lane;     // TMEM lane = state row (dk)
        const uint32_t tlane = tbase + ((uint32_t)(32 * q) << 16) + cg * kCols;
        const size_t sidx = (((size_t)n * hv + h) * kD + row) * kD + r * kNv + cg * kCols;
        float S[kCols];
        if (p.init_state) {
#pragma unroll
            for (int j = 0; j < kCols / 4; ++j) {
                const float4 a = reinterpret_cast<const float4 *>(p.init_state + sidx)[j];
                S[4 * j] = a.x; S[4 * j + 1] = a.y; S[4 * j + 2] = a.z; S[4 * j + 3] = a.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < kCols; ++j) S[j] = 0.f;
        }
        bool over = false;   // a state value left the fp16 operand range
        auto put_state = [&](int b) {
            float v[8];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    v[j] = S[8 * hh + j];
                    over |= !(fabsf(v[j]) <= kHalfMax);
                }
                *reinterpret_cast<uint4 *>(sm + kOffS + b * 8192 + sw64_chunk_offset(row, 2 * cg + hh)) = pack8h(v);
            }
            fence_async_smem();
            tc_fence_before();
            named_arrive(kBarS, kCntS);
        };
        if (nck > 0)
            put_state(0);
        // e^{G_last} of chunks c and c+1 in registers, c+2 requested two chunks ahead
        float gl = (nck > 0) ? *reinterpret_cast<const float *>(record(0) + kWsScal) : 0.f;
        float gl1 = (nck > 1) ? *reinterpret_cast<const float *>(record(1) + kWsScal) : 0.f;
        for (int c = 0; c < nck; ++c) {
            const float gl2 = (c + 2 < nck) ? *reinterpret_cast<const float *>(record(c + 2) + kWsScal) : 0.f;
            wait_bar(s, &s->bar_chain, (uint32_t)c & 1, p.status);
            tc_fence_after();
            float dv[kCols];
            tmem_ld16(tlane + (c & 1) * kNv, dv);
#pragma unroll
            for (int j = 0; j < kCols; ++j) S[j] = fmaf(gl, S[j], dv[j]);
            if (c + 1 < nck)
                put_state((c + 1) & 1);
            gl = gl1;
            gl1 = gl2;
        }
        if (over)
            set_status(p.status, kStatusRange);
#pragma unroll
        for (int j = 0; j < kCols / 4; ++j)
            reinterpret_cast<float4 *>(p.final_state + sidx)[j] = make_float4(S[4 * j], S[4 * j + 1], S[4 * j + 2], S[4 * j + 3]);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tbase, kTmemCols);
    }
}

}  // namespace

cudaError_t launch_prefill_scan(const PrefillArgs &p, cudaStream_t stream)
{
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e != cudaSuccess)
            return e;
        configured = true;
    }
    dim3 grid(kTiles, p.hv, p.num_seqs);
    scan_kernel<<<grid, kThreads, kSmemBytes, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace gdn
