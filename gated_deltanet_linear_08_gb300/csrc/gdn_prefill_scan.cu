// gdn_prefill_scan.cu -- serial half of the chunked GDN prefill: the fp32
// inter-chunk state scan, the chunk outputs and the optional gated RMSNorm
// epilogue (JevAny page "Add opt-in fused Qwen3.5 inference kernels",
// Summary: chunked kernel followed by a fused gated RMSNorm; pegainfer page
// "feat(qwen35): add SM120 FlashInfer GDN prefill candidate", Correctness:
// chunked vs unchunked prefill, initial/final states).
//
// One CTA per (sequence, value head, 32-column slice of Dv).  The recurrence
// is independent per value column, so the four slices of a head run in
// parallel; with the epilogue on, the four CTAs of a head form a cluster and
// exchange per-row sums of squares through distributed shared memory.
//
// The prep kernel turns each chunk into an affine map of the state (tcgen05,
// M = 128, fp16 operands; S is the fp32 slice, 128 x 32):
//   S'  = e^{G_last} S + [Mc | Ec] [S; V]     one MMA chain, the only serial step
//   o   = scale [Qc | Fc] [S; V]              off the chain
// Ec V does not depend on S and is issued ahead, so the chain per chunk is
// S (fp16 operand) -> 8 MMAs -> TMEM -> S' in registers.  Qc and Fc are
// staged so that a 128-row operand starting 8 KB before them has them as
// rows 64-127: the outputs land in TMEM lanes 64-127.
//
// Roles (16 warps):
//   warps 0-7   state: warp w holds TMEM lane quadrant w % 4 = state rows
//               32 (w % 4) .. +31 and value columns 16 (w / 4) .. +15
//   warp 8      issues every MMA
//   warp 9      issues every bulk copy (two stages of 77 KB)
//   warps 10, 11, 14, 15
//               outputs: lane quadrants 2-3 = chunk rows 0-63, value
//               columns 16 ((w - 10) / 4) .. +15; scale, gated RMSNorm and
//               the stores, never on the state chain
//   warps 12, 13 idle
// With the epilogue on, each CTA sums its row partials over its 32 columns
// and pushes them into every cluster CTA's receive buffer with asynchronous
// remote stores that complete bytes on the receiver's mbarrier: no
// cluster-scope fence, no cluster-wide barrier per chunk.
#include "common.cuh"
#include "kernels.h"
#include "tc05.cuh"

namespace gdn {

cudaError_t launch_prefill_prep(const PrefillArgs &p, cudaStream_t stream);

namespace {

constexpr int kThreads = 16 * 32;
constexpr int kStateWarps = 8;
constexpr int kIssuerWarp = 8;
constexpr int kLoaderWarp = 9;
__device__ __forceinline__ bool is_output_warp(int w) { return w == 10 || w == 11 || w == 14 || w == 15; }
// Named barriers (id, participating threads): producers arrive, consumers sync.
constexpr uint32_t kBarS = 1, kCntS = kStateWarps * 32 + 32;   // S operand written
constexpr uint32_t kBarRed = 2, kCntRed = 4 * 32;               // output warps' row partials
constexpr int kNv = 32;                 // value columns per CTA
constexpr int kTiles = kD / kNv;        // 4 CTAs per (sequence, head)
constexpr int kCols = 16;               // value columns per thread

// Stage: the chunk's operand record (Mc, Qc, Ec, Fc as laid out in the
// workspace) and this CTA's V slice.
constexpr uint32_t kStV = (uint32_t)kOpsBytes;
constexpr uint32_t kStageBytes = (uint32_t)kOpsBytes + 5120;
constexpr int kStages = 2;
constexpr uint32_t kLoadBytes = (uint32_t)kOpsBytes + 4096;
constexpr uint32_t kOpsPiece = (uint32_t)kOpsBytes / 3;   // copied in three pieces

constexpr uint32_t kOffS = kStages * kStageBytes;   // two S operands [dk][32] fp16, MN-major, 8 KB each
constexpr uint32_t kOffSmall = kOffS + 16384;

// TMEM columns: chain accumulators at 0 / 32, output accumulators at 64 / 96.
constexpr uint32_t kTmemCols = 128;
constexpr uint32_t kColS = 0, kColO = 64;

constexpr float kScale = 0.088388347648318440550f;  // 1/sqrt(128)

struct Small {
    float red_local[2][2][64];  // output-row partial sums of squares [parity][column group][row]
    float red_in[2][4][64];     // this CTA's row sums as received from [parity][cluster rank][row]
    float w[kNv];               // gated-norm weight slice
    uint64_t full[kStages];     // stage landed (one arrival + bytes)
    uint64_t sfree[kStages];    // every MMA reading the stage has completed
    uint64_t ofree[2];          // output accumulator read by the four output warps
    uint64_t bar_chain;
    uint64_t bar_out[2];        // one per output accumulator, so it never runs two phases ahead
    uint64_t red_full[2];       // all cluster CTAs' row sums received (1 arrival + 1 KB)
    uint32_t tmem_base;
    int fail;
};
constexpr uint32_t kSmemBytes = kOffSmall + ((sizeof(Small) + 127) / 128) * 128 + 1024;

__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

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

__device__ __forceinline__ bool wait_bar_cluster(Small *s, uint64_t *bar, uint32_t parity, uint32_t *status)
{
    if (failed(s))
        return false;
    for (uint32_t i = 0; i < kWaitPolls; ++i)
        if (mbar_try_wait_cluster(bar, parity))
            return true;
    s->fail = 1;
    set_status(status, kStatusWaitTimeout);
    return false;
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
__device__ __forceinline__ uint64_t desc_v(uint32_t st) { return make_desc(st + kStV, 512, 512, kSw64); }

// D += X V (X = Ec, or Fc read as rows 64-127 of an operand starting 8 KB
// earlier): four K steps over the chunk's 64 tokens.
__device__ __forceinline__ void issue_xv(uint32_t d, uint32_t a_addr, uint32_t st, uint32_t idesc, bool acc)
{
    const uint64_t a = desc_k128(a_addr), b = desc_v(st);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
        mma_f16(d, a + (uint64_t)(kk * 2), b + (uint64_t)(kk * 64), idesc, (acc || kk != 0) ? 1u : 0u);
}
// D += X S over the two 64-wide K halves of the state (X = Mc, or Qc as rows
// 64-127 of operands starting 8 KB before each of its halves).
__device__ __forceinline__ void issue_xs(uint32_t d, uint32_t a_lo, uint32_t a_hi, uint64_t ds, uint32_t idesc)
{
    const uint64_t a0 = desc_k128(a_lo), a1 = desc_k128(a_hi);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
        mma_f16(d, (kk < 4 ? a0 : a1) + (uint64_t)((kk & 3) * 2), ds + (uint64_t)(kk * 64), idesc, 1u);
}


template <bool kNorm>
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
        mbar_init(&s->ofree[0], 4);
        mbar_init(&s->ofree[1], 4);
        mbar_init(&s->bar_chain, 1);
        mbar_init(&s->bar_out[0], 1);
        mbar_init(&s->bar_out[1], 1);
        mbar_init(&s->red_full[0], 1);
        mbar_init(&s->red_full[1], 1);
        mbar_fence_init();
        s->fail = 0;
    }
    if (kNorm && tid < kNv)
        s->w[tid] = bf2f(reinterpret_cast<const __nv_bfloat16 *>(p.norm_w)[r * kNv + tid]);
    if (warp == 0) {
        tmem_alloc(&s->tmem_base, kTmemCols);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    if (kNorm) {   // every CTA of the cluster is running before any DSMEM access
        cluster_arrive();
        cluster_wait();
    }
    const uint32_t tbase = s->tmem_base;
    const uint32_t idesc = make_idesc_f16(128, kNv, false, true);

    if (warp == kIssuerWarp) {
        // ------------------------------------------------------------ issuer
        bool pre = false;   // Ec V of the current chunk already issued
        for (int c = 0; c < nck; ++c) {
            const int b = c & 1;   // stage = S operand = accumulator buffer
            const uint32_t st = sbase + b * kStageBytes;
            const uint32_t dS = tbase + kColS + b * kNv, dO = tbase + kColO + b * kNv;
            const uint64_t ds = make_desc(sbase + kOffS + b * 8192, 512, 512, kSw64);
            if (lane == 0 && !pre && wait_bar(s, &s->full[b], (uint32_t)(c >> 1) & 1, p.status)) {
                tc_fence_after();
                issue_xv(dS, st + (uint32_t)kWsEc, st, idesc, false);
            }
            __syncwarp();
            named_sync(kBarS, kCntS);            // S(c) operand written
            if (lane == 0) {
                if (!failed(s)) {
                    tc_fence_after();
                    issue_xs(dS, st + (uint32_t)kWsMc0, st + (uint32_t)kWsMc1, ds, idesc);
                }
                mma_commit(&s->bar_chain);
                // outputs into an accumulator the output warps have finished reading
                if (c < 2 || wait_bar(s, &s->ofree[b], ((uint32_t)(c >> 1) & 1) ^ 1, p.status)) {
                    if (!failed(s)) {
                        tc_fence_after();
                        issue_xv(dO, st + (uint32_t)kWsFc - 8192, st, idesc, false);
                        issue_xs(dO, st + (uint32_t)kWsQc0 - 8192, st + (uint32_t)kWsQc1 - 8192, ds, idesc);
                    }
                }
                mma_commit(&s->bar_out[b]);
                mma_commit(&s->sfree[b]);
                pre = false;
                if (c + 1 < nck && !failed(s) && mbar_test(&s->full[b ^ 1], (uint32_t)((c + 1) >> 1) & 1)) {
                    tc_fence_after();
                    issue_xv(tbase + kColS + (b ^ 1) * kNv, sbase + (b ^ 1) * kStageBytes + (uint32_t)kWsEc,
                             sbase + (b ^ 1) * kStageBytes, idesc, false);
                    pre = true;
                }
            }
            __syncwarp();
        }
    } else if (warp == kLoaderWarp) {
        // ------------------------------------------------------------ loader
        int issued[kStages] = {0, 0};
        if (lane == 0) {
            for (int c = 0; c < nck; ++c) {
                const int b = c & 1;
                // chunk c goes into the stage chunk c-2 used, once every MMA
                // that read it has completed
                if (c >= 2 && !wait_bar(s, &s->sfree[b], ((uint32_t)(c >> 1) & 1) ^ 1, p.status))
                    break;
                unsigned char *stage = sm + b * kStageBytes;
                const unsigned char *rec = record(c);
                mbar_arrive_expect_tx(&s->full[b], kLoadBytes);
#pragma unroll
                for (int k = 0; k < 3; ++k)
                    bulk_g2s(stage + k * kOpsPiece, rec + k * kOpsPiece, kOpsPiece, &s->full[b]);
                bulk_g2s(stage + kStV, rec + kWsV + r * 4096, 4096, &s->full[b]);
                ++issued[b];
            }
            // no copy may still be landing in shared memory when the CTA exits
            if (failed(s)) {
                for (int qq = 0; qq < kStages; ++qq)
                    if (issued[qq] > 0)
                        mbar_wait(&s->full[qq], (uint32_t)(issued[qq] - 1) & 1);
            }
        }
        __syncwarp();
    } else if (warp < kStateWarps) {
        // ------------------------------------------------------------ state
        const int q = warp & 3, cg = warp >> 2;
        const int row = 32 * q + lane;     // TMEM lane = state row (dk)
        const uint32_t tlane = tbase + ((uint32_t)(32 * q) << 16) + kColS + cg * kCols;
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
        float gl = (nck > 0) ? *reinterpret_cast<const float *>(record(0) + kWsScal) : 0.f;
        for (int c = 0; c < nck; ++c) {
            const float gnext = (c + 1 < nck) ? *reinterpret_cast<const float *>(record(c + 1) + kWsScal) : 0.f;
            wait_bar(s, &s->bar_chain, (uint32_t)c & 1, p.status);
            tc_fence_after();
            float dv[kCols];
            tmem_ld16(tlane + (c & 1) * kNv, dv);
#pragma unroll
            for (int j = 0; j < kCols; ++j) S[j] = fmaf(gl, S[j], dv[j]);
            if (c + 1 < nck)
                put_state((c + 1) & 1);
            gl = gnext;
        }
        if (over)
            set_status(p.status, kStatusRange);
#pragma unroll
        for (int j = 0; j < kCols / 4; ++j)
            reinterpret_cast<float4 *>(p.final_state + sidx)[j] = make_float4(S[4 * j], S[4 * j + 1], S[4 * j + 2], S[4 * j + 3]);
    } else if (is_output_warp(warp)) {
        // ------------------------------------------------------------ outputs
        const int q = warp & 3, cg = (warp - 10) >> 2;
        const int orow = 32 * (q - 2) + lane;   // chunk row (TMEM lane 64 + orow)
        const uint32_t tlane = tbase + ((uint32_t)(32 * q) << 16) + kColO + cg * kCols;
        const size_t col0 = (size_t)r * kNv + cg * kCols;
        const __nv_bfloat16 *zg = reinterpret_cast<const __nv_bfloat16 *>(p.z);
        __nv_bfloat16 *outg = reinterpret_cast<__nv_bfloat16 *>(p.out);
        const uint32_t my_rank = kNorm ? cluster_ctarank() : 0;
        for (int c = 0; c < nck; ++c) {
            const int pp = c & 1;
            const int Lc = min(kC, len - c * kC);
            const size_t oidx = ((size_t)(tok0 + c * kC + orow) * hv + h) * kD + col0;
            float zc[kCols];
            if (kNorm && orow < Lc) {   // z of this chunk, loaded while the MMAs run
                unpack8(reinterpret_cast<const uint4 *>(zg + oidx)[0], *reinterpret_cast<float(*)[8]>(zc));
                unpack8(reinterpret_cast<const uint4 *>(zg + oidx)[1], *reinterpret_cast<float(*)[8]>(zc + 8));
            }
            wait_bar(s, &s->bar_out[pp], (uint32_t)(c >> 1) & 1, p.status);
            tc_fence_after();
            float o[kCols];
            tmem_ld16(tlane + pp * kNv, o);
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&s->ofree[pp]);
            float ss = 0.f;
#pragma unroll
            for (int j = 0; j < kCols; ++j) {
                o[j] *= kScale;
                ss = fmaf(o[j], o[j], ss);
            }
            if (kNorm) {
                // row sums over this CTA's 32 columns, pushed to all four
                // CTAs' receive buffers (slot = this CTA's rank)
                s->red_local[pp][cg][orow] = ss;
                named_sync(kBarRed, kCntRed);
                if (cg == 0) {
                    if (orow == 0)
                        mbar_arrive_expect_tx(&s->red_full[pp], kTiles * 64 * 4);
                    const float t = s->red_local[pp][0][orow] + s->red_local[pp][1][orow];
#pragma unroll
                    for (uint32_t rk = 0; rk < kTiles; ++rk)
                        st_async_remote(&s->red_in[pp][my_rank][orow], t, &s->red_full[pp], rk);
                }
                const bool ok = wait_bar_cluster(s, &s->red_full[pp], (uint32_t)(c >> 1) & 1, p.status);
                if (ok && orow < Lc) {
                    float tot = 0.f;
#pragma unroll
                    for (int rk = 0; rk < kTiles; ++rk)
                        tot += s->red_in[pp][rk][orow];
                    const float rn = rsqrtf(tot * (1.f / kD) + p.eps);
#pragma unroll
                    for (int j = 0; j < kCols; ++j)
                        o[j] = o[j] * rn * s->w[cg * kCols + j] * (zc[j] * sigmoid_f(zc[j]));
                }
            }
            if (orow < Lc) {
                float o8[8];
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) o8[j] = o[8 * hh + j];
                    reinterpret_cast<uint4 *>(outg + oidx)[hh] = pack8(o8);
                }
            }
        }
    }

    if (kNorm) {   // peers may still be reading this CTA's partial sums
        cluster_arrive();
        cluster_wait();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tbase, kTmemCols);
    }
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs &p, cudaStream_t stream)
{
    if (p.num_seqs == 0)
        return cudaSuccess;
    if (p.total_tokens > 0) {
        cudaError_t e = launch_prefill_prep(p, stream);
        if (e != cudaSuccess)
            return e;
    }
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(scan_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(scan_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e != cudaSuccess)
            return e;
        configured = true;
    }
    dim3 grid(kTiles, p.hv, p.num_seqs);
    if (!p.z) {
        scan_kernel<false><<<grid, kThreads, kSmemBytes, stream>>>(p);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kTiles;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, scan_kernel<true>, p);
}

}  // namespace gdn
