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
// Per chunk, with S the fp32 state slice (128 x 32) held in registers, and the
// chunk operands built by the prep kernel (tcgen05, M = 128, fp16 operands):
//   X  = MT V + WQ S                one TMEM accumulator
//   U  = X[0:64]                    (= T diag(beta) V - W S)
//   o  = X[64:128] / sqrt(Dk)       (= chunk outputs)
//   Z  = Kn^T (diag(e^{G_last - G}) U)
//   S  = e^{G_last} S + Z
// Only WQ S and Z lie on the serial chain S -> X -> U -> Z -> S: MT V does not
// depend on S and is issued after the previous chunk's Z when its operands
// have already landed.  Operands stream through three stages; the copies for
// chunk c+2 are issued, split over two threads, while Z(c) runs.  The tensor core accepts about one M=128 MMA per ~50
// cycles at these widths, so the chain is counted in MMA instructions: 12 per
// chunk.  The cluster exchange of row norms is deferred by one chunk and the
// output stores follow the next cluster arrival, so neither the exchange nor
// a store waits on the chain.
//
// 16 compute warps: warp w reads TMEM lane quadrant q = w % 4 and value
// columns 8 (w / 4) .. +7 of each accumulator; thread (q, lane) owns state row
// 32 q + lane.  Quadrants 0-1 form U (chunk rows 0-63), quadrants 2-3 the
// outputs.  Every operand they write is MN-major, so each thread stores its 8
// values as one 16-byte vector, then arrives on a named barrier without
// waiting.  An issuer warp syncs on those barriers and issues every MMA, and a
// loader warp issues the bulk copies, so no compute warp is held up issuing.
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

constexpr int kComputeWarps = 16;
constexpr int kIssuerWarp = kComputeWarps;        // issues every MMA
constexpr int kLoaderWarp = kComputeWarps + 1;    // issues every bulk copy
constexpr int kThreads = (kComputeWarps + 2) * 32;
// Named barriers (id, participating threads): producers arrive, consumer warps
// sync.
constexpr uint32_t kBarS = 1, kCntS = kComputeWarps * 32 + 64;   // S operand written
constexpr uint32_t kBarU = 2, kCntU = 8 * 32 + 32;               // U operand written
constexpr uint32_t kBarRed = 3, kCntRed = 8 * 32;                // output warps' row partials
constexpr int kNv = 32;                 // value columns per CTA
constexpr int kTiles = kD / kNv;        // 4 CTAs per (sequence, head)
constexpr int kCols = 8;                // value columns per thread

// Stage layout (offsets within a stage; all 1024-byte aligned).
constexpr uint32_t kStWQ = 0;           // 32 KB  WQ, K-major, K halves of 16 KB
constexpr uint32_t kStMT = 32768;       // 16 KB  MT, K-major
constexpr uint32_t kStK = 49152;        // 16 KB  Kn [token][dk], MN-major A
constexpr uint32_t kStV = 65536;        //  4 KB  V slice [token][32], MN-major B
constexpr uint32_t kStScal = 69632;     //  272 B used
constexpr uint32_t kScalCopy = 272;     //  65 floats rounded up to 16 bytes
constexpr uint32_t kStageBytes = 70656;
constexpr int kStages = 3;
// bytes of the two halves of a stage's copies (one issuing thread each)
constexpr uint32_t kLoadBytesA = (uint32_t)(kWQBytes + kMTBytes);
constexpr uint32_t kLoadBytesB = (uint32_t)kKBytes + 4096 + kScalCopy;

constexpr uint32_t kOffS = kStages * kStageBytes;   // S operand [dk][32] fp16, MN-major, 8 KB
constexpr uint32_t kOffU = kOffS + 8192;      // U operand [token][32] fp16, MN-major, 4 KB
constexpr uint32_t kOffSmall = kOffU + 4096;
constexpr uint32_t kSmemBytes = kOffSmall + 5120 + 1024;

// TMEM columns: X[2] at 0 / 32, Z at 64.
constexpr uint32_t kTmemCols = 128;
constexpr uint32_t kColX = 0, kColZ = 64;

constexpr float kScale = 0.088388347648318440550f;  // 1/sqrt(128)

struct Small {
    float red_local[2][4][64];  // row partial sums of squares [parity][column group][row]
    float red_in[2][4][64];     // this CTA's row sums as received from [parity][cluster rank][row]
    float w[kNv];               // gated-norm weight slice
    uint64_t bar_load[kStages];   // two arrivals (one per issuing thread) + bytes
    uint64_t bar_x, bar_z;
    uint64_t red_full[2];   // all cluster CTAs' row sums received (1 arrival + 1 KB)
    uint32_t tmem_base;
    int fail;
};

__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

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

__device__ __forceinline__ bool wait_bar_cluster(Small *s, uint64_t *bar, uint32_t parity, uint32_t *status)
{
    if (*reinterpret_cast<volatile int *>(&s->fail))
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

// The stage's copies are split over two issuing threads: half A (WQ, MT) and
// half B (Kn, the V slice, the row scales).
__device__ __forceinline__ void issue_loads_a(const PrefillArgs &p, unsigned char *stage, uint64_t *bar,
                                              int gc, int h)
{
    const unsigned char *wv = p.workspace + ((size_t)gc * p.hv + h) * kPerVHead;
    mbar_arrive_expect_tx(bar, kLoadBytesA);
    bulk_g2s(stage + kStWQ, wv, (uint32_t)kWQBytes, bar);
    bulk_g2s(stage + kStMT, wv + kWQBytes, (uint32_t)kMTBytes, bar);
}
__device__ __forceinline__ void issue_loads_b(const PrefillArgs &p, unsigned char *stage, uint64_t *bar,
                                              int gc, int h, int hq, int r)
{
    const unsigned char *wv = p.workspace + ((size_t)gc * p.hv + h) * kPerVHead;
    const unsigned char *wk = p.workspace + (size_t)p.max_chunks * p.hv * kPerVHead
                              + ((size_t)gc * p.hk + hq) * kKBytes;
    mbar_arrive_expect_tx(bar, kLoadBytesB);
    bulk_g2s(stage + kStK, wk, (uint32_t)kKBytes, bar);
    bulk_g2s(stage + kStV, wv + kWQBytes + kMTBytes + r * 4096, 4096, bar);
    bulk_g2s(stage + kStScal, wv + kWQBytes + kMTBytes + kVBytes, kScalCopy, bar);
}

// X(stage) += MT V: four K steps over the 64 tokens.
__device__ __forceinline__ void issue_mtv(uint32_t dx, uint32_t soff, uint32_t idesc)
{
    const uint64_t a = make_desc(soff + kStMT, 16, 1024, kSw128);
    const uint64_t b = make_desc(soff + kStV, 512, 512, kSw64);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
        mma_f16(dx, a + (uint64_t)(kk * 2), b + (uint64_t)(kk * 64), idesc, kk != 0);
}

template <bool kNorm>
__global__ void __launch_bounds__(kThreads, 1)
scan_kernel(PrefillArgs p)
{
    const int r = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
    const int hv = p.hv, hq = h / (hv / p.hk);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Small *s = reinterpret_cast<Small *>(sm + kOffSmall);
    const uint32_t sbase = smem_u32(sm);

    int tok0 = 0, len = 0;
    const int cbase = chunk_base_of(p, n, tok0, len);
    const int nck = (len + kC - 1) / kC;

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i)
            mbar_init(&s->bar_load[i], 2);
        mbar_init(&s->bar_x, 1);
        mbar_init(&s->bar_z, 1);
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
    const uint32_t idesc_x = make_idesc_f16(128, kNv, false, true);
    const uint32_t idesc_z = make_idesc_f16(128, kNv, true, true);

    if (warp == kIssuerWarp) {
        // ------------------------------------------------------------ issuer
        const uint64_t desc_s = make_desc(sbase + kOffS, 512, 512, kSw64);
        const uint64_t desc_u = make_desc(sbase + kOffU, 512, 512, kSw64);
        bool mtv_pre = false;
        for (int c = 0; c < nck; ++c) {
            const int st = c % kStages;
            const uint32_t soff = sbase + st * kStageBytes;
            named_sync(kBarS, kCntS);            // S(c) operand written
            if (lane == 0) {
                if (wait_bar(s, &s->bar_load[st], (uint32_t)(c / kStages) & 1, p.status)) {
                    tc_fence_after();
                    const uint32_t dx = tbase + kColX + (c & 1) * kNv;
                    if (!mtv_pre)
                        issue_mtv(dx, soff, idesc_x);
                    const uint64_t a = make_desc(soff + kStWQ, 16, 1024, kSw128);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_f16(dx, a + (uint64_t)((kk >> 2) * 1024 + (kk & 3) * 2),
                                desc_s + (uint64_t)(kk * 64), idesc_x, 1);
                }
                mma_commit(&s->bar_x);
            }
            __syncwarp();
            named_sync(kBarU, kCntU);            // U(c) operand written
            if (lane == 0) {
                if (!*reinterpret_cast<volatile int *>(&s->fail)) {
                    tc_fence_after();
                    const uint64_t a = make_desc(soff + kStK, 8192, 1024, kSw128);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_f16(tbase + kColZ, a + (uint64_t)(kk * 128), desc_u + (uint64_t)(kk * 64),
                                idesc_z, kk != 0);
                }
                mma_commit(&s->bar_z);
                mtv_pre = false;
                if (c + 1 < nck && !*reinterpret_cast<volatile int *>(&s->fail)) {
                    const int ns = (c + 1) % kStages;
                    if (mbar_test(&s->bar_load[ns], (uint32_t)((c + 1) / kStages) & 1)) {
                        tc_fence_after();
                        issue_mtv(tbase + kColX + ((c + 1) & 1) * kNv, sbase + ns * kStageBytes, idesc_x);
                        mtv_pre = true;
                    }
                }
            }
            __syncwarp();
        }
    } else if (warp == kLoaderWarp) {
        // ------------------------------------------------------------ loader
        int issued[kStages] = {0, 0, 0};
        auto issue_stage = [&](int cc) {
            const int st = cc % kStages;
            issue_loads_a(p, sm + st * kStageBytes, &s->bar_load[st], cbase + cc, h);
            issue_loads_b(p, sm + st * kStageBytes, &s->bar_load[st], cbase + cc, h, hq, r);
            ++issued[st];
        };
        if (lane == 0)
            for (int cc = 0; cc < 2 && cc < nck; ++cc)
                issue_stage(cc);
        for (int c = 0; c < nck; ++c) {
            named_sync(kBarS, kCntS);
            // chunk c+2 goes into the stage chunk c-1 used: Z(c-1) was read
            // and every read of that stage's row scales happened before the
            // S(c) barrier
            if (lane == 0 && c + 2 < nck)
                issue_stage(c + 2);
            __syncwarp();
        }
        // no copy may still be landing in shared memory when the CTA exits
        if (lane == 0 && *reinterpret_cast<volatile int *>(&s->fail)) {
            for (int qq = 0; qq < kStages; ++qq)
                if (issued[qq] > 0)
                    mbar_wait(&s->bar_load[qq], (issued[qq] - 1) & 1);
        }
    } else {
        // ------------------------------------------------------------ compute
        const int q = warp & 3, g = warp >> 2;
        const int row = 32 * q + lane;     // TMEM lane = state row = chunk row
        const int orow = row - 64;         // output row for quadrants 2-3
        const uint32_t tlane = tbase + ((uint32_t)(32 * q) << 16) + g * kCols;
        const size_t sidx = (((size_t)n * hv + h) * kD + row) * kD + r * kNv + g * kCols;
        const size_t col0 = (size_t)r * kNv + g * kCols;
        const __nv_bfloat16 *zg = reinterpret_cast<const __nv_bfloat16 *>(p.z);
        __nv_bfloat16 *outg = reinterpret_cast<__nv_bfloat16 *>(p.out);

        float S[kCols];
        if (p.init_state) {
            const float4 a0 = reinterpret_cast<const float4 *>(p.init_state + sidx)[0];
            const float4 a1 = reinterpret_cast<const float4 *>(p.init_state + sidx)[1];
            S[0] = a0.x; S[1] = a0.y; S[2] = a0.z; S[3] = a0.w;
            S[4] = a1.x; S[5] = a1.y; S[6] = a1.z; S[7] = a1.w;
        } else {
#pragma unroll
            for (int j = 0; j < kCols; ++j) S[j] = 0.f;
        }
        const uint32_t my_rank = kNorm ? cluster_ctarank() : 0;
        float o_prev[kCols], z_prev[kCols];   // outputs of the previous chunk awaiting its norm
#pragma unroll
        for (int j = 0; j < kCols; ++j) { o_prev[j] = 0.f; z_prev[j] = 0.f; }
        bool over = false;   // a state value left the fp16 operand range

        // gated RMSNorm and store of chunk c's output rows, once every CTA of
        // the cluster has published its partial sums for them
        auto finish = [&](int c) {
            const int Lc = min(kC, len - c * kC);
            const bool ok = wait_bar_cluster(s, &s->red_full[c & 1], (uint32_t)(c >> 1) & 1, p.status);
            if (!ok || orow >= Lc)
                return;
            float tot = 0.f;
#pragma unroll
            for (int rk = 0; rk < kTiles; ++rk)
                tot += s->red_in[c & 1][rk][orow];
            const float rn = rsqrtf(tot * (1.f / kD) + p.eps);
            float y[kCols];
#pragma unroll
            for (int j = 0; j < kCols; ++j)
                y[j] = o_prev[j] * rn * s->w[g * kCols + j] * (z_prev[j] * sigmoid_f(z_prev[j]));
            *reinterpret_cast<uint4 *>(outg + ((size_t)(tok0 + c * kC + orow) * hv + h) * kD + col0) = pack8(y);
        };

        for (int c = 0; c < nck; ++c) {
            const int pp = c & 1;
            const int st = c % kStages;
            const int Lc = min(kC, len - c * kC);
            const float *scal = reinterpret_cast<const float *>(sm + st * kStageBytes + kStScal);

            // (A) state -> fp16 operand S
            {
                float v[kCols];
#pragma unroll
                for (int j = 0; j < kCols; ++j) {
                    v[j] = S[j];
                    over |= !(fabsf(S[j]) <= kHalfMax);
                }
                *reinterpret_cast<uint4 *>(sm + kOffS + sw64_chunk_offset(row, g)) = pack8h(v);
            }
            fence_async_smem();
            tc_fence_before();
            named_arrive(kBarS, kCntS);

            // (D) the previous chunk's outputs (their norms are complete by now)
            if (kNorm && c >= 1 && q >= 2)
                finish(c - 1);

            // (C) U rows -> scaled operand; output rows -> epilogue
            float zc[kCols];
            if (kNorm && q >= 2 && orow < Lc) {   // z of this chunk, loaded under the MMA
                unpack8(*reinterpret_cast<const uint4 *>(zg + ((size_t)(tok0 + c * kC + orow) * hv + h) * kD + col0), zc);
            } else {
#pragma unroll
                for (int j = 0; j < kCols; ++j) zc[j] = 0.f;
            }
            wait_bar(s, &s->bar_x, pp, p.status);
            wait_bar(s, &s->bar_load[st], (uint32_t)(c / kStages) & 1, p.status);   // row scales visible
            tc_fence_after();
            float xv[kCols];
            tmem_ld8(tlane + kColX + pp * kNv, xv);
            if (q < 2) {
                const float sc = scal[row];
                float u[kCols];
#pragma unroll
                for (int j = 0; j < kCols; ++j) u[j] = xv[j] * sc;
                *reinterpret_cast<uint4 *>(sm + kOffU + sw64_chunk_offset(row, g)) = pack8h(u);
                fence_async_smem();
                tc_fence_before();
                named_arrive(kBarU, kCntU);
            } else {
                float ss = 0.f;
#pragma unroll
                for (int j = 0; j < kCols; ++j) {
                    o_prev[j] = xv[j] * kScale;
                    ss = fmaf(o_prev[j], o_prev[j], ss);
                    z_prev[j] = zc[j];
                }
                if (kNorm) {
                    // row sums over this CTA's 32 columns, pushed to all four
                    // CTAs' receive buffers (slot = this CTA's rank)
                    s->red_local[pp][g][orow] = ss;
                    named_sync(kBarRed, kCntRed);
                    if (g == 0) {
                        if (orow == 0)
                            mbar_arrive_expect_tx(&s->red_full[pp], kTiles * 64 * 4);
                        const float t = s->red_local[pp][0][orow] + s->red_local[pp][1][orow]
                                      + s->red_local[pp][2][orow] + s->red_local[pp][3][orow];
#pragma unroll
                        for (uint32_t rk = 0; rk < kTiles; ++rk)
                            st_async_remote(&s->red_in[pp][my_rank][orow], t, &s->red_full[pp], rk);
                    }
                } else if (orow < Lc) {
                    *reinterpret_cast<uint4 *>(outg + ((size_t)(tok0 + c * kC + orow) * hv + h) * kD + col0) = pack8(o_prev);
                }
            }

            // (F) S = e^{G_last} S + Z
            wait_bar(s, &s->bar_z, pp, p.status);
            tc_fence_after();
            float zv[kCols];
            tmem_ld8(tlane + kColZ, zv);
            const float gl = scal[64];
#pragma unroll
            for (int j = 0; j < kCols; ++j) S[j] = fmaf(gl, S[j], zv[j]);
        }
        if (kNorm && nck >= 1 && q >= 2)
            finish(nck - 1);

        if (over)
            set_status(p.status, kStatusRange);
        float4 *dst = reinterpret_cast<float4 *>(p.final_state + sidx);
        dst[0] = make_float4(S[0], S[1], S[2], S[3]);
        dst[1] = make_float4(S[4], S[5], S[6], S[7]);
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
