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
// Per chunk, with S the fp32 state slice (128 x 32) held in registers (thread
// t owns key row t) and the chunk operands built by the prep kernel:
//   X  = MT V + WQ S           one TMEM accumulator (tcgen05, M = 128)
//   U  = X[0:64]               (= T diag(beta) V - W S)
//   o  = X[64:128] / sqrt(Dk)  (= chunk outputs)
//   Z  = K^T (diag(e^{G_last - G} r_k) U)   U split hi/lo bf16, raw K exact
//   S  = e^{G_last} S + Z
// Operands arrive by bulk asynchronous copy (one mbarrier per stage, two
// stages); the next chunk's copy is in flight while this chunk computes.
#include "common.cuh"
#include "kernels.h"
#include "tc05.cuh"

namespace gdn {

cudaError_t launch_prefill_prep(const PrefillArgs &p, cudaStream_t stream);

namespace {

constexpr int kThreads = 128;
constexpr int kNv = 32;                 // value columns per CTA
constexpr int kTiles = kD / kNv;        // 4 CTAs per (sequence, head)

// Stage layout (offsets within a stage; all 1024-byte aligned)
constexpr uint32_t kStWQ = 0;           // 32 KB
constexpr uint32_t kStMT = 32768;       // 16 KB
constexpr uint32_t kStKT = 49152;       // 16 KB
constexpr uint32_t kStVT = 65536;       //  4 KB (this CTA's 32 value rows)
constexpr uint32_t kStScal = 69632;     //  272 B used
constexpr uint32_t kScalCopy = 272;     //  65 floats rounded up to 16 bytes
constexpr uint32_t kStageBytes = 70656;
constexpr uint32_t kLoadBytes = 32768 + 16384 + 16384 + 4096 + kScalCopy;

constexpr uint32_t kOffST = 2 * kStageBytes;        // S^T bf16: 2 halves x 32 rows x 128 B
constexpr uint32_t kOffUhi = kOffST + 8192;         // (scaled U)^T hi: 32 rows x 128 B
constexpr uint32_t kOffUlo = kOffUhi + 4096;
constexpr uint32_t kOffSmall = kOffUlo + 4096;
constexpr uint32_t kSmemBytes = kOffSmall + 1024 + 1024;

constexpr uint32_t kTmemCols = 128;     // X[2] at 0 and 32, Z at 64

constexpr float kScale = 0.088388347648318440550f;  // 1/sqrt(128)

struct Small {
    float red[2][64];       // per-row partial sums of squares (epilogue)
    float w[kNv];           // gated-norm weight slice
    uint64_t bar_load[2];
    uint64_t bar_x, bar_z;
    uint32_t tmem_base;
    int fail;
};

__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

__device__ __forceinline__ float ld_peer_f32(const float *local, uint32_t rank)
{
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
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

// Chunks that precede sequence n, with the same clamping of malformed
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

__device__ __forceinline__ void issue_loads(const PrefillArgs &p, unsigned char *stage, uint64_t *bar,
                                            int gc, int h, int hq, int r)
{
    const unsigned char *wv = p.workspace + ((size_t)gc * p.hv + h) * kPerVHead;
    const unsigned char *wk = p.workspace + (size_t)p.max_chunks * p.hv * kPerVHead
                              + ((size_t)gc * p.hk + hq) * kKTBytes;
    mbar_arrive_expect_tx(bar, kLoadBytes);
    bulk_g2s(stage + kStWQ, wv, 32768, bar);
    bulk_g2s(stage + kStMT, wv + kWQBytes, 16384, bar);
    bulk_g2s(stage + kStKT, wk, 16384, bar);
    bulk_g2s(stage + kStVT, wv + kWQBytes + kMTBytes + r * 4096, 4096, bar);
    bulk_g2s(stage + kStScal, wv + kWQBytes + kMTBytes + kVTBytes, kScalCopy, bar);
}

template <bool kNorm>
__global__ void __launch_bounds__(kThreads, 1)
scan_kernel(PrefillArgs p)
{
    const int r = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
    const int hv = p.hv, hq = h / (hv / p.hk);
    const int tid = threadIdx.x, warp = tid >> 5;

    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Small *s = reinterpret_cast<Small *>(sm + kOffSmall);
    const uint32_t sbase = smem_u32(sm);

    int tok0 = 0, len = 0;
    const int cbase = chunk_base_of(p, n, tok0, len);
    const int nck = (len + kC - 1) / kC;

    if (tid == 0) {
        mbar_init(&s->bar_load[0], 1);
        mbar_init(&s->bar_load[1], 1);
        mbar_init(&s->bar_x, 1);
        mbar_init(&s->bar_z, 1);
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
    if (kNorm) {   // every CTA of the cluster has started before any DSMEM access
        cluster_arrive();
        cluster_wait();
    }
    const uint32_t tbase = s->tmem_base;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;

    // state slice: key row tid, value columns [32r, 32r+32)
    const size_t srow = (((size_t)n * hv + h) * kD + tid) * kD + r * kNv;
    float S[kNv];
    if (p.init_state) {
        const float4 *src = reinterpret_cast<const float4 *>(p.init_state + srow);
#pragma unroll
        for (int j = 0; j < kNv / 4; ++j) {
            const float4 x = src[j];
            S[4 * j] = x.x; S[4 * j + 1] = x.y; S[4 * j + 2] = x.z; S[4 * j + 3] = x.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < kNv; ++j) S[j] = 0.f;
    }

    int issued[2] = {0, 0};   // loads issued per stage (thread 0 only)
    if (tid == 0 && nck > 0) {
        issue_loads(p, sm, &s->bar_load[0], cbase, h, hq, r);
        issued[0] = 1;
    }

    for (int ci = 0; ci < nck; ++ci) {
        const int st = ci & 1;
        unsigned char *stage = sm + st * kStageBytes;
        const uint32_t soff = st * kStageBytes;
        const int t0 = tok0 + ci * kC;
        const int L = min(kC, tok0 + len - t0);

        // (1) S -> bf16 S^T operand (value row j, key column tid)
        {
            const uint32_t off = kOffST + (tid >> 6) * 4096;
#pragma unroll
            for (int j = 0; j < kNv; ++j)
                *reinterpret_cast<uint16_t *>(sm + off + sw128_offset(j, tid & 63)) = bf16_bits(S[j]);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();

        // (2) prefetch the next chunk; X = MT V + WQ S
        if (tid == 0) {
            if (ci + 1 < nck) {
                const int nst = (ci + 1) & 1;
                issue_loads(p, sm + nst * kStageBytes, &s->bar_load[nst], cbase + ci + 1, h, hq, r);
                ++issued[nst];
            }
            if (wait_bar(s, &s->bar_load[st], (ci >> 1) & 1, p.status)) {
                tc_fence_after();
                const uint32_t dx = tbase + st * kNv;
                constexpr uint32_t idesc = make_idesc_bf16(128, kNv);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(dx, make_sw128_desc(sbase + soff + kStMT + kk * 32),
                             make_sw128_desc(sbase + soff + kStVT + kk * 32), idesc, kk != 0);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16(dx, make_sw128_desc(sbase + soff + kStWQ + (kk >> 2) * 16384 + (kk & 3) * 32),
                             make_sw128_desc(sbase + kOffST + (kk >> 2) * 4096 + (kk & 3) * 32), idesc, 1);
            }
            mma_commit(&s->bar_x);
        }
        __syncwarp();

        // z slice for the epilogue (loads overlap the MMA)
        float zf[kNv];
        const int i_out = tid - 64;
        const bool row_ok = tid >= 64 && i_out < L;
        if (kNorm) {
            if (row_ok) {
                const uint4 *zp = reinterpret_cast<const uint4 *>(
                    reinterpret_cast<const __nv_bfloat16 *>(p.z) + ((size_t)(t0 + i_out) * hv + h) * kD + r * kNv);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    float f[8];
                    unpack8(zp[u], f);
#pragma unroll
                    for (int e = 0; e < 8; ++e) zf[u * 8 + e] = f[e];
                }
            } else {
#pragma unroll
                for (int e = 0; e < kNv; ++e) zf[e] = 0.f;
            }
        }

        // (3) U rows -> scaled hi/lo operand; output rows -> epilogue
        wait_bar(s, &s->bar_x, ci & 1, p.status);
        wait_bar(s, &s->bar_load[st], (ci >> 1) & 1, p.status);   // scal visibility
        tc_fence_after();
        float xv[kNv];
        tmem_ld32(tbase + lane_base + st * kNv, xv);
        const float *scal = reinterpret_cast<const float *>(stage + kStScal);
        float o[kNv];
        if (tid < 64) {
            const float sc = scal[tid];
#pragma unroll
            for (int j = 0; j < kNv; ++j) {
                const float u = xv[j] * sc;
                const float hi = bf16_round(u);
                *reinterpret_cast<uint16_t *>(sm + kOffUhi + sw128_offset(j, tid)) = bf16_bits(hi);
                *reinterpret_cast<uint16_t *>(sm + kOffUlo + sw128_offset(j, tid)) = bf16_bits(u - hi);
            }
        } else {
            float ss = 0.f;
#pragma unroll
            for (int j = 0; j < kNv; ++j) {
                o[j] = xv[j] * kScale;
                ss = fmaf(o[j], o[j], ss);
            }
            if (kNorm)
                s->red[ci & 1][i_out] = ss;
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (kNorm)
            cluster_arrive();

        // (4) Z = K^T U_hi + K^T U_lo
        if (tid == 0) {
            if (!*reinterpret_cast<volatile int *>(&s->fail)) {
                tc_fence_after();
                const uint32_t dz = tbase + 2 * kNv;
                constexpr uint32_t idesc = make_idesc_bf16(128, kNv);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16(dz, make_sw128_desc(sbase + soff + kStKT + (kk & 3) * 32),
                             make_sw128_desc(sbase + ((kk >> 2) ? kOffUlo : kOffUhi) + (kk & 3) * 32),
                             idesc, kk != 0);
            }
            mma_commit(&s->bar_z);
        }
        __syncwarp();
        if (tid >= 64) {
            if (kNorm) {
                cluster_wait();
                float tot = 0.f;
#pragma unroll
                for (uint32_t q = 0; q < kTiles; ++q)
                    tot += ld_peer_f32(&s->red[ci & 1][i_out], q);
                const float rn = rsqrtf(tot * (1.f / kD) + p.eps);
#pragma unroll
                for (int j = 0; j < kNv; ++j)
                    o[j] = o[j] * rn * s->w[j] * (zf[j] * sigmoid_f(zf[j]));
            }
            if (row_ok) {
                uint4 *dst = reinterpret_cast<uint4 *>(
                    reinterpret_cast<__nv_bfloat16 *>(p.out) + ((size_t)(t0 + i_out) * hv + h) * kD + r * kNv);
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    dst[u] = make_uint4(pack2(o[8 * u], o[8 * u + 1]), pack2(o[8 * u + 2], o[8 * u + 3]),
                                        pack2(o[8 * u + 4], o[8 * u + 5]), pack2(o[8 * u + 6], o[8 * u + 7]));
            }
        }

        // (5) S = e^{G_last} S + Z
        wait_bar(s, &s->bar_z, ci & 1, p.status);
        tc_fence_after();
        float zv[kNv];
        tmem_ld32(tbase + lane_base + 2 * kNv, zv);
        const float gl = scal[64];
#pragma unroll
        for (int j = 0; j < kNv; ++j)
            S[j] = fmaf(gl, S[j], zv[j]);
        if (kNorm && tid < 64)
            cluster_wait();
    }

    // final state slice
    {
        float4 *dst = reinterpret_cast<float4 *>(p.final_state + srow);
#pragma unroll
        for (int j = 0; j < kNv / 4; ++j)
            dst[j] = make_float4(S[4 * j], S[4 * j + 1], S[4 * j + 2], S[4 * j + 3]);
    }
    // no copy may still be landing in shared memory when the CTA exits
    if (tid == 0 && *reinterpret_cast<volatile int *>(&s->fail)) {
        for (int q = 0; q < 2; ++q)
            if (issued[q] > 0)
                mbar_wait(&s->bar_load[q], (issued[q] - 1) & 1);
    }
    if (kNorm) {   // peers may still read this CTA's partial sums
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
