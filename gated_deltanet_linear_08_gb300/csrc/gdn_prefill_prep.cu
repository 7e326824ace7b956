// gdn_prefill_prep.cu -- chunk-parallel half of the chunked GDN prefill.
//
// One CTA per (64-token chunk, value head).  Everything here depends only on
// the chunk's own tokens, never on the recurrent state, so all chunks of all
// sequences run at once (the "chunked kernel" of the JevAny page, "Add opt-in
// fused Qwen3.5 inference kernels", Summary; chunk boundaries as in the
// pegainfer page, Correctness: T = 63/64/65/127/128).
//
// Per chunk (L <= 64 valid rows; padded rows are zero and change nothing),
// with r_k, r_q the inverse L2 norms, g/beta the gate and beta, G the in-chunk
// cumulative gate, Gam_i = e^{G_i}, Kn = diag(r_k) K:
//   D_a  = [K; Q] K^T                       raw bf16 q/k (exact), tcgen05
//   A_ij = beta_i e^{G_i-G_j} r_ki r_kj (K K^T)_ij      (j < i)
//   P_ij = e^{G_i-G_j} r_qi r_kj (Q K^T)_ij             (j <= i)
//   T    = (I + A)^{-1}                     fp32, blocked 16x16 substitution
//   MT   = [I; P] T diag(beta)              tcgen05, fp16 operands
//   [W; R] = MT diag(Gam) Kn                tcgen05, fp16 operands
//   WQ   = [-W; diag(Gam r_q) Q - R]
// and it writes, as the fp16 swizzled byte images the scan kernel copies
// straight into shared memory: WQ (128x128), MT (128x64), V (four [token][32]
// value slices), Kn ([token][dk], once per key head) and the row scales
// e^{G_last - G_i} and e^{G_last}.
// With U = T diag(beta) V - W S0 the chunk's outputs are
//   scale (P T diag(beta) V + (diag(Gam) Qn - P W) S0) = scale [MT V + WQ S0]_bottom
// and U = [MT V + WQ S0]_top, so the serial scan needs one accumulator.
// fp16 operands (10-bit mantissa) keep the rounding of the state-side
// products 8x below bf16's; the bf16 inputs convert exactly.  A value of v
// outside the fp16 range sets the range status bit.
#include "common.cuh"
#include "kernels.h"
#include "tc05.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 128;
constexpr int kApad = 65;   // fp32 row stride of the A/T matrix (bank-conflict free)

// Shared-memory map (offsets from a 1024-byte aligned base), ~51 KB so that
// four CTAs share an SM.  Region R0 is reused as the kernel goes:
//   [K;Q] bf16 image (until D_a completes)
//   -> fp32 A/T [64][65], fp32 X [16][48], fp16 (T diag(beta))^T
//   -> fp16 Kn image (after T diag(beta) has been consumed by the MT product)
constexpr uint32_t kOffKQ = 0;          // bf16 [K;Q] raw, 2 halves x 128 rows x 128 B
constexpr uint32_t kOffA = 0;           // fp32 A, then T, [64][65]
constexpr uint32_t kOffX = 16640;       // fp32 X [16][48] of the blocked inverse
constexpr uint32_t kOffTb = 20480;      // fp16 (T diag(beta))^T, 64 rows x 128 B
constexpr uint32_t kOffKn = 0;          // fp16 Kn [token][dk], dk halves of 8 KB
constexpr uint32_t kOffP = 32768;       // fp16 [I; P], 128 rows x 128 B; then A'
constexpr uint32_t kOffSmall = 49152;   // per-row scalars, barrier, TMEM slot
constexpr uint32_t kSmemBytes = kOffSmall + 2048 + 1024;  // + alignment slack

// TMEM: D_a in [0,64), MT in [64,128); [W; R] reuses [0,128) once both have
// been read.
constexpr uint32_t kTmemCols = 128;

struct Small {
    float rk[64], rq[64], G[64], gam[64], beta[64];
    uint64_t mbar;
    uint32_t tmem_base;
    int fail;
};

// Locate global chunk `gc`: first token and valid rows.  Returns false when gc
// lies past the last chunk.  Malformed cu_seqlens (decreasing or outside
// [0, T]) are treated as empty sequences and flagged.
__device__ bool locate_chunk(const PrefillArgs &p, int gc, int &tok0, int &L, bool &bad)
{
    int c = 0;
    bad = false;
    for (int n = 0; n < p.num_seqs; ++n) {
        int s = p.cu_seqlens[n], e = p.cu_seqlens[n + 1];
        if (s < 0 || e < s || e > p.total_tokens) {
            bad = true;
            continue;
        }
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

// Bounded wait on the CTA's MMA barrier; a timeout is recorded once and later
// waits are skipped so the CTA runs to its end without hanging.
__device__ __forceinline__ void wait_mma(Small *sm, uint32_t parity, uint32_t *status)
{
    if (*reinterpret_cast<volatile int *>(&sm->fail))
        return;
    if (!mbar_wait(&sm->mbar, parity)) {
        sm->fail = 1;
        set_status(status, kStatusWaitTimeout);
    }
}

// Inverse of the unit lower-triangular (I + A), in place in fp32 (row stride
// kApad).  16x16 diagonal blocks by forward substitution (one thread per
// column), then block rows a = 1..3: X = sum_c A_ac T_cb, T_ab = -T_aa X.
template <int a>
__device__ __forceinline__ void invert_block_row(float *A, float *X, int tid)
{
    constexpr int ncols = 16 * a;                    // columns 0 .. 16a-1
    constexpr int per = 16 * ncols / kThreads;       // outputs per thread (2, 4, 6)
    static_assert(16 * ncols % kThreads == 0, "outputs divide evenly");
    // X[r][col] = sum over blocks b = col/16 .. a-1 of A[16a+r][16b..] T[16b..][col]
#pragma unroll
    for (int k = 0; k < per; ++k) {
        const int e = tid + k * kThreads;
        const int r = e / ncols, col = e % ncols, cb = col >> 4;
        const float *arow = A + (16 * a + r) * kApad;
        float acc = 0.f;
#pragma unroll
        for (int b = 0; b < a; ++b) {
            if (b >= cb) {
#pragma unroll
                for (int m = 0; m < 16; ++m)
                    acc = fmaf(arow[16 * b + m], A[(16 * b + m) * kApad + col], acc);
            }
        }
        X[r * 48 + col] = acc;
    }
    __syncthreads();
    // T[16a+r][col] = -sum_m T_aa[r][m] X[m][col]; T_aa's upper part is stored
    // as zeros, so the sum runs over all 16 m
#pragma unroll
    for (int k = 0; k < per; ++k) {
        const int e = tid + k * kThreads;
        const int r = e / ncols, col = e % ncols;
        const float *trow = A + (16 * a + r) * kApad + 16 * a;
        float acc = 0.f;
#pragma unroll
        for (int m = 0; m < 16; ++m)
            acc = fmaf(trow[m], X[m * 48 + col], acc);
        A[(16 * a + r) * kApad + col] = -acc;
    }
    __syncthreads();
}

__device__ void invert_unit_lower(float *A, float *X, int tid)
{
    const int b = (tid >> 4) & 3, l = tid & 15, o = b * 16;
    float x[16];
    if (tid < 64) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float acc = (i == l) ? 1.f : 0.f;
#pragma unroll
            for (int j = 0; j < i; ++j)
                acc = fmaf(-A[(o + i) * kApad + o + j], x[j], acc);
            x[i] = (i < l) ? 0.f : acc;
        }
    }
    __syncthreads();   // every read of the diagonal blocks precedes the writes
    if (tid < 64) {
#pragma unroll
        for (int i = 0; i < 16; ++i)
            A[(o + i) * kApad + o + l] = x[i];
    }
    __syncthreads();
    invert_block_row<1>(A, X, tid);
    invert_block_row<2>(A, X, tid);
    invert_block_row<3>(A, X, tid);
}

__global__ void __launch_bounds__(kThreads, 4)
prep_kernel(PrefillArgs p)
{
    const int gc = blockIdx.x, h = blockIdx.y;
    const int hv = p.hv, hk = p.hk, group = hv / hk, hq = h / group;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    int tok0 = 0, L = 0;
    bool bad = false;
    const bool live = locate_chunk(p, gc, tok0, L, bad);
    if (bad && gc == 0 && h == 0 && tid == 0)
        set_status(p.status, kStatusBadSeqlens);
    if (!live)
        return;

    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Small *s = reinterpret_cast<Small *>(sm + kOffSmall);
    const uint32_t sbase = smem_u32(sm);

    unsigned char *ws_wq = p.workspace + ((size_t)gc * hv + h) * kPerVHead;
    unsigned char *ws_mt = ws_wq + kWQBytes;
    unsigned char *ws_vimg = ws_mt + kMTBytes;
    float *ws_scal = reinterpret_cast<float *>(ws_vimg + kVBytes);
    unsigned char *ws_k = p.workspace + (size_t)p.max_chunks * hv * kPerVHead
                          + ((size_t)gc * hk + hq) * kKBytes;

    if (tid == 0) {
        mbar_init(&s->mbar, 1);
        mbar_fence_init();
        s->fail = 0;
    }
    if (warp == 0) {
        tmem_alloc(&s->tmem_base, kTmemCols);
        tmem_relinquish();
        tc_fence_before();
    }

    // ---- 1. raw K, Q (rows 0-63 K, 64-127 Q) -> bf16 [K;Q] image and sums of
    //         squares; V -> four fp16 [token][32] value-slice images in the
    //         workspace.  16 threads per 256-byte row.
    const __nv_bfloat16 *qg = reinterpret_cast<const __nv_bfloat16 *>(p.q);
    const __nv_bfloat16 *kg = reinterpret_cast<const __nv_bfloat16 *>(p.k);
    const __nv_bfloat16 *vg = reinterpret_cast<const __nv_bfloat16 *>(p.v);
    {
        const int chunk = tid & 15;
        for (int m = 0; m < 16; ++m) {
            const int r = (tid >> 4) + 8 * m;      // 0..127
            const int i = r & 63;
            uint4 u = make_uint4(0, 0, 0, 0);
            if (i < L) {
                const __nv_bfloat16 *src = (r < 64 ? kg : qg) + ((size_t)(tok0 + i) * hk + hq) * kD;
                u = *reinterpret_cast<const uint4 *>(src + chunk * 8);
            }
            float f[8];
            unpack8(u, f);
            float ss = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e)
                ss = fmaf(f[e], f[e], ss);
#pragma unroll
            for (int o = 8; o > 0; o >>= 1)
                ss += __shfl_xor_sync(0xffffffffu, ss, o);
            if (chunk == 0) {
                const float rn = (i < L) ? 1.f / sqrtf(ss + kL2Eps) : 0.f;
                if (r < 64) s->rk[i] = rn; else s->rq[i] = rn;
            }
            *reinterpret_cast<uint4 *>(sm + kOffKQ + (chunk >> 3) * 16384
                                       + sw128_chunk_offset(r, chunk & 7)) = u;
        }
        bool over = false;
        for (int m = 0; m < 8; ++m) {
            const int i = (tid >> 4) + 8 * m;      // token 0..63
            uint4 u = make_uint4(0, 0, 0, 0);
            if (i < L)
                u = *reinterpret_cast<const uint4 *>(vg + ((size_t)(tok0 + i) * hv + h) * kD + chunk * 8);
            float f[8];
            unpack8(u, f);
#pragma unroll
            for (int e = 0; e < 8; ++e)
                over |= !(fabsf(f[e]) <= kHalfMax);
            // value columns 8*chunk..+7 sit in slice chunk/4, 16-byte chunk chunk%4
            *reinterpret_cast<uint4 *>(ws_vimg + (chunk >> 2) * 4096 + sw64_chunk_offset(i, chunk & 3)) = pack8h(f);
        }
        if (over)
            set_status(p.status, kStatusRange);
    }
    // ---- 2. gates: g, beta, in-chunk inclusive cumsum G
    if (tid < 64) {
        float gv = 0.f, bv = 0.f;
        if (tid < L) {
            const size_t idx = (size_t)(tok0 + tid) * hv + h;
            gv = gate_f(bf2f(reinterpret_cast<const __nv_bfloat16 *>(p.a)[idx]), p.A_log[h], p.dt_bias[h]);
            bv = sigmoid_f(bf2f(reinterpret_cast<const __nv_bfloat16 *>(p.b)[idx]));
        }
        float c = gv;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float t = __shfl_up_sync(0xffffffffu, c, o);
            if (lane >= o) c += t;
        }
        s->G[tid] = c;
        s->beta[tid] = bv;
    }
    fence_async_smem();
    __syncthreads();
    if (tid >= 32 && tid < 64)
        s->G[tid] += s->G[31];
    if (warp == 0) {
        // D_a = [K;Q] K^T in bf16: the B operand is the K rows of the same image
        tc_fence_after();
        if (lane == 0) {
            const uint32_t d = s->tmem_base;   // columns [0, 64)
            constexpr uint32_t idesc = make_idesc_bf16(128, 64);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t off = kOffKQ + (kk >> 2) * 16384 + (kk & 3) * 32;
                mma_f16(d, make_sw128_desc(sbase + off), make_sw128_desc(sbase + off), idesc, kk > 0);
            }
            mma_commit(&s->mbar);
        }
        __syncwarp();
    }
    __syncthreads();   // G complete before gam
    if (tid < 64)
        s->gam[tid] = expf(s->G[tid]);
    wait_mma(s, 0, p.status);
    tc_fence_after();

    // ---- 3. A (fp32, rows 0-63) and P (fp16, rows 64-127 of [I; P]); A
    //         overwrites the [K;Q] image, which D_a has finished reading.
    //         Columns are taken 32 at a time to bound register use.
    float *sA = reinterpret_cast<float *>(sm + kOffA);
    float *sX = reinterpret_cast<float *>(sm + kOffX);
    {
        const uint32_t ta = s->tmem_base + ((uint32_t)(warp * 32) << 16);
        const int i = tid & 63;
        const float Gi = s->G[i];
        const float ci = (tid < 64) ? s->beta[i] * s->rk[i] : s->rq[i];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            float d[32];
            tmem_ld32(ta + half * 32, d);
            if (tid < 64) {
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    const int j = half * 32 + jj;
                    sA[i * kApad + j] = (j < i) ? ci * __expf(Gi - s->G[j]) * s->rk[j] * d[jj] : 0.f;
                }
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    float pv[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int j = half * 32 + c * 8 + e;
                        pv[e] = (j <= i) ? ci * __expf(Gi - s->G[j]) * s->rk[j] * d[c * 8 + e] : 0.f;
                    }
                    *reinterpret_cast<uint4 *>(sm + kOffP + sw128_chunk_offset(64 + i, half * 4 + c)) = pack8h(pv);
                }
            }
        }
        if (tid < 64) {   // identity rows of [I; P]
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                uint32_t w[4] = {0, 0, 0, 0};
                if ((i >> 3) == c)
                    w[(i & 7) >> 1] = (i & 1) ? 0x3C000000u : 0x00003C00u;   // fp16 1.0
                *reinterpret_cast<uint4 *>(sm + kOffP + sw128_chunk_offset(i, c)) = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
    }
    __syncthreads();

    // ---- 4. T = (I + A)^{-1} in fp32, then (T diag(beta))^T in fp16
    invert_unit_lower(sA, sX, tid);
    {
        const int l = tid & 63, jh = tid >> 6;
        const float bl = s->beta[l];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
            const int c = jh * 4 + cc;
            float v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
                v[e] = sA[(c * 8 + e) * kApad + l] * bl;
            *reinterpret_cast<uint4 *>(sm + kOffTb + sw128_chunk_offset(l, c)) = pack8h(v);
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- 5. MT = [I; P] T diag(beta)   (fp32 in TMEM columns 64..127)
    if (warp == 0) {
        tc_fence_after();
        if (lane == 0) {
            const uint32_t d = s->tmem_base + 64;
            constexpr uint32_t idesc = make_idesc_f16(128, 64);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_f16(d, make_sw128_desc(sbase + kOffP + kk * 32),
                        make_sw128_desc(sbase + kOffTb + kk * 32), idesc, kk != 0);
            mma_commit(&s->mbar);
        }
        __syncwarp();
    }
    // Kn = diag(r_k) K in fp16, [token][dk] in dk halves of 8 KB (the operand
    // layout of [W; R] below and of the scan kernel's state update), built
    // from a second read of K while the MMA runs; it overwrites A, which is
    // no longer needed (T diag(beta) lives elsewhere)
    for (int e = tid; e < 1024; e += kThreads) {
        const int half = e >> 9, i = (e >> 3) & 63, cc = e & 7;
        float f[8];
        if (i < L) {
            unpack8(*reinterpret_cast<const uint4 *>(kg + ((size_t)(tok0 + i) * hk + hq) * kD + half * 64 + cc * 8), f);
            const float rk = s->rk[i];
#pragma unroll
            for (int j = 0; j < 8; ++j) f[j] *= rk;
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) f[j] = 0.f;
        }
        const uint4 hv8 = pack8h(f);
        const uint32_t off = sw128_chunk_offset(i, cc);
        *reinterpret_cast<uint4 *>(sm + kOffKn + half * 8192 + off) = hv8;
        if (h % group == 0)
            *reinterpret_cast<uint4 *>(ws_k + half * 8192 + off) = hv8;
    }
    wait_mma(s, 1, p.status);
    tc_fence_after();

    // ---- 6. MT row t -> workspace (fp16 image); A' = MT diag(Gam) -> smem
    //         (A' reuses the [I; P] buffer: the MMA that read it has completed)
    {
        const uint32_t ta = s->tmem_base + ((uint32_t)(warp * 32) << 16) + 64;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            float mrow[32];
            tmem_ld32(ta + half * 32, mrow);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                float m8[8], a8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    m8[e] = mrow[c * 8 + e];
                    a8[e] = m8[e] * s->gam[half * 32 + c * 8 + e];
                }
                *reinterpret_cast<uint4 *>(ws_mt + sw128_chunk_offset(tid, half * 4 + c)) = pack8h(m8);
                *reinterpret_cast<uint4 *>(sm + kOffP + sw128_chunk_offset(tid, half * 4 + c)) = pack8h(a8);
            }
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- 7. [W; R] = A' Kn into TMEM columns 0..127 (D_a and MT have been
    //         read).  B = Kn read MN-major: dk halves 8 KB apart, 8-token
    //         groups 1024 bytes apart; N = 128 key dims.
    if (warp == 0) {
        tc_fence_after();
        if (lane == 0) {
            const uint32_t d = s->tmem_base;
            constexpr uint32_t idesc = make_idesc_f16(128, 128, false, true);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_f16(d, make_sw128_desc(sbase + kOffP + kk * 32),
                        make_desc(sbase + kOffKn + kk * 2048, 8192, 1024, kSw128), idesc, kk != 0);
            mma_commit(&s->mbar);
        }
        __syncwarp();
    }
    // row scales for the state update while the MMA runs
    if (tid < 64) {
        const float Gl = s->G[63];
        ws_scal[tid] = (tid < L) ? expf(Gl - s->G[tid]) : 0.f;
        if (tid == 0)
            ws_scal[64] = expf(Gl);
    }
    wait_mma(s, 0, p.status);
    tc_fence_after();

    // ---- 8. WQ = [-W; diag(Gam r_q) Q - R] -> workspace (two 64-wide halves)
    {
        const int i = tid - 64;   // token row of the Q part (warps 2-3)
        const float qs = (tid >= 64) ? s->gam[i] * s->rq[i] : 0.f;
        for (int gq = 0; gq < 4; ++gq) {
            float dv[32];
            tmem_ld32(s->tmem_base + ((uint32_t)(warp * 32) << 16) + gq * 32, dv);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                float qv[8];
                if (tid >= 64 && i < L)
                    unpack8(reinterpret_cast<const uint4 *>(qg + ((size_t)(tok0 + i) * hk + hq) * kD + gq * 32)[u], qv);
                else
#pragma unroll
                    for (int e = 0; e < 8; ++e) qv[e] = 0.f;
                float w8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    w8[e] = (tid < 64) ? -dv[u * 8 + e] : fmaf(qs, qv[e], -dv[u * 8 + e]);
                const int col = gq * 32 + u * 8;   // 0..127
                *reinterpret_cast<uint4 *>(ws_wq + (col >> 6) * 16384 + sw128_chunk_offset(tid, (col & 63) >> 3)) = pack8h(w8);
            }
        }
    }

    // ---- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(s->tmem_base, kTmemCols);
    }
}

}  // namespace

cudaError_t launch_prefill_prep(const PrefillArgs &p, cudaStream_t stream)
{
    static bool configured = false;   // attribute is per function, process-wide
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e != cudaSuccess)
            return e;
        configured = true;
    }
    dim3 grid(p.max_chunks, p.hv);
    prep_kernel<<<grid, kThreads, kSmemBytes, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace gdn
