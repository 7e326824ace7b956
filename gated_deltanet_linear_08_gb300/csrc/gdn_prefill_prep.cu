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
// cumulative gate, Gam_i = e^{G_i}:
//   D_a  = [K; Q] K^T                      raw bf16 q/k (exact), tcgen05
//   A_ij = beta_i e^{G_i-G_j} r_ki r_kj (K K^T)_ij      (j < i)
//   P_ij = e^{G_i-G_j} r_qi r_kj (Q K^T)_ij             (j <= i)
//   T    = (I + A)^{-1}                    fp32, blocked 16x16 substitution
//   MT   = [T diag(beta); P T diag(beta)]  tcgen05, hi/lo-split bf16 operands
//   [W; R] = MT diag(Gam r_k) K            tcgen05, raw K as exact operand
//   WQ   = [-W; diag(Gam r_q) Q - R]
// and it writes, in the 128-byte swizzled K-major byte image the scan kernel
// copies straight into shared memory:
//   WQ (128x128), MT (128x64), V^T (128 dv x 64 tokens), K^T (128 dk x 64,
//   once per key head) and the row scales e^{G_last - G_i} r_ki, e^{G_last}.
// The algebra: with U = Ut - W S0 (Ut = T diag(beta) V) the chunk's outputs
// are scale (P Ut + (diag(Gam) Qn - P W) S0) = scale ([MT V]_bottom + [WQ S0]_bottom)
// and U = [MT V]_top + [WQ S0]_top, so the serial scan needs one accumulator.
#include "common.cuh"
#include "kernels.h"
#include "tc05.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 128;
constexpr int kApad = 65;   // fp32 row stride of the A/T matrix (bank-conflict free)

// Shared-memory map (offsets from a 1024-byte aligned base).
constexpr uint32_t kOffKQ = 0;          // [K;Q] raw, 2 halves x 128 rows x 128 B
constexpr uint32_t kOffA = 0;           //   reused after D_a: fp32 A/T [64][65]
constexpr uint32_t kOffX = 16640;       //   reused after D_a: fp32 X [16][48]
constexpr uint32_t kOffKT = 32768;      // K^T raw, 128 rows x 128 B
constexpr uint32_t kOffAhi = 49152;     // [I; P_hi]   (V^T image before that)
constexpr uint32_t kOffAlo = 65536;     // [0; P_lo]   (A' after MT is built)
constexpr uint32_t kOffBhi = 81920;     // (T diag(beta))^T hi, 64 rows x 128 B
constexpr uint32_t kOffBlo = 90112;     // (T diag(beta))^T lo
constexpr uint32_t kOffSmall = 98304;   // per-row scalars, barrier, TMEM slot
constexpr uint32_t kSmemBytes = kOffSmall + 2048 + 1024;  // + alignment slack

constexpr uint32_t kTmemCols = 256;     // [0,64) D_a  [64,128) MT  [128,256) [W;R]

struct Small {
    float rk[64], rq[64], G[64], gam[64], beta[64];
    uint64_t mbar;
    uint32_t tmem_base;
    int fail;
};

// Locate global chunk `gc`: sequence n, first token, valid rows.  Returns
// false when gc lies past the last chunk.  Malformed cu_seqlens (decreasing
// or outside [0, T]) are clamped to empty sequences and flagged.
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
    for (int a = 1; a < 4; ++a) {
        const int ncols = 16 * a;              // columns 0 .. 16a-1
        for (int e = tid; e < 16 * ncols; e += kThreads) {
            const int r = e / ncols, col = e % ncols;
            const int j0 = (col >> 4) << 4;    // first row of block b = col/16
            float acc = 0.f;
            for (int j = j0; j < 16 * a; ++j)
                acc = fmaf(A[(16 * a + r) * kApad + j], A[j * kApad + col], acc);
            X[r * 48 + col] = acc;
        }
        __syncthreads();
        for (int e = tid; e < 16 * ncols; e += kThreads) {
            const int r = e / ncols, col = e % ncols;
            float acc = 0.f;
            for (int m = 0; m <= r; ++m)
                acc = fmaf(A[(16 * a + r) * kApad + 16 * a + m], X[m * 48 + col], acc);
            A[(16 * a + r) * kApad + col] = -acc;
        }
        __syncthreads();
    }
}

__global__ void __launch_bounds__(kThreads, 2)
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

    unsigned char *ws_v = p.workspace + ((size_t)gc * hv + h) * kPerVHead;
    unsigned char *ws_wq = ws_v;
    unsigned char *ws_mt = ws_v + kWQBytes;
    unsigned char *ws_vt = ws_mt + kMTBytes;
    float *ws_scal = reinterpret_cast<float *>(ws_vt + kVTBytes);
    unsigned char *ws_kt = p.workspace + (size_t)p.max_chunks * hv * kPerVHead
                           + ((size_t)gc * hk + hq) * kKTBytes;

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

    // ---- 1. raw K, Q (rows 0-63 K, 64-127 Q) -> [K;Q] image, K^T image,
    //         sums of squares; V -> V^T image.  16 threads per 256-byte row.
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
            if (r < 64) {
                const uint16_t *hw = reinterpret_cast<const uint16_t *>(&u);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    *reinterpret_cast<uint16_t *>(sm + kOffKT + sw128_offset(chunk * 8 + e, i)) = hw[e];
            }
        }
        for (int m = 0; m < 8; ++m) {
            const int i = (tid >> 4) + 8 * m;      // token 0..63
            uint4 u = make_uint4(0, 0, 0, 0);
            if (i < L)
                u = *reinterpret_cast<const uint4 *>(vg + ((size_t)(tok0 + i) * hv + h) * kD + chunk * 8);
            const uint16_t *hw = reinterpret_cast<const uint16_t *>(&u);
#pragma unroll
            for (int e = 0; e < 8; ++e)
                *reinterpret_cast<uint16_t *>(sm + kOffAhi + sw128_offset(chunk * 8 + e, i)) = hw[e];
        }
    }
    // ---- 2. gates: g, beta, in-chunk inclusive cumsum G, Gam = e^G
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
        // the MMA reads [K;Q] and K (rows 0-63 of the same image)
        tc_fence_after();
        if (lane == 0) {
            const uint32_t d = s->tmem_base;   // columns [0, 64)
            constexpr uint32_t idesc = make_idesc_bf16(128, 64);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t off = kOffKQ + (kk >> 2) * 16384 + (kk & 3) * 32;
                mma_bf16(d, make_sw128_desc(sbase + off), make_sw128_desc(sbase + off), idesc, kk > 0);
            }
            mma_commit(&s->mbar);
        }
        __syncwarp();
    }
    // V^T image and K^T image out to the workspace (16-byte coalesced)
    for (int e = tid; e < 1024; e += kThreads) {
        reinterpret_cast<uint4 *>(ws_vt)[e] = reinterpret_cast<const uint4 *>(sm + kOffAhi)[e];
        if (h % group == 0)
            reinterpret_cast<uint4 *>(ws_kt)[e] = reinterpret_cast<const uint4 *>(sm + kOffKT)[e];
    }
    __syncthreads();
    if (tid < 64)
        s->gam[tid] = expf(s->G[tid]);
    wait_mma(s, 0, p.status);
    tc_fence_after();

    // ---- 3. A (fp32, rows 0-63) and P split hi/lo (bf16 rows 64-127 of the
    //         [I; P_hi] and [0; P_lo] operands).
    float *sA = reinterpret_cast<float *>(sm + kOffA);
    float *sX = reinterpret_cast<float *>(sm + kOffX);
    {
        float d[64];
        {
            float t0[32], t1[32];
            const uint32_t ta = s->tmem_base + ((uint32_t)(warp * 32) << 16);
            tmem_ld32(ta, t0);
            tmem_ld32(ta + 32, t1);
#pragma unroll
            for (int j = 0; j < 32; ++j) { d[j] = t0[j]; d[32 + j] = t1[j]; }
        }
        if (tid < 64) {
            const int i = tid;
            const float Gi = s->G[i], ci = s->beta[i] * s->rk[i];
#pragma unroll
            for (int j = 0; j < 64; ++j)
                sA[i * kApad + j] = (j < i) ? ci * expf(Gi - s->G[j]) * s->rk[j] * d[j] : 0.f;
            // identity rows of [I; P_hi], zero rows of [0; P_lo]
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                uint32_t w[4] = {0, 0, 0, 0};
                if ((i >> 3) == c)
                    w[(i & 7) >> 1] = (i & 1) ? 0x3F800000u : 0x00003F80u;
                *reinterpret_cast<uint4 *>(sm + kOffAhi + sw128_chunk_offset(i, c)) = make_uint4(w[0], w[1], w[2], w[3]);
                *reinterpret_cast<uint4 *>(sm + kOffAlo + sw128_chunk_offset(i, c)) = make_uint4(0, 0, 0, 0);
            }
        } else {
            const int i = tid - 64;
            const float Gi = s->G[i], ci = s->rq[i];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                uint32_t whi[4], wlo[4];
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    float pv[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int j = c * 8 + e + u;
                        pv[u] = (j <= i) ? ci * expf(Gi - s->G[j]) * s->rk[j] * d[j] : 0.f;
                    }
                    const float h0 = bf16_round(pv[0]), h1 = bf16_round(pv[1]);
                    whi[e >> 1] = pack2(h0, h1);
                    wlo[e >> 1] = pack2(pv[0] - h0, pv[1] - h1);
                }
                *reinterpret_cast<uint4 *>(sm + kOffAhi + sw128_chunk_offset(64 + i, c)) = make_uint4(whi[0], whi[1], whi[2], whi[3]);
                *reinterpret_cast<uint4 *>(sm + kOffAlo + sw128_chunk_offset(64 + i, c)) = make_uint4(wlo[0], wlo[1], wlo[2], wlo[3]);
            }
        }
    }
    __syncthreads();

    // ---- 4. T = (I + A)^{-1} in fp32, then (T diag(beta))^T split hi/lo.
    invert_unit_lower(sA, sX, tid);
    {
        const int l = tid & 63, jh = tid >> 6;
        const float bl = s->beta[l];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
            const int c = jh * 4 + cc;
            uint32_t whi[4], wlo[4];
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
                const float v0 = sA[(c * 8 + e) * kApad + l] * bl;
                const float v1 = sA[(c * 8 + e + 1) * kApad + l] * bl;
                const float h0 = bf16_round(v0), h1 = bf16_round(v1);
                whi[e >> 1] = pack2(h0, h1);
                wlo[e >> 1] = pack2(v0 - h0, v1 - h1);
            }
            *reinterpret_cast<uint4 *>(sm + kOffBhi + sw128_chunk_offset(l, c)) = make_uint4(whi[0], whi[1], whi[2], whi[3]);
            *reinterpret_cast<uint4 *>(sm + kOffBlo + sw128_chunk_offset(l, c)) = make_uint4(wlo[0], wlo[1], wlo[2], wlo[3]);
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- 5. MT = [I; P_hi] Tb_hi + [I; P_hi] Tb_lo + [0; P_lo] Tb_hi  (fp32 in TMEM)
    if (warp == 0) {
        tc_fence_after();
        if (lane == 0) {
            const uint32_t d = s->tmem_base + 64;
            constexpr uint32_t idesc = make_idesc_bf16(128, 64);
            const uint32_t aoff[3] = {kOffAhi, kOffAhi, kOffAlo};
            const uint32_t boff[3] = {kOffBhi, kOffBlo, kOffBhi};
#pragma unroll
            for (int t = 0; t < 3; ++t)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(d, make_sw128_desc(sbase + aoff[t] + kk * 32),
                             make_sw128_desc(sbase + boff[t] + kk * 32), idesc, (t | kk) != 0);
            mma_commit(&s->mbar);
        }
        __syncwarp();
    }
    wait_mma(s, 1, p.status);
    tc_fence_after();

    // ---- 6. MT row t -> workspace (bf16 image); A' = MT diag(Gam r_k) -> smem
    {
        float mrow[64];
        {
            float t0[32], t1[32];
            const uint32_t ta = s->tmem_base + ((uint32_t)(warp * 32) << 16) + 64;
            tmem_ld32(ta, t0);
            tmem_ld32(ta + 32, t1);
#pragma unroll
            for (int j = 0; j < 32; ++j) { mrow[j] = t0[j]; mrow[32 + j] = t1[j]; }
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            uint32_t wm[4], wa[4];
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
                const int j = c * 8 + e;
                wm[e >> 1] = pack2(mrow[j], mrow[j + 1]);
                wa[e >> 1] = pack2(mrow[j] * s->gam[j] * s->rk[j], mrow[j + 1] * s->gam[j + 1] * s->rk[j + 1]);
            }
            *reinterpret_cast<uint4 *>(ws_mt + sw128_chunk_offset(tid, c)) = make_uint4(wm[0], wm[1], wm[2], wm[3]);
            *reinterpret_cast<uint4 *>(sm + kOffAlo + sw128_chunk_offset(tid, c)) = make_uint4(wa[0], wa[1], wa[2], wa[3]);
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- 7. [W; R] = A' K  (B operand: K^T image, N = 128 key dims)
    if (warp == 0) {
        tc_fence_after();
        if (lane == 0) {
            const uint32_t d = s->tmem_base + 128;
            constexpr uint32_t idesc = make_idesc_bf16(128, 128);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16(d, make_sw128_desc(sbase + kOffAlo + kk * 32),
                         make_sw128_desc(sbase + kOffKT + kk * 32), idesc, kk != 0);
            mma_commit(&s->mbar);
        }
        __syncwarp();
    }
    // row scales for the state update while the MMA runs
    if (tid < 64) {
        const float Gl = s->G[63];
        ws_scal[tid] = (tid < L) ? expf(Gl - s->G[tid]) * s->rk[tid] : 0.f;
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
            tmem_ld32(s->tmem_base + ((uint32_t)(warp * 32) << 16) + 128 + gq * 32, dv);
            float qv[32];
            if (tid >= 64 && i < L) {
                const uint4 *src = reinterpret_cast<const uint4 *>(qg + ((size_t)(tok0 + i) * hk + hq) * kD + gq * 32);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    float f[8];
                    unpack8(src[u], f);
#pragma unroll
                    for (int e = 0; e < 8; ++e) qv[u * 8 + e] = f[e];
                }
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) qv[e] = 0.f;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    const int j = u * 8 + e;
                    float v0, v1;
                    if (tid < 64) { v0 = -dv[j]; v1 = -dv[j + 1]; }
                    else { v0 = fmaf(qs, qv[j], -dv[j]); v1 = fmaf(qs, qv[j + 1], -dv[j + 1]); }
                    w[e >> 1] = pack2(v0, v1);
                }
                const int col = gq * 32 + u * 8;   // 0..127
                *reinterpret_cast<uint4 *>(ws_wq + (col >> 6) * 16384 + sw128_chunk_offset(tid, (col & 63) >> 3))
                    = make_uint4(w[0], w[1], w[2], w[3]);
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
