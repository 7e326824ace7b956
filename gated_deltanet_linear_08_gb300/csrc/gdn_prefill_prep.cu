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
// cumulative gate, Gam_i = e^{G_i}, eps_i = e^{G_last - G_i}, Kn = diag(r_k) K:
//   D_a  = [K; Q] K^T                       raw bf16 q/k (exact), tcgen05
//   A_ij = beta_i e^{G_i-G_j} r_ki r_kj (K K^T)_ij      (j < i)
//   P_ij = e^{G_i-G_j} r_qi r_kj (Q K^T)_ij             (j <= i)
//   T    = (I + A)^{-1}                     16x16 diagonal blocks exactly in
//                                           fp32, the blocks below them by
//                                           warp-level fp16 products
//   MT   = [I; P] T diag(beta)              tcgen05, fp16 operands
//   [W; R] = MT diag(Gam) Kn                tcgen05
//   Ec   = Kn^T diag(eps) T diag(beta)      tcgen05 (A = Kn read MN-major)
//   Mc   = -Kn^T diag(eps) W                tcgen05
//   Bc   = Ec V                             tcgen05
// Within the chunk the delta rule gives U = T diag(beta) V - W S0 (the
// UT/WY form), S1 = e^{G_last} S0 + Kn^T diag(eps) U and outputs
// scale (diag(Gam) Qn S0 + P U), so
//   S1 = e^{G_last} S0 + Mc S0 + Bc,  Bc = Ec V
//   o  = scale (Qc S0 + Fc V),  Qc = diag(Gam r_q) Q - R,  Fc = P T diag(beta)
// and the serial scan needs one tensor-core product per chunk on its chain.
// Everything is written as the fp16 swizzled byte images the scan and output
// kernels copy straight into shared memory (layout in kernels.h).  fp16 operands
// (10-bit mantissa) keep the rounding of the state-side products 8x below
// bf16's; the bf16 inputs convert exactly.  A value of v outside the fp16
// range sets the range status bit.
//
// The chunk's q, k and v tiles arrive by tensor-map copies issued at entry:
// k and q land directly in the 128-byte-swizzled layout the first tcgen05
// product reads, so no thread waits on a global load.
#include <atomic>

#include <cuda.h>

#include "chunks.cuh"
#include "common.cuh"
#include "kernels.h"
#include "tc05.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 256;

// Shared-memory map (offsets from a 1024-byte aligned base), ~100 KB so that
// two CTAs share an SM.
//   KQ: bf16 [K;Q] as the 128-row A operand of D_a, dk halves 16 KB apart
//       (K rows of half h at h*16K, Q rows at h*16K + 8K); after D_a the K
//       rows are rescaled in place into the fp16 Kn operand.
//   V : bf16 tile of v (dk halves of 8 KB); after its conversion the fp16
//       [I; P] operand; after MT the fp16 A' = MT diag(Gam) operand.
//   Tb: fp16 (T diag(beta))^T, B operand of MT.
//   Ah, Th, Xs: 16x16 fp16 blocks for the inverse (512 B each): the six
//       blocks of A below the diagonal blocks (row-major), the ten lower
//       blocks of T stored transposed, one scratch block per merging warp.
//   Ad: fp32 diagonal 16x16 blocks of A.
//   StV: fp16 V slices [token][32] x 4, kept to the end as the B operand of Bc.
//   BE: fp16 diag(eps) T diag(beta) [token][64], MN-major B operand of Ec.
//   BM: fp16 -diag(eps) W [token][dk], MN-major B operand of Mc, dk halves
//       8 KB apart (in place of BE, once Ec is computed).
constexpr uint32_t kOffKQ = 0;
constexpr uint32_t kOffQ = 8192;        // + h * 16384
constexpr uint32_t kOffV = 32768;
constexpr uint32_t kOffP = 32768;
constexpr uint32_t kOffTb = 49152;
constexpr uint32_t kOffAh = 57344;
constexpr uint32_t kOffTh = kOffAh + 6 * 512;
constexpr uint32_t kOffXs = kOffTh + 10 * 512;
constexpr uint32_t kOffAd = kOffXs + 3 * 512;
constexpr uint32_t kOffStV = 73728;      // fp16 V slices: bulk-copied out, and the B operand of Bc
constexpr uint32_t kOffBE = 90112;
constexpr uint32_t kOffBM = 90112;       // after Ec has been computed (BE no longer needed)
constexpr uint32_t kOffSmall = kOffBM + 16384;
// Staging of the images bulk-copied to the workspace (regions free at the time).
constexpr uint32_t kOffStFc = kOffTb;    // Fc, after MT
constexpr uint32_t kOffStEc = kOffAh;    // Ec as the fp16 A operand of Bc, after the inverse
constexpr uint32_t kOffStQc = kOffP;     // Qc, after [W; R]
constexpr uint32_t kOffStMc = kOffKQ;    // Mc, after Mc
constexpr uint32_t kOffStBc = kOffAh;    // Bc (over Ec and the V slices), after Bc
constexpr uint32_t kTmaBytes = 6 * 8192;   // k, q, v: two 64x64 bf16 boxes each

// TMEM: D_a in [0,64), MT in [64,128); then Ec in [0,64) and [W; R] in
// [128,256); then Mc in [0,128) and Bc in [128,256).
constexpr uint32_t kTmemCols = 256;

constexpr float kLog2e = 1.4426950408889634f;

struct Small {
    float rk[64], rq[64];
    float G2[64];      // in-chunk cumulative gate times log2(e)
    float gam[64];     // e^{G_i}
    float beta[64];
    float eps[64];     // e^{G_last - G_i}, 0 past the chunk's end
    uint64_t mbar_tma, mbar_mma;
    uint32_t tmem_base;
    int fail;
};
constexpr uint32_t kSmemBytes = kOffSmall + ((sizeof(Small) + 127) / 128) * 128 + 1024;

// Bounded wait on one of the CTA's barriers; a timeout is recorded once and
// later waits are skipped so the CTA runs to its end without hanging.
__device__ __forceinline__ void wait_bar(Small *sm, uint64_t *bar, uint32_t parity, uint32_t *status)
{
    if (*reinterpret_cast<volatile int *>(&sm->fail))
        return;
    if (!mbar_wait(bar, parity)) {
        sm->fail = 1;
        set_status(status, kStatusWaitTimeout);
    }
}

// 16x16 fp16 block, 32-byte rows; the two 16-byte halves of row r swap places
// when bit 2 of r is set, so the eight rows ldmatrix reads at once fall in
// distinct banks.
__device__ __forceinline__ uint32_t blk_off(int r, int half)
{
    return (uint32_t)(r * 32 + ((half ^ ((r >> 2) & 1)) << 4));
}
__device__ __forceinline__ int ah_index(int a, int b) { return a * (a - 1) / 2 + b; }   // a > b
__device__ __forceinline__ int th_index(int a, int b) { return a * (a + 1) / 2 + b; }   // a >= b
// Row address lane t contributes to an x4 ldmatrix over one block.
__device__ __forceinline__ uint32_t ldsm_addr(uint32_t blk, int lane)
{
    return blk + blk_off((lane & 7) + ((lane >> 3) & 1) * 8, lane >> 4);
}
// Byte offset of (row n, k index i) in the Tb image (64 rows of 64 fp16).
__device__ __forceinline__ uint32_t tb_off(int n, int i)
{
    return (uint32_t)(n * 128 + ((((i >> 3) ^ n) & 7) << 4) + (i & 7) * 2);
}

// One block of T below the diagonal blocks, for warp-level products:
//   X = sum_{c=b}^{a-1} A_ac T_cb,   T_ab = -T_aa X
// written (transposed) into Th and, scaled by beta of its column, into Tb.
__device__ void merge_block(unsigned char *sm, const Small *s, int a, int b, int lane, int warp)
{
    const uint32_t sbase = smem_u32(sm);
    const int g = lane >> 2, t4 = lane & 3;
    float x[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    for (int c = b; c < a; ++c) {
        uint32_t fa[4], fb[4];
        ldsm_x4(ldsm_addr(sbase + kOffAh + ah_index(a, c) * 512, lane), fa);   // A_ac, row-major
        ldsm_x4(ldsm_addr(sbase + kOffTh + th_index(c, b) * 512, lane), fb);   // T_cb, stored as T^T
        mma16816(x[0], fa[0], fa[1], fa[2], fa[3], fb[0], fb[2]);
        mma16816(x[1], fa[0], fa[1], fa[2], fa[3], fb[1], fb[3]);
    }
    // X -> fp16 scratch, row-major [k][n]
    unsigned char *xs = sm + kOffXs + warp * 512;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        *reinterpret_cast<uint32_t *>(xs + blk_off(g, j) + t4 * 4) = pack2h(x[j][0], x[j][1]);
        *reinterpret_cast<uint32_t *>(xs + blk_off(g + 8, j) + t4 * 4) = pack2h(x[j][2], x[j][3]);
    }
    __syncwarp();
    uint32_t fx[4], ft[4];
    ldsm_x4_t(ldsm_addr(sbase + kOffXs + warp * 512, lane), fx);            // B = X
    ldsm_x4_t(ldsm_addr(sbase + kOffTh + th_index(a, a) * 512, lane), ft);  // A = T_aa from T^T
    float d[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    mma16816(d[0], ft[0], ft[2], ft[1], ft[3], fx[0], fx[1]);
    mma16816(d[1], ft[0], ft[2], ft[1], ft[3], fx[2], fx[3]);
    __half *th = reinterpret_cast<__half *>(sm + kOffTh + th_index(a, b) * 512);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int r = g + (e >> 1) * 8, cc = 8 * j + 2 * t4 + (e & 1);   // element (r, cc) of T_ab
            const float v = -d[j][e];
            th[(blk_off(cc, r >> 3) >> 1) + (r & 7)] = __float2half_rn(v);
            *reinterpret_cast<__half *>(sm + kOffTb + tb_off(16 * b + cc, 16 * a + r)) =
                __float2half_rn(v * s->beta[16 * b + cc]);
        }
    }
}



// kSingle: the call's single-chunk form (see below); a separate kernel, so
// that the general form is the code it would be without it.
template <bool kSingle>
__global__ void __launch_bounds__(kThreads, 2)
prep_kernel(PrefillArgs p, const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
            const __grid_constant__ CUtensorMap tm_v)
{
    const int gc = blockIdx.x, h = blockIdx.y;
    const int hv = p.hv, hq = h / (hv / p.hk);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // warp w reads TMEM lane quadrant q = w % 4 and column half ch = w / 4
    const int q = warp & 3, ch = warp >> 2;
    const int row = 32 * q + lane;          // TMEM lane of this thread

    int seq = 0, tok0 = 0, L = 0;
    bool bad = false;
    const bool live = find_chunk(p, gc, seq, tok0, L, bad);
    if (bad && gc == 0 && h == 0 && tid == 0)
        set_status(p.status, kStatusBadSeqlens);
    if (!live) {
        // single-chunk call: the last chunk index never exists, and its CTA
        // of head h writes the zero final state of every empty (or
        // malformed) sequence for h, which no chunk covers
        if (kSingle && gc == p.max_chunks - 1) {
            for (int n = 0; n < p.num_seqs; ++n) {
                const int s0 = p.cu_seqlens[n], e0 = p.cu_seqlens[n + 1];
                if (seq_ok(p, s0, e0) && e0 > s0)
                    continue;
                float4 *dst = reinterpret_cast<float4 *>(p.final_state + ((size_t)n * hv + h) * kD * kD);
                for (int e = tid; e < kD * kD / 4; e += kThreads)
                    dst[e] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        return;
    }
    // single-chunk call (every sequence within one chunk, zero initial
    // state): the state entering the chunk is zero, so this CTA finishes it:
    // final state S1 = Bc (as the scan would add it, through fp16) and
    // outputs o = scale Fc V (the output kernel's Qc S0 term is zero); no
    // record is written and the scan and output kernels do not run
    constexpr bool single = kSingle;
    // The scan kernel may be scheduled as soon as every prep CTA has started:
    // its CTAs take SMs that prep's last wave leaves free and run their
    // prologue there; griddepcontrol.wait still holds them until this whole
    // grid has finished and its writes are visible.
    grid_dep_launch();

    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Small *s = reinterpret_cast<Small *>(sm + kOffSmall);
    const uint32_t sbase = smem_u32(sm);
    unsigned char *ws = p.workspace + ((size_t)gc * hv + h) * kPerVHead;

    // ---- 1. tile copies of k, q (straight into the D_a operand layout) and v
    if (tid == 0) {
        mbar_init(&s->mbar_tma, 1);
        mbar_init(&s->mbar_mma, 1);
        mbar_fence_init();
        s->fail = 0;
        mbar_arrive_expect_tx(&s->mbar_tma, kTmaBytes);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            tma_load_3d(sm + kOffKQ + hf * 16384, &tm_k, hf * 64, hq, tok0, &s->mbar_tma);
            tma_load_3d(sm + kOffQ + hf * 16384, &tm_q, hf * 64, hq, tok0, &s->mbar_tma);
            tma_load_3d(sm + kOffV + hf * 8192, &tm_v, hf * 64, h, tok0, &s->mbar_tma);
        }
    }
    if (warp == 0) {
        tmem_alloc(&s->tmem_base, kTmemCols);
        tmem_relinquish();
        tc_fence_before();
    }
    // ---- 2. gates: g, beta, in-chunk inclusive cumsum G (under the copies)
    if (tid < 64) {
        float gv = 0.f, bv = 0.f;
        if (tid < L) {
            const int64_t tok = tok0 + tid;
            gv = gate_f(bf2f(reinterpret_cast<const __nv_bfloat16 *>(p.a)[tok * p.in.a.t + h * p.in.a.h]),
                        p.A_log[h], p.dt_bias[h]);
            bv = sigmoid_f(bf2f(reinterpret_cast<const __nv_bfloat16 *>(p.b)[tok * p.in.b.t + h * p.in.b.h]));
        }
        float c = gv;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float t = __shfl_up_sync(0xffffffffu, c, o);
            if (lane >= o) c += t;
        }
        s->G2[tid] = c;
        s->beta[tid] = bv;
    }
    __syncthreads();
    float Gnat = 0.f;
    if (tid < 64)
        Gnat = s->G2[tid] + (tid >= 32 ? s->G2[31] : 0.f);
    __syncthreads();
    if (tid < 64) {
        s->G2[tid] = Gnat * kLog2e;
        s->gam[tid] = expf(Gnat);
    }
    __syncthreads();
    if (tid < 64)
        s->eps[tid] = (tid < L) ? exp2f(s->G2[63] - s->G2[tid]) : 0.f;
    if (tid == 0 && !single)
        *reinterpret_cast<float4 *>(ws + kWsScal) = make_float4(exp2f(s->G2[63]), 0.f, 0.f, 0.f);
    wait_bar(s, &s->mbar_tma, 0, p.status);

    // rows past the chunk's end hold the next sequence's tokens (or the
    // copy's zero fill): clear them in all six tiles
    if (L < kC) {
        const int nr = kC - L;
        for (int e = tid; e < 6 * nr * 8; e += kThreads) {
            const int tile = e / (nr * 8), rem = e - tile * nr * 8;
            const uint32_t base = tile < 4 ? (uint32_t)((tile >> 1) * 16384 + (tile & 1) * 8192)
                                           : kOffV + (uint32_t)(tile - 4) * 8192;
            *reinterpret_cast<uint4 *>(sm + base + (L + (rem >> 3)) * 128 + (rem & 7) * 16) = make_uint4(0, 0, 0, 0);
        }
        __syncthreads();
    }
    // inverse L2 norms: threads 2r, 2r+1 sum the two dk halves of row r of [K; Q]
    {
        const int r = tid >> 1, hf = tid & 1, i = r & 63;
        const uint32_t rb = (uint32_t)hf * 16384u + (r < 64 ? 0u : 8192u) + (uint32_t)i * 128u;
        float ss = 0.f;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            float f[8];
            // rotate the chunk by row so the lanes of a warp hit distinct banks
            unpack8(*reinterpret_cast<const uint4 *>(sm + rb + ((c + i) & 7) * 16), f);
#pragma unroll
            for (int e = 0; e < 8; ++e)
                ss = fmaf(f[e], f[e], ss);
        }
        ss += __shfl_xor_sync(0xffffffffu, ss, 1);
        const float rn = (i < L) ? 1.f / sqrtf(ss + kL2Eps) : 0.f;
        if (hf == 0) {
            if (r < 64) s->rk[i] = rn; else s->rq[i] = rn;
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
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
            mma_commit(&s->mbar_mma);
        }
        __syncwarp();
    }

    // ---- 3. v -> four fp16 [token][32] value-slice images, staged for one bulk
    //         copy to the workspace
    {
        bool over = false;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int e = tid + k * kThreads;
            const int i = e >> 4, c16 = e & 15;
            float f[8];
            unpack8(*reinterpret_cast<const uint4 *>(sm + kOffV + (c16 >> 3) * 8192 + sw128_chunk_offset(i, c16 & 7)), f);
#pragma unroll
            for (int j = 0; j < 8; ++j)
                over |= !(fabsf(f[j]) <= kHalfMax);
            // value columns 8*c16..+7 sit in slice c16/4, 16-byte chunk c16%4
            *reinterpret_cast<uint4 *>(sm + kOffStV + (c16 >> 2) * 4096 + sw64_chunk_offset(i, c16 & 3)) = pack8h(f);
        }
        if (over)
            set_status(p.status, kStatusRange);
    }
    wait_bar(s, &s->mbar_mma, 0, p.status);
    tc_fence_after();
    // Kn = diag(r_k) K in fp16, in place of the K rows (the operand of the
    // [W; R], Ec and Mc products)
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int e = tid + k * kThreads;
        const int hf = e >> 9, i = (e >> 3) & 63, c = e & 7;
        uint4 *ptr = reinterpret_cast<uint4 *>(sm + kOffKQ + hf * 16384 + sw128_chunk_offset(i, c));
        float f[8];
        unpack8(*ptr, f);
        const float rk = s->rk[i];
#pragma unroll
        for (int j = 0; j < 8; ++j) f[j] *= rk;
        *ptr = pack8h(f);
    }
    fence_async_smem();
    __syncthreads();   // the v tile is consumed before [I; P] overwrites it
    if (tid == 0 && !single)
        bulk_s2g(ws + kWsV, sm + kOffStV, (uint32_t)kVBytes);
    __syncwarp();   // warp 0 whole again before the .aligned TMEM loads

    // ---- 4. A (fp16 blocks below the diagonal, fp32 diagonal blocks) from
    //         lanes 0-63 and P (fp16, rows 64-127 of [I; P]) from lanes
    //         64-127, columns 32 ch .. 32 ch + 31.  Rows 0-31 of A and of P
    //         have nothing at columns 32-63.
    {
        const int i = row & 63, a = i >> 4;
        if (ch == 1 && (q & 1) == 0) {
            if (q == 2) {
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    *reinterpret_cast<uint4 *>(sm + kOffP + sw128_chunk_offset(64 + i, 4 + c)) = make_uint4(0, 0, 0, 0);
            }
        } else {
            const float G2i = s->G2[i];
            const float ci = (q < 2) ? s->beta[i] * s->rk[i] : s->rq[i];
            float *Ad = reinterpret_cast<float *>(sm + kOffAd);
            float d[32];
            tmem_ld32(s->tmem_base + ((uint32_t)(32 * q) << 16) + ch * 32, d);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int j0 = ch * 32 + c * 8, b = j0 >> 4;
                float v[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int j = j0 + e;
                    const bool keep = (q < 2) ? (j < i) : (j <= i);
                    v[e] = keep ? ci * exp2f(G2i - s->G2[j]) * s->rk[j] * d[c * 8 + e] : 0.f;
                }
                if (q >= 2) {
                    *reinterpret_cast<uint4 *>(sm + kOffP + sw128_chunk_offset(64 + i, ch * 4 + c)) = pack8h(v);
                } else if (b < a) {
                    *reinterpret_cast<uint4 *>(sm + kOffAh + ah_index(a, b) * 512 + blk_off(i & 15, (j0 >> 3) & 1)) = pack8h(v);
                } else if (b == a) {
                    float4 *dst = reinterpret_cast<float4 *>(Ad + a * 256 + (i & 15) * 16 + (j0 & 15));
                    dst[0] = make_float4(v[0], v[1], v[2], v[3]);
                    dst[1] = make_float4(v[4], v[5], v[6], v[7]);
                }
            }
        }
        if (tid < 64) {   // identity rows of [I; P]
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                uint32_t w[4] = {0, 0, 0, 0};
                if ((tid >> 3) == c)
                    w[(tid & 7) >> 1] = (tid & 1) ? 0x3C000000u : 0x00003C00u;   // fp16 1.0
                *reinterpret_cast<uint4 *>(sm + kOffP + sw128_chunk_offset(tid, c)) = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
    }
    __syncthreads();

    // ---- 5. T = (I + A)^{-1}: diagonal blocks by forward substitution in
    //         fp32 (one thread per column), the upper blocks of Tb cleared
    //         meanwhile, then the blocks below the diagonal by three rounds of
    //         warp-level products (block distance 1, 2, 3)
    if (tid < 64) {
        const int b = tid >> 4, l = tid & 15;
        const float *Ad = reinterpret_cast<const float *>(sm + kOffAd) + b * 256;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float acc = (r == l) ? 1.f : 0.f;
#pragma unroll
            for (int j = 0; j < r; ++j)
                acc = fmaf(-Ad[r * 16 + j], x[j], acc);
            x[r] = (r < l) ? 0.f : acc;
        }
        // column l of T_bb: row l of the transposed block in Th, row 16b+l of Tb
        unsigned char *th = sm + kOffTh + th_index(b, b) * 512;
        const float bl = s->beta[16 * b + l];
        const int n = 16 * b + l;
#pragma unroll
        for (int qq = 0; qq < 2; ++qq) {
            float v[8], w[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                v[e] = x[8 * qq + e];
                w[e] = x[8 * qq + e] * bl;
            }
            *reinterpret_cast<uint4 *>(th + blk_off(l, qq)) = pack8h(v);
            *reinterpret_cast<uint4 *>(sm + kOffTb + n * 128 + ((((2 * b + qq) ^ n) & 7) << 4)) = pack8h(w);
        }
    } else {
        for (int e = tid - 64; e < 64 * 8; e += kThreads - 64) {
            const int n = e >> 3, k8 = e & 7;
            if (k8 < 2 * (n >> 4))
                *reinterpret_cast<uint4 *>(sm + kOffTb + n * 128 + (((k8 ^ n) & 7) << 4)) = make_uint4(0, 0, 0, 0);
        }
    }
    __syncthreads();
    if (warp < 3)
        merge_block(sm, s, warp + 1, warp, lane, warp);
    __syncthreads();
    if (warp < 2)
        merge_block(sm, s, warp + 2, warp, lane, warp);
    __syncthreads();
    if (warp == 0)
        merge_block(sm, s, 3, 0, lane, warp);
    fence_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- 6. MT = [I; P] T diag(beta)   (fp32 in TMEM columns 64..127)
    if (warp == 0) {
        tc_fence_after();
        if (lane == 0) {
            const uint32_t d = s->tmem_base + 64;
            constexpr uint32_t idesc = make_idesc_f16(128, 64);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_f16(d, make_sw128_desc(sbase + kOffP + kk * 32),
                        make_sw128_desc(sbase + kOffTb + kk * 32), idesc, kk != 0);
            mma_commit(&s->mbar_mma);
        }
        __syncwarp();
    }
    wait_bar(s, &s->mbar_mma, 1, p.status);
    tc_fence_after();

    // ---- 7. MT (row = lane, columns 32 ch ..) -> A' = MT diag(Gam) for
    //         [W; R]; rows 64-127 are Fc; rows 0-63 scaled by eps form BE.
    //         A' reuses the [I; P] buffer: the MMA that read it has completed.
    {
        float mrow[32];
        tmem_ld32(s->tmem_base + ((uint32_t)(32 * q) << 16) + 64 + ch * 32, mrow);
        const int i = row & 63;
        const float ei = (q < 2) ? s->eps[i] : 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            float m8[8], a8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                m8[e] = mrow[c * 8 + e];
                a8[e] = m8[e] * s->gam[ch * 32 + c * 8 + e];
            }
            const uint32_t off = sw128_chunk_offset(i, ch * 4 + c);
            *reinterpret_cast<uint4 *>(sm + kOffP + sw128_chunk_offset(row, ch * 4 + c)) = pack8h(a8);
            if (q >= 2) {
                *reinterpret_cast<uint4 *>(sm + kOffStFc + off) = pack8h(m8);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) m8[e] *= ei;
                *reinterpret_cast<uint4 *>(sm + kOffBE + off) = pack8h(m8);
            }
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();

    if (tid == 0 && !single)
        bulk_s2g(ws + kWsFc, sm + kOffStFc, 8192);
    __syncwarp();
    // ---- 8. Ec = Kn^T BE (TMEM [0,64); A = Kn read MN-major: dk halves 16 KB
    //         apart, 16-token steps of 2 KB) and [W; R] = A' Kn (TMEM
    //         [128,256); B = Kn read MN-major)
    if (warp == 0) {
        tc_fence_after();
        if (lane == 0) {
            constexpr uint32_t idesc_e = make_idesc_f16(128, 64, true, true);
            constexpr uint32_t idesc_w = make_idesc_f16(128, 128, false, true);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_f16(s->tmem_base, make_desc(sbase + kOffKQ + kk * 2048, 16384, 1024, kSw128),
                        make_desc(sbase + kOffBE + kk * 2048, 8192, 1024, kSw128), idesc_e, kk != 0);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_f16(s->tmem_base + 128, make_sw128_desc(sbase + kOffP + kk * 32),
                        make_desc(sbase + kOffKQ + kk * 2048, 16384, 1024, kSw128), idesc_w, kk != 0);
            mma_commit(&s->mbar_mma);
        }
        __syncwarp();
    }
    wait_bar(s, &s->mbar_mma, 0, p.status);
    tc_fence_after();

    // ---- 9. every lane's Ec row -> the fp16 A operand of Bc; rows 0-63 of
    //         [W; R] -> BM = -diag(eps) W.  Columns: dk half ch.  The Mc and
    //         Bc products need only these two images (and TMEM free of Ec
    //         and [W; R]), so they are issued as soon as both are staged; the
    //         R rows (64-127) become Qc = diag(Gam r_q) Q - R meanwhile.
    const int i = row & 63;
    {
        float ev[32];
        tmem_ld32(s->tmem_base + ((uint32_t)(32 * q) << 16) + ch * 32, ev);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            float e8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) e8[e] = ev[c * 8 + e];
            *reinterpret_cast<uint4 *>(sm + kOffStEc + sw128_chunk_offset(row, ch * 4 + c)) = pack8h(e8);
        }
    }
    float wr[2][32];
    tmem_ld32x2(s->tmem_base + ((uint32_t)(32 * q) << 16) + 128 + ch * 64,
                s->tmem_base + ((uint32_t)(32 * q) << 16) + 128 + ch * 64 + 32, wr[0], wr[1]);
    if (q < 2 && !single) {
        const float ei = s->eps[i];
#pragma unroll
        for (int g = 0; g < 2; ++g)
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                float w8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    w8[e] = -ei * wr[g][u * 8 + e];
                *reinterpret_cast<uint4 *>(sm + kOffBM + ch * 8192 + sw128_chunk_offset(i, g * 4 + u)) = pack8h(w8);
            }
    }
    if (tid == 0)
        bulk_wait_read<0>();   // the V and Fc copies are done with their staging (Bc goes there)
    __syncwarp();
    fence_async_smem();
    tc_fence_before();
    // barrier 1: the W warps (q < 2, warp 0 among them) wait for every thread
    // to have staged its Ec row and read [W; R]; the R warps only arrive
    if (q < 2)
        named_sync(1, kThreads);
    else
        named_arrive(1, kThreads);

    // ---- 10. Mc = Kn^T BM into TMEM [0,128) and Bc = Ec V into [128,256);
    //          A = the fp16 Ec image, B = the V slices read MN-major (slices
    //          4 KB apart)
    if (warp == 0) {
        tc_fence_after();
        if (lane == 0) {
            constexpr uint32_t idesc = make_idesc_f16(128, 128, true, true);
            constexpr uint32_t idesc_b = make_idesc_f16(128, 128, false, true);
            if (!single) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_f16(s->tmem_base, make_desc(sbase + kOffKQ + kk * 2048, 16384, 1024, kSw128),
                            make_desc(sbase + kOffBM + kk * 2048, 8192, 1024, kSw128), idesc, kk != 0);
            } else {
                // o = Fc V into [0,128), as the output kernel forms it: the
                // 64-row Fc image as a 128-row operand (its rows 64-127, the
                // next 8 KB, land in lanes that are not read)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_f16(s->tmem_base, make_desc(sbase + kOffStFc + kk * 32, 16, 1024, kSw128),
                            make_desc(sbase + kOffStV + kk * 1024, 4096, 512, kSw64), idesc_b, kk != 0);
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_f16(s->tmem_base + 128, make_desc(sbase + kOffStEc + kk * 32, 16, 1024, kSw128),
                        make_desc(sbase + kOffStV + kk * 1024, 4096, 512, kSw64), idesc_b, kk != 0);
            mma_commit(&s->mbar_mma);
        }
        __syncwarp();
    }
    // the R warps (q >= 2: warps 2, 3, 6, 7) turn R into Qc under the products
    // (q from the tile still in shared memory) and copy it out
    if (q >= 2 && !single) {
        const float qs = s->gam[i] * s->rq[i];
#pragma unroll
        for (int g = 0; g < 2; ++g)
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int c = g * 4 + u;   // 16-byte chunk within the dk half
                float qv[8], w8[8];
                unpack8(*reinterpret_cast<const uint4 *>(sm + kOffQ + ch * 16384 + sw128_chunk_offset(i, c)), qv);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    w8[e] = fmaf(qs, qv[e], -wr[g][u * 8 + e]);
                *reinterpret_cast<uint4 *>(sm + kOffStQc + ch * 8192 + sw128_chunk_offset(i, c)) = pack8h(w8);
            }
        // this warp's 32 Qc rows of dk half ch are 4 KB of the image: out now
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
            const uint32_t off = ch * 8192 + (q - 2) * 4096;
            bulk_s2g(ws + kWsQc0 + off, sm + kOffStQc + off, 4096);
        }
    }
    wait_bar(s, &s->mbar_mma, 1, p.status);
    tc_fence_after();
    if (single) {
        // final state row = lane (dk), value columns 64 ch ..: Bc through fp16,
        // as the scan adds it to a zero state
        float* fs = p.final_state + (((size_t)seq * hv + h) * kD + row) * kD + 64 * ch;
        {
            float bv[2][32];
            tmem_ld32x2(s->tmem_base + ((uint32_t)(32 * q) << 16) + 128 + ch * 64,
                        s->tmem_base + ((uint32_t)(32 * q) << 16) + 128 + ch * 64 + 32, bv[0], bv[1]);
#pragma unroll
            for (int g = 0; g < 2; ++g)
#pragma unroll
                for (int e = 0; e < 32; e += 4)
                    *reinterpret_cast<float4 *>(fs + 32 * g + e) =
                        make_float4(__half2float(__float2half_rn(bv[g][e])), __half2float(__float2half_rn(bv[g][e + 1])),
                                    __half2float(__float2half_rn(bv[g][e + 2])), __half2float(__float2half_rn(bv[g][e + 3])));
        }
        // outputs: token row = lane of quadrants 0-1 (warps 0, 1, 4, 5), value
        // columns 64 ch .. as two 32-column quarters, with the output kernel's
        // arithmetic: scale, the row's sum of squares over the four quarters
        // in order, gated RMSNorm, bf16 of the valid rows
        if (q < 2) {
            constexpr float kScale = 0.088388347648318440550f;   // 1/sqrt(128)
            float *red = reinterpret_cast<float *>(sm + kOffBM);   // [quarter][row]: BM is not used here
            const uint32_t ta = s->tmem_base + ((uint32_t)(32 * q) << 16) + 64 * ch;
            const bool norm = p.z != nullptr;
            const __nv_bfloat16 *zp = norm ? reinterpret_cast<const __nv_bfloat16 *>(p.z)
                                             + (int64_t)(tok0 + row) * p.in.z.t + (int64_t)h * p.in.z.h + 64 * ch
                                           : nullptr;
            float rn = 1.f;
            if (norm) {
#pragma unroll
                for (int g = 0; g < 2; ++g) {
                    float o[32];
                    tmem_ld32(ta + 32 * g, o);
                    float ss = 0.f;
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        o[e] *= kScale;
                        ss = fmaf(o[e], o[e], ss);
                    }
                    red[(2 * ch + g) * 64 + row] = ss;
                }
                named_sync(2, 128);   // warps 0, 1, 4, 5
                rn = rsqrtf((red[row] + red[64 + row] + red[128 + row] + red[192 + row]) * (1.f / kD) + p.eps);
            }
#pragma unroll
            for (int g = 0; g < 2; ++g) {
                float o[32];
                tmem_ld32(ta + 32 * g, o);
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] *= kScale;
                if (norm) {
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        float zf[8], wf[8];
                        unpack8(row < L ? reinterpret_cast<const uint4 *>(zp + 32 * g)[u] : make_uint4(0, 0, 0, 0), zf);
                        unpack8(reinterpret_cast<const uint4 *>(p.norm_w)[8 * ch + 4 * g + u], wf);
#pragma unroll
                        for (int e = 0; e < 8; ++e)   // silu(z) = z / (1 + e^-z)
                            o[8 * u + e] = o[8 * u + e] * rn * wf[e] * __fdividef(zf[e], 1.f + __expf(-zf[e]));
                    }
                }
                if (row < L) {
                    uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(p.out)
                                                           + ((size_t)(tok0 + row) * hv + h) * kD + 64 * ch + 32 * g);
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        float v8[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) v8[e] = o[8 * u + e];
                        dst[u] = pack8(v8);
                    }
                }
            }
        }
    } else {
    // Mc row = lane (output dk), columns = input dk half ch
    {
        float mv[2][32];
        tmem_ld32x2(s->tmem_base + ((uint32_t)(32 * q) << 16) + ch * 64,
                    s->tmem_base + ((uint32_t)(32 * q) << 16) + ch * 64 + 32, mv[0], mv[1]);
#pragma unroll
        for (int g = 0; g < 2; ++g)
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                float m8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) m8[e] = mv[g][u * 8 + e];
                *reinterpret_cast<uint4 *>(sm + kOffStMc + ch * 16384 + sw128_chunk_offset(row, g * 4 + u)) = pack8h(m8);
            }
        // this warp's 32 rows of dk half ch: 4 KB of the Mc image
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
            const uint32_t off = ch * 16384 + q * 4096;
            bulk_s2g(ws + kWsMc0 + off, sm + kOffStMc + off, 4096);
        }
    }

    // Bc row = lane (dk), value columns 64 ch .. = slices 2 ch, 2 ch + 1, in
    // 64-byte-swizzled rows, staged over Ec and the V slices (both read by
    // the finished products) for one bulk copy
    {
        float bv[2][32];
        tmem_ld32x2(s->tmem_base + ((uint32_t)(32 * q) << 16) + 128 + ch * 64,
                    s->tmem_base + ((uint32_t)(32 * q) << 16) + 128 + ch * 64 + 32, bv[0], bv[1]);
#pragma unroll
        for (int g = 0; g < 2; ++g) {
            unsigned char *dst = sm + kOffStBc + (2 * ch + g) * 8192;   // the record's byte image
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                float b8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) b8[e] = bv[g][u * 8 + e];
                *reinterpret_cast<uint4 *>(dst + sw64_chunk_offset(row, u)) = pack8h(b8);
            }
        }
        // this warp's 32 rows of slices 2 ch and 2 ch + 1: 2 KB of each
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
#pragma unroll
            for (int g = 0; g < 2; ++g) {
                const uint32_t off = (2 * ch + g) * 8192 + q * 2048;
                bulk_s2g(ws + kWsBc + off, sm + kOffStBc + off, 2048);
            }
        }
    }

    }   // the records of a call that continues in the scan and output kernels

    // ---- teardown: every record copy has completed before the CTA exits (each
    //      issuing lane waits for its own).  Waiting only for the copies to
    //      have read shared memory is not enough: a dependent kernel read
    //      stale records that way.
    tc_fence_before();
    __syncthreads();
    if (lane == 0)
        bulk_wait_all();
    __syncwarp();        // warp 0 whole again for the .aligned dealloc
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(s->tmem_base, kTmemCols);
    }
}

}  // namespace

namespace {
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once through the runtime.
EncodeTiledFn encode_fn()
{
    static const EncodeTiledFn fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess
            || q != cudaDriverEntryPointSuccess)
            f = nullptr;
        return reinterpret_cast<EncodeTiledFn>(f);
    }();
    return fn;
}

}  // namespace

// Tensor map over token x head rows of 128 bf16 (see kernels.h).
bool encode_tile_map(CUtensorMap *map, const void *base, int heads, int tokens, int64_t st, int64_t sh)
{
    const EncodeTiledFn fn = encode_fn();
    if (!fn || st <= 0 || sh <= 0)
        return false;
    const cuuint64_t dims[3] = {128, (cuuint64_t)heads, (cuuint64_t)tokens};
    const cuuint64_t strides[2] = {(cuuint64_t)sh * 2, (cuuint64_t)st * 2};
    const cuuint32_t box[3] = {64, 1, 64};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}


namespace {

// The chunk index: chunk_off[n] = chunks before sequence n (n = 0..N), by one
// CTA: tiles of 1024 sequences, a block-wide exclusive scan of their chunk
// counts, and a running carry.  Malformed sequences count no chunks and set
// the status bit.
constexpr int kIndexThreads = 1024;

__global__ void __launch_bounds__(kIndexThreads)
chunk_index_kernel(PrefillArgs p, int32_t *off)
{
    __shared__ int wsum[kIndexThreads / 32];
    __shared__ int carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0)
        carry = 0;
    bool bad = false;
    __syncthreads();
    for (int base = 0; base < p.num_seqs; base += kIndexThreads) {
        const int n = base + tid;
        int nc = 0;
        if (n < p.num_seqs) {
            const int s = p.cu_seqlens[n], e = p.cu_seqlens[n + 1];
            if (seq_ok(p, s, e))
                nc = (e - s + kC - 1) / kC;
            else
                bad = true;
        }
        int v = nc;   // inclusive scan within the warp
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += t;
        }
        if (lane == 31)
            wsum[warp] = v;
        __syncthreads();
        if (warp == 0) {   // inclusive scan of the warp totals
            int w = wsum[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += t;
            }
            wsum[lane] = w;
        }
        __syncthreads();
        if (n < p.num_seqs)
            off[n] = carry + (warp ? wsum[warp - 1] : 0) + v - nc;
        __syncthreads();
        if (tid == 0)
            carry += wsum[kIndexThreads / 32 - 1];
        __syncthreads();
    }
    if (tid == 0)
        off[p.num_seqs] = carry;
    if (bad)
        set_status(p.status, kStatusBadSeqlens);
}

}  // namespace

cudaError_t launch_chunk_index(const PrefillArgs &p, cudaStream_t stream)
{
    chunk_index_kernel<<<1, kIndexThreads, 0, stream>>>(p, const_cast<int32_t *>(p.chunk_off));
    return cudaGetLastError();
}

cudaError_t launch_prefill_prep(const PrefillArgs &p, cudaStream_t stream)
{
    // the shared-memory attribute, once per device (a repeat from a racing
    // host thread sets the same value)
    static std::atomic<bool> configured[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    if (!configured[dev].load(std::memory_order_relaxed)) {
        cudaError_t e = cudaFuncSetAttribute(prep_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(prep_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e != cudaSuccess)
            return e;
        configured[dev].store(true, std::memory_order_relaxed);
    }
    CUtensorMap tq, tk, tv;
    if (!encode_tile_map(&tq, p.q, p.hk, p.total_tokens, p.in.q.t, p.in.q.h)
        || !encode_tile_map(&tk, p.k, p.hk, p.total_tokens, p.in.k.t, p.in.k.h)
        || !encode_tile_map(&tv, p.v, p.hv, p.total_tokens, p.in.v.t, p.in.v.h))
        return cudaErrorInvalidValue;
    dim3 grid(p.max_chunks, p.hv);
    if (p.single_chunk)
        prep_kernel<true><<<grid, kThreads, kSmemBytes, stream>>>(p, tq, tk, tv);
    else
        prep_kernel<false><<<grid, kThreads, kSmemBytes, stream>>>(p, tq, tk, tv);
    return cudaGetLastError();
}

}  // namespace gdn
