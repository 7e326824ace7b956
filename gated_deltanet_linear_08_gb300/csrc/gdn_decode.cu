// gdn_decode.cu -- GDN decode with the fp32 state updated in place: one
// token per sequence, or a few consecutive tokens (a speculative draft),
// against a pool of recurrent-state slots (the per-request state slots of
// serving: SGLang page "[Perf] Pack the Qwen3.5 GDN input projection on
// CUDA", Accuracy Tests, "16 mamba slots").
//
// One CTA per (sequence, value head) streams its 128x128 fp32 state (64 KB)
// exactly once: every thread keeps 16 rows x 4 columns of the state in
// registers from the read to the write.  For one token
//   r_k = S_old^T kn,  r_q = S_old^T qn          (reductions over Dk)
//   delta = beta (v - e^g r_k)
//   o = scale (e^g r_q + (kn . qn) delta)        (= scale * S_new^T qn)
//   S_new = e^g S_old + kn delta^T
// so both reductions come from the old state and the update needs no second
// pass (decode_kernel); a draft of 2..8 tokens unrolls the same recurrence
// over its tokens and still reads the state once (decode_draft_kernel).  The
// path is HBM-bound (about 7 flop per 8 bytes of state for one token): loads
// and stores are 16-byte, warp-contiguous rows of 512 bytes, marked streaming
// so they do not displace other data in L2, and each CTA prefetches into L2
// the state of the CTA one resident wave after it.
#include <atomic>

#include "common.cuh"
#include "conv.cuh"
#include "kernels.h"
#include "tc05.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRowsPerThread = kD / kWarps;  // 16

// The state slot of sequence n, or -1 when it has none: a negative index
// (skipped), or one past the pool (flagged).  Such a sequence gets zero
// outputs: every thread of the first four warps stores its column first, and
// the one-lane status update of an out-of-pool index comes after the stores.
// (With that update ahead of the stores, a build of the decode kernel lost the
// stores of lanes 1-31 of warp 0.)
__device__ __forceinline__ int resolve_slot(const DecodeArgs &p, int n, int h, int tid)
{
    int slot = n;
    bool out_of_pool = false;
    if (p.state_idx) {
        slot = p.state_idx[n];
        if (slot >= p.num_slots) {
            out_of_pool = true;
            slot = -1;
        }
    }
    if (slot < 0) {
        __nv_bfloat16 *outg = reinterpret_cast<__nv_bfloat16 *>(p.out);
        if (tid < kD)
            for (int t = 0; t < p.tokens; ++t)
                outg[(((size_t)n * p.tokens + t) * p.hv + h) * kD + tid] = __float2bfloat16_rn(0.f);
        if (out_of_pool && tid == 0)
            set_status(p.status, kStatusRange);
    }
    return slot;
}

// Conv channel of lane `lane` in warps 0-2 (k, q, v of head h / group hq).
__device__ __forceinline__ int conv_channel(int warp, int lane, int hk, int hq, int h)
{
    return (warp == 0 ? (hk + hq) * kD : warp == 1 ? hq * kD : (2 * hk + h) * kD) + lane * 4;
}

// One token of the causal conv + SiLU on four channels: f holds the raw
// inputs and receives the bf16-rounded outputs; the window of the K-1
// previous raw inputs moves on.
template <int KW>
__device__ __forceinline__ void conv_token4(const float (&cw)[KW > 0 ? KW : 1][4],
                                            float (&win)[KW > 1 ? KW - 1 : 1][4], float (&f)[4])
{
    if constexpr (KW > 0) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            float acc = cw[KW - 1][e] * f[e];
#pragma unroll
            for (int j = 0; j < KW - 1; ++j)
                acc = fmaf(cw[j][e], win[j][e], acc);
            if constexpr (KW > 1) {
#pragma unroll
                for (int j = 0; j + 1 < KW - 1; ++j)
                    win[j][e] = win[j + 1][e];
                win[KW - 2][e] = f[e];
            }
            f[e] = bf16_round(silu_f(acc));
        }
    }
}

// Conv weights and the carried window of this lane's channels (warps 0-2).
template <int KW>
__device__ __forceinline__ void conv_load4(const DecodeArgs &p, int slot, int chan,
                                           float (&cw)[KW > 0 ? KW : 1][4], float (&win)[KW > 1 ? KW - 1 : 1][4])
{
    if constexpr (KW > 0) {
        conv_weights<4, KW>(p.conv.weight, chan, cw);
#pragma unroll
        for (int j = 0; j < KW - 1; ++j)
            unpack4(*reinterpret_cast<const uint2 *>(
                        p.conv.state_in + (((size_t)slot * (KW - 1) + j) * p.conv.channels + chan)),
                    win[j]);
    }
}

// The window after the call into a separate conv-state pool (an in-place
// pool is rolled by the follow-up kernel instead).  q and k channels come
// from the group's first value head, v channels from every head.
template <int KW>
__device__ __forceinline__ void conv_store4(const DecodeArgs &p, int slot, int chan, int warp, int h,
                                            const float (&win)[KW > 1 ? KW - 1 : 1][4])
{
    if constexpr (KW > 1) {
        if (p.conv.state_out && p.conv.state_out != p.conv.state_in && (warp == 2 || h % (p.hv / p.hk) == 0)) {
#pragma unroll
            for (int j = 0; j < KW - 1; ++j)
                *reinterpret_cast<uint2 *>(p.conv.state_out + (((size_t)slot * (KW - 1) + j) * p.conv.channels + chan))
                    = make_uint2(pack2(win[j][0], win[j][1]), pack2(win[j][2], win[j][3]));
        }
    }
}

constexpr int kMaxTokens = 8;   // tokens per sequence in one call

// L2 prefetch of the 128-byte lines of one 256-byte token row, by two lanes.
__device__ __forceinline__ void prefetch_row_l2(const void *row, int half)
{
    asm volatile("prefetch.global.L2 [%0];" :: "l"(reinterpret_cast<const char *>(row) + half * 128));
}

// The state and token rows of the CTA `ahead` places later in launch order
// (about one wave of resident CTAs later) are prefetched into L2, so that
// CTA's loads hit L2 while HBM keeps streaming the following wave.  Warp 4
// (lane 0) prefetches the 64 KB state with one bulk prefetch, warp 5 the
// token rows.
__device__ __forceinline__ void prefetch_ahead_l2(const DecodeArgs &p, int ahead, int warp, int lane)
{
    const int b = blockIdx.x + blockIdx.y * gridDim.x + ahead;
    if (ahead <= 0 || b >= gridDim.x * gridDim.y)
        return;
    const int h = b % gridDim.x, n = b / gridDim.x;
    if (warp == 4 && lane == 0) {
        const int slot = p.state_idx ? p.state_idx[n] : n;
        if (slot >= 0 && slot < p.num_slots) {
            const float *S = p.state + ((size_t)slot * p.hv + h) * (size_t)(kD * kD);
            bulk_prefetch_l2(S, (uint32_t)(kD * kD * sizeof(float)));
        }
    } else if (warp == 5 && lane < 2 * kMaxTokens) {
        const int t = lane >> 1, half = lane & 1;
        if (t < p.tokens) {
            const int64_t tok = (int64_t)n * p.tokens + t;
            const int hq = h / (p.hv / p.hk);
            prefetch_row_l2(reinterpret_cast<const __nv_bfloat16 *>(p.k) + tok * p.in.k.t + (int64_t)hq * p.in.k.h, half);
            prefetch_row_l2(reinterpret_cast<const __nv_bfloat16 *>(p.q) + tok * p.in.q.t + (int64_t)hq * p.in.q.h, half);
            prefetch_row_l2(reinterpret_cast<const __nv_bfloat16 *>(p.v) + tok * p.in.v.t + (int64_t)h * p.in.v.h, half);
            if (p.z)
                prefetch_row_l2(reinterpret_cast<const __nv_bfloat16 *>(p.z) + tok * p.in.z.t + (int64_t)h * p.in.z.h, half);
        }
    }
}

// One token per sequence.  KW: width of the causal conv ahead of the core
// (0: none); warps 0-2 keep, per lane, the conv weights and the K-1 previous
// raw inputs of their four k, q or v channels in registers.
template <bool kNorm, int KW>
__global__ void __launch_bounds__(kThreads, 2)
decode_kernel(DecodeArgs p, int ahead)
{
    const int h = blockIdx.x, n = blockIdx.y;
    const int hv = p.hv, hk = p.hk;
    const int hq = h / (hv / hk);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    __shared__ float s_k[kD], s_q[kD], s_v[kD], s_delta[kD];
    __shared__ float s_part[2][kWarps][kD];
    __shared__ float s_scal[4];   // e^g, beta, kn.qn
    __shared__ float s_red[4];

    __nv_bfloat16 *outg = reinterpret_cast<__nv_bfloat16 *>(p.out);
    const int slot = resolve_slot(p, n, h, tid);
    if (slot < 0)
        return;
    float *S = p.state + ((size_t)slot * hv + h) * (size_t)(kD * kD);

    // 1. Issue every state load first so the whole 64 KB is in flight.
    float4 st[kRowsPerThread];
#pragma unroll
    for (int i = 0; i < kRowsPerThread; ++i)
        st[i] = __ldcs(reinterpret_cast<const float4 *>(S + (size_t)(warp + kWarps * i) * kD) + lane);

    // conv channels of this lane (warps 0-2: k, q, v), weights and history
    float cw[KW > 0 ? KW : 1][4], win[KW > 1 ? KW - 1 : 1][4];
    if (KW > 0 && warp < 3)
        conv_load4<KW>(p, slot, conv_channel(warp, lane, hk, hq, h), cw, win);

    const float scale = rsqrtf((float)kD);
    {
        const size_t tok = (size_t)n;   // one token per sequence
        // 2. Per-token inputs: warp 0 normalises k, warp 1 q, warp 2 loads v,
        //    warp 3 computes the gate and beta.
        if (warp < 2) {
            const Stride sd = warp == 0 ? p.in.k : p.in.q;
            const __nv_bfloat16 *src = reinterpret_cast<const __nv_bfloat16 *>(warp == 0 ? p.k : p.q)
                                       + (int64_t)tok * sd.t + (int64_t)hq * sd.h + lane * 4;
            float f[4];
            unpack4(*reinterpret_cast<const uint2 *>(src), f);
            conv_token4<KW>(cw, win, f);
            float ss = f[0] * f[0] + f[1] * f[1] + f[2] * f[2] + f[3] * f[3];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                ss += __shfl_xor_sync(0xffffffffu, ss, o);
            const float r = 1.f / sqrtf(ss + kL2Eps);
            float *dst = warp == 0 ? s_k : s_q;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                dst[lane * 4 + j] = f[j] * r;
        } else if (warp == 2) {
            const __nv_bfloat16 *src = reinterpret_cast<const __nv_bfloat16 *>(p.v)
                                       + (int64_t)tok * p.in.v.t + (int64_t)h * p.in.v.h + lane * 4;
            float f[4];
            unpack4(*reinterpret_cast<const uint2 *>(src), f);
            conv_token4<KW>(cw, win, f);
#pragma unroll
            for (int j = 0; j < 4; ++j)
                s_v[lane * 4 + j] = f[j];
        } else if (warp >= 4) {
            prefetch_ahead_l2(p, ahead, warp, lane);
        } else if (warp == 3 && lane == 0) {
            const float av = bf2f(reinterpret_cast<const __nv_bfloat16 *>(p.a)[(int64_t)tok * p.in.a.t + (int64_t)h * p.in.a.h]);
            const float bv = bf2f(reinterpret_cast<const __nv_bfloat16 *>(p.b)[(int64_t)tok * p.in.b.t + (int64_t)h * p.in.b.h]);
            s_scal[0] = expf(gate_f(av, p.A_log[h], p.dt_bias[h]));
            s_scal[1] = sigmoid_f(bv);
        }
        __syncthreads();

        // 3. Partial reductions over this thread's 16 rows, for 4 columns.
        float rk[4] = {0.f, 0.f, 0.f, 0.f}, rq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < kRowsPerThread; ++i) {
            const int r = warp + kWarps * i;
            const float kk = s_k[r], qq = s_q[r];
            rk[0] = fmaf(st[i].x, kk, rk[0]); rq[0] = fmaf(st[i].x, qq, rq[0]);
            rk[1] = fmaf(st[i].y, kk, rk[1]); rq[1] = fmaf(st[i].y, qq, rq[1]);
            rk[2] = fmaf(st[i].z, kk, rk[2]); rq[2] = fmaf(st[i].z, qq, rq[2]);
            rk[3] = fmaf(st[i].w, kk, rk[3]); rq[3] = fmaf(st[i].w, qq, rq[3]);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            s_part[0][warp][lane * 4 + j] = rk[j];
            s_part[1][warp][lane * 4 + j] = rq[j];
        }
        if (warp == 0) {
            float kq = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                kq = fmaf(s_k[lane * 4 + j], s_q[lane * 4 + j], kq);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                kq += __shfl_xor_sync(0xffffffffu, kq, o);
            if (lane == 0)
                s_scal[2] = kq;
        }
        __syncthreads();

        // 4. Column c = tid (< 128): delta and the output.
        const float eg = s_scal[0], beta = s_scal[1];
        float o = 0.f;
        if (tid < kD) {
            float sk = 0.f, sq = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                sk += s_part[0][w][tid];
                sq += s_part[1][w][tid];
            }
            const float delta = beta * (s_v[tid] - eg * sk);
            s_delta[tid] = delta;
            o = scale * (eg * sq + s_scal[2] * delta);
            if (kNorm) {
                float ss = o * o;
#pragma unroll
                for (int off = 16; off > 0; off >>= 1)
                    ss += __shfl_xor_sync(0xffffffffu, ss, off);
                if (lane == 0)
                    s_red[warp] = ss;
            }
        }
        __syncthreads();
        if (tid < kD) {
            if (kNorm) {
                const float ms = (s_red[0] + s_red[1] + s_red[2] + s_red[3]) * (1.f / kD);
                const float zz = bf2f(reinterpret_cast<const __nv_bfloat16 *>(p.z)[(int64_t)tok * p.in.z.t
                                                                                   + (int64_t)h * p.in.z.h + tid]);
                const float ww = bf2f(reinterpret_cast<const __nv_bfloat16 *>(p.norm_w)[tid]);
                o = o * rsqrtf(ms + p.eps) * ww * (zz * sigmoid_f(zz));
            }
            outg[(tok * hv + h) * kD + tid] = __float2bfloat16_rn(o);
        }

        // 5. S_new = e^g S_old + kn delta^T, kept in registers.
        const float4 d4 = *reinterpret_cast<const float4 *>(&s_delta[lane * 4]);
#pragma unroll
        for (int i = 0; i < kRowsPerThread; ++i) {
            const float kk = s_k[warp + kWarps * i];
            st[i].x = fmaf(eg, st[i].x, kk * d4.x);
            st[i].y = fmaf(eg, st[i].y, kk * d4.y);
            st[i].z = fmaf(eg, st[i].z, kk * d4.z);
            st[i].w = fmaf(eg, st[i].w, kk * d4.w);
        }
    }

    // 6. Written back in place, once.
#pragma unroll
    for (int i = 0; i < kRowsPerThread; ++i)
        __stcs(reinterpret_cast<float4 *>(S + (size_t)(warp + kWarps * i) * kD) + lane, st[i]);

    // 7. A separate conv-state pool receives the window now in registers: the
    //    K-1 last raw inputs of [old state; tokens].
    if (KW > 1 && warp < 3)
        conv_store4<KW>(p, slot, conv_channel(warp, lane, hk, hq, h), warp, h, win);
}

// A draft of 2..8 tokens per sequence, taken in one pass over the state.
// With G_t the gate summed over the draft's tokens 0..t, Gam_t = e^{G_t},
// r_ts = e^{G_t - G_s} (s <= t, never above 1) and S0 the state before the
// draft, the per-token recurrence unrolls to
//   delta_t = beta_t (v_t - Gam_t S0^T k_t) - sum_{s<t} beta_t r_ts (k_s.k_t) delta_s
//   o_t     = scale (Gam_t S0^T q_t + sum_{s<=t} r_ts (k_s.q_t) delta_s)
//   S_T     = Gam_{T-1} S0 + sum_s (r_{T-1,s} k_s) delta_s^T
// (the UT form of a prefill chunk, solved by forward substitution in each
// value column).  Every reduction reads the old state, so all 2T of them run
// in one pass, and every token's inputs are requested at entry instead of one
// token at a time.  The dot products and decay ratios are formed by warps
// that would otherwise wait on those loads, so after them the CTA meets three
// block barriers whatever the draft length.  The state is streamed once, as
// in the single-token kernel, with the same thread layout (warp w: rows
// w + 8i; lane: four columns).
constexpr int kMaxDraft = 8;
constexpr int kDotWarps = 4;   // warps 4-7 form the dot products under the input loads

template <bool kNorm>
struct DraftSmem {
    // k_t, q_t normalised, and r_{T-1,s} k_s: permuted so that the 16 rows a
    // thread of warp w owns (w + 8i) sit contiguous at [w][i] (the dot
    // products k_s.k_t and k_s.q_t run over the same permuted order)
    float kp[kMaxDraft][kWarps][kRowsPerThread], qp[kMaxDraft][kWarps][kRowsPerThread];
    float kwp[kMaxDraft][kWarps][kRowsPerThread];
    float v[kMaxDraft][kD];                    // v_t; then o_t before the norm
    float dl[kMaxDraft][kD];                   // delta_t
    float z[kNorm ? kMaxDraft : 1][kD];
    float beta[kMaxDraft], gam[kMaxDraft];
    float rat[kMaxDraft][kMaxDraft];           // r_ts, s <= t
    float kk[kMaxDraft][kMaxDraft];            // k_s . k_t, s < t
    float kq[kMaxDraft][kMaxDraft];            // k_s . q_t, s <= t
    float red[kMaxDraft][4];                   // sum of o_t^2 per column warp
};

// Two fp32 fused multiply-adds in one instruction, each rounded as fmaf:
// (x0, x1) * (y0, y1) + (z0, z1).
__device__ __forceinline__ float2 fma2(float2 x, float2 y, float2 z)
{
    unsigned long long r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;"
        : "=l"(r)
        : "l"(*reinterpret_cast<unsigned long long *>(&x)), "l"(*reinterpret_cast<unsigned long long *>(&y)),
          "l"(*reinterpret_cast<unsigned long long *>(&z)));
    return *reinterpret_cast<float2 *>(&r);
}

// Per-warp partial sums of NT consecutive tokens from t0:
// part[2t] = (S0^T k_t) and part[2t+1] = (S0^T q_t) over this warp's rows.
template <int NT, bool kNorm>
__device__ __forceinline__ void draft_partials(const float4 (&st)[kRowsPerThread], int t0, int warp, int lane,
                                               const DraftSmem<kNorm> &sm, float *s_part)
{
    float2 rk[NT][2], rq[NT][2];
#pragma unroll
    for (int u = 0; u < NT; ++u)
#pragma unroll
        for (int j = 0; j < 2; ++j)
            rk[u][j] = rq[u][j] = make_float2(0.f, 0.f);
#pragma unroll
    for (int i4 = 0; i4 < kRowsPerThread; i4 += 4) {
#pragma unroll
        for (int u = 0; u < NT; ++u) {
            const float4 k4 = *reinterpret_cast<const float4 *>(&sm.kp[t0 + u][warp][i4]);
            const float4 q4 = *reinterpret_cast<const float4 *>(&sm.qp[t0 + u][warp][i4]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 lo = make_float2(st[i4 + e].x, st[i4 + e].y), hi = make_float2(st[i4 + e].z, st[i4 + e].w);
                const float kk = e == 0 ? k4.x : e == 1 ? k4.y : e == 2 ? k4.z : k4.w;
                const float qq = e == 0 ? q4.x : e == 1 ? q4.y : e == 2 ? q4.z : q4.w;
                rk[u][0] = fma2(lo, make_float2(kk, kk), rk[u][0]);
                rk[u][1] = fma2(hi, make_float2(kk, kk), rk[u][1]);
                rq[u][0] = fma2(lo, make_float2(qq, qq), rq[u][0]);
                rq[u][1] = fma2(hi, make_float2(qq, qq), rq[u][1]);
            }
        }
    }
#pragma unroll
    for (int u = 0; u < NT; ++u) {
        const int t = t0 + u;
        *reinterpret_cast<float4 *>(s_part + ((2 * t) * kWarps + warp) * kD + lane * 4)
            = make_float4(rk[u][0].x, rk[u][0].y, rk[u][1].x, rk[u][1].y);
        *reinterpret_cast<float4 *>(s_part + ((2 * t + 1) * kWarps + warp) * kD + lane * 4)
            = make_float4(rq[u][0].x, rq[u][0].y, rq[u][1].x, rq[u][1].y);
    }
}

// Dynamic shared memory of a draft of T tokens: the per-warp partial sums.
__host__ __device__ constexpr size_t draft_part_bytes(int T)
{
    return (size_t)2 * T * kWarps * kD * sizeof(float);
}

template <bool kNorm, int KW>
__global__ void __launch_bounds__(kThreads, 2)
decode_draft_kernel(DecodeArgs p, int ahead)
{
    const int h = blockIdx.x, n = blockIdx.y;
    const int hv = p.hv, hk = p.hk, T = p.tokens;
    const int hq = h / (hv / hk);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    extern __shared__ float4 s_dyn[];
    float *s_part = reinterpret_cast<float *>(s_dyn);   // [2T][kWarps][kD]
    __shared__ __align__(16) DraftSmem<kNorm> sm;

    const int slot = resolve_slot(p, n, h, tid);
    if (slot < 0)
        return;
    float *S = p.state + ((size_t)slot * hv + h) * (size_t)(kD * kD);
    const size_t tok0 = (size_t)n * T;

    // 1. Every state load first, then every token input of the draft:
    //    warps 0-2 the k, q and v rows (through the conv, if any; k and q
    //    normalised), warp 3 the gates and decay ratios, warps 4-7 the z rows
    //    of the norm and, once warps 0-1 have stored k and q, the dot products.
    float4 st[kRowsPerThread];
#pragma unroll
    for (int i = 0; i < kRowsPerThread; ++i)
        st[i] = __ldcs(reinterpret_cast<const float4 *>(S + (size_t)(warp + kWarps * i) * kD) + lane);

    if (warp < 3) {
        const Stride sd = warp == 0 ? p.in.k : warp == 1 ? p.in.q : p.in.v;
        const void *base = warp == 0 ? p.k : warp == 1 ? p.q : p.v;
        const __nv_bfloat16 *src = reinterpret_cast<const __nv_bfloat16 *>(base) + (int64_t)tok0 * sd.t
                                   + (int64_t)(warp < 2 ? hq : h) * sd.h + lane * 4;
        uint2 raw[kMaxDraft];
#pragma unroll
        for (int t = 0; t < kMaxDraft; ++t)
            if (t < T)
                raw[t] = *reinterpret_cast<const uint2 *>(src + (int64_t)t * sd.t);
        float cw[KW > 0 ? KW : 1][4], win[KW > 1 ? KW - 1 : 1][4];
        const int chan = conv_channel(warp, lane, hk, hq, h);
        conv_load4<KW>(p, slot, chan, cw, win);
        float(*dstp)[kWarps][kRowsPerThread] = warp == 0 ? sm.kp : sm.qp;
#pragma unroll
        for (int t = 0; t < kMaxDraft; ++t) {
            if (t < T) {
                float f[4];
                unpack4(raw[t], f);
                conv_token4<KW>(cw, win, f);
                if (warp < 2) {
                    float ss = f[0] * f[0] + f[1] * f[1] + f[2] * f[2] + f[3] * f[3];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1)
                        ss += __shfl_xor_sync(0xffffffffu, ss, o);
                    const float r = 1.f / sqrtf(ss + kL2Eps);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        f[j] *= r;
                        const int e = lane * 4 + j;   // row e = (e % 8) + 8 (e / 8)
                        dstp[t][e & 7][e >> 3] = f[j];
                    }
                } else {
                    *reinterpret_cast<float4 *>(&sm.v[t][lane * 4]) = make_float4(f[0], f[1], f[2], f[3]);
                }
            }
        }
        if (warp < 2)
            named_arrive(1, (2 + kDotWarps) * 32);   // k and q stored
        conv_store4<KW>(p, slot, chan, warp, h, win);
    } else if (warp == 3) {
        float g = 0.f, bt = 0.f;
        if (lane < T) {
            const int64_t tok = (int64_t)tok0 + lane;
            g = gate_f(bf2f(reinterpret_cast<const __nv_bfloat16 *>(p.a)[tok * p.in.a.t + (int64_t)h * p.in.a.h]),
                       p.A_log[h], p.dt_bias[h]);
            bt = sigmoid_f(bf2f(reinterpret_cast<const __nv_bfloat16 *>(p.b)[tok * p.in.b.t + (int64_t)h * p.in.b.h]));
        }
#pragma unroll
        for (int o = 1; o < kMaxDraft; o <<= 1) {   // G: inclusive sum over the draft
            const float x = __shfl_up_sync(0xffffffffu, g, o);
            if (lane >= o)
                g += x;
        }
#pragma unroll
        for (int e0 = 0; e0 < kMaxDraft * kMaxDraft; e0 += 32) {
            const int e = e0 + lane, t = e / kMaxDraft, s = e % kMaxDraft;
            const float Gt = __shfl_sync(0xffffffffu, g, t), Gs = __shfl_sync(0xffffffffu, g, s);
            if (t < T && s <= t)
                sm.rat[t][s] = expf(Gt - Gs);
        }
        if (lane < T) {
            sm.beta[lane] = bt;
            sm.gam[lane] = expf(g);
        }
    } else {
        prefetch_ahead_l2(p, ahead, warp, lane);
        if (kNorm) {
            const int c = tid - 4 * 32;
            for (int t = 0; t < T; ++t)
                sm.z[t][c] = bf2f(reinterpret_cast<const __nv_bfloat16 *>(p.z)[((int64_t)tok0 + t) * p.in.z.t
                                                                               + (int64_t)h * p.in.z.h + c]);
        }
        named_sync(1, (2 + kDotWarps) * 32);
        for (int pi = warp - 4; pi < T * T; pi += kDotWarps) {
            const int s = pi / T, t = pi - s * T;
            if (s > t)
                continue;
            const float4 ks = *reinterpret_cast<const float4 *>(&sm.kp[s][0][0] + lane * 4);
            const float4 kt = *reinterpret_cast<const float4 *>(&sm.kp[t][0][0] + lane * 4);
            const float4 qt = *reinterpret_cast<const float4 *>(&sm.qp[t][0][0] + lane * 4);
            float dk = ks.x * kt.x + ks.y * kt.y + ks.z * kt.z + ks.w * kt.w;
            float dq = ks.x * qt.x + ks.y * qt.y + ks.z * qt.z + ks.w * qt.w;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                dk += __shfl_xor_sync(0xffffffffu, dk, o);
                dq += __shfl_xor_sync(0xffffffffu, dq, o);
            }
            if (lane == 0) {
                sm.kq[s][t] = dq;
                if (s < t)
                    sm.kk[s][t] = dk;
            }
        }
    }
    __syncthreads();

    // 2. The 2T reductions of the old state: per-warp partial sums, four
    //    tokens at a time.
    {
        int t0 = 0;
        for (; t0 + 4 <= T; t0 += 4)
            draft_partials<4, kNorm>(st, t0, warp, lane, sm, s_part);
        switch (T - t0) {
        case 1: draft_partials<1, kNorm>(st, t0, warp, lane, sm, s_part); break;
        case 2: draft_partials<2, kNorm>(st, t0, warp, lane, sm, s_part); break;
        case 3: draft_partials<3, kNorm>(st, t0, warp, lane, sm, s_part); break;
        default: break;
        }
    }
    __syncthreads();

    // 3. Column c = tid (< 128): delta_t and o_t by forward substitution over
    //    the draft; warps 4-7 meanwhile form the update's row factors.
    const float scale = rsqrtf((float)kD);
    if (tid < kD) {
        const int c = tid;
        float dl[kMaxDraft];
#pragma unroll
        for (int t = 0; t < kMaxDraft; ++t) {
            if (t < T) {
                float sk = 0.f, sq = 0.f;
#pragma unroll
                for (int w = 0; w < kWarps; ++w) {
                    sk += s_part[((2 * t) * kWarps + w) * kD + c];
                    sq += s_part[((2 * t + 1) * kWarps + w) * kD + c];
                }
                const float bt = sm.beta[t], gt = sm.gam[t];
                float x = bt * (sm.v[t][c] - gt * sk);
                float o = gt * sq;
#pragma unroll
                for (int s = 0; s < t; ++s) {
                    const float rts = sm.rat[t][s];
                    x = fmaf(-bt * rts * sm.kk[s][t], dl[s], x);
                    o = fmaf(rts * sm.kq[s][t], dl[s], o);
                }
                dl[t] = x;
                o = scale * fmaf(sm.kq[t][t], x, o);
                sm.dl[t][c] = x;
                sm.v[t][c] = o;
                if (kNorm) {
                    float ss = o * o;
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1)
                        ss += __shfl_xor_sync(0xffffffffu, ss, off);
                    if (lane == 0)
                        sm.red[t][warp] = ss;
                }
            }
        }
    } else {
        const int e = tid - kD;   // permuted position: warp e / 16, row slot e % 16
        const float *rl = sm.rat[T - 1];
        const float *kp = &sm.kp[0][0][0];
        for (int s = 0; s < T; ++s)
            (&sm.kwp[s][0][0])[e] = rl[s] * kp[s * kD + e];
    }
    __syncthreads();

    // 4. Outputs (through the gated norm), then S_T = Gam_{T-1} S0 + sum_s
    //    (r_{T-1,s} k_s) delta_s^T in registers, written back in place once.
    if (tid < kD) {
        __nv_bfloat16 *outg = reinterpret_cast<__nv_bfloat16 *>(p.out);
        const float ww = kNorm ? bf2f(reinterpret_cast<const __nv_bfloat16 *>(p.norm_w)[tid]) : 0.f;
        for (int t = 0; t < T; ++t) {
            float o = sm.v[t][tid];
            if (kNorm) {
                const float ms = (sm.red[t][0] + sm.red[t][1] + sm.red[t][2] + sm.red[t][3]) * (1.f / kD);
                const float zz = sm.z[t][tid];
                o = o * rsqrtf(ms + p.eps) * ww * (zz * sigmoid_f(zz));
            }
            outg[(((size_t)tok0 + t) * hv + h) * kD + tid] = __float2bfloat16_rn(o);
        }
    }
    const float gT = sm.gam[T - 1];
#pragma unroll
    for (int i = 0; i < kRowsPerThread; ++i) {
        st[i].x *= gT; st[i].y *= gT; st[i].z *= gT; st[i].w *= gT;
    }
    for (int s = 0; s < T; ++s) {
        const float4 d4 = *reinterpret_cast<const float4 *>(&sm.dl[s][lane * 4]);
        const float2 dlo = make_float2(d4.x, d4.y), dhi = make_float2(d4.z, d4.w);
#pragma unroll
        for (int i4 = 0; i4 < kRowsPerThread; i4 += 4) {
            const float4 kw4 = *reinterpret_cast<const float4 *>(&sm.kwp[s][warp][i4]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float kw = e == 0 ? kw4.x : e == 1 ? kw4.y : e == 2 ? kw4.z : kw4.w;
                float2 lo = make_float2(st[i4 + e].x, st[i4 + e].y), hi = make_float2(st[i4 + e].z, st[i4 + e].w);
                lo = fma2(make_float2(kw, kw), dlo, lo);
                hi = fma2(make_float2(kw, kw), dhi, hi);
                st[i4 + e] = make_float4(lo.x, lo.y, hi.x, hi.y);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < kRowsPerThread; ++i)
        __stcs(reinterpret_cast<float4 *>(S + (size_t)(warp + kWarps * i) * kD) + lane, st[i]);
}

// The in-place conv-state roll after a decode call: one thread per 8
// channels of a sequence's slot.  It runs once the decode grid has finished
// (every value head of a group reads the same q and k history, so none of it
// may change while any of them still runs).
constexpr int kRollThreads = 128;

__global__ void __launch_bounds__(kRollThreads)
conv_roll_kernel(DecodeArgs p)
{
    grid_dep_wait();
    const int n = blockIdx.y;
    const int c = (blockIdx.x * kRollThreads + threadIdx.x) * 8;
    if (c >= p.conv.channels)
        return;
    int slot = n;
    if (p.state_idx) {
        slot = p.state_idx[n];
        if (slot >= p.num_slots)
            return;
    }
    if (slot < 0)
        return;
    conv_roll8(p.conv, p.q, p.k, p.v, p.in, p.hk, c, slot, slot, (int64_t)n * p.tokens, p.tokens);
}

// CTAs of `kernel` resident on the current device at once (the distance of
// the one-wave-ahead L2 prefetch), computed once per device and kernel.
template <typename Kernel>
cudaError_t resident_ctas(Kernel kernel, size_t smem, std::atomic<int> (&cache)[kMaxDevices], int &out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    out = cache[dev].load(std::memory_order_relaxed);
    if (!out) {
        int sms = 0, per_sm = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, smem);
        if (e != cudaSuccess)
            return e;
        out = sms * (per_sm > 0 ? per_sm : 1);
        cache[dev].store(out, std::memory_order_relaxed);
    }
    return cudaSuccess;
}

template <bool kNorm, int KW>
cudaError_t launch_one(const DecodeArgs &args, dim3 grid, cudaStream_t stream)
{
    static std::atomic<int> resident[kMaxDevices];
    int ahead = 0;
    cudaError_t e = resident_ctas(decode_kernel<kNorm, KW>, 0, resident, ahead);
    if (e != cudaSuccess)
        return e;
    decode_kernel<kNorm, KW><<<grid, kThreads, 0, stream>>>(args, ahead);
    return cudaGetLastError();
}

template <bool kNorm>
cudaError_t launch_width(const DecodeArgs &args, dim3 grid, cudaStream_t stream)
{
    switch (args.conv.width) {
    case 1: return launch_one<kNorm, 1>(args, grid, stream);
    case 2: return launch_one<kNorm, 2>(args, grid, stream);
    case 3: return launch_one<kNorm, 3>(args, grid, stream);
    case 4: return launch_one<kNorm, 4>(args, grid, stream);
    default: return launch_one<kNorm, 0>(args, grid, stream);
    }
}

template <bool kNorm, int KW>
cudaError_t launch_draft_width(const DecodeArgs &args, dim3 grid, cudaStream_t stream)
{
    // the partial sums of the longest draft exceed the default dynamic
    // shared-memory limit: the attribute is set with the first launch on a
    // device, before the occupancy query (a racing repeat sets the same value)
    static std::atomic<bool> configured[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    if (!configured[dev].load(std::memory_order_relaxed)) {
        const cudaError_t attr = cudaFuncSetAttribute(decode_draft_kernel<kNorm, KW>,
                                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                      (int)draft_part_bytes(kMaxDraft));
        if (attr != cudaSuccess)
            return attr;
        configured[dev].store(true, std::memory_order_relaxed);
    }
    static std::atomic<int> resident[kMaxDevices];
    int ahead = 0;   // sized for the longest draft: the fewest CTAs resident
    cudaError_t e = resident_ctas(decode_draft_kernel<kNorm, KW>, draft_part_bytes(kMaxDraft), resident, ahead);
    if (e != cudaSuccess)
        return e;
    decode_draft_kernel<kNorm, KW><<<grid, kThreads, draft_part_bytes(args.tokens), stream>>>(args, ahead);
    return cudaGetLastError();
}

template <bool kNorm>
cudaError_t launch_draft(const DecodeArgs &args, dim3 grid, cudaStream_t stream)
{
    switch (args.conv.width) {
    case 1: return launch_draft_width<kNorm, 1>(args, grid, stream);
    case 2: return launch_draft_width<kNorm, 2>(args, grid, stream);
    case 3: return launch_draft_width<kNorm, 3>(args, grid, stream);
    case 4: return launch_draft_width<kNorm, 4>(args, grid, stream);
    default: return launch_draft_width<kNorm, 0>(args, grid, stream);
    }
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs &args, cudaStream_t stream)
{
    if (args.batch == 0)
        return cudaSuccess;
    dim3 grid(args.hv, args.batch);
    cudaError_t e;
    if (args.tokens > 1) {
        e = args.z ? launch_draft<true>(args, grid, stream) : launch_draft<false>(args, grid, stream);
    } else {
        e = args.z ? launch_width<true>(args, grid, stream) : launch_width<false>(args, grid, stream);
    }
    if (e != cudaSuccess || args.conv.width <= 1 || !args.conv.state_out || args.conv.state_out != args.conv.state_in)
        return e;
    // launched early behind the decode grid; it waits for that grid's end
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((args.conv.channels / 8 + kRollThreads - 1) / kRollThreads, args.batch);
    cfg.blockDim = dim3(kRollThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, conv_roll_kernel, args);
}

}  // namespace gdn
