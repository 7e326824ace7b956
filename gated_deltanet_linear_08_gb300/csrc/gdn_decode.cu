// gdn_decode.cu -- GDN decode with the fp32 state updated in place: one
// token per sequence, or a few consecutive tokens (a speculative draft),
// against a pool of recurrent-state slots (the per-request state slots of
// serving: SGLang page "[Perf] Pack the Qwen3.5 GDN input projection on
// CUDA", Accuracy Tests, "16 mamba slots").
//
// One CTA per (sequence, value head) streams its 128x128 fp32 state (64 KB)
// exactly once: every thread keeps 16 rows x 4 columns of the state in
// registers from the read, through every token, to the write.  Per token
//   r_k = S_old^T kn,  r_q = S_old^T qn          (reductions over Dk)
//   delta = beta (v - e^g r_k)
//   o = scale (e^g r_q + (kn . qn) delta)        (= scale * S_new^T qn)
//   S_new = e^g S_old + kn delta^T
// so both reductions come from the old state and the update needs no second
// pass.  The path is HBM-bound (about 7 flop per 8 bytes of state for one
// token): loads and stores are 16-byte, warp-contiguous rows of 512 bytes,
// marked streaming so they do not displace other data in L2.
#include "common.cuh"
#include "conv.cuh"
#include "kernels.h"
#include "tc05.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRowsPerThread = kD / kWarps;  // 16

// KW: width of the causal conv ahead of the core (0: none).  Warps 0-2 keep,
// per lane, the conv weights and the K-1 previous raw inputs of their four
// k, q or v channels in registers across the tokens.
template <bool kNorm, int KW>
__global__ void __launch_bounds__(kThreads, 2)
decode_kernel(DecodeArgs p)
{
    const int h = blockIdx.x, n = blockIdx.y;
    const int hv = p.hv, hk = p.hk, T = p.tokens;
    const int hq = h / (hv / hk);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    __shared__ float s_k[kD], s_q[kD], s_v[kD], s_delta[kD];
    __shared__ float s_part[2][kWarps][kD];
    __shared__ float s_scal[4];   // e^g, beta, kn.qn
    __shared__ float s_red[4];

    __nv_bfloat16 *outg = reinterpret_cast<__nv_bfloat16 *>(p.out);
    int slot = n;
    bool out_of_pool = false;
    if (p.state_idx) {
        slot = p.state_idx[n];
        if (slot >= p.num_slots) {   // out of the pool: flagged and skipped
            out_of_pool = true;
            slot = -1;
        }
    }
    if (slot < 0) {
        // No state for this sequence: zero outputs.  Every thread of the
        // first four warps stores its column first; the one-lane status
        // update of an out-of-pool index comes after the stores.  (With that
        // update ahead of the stores, a build of this kernel lost the stores
        // of lanes 1-31 of warp 0.)
        if (tid < kD)
            for (int t = 0; t < T; ++t)
                outg[(((size_t)n * T + t) * hv + h) * kD + tid] = __float2bfloat16_rn(0.f);
        if (out_of_pool && tid == 0)
            set_status(p.status, kStatusRange);
        return;
    }
    float *S = p.state + ((size_t)slot * hv + h) * (size_t)(kD * kD);

    // 1. Issue every state load first so the whole 64 KB is in flight.
    float4 st[kRowsPerThread];
#pragma unroll
    for (int i = 0; i < kRowsPerThread; ++i)
        st[i] = __ldcs(reinterpret_cast<const float4 *>(S + (size_t)(warp + kWarps * i) * kD) + lane);

    // conv channels of this lane (warps 0-2: k, q, v), weights and history
    constexpr int kHist = KW > 1 ? KW - 1 : 1;
    float cw[KW > 0 ? KW : 1][4], win[kHist][4];
    if constexpr (KW > 0) {
        if (warp < 3) {
            const int chan = (warp == 0 ? (hk + hq) * kD : warp == 1 ? hq * kD : (2 * hk + h) * kD) + lane * 4;
            conv_weights<4, KW>(p.conv.weight, chan, cw);
#pragma unroll
            for (int j = 0; j < KW - 1; ++j)
                unpack4(*reinterpret_cast<const uint2 *>(
                            p.conv.state_in + (((size_t)slot * (KW - 1) + j) * p.conv.channels + chan)),
                        win[j]);
        }
    }
    // raw token inputs -> conv + SiLU, rounded to bf16; the window moves on
    auto conv4 = [&](float (&f)[4]) {
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
    };

    const float scale = rsqrtf((float)kD);
    for (int t = 0; t < T; ++t) {
        const size_t tok = (size_t)n * T + t;
        // 2. Per-token inputs: warp 0 normalises k, warp 1 q, warp 2 loads v,
        //    warp 3 computes the gate and beta.
        if (warp < 2) {
            const Stride sd = warp == 0 ? p.in.k : p.in.q;
            const __nv_bfloat16 *src = reinterpret_cast<const __nv_bfloat16 *>(warp == 0 ? p.k : p.q)
                                       + (int64_t)tok * sd.t + (int64_t)hq * sd.h + lane * 4;
            float f[4];
            unpack4(*reinterpret_cast<const uint2 *>(src), f);
            conv4(f);
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
            conv4(f);
#pragma unroll
            for (int j = 0; j < 4; ++j)
                s_v[lane * 4 + j] = f[j];
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
        if (t + 1 < T)
            __syncthreads();   // the next token overwrites the shared inputs
    }

    // 6. Written back in place, once.
#pragma unroll
    for (int i = 0; i < kRowsPerThread; ++i)
        __stcs(reinterpret_cast<float4 *>(S + (size_t)(warp + kWarps * i) * kD) + lane, st[i]);

    // 7. A separate conv-state pool receives the window now in registers: the
    //    K-1 last raw inputs of [old state; tokens].  q and k channels come
    //    from the group's first value head, v channels from every head.  (An
    //    in-place pool is rolled by the follow-up kernel instead.)
    if constexpr (KW > 1) {
        if (warp < 3 && p.conv.state_out && p.conv.state_out != p.conv.state_in
            && (warp == 2 || h % (hv / hk) == 0)) {
            const int chan = (warp == 0 ? (hk + hq) * kD : warp == 1 ? hq * kD : (2 * hk + h) * kD) + lane * 4;
#pragma unroll
            for (int j = 0; j < KW - 1; ++j)
                *reinterpret_cast<uint2 *>(p.conv.state_out + (((size_t)slot * (KW - 1) + j) * p.conv.channels + chan))
                    = make_uint2(pack2(win[j][0], win[j][1]), pack2(win[j][2], win[j][3]));
        }
    }
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

template <bool kNorm>
void launch_width(const DecodeArgs &args, dim3 grid, cudaStream_t stream)
{
    switch (args.conv.width) {
    case 1: decode_kernel<kNorm, 1><<<grid, kThreads, 0, stream>>>(args); break;
    case 2: decode_kernel<kNorm, 2><<<grid, kThreads, 0, stream>>>(args); break;
    case 3: decode_kernel<kNorm, 3><<<grid, kThreads, 0, stream>>>(args); break;
    case 4: decode_kernel<kNorm, 4><<<grid, kThreads, 0, stream>>>(args); break;
    default: decode_kernel<kNorm, 0><<<grid, kThreads, 0, stream>>>(args);
    }
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs &args, cudaStream_t stream)
{
    if (args.batch == 0)
        return cudaSuccess;
    dim3 grid(args.hv, args.batch);
    if (args.z)
        launch_width<true>(args, grid, stream);
    else
        launch_width<false>(args, grid, stream);
    cudaError_t e = cudaGetLastError();
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
