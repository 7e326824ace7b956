// conv.cuh -- the short causal conv1d + SiLU over the q | k | v channels that
// runs ahead of the GDN core in a Qwen3-Next / Qwen3.5 linear-attention layer
// (JevAny page "Add opt-in fused Qwen3.5 inference kernels", Measurements:
// causal-conv1d is one of the path's dependencies), and the roll of the
// per-sequence conv state that carries it across calls.
//
// Channels: q heads (Hk x 128), then k heads (Hk x 128), then v heads
// (Hv x 128); weight [C][K] bf16; state [rows][K-1][C] bf16, oldest first.
//   y[t, c] = silu( sum_j w[c][j] x[t-(K-1)+j, c] ),  rounded to bf16
// The products and the sum run in fp32 (bf16 x bf16 products are exact in
// fp32), so only the final bf16 rounding is visible in the core's inputs.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace gdn {

constexpr int kMaxConvWidth = 4;

// SiLU in fp32: x sigmoid(x), exact to a few fp32 ulps.
__device__ __forceinline__ float silu_f(float x) { return __fdividef(x, 1.f + __expf(-x)); }

// Weights of the N channels c .. c+N-1 (c a multiple of 4), w[j][e] for tap
// j of channel c+e: N*KW contiguous bf16 read as 8-byte vectors (the weight
// array is 16-byte aligned and a channel group starts at a multiple of 8 B).
template <int N, int KW>
__device__ __forceinline__ void conv_weights(const __nv_bfloat16 *weight, int c, float (&w)[KW][N])
{
    static_assert((N * KW) % 4 == 0, "whole 8-byte vectors");
    const uint2 *src = reinterpret_cast<const uint2 *>(weight + (size_t)c * KW);
#pragma unroll
    for (int v = 0; v < N * KW / 4; ++v) {
        const uint2 u = src[v];
        const uint32_t h[2] = {u.x, u.y};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int f = 4 * v + k;   // flat index e * KW + j
            w[f % KW][f / KW] = __uint_as_float(k & 1 ? (h[k >> 1] & 0xFFFF0000u) : (h[k >> 1] << 16));
        }
    }
}

// First element of conv channels c, c+1, ... (c a multiple of 4) of token
// `tok` in the token inputs, which hold each head as 128 contiguous channels.
__device__ __forceinline__ const __nv_bfloat16 *conv_src(const void *q, const void *k, const void *v,
                                                         const InputStrides &in, int hk, int c, int64_t tok)
{
    const int qk = hk * kD;
    const void *base = q;
    Stride sd = in.q;
    if (c >= 2 * qk) {
        base = v; sd = in.v; c -= 2 * qk;
    } else if (c >= qk) {
        base = k; sd = in.k; c -= qk;
    }
    return reinterpret_cast<const __nv_bfloat16 *>(base) + tok * sd.t + (int64_t)(c / kD) * sd.h + (c % kD);
}

// The carried state after `len` tokens starting at `tok0`: the last K-1 raw
// inputs of [state_in row in_row; the tokens], for channels c .. c+7.  The
// thread reads every value before it writes any, so state_out may be
// state_in (each thread owns its channels of the row).
__device__ __forceinline__ void conv_roll8(const ConvArgs &cv, const void *q, const void *k, const void *v,
                                           const InputStrides &in, int hk, int c, int64_t in_row, int64_t out_row,
                                           int64_t tok0, int len)
{
    const int W = cv.width - 1;
    if (!cv.state_out || W <= 0)
        return;
    uint4 r[kMaxConvWidth - 1];
#pragma unroll
    for (int j = 0; j < kMaxConvWidth - 1; ++j) {
        r[j] = make_uint4(0, 0, 0, 0);
        if (j < W) {
            const int pos = len - W + j;   // relative to the first token
            if (pos >= 0)
                r[j] = *reinterpret_cast<const uint4 *>(conv_src(q, k, v, in, hk, c, tok0 + pos));
            else if (cv.state_in)
                r[j] = *reinterpret_cast<const uint4 *>(cv.state_in + ((in_row * W + (W + pos)) * cv.channels + c));
        }
    }
#pragma unroll
    for (int j = 0; j < kMaxConvWidth - 1; ++j)
        if (j < W)
            *reinterpret_cast<uint4 *>(cv.state_out + ((out_row * W + j) * cv.channels + c)) = r[j];
}

}  // namespace gdn
