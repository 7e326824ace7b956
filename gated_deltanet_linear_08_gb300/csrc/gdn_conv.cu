// gdn_conv.cu -- the causal conv1d + SiLU ahead of the prefill core, as its
// own HBM-bound pass (the definition and its rounding are in conv.cuh).
//
// Every token's q | k | v channels are read once and the bf16 result written
// once to the workspace, from where the prep kernel's tensor-map copies read
// it like any strided input.  One thread owns 4 channels (8 bytes) over a
// run of 8 consecutive tokens and keeps the window of the K-1 previous raw
// inputs in registers; a warp covers 128 contiguous channels of a token, so
// every load and store is a 256-byte coalesced row.  The per-element cost is
// four fp32 products and a SiLU (an exponential and a reciprocal on the
// special-function units, whose rate bounds the kernel next to HBM); small
// threads keep four CTAs per SM so loads and arithmetic overlap.  Every
// thread requests its run's rows and the K-1 rows before them before it looks
// up the sequence, and each CTA prefetches into L2 the rows of the CTA one
// resident wave later, so a CTA's loads mostly hit L2 while HBM streams the
// next wave.  A run that a sequence start crosses (or whose window does)
// instead resets the window from that sequence's carried state.  Grouped q
// and k heads are convolved once, not once per value head.
#include <atomic>

#include "common.cuh"
#include "conv.cuh"
#include "kernels.h"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kRun = 8;   // tokens per thread
constexpr int kCh = 4;    // channels per thread (one 8-byte vector)

// Sequence holding token t: the last n with cu[n] <= t (cu nondecreasing in
// a well-formed call; otherwise any n in range, which only ever reads
// in-bounds state rows).
__device__ __forceinline__ int seq_of(const int32_t *cu, int num_seqs, int t)
{
    int lo = 0, hi = num_seqs - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cu[mid] <= t)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

// The rows of the CTA `ahead` places later in launch order (about one wave
// of resident CTAs later) are prefetched into L2: 8 tokens x 16 lines of 128
// bytes (the CTA's 1024 channels, 8 heads of one of q, k, v), one line per
// thread of the first 128.
__device__ __forceinline__ void conv_prefetch_ahead(const PrefillArgs &p, int ahead)
{
    const ConvArgs &cv = p.conv;
    const int b = blockIdx.x + blockIdx.y * gridDim.x + ahead;
    if (ahead <= 0 || b >= gridDim.x * gridDim.y || threadIdx.x >= kRun * 16)
        return;
    const int bx = b % gridDim.x, by = b / gridDim.x;
    const int c = bx * kThreads * kCh + (threadIdx.x & 15) * 64;   // 64 channels per 128-byte line
    const int t = by * kRun + (threadIdx.x >> 4);
    if (c < cv.channels && t < p.total_tokens)
        asm volatile("prefetch.global.L2 [%0];" :: "l"(conv_src(cv.x_q, cv.x_k, cv.x_v, cv.x_in, p.hk, c, t)));
}

template <int KW>
__global__ void __launch_bounds__(kThreads, 4)
conv_prefill_kernel(PrefillArgs p, int ahead)
{
    const ConvArgs &cv = p.conv;
    conv_prefetch_ahead(p, ahead);
    const int c = (blockIdx.x * kThreads + threadIdx.x) * kCh;
    const int t0 = blockIdx.y * kRun;
    if (c >= cv.channels || t0 >= p.total_tokens)
        return;
    const int nt = min(kRun, p.total_tokens - t0);
    // this thread's channels: one input row per token at a fixed stride
    const __nv_bfloat16 *xb = conv_src(cv.x_q, cv.x_k, cv.x_v, cv.x_in, p.hk, c, 0);
    const int64_t xt = c < p.hk * kD ? cv.x_in.q.t : c < 2 * p.hk * kD ? cv.x_in.k.t : cv.x_in.v.t;
    __nv_bfloat16 *yb = cv.y + c;
    auto src = [&](int t) { return *reinterpret_cast<const uint2 *>(xb + (int64_t)t * xt); };

    // The run's rows and the K-1 rows before it are requested first, as if
    // one sequence held them all (the common case); the sequence lookup runs
    // under those loads.
    constexpr int kHist = KW > 1 ? KW - 1 : 1;
    uint2 raw[kRun], pre[kHist];
#pragma unroll
    for (int i = 0; i < kRun; ++i)
        if (i < nt)
            raw[i] = src(t0 + i);
#pragma unroll
    for (int j = 0; j < KW - 1; ++j) {
        const int pos = t0 - (KW - 1) + j;
        pre[j] = pos >= 0 ? src(pos) : make_uint2(0, 0);
    }
    float w[KW][kCh];
    conv_weights<kCh, KW>(cv.weight, c, w);

    int n = seq_of(p.cu_seqlens, p.num_seqs, t0);
    int s = p.cu_seqlens[n], e = p.cu_seqlens[n + 1];
    // a full run whose window lies inside one sequence too
    const bool fast = nt == kRun && t0 - (KW - 1) >= s && t0 + kRun <= e;

    // the K-1 raw inputs before position t of sequence n (which starts at s)
    float win[kHist][kCh];
    auto load_window = [&](int t) {
#pragma unroll
        for (int j = 0; j < KW - 1; ++j) {
            const int pos = t - (KW - 1) + j;
            uint2 u = make_uint2(0, 0);   // (bounds hold for malformed cu_seqlens too)
            if (pos >= s && pos >= 0)
                u = src(pos);
            else if (cv.state_in && pos < s && pos - s >= -(KW - 1))
                u = *reinterpret_cast<const uint2 *>(
                    cv.state_in + (((size_t)n * (KW - 1) + (KW - 1) + (pos - s)) * cv.channels + c));
            unpack4(u, win[j]);
        }
    };
    auto step = [&](const uint2 &u, int t) {
        float x[kCh], y[kCh];
        unpack4(u, x);
#pragma unroll
        for (int q = 0; q < kCh; ++q) {
            float acc = w[KW - 1][q] * x[q];
#pragma unroll
            for (int j = 0; j < KW - 1; ++j)
                acc = fmaf(w[j][q], win[j][q], acc);
            y[q] = silu_f(acc);
            if constexpr (KW > 1) {
#pragma unroll
                for (int j = 0; j + 1 < KW - 1; ++j)
                    win[j][q] = win[j + 1][q];
                win[KW - 2][q] = x[q];
            }
        }
        *reinterpret_cast<uint2 *>(yb + (size_t)t * cv.channels) = make_uint2(pack2(y[0], y[1]), pack2(y[2], y[3]));
    };

    if (fast) {
#pragma unroll
        for (int j = 0; j < KW - 1; ++j)
            unpack4(pre[j], win[j]);
#pragma unroll
        for (int i = 0; i < kRun; ++i)
            step(raw[i], t0 + i);
    } else {
        // a sequence starts inside the run or its window (or cu_seqlens do
        // not cover it)
        load_window(t0);
#pragma unroll 1
        for (int t = t0; t < t0 + nt; ++t) {
            if (t >= e) {
                while (n + 1 < p.num_seqs && p.cu_seqlens[n + 1] <= t)
                    ++n;
                s = p.cu_seqlens[n];
                e = p.cu_seqlens[n + 1];
                load_window(t);
            }
            step(src(t), t);
        }
    }
}

template <int KW>
cudaError_t launch_width(const PrefillArgs &p, cudaStream_t stream)
{
    // prefetch distance: the CTAs resident at once, once per device
    static std::atomic<int> resident[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    int ahead = resident[dev].load(std::memory_order_relaxed);
    if (!ahead) {
        int sms = 0, per_sm = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, conv_prefill_kernel<KW>, kThreads, 0);
        if (e != cudaSuccess)
            return e;
        ahead = sms * (per_sm > 0 ? per_sm : 1);
        resident[dev].store(ahead, std::memory_order_relaxed);
    }
    const dim3 grid((p.conv.channels / kCh + kThreads - 1) / kThreads, (p.total_tokens + kRun - 1) / kRun);
    conv_prefill_kernel<KW><<<grid, kThreads, 0, stream>>>(p, ahead);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_conv(const PrefillArgs &p, cudaStream_t stream)
{
    switch (p.conv.width) {
    case 1: return launch_width<1>(p, stream);
    case 2: return launch_width<2>(p, stream);
    case 3: return launch_width<3>(p, stream);
    case 4: return launch_width<4>(p, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace gdn
