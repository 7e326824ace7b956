// gdn_prefill_scan.cu -- serial half of the chunked GDN prefill: the fp32
// inter-chunk state scan (JevAny page "Add opt-in fused Qwen3.5 inference
// kernels", Summary: chunked kernel; pegainfer page "feat(qwen35): add SM120
// FlashInfer GDN prefill candidate", Correctness: chunked vs unchunked
// prefill, initial/final states).
//
// A chain is one (sequence, value head, 32-column slice of Dv): the
// recurrence is independent per value column, so the four slices of a head
// run in parallel with no communication.  The grid is persistent: each CTA
// runs chains one after another (all of them at once when there are no more
// chains than CTAs), and its loader streams the stages across chain
// boundaries, so a batch of many short sequences pays the pipeline's start-up
// once per CTA instead of once per chain.
//
// The prep kernel turns each chunk into an affine map of the state (S is the
// fp32 slice, 128 x 32):
//   S' = e^{G_last} S + Mc S + Bc
// with Mc an fp16 tcgen05 operand (M = 128) and Bc, the value input, added
// by the state threads.  The serial chain per chunk is S (fp16 operand) ->
// 8 MMAs -> TMEM -> S' in registers; the state threads touch no global
// memory inside it.  Each chunk's fp16 S operand is also copied to the
// workspace, where the output kernel, fully parallel over chunks, turns it
// into the chunk's outputs.
//
// Roles (11 warps):
//   warps 0-7   state: warp w holds TMEM lane quadrant w % 4 = state rows
//               32 (w % 4) .. +31 and value columns 16 (w / 4) .. +15
//   warps 8, 10 issue the MMAs of the first and second 64-row K half of the
//               state into two accumulators (issuing them is the chain's
//               largest cost, and two issuing threads overlap it), which the
//               state threads add; warp 8 also copies S to the workspace
//   warp 9      issues the stage copies (Mc, the chain's Bc slice,
//               e^{G_last}) for every chunk of every chain of the CTA, then
//               rolls the chains' share of the carried conv states
// One CTA per SM with four stages (copies run well ahead of the chain); with
// more chains than CTAs, each CTA runs its share in turn, the next chain's
// initial state loaded while the current one runs.
#include <atomic>

#include "chunks.cuh"
#include "common.cuh"
#include "conv.cuh"
#include "kernels.h"
#include "tc05.cuh"

namespace gdn {


namespace {

constexpr int kThreads = 11 * 32;
constexpr int kStateWarps = 8;
constexpr int kIssuerWarp = 8;
constexpr int kLoaderWarp = 9;
constexpr int kIssuer2Warp = 10;   // the second K half's MMAs
// Named barrier (id, participating threads): state warps arrive, the issuer syncs.
constexpr uint32_t kBarS = 1, kCntS = kStateWarps * 32 + 64;   // S operand written
constexpr int kNv = 32;                 // value columns per CTA
constexpr int kTiles = kD / kNv;        // 4 CTAs per (sequence, head)
constexpr int kCols = 16;               // value columns per thread

// Stage: the chunk's Mc (the first 32 KB of its record), this CTA's Bc slice
// and e^{G_last}.
constexpr uint32_t kStBc = 32768, kStScal = 40960;
constexpr uint32_t kStageBytes = 41984;
constexpr uint32_t kLoadBytes = 32768 + 8192 + 16;

// TMEM columns: chain accumulators at 0 / 32.
constexpr uint32_t kTmemCols = 128;
constexpr uint32_t kAccHalf = 64;   // the second K half's accumulators

// NS stages of copies ahead of the chain (four: one CTA per SM).
template <int NS>
struct SmallT {
    uint64_t full[NS];          // stage landed (one arrival + bytes)
    uint64_t sfree[NS];         // stage read: the MMAs (one commit) and the eight state warps
    uint64_t bar_chain;
    uint32_t tmem_base;
    int fail;
};
template <int NS>
struct ScanCfg {
    static constexpr uint32_t kOffS = NS * kStageBytes;   // two S operands [dk][32] fp16, MN-major, 8 KB each
    static constexpr uint32_t kOffSmall = kOffS + 16384;
    static constexpr uint32_t kSmemBytes = kOffSmall + ((sizeof(SmallT<NS>) + 127) / 128) * 128 + 1024;
};

template <class Small>
__device__ __forceinline__ bool failed(Small *s) { return *reinterpret_cast<volatile int *>(&s->fail) != 0; }

template <class Small>
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

// Wait that first tests without suspending: a phase that has already
// completed costs one test.  Spins a little before suspending, for waits on
// the state chain where the wake-up delay would add to every chunk.
template <class Small>
__device__ __forceinline__ bool wait_quick(Small *s, uint64_t *bar, uint32_t parity, uint32_t *status, int spins)
{
    for (int i = 0; i < spins; ++i)
        if (mbar_test(bar, parity))
            return true;
    return wait_bar(s, bar, parity, status);
}

// Descriptors of the stage operands (shared-memory byte address `st`).
__device__ __forceinline__ uint64_t desc_k128(uint32_t addr) { return make_desc(addr, 16, 1024, kSw128); }

// D = Mc S over one 64-wide K half of the state (4 MMAs).
__device__ __forceinline__ void issue_mcs(uint32_t d, uint32_t st, uint64_t ds, uint32_t idesc, int half)
{
    const uint64_t a = desc_k128(st + (uint32_t)(half ? kWsMc1 : kWsMc0));
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
        mma_f16(d, a + (uint64_t)(kk * 2), ds + (uint64_t)((4 * half + kk) * 64), idesc, kk != 0);
}

// Chain i: (sequence n, value head h, slice r), sequence-major.
struct Chain {
    int n, h, r;
    int cbase, tok0, len, nck;
};
__device__ __forceinline__ Chain chain_at(const PrefillArgs &p, int i)
{
    Chain c;
    c.n = i / (p.hv * kTiles);
    const int rem = i - c.n * p.hv * kTiles;
    c.h = rem / kTiles;
    c.r = rem - c.h * kTiles;
    c.cbase = chunks_before(p, c.n, c.tok0, c.len);
    c.nck = (c.len + kC - 1) / kC;
    return c;
}

template <int NS>
__global__ void __launch_bounds__(kThreads, NS >= 4 ? 1 : 2)
scan_kernel(PrefillArgs p)
{
    constexpr int kStages = NS;
    constexpr uint32_t kOffS = ScanCfg<NS>::kOffS, kOffSmall = ScanCfg<NS>::kOffSmall;
    using Small = SmallT<NS>;
    const int hv = p.hv;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nchains = p.num_seqs * hv * kTiles;
    const int first = blockIdx.x, stride = gridDim.x;

    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Small *s = reinterpret_cast<Small *>(sm + kOffSmall);
    const uint32_t sbase = smem_u32(sm);
    auto record = [&](const Chain &c, int k) {
        return p.workspace + ((size_t)(c.cbase + k) * hv + c.h) * kPerVHead;
    };

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&s->full[i], 1);
            mbar_init(&s->sfree[i], kStateWarps + 2);
        }
        mbar_init(&s->bar_chain, 2);
        mbar_fence_init();
        s->fail = 0;
    }
    if (warp == 0) {
        tmem_alloc(&s->tmem_base, kTmemCols);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    // launched early behind the prep kernel: its records are read below
    grid_dep_wait();
    // the output kernel may be scheduled now (its CTAs take the SMs no chain
    // uses and fetch their z tiles); it waits for this grid's end to read S
    grid_dep_launch();
    const uint32_t tbase = s->tmem_base;
    const uint32_t idesc = make_idesc_f16(128, kNv, false, true);

    if (warp == kIssuerWarp || warp == kIssuer2Warp) {
        // ----------------------------------------------------------- issuers
        // each issues one K half's MMAs into its own accumulator; the first
        // also copies S to the workspace.  g counts this CTA's chunks over
        // all its chains: it picks the stage, the buffers and the parities.
        const int half = warp == kIssuer2Warp;
        uint32_t g = 0;
        for (int i = first; i < nchains; i += stride) {
            const Chain ch = chain_at(p, i);
            for (int c = 0; c < ch.nck; ++c, ++g) {
                const int b = g & 1, st = g % kStages;   // S operand and accumulator buffer; stage
                const uint32_t sst = sbase + st * kStageBytes;
                const uint32_t dS = tbase + half * kAccHalf + b * kNv;
                bool ok = true;
                if (lane == 0) {
                    // the copy of the previous S has read its buffer before this
                    // chunk's chain releases the state warps to write the next S there
                    if (!half)
                        bulk_wait_read<0>();
                    ok = wait_quick(s, &s->full[st], (g / kStages) & 1, p.status, 1);
                }
                __syncwarp();
                named_sync(kBarS, kCntS);            // S(c) operand written
                if (lane == 0) {
                    if (ok && !failed(s)) {
                        tc_fence_after();
                        issue_mcs(dS, sst, make_desc(sbase + kOffS + b * 8192, 512, 512, kSw64), idesc, half);
                    }
                    mma_commit(&s->bar_chain);
                    mma_commit(&s->sfree[st]);
                    // S(c) -> workspace, for the output kernel
                    if (!half)
                        bulk_s2g(record(ch, c) + kWsS + ch.r * 8192, sm + kOffS + b * 8192, 8192);
                }
                __syncwarp();
            }
        }
        if (lane == 0 && !half)
            bulk_wait_all();   // every S copy complete before exit (the output kernel reads them)
        __syncwarp();
    } else if (warp == kLoaderWarp) {
        // ------------------------------------------------------------ loader
        int issued[kStages] = {};
        if (lane == 0) {
            uint32_t g = 0;
            for (int i = first; i < nchains && !failed(s); i += stride) {
                const Chain ch = chain_at(p, i);
                for (int c = 0; c < ch.nck; ++c, ++g) {
                    const int st = g % kStages;
                    // step g goes into the stage step g - NS used, once its MMAs
                    // and the state warps have read it
                    if (g >= (uint32_t)kStages && !wait_bar(s, &s->sfree[st], (g / kStages - 1) & 1, p.status))
                        break;
                    unsigned char *stage = sm + st * kStageBytes;
                    const unsigned char *rec = record(ch, c);
                    mbar_arrive_expect_tx(&s->full[st], kLoadBytes);
                    bulk_g2s(stage, rec, 16384, &s->full[st]);
                    bulk_g2s(stage + 16384, rec + 16384, 16384, &s->full[st]);
                    bulk_g2s(stage + kStBc, rec + kWsBc + ch.r * 8192, 8192, &s->full[st]);
                    bulk_g2s(stage + kStScal, rec + kWsScal, 16, &s->full[st]);
                    ++issued[st];
                }
            }
            // no copy may still be landing in shared memory when the CTA exits
            if (failed(s)) {
                for (int qq = 0; qq < kStages; ++qq)
                    if (issued[qq] > 0)
                        mbar_wait(&s->full[qq], (uint32_t)(issued[qq] - 1) & 1);
            }
        }
        __syncwarp();
        // The carried conv states.  Every prep CTA has read the old ones (the
        // dependency wait above), so they may be rewritten in place.  Each
        // chain rolls its value slice of head h and, for the first value head
        // of a group, the same slice of q and k head h / group.
        if (p.conv.width > 1 && p.conv.state_out) {
            for (int i = first; i < nchains; i += stride) {
                const int n = i / (hv * kTiles), rem = i - n * hv * kTiles, h = rem / kTiles,
                          r = rem - h * kTiles;
                int tok0 = 0, len = 0;
                chunks_before(p, n, tok0, len);
                const int grp = hv / p.hk, hq = h / grp;
                if (lane < (h % grp == 0 ? 12 : 4)) {
                    const int part = lane >> 2, c = r * kNv + (lane & 3) * 8;
                    const int chan = part == 0 ? (2 * p.hk + h) * kD + c
                                   : part == 1 ? hq * kD + c : (p.hk + hq) * kD + c;
                    conv_roll8(p.conv, p.conv.x_q, p.conv.x_k, p.conv.x_v, p.conv.x_in, p.hk, chan, n, n, tok0, len);
                }
            }
        }
    } else {
        // ------------------------------------------------------------ state
        const int q = warp & 3, cg = warp >> 2;
        const int row = 32 * q + lane;     // TMEM lane = state row (dk)
        const uint32_t tlane = tbase + ((uint32_t)(32 * q) << 16) + cg * kCols;
        float S[kCols];
        bool over = false;   // a state value left the fp16 operand range
        // S -> fp16 operand buffer b
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
        // this thread's part of chain i's state, at element offset sidx(i)
        auto sidx_of = [&](const Chain &c) {
            return (((size_t)c.n * hv + c.h) * kD + row) * kD + c.r * kNv + cg * kCols;
        };
        // the next chain's initial state is loaded while the current chain
        // runs, so a CTA with many short chains does not wait for it between them
        float4 nxt[kCols / 4];
        auto load_init = [&](int i) {
#pragma unroll
            for (int j = 0; j < kCols / 4; ++j)
                nxt[j] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (p.init_state && i < nchains) {
                const size_t o = sidx_of(chain_at(p, i));
#pragma unroll
                for (int j = 0; j < kCols / 4; ++j)
                    nxt[j] = reinterpret_cast<const float4 *>(p.init_state + o)[j];
            }
        };
        load_init(first);
        uint32_t g = 0;
        for (int i = first; i < nchains; i += stride) {
            const Chain ch = chain_at(p, i);
            if (tid == 0 && ch.h == 0 && ch.r == 0 && !seq_ok(p, p.cu_seqlens[ch.n], p.cu_seqlens[ch.n + 1]))
                set_status(p.status, kStatusBadSeqlens);   // treated as empty: final state = initial state
            const size_t sidx = sidx_of(ch);
#pragma unroll
            for (int j = 0; j < kCols / 4; ++j) {
                S[4 * j] = nxt[j].x; S[4 * j + 1] = nxt[j].y; S[4 * j + 2] = nxt[j].z; S[4 * j + 3] = nxt[j].w;
            }
            load_init(i + stride);
            const int nck = ch.nck;
            if (nck > 0)
                put_state(g & 1);
            for (int c = 0; c < nck; ++c, ++g) {
                const int st = g % kStages;
                const unsigned char *stage = sm + st * kStageBytes;
                wait_quick(s, &s->full[st], (g / kStages) & 1, p.status, 1);   // Bc, e^{G_last} visible
                wait_quick(s, &s->bar_chain, g & 1, p.status, 256);
                __syncwarp();   // converged for the .aligned TMEM load
                tc_fence_after();
                float dv[kCols];
                tmem_ld16_sum2(tlane + (g & 1) * kNv, tlane + kAccHalf + (g & 1) * kNv, dv);
                const float eg = *reinterpret_cast<const float *>(stage + kStScal);
                uint4 bc[2];
                bc[0] = *reinterpret_cast<const uint4 *>(stage + kStBc + sw64_chunk_offset(row, 2 * cg));
                bc[1] = *reinterpret_cast<const uint4 *>(stage + kStBc + sw64_chunk_offset(row, 2 * cg + 1));
                const __half2 *hp = reinterpret_cast<const __half2 *>(bc);
#pragma unroll
                for (int j = 0; j < kCols / 2; ++j) {
                    const float2 f2 = __half22float2(hp[j]);
                    S[2 * j] = fmaf(eg, S[2 * j], dv[2 * j] + f2.x);
                    S[2 * j + 1] = fmaf(eg, S[2 * j + 1], dv[2 * j + 1] + f2.y);
                }
                // The loader refills this stage by TMA (the async proxy) once it is
                // free: the generic reads of Bc and e^{G_last} above are ordered
                // before that write only by a proxy fence, not by the mbarrier.
                // Without it, with two CTAs per SM, a refill now and then landed
                // under these reads and S(c+1) took chunk c+2's Bc.  put_state's
                // fence serves both its S writes and these reads, and the stage
                // is released after it, off the chain.
                if (c + 1 < nck)
                    put_state((g + 1) & 1);
                else
                    fence_async_smem();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&s->sfree[st]);
                __syncwarp();
            }
#pragma unroll
            for (int j = 0; j < kCols / 4; ++j)
                reinterpret_cast<float4 *>(p.final_state + sidx)[j] = make_float4(S[4 * j], S[4 * j + 1], S[4 * j + 2], S[4 * j + 3]);
        }
        if (over)
            set_status(p.status, kStatusRange);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tbase, kTmemCols);
    }
}

}  // namespace

namespace {

template <int NS>
cudaError_t launch_stages(const PrefillArgs &p, int resident, cudaStream_t stream)
{
    const int64_t chains = (int64_t)p.num_seqs * p.hv * kTiles;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(chains < resident ? chains : resident));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = ScanCfg<NS>::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, scan_kernel<NS>, p);
}

}  // namespace

namespace {
// CTAs of scan_kernel<NS> that fit on the device at once, per device.
template <int NS>
cudaError_t resident_ctas(int &out)
{
    static std::atomic<int> cache[kMaxDevices];   // a racing repeat stores the same value
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    int n = cache[dev].load(std::memory_order_relaxed);
    if (!n) {
        e = cudaFuncSetAttribute(scan_kernel<NS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)ScanCfg<NS>::kSmemBytes);
        int sms = 0, per_sm = 0;
        if (e == cudaSuccess)
            e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, scan_kernel<NS>, kThreads,
                                                              ScanCfg<NS>::kSmemBytes);
        if (e != cudaSuccess)
            return e;
        n = sms * (per_sm > 0 ? per_sm : 1);
        cache[dev].store(n, std::memory_order_relaxed);
    }
    out = n;
    return cudaSuccess;
}
}  // namespace

cudaError_t launch_prefill_scan(const PrefillArgs &p, cudaStream_t stream)
{
    // One CTA per chain while they all fit at once; past that, every CTA
    // that fits, each running its share of the chains in turn.  (Two stages
    // at two CTAs per SM measured slower on many short chains: each chunk
    // then waits on its copies.)
    int resident = 0;
    cudaError_t e = resident_ctas<4>(resident);
    if (e != cudaSuccess)
        return e;
    return launch_stages<4>(p, resident, stream);
}

}  // namespace gdn
