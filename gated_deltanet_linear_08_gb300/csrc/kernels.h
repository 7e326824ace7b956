// kernels.h -- internal launcher interface between the C-ABI layer
// (gdn_api.cu) and the kernel translation units.  Not installed; the public
// boundary is include/gdn.h.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace gdn {

// Devices one process may drive: the size of the per-device caches (device
// addresses, resident CTA counts).
constexpr int kMaxDevices = 64;

// Element strides of one token input: between consecutive tokens and
// between consecutive heads (rows of 128 elements for q, k, v, z; one element
// for a, b).
struct Stride {
    int64_t t, h;
};
struct InputStrides {
    Stride q, k, v, z, a, b;
};

// Causal conv1d + SiLU over the q | k | v channels ahead of the core
// (width 0: none).  state_in / state_out: bf16 [rows][width-1][channels].
// x_q, x_k, x_v / x_in: the raw token inputs the conv reads (and the state
// roll copies); for prefill the core then reads the conv output y instead.
struct ConvArgs {
    int width;
    int channels;               // Hk*128 + Hk*128 + Hv*128
    const __nv_bfloat16 *weight;   // [channels][width]
    const __nv_bfloat16 *state_in;
    __nv_bfloat16 *state_out;
    const void *x_q, *x_k, *x_v;
    InputStrides x_in;
    __nv_bfloat16 *y;           // prefill: conv output [tokens][channels]
};

struct DecodeArgs {
    int batch, hk, hv;
    int tokens;                    // consecutive tokens per sequence (1..8)
    int num_slots;                 // slots in the state pool
    const int32_t *state_idx;      // slot per sequence, or null for slot n
    InputStrides in;
    ConvArgs conv;
    const void *q, *k, *v, *a, *b;
    const float *A_log, *dt_bias;
    float *state;                  // state pool [num_slots, hv, 128, 128]
    const void *z, *norm_w;
    float eps;
    void *out;
    uint32_t *status;
};

struct PrefillArgs {
    int num_seqs, total_tokens, hk, hv;
    int max_chunks;                // upper bound on chunks: ceil(T/64) + N
    InputStrides in;
    ConvArgs conv;
    const void *q, *k, *v, *a, *b;
    const float *A_log, *dt_bias;
    const float *init_state;
    const int32_t *cu_seqlens;
    const int32_t *chunk_off;      // [N+1] chunks before sequence n, or null (walk cu_seqlens)
    const void *z, *norm_w;
    float eps;
    void *out;
    float *final_state;
    unsigned char *workspace;
    uint32_t *status;
    int single_chunk;              // set by launch_prefill: prep finishes the call (see there)
};

// Workspace layout of the chunked prefill (all offsets 1024-byte aligned).
// Per (chunk, value head) one 137 KB record, ordered so that the scan kernel
// copies its operand (Mc) and the output kernel its operands (Qc, Fc, V, S)
// each as one contiguous run.  Images are fp16 byte-exact shared-memory
// operand layouts (see tc05.cuh):
//   Mc  128x128  state-to-state map -Kn^T diag(eps) W, K-major 128B swizzle,
//                two 64-wide K halves of 16 KB                         [0, 32K)
//   Bc  [slice 4][dk 128][dv 32] fp16 in 64-byte-swizzled rows: the
//       chunk's value input to the state, Kn^T diag(eps) T diag(beta) V,
//       added by the scan's state threads                              [32K, 64K)
//   Qc   64x128  state-to-output map diag(Gam r_q) Q - R, two K halves
//                of 8 KB                                               [64K, 80K)
//   Fc   64x64   value-to-output map P T diag(beta)                    [80K, 88K)
//   V   [token 64][dv 32] x 4 value slices, MN-major 64B swizzle       [88K, 104K)
//   S   [dk 128][dv 32] x 4 value slices: the fp16 state entering the
//       chunk, written by the scan kernel, MN-major 64B swizzle        [104K, 136K)
//   scal fp32 e^{G_last}                                               [136K]
// with eps_i = e^{G_last - G_i} for the chunk's valid rows, 0 past them.
constexpr size_t kWsMc0 = 0, kWsMc1 = 16384, kWsBc = 32768;
constexpr size_t kWsQc0 = 65536, kWsQc1 = 73728, kWsFc = 81920;
constexpr size_t kWsV = 90112, kWsS = 106496, kWsScal = 139264;
constexpr size_t kVBytes = 16384, kSBytes = 32768;
constexpr size_t kPerVHead = 140288;

inline int prefill_max_chunks(int num_seqs, int total_tokens)
{
    return (total_tokens + 63) / 64 + num_seqs;
}
// From this many sequences on, a one-CTA kernel builds the chunk index
// (chunks before each sequence) ahead of prep; below it, walking cu_seqlens
// is cheaper than the launch.
constexpr int kIndexMinSeqs = 16;
// The workspace: the records, then the chunk index (int32 [N+1], 1 KB
// aligned), then (with the conv) the conv output.
inline size_t prefill_index_offset(int num_seqs, int total_tokens, int hv)
{
    return (size_t)prefill_max_chunks(num_seqs, total_tokens) * (size_t)hv * kPerVHead;
}
inline size_t prefill_workspace_bytes(int num_seqs, int total_tokens, int hk, int hv)
{
    (void)hk;
    if (total_tokens <= 0)
        return 0;
    const size_t idx = ((size_t)(num_seqs + 1) * 4 + 1023) & ~size_t(1023);
    return prefill_index_offset(num_seqs, total_tokens, hv) + idx;
}

// With the conv, the prefill workspace also holds its output y, bf16
// [tokens][channels], after the records.
inline size_t prefill_conv_bytes(int total_tokens, int hk, int hv)
{
    const size_t b = (size_t)(total_tokens > 0 ? total_tokens : 0) * (size_t)(2 * hk + hv) * 128 * 2;
    return (b + 1023) & ~size_t(1023);
}

// Tensor map over a bf16 tensor of `tokens` x `heads` rows of 128 elements,
// `st` elements between tokens and `sh` between heads (multiples of 8): boxes
// of 64 tokens x 64 elements of one head, 128-byte swizzled in shared memory,
// zero fill past the last token.  Host only; false if the driver's encoder is
// unavailable or rejects the tensor.
bool encode_tile_map(CUtensorMap *map, const void *base, int heads, int tokens, int64_t st, int64_t sh);

cudaError_t launch_decode(const DecodeArgs &args, cudaStream_t stream);
// The chunked prefill runs three kernels in stream order: prep (chunk-parallel
// maps), scan (serial state chain, one CTA per sequence, head and Dv slice)
// and out (chunk-parallel outputs and epilogue).
cudaError_t launch_prefill_prep(const PrefillArgs &args, cudaStream_t stream);
cudaError_t launch_prefill_scan(const PrefillArgs &args, cudaStream_t stream);
cudaError_t launch_prefill_out(const PrefillArgs &args, cudaStream_t stream);
// The conv ahead of the prefill core: y = silu(conv(x)) for every token into
// args.conv.y, in stream order before prep (which then reads y through
// args.q/k/v); also the whole of gdn_conv_prefill.
cudaError_t launch_prefill_conv(const PrefillArgs &args, cudaStream_t stream);
// The chunk index args.chunk_off (when set), built before the other kernels.
cudaError_t launch_chunk_index(const PrefillArgs &args, cudaStream_t stream);
inline cudaError_t launch_prefill(const PrefillArgs &args, cudaStream_t stream)
{
    if (args.num_seqs == 0)
        return cudaSuccess;
    if (args.chunk_off) {
        cudaError_t e = launch_chunk_index(args, stream);
        if (e != cudaSuccess)
            return e;
    }
    if (args.total_tokens > 0 && args.conv.width > 0) {
        cudaError_t e = launch_prefill_conv(args, stream);
        if (e != cudaSuccess)
            return e;
    }
    // Every sequence within one chunk (64 tokens or fewer in all), a zero
    // initial state and no conv: the state entering each chunk is zero, so
    // prep computes the outputs and final states itself and the scan and
    // output kernels do not run.
    const bool single = args.total_tokens > 0 && args.total_tokens <= 64 && !args.init_state
                        && args.conv.width == 0;
    if (args.total_tokens > 0) {
        PrefillArgs a = args;
        a.single_chunk = single ? 1 : 0;
        cudaError_t e = launch_prefill_prep(a, stream);
        if (e != cudaSuccess || single)
            return e;
    }
    cudaError_t e = launch_prefill_scan(args, stream);
    if (e != cudaSuccess || args.total_tokens == 0)
        return e;
    return launch_prefill_out(args, stream);
}

}  // namespace gdn
