// kernels.h -- internal launcher interface between the C-ABI layer
// (gdn_api.cu) and the kernel translation units.  Not installed; the public
// boundary is include/gdn.h.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace gdn {

struct DecodeArgs {
    int batch, hk, hv;
    const void *q, *k, *v, *a, *b;
    const float *A_log, *dt_bias;
    float *state;
    const void *z, *norm_w;
    float eps;
    void *out;
    uint32_t *status;
};

struct PrefillArgs {
    int num_seqs, total_tokens, hk, hv;
    int max_chunks;                // upper bound on chunks: ceil(T/64) + N
    const void *q, *k, *v, *a, *b;
    const float *A_log, *dt_bias;
    const float *init_state;
    const int32_t *cu_seqlens;
    const void *z, *norm_w;
    float eps;
    void *out;
    float *final_state;
    unsigned char *workspace;
    uint32_t *status;
};

// Workspace layout of the chunked prefill (all offsets 1024-byte aligned).
// Images are byte-exact shared-memory operand layouts (see tc05.cuh), fp16.
// Per (chunk, value head):  WQ   128x128, K-major 128B swizzle, two 64-wide K
//                                halves of 16 KB, 32 KB
//                           MT   128x64, K-major 128B swizzle, 16 KB
//                           V    [token 64][dv 32] x 4 value slices,
//                                MN-major 64B swizzle, 4 KB each, 16 KB
//                           scal fp32: [0,64) state-update row scales
//                                e^{G_last - G_i}, [64] e^{G_last}, 1 KB
// Per (chunk, key head):    Kn   L2-normalised keys [token 64][dk 128],
//                                MN-major 128B swizzle, dk halves of 8 KB
constexpr size_t kWQBytes = 32768;
constexpr size_t kMTBytes = 16384;
constexpr size_t kVBytes = 16384;
constexpr size_t kScalBytes = 1024;
constexpr size_t kPerVHead = kWQBytes + kMTBytes + kVBytes + kScalBytes;  // 66560
constexpr size_t kKBytes = 16384;

inline int prefill_max_chunks(int num_seqs, int total_tokens)
{
    return (total_tokens + 63) / 64 + num_seqs;
}
inline size_t prefill_workspace_bytes(int num_seqs, int total_tokens, int hk, int hv)
{
    if (total_tokens <= 0)
        return 0;
    const size_t c = (size_t)prefill_max_chunks(num_seqs, total_tokens);
    return c * (size_t)hv * kPerVHead + c * (size_t)hk * kKBytes;
}

cudaError_t launch_decode(const DecodeArgs &args, cudaStream_t stream);
cudaError_t launch_prefill(const PrefillArgs &args, cudaStream_t stream);

}  // namespace gdn
