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
// Per (chunk, value head) one 89 KB record of fp16 byte-exact shared-memory
// operand images (see tc05.cuh), in the order the scan kernel stages them:
//   Mc  128x128  state-to-state map -Kn^T diag(eps) W, K-major 128B swizzle,
//                two 64-wide K halves of 16 KB (at 0 and 24 KB)
//   Qc   64x128  state-to-output map diag(Gam r_q) Q - R, K-major, two K
//                halves of 8 KB (at 16 KB and 40 KB, each directly after a
//                Mc half, so a 128-row operand starting 8 KB earlier has
//                Qc as rows 64-127)
//   Ec  128x64   value-to-state map Kn^T diag(eps) T diag(beta), K-major (48 KB)
//   Fc   64x64   value-to-output map P T diag(beta), K-major (64 KB, after Ec)
//   V   [token 64][dv 32] x 4 value slices, MN-major 64B swizzle (72 KB)
//   scal fp32 e^{G_last} (88 KB)
// with eps_i = e^{G_last - G_i} for the chunk's valid rows, 0 past them.
constexpr size_t kWsMc0 = 0, kWsQc0 = 16384, kWsMc1 = 24576, kWsQc1 = 40960;
constexpr size_t kWsEc = 49152, kWsFc = 65536;
constexpr size_t kOpsBytes = 73728;          // Mc, Qc, Ec, Fc
constexpr size_t kWsV = 73728;
constexpr size_t kVBytes = 16384;
constexpr size_t kWsScal = 90112;
constexpr size_t kPerVHead = 91136;

inline int prefill_max_chunks(int num_seqs, int total_tokens)
{
    return (total_tokens + 63) / 64 + num_seqs;
}
inline size_t prefill_workspace_bytes(int num_seqs, int total_tokens, int hk, int hv)
{
    (void)hk;
    if (total_tokens <= 0)
        return 0;
    const size_t c = (size_t)prefill_max_chunks(num_seqs, total_tokens);
    return c * (size_t)hv * kPerVHead;
}

cudaError_t launch_decode(const DecodeArgs &args, cudaStream_t stream);
cudaError_t launch_prefill(const PrefillArgs &args, cudaStream_t stream);

}  // namespace gdn
