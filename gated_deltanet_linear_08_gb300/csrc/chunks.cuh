// chunks.cuh -- chunk bookkeeping of the packed prefill, shared by its kernels.
//
// Sequence n owns ceil(len_n / 64) chunks, numbered consecutively in sequence
// order (pegainfer page "feat(qwen35): add SM120 FlashInfer GDN prefill
// candidate", Correctness: packed varlen prefill, chunk boundaries).  A
// malformed sequence (decreasing cu_seqlens, or outside [0, T]) owns none and
// is flagged.  With many sequences the chunk index (chunk_off[n] = chunks
// before sequence n, n = 0..N, built once per call by a one-CTA kernel) turns
// every lookup into a binary search or a single load; with few, a walk over
// cu_seqlens is cheaper than the extra launch.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace gdn {

__device__ __forceinline__ bool seq_ok(const PrefillArgs &p, int s, int e)
{
    return !(s < 0 || e < s || e > p.total_tokens);
}

// Global chunk gc: its sequence, first token and valid rows; false when gc
// lies past the last chunk.  `bad` reports a malformed sequence met on the walk.
__device__ __forceinline__ bool find_chunk(const PrefillArgs &p, int gc, int &n, int &tok0, int &L, bool &bad)
{
    bad = false;
    if (p.chunk_off) {
        int lo = 0, hi = p.num_seqs;   // the last n with chunk_off[n] <= gc
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (p.chunk_off[mid] <= gc)
                lo = mid;
            else
                hi = mid - 1;
        }
        if (lo >= p.num_seqs)
            return false;
        n = lo;
        const int s = p.cu_seqlens[n], e = p.cu_seqlens[n + 1];
        tok0 = s + (gc - p.chunk_off[n]) * kC;
        L = min(kC, e - tok0);
        return true;
    }
    int c = 0;
    for (int m = 0; m < p.num_seqs; ++m) {
        const int s = p.cu_seqlens[m], e = p.cu_seqlens[m + 1];
        if (!seq_ok(p, s, e)) {
            bad = true;
            continue;
        }
        const int nc = (e - s + kC - 1) / kC;
        if (gc < c + nc) {
            n = m;
            tok0 = s + (gc - c) * kC;
            L = min(kC, e - tok0);
            return true;
        }
        c += nc;
    }
    return false;
}

// Chunks before sequence n, its first token and its length (0 when malformed).
__device__ __forceinline__ int chunks_before(const PrefillArgs &p, int n, int &tok0, int &len)
{
    const int s = p.cu_seqlens[n], e = p.cu_seqlens[n + 1];
    const bool ok = seq_ok(p, s, e);
    tok0 = ok ? s : 0;
    len = ok ? e - s : 0;
    if (p.chunk_off)
        return p.chunk_off[n];
    int c = 0;
    for (int m = 0; m < n; ++m) {
        const int sm = p.cu_seqlens[m], em = p.cu_seqlens[m + 1];
        if (seq_ok(p, sm, em))
            c += (em - sm + kC - 1) / kC;
    }
    return c;
}

}  // namespace gdn
