// gdn_noalloc.cu -- gdn_prefill for callers that cannot allocate device
// memory: some hosts hand a kernel only their own pre-registered input and
// output buffers and forbid device allocation once they are running (a
// cudaMalloc synchronises the device and can fragment a pool sized at
// start-up), and some plain-C callers carry no device allocator at all.  This
// entry point runs the same chunked prefill with its scratch in a fixed array
// that the library itself holds in device memory.
//
// The array is file-scope and static: every GPU that loads the library keeps
// kNoAllocScratchBytes of device memory for it until the process exits.  In
// host code its name is only a host-side stand-in, never a device address;
// the device address comes from cudaGetSymbolAddress, looked up once per
// device (with that device current) on the first call made on it.
#include <atomic>

#include <cuda_runtime.h>

#include "../../include/gdn.h"
#include "kernels.h"

namespace {

// 64 MiB.  The workspace takes one record per (64-token chunk, value head)
// for ceil(T/64) + N chunks, plus the chunk index, so at Hv = 32 this covers
// ceil(T/64) + N <= 14 (one sequence of up to 832 tokens).  The extra 1 KB
// lets the base be rounded up to the 1024-byte alignment gdn_prefill requires.
constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes + 1024];

// Device address of g_noalloc_scratch, per device.  Two host threads making
// their first call on one device at the same time both look it up and store
// the same value; the atomic keeps that race well defined.
std::atomic<void *> g_scratch_ptr[gdn::kMaxDevices];

}  // namespace

extern "C" gdn_status_t gdn_prefill_noalloc(const gdn_shape_t *s, const void *q, const void *k,
                                            const void *v, const void *a, const void *b,
                                            const float *A_log, const float *dt_bias,
                                            const float *init_state, const int32_t *cu_seqlens,
                                            const void *z, const void *norm_w, float eps,
                                            void *out, float *final_state, void *stream)
{
    const size_t need = gdn_prefill_workspace_bytes(s);
    if (need > kNoAllocScratchBytes)
        return GDN_ERR_WORKSPACE;   // the problem is larger than the built-in scratch
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= gdn::kMaxDevices)
        return GDN_ERR_CUDA;
    void *ptr = g_scratch_ptr[dev].load(std::memory_order_relaxed);
    if (!ptr) {
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr)
            return GDN_ERR_CUDA;
        g_scratch_ptr[dev].store(ptr, std::memory_order_relaxed);
    }
    uintptr_t base = reinterpret_cast<uintptr_t>(ptr);
    base = (base + 1023) & ~uintptr_t(1023);
    return gdn_prefill(s, q, k, v, a, b, A_log, dt_bias, init_state, cu_seqlens, z, norm_w, eps,
                       out, final_state, reinterpret_cast<void *>(base), kNoAllocScratchBytes, stream);
}
