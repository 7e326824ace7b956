// gdn_api.cu -- the C ABI of libgdn (include/gdn.h): host-side validation,
// status codes and dispatch onto the caller's stream.  Unsupported shapes are
// explicit errors returned before any launch, as the pegainfer review asks of
// a stable C ABI ("feat(qwen35): add SM120 FlashInfer GDN prefill
// candidate", maintainer review: unsupported shapes handled explicitly).
// Nothing here allocates device memory, prints, aborts or synchronises,
// except gdn_check_device_status, which is documented as off the hot path.
#include <cuda_runtime.h>

#include "../../include/gdn.h"
#include "kernels.h"

namespace {

// Status word the kernels OR bits into when a bounded wait runs out.
__device__ uint32_t g_device_status;

constexpr int kMaxDevices = 64;
uint32_t *g_status_ptr[kMaxDevices];   // device address of g_device_status, per device

uint32_t *status_ptr()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return nullptr;
    if (!g_status_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess)
            return nullptr;
        g_status_ptr[dev] = static_cast<uint32_t *>(p);
    }
    return g_status_ptr[dev];
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool overlaps(const void *a, size_t na, const void *b, size_t nb)
{
    if (!a || !b || na == 0 || nb == 0)
        return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

gdn_status_t check_shape(const gdn_shape_t *s)
{
    if (!s)
        return GDN_ERR_INVALID_ARG;
    if (s->num_seqs < 0 || s->total_tokens < 0 || s->hq <= 0 || s->hk <= 0 || s->hv <= 0
        || s->dk <= 0 || s->dv <= 0)
        return GDN_ERR_INVALID_ARG;
    if (s->dk != 128 || s->dv != 128 || s->hq != s->hk || s->hv % s->hk != 0)
        return GDN_ERR_UNSUPPORTED;
    if (s->hv > 65535 || s->num_seqs > 65535)
        return GDN_ERR_UNSUPPORTED;
    return GDN_OK;
}

}  // namespace

extern "C" {

const char *gdn_status_string(gdn_status_t status)
{
    switch (status) {
    case GDN_OK: return "GDN_OK";
    case GDN_ERR_INVALID_ARG: return "GDN_ERR_INVALID_ARG: null pointer, negative size or aliasing";
    case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED: needs Dk=Dv=128, Hq==Hk, Hv%Hk==0";
    case GDN_ERR_ALIGNMENT: return "GDN_ERR_ALIGNMENT: tensors need 16-byte, workspace 1024-byte alignment";
    case GDN_ERR_CUDA: return "GDN_ERR_CUDA: a CUDA call or kernel launch failed";
    case GDN_ERR_DEVICE_STATUS: return "GDN_ERR_DEVICE_STATUS: a kernel recorded an error";
    case GDN_ERR_WORKSPACE: return "GDN_ERR_WORKSPACE: workspace missing or too small";
    }
    return "GDN_ERR_UNKNOWN";
}

size_t gdn_prefill_workspace_bytes(const gdn_shape_t *s)
{
    if (check_shape(s) != GDN_OK)
        return 0;
    return gdn::prefill_workspace_bytes(s->num_seqs, s->total_tokens, s->hk, s->hv);
}

gdn_status_t gdn_prefill(const gdn_shape_t *s, const void *q, const void *k, const void *v,
                         const void *a, const void *b, const float *A_log, const float *dt_bias,
                         const float *init_state, const int32_t *cu_seqlens, const void *z,
                         const void *norm_w, float eps, void *out, float *final_state,
                         void *workspace, size_t workspace_bytes, void *stream)
{
    gdn_status_t st = check_shape(s);
    if (st != GDN_OK)
        return st;
    const size_t T = (size_t)s->total_tokens, N = (size_t)s->num_seqs;
    if (N == 0)
        return T == 0 ? GDN_OK : GDN_ERR_INVALID_ARG;
    if (!cu_seqlens || !A_log || !dt_bias || !final_state)
        return GDN_ERR_INVALID_ARG;
    if (T > 0 && (!q || !k || !v || !a || !b || !out))
        return GDN_ERR_INVALID_ARG;
    if (z && !norm_w)
        return GDN_ERR_INVALID_ARG;
    if (!(eps >= 0.f))
        return GDN_ERR_INVALID_ARG;
    const void *al16[] = {q, k, v, a, b, init_state, z, norm_w, out, final_state};
    for (const void *p : al16)
        if (p && !aligned(p, 16))
            return GDN_ERR_ALIGNMENT;
    // a, b rows are Hv bf16 wide: every row start need not be 16-byte aligned,
    // but the tensor base must be (checked above).
    const size_t need = gdn::prefill_workspace_bytes(s->num_seqs, s->total_tokens, s->hk, s->hv);
    if (need > 0 && (!workspace || workspace_bytes < need))
        return GDN_ERR_WORKSPACE;
    if (workspace && !aligned(workspace, 1024))
        return GDN_ERR_ALIGNMENT;
    const size_t hk = s->hk, hv = s->hv;
    const size_t out_b = T * hv * 128 * 2;
    const size_t st_b = N * hv * 128 * 128 * 4;
    const struct { const void *p; size_t n; } ins[] = {
        {q, T * hk * 256}, {k, T * hk * 256}, {v, T * hv * 256}, {a, T * hv * 2},
        {b, T * hv * 2}, {z, z ? T * hv * 256 : 0}, {init_state, init_state ? st_b : 0},
        {cu_seqlens, (N + 1) * 4}, {workspace, need}};
    for (const auto &x : ins)
        if (overlaps(out, out_b, x.p, x.n))
            return GDN_ERR_INVALID_ARG;
    if (init_state != final_state && overlaps(final_state, st_b, init_state, init_state ? st_b : 0))
        return GDN_ERR_INVALID_ARG;   // partial overlap; exact equality is the in-place case
    if (overlaps(final_state, st_b, out, out_b) || overlaps(final_state, st_b, workspace, need))
        return GDN_ERR_INVALID_ARG;

    gdn::PrefillArgs p{};
    p.num_seqs = s->num_seqs;
    p.total_tokens = s->total_tokens;
    p.hk = s->hk;
    p.hv = s->hv;
    p.max_chunks = gdn::prefill_max_chunks(s->num_seqs, s->total_tokens);
    p.q = q; p.k = k; p.v = v; p.a = a; p.b = b;
    p.A_log = A_log; p.dt_bias = dt_bias;
    p.init_state = init_state;
    p.cu_seqlens = cu_seqlens;
    p.z = z; p.norm_w = norm_w; p.eps = eps;
    p.out = out;
    p.final_state = final_state;
    p.workspace = static_cast<unsigned char *>(workspace);
    p.status = status_ptr();
    if (!p.status)
        return GDN_ERR_CUDA;
    return gdn::launch_prefill(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

gdn_status_t gdn_decode_slots(const gdn_shape_t *s, int32_t tokens, int32_t num_slots, const void *q,
                              const void *k, const void *v, const void *a, const void *b, const float *A_log,
                              const float *dt_bias, float *state, const int32_t *state_idx, const void *z,
                              const void *norm_w, float eps, void *out, void *stream)
{
    gdn_status_t st = check_shape(s);
    if (st != GDN_OK)
        return st;
    if (tokens < 1 || tokens > 8 || num_slots < 0)
        return GDN_ERR_INVALID_ARG;
    if ((int64_t)s->total_tokens != (int64_t)s->num_seqs * tokens)
        return GDN_ERR_INVALID_ARG;
    const size_t B = (size_t)s->num_seqs;
    if (B == 0)
        return GDN_OK;
    if (!state_idx && (size_t)num_slots < B)
        return GDN_ERR_INVALID_ARG;
    if (!q || !k || !v || !a || !b || !A_log || !dt_bias || !out || (num_slots > 0 && !state))
        return GDN_ERR_INVALID_ARG;
    if (z && !norm_w)
        return GDN_ERR_INVALID_ARG;
    if (!(eps >= 0.f))
        return GDN_ERR_INVALID_ARG;
    const void *al16[] = {q, k, v, a, b, state, z, norm_w, out};
    for (const void *p : al16)
        if (p && !aligned(p, 16))
            return GDN_ERR_ALIGNMENT;
    if (state_idx && !aligned(state_idx, 4))
        return GDN_ERR_ALIGNMENT;
    const size_t hk = s->hk, hv = s->hv, BT = B * (size_t)tokens;
    const size_t out_b = BT * hv * 256;
    const struct { const void *p; size_t n; } ins[] = {
        {q, BT * hk * 256}, {k, BT * hk * 256}, {v, BT * hv * 256}, {a, BT * hv * 2},
        {b, BT * hv * 2}, {z, z ? BT * hv * 256 : 0}, {state, (size_t)num_slots * hv * 128 * 128 * 4},
        {state_idx, state_idx ? B * 4 : 0}};
    for (const auto &x : ins)
        if (overlaps(out, out_b, x.p, x.n))
            return GDN_ERR_INVALID_ARG;

    gdn::DecodeArgs p{};
    p.batch = s->num_seqs;
    p.hk = s->hk;
    p.hv = s->hv;
    p.tokens = tokens;
    p.num_slots = num_slots;
    p.state_idx = state_idx;
    p.q = q; p.k = k; p.v = v; p.a = a; p.b = b;
    p.A_log = A_log; p.dt_bias = dt_bias;
    p.state = state;
    p.z = z; p.norm_w = norm_w; p.eps = eps;
    p.out = out;
    p.status = status_ptr();
    if (!p.status)
        return GDN_ERR_CUDA;
    return gdn::launch_decode(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

gdn_status_t gdn_decode(const gdn_shape_t *s, const void *q, const void *k, const void *v,
                        const void *a, const void *b, const float *A_log, const float *dt_bias,
                        float *state, const void *z, const void *norm_w, float eps, void *out,
                        void *stream)
{
    gdn_status_t st = check_shape(s);
    if (st != GDN_OK)
        return st;
    if (s->total_tokens != s->num_seqs)
        return GDN_ERR_INVALID_ARG;
    if (s->num_seqs > 0 && !state)
        return GDN_ERR_INVALID_ARG;
    return gdn_decode_slots(s, 1, s->num_seqs, q, k, v, a, b, A_log, dt_bias, state, nullptr, z, norm_w,
                            eps, out, stream);
}

gdn_status_t gdn_check_device_status(uint32_t *bits)
{
    uint32_t h = 0;
    const uint32_t zero = 0;
    if (cudaDeviceSynchronize() != cudaSuccess)
        return GDN_ERR_CUDA;
    if (cudaMemcpyFromSymbol(&h, g_device_status, sizeof(h)) != cudaSuccess)
        return GDN_ERR_CUDA;
    if (h && cudaMemcpyToSymbol(g_device_status, &zero, sizeof(zero)) != cudaSuccess)
        return GDN_ERR_CUDA;
    if (bits)
        *bits = h;
    return h ? GDN_ERR_DEVICE_STATUS : GDN_OK;
}

}  // extern "C"
