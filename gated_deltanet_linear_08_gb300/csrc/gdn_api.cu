// gdn_api.cu -- the C ABI of libgdn (include/gdn.h): host-side validation,
// status codes and dispatch onto the caller's stream.  Unsupported shapes are
// explicit errors returned before any launch, as the pegainfer review asks of
// a stable C ABI ("feat(qwen35): add SM120 FlashInfer GDN prefill
// candidate", maintainer review: unsupported shapes handled explicitly).
// Nothing here allocates device memory, prints, aborts or synchronises,
// except gdn_check_device_status, which is documented as off the hot path.
#include <atomic>

#include <cuda_runtime.h>

#include "../../include/gdn.h"
#include "kernels.h"

namespace {

// Status word the kernels OR bits into when a bounded wait runs out.
__device__ uint32_t g_device_status;

// Device address of g_device_status, per device.  Host threads may make their
// first call on a device at the same time: each then looks the address up and
// stores the same value, which the atomic makes a well-defined race.
std::atomic<uint32_t *> g_status_ptr[gdn::kMaxDevices];

uint32_t *status_ptr()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= gdn::kMaxDevices)
        return nullptr;
    uint32_t *cached = g_status_ptr[dev].load(std::memory_order_relaxed);
    if (!cached) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess)
            return nullptr;
        cached = static_cast<uint32_t *>(p);
        g_status_ptr[dev].store(cached, std::memory_order_relaxed);
    }
    return cached;
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

// The caller's strides, or the dense layouts when none are given; false if
// they break the rules of gdn_strides_t.
bool resolve_strides(const gdn_strides_t *u, int hk, int hv, bool with_z, gdn::InputStrides &o)
{
    const int64_t k = 128;
    o.q = {hk * k, k}; o.k = {hk * k, k}; o.v = {hv * k, k}; o.z = {hv * k, k};
    o.a = {hv, 1}; o.b = {hv, 1};
    if (!u)
        return true;
    o.q = {u->q.token, u->q.head}; o.k = {u->k.token, u->k.head}; o.v = {u->v.token, u->v.head};
    o.a = {u->a.token, u->a.head}; o.b = {u->b.token, u->b.head};
    if (with_z)
        o.z = {u->z.token, u->z.head};
    for (const gdn::Stride &x : {o.q, o.k, o.v, o.z})
        if (x.t <= 0 || x.h < 128 || x.t % 8 || x.h % 8)
            return false;
    for (const gdn::Stride &x : {o.a, o.b})
        if (x.t <= 0 || x.h <= 0)
            return false;
    return true;
}

// Bytes spanned by a strided bf16 input of `tokens` x `heads` rows of `row`
// elements (0 for an absent tensor).
size_t span(const void *p, size_t tokens, size_t heads, const gdn::Stride &x, size_t row)
{
    if (!p || tokens == 0)
        return 0;
    return ((tokens - 1) * (size_t)x.t + (heads - 1) * (size_t)x.h + row) * 2;
}

// The caller's conv descriptor (NULL: no conv), checked against the shape.
// `rows` is the number of state rows: sequences for prefill, slots for
// decode.  state_out may equal state_in; any other overlap is rejected.
gdn_status_t resolve_conv(const gdn_conv_t *c, const gdn_shape_t *s, size_t rows, bool decode,
                          gdn::ConvArgs &o, size_t &state_bytes)
{
    o = gdn::ConvArgs{};
    state_bytes = 0;
    if (!c)
        return GDN_OK;
    if (c->width < 1 || c->width > 4 || !c->weight)
        return GDN_ERR_INVALID_ARG;
    if (decode && c->width > 1 && !c->state_in)
        return GDN_ERR_INVALID_ARG;   // the slot pool holds the history
    o.width = c->width;
    o.channels = (2 * s->hk + s->hv) * 128;
    o.weight = static_cast<const __nv_bfloat16 *>(c->weight);
    o.state_in = static_cast<const __nv_bfloat16 *>(c->state_in);
    o.state_out = static_cast<__nv_bfloat16 *>(c->state_out);
    if (!aligned(c->weight, 16) || !aligned(c->state_in, 16) || !aligned(c->state_out, 16))
        return GDN_ERR_ALIGNMENT;
    state_bytes = rows * (size_t)(c->width - 1) * (size_t)o.channels * 2;
    if (c->state_in != c->state_out && overlaps(c->state_in, state_bytes, c->state_out, state_bytes))
        return GDN_ERR_INVALID_ARG;
    const size_t wb = (size_t)o.channels * c->width * 2;
    if (overlaps(c->state_out, state_bytes, c->weight, wb))
        return GDN_ERR_INVALID_ARG;
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

size_t gdn_prefill_conv_workspace_bytes(const gdn_shape_t *s)
{
    if (check_shape(s) != GDN_OK || s->total_tokens <= 0)
        return 0;
    return gdn::prefill_workspace_bytes(s->num_seqs, s->total_tokens, s->hk, s->hv)
           + gdn::prefill_conv_bytes(s->total_tokens, s->hk, s->hv);
}

gdn_status_t gdn_prefill_conv(const gdn_shape_t *s, const gdn_strides_t *strides, const gdn_conv_t *conv,
                              const void *q, const void *k, const void *v, const void *a, const void *b,
                              const float *A_log, const float *dt_bias, const float *init_state,
                              const int32_t *cu_seqlens, const void *z, const void *norm_w, float eps, void *out,
                              float *final_state, void *workspace, size_t workspace_bytes, void *stream)
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
    gdn::InputStrides in;
    if (!resolve_strides(strides, s->hk, s->hv, z != nullptr, in))
        return GDN_ERR_INVALID_ARG;
    const void *al16[] = {q, k, v, init_state, z, norm_w, out, final_state};
    for (const void *p : al16)
        if (p && !aligned(p, 16))
            return GDN_ERR_ALIGNMENT;
    if (!aligned(a, 2) || !aligned(b, 2))   // read one element at a time
        return GDN_ERR_ALIGNMENT;
    const size_t core_need = gdn::prefill_workspace_bytes(s->num_seqs, s->total_tokens, s->hk, s->hv);
    const size_t need = core_need + (conv ? gdn::prefill_conv_bytes(s->total_tokens, s->hk, s->hv) : 0);
    if (need > 0 && (!workspace || workspace_bytes < need))
        return GDN_ERR_WORKSPACE;
    if (workspace && !aligned(workspace, 1024))
        return GDN_ERR_ALIGNMENT;
    const size_t hk = s->hk, hv = s->hv;
    const size_t out_b = T * hv * 128 * 2;
    const size_t st_b = N * hv * 128 * 128 * 4;
    // everything the call reads; the workspace, out and final_state (the
    // buffers it writes) may overlap none of them, except that final_state
    // may be exactly init_state (the in-place case)
    const struct { const void *p; size_t n; } ins[] = {
        {q, span(q, T, hk, in.q, 128)}, {k, span(k, T, hk, in.k, 128)}, {v, span(v, T, hv, in.v, 128)},
        {a, span(a, T, hv, in.a, 1)}, {b, span(b, T, hv, in.b, 1)}, {z, span(z, T, hv, in.z, 128)},
        {init_state, init_state ? st_b : 0}, {cu_seqlens, (N + 1) * 4}, {A_log, hv * 4}, {dt_bias, hv * 4},
        {norm_w, z ? 256u : 0u}};
    for (const auto &x : ins)
        if (overlaps(out, out_b, x.p, x.n) || overlaps(workspace, need, x.p, x.n))
            return GDN_ERR_INVALID_ARG;
    for (const auto &x : ins)   // ins[6] is init_state, checked below
        if (&x != &ins[6] && overlaps(final_state, st_b, x.p, x.n))
            return GDN_ERR_INVALID_ARG;
    if (init_state != final_state && overlaps(final_state, st_b, init_state, init_state ? st_b : 0))
        return GDN_ERR_INVALID_ARG;   // partial overlap; exact equality is the in-place case
    if (overlaps(final_state, st_b, out, out_b) || overlaps(final_state, st_b, workspace, need)
        || overlaps(out, out_b, workspace, need))
        return GDN_ERR_INVALID_ARG;
    gdn::ConvArgs cv;
    size_t cs_b = 0;
    if ((st = resolve_conv(conv, s, N, false, cv, cs_b)) != GDN_OK)
        return st;
    if (cv.state_out) {
        // the state written must not alias anything the call reads or writes
        for (const auto &x : ins)
            if (overlaps(cv.state_out, cs_b, x.p, x.n))
                return GDN_ERR_INVALID_ARG;
        if (overlaps(cv.state_out, cs_b, out, out_b) || overlaps(cv.state_out, cs_b, final_state, st_b)
            || overlaps(cv.state_out, cs_b, workspace, need))
            return GDN_ERR_INVALID_ARG;
    }
    if (overlaps(cv.state_in, cs_b, out, out_b) || overlaps(cv.state_in, cs_b, final_state, st_b)
        || overlaps(cv.state_in, cs_b, workspace, need))
        return GDN_ERR_INVALID_ARG;
    if (conv) {
        const size_t wb = (size_t)cv.channels * cv.width * 2;
        if (overlaps(cv.weight, wb, out, out_b) || overlaps(cv.weight, wb, final_state, st_b)
            || overlaps(cv.weight, wb, workspace, need))
            return GDN_ERR_INVALID_ARG;
    }

    gdn::PrefillArgs p{};
    p.num_seqs = s->num_seqs;
    p.total_tokens = s->total_tokens;
    p.hk = s->hk;
    p.hv = s->hv;
    p.max_chunks = gdn::prefill_max_chunks(s->num_seqs, s->total_tokens);
    p.in = in;
    p.q = q; p.k = k; p.v = v; p.a = a; p.b = b;
    if (conv) {
        // the conv reads the raw inputs; the core reads its output, q | k | v
        // rows of `channels` elements in the workspace after the records
        cv.x_q = q; cv.x_k = k; cv.x_v = v;
        cv.x_in = in;
        cv.y = reinterpret_cast<__nv_bfloat16 *>(static_cast<unsigned char *>(workspace) + core_need);
        const int64_t C = cv.channels;
        p.q = cv.y;
        p.k = cv.y + (size_t)s->hk * 128;
        p.v = cv.y + (size_t)2 * s->hk * 128;
        p.in.q = {C, 128}; p.in.k = {C, 128}; p.in.v = {C, 128};
    }
    p.conv = cv;
    p.A_log = A_log; p.dt_bias = dt_bias;
    p.init_state = init_state;
    p.cu_seqlens = cu_seqlens;
    if (s->num_seqs >= gdn::kIndexMinSeqs && T > 0)
        p.chunk_off = reinterpret_cast<int32_t *>(static_cast<unsigned char *>(workspace)
                                                  + gdn::prefill_index_offset(s->num_seqs, s->total_tokens, s->hv));
    p.z = z; p.norm_w = norm_w; p.eps = eps;
    p.out = out;
    p.final_state = final_state;
    p.workspace = static_cast<unsigned char *>(workspace);
    p.status = status_ptr();
    if (!p.status)
        return GDN_ERR_CUDA;
    return gdn::launch_prefill(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

gdn_status_t gdn_conv_prefill(const gdn_shape_t *s, const gdn_strides_t *strides, const gdn_conv_t *conv,
                              const void *q, const void *k, const void *v, const int32_t *cu_seqlens, void *y,
                              void *stream)
{
    gdn_status_t st = check_shape(s);
    if (st != GDN_OK)
        return st;
    const size_t T = (size_t)s->total_tokens, N = (size_t)s->num_seqs;
    if (N == 0)
        return T == 0 ? GDN_OK : GDN_ERR_INVALID_ARG;
    if (!conv || !cu_seqlens)
        return GDN_ERR_INVALID_ARG;
    if (conv->state_out)
        return GDN_ERR_INVALID_ARG;   // this entry point writes y only
    if (T == 0)
        return GDN_OK;
    if (!q || !k || !v || !y)
        return GDN_ERR_INVALID_ARG;
    // only q, k and v are read: the caller's a, b strides do not matter here
    gdn_strides_t qkv;
    if (strides) {
        qkv = *strides;
        qkv.a = qkv.b = gdn_stride_t{1, 1};
    }
    gdn::InputStrides in;
    if (!resolve_strides(strides ? &qkv : nullptr, s->hk, s->hv, false, in))
        return GDN_ERR_INVALID_ARG;
    const void *al16[] = {q, k, v, y};
    for (const void *ptr : al16)
        if (!aligned(ptr, 16))
            return GDN_ERR_ALIGNMENT;
    gdn::ConvArgs cv;
    size_t cs_b = 0;
    if ((st = resolve_conv(conv, s, N, false, cv, cs_b)) != GDN_OK)
        return st;
    const size_t hk = s->hk, hv = s->hv;
    const size_t y_b = T * (size_t)cv.channels * 2;
    const struct { const void *p; size_t n; } ins[] = {
        {q, span(q, T, hk, in.q, 128)}, {k, span(k, T, hk, in.k, 128)}, {v, span(v, T, hv, in.v, 128)},
        {cu_seqlens, (N + 1) * 4}, {cv.weight, (size_t)cv.channels * cv.width * 2}, {cv.state_in, cs_b}};
    for (const auto &x : ins)
        if (overlaps(y, y_b, x.p, x.n))
            return GDN_ERR_INVALID_ARG;
    cv.x_q = q; cv.x_k = k; cv.x_v = v;
    cv.x_in = in;
    cv.y = static_cast<__nv_bfloat16 *>(y);
    gdn::PrefillArgs p{};
    p.num_seqs = s->num_seqs;
    p.total_tokens = s->total_tokens;
    p.hk = s->hk;
    p.hv = s->hv;
    p.cu_seqlens = cu_seqlens;
    p.conv = cv;
    p.status = status_ptr();
    if (!p.status)
        return GDN_ERR_CUDA;
    return gdn::launch_prefill_conv(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

gdn_status_t gdn_prefill_strided(const gdn_shape_t *s, const gdn_strides_t *strides, const void *q,
                                 const void *k, const void *v, const void *a, const void *b, const float *A_log,
                                 const float *dt_bias, const float *init_state, const int32_t *cu_seqlens,
                                 const void *z, const void *norm_w, float eps, void *out, float *final_state,
                                 void *workspace, size_t workspace_bytes, void *stream)
{
    return gdn_prefill_conv(s, strides, nullptr, q, k, v, a, b, A_log, dt_bias, init_state, cu_seqlens, z, norm_w,
                            eps, out, final_state, workspace, workspace_bytes, stream);
}

gdn_status_t gdn_prefill(const gdn_shape_t *s, const void *q, const void *k, const void *v,
                         const void *a, const void *b, const float *A_log, const float *dt_bias,
                         const float *init_state, const int32_t *cu_seqlens, const void *z,
                         const void *norm_w, float eps, void *out, float *final_state,
                         void *workspace, size_t workspace_bytes, void *stream)
{
    return gdn_prefill_strided(s, nullptr, q, k, v, a, b, A_log, dt_bias, init_state, cu_seqlens, z, norm_w,
                               eps, out, final_state, workspace, workspace_bytes, stream);
}

gdn_status_t gdn_decode_conv(const gdn_shape_t *s, const gdn_strides_t *strides, const gdn_conv_t *conv,
                             int32_t tokens, int32_t num_slots, const void *q, const void *k, const void *v,
                             const void *a, const void *b, const float *A_log, const float *dt_bias, float *state,
                             const int32_t *state_idx, const void *z, const void *norm_w, float eps, void *out,
                             void *stream)
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
    gdn::InputStrides in;
    if (!resolve_strides(strides, s->hk, s->hv, z != nullptr, in))
        return GDN_ERR_INVALID_ARG;
    const void *al16[] = {q, k, v, state, z, norm_w, out};
    for (const void *p : al16)
        if (p && !aligned(p, 16))
            return GDN_ERR_ALIGNMENT;
    if (!aligned(a, 2) || !aligned(b, 2))   // read one element at a time
        return GDN_ERR_ALIGNMENT;
    if (state_idx && !aligned(state_idx, 4))
        return GDN_ERR_ALIGNMENT;
    const size_t hk = s->hk, hv = s->hv, BT = B * (size_t)tokens;
    const size_t out_b = BT * hv * 256;
    const size_t pool_b = (size_t)num_slots * hv * 128 * 128 * 4;
    const struct { const void *p; size_t n; } ins[] = {
        {q, span(q, BT, hk, in.q, 128)}, {k, span(k, BT, hk, in.k, 128)}, {v, span(v, BT, hv, in.v, 128)},
        {a, span(a, BT, hv, in.a, 1)}, {b, span(b, BT, hv, in.b, 1)}, {z, span(z, BT, hv, in.z, 128)},
        {state, pool_b}, {state_idx, state_idx ? B * 4 : 0}, {A_log, hv * 4}, {dt_bias, hv * 4},
        {norm_w, z ? 256u : 0u}};
    for (const auto &x : ins)
        if (overlaps(out, out_b, x.p, x.n))
            return GDN_ERR_INVALID_ARG;
    // the pool is read and written in place: no other input may lie in it
    for (const auto &x : ins)   // ins[6] is the pool itself
        if (&x != &ins[6] && overlaps(state, pool_b, x.p, x.n))
            return GDN_ERR_INVALID_ARG;
    gdn::ConvArgs cv;
    size_t cs_b = 0;
    if ((st = resolve_conv(conv, s, (size_t)num_slots, true, cv, cs_b)) != GDN_OK)
        return st;
    if (conv) {
        // neither conv state may alias the outputs; the one written, nothing read
        if (overlaps(out, out_b, cv.state_in, cs_b) || overlaps(out, out_b, cv.state_out, cs_b)
            || overlaps(cv.state_in, cs_b, state, (size_t)num_slots * hv * 128 * 128 * 4))
            return GDN_ERR_INVALID_ARG;
        for (const auto &x : ins)
            if (overlaps(cv.state_out, cs_b, x.p, x.n))
                return GDN_ERR_INVALID_ARG;
    }

    gdn::DecodeArgs p{};
    p.batch = s->num_seqs;
    p.hk = s->hk;
    p.hv = s->hv;
    p.tokens = tokens;
    p.num_slots = num_slots;
    p.state_idx = state_idx;
    p.in = in;
    p.conv = cv;
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

gdn_status_t gdn_decode_strided(const gdn_shape_t *s, const gdn_strides_t *strides, int32_t tokens,
                                int32_t num_slots, const void *q, const void *k, const void *v, const void *a,
                                const void *b, const float *A_log, const float *dt_bias, float *state,
                                const int32_t *state_idx, const void *z, const void *norm_w, float eps,
                                void *out, void *stream)
{
    return gdn_decode_conv(s, strides, nullptr, tokens, num_slots, q, k, v, a, b, A_log, dt_bias, state, state_idx,
                           z, norm_w, eps, out, stream);
}

gdn_status_t gdn_decode_slots(const gdn_shape_t *s, int32_t tokens, int32_t num_slots, const void *q,
                              const void *k, const void *v, const void *a, const void *b, const float *A_log,
                              const float *dt_bias, float *state, const int32_t *state_idx, const void *z,
                              const void *norm_w, float eps, void *out, void *stream)
{
    return gdn_decode_strided(s, nullptr, tokens, num_slots, q, k, v, a, b, A_log, dt_bias, state, state_idx, z,
                              norm_w, eps, out, stream);
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
