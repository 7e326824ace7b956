// common.cuh -- device helpers shared by the GDN kernels: the per-token gate
// and beta (JevAny page "Add opt-in fused Qwen3.5 inference kernels",
// Summary: gate from A_log and dt_bias, beta sigmoid), bf16/fp16 packing, and the
// device status bits that bounded waits set.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace gdn {

constexpr int kD = 128;      // Dk = Dv
constexpr int kC = 64;       // chunk length
constexpr float kL2Eps = 1e-6f;

// Device status bits (OR-ed into the status word by kernels).
constexpr uint32_t kStatusWaitTimeout = 1u << 0;
constexpr uint32_t kStatusBadSeqlens = 1u << 1;
constexpr uint32_t kStatusRange = 1u << 2;   // a value outside the fp16 operand range
constexpr float kHalfMax = 65504.f;

// softplus(x) = log(1 + e^x); above 20 the correction log1p(e^-x) < 2.1e-9
// is below fp32 resolution of x, so x itself is returned.
__device__ __forceinline__ float softplus_f(float x)
{
    return x > 20.f ? x : log1pf(expf(x));
}
__device__ __forceinline__ float sigmoid_f(float x) { return 1.f / (1.f + expf(-x)); }

// g = -exp(A_log) * softplus(a + dt_bias)
__device__ __forceinline__ float gate_f(float a, float A_log, float dt_bias)
{
    return -expf(A_log) * softplus_f(a + dt_bias);
}

__device__ __forceinline__ float bf2f(__nv_bfloat16 x) { return __bfloat162float(x); }

// Unpack 8 bf16 held in a 16-byte vector.
__device__ __forceinline__ void unpack8(const uint4 &u, float (&f)[8])
{
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}
// Unpack 4 bf16 held in an 8-byte vector.
__device__ __forceinline__ void unpack4(const uint2 &u, float (&f)[4])
{
    f[0] = __uint_as_float(u.x << 16);
    f[1] = __uint_as_float(u.x & 0xFFFF0000u);
    f[2] = __uint_as_float(u.y << 16);
    f[3] = __uint_as_float(u.y & 0xFFFF0000u);
}
// Pack two floats into bf16x2 (round to nearest even), lo in the low half.
__device__ __forceinline__ uint32_t pack2(float lo, float hi)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ uint4 pack8(const float (&v)[8])
{
    return make_uint4(pack2(v[0], v[1]), pack2(v[2], v[3]), pack2(v[4], v[5]), pack2(v[6], v[7]));
}
// Pack two floats into f16x2 (round to nearest even), lo in the low half.
__device__ __forceinline__ uint32_t pack2h(float lo, float hi)
{
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ uint4 pack8h(const float (&v)[8])
{
    return make_uint4(pack2h(v[0], v[1]), pack2h(v[2], v[3]), pack2h(v[4], v[5]), pack2h(v[6], v[7]));
}
__device__ __forceinline__ float bf16_round(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

__device__ __forceinline__ void set_status(uint32_t *status, uint32_t bits)
{
    if (status)
        atomicOr(status, bits);
}

}  // namespace gdn
