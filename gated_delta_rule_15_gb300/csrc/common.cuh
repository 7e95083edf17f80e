// common.cuh -- small device helpers shared by the library's kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dr {

// Loads of one storage element as fp32.
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// Four consecutive storage elements as fp32 (the address is 8- or 16-byte aligned).
__device__ __forceinline__ float4 load4(const float *p) {
    return *reinterpret_cast<const float4 *>(p);
}
__device__ __forceinline__ float4 load4(const __nv_bfloat16 *p) {
    uint2 u = *reinterpret_cast<const uint2 *>(p);
    __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162 *>(&u.x);
    __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162 *>(&u.y);
    float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
    return make_float4(fa.x, fa.y, fb.x, fb.y);
}

__device__ __forceinline__ void store4(float *p, float4 v) {
    *reinterpret_cast<float4 *>(p) = v;
}
__device__ __forceinline__ void store4(__nv_bfloat16 *p, float4 v) {
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
    __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t *>(&a);
    u.y = *reinterpret_cast<uint32_t *>(&b);
    *reinterpret_cast<uint2 *>(p) = u;
}

// Neighbours of the operation that the kernels fuse (DR_FUSE_* of include/dr.h).
// L2-normalisation epsilon under the square root (DR_L2NORM_EPS).
constexpr float kL2NormEps = 1e-6f;
// 1 / (1 + exp(-x)) and x / (1 + exp(-x)) with the fast intrinsics (two MUFU operations;
// relative error a few 1e-6 for |x| < 20).  For x below about -88, exp(-x) overflows to
// infinity and the quotient is 0 (the exact values are below 1e-36 in magnitude).
__device__ __forceinline__ float sigmoid_f(float x) { return __fdividef(1.f, 1.f + __expf(-x)); }
__device__ __forceinline__ float silu_f(float x) { return __fdividef(x, 1.f + __expf(-x)); }
// x sigmoid(x) = x (1 + tanh(x / 2)) / 2 with one MUFU operation (PTX tanh.approx.f32,
// relative error about 2^-11): for the bf16-input kernels, where it is far below the
// inputs' own rounding.
__device__ __forceinline__ float silu_tanh(float x) {
    const float h = 0.5f * x;
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(h));
    return fmaf(h, t, h);
}
// Round to the nearest bf16 (ties to even), back as fp32.
__device__ __forceinline__ float round_bf16(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

// Library status codes (mirrors include/dr.h).
enum : int {
    kOk = 0, kErrInvalid = -1, kErrUnsupported = -2, kErrCuda = -3, kErrTimeout = -4,
    kErrWorkspace = -5
};

}  // namespace dr
