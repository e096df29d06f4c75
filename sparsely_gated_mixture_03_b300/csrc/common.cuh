// Device helpers shared by the library's kernels (GPU side only).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace moe {

// Codes of the device error word (set once, first error wins).
enum DeviceError : int {
    DEV_OK = 0,
    DEV_TIMEOUT = 1,      // a bounded spin on an mbarrier or flag gave up
    DEV_BAD_INDEX = 2,    // an expert index outside [0, n)
};

__device__ __forceinline__ void raise_error(int* err, int code) {
    if (err != nullptr) atomicCAS(err, 0, code);
}

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}
template <> __device__ __forceinline__ __half from_f32<__half>(float v) {
    return __float2half_rn(v);
}

// 1/x by the SFU's approximate reciprocal (relative error about 2^-23).
__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// a / b to about 1 ulp: the approximate reciprocal and one residual correction.
__device__ __forceinline__ float div_refined(float a, float b) {
    const float r = rcp_approx(b);
    const float q = a * r;
    return fmaf(fmaf(-b, q, a), r, q);
}

// Softplus(z) = log(1 + e^z) = max(z, 0) + log1p(u), u = e^-|z| in (0, 1].
// log1p(u) = 2 atanh(s) with s = u / (2 + u) <= 1/3, summed as the series
// 2 s (1 + s^2/3 + s^4/5 + ... + s^12/13); the first omitted term is below
// (1/9)^7 / 15 < 2^-26 of the sum.  For z < 0 the result keeps full relative
// accuracy down to e^z itself; for large z it rounds to z.
__device__ __forceinline__ float softplus_f32(float z) {
    const float u = expf(-fabsf(z));
    const float s = div_refined(u, 2.0f + u);
    const float s2 = s * s;
    float p = 1.0f / 13.0f;
    p = fmaf(p, s2, 1.0f / 11.0f);
    p = fmaf(p, s2, 1.0f / 9.0f);
    p = fmaf(p, s2, 1.0f / 7.0f);
    p = fmaf(p, s2, 1.0f / 5.0f);
    p = fmaf(p, s2, 1.0f / 3.0f);
    p = fmaf(p, s2, 1.0f);
    return fmaxf(z, 0.0f) + 2.0f * s * p;
}

// Standard normal CDF Phi(z), by the rational approximation of the upper tail in
// Abramowitz & Stegun, Handbook of Mathematical Functions, 26.2.17 (after Hastings):
// for x >= 0, 1 - Phi(x) = phi(x) (b1 t + b2 t^2 + b3 t^3 + b4 t^4 + b5 t^5),
// t = 1 / (1 + p x), with absolute error below 7.5e-8; Phi(-x) = 1 - Phi(x).
// |z| is capped at 40, where the tail is below the smallest fp32 (z = +-inf, a
// threshold of -inf when every expert is kept, gives exactly 1 or 0).
__device__ __forceinline__ float normal_cdf_f32(float z) {
    const float x = fminf(fabsf(z), 40.0f);
    const float t = div_refined(1.0f, fmaf(0.2316419f, x, 1.0f));
    float poly = 1.330274429f;
    poly = fmaf(poly, t, -1.821255978f);
    poly = fmaf(poly, t, 1.781477937f);
    poly = fmaf(poly, t, -0.356563782f);
    poly = fmaf(poly, t, 0.319381530f);
    poly *= t;
    const float pdf = 0.3989422804f * expf(-0.5f * x * x);   // phi(x) = e^(-x^2/2) / sqrt(2 pi)
    const float tail = pdf * poly;                           // 1 - Phi(x)
    return z >= 0.0f ? 1.0f - tail : tail;
}

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm volatile("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

}  // namespace moe
