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
    DEV_RANGE = 3,        // an fp16 output beyond fp16's finite range (or NaN)
};

__device__ __forceinline__ void raise_error(int* err, int code) {
    if (err != nullptr) atomicCAS(err, 0, code);
}

// fp16 outputs: |v| >= 65520 rounds to infinity (65504 is fp16's largest finite
// value); a value that would leave the finite range, or NaN, sets DEV_RANGE.
__device__ __forceinline__ void check_half_range(float v0, float v1, int* err) {
    if (!(fabsf(v0) < 65520.0f) || !(fabsf(v1) < 65520.0f)) raise_error(err, DEV_RANGE);
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

// e^x for x <= 0 as 2^(x log2 e) on the SFU (ex2.approx, relative error about 2^-22):
// the rounding of the product x log2 e adds |x| * 2^-24 relative, so the result is
// within about (2 + |x|) 1e-7 of e^x (for |x| <= 20, 2.4e-6).
__device__ __forceinline__ float exp_nonpos_f32(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x * 1.44269504f));
    return r;
}

// Softplus(z) = log(1 + e^z) = max(z, 0) + log1p(u), u = e^-|z| in (0, 1].
// log1p(u) = 2 atanh(s) with s = u / (2 + u) <= 1/3, summed as the series
// 2 s (1 + s^2/3 + s^4/5 + ... + s^12/13); the first omitted term is below
// (1/9)^7 / 15 < 2^-26 of the sum.  For z < 0 the result keeps the relative accuracy
// of e^z itself (exp_nonpos_f32: about (2 + |z|) 1e-7; s by the SFU reciprocal, one
// more ulp); for large z it rounds to z.
__device__ __forceinline__ float softplus_f32(float z) {
    const float u = exp_nonpos_f32(-fabsf(z));
    const float s = u * rcp_approx(2.0f + u);
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

// erfc(x) for x >= 0 with a small RELATIVE error at every x (the Load sums tails of
// the normal distribution, so relative accuracy in the tail matters): the Chebyshev
// fit of Numerical Recipes (Press et al., 2nd ed., section 6.2, erfcc),
// erfc(x) = t exp(-x^2 + P(t)), t = 1 / (1 + x/2), P of degree 9, fractional error
// below 1.2e-7.  In fp32 the exponent -x^2 + P(t) is carried with the rounding errors
// of x*x and of the sum, which keeps the error near 5e-7 up to x = 9 instead of
// growing like x^2 ulp.
__device__ __forceinline__ float erfc_pos_f32(float x) {
    const float t = rcp_approx(fmaf(0.5f, x, 1.0f));   // (1 ulp: 2e-7 more relative error)
    float p = 0.17087277f;
    p = fmaf(p, t, -0.82215223f);
    p = fmaf(p, t, 1.48851587f);
    p = fmaf(p, t, -1.13520398f);
    p = fmaf(p, t, 0.27886807f);
    p = fmaf(p, t, -0.18628806f);
    p = fmaf(p, t, 0.09678418f);
    p = fmaf(p, t, 0.37409196f);
    p = fmaf(p, t, 1.00002368f);
    p = fmaf(p, t, -1.26551223f);
    const float x2 = x * x;
    const float e2 = fmaf(x, x, -x2);                  // x*x = x2 + e2 exactly
    const float sx = p - x2;
    const float bb = sx - p;
    const float es = (p - (sx - bb)) + (-x2 - bb);     // p - x2 = sx + es exactly
    return t * expf(sx) * (1.0f + (es - e2));
}

// Standard normal CDF Phi(z) = erfc(-z / sqrt 2) / 2; |z| is capped at 40, where the
// tail is below the smallest fp32 (z = +-inf, a threshold of -inf when every expert is
// kept, gives exactly 1 or 0).
__device__ __forceinline__ float normal_cdf_f32(float z) {
    const float x = fminf(fabsf(z), 40.0f) * 0.70710678f;
    const float q = 0.5f * erfc_pos_f32(x);
    return z >= 0.0f ? 1.0f - q : q;
}

// Programmatic dependent launch.  Every kernel of the library is launched with
// programmatic stream serialization (launch_pdl below), so it may start while the
// previous kernel on the stream is still running; griddep_wait() blocks until that
// kernel has completed and its writes are visible, and must come before the first
// global-memory read (its own setup -- barriers, TMEM, tensor-map prefetch -- may
// precede it).  griddep_launch_dependents() lets the next kernel start launching.
// Both are no-ops for a kernel launched without the attribute.
__device__ __forceinline__ void griddep_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm volatile("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Launch `kernel` on `s` with programmatic stream serialization (and a cluster of
// cluster_x CTAs along x when cluster_x > 1).
template <typename... Params, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, int cluster_x, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int na = 0;
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    if (cluster_x > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = cluster_x;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Params>(args)...);
}

}  // namespace moe
