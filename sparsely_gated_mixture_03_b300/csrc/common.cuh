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

// Softplus(z) = log(1 + e^z).  Above z = 20 the correction log1p(e^-z) is
// below 2.1e-9, under half an fp32 ulp of z, so z itself is returned.
__device__ __forceinline__ float softplus_f32(float z) {
    return z > 20.0f ? z : log1pf(expf(z));
}

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm volatile("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

}  // namespace moe
