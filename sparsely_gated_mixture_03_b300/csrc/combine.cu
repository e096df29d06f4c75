// Gate-weighted combine, eq (1) of "Mixture of Experts: Outrageously Large Neural
// Networks" (intuitivepapers.ai), section "How a mixture-of-experts layer works":
// y = sum_i G(x)_i E_i(x).  G is zero outside the k kept experts, so the sum runs
// over the token's k expert outputs, gathered through inv, in slot order j = 0..k-1
// with fp32 accumulation: a fixed order, so y is bitwise reproducible.
#include <stdint.h>

#include "common.cuh"
#include "launch.h"

namespace moe {
namespace {

__device__ __forceinline__ void load8(const __half* p, float o[8]) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    const __half2* h = reinterpret_cast<const __half2*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __half22float2(h[i]);
        o[2 * i] = f.x;
        o[2 * i + 1] = f.y;
    }
}
__device__ __forceinline__ void load8(const float* p, float o[8]) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    const float4 b = *reinterpret_cast<const float4*>(p + 4);
    o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w; o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
}

// One warp per token; each lane owns 8 consecutive columns per 256-column stripe.  The
// token's K expert rows of a stripe are loaded together (K 16-byte loads a lane in
// flight), then added in slot order.
template <typename TY, int K>
__global__ void __launch_bounds__(256)
combine_kernel(const TY* __restrict__ y_perm, const int32_t* __restrict__ inv,
               const float* __restrict__ gates, int T, int d, long long R,
               float* __restrict__ y) {
    griddep_wait();
    griddep_launch_dependents();
    const int lane = threadIdx.x & 31;
    const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
    for (long long t = warp; t < T; t += nwarps) {
        int32_t pos[K];
        float g[K];
#pragma unroll
        for (int j = 0; j < K; ++j) {
            pos[j] = inv[t * K + j];
            g[j] = gates[t * K + j];
        }
        for (int c = lane * 8; c < d; c += 256) {
            float v[K][8];
#pragma unroll
            for (int j = 0; j < K; ++j) {
                if (pos[j] >= 0 && pos[j] < R) {
                    load8(y_perm + (size_t)pos[j] * d + c, v[j]);
                } else {                           // only after a reported bad idx
#pragma unroll
                    for (int q = 0; q < 8; ++q) v[j][q] = 0.0f;
                }
            }
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int j = 0; j < K; ++j) {
                if (pos[j] < 0 || pos[j] >= R) continue;
#pragma unroll
                for (int q = 0; q < 8; ++q) acc[q] = fmaf(g[j], v[j][q], acc[q]);
            }
            float4* out = reinterpret_cast<float4*>(y + (size_t)t * d + c);
            out[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
            out[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
        }
    }
}

template <typename TY>
cudaError_t launch_k(const TY* y_perm, const int32_t* inv, const float* gates, int T, int k, int d,
                     long long R, float* y, unsigned blocks, cudaStream_t s) {
    switch (k) {
#define MOE_COMBINE_CASE(K)                                                                     \
    case K:                                                                                     \
        return launch_pdl(combine_kernel<TY, K>, dim3(blocks), dim3(256), 0, s, 1, y_perm, inv, \
                          gates, T, d, R, y);
        MOE_COMBINE_CASE(1) MOE_COMBINE_CASE(2) MOE_COMBINE_CASE(3) MOE_COMBINE_CASE(4)
        MOE_COMBINE_CASE(5) MOE_COMBINE_CASE(6) MOE_COMBINE_CASE(7) MOE_COMBINE_CASE(8)
#undef MOE_COMBINE_CASE
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_combine(const void* y_perm, bool half_rows, const int32_t* inv,
                           const float* gates, int T, int k, int d, float* y, cudaStream_t s) {
    long long blocks = ((long long)T + 7) / 8;
    if (blocks > 148 * 16) blocks = 148 * 16;
    if (blocks < 1) blocks = 1;
    const long long R = (long long)T * k;
    const cudaError_t e =
        half_rows ? launch_k(static_cast<const __half*>(y_perm), inv, gates, T, k, d, R, y,
                             (unsigned)blocks, s)
                  : launch_k(static_cast<const float*>(y_perm), inv, gates, T, k, d, R, y,
                             (unsigned)blocks, s);
    note_launch();
    return e;
}

}  // namespace moe
