// Balancing losses of "Mixture of Experts: Outrageously Large Neural Networks"
// (intuitivepapers.ai):
//   section "Why experts collapse, and the balancing losses":
//     Importance(X)_e = sum_x G(x)_e (eq (6)); L_importance = w CV(Importance)^2 (eq (7)),
//     CV^2 = population variance / mean^2;
//   section "A differentiable count of examples": L_load = w CV(Load)^2 (eq (10)).
// Sums run in fixed orders in fp64, so the losses are bitwise reproducible.
#include <stdint.h>

#include "common.cuh"
#include "launch.h"

namespace moe {
namespace {

// One warp per expert: sum the gates of its rows in ascending routed-row order
// (lane-strided fp64 partials, then a fixed xor-butterfly).
__global__ void __launch_bounds__(256)
importance_kernel(const float* __restrict__ gates, const int32_t* __restrict__ perm,
                  const int32_t* __restrict__ offsets, int n, float* __restrict__ importance) {
    const int lane = threadIdx.x & 31;
    const int e = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (e >= n) return;
    const int32_t p0 = offsets[e], p1 = offsets[e + 1];
    double s = 0.0;
    for (int32_t p = p0 + lane; p < p1; p += 32) s += (double)gates[perm[p]];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) importance[e] = (float)s;
}

__device__ double block_sum(double v, double* scratch) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    __syncthreads();
    if (lane == 0) scratch[wid] = v;
    __syncthreads();
    double t = 0.0;
    const int nw = blockDim.x >> 5;
    for (int w = 0; w < nw; ++w) t += scratch[w];
    return t;
}

__device__ double cv2_of(const float* v, int n, double* scratch) {
    double s = 0.0;
    for (int i = threadIdx.x; i < n; i += blockDim.x) s += (double)v[i];
    const double mean = block_sum(s, scratch) / n;
    double q = 0.0;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const double dv = (double)v[i] - mean;
        q += dv * dv;
    }
    const double var = block_sum(q, scratch) / n;
    if (n <= 1 || mean == 0.0) return 0.0;
    return var / (mean * mean);
}

// losses = (CV^2(importance), CV^2(load), w_imp * CV^2(importance) + w_load * CV^2(load)).
__global__ void __launch_bounds__(1024)
cv2_losses_kernel(const float* __restrict__ importance, const float* __restrict__ load, int n,
                  float w_imp, float w_load, float* __restrict__ losses) {
    __shared__ double scratch[32];
    const double ci = cv2_of(importance, n, scratch);
    const double cl = cv2_of(load, n, scratch);
    if (threadIdx.x == 0) {
        losses[0] = (float)ci;
        losses[1] = (float)cl;
        losses[2] = (float)((double)w_imp * ci + (double)w_load * cl);
    }
}

}  // namespace

cudaError_t launch_importance(const float* gates, const int32_t* perm, const int32_t* offsets,
                              int n, float* importance, cudaStream_t s) {
    importance_kernel<<<(n + 7) / 8, 256, 0, s>>>(gates, perm, offsets, n, importance); note_launch();
    return cudaGetLastError();
}

cudaError_t launch_cv2_losses(const float* importance, const float* load, int n, float w_imp,
                              float w_load, float* losses, cudaStream_t s) {
    cv2_losses_kernel<<<1, 1024, 0, s>>>(importance, load, n, w_imp, w_load, losses); note_launch();
    return cudaGetLastError();
}

}  // namespace moe
