// Balancing losses of "Mixture of Experts: Outrageously Large Neural Networks"
// (intuitivepapers.ai):
//   section "Why experts collapse, and the balancing losses":
//     Importance(X)_e = sum_x G(x)_e (eq (6)); L_importance = w CV(Importance)^2 (eq (7)),
//     CV^2 = population variance / mean^2;
//   section "A differentiable count of examples": L_load = w CV(Load)^2 (eq (10)).
// Sums run in fixed orders (reduce.cuh), so the losses are bitwise reproducible.
#include <stdint.h>

#include "common.cuh"
#include "launch.h"
#include "reduce.cuh"

namespace moe {
namespace {

// One warp per expert: sum the gates of its rows in ascending routed-row order
// (lane-strided fp64 partials, then a fixed xor-butterfly).
__global__ void __launch_bounds__(256)
importance_kernel(const float* __restrict__ gates, const int32_t* __restrict__ perm,
                  const int32_t* __restrict__ offsets, int n, float* __restrict__ importance) {
    griddep_wait();
    griddep_launch_dependents();
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

// The sums without the losses (moe_gate's Load, the Switch sums, the hierarchical
// layer's primary vectors): the order of tile_sums_512, which the dispatch's column scan
// also uses for the forward pass.
__global__ void __launch_bounds__(32 * RED_WARPS)
tile_reduce_kernel(const float* __restrict__ part, const float* __restrict__ imp_part, int chunks,
                   int n, float* __restrict__ load, float* __restrict__ importance) {
    griddep_wait();
    griddep_launch_dependents();
    tile_sums_512(part, imp_part, chunks, n, blockIdx.x * 32, load, importance);
}

// losses = (CV^2(importance), CV^2(load), w_imp * CV^2(importance) + w_load * CV^2(load)),
// or with switch_scale > 0 (the Switch gate) (L_switch, 0, w_imp * L_switch): the same
// computation, in the same order, as the forward pass's (losses_512).
__global__ void __launch_bounds__(32 * RED_WARPS)
cv2_losses_kernel(const float* __restrict__ importance, const float* __restrict__ load, int n,
                  float w_imp, float w_load, double switch_scale, float* __restrict__ losses) {
    griddep_wait();
    griddep_launch_dependents();
    losses_512(importance, load, n, w_imp, w_load, switch_scale, losses);
}

}  // namespace

cudaError_t launch_importance(const float* gates, const int32_t* perm, const int32_t* offsets,
                              int n, float* importance, cudaStream_t s) {
    const cudaError_t e = launch_pdl(importance_kernel, dim3((n + 7) / 8), dim3(256), 0, s, 1,
                                     gates, perm, offsets, n, importance);
    note_launch();
    return e;
}

cudaError_t launch_cv2_losses(const float* importance, const float* load, int n, float w_imp,
                              float w_load, float* losses, cudaStream_t s, double switch_scale) {
    const cudaError_t e =
        launch_pdl(cv2_losses_kernel, dim3(1), dim3(32 * RED_WARPS), 0, s, 1, importance, load,
                   n, w_imp, w_load, switch_scale, losses);
    note_launch();
    return e;
}

cudaError_t launch_partial_reduce(const float* part, const float* imp_part, int chunks, int n,
                                  float* load, float* importance, cudaStream_t s) {
    const cudaError_t e = launch_pdl(tile_reduce_kernel, dim3((n + 31) / 32), dim3(32 * RED_WARPS),
                                     0, s, 1, part, imp_part, chunks, n, load, importance);
    note_launch();
    return e;
}

}  // namespace moe
