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

__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// CV^2 of v[0..n) by one warp in fp64: lane-strided sums, then a fixed butterfly.
__device__ double warp_cv2(const float* __restrict__ v, int n) {
    const int lane = threadIdx.x & 31;
    double s = 0.0;
    for (int i = lane; i < n; i += 32) s += (double)v[i];
    const double mean = warp_sum(s) / n;
    double q = 0.0;
    for (int i = lane; i < n; i += 32) {
        const double dv = (double)v[i] - mean;
        q += dv * dv;
    }
    const double var = warp_sum(q) / n;
    if (n <= 1 || mean == 0.0) return 0.0;
    return var / (mean * mean);
}

// The Switch balancing loss ("From LSTMs to Switch and Mixtral": one loss on the
// product of each expert's token fraction and mean gate probability):
// scale * sum_i load_i importance_i, with scale = n / (routed rows * tokens), so that
// f_i = load_i / rows and P_i = importance_i / tokens; fp64, lane-strided, fixed butterfly.
__device__ double warp_switch_loss(const float* __restrict__ importance,
                                   const float* __restrict__ load, int n, double scale) {
    const int lane = threadIdx.x & 31;
    double s = 0.0;
    for (int i = lane; i < n; i += 32) s += (double)load[i] * (double)importance[i];
    return warp_sum(s) * scale;
}

// losses = (CV^2(importance), CV^2(load), w_imp * CV^2(importance) + w_load * CV^2(load)),
// or with switch_scale > 0 (the Switch gate) (L_switch, 0, w_imp * L_switch).
// Warp 0 takes the importance, warp 1 the load.
__global__ void __launch_bounds__(64)
cv2_losses_kernel(const float* __restrict__ importance, const float* __restrict__ load, int n,
                  float w_imp, float w_load, double switch_scale, float* __restrict__ losses) {
    griddep_wait();
    griddep_launch_dependents();
    __shared__ double cv[2];
    const int w = threadIdx.x >> 5;
    const double c = switch_scale > 0.0
                         ? (w == 0 ? warp_switch_loss(importance, load, n, switch_scale) : 0.0)
                         : warp_cv2(w == 0 ? importance : load, n);
    if ((threadIdx.x & 31) == 0) cv[w] = c;
    __syncthreads();
    if (threadIdx.x == 0) {
        losses[0] = (float)cv[0];
        losses[1] = (float)cv[1];
        losses[2] = (float)((double)w_imp * cv[0] + (double)w_load * cv[1]);
    }
}

// The end of the forward pass in one launch.  A CTA owns 32 experts (lane = expert) and
// its 32 warps split the token tiles (warp w takes tiles w, w + 32, ...), so every warp
// load reads 32 consecutive floats of one tile's partials; each (warp, expert) sum is
// fp64 in ascending tile order, then warp 0 adds the 32 warps' sums in warp order (a
// fixed order: the results are bitwise reproducible).  The last CTA to finish (a ticket
// counter, zeroed by the gate kernel before this launch and again by that CTA) forms the
// CV^2 losses.
constexpr int TAIL_WARPS = 32;

__global__ void __launch_bounds__(32 * TAIL_WARPS)
forward_tail_kernel(const float* __restrict__ load_part, const float* __restrict__ imp_part,
                    int chunks, int n, float* __restrict__ load, float* __restrict__ importance,
                    float w_imp, float w_load, double switch_scale, float* __restrict__ losses,
                    unsigned* __restrict__ ticket) {
    griddep_wait();
    griddep_launch_dependents();
    __shared__ double part_l[TAIL_WARPS][33], part_i[TAIL_WARPS][33];
    __shared__ bool last;
    __shared__ double cv[2];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int e = blockIdx.x * 32 + lane;
    double sl = 0.0, si = 0.0;
    if (e < n) {
#pragma unroll 4
        for (int c = wid; c < chunks; c += TAIL_WARPS) {
            sl += (double)load_part[(size_t)c * n + e];
            si += (double)imp_part[(size_t)c * n + e];
        }
    }
    part_l[wid][lane] = sl;
    part_i[wid][lane] = si;
    __syncthreads();
    if (wid == 0 && e < n) {
        double tl = 0.0, ti = 0.0;
#pragma unroll 8
        for (int w = 0; w < TAIL_WARPS; ++w) {
            tl += part_l[w][lane];
            ti += part_i[w][lane];
        }
        load[e] = (float)tl;
        importance[e] = (float)ti;
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) last = atomicAdd(ticket, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!last) return;
    __threadfence();                       // every CTA's sums are visible
    if (wid < 2) {
        const double c = switch_scale > 0.0
                             ? (wid == 0 ? warp_switch_loss(importance, load, n, switch_scale) : 0.0)
                             : warp_cv2(wid == 0 ? importance : load, n);
        if (lane == 0) cv[wid] = c;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        losses[0] = (float)cv[0];
        losses[1] = (float)cv[1];
        losses[2] = (float)((double)w_imp * cv[0] + (double)w_load * cv[1]);
        *ticket = 0u;                      // ready for the next call
    }
}

}  // namespace

cudaError_t launch_forward_tail(const float* load_part, const float* imp_part, int chunks, int n,
                                float* load, float* importance, float w_imp, float w_load,
                                float* losses, unsigned* ticket, cudaStream_t s,
                                double switch_scale) {
    const cudaError_t e =
        launch_pdl(forward_tail_kernel, dim3((n + 31) / 32), dim3(32 * TAIL_WARPS), 0, s, 1,
                   load_part, imp_part, chunks, n, load, importance, w_imp, w_load, switch_scale,
                   losses, ticket);
    note_launch();
    return e;
}

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
        launch_pdl(cv2_losses_kernel, dim3(1), dim3(64), 0, s, 1, importance, load, n, w_imp,
                   w_load, switch_scale, losses);
    note_launch();
    return e;
}

}  // namespace moe
