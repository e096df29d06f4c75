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

// The end of the forward pass in one launch.  A CTA owns 32 experts (lane = expert) and
// its 32 warps split the token tiles (warp w takes tiles w, w + 32, ...), so every warp
// load reads 32 consecutive floats of one tile's partials.  Each (warp, expert) sum is
// fp32 in ascending tile order; warp 0 then adds the 32 warps' sums in a fixed pairwise
// tree (fp32: B300's fp64 rate is a small fraction of its fp32 rate, and a sum of at most
// a few hundred fp32 terms in this order stays within 1e-6 relative).  The order is fixed,
// so the results are bitwise reproducible.  The last CTA to finish (a ticket counter,
// zeroed by the gate kernel before this launch and again by that CTA) forms the losses
// with 16 warps a vector (fp64 partials over slices of the experts, added in order).
constexpr int TAIL_WARPS = 32;

// Sum of v over the 16 warps of group slot / 16 of a 1024-thread CTA: a butterfly inside
// each warp, then one thread a group adds the 16 warp results in warp order (fp64 issues
// at a small fraction of the fp32 rate on B300, so no other thread repeats that sum).
// red: 34 doubles of shared memory.
__device__ __forceinline__ double block16_sum(double v, double* red, int slot) {
    v = warp_sum(v);
    if ((threadIdx.x & 31) == 0) red[slot] = v;
    __syncthreads();
    if ((threadIdx.x & 511) == 0) {
        const int g0 = (slot / 16) * 16;
        double t = 0.0;
#pragma unroll
        for (int w = 0; w < 16; ++w) t += red[g0 + w];
        red[32 + slot / 16] = t;
    }
    __syncthreads();
    return red[32 + slot / 16];
}

// The Switch balancing loss ("From LSTMs to Switch and Mixtral": one loss on the product
// of each expert's token fraction and mean gate probability) is
// scale * sum_i load_i importance_i with scale = n / (routed rows * tokens), so that
// f_i = load_i / rows and P_i = importance_i / tokens.
//
// CV^2 of v[0..n), or with sw the Switch loss scale * sum_i v_i other_i, by the 16 warps
// of group g (0 or 1) of a 1024-thread CTA: every thread of the CTA calls this once, and
// each call makes exactly two block16_sum calls, so the CTA's barriers line up.
__device__ double group_cv2(const float* __restrict__ v, const float* __restrict__ other, int n,
                            bool sw, double scale, double* red, int g) {
    const int gw = (threadIdx.x >> 5) & 15;
    const int i0 = gw * 32 + (threadIdx.x & 31);
    double s = 0.0;
    for (int i = i0; i < n; i += 16 * 32) s += sw ? (double)v[i] * (double)other[i] : (double)v[i];
    const double s_tot = block16_sum(s, red, 16 * g + gw);
    const double mean = s_tot / n;
    double q = 0.0;
    if (!sw)
        for (int i = i0; i < n; i += 16 * 32) {
            const double dv = (double)v[i] - mean;
            q += dv * dv;
        }
    const double q_tot = block16_sum(q, red, 16 * g + gw);
    if (sw) return s_tot * scale;
    if (n <= 1 || mean == 0.0) return 0.0;
    return (q_tot / n) / (mean * mean);
}

// load[e] and importance[e] (imp_part may be null) for the 32 experts of this CTA: sums
// over the tiles' partials in the fixed order described above.
__device__ __forceinline__ void tile_sums32(const float* __restrict__ load_part,
                                            const float* __restrict__ imp_part, int chunks, int n,
                                            float* __restrict__ load,
                                            float* __restrict__ importance) {
    __shared__ float part_l[TAIL_WARPS][33], part_i[TAIL_WARPS][33];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int e = blockIdx.x * 32 + lane;
    float sl = 0.0f, si = 0.0f;
    if (e < n) {
#pragma unroll 4
        for (int c = wid; c < chunks; c += TAIL_WARPS) {
            sl += load_part[(size_t)c * n + e];
            if (imp_part != nullptr) si += imp_part[(size_t)c * n + e];
        }
    }
    part_l[wid][lane] = sl;
    part_i[wid][lane] = si;
    __syncthreads();
    if (wid == 0 && e < n) {
        float tl[TAIL_WARPS], ti[TAIL_WARPS];
#pragma unroll
        for (int w = 0; w < TAIL_WARPS; ++w) { tl[w] = part_l[w][lane]; ti[w] = part_i[w][lane]; }
#pragma unroll
        for (int h = TAIL_WARPS / 2; h > 0; h >>= 1)
#pragma unroll
            for (int w = 0; w < h; ++w) { tl[w] += tl[w + h]; ti[w] += ti[w + h]; }
        load[e] = tl[0];
        if (importance != nullptr) importance[e] = ti[0];
    }
}

// The losses from the finished load / importance vectors by the whole 1024-thread CTA:
// warps 0-15 the importance's CV^2 (or the Switch loss), warps 16-31 the load's.
__device__ __forceinline__ void losses_block(const float* __restrict__ importance,
                                             const float* __restrict__ load, int n, float w_imp,
                                             float w_load, double switch_scale,
                                             float* __restrict__ losses) {
    __shared__ double red[34];
    const int g = (threadIdx.x >> 5) >= 16 ? 1 : 0;
    const bool sw = switch_scale > 0.0;
    const double c = group_cv2(g ? load : importance, load, n, sw && g == 0, switch_scale, red, g);
    if ((threadIdx.x & 511) == 0) red[16 * g] = (sw && g == 1) ? 0.0 : c;
    __syncthreads();
    if (threadIdx.x == 0) {
        const double c0 = red[0], c1 = red[16];
        losses[0] = (float)c0;
        losses[1] = (float)c1;
        losses[2] = (float)((double)w_imp * c0 + (double)w_load * c1);
    }
}

__global__ void __launch_bounds__(32 * TAIL_WARPS)
forward_tail_kernel(const float* __restrict__ load_part, const float* __restrict__ imp_part,
                    int chunks, int n, float* __restrict__ load, float* __restrict__ importance,
                    float w_imp, float w_load, double switch_scale, float* __restrict__ losses,
                    unsigned* __restrict__ ticket) {
    griddep_wait();
    griddep_launch_dependents();
    __shared__ bool last;
    tile_sums32(load_part, imp_part, chunks, n, load, importance);
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) last = atomicAdd(ticket, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!last) return;
    __threadfence();                       // every CTA's sums are visible
    losses_block(importance, load, n, w_imp, w_load, switch_scale, losses);
    if (threadIdx.x == 0) *ticket = 0u;    // ready for the next call
}

// The same sums without the losses (moe_gate's Load and the Switch sums).
__global__ void __launch_bounds__(32 * TAIL_WARPS)
tile_reduce_kernel(const float* __restrict__ part, const float* __restrict__ imp_part, int chunks,
                   int n, float* __restrict__ load, float* __restrict__ importance) {
    griddep_wait();
    griddep_launch_dependents();
    tile_sums32(part, imp_part, chunks, n, load, importance);
}

// losses = (CV^2(importance), CV^2(load), w_imp * CV^2(importance) + w_load * CV^2(load)),
// or with switch_scale > 0 (the Switch gate) (L_switch, 0, w_imp * L_switch): the same
// computation, in the same order, as the forward pass's tail.
__global__ void __launch_bounds__(32 * TAIL_WARPS)
cv2_losses_kernel(const float* __restrict__ importance, const float* __restrict__ load, int n,
                  float w_imp, float w_load, double switch_scale, float* __restrict__ losses) {
    griddep_wait();
    griddep_launch_dependents();
    losses_block(importance, load, n, w_imp, w_load, switch_scale, losses);
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
        launch_pdl(cv2_losses_kernel, dim3(1), dim3(32 * TAIL_WARPS), 0, s, 1, importance, load,
                   n, w_imp, w_load, switch_scale, losses);
    note_launch();
    return e;
}

cudaError_t launch_partial_reduce(const float* part, const float* imp_part, int chunks, int n,
                                  float* load, float* importance, cudaStream_t s) {
    const cudaError_t e = launch_pdl(tile_reduce_kernel, dim3((n + 31) / 32), dim3(32 * TAIL_WARPS),
                                     0, s, 1, part, imp_part, chunks, n, load, importance);
    note_launch();
    return e;
}

}  // namespace moe
