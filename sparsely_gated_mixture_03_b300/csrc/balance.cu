// Balancing losses of "Mixture of Experts: Outrageously Large Neural Networks"
// (intuitivepapers.ai):
//   section "Why experts collapse, and the balancing losses":
//     Importance(X)_e = sum_x G(x)_e (eq (6)); L_importance = w CV(Importance)^2 (eq (7)),
//     CV^2 = population variance / mean^2;
//   section "A differentiable count of examples": L_load = w CV(Load)^2 (eq (10)).
// Sums run in fixed orders, so the losses are bitwise reproducible.  B300 issues fp64 at a
// small fraction of its fp32 rate, so the sums on the forward path are fp32: plain for
// the few hundred per-tile partials of an expert, compensated for the CV^2.
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

constexpr int TAIL_WARPS = 32;

// Compensated fp32 sums.  A sum is carried as s + c: every addition is an exact two-sum
// whose rounding error goes into c (Neumaier's variant of Kahan summation), so a sum of
// up to a few ten thousand terms keeps about fp32's relative precision whatever the
// number of terms.
struct CSum {
    float s, c;
};
__device__ __forceinline__ CSum two_sum(float a, float b) {
    const float s = a + b;
    const float bb = s - a;
    return {s, (a - (s - bb)) + (b - bb)};
}
__device__ __forceinline__ CSum cadd(CSum x, float v) {
    const CSum t = two_sum(x.s, v);
    return {t.s, x.c + t.c};
}
__device__ __forceinline__ CSum cmerge(CSum x, CSum y) {
    const CSum t = two_sum(x.s, y.s);
    return {t.s, (x.c + y.c) + t.c};
}

// Sum over the 16 warps of group g (0 or 1) of a 1024-thread CTA: a fixed butterfly
// inside each warp, then one thread a group merges the 16 warp results in warp order.
// red: 34 CSum slots of shared memory.
__device__ __forceinline__ float block16_sum(CSum v, CSum* red, int g) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const CSum o = {__shfl_xor_sync(0xffffffffu, v.s, off),
                        __shfl_xor_sync(0xffffffffu, v.c, off)};
        v = (threadIdx.x & off) ? cmerge(o, v) : cmerge(v, o);   // lower lane first
    }
    const int gw = (threadIdx.x >> 5) & 15;
    if ((threadIdx.x & 31) == 0) red[16 * g + gw] = v;
    __syncthreads();
    if ((threadIdx.x & 511) == 0) {
        CSum t = red[16 * g];
#pragma unroll
        for (int w = 1; w < 16; ++w) t = cmerge(t, red[16 * g + w]);
        red[32 + g] = t;
    }
    __syncthreads();
    const CSum r = red[32 + g];
    return r.s + r.c;
}

// The Switch balancing loss ("From LSTMs to Switch and Mixtral": one loss on the product
// of each expert's token fraction and mean gate probability) is
// scale * sum_i load_i importance_i with scale = n / (routed rows * tokens), so that
// f_i = load_i / rows and P_i = importance_i / tokens.
//
// CV^2 of v[0..n), or with sw the Switch loss scale * sum_i v_i other_i, by the 16 warps
// of group g of a 1024-thread CTA: every thread of the CTA calls this once, and each call
// makes exactly two block16_sum calls, so the CTA's barriers line up.  The mean first,
// then the squared deviations from it (each deviation v - mean carries one fp32
// rounding, so the CV^2 keeps fp32's relative precision even for nearly equal v).
__device__ float group_cv2(const float* __restrict__ v, const float* __restrict__ other, int n,
                           bool sw, double scale, CSum* red, int g) {
    const int gw = (threadIdx.x >> 5) & 15;
    const int i0 = gw * 32 + (threadIdx.x & 31);
    CSum s = {0.0f, 0.0f};
    for (int i = i0; i < n; i += 16 * 32) s = cadd(s, sw ? v[i] * other[i] : v[i]);
    const float s_tot = block16_sum(s, red, g);
    const float mean = s_tot / (float)n;
    CSum q = {0.0f, 0.0f};
    if (!sw)
        for (int i = i0; i < n; i += 16 * 32) {
            const float dv = v[i] - mean;
            q = cadd(q, dv * dv);
        }
    const float q_tot = block16_sum(q, red, g);
    if (sw) return (float)((double)s_tot * scale);
    if (n <= 1 || mean == 0.0f) return 0.0f;
    return (q_tot / (float)n) / (mean * mean);
}

// load[e] and importance[e] (imp_part may be null) for the 32 experts of this CTA: a CTA
// owns 32 experts (lane = expert) and its 32 warps split the token tiles (warp w takes
// tiles w, w + 32, ...), so every warp load reads 32 consecutive floats of one tile's
// partials; each (warp, expert) sum is fp32 in ascending tile order, and warp 0 adds the
// 32 warps' sums in a fixed pairwise tree (a sum of at most a few hundred fp32 terms in
// this order stays within 1e-6 relative).
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
    __shared__ CSum red[34];
    __shared__ float cv[2];
    const int g = (threadIdx.x >> 5) >= 16 ? 1 : 0;
    const bool sw = switch_scale > 0.0;
    const float c = group_cv2(g ? load : importance, load, n, sw && g == 0, switch_scale, red, g);
    if ((threadIdx.x & 511) == 0) cv[g] = (sw && g == 1) ? 0.0f : c;
    __syncthreads();
    if (threadIdx.x == 0) {
        losses[0] = cv[0];
        losses[1] = cv[1];
        losses[2] = w_imp * cv[0] + w_load * cv[1];
    }
}

// The end of the forward pass in one launch: the tile sums, then the last CTA to finish
// (a ticket counter, zeroed by the gate kernel before this launch and again by that CTA)
// forms the losses.
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
