// Fixed-order reductions shared by the balancing losses (balance.cu) and the dispatch's
// column scan (dispatch.cu), which forms the forward pass's losses in its last CTA.
//
// "Mixture of Experts: Outrageously Large Neural Networks" (intuitivepapers.ai):
// Importance and Load are batch sums (eqs (6), (10)); the losses are CV^2 = population
// variance / mean^2 of each (eq (7)).  Every sum below runs in a fixed order, so the
// results are bitwise reproducible, and every path that forms them (the forward pass,
// moe_gate, moe_balance_losses, moe_losses_from_sums, the hierarchical layer) uses these
// functions with 512-thread CTAs, so they agree bit for bit.  B300 issues fp64 at a
// small fraction of its fp32 rate, so the sums are fp32: plain for an expert's few
// hundred per-tile partials, compensated for the CV^2.
#pragma once

#include <stdint.h>

#include "common.cuh"

namespace moe {

constexpr int RED_WARPS = 16;                  // every CTA using these runs 512 threads

// Compensated fp32 sums.  A sum is carried as s + c: every addition is an exact two-sum
// whose rounding error goes into c (Neumaier's variant of Kahan summation), so a sum of
// up to a few ten thousand terms keeps about fp32's relative precision.
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

// Sum over the 16 warps of the CTA: a fixed butterfly inside each warp, then thread 0
// merges the 16 warp results in warp order.  red: 17 CSum slots of shared memory.
__device__ __forceinline__ float block16_sum(CSum v, CSum* red) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const CSum o = {__shfl_xor_sync(0xffffffffu, v.s, off),
                        __shfl_xor_sync(0xffffffffu, v.c, off)};
        v = (threadIdx.x & off) ? cmerge(o, v) : cmerge(v, o);   // lower lane first
    }
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    if (threadIdx.x == 0) {
        CSum t = red[0];
#pragma unroll
        for (int w = 1; w < RED_WARPS; ++w) t = cmerge(t, red[w]);
        red[RED_WARPS] = t;
    }
    __syncthreads();
    const CSum r = red[RED_WARPS];
    __syncthreads();                               // red is free for the next call
    return r.s + r.c;
}

// w_imp c0 + w_load c1 with every rounding explicit (no contraction into an FMA), so
// each kernel that forms the losses gets the same bits.
__device__ __forceinline__ float weighted_losses(float w_imp, float c0, float w_load, float c1) {
    return __fadd_rn(__fmul_rn(w_imp, c0), __fmul_rn(w_load, c1));
}

// CV^2 of v[0..n) by the CTA's 512 threads (every thread calls it): the mean first, then
// the squared deviations from it (each deviation v - mean carries one fp32 rounding, so
// the CV^2 keeps fp32's relative precision even for nearly equal v).  With sw: the Switch
// loss scale * sum_i v_i other_i ("From LSTMs to Switch and Mixtral": one loss on the
// product of each expert's token fraction and mean gate probability, scale = n / (routed
// rows * tokens)).  Zero mean or n = 1 gives 0.
__device__ __forceinline__ float cv2_512(const float* __restrict__ v,
                                         const float* __restrict__ other, int n, bool sw,
                                         double scale, CSum* red) {
    CSum s = {0.0f, 0.0f};
    for (int i = threadIdx.x; i < n; i += 32 * RED_WARPS) s = cadd(s, sw ? v[i] * other[i] : v[i]);
    const float s_tot = block16_sum(s, red);
    if (sw) return (float)((double)s_tot * scale);
    const float mean = s_tot / (float)n;
    CSum q = {0.0f, 0.0f};
    for (int i = threadIdx.x; i < n; i += 32 * RED_WARPS) {
        const float dv = v[i] - mean;
        q = cadd(q, dv * dv);
    }
    const float q_tot = block16_sum(q, red);
    if (n <= 1 || mean == 0.0f) return 0.0f;
    return (q_tot / (float)n) / (mean * mean);
}

// losses = (CV^2(importance), CV^2(load), w_imp CV^2(importance) + w_load CV^2(load)), or
// with switch_scale > 0 (L_switch, 0, w_imp L_switch), by the CTA's 512 threads.
__device__ __forceinline__ void losses_512(const float* __restrict__ importance,
                                           const float* __restrict__ load, int n, float w_imp,
                                           float w_load, double switch_scale,
                                           float* __restrict__ losses) {
    __shared__ CSum red[RED_WARPS + 1];
    const bool sw = switch_scale > 0.0;
    const float c0 = cv2_512(importance, load, n, sw, switch_scale, red);
    const float c1 = sw ? 0.0f : cv2_512(load, nullptr, n, false, 0.0, red);
    if (threadIdx.x == 0) {
        losses[0] = c0;
        losses[1] = c1;
        losses[2] = weighted_losses(w_imp, c0, w_load, c1);
    }
}

// The fixed pairwise tree over the 16 warps' partial sums part_l / part_i [16][33]
// (written before the call, the barrier inside makes them visible): warp 0 adds them for
// expert e = e0 + lane and writes load[e] and importance[e] (importance may be null).
// Every thread of the 512-thread CTA calls it.
__device__ __forceinline__ void tile_sums_tree(const float (*part_l)[33], const float (*part_i)[33],
                                               int n, int e0, float* __restrict__ load,
                                               float* __restrict__ importance) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int e = e0 + lane;
    __syncthreads();
    if (wid == 0 && e < n) {
        float tl[RED_WARPS], ti[RED_WARPS];
#pragma unroll
        for (int w = 0; w < RED_WARPS; ++w) { tl[w] = part_l[w][lane]; ti[w] = part_i[w][lane]; }
#pragma unroll
        for (int h = RED_WARPS / 2; h > 0; h >>= 1)
#pragma unroll
            for (int w = 0; w < h; ++w) { tl[w] += tl[w + h]; ti[w] += ti[w + h]; }
        load[e] = tl[0];
        if (importance != nullptr) importance[e] = ti[0];
    }
    __syncthreads();
}

// load[e] and importance[e] (imp_part may be null) for the 32 experts e = e0 + lane of
// this CTA from per-tile partials [chunks][n]: warp w sums the tiles of its contiguous
// span [w span, (w+1) span), span = ceil(chunks / 16), in ascending order (fp32), and
// warp 0 adds the 16 warps' sums in a fixed pairwise tree (a sum of at most a few hundred
// fp32 terms in this order stays within 1e-6 relative).  Every warp load reads 32
// consecutive floats of one tile's partials.
__device__ __forceinline__ void tile_sums_512(const float* __restrict__ load_part,
                                              const float* __restrict__ imp_part, int chunks,
                                              int n, int e0, float* __restrict__ load,
                                              float* __restrict__ importance) {
    __shared__ float part_l[RED_WARPS][33], part_i[RED_WARPS][33];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int e = e0 + lane;
    const int span = (chunks + RED_WARPS - 1) / RED_WARPS;
    const int t0 = min(chunks, wid * span), t1 = min(chunks, t0 + span);
    float sl = 0.0f, si = 0.0f;
    if (e < n) {
#pragma unroll 4
        for (int c = t0; c < t1; ++c) {
            sl += load_part[(size_t)c * n + e];
            if (imp_part != nullptr) si += imp_part[(size_t)c * n + e];
        }
    }
    part_l[wid][lane] = sl;
    part_i[wid][lane] = si;
    tile_sums_tree(part_l, part_i, n, e0, load, importance);
}

}  // namespace moe
