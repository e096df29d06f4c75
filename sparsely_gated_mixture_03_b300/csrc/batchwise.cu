// The batchwise top-m gate: each expert takes exactly the m = floor(k T / n) tokens of
// the batch with its largest noisy logits.
//
// "Mixture of Experts: Outrageously Large Neural Networks" (intuitivepapers.ai), "What
// the paper measured": the single-pair translation models use the gate of Appendix F,
// in which during training each expert takes exactly the top m = k |X| / n inputs of the
// batch, so every expert gets the same batch size.  Readings: the score is the noisy
// logit H of eq (4); an expert ranks tokens by H, larger first, equal H -> lower token
// index; a token's gates over the experts that took it are the softmax of their H; a
// token no expert took gets y = 0.
//
// Kernels: the logits transposed to [n, T] (coalesced columns); one CTA an expert finds
// its m-th largest logit by a four-pass radix select on order-preserving 32-bit keys and
// writes its tokens in ascending order (sel, and rowmap [T, n] = the routed row or -1),
// the ties at the m-th value going to the lowest token indices; one warp a token forms
// the softmax over the experts that took it; the expert-major rows are copied to x_perm
// (each expert's segment is exactly m rows, offsets e m); after the grouped FFN one warp a
// token adds its experts' outputs in ascending expert order.
//
// Inference mode (the learned per-expert threshold that replaces the batch-wise choice):
// expert i takes the tokens with H > threshold_i, so its segment length varies: one CTA
// an expert counts them, one CTA scans the counts into offsets (clamped to the rows the
// workspace holds, an excess reported as DEV_RANGE), one CTA an expert writes its tokens
// in ascending order at offsets[i] + rank; the rest is the training mode's.
#include <stdint.h>

#include "common.cuh"
#include "launch.h"

namespace moe {
namespace {

// Order-preserving map of a float to an unsigned key (larger float -> larger key; -0
// and +0, equal as floats, get the same key).
__device__ __forceinline__ uint32_t float_key(float f) {
    const uint32_t u0 = __float_as_uint(f);
    const uint32_t u = u0 == 0x80000000u ? 0u : u0;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Ht[i][t] = H[t][i], 32 x 32 tiles through shared memory.
__global__ void __launch_bounds__(256)
transpose_kernel(const float* __restrict__ H, int T, int n, float* __restrict__ Ht) {
    griddep_wait();
    griddep_launch_dependents();
    __shared__ float tile[32][33];
    const int t0 = blockIdx.x * 32, i0 = blockIdx.y * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;   // 32 x 8
    for (int r = ty; r < 32; r += 8) {
        const int t = t0 + r, i = i0 + tx;
        tile[r][tx] = (t < T && i < n) ? H[(size_t)t * n + i] : 0.0f;
    }
    __syncthreads();
    for (int r = ty; r < 32; r += 8) {
        const int i = i0 + r, t = t0 + tx;
        if (i < n && t < T) Ht[(size_t)i * T + t] = tile[tx][r];
    }
}

__global__ void fill_kernel(int32_t* __restrict__ p, long long count, int32_t v) {
    griddep_wait();
    griddep_launch_dependents();
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < count;
         i += (long long)gridDim.x * blockDim.x)
        p[i] = v;
}

constexpr int TM_THREADS = 1024;

// Block-wide exclusive scan of v over the 1024 threads; *total receives the sum.
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) warp_sums[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        int w = warp_sums[lane];
        int wi = w;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, wi, off);
            if (lane >= off) wi += o;
        }
        warp_sums[lane] = wi - w;                 // exclusive over warps
        if (lane == 31) warp_sums[32] = wi;       // block total
    }
    __syncthreads();
    const int r = warp_sums[wid] + incl - v;
    *total = warp_sums[32];
    __syncthreads();                              // warp_sums is reused by the next call
    return r;
}

// One CTA an expert: the m tokens with its largest logits, ascending token order.
__global__ void __launch_bounds__(TM_THREADS)
expert_topm_kernel(const float* __restrict__ Ht, int T, int n, int m, int32_t* __restrict__ sel,
                   int32_t* __restrict__ rowmap) {
    griddep_wait();
    griddep_launch_dependents();
    __shared__ int hist[256];
    __shared__ int warp_sums[33];
    __shared__ uint32_t s_prefix;
    __shared__ int s_want;
    const int tid = threadIdx.x;
    const int i = blockIdx.x;
    const float* col = Ht + (size_t)i * T;
    uint32_t prefix = 0, mask = 0;
    int want = m;
    // radix select, 8 bits a pass from the top: the key of the m-th largest logit
    for (int shift = 24; shift >= 0; shift -= 8) {
        if (tid < 256) hist[tid] = 0;
        __syncthreads();
        for (int t = tid; t < T; t += TM_THREADS) {
            const uint32_t key = float_key(col[t]);
            if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1);
        }
        __syncthreads();
        if (tid == 0) {
            int acc = 0, b = 255;
            for (; b > 0; --b) {
                if (acc + hist[b] >= want) break;
                acc += hist[b];
            }
            s_prefix = prefix | ((uint32_t)b << shift);
            s_want = want - acc;
        }
        __syncthreads();
        prefix = s_prefix;
        want = s_want;
        mask |= 0xffu << shift;
        __syncthreads();
    }
    // prefix: the m-th largest key; want: how many keys equal to it are taken (lowest
    // token indices first).  Compaction in token order.
    int carry_tie = 0, carry_take = 0;
    for (int t0 = 0; t0 < T; t0 += TM_THREADS) {
        const int t = t0 + tid;
        const uint32_t key = t < T ? float_key(col[t]) : 0u;
        const int gt = (t < T && key > prefix) ? 1 : 0;
        const int eq = (t < T && key == prefix) ? 1 : 0;
        int tot_eq = 0, tot_take = 0;
        const int tie_rank = carry_tie + block_exclusive_scan(eq, warp_sums, &tot_eq);
        const int take = (gt || (eq && tie_rank < want)) ? 1 : 0;
        const int pos = carry_take + block_exclusive_scan(take, warp_sums, &tot_take);
        if (take && pos < m) {
            sel[(size_t)i * m + pos] = t;
            rowmap[(size_t)t * n + i] = i * m + pos;
        }
        carry_tie += tot_eq;
        carry_take += tot_take;
    }
}

// One CTA an expert: how many tokens have H > threshold[i].
__global__ void __launch_bounds__(TM_THREADS)
threshold_count_kernel(const float* __restrict__ Ht, int T, const float* __restrict__ threshold,
                       int32_t* __restrict__ counts) {
    griddep_wait();
    griddep_launch_dependents();
    __shared__ int warp_c[TM_THREADS / 32];
    const int i = blockIdx.x;
    const float thr = threshold[i];
    const float* col = Ht + (size_t)i * T;
    int c = 0;
    for (int t = threadIdx.x; t < T; t += TM_THREADS) c += col[t] > thr ? 1 : 0;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) c += __shfl_xor_sync(0xffffffffu, c, off);
    if ((threadIdx.x & 31) == 0) warp_c[threadIdx.x >> 5] = c;
    __syncthreads();
    if (threadIdx.x == 0) {
        int tot = 0;
        for (int w = 0; w < TM_THREADS / 32; ++w) tot += warp_c[w];
        counts[i] = tot;
    }
}

// One CTA: offsets = exclusive prefix of the counts, each clamped to cap (the rows the
// workspace holds); more than cap rows in all sets DEV_RANGE.
__global__ void __launch_bounds__(TM_THREADS)
threshold_offsets_kernel(const int32_t* __restrict__ counts, int n, long long cap,
                         int32_t* __restrict__ offsets, int* err) {
    griddep_wait();
    griddep_launch_dependents();
    __shared__ int warp_sums[33];
    long long carry = 0;
    for (int e0 = 0; e0 < n; e0 += TM_THREADS) {
        const int e = e0 + threadIdx.x;
        const int v = e < n ? counts[e] : 0;
        int tot = 0;
        const long long ex = carry + block_exclusive_scan(v, warp_sums, &tot);
        if (e < n) offsets[e] = (int32_t)(ex < cap ? ex : cap);
        carry += tot;
    }
    if (threadIdx.x == 0) {
        offsets[n] = (int32_t)(carry < cap ? carry : cap);
        if (carry > cap) raise_error(err, DEV_RANGE);
    }
}

// One CTA an expert: its tokens with H > threshold[i], ascending, at offsets[i] + rank
// (rows past offsets[i+1], cut by the capacity clamp, are not written).
__global__ void __launch_bounds__(TM_THREADS)
threshold_select_kernel(const float* __restrict__ Ht, int T, int n,
                        const float* __restrict__ threshold, const int32_t* __restrict__ offsets,
                        int32_t* __restrict__ sel, int32_t* __restrict__ rowmap) {
    griddep_wait();
    griddep_launch_dependents();
    __shared__ int warp_sums[33];
    const int i = blockIdx.x;
    const float thr = threshold[i];
    const float* col = Ht + (size_t)i * T;
    const int p0 = offsets[i], p1 = offsets[i + 1];
    int carry = 0;
    for (int t0 = 0; t0 < T; t0 += TM_THREADS) {
        const int t = t0 + threadIdx.x;
        const int take = (t < T && col[t] > thr) ? 1 : 0;
        int tot = 0;
        const int p = p0 + carry + block_exclusive_scan(take, warp_sums, &tot);
        if (take && p < p1) {
            sel[p] = t;
            rowmap[(size_t)t * n + i] = p;
        }
        carry += tot;
    }
}

// One warp a token: the softmax of H over the experts that took it (lane-strided sums,
// fixed butterfly); gates_r[r] for each of its routed rows r.
__global__ void __launch_bounds__(256)
token_gates_kernel(const float* __restrict__ H, const int32_t* __restrict__ rowmap, int T, int n,
                   float* __restrict__ gates_r) {
    griddep_wait();
    griddep_launch_dependents();
    const int lane = threadIdx.x & 31;
    const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
    for (long long t = warp; t < T; t += nwarps) {
        const float* hr = H + (size_t)t * n;
        const int32_t* rr = rowmap + (size_t)t * n;
        float mx = -INFINITY;
        for (int i = lane; i < n; i += 32)
            if (rr[i] >= 0) mx = fmaxf(mx, hr[i]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        if (mx == -INFINITY) continue;            // no expert took this token
        float s = 0.0f;
        for (int i = lane; i < n; i += 32)
            if (rr[i] >= 0) s += expf(hr[i] - mx);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        const float inv = 1.0f / s;
        for (int i = lane; i < n; i += 32)
            if (rr[i] >= 0) gates_r[rr[i]] = expf(hr[i] - mx) * inv;
    }
}

// One warp an expert: importance = the gates of its segment summed in order (fp64);
// load = the segment's rows.  Segments: [e m, (e+1) m), or [offsets[e], offsets[e+1])
// when offsets is given (the inference mode).
__global__ void __launch_bounds__(256)
batch_importance_kernel(const float* __restrict__ gates_r, int n, int m,
                        const int32_t* __restrict__ offsets, float* __restrict__ importance,
                        float* __restrict__ load) {
    griddep_wait();
    griddep_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int e = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (e >= n) return;
    const long long p0 = offsets != nullptr ? offsets[e] : (long long)e * m;
    const long long p1 = offsets != nullptr ? offsets[e + 1] : p0 + m;
    double s = 0.0;
    for (long long p = p0 + lane; p < p1; p += 32) s += (double)gates_r[p];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) {
        importance[e] = (float)s;
        load[e] = (float)(p1 - p0);
    }
}

// x_perm[r] = x[sel[r]] (one warp a row, 16-byte vectors).  Training: rows = n m and
// offsets[e] = e m are written here; inference (given_offsets): rows = offsets[n].
__global__ void __launch_bounds__(256)
batch_gather_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ sel, long long rows,
                    int row_vecs, uint4* __restrict__ out, int n, int m,
                    int32_t* __restrict__ offsets, int given_offsets) {
    griddep_wait();
    griddep_launch_dependents();
    const int lane = threadIdx.x & 31;
    const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
    if (given_offsets) {
        rows = offsets[n];
    } else if (warp == 0) {
        for (int e = lane; e <= n; e += 32) offsets[e] = e * m;
    }
    for (long long r = warp; r < rows; r += nwarps) {
        const int32_t t = sel[r];
        for (int v = lane; v < row_vecs; v += 32)
            out[(size_t)r * row_vecs + v] = x[(size_t)t * row_vecs + v];
    }
}

__device__ __forceinline__ float as_float(const __half* p) { return __half2float(*p); }
__device__ __forceinline__ float as_float(const float* p) { return *p; }

// One warp a token: y[t] = sum over the experts that took it, ascending expert index,
// of gates_r[r] y_perm[r] (fp32); 0 when none did.
template <typename TY>
__global__ void __launch_bounds__(256)
batch_combine_kernel(const TY* __restrict__ y_perm, const int32_t* __restrict__ rowmap,
                     const float* __restrict__ gates_r, int T, int n, int d,
                     float* __restrict__ y) {
    griddep_wait();
    griddep_launch_dependents();
    const int lane = threadIdx.x & 31;
    const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
    for (long long t = warp; t < T; t += nwarps) {
        const int32_t* rr = rowmap + (size_t)t * n;
        for (int c0 = 0; c0 < d; c0 += 32 * 8) {
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            for (int i0 = 0; i0 < n; i0 += 32) {
                const int32_t v = i0 + lane < n ? rr[i0 + lane] : -1;
                unsigned live = __ballot_sync(0xffffffffu, v >= 0);
                while (live != 0u) {
                    const int b = __ffs(live) - 1;
                    live &= live - 1u;
                    const int32_t r = __shfl_sync(0xffffffffu, v, b);
                    const float g = gates_r[r];
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const int c = c0 + lane * 8 + q;
                        if (c < d) acc[q] = fmaf(g, as_float(y_perm + (size_t)r * d + c), acc[q]);
                    }
                }
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int c = c0 + lane * 8 + q;
                if (c < d) y[(size_t)t * d + c] = acc[q];
            }
        }
    }
}

int warp_blocks(long long units) {
    long long b = (units + 7) / 8;
    if (b > 148 * 16) b = 148 * 16;
    return (int)(b < 1 ? 1 : b);
}

}  // namespace

cudaError_t launch_batch_select(const float* H, int T, int n, int m, float* Ht, int32_t* sel,
                                int32_t* rowmap, float* gates_r, float* importance, float* load,
                                cudaStream_t s) {
    cudaError_t e = launch_pdl(transpose_kernel, dim3((T + 31) / 32, (n + 31) / 32), dim3(256), 0,
                               s, 1, H, T, n, Ht);
    note_launch();
    if (e != cudaSuccess) return e;
    e = launch_pdl(fill_kernel, dim3(148 * 4), dim3(256), 0, s, 1, rowmap, (long long)T * n,
                   (int32_t)-1);
    note_launch();
    if (e != cudaSuccess) return e;
    e = launch_pdl(expert_topm_kernel, dim3(n), dim3(TM_THREADS), 0, s, 1,
                   static_cast<const float*>(Ht), T, n, m, sel, rowmap);
    note_launch();
    if (e != cudaSuccess) return e;
    e = launch_pdl(token_gates_kernel, dim3(warp_blocks(T)), dim3(256), 0, s, 1, H,
                   static_cast<const int32_t*>(rowmap), T, n, gates_r);
    note_launch();
    if (e != cudaSuccess) return e;
    e = launch_pdl(batch_importance_kernel, dim3((n + 7) / 8), dim3(256), 0, s, 1,
                   static_cast<const float*>(gates_r), n, m, static_cast<const int32_t*>(nullptr),
                   importance, load);
    note_launch();
    return e;
}

cudaError_t launch_threshold_select(const float* H, int T, int n, const float* threshold,
                                    long long cap, float* Ht, int32_t* counts, int32_t* offsets,
                                    int32_t* sel, int32_t* rowmap, float* gates_r,
                                    float* importance, float* load, int* err, cudaStream_t s) {
    cudaError_t e = launch_pdl(transpose_kernel, dim3((T + 31) / 32, (n + 31) / 32), dim3(256), 0,
                               s, 1, H, T, n, Ht);
    note_launch();
    if (e != cudaSuccess) return e;
    e = launch_pdl(fill_kernel, dim3(148 * 4), dim3(256), 0, s, 1, rowmap, (long long)T * n,
                   (int32_t)-1);
    note_launch();
    if (e != cudaSuccess) return e;
    e = launch_pdl(threshold_count_kernel, dim3(n), dim3(TM_THREADS), 0, s, 1,
                   static_cast<const float*>(Ht), T, threshold, counts);
    note_launch();
    if (e != cudaSuccess) return e;
    e = launch_pdl(threshold_offsets_kernel, dim3(1), dim3(TM_THREADS), 0, s, 1,
                   static_cast<const int32_t*>(counts), n, cap, offsets, err);
    note_launch();
    if (e != cudaSuccess) return e;
    e = launch_pdl(threshold_select_kernel, dim3(n), dim3(TM_THREADS), 0, s, 1,
                   static_cast<const float*>(Ht), T, n, threshold,
                   static_cast<const int32_t*>(offsets), sel, rowmap);
    note_launch();
    if (e != cudaSuccess) return e;
    e = launch_pdl(token_gates_kernel, dim3(warp_blocks(T)), dim3(256), 0, s, 1, H,
                   static_cast<const int32_t*>(rowmap), T, n, gates_r);
    note_launch();
    if (e != cudaSuccess) return e;
    e = launch_pdl(batch_importance_kernel, dim3((n + 7) / 8), dim3(256), 0, s, 1,
                   static_cast<const float*>(gates_r), n, 0, static_cast<const int32_t*>(offsets),
                   importance, load);
    note_launch();
    return e;
}

cudaError_t launch_batch_gather(const void* x, size_t row_bytes, const int32_t* sel, int n, int m,
                                void* x_perm, int32_t* offsets, cudaStream_t s,
                                long long given_rows_cap) {
    const bool given = given_rows_cap > 0;
    const long long rows = given ? given_rows_cap : (long long)n * m;
    const cudaError_t e =
        launch_pdl(batch_gather_kernel, dim3(warp_blocks(rows)), dim3(256), 0, s, 1,
                   static_cast<const uint4*>(x), sel, rows, (int)(row_bytes / 16),
                   static_cast<uint4*>(x_perm), n, m, offsets, given ? 1 : 0);
    note_launch();
    return e;
}

cudaError_t launch_batch_combine(const void* y_perm, bool half_rows, const int32_t* rowmap,
                                 const float* gates_r, int T, int n, int d, float* y,
                                 cudaStream_t s) {
    const cudaError_t e =
        half_rows ? launch_pdl(batch_combine_kernel<__half>, dim3(warp_blocks(T)), dim3(256), 0, s,
                               1, static_cast<const __half*>(y_perm), rowmap, gates_r, T, n, d, y)
                  : launch_pdl(batch_combine_kernel<float>, dim3(warp_blocks(T)), dim3(256), 0, s,
                               1, static_cast<const float*>(y_perm), rowmap, gates_r, T, n, d, y);
    note_launch();
    return e;
}

}  // namespace moe
