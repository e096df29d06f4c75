// Backward pass of the layer: the exact derivative of the forward pass for the loss
//   L = sum(dy * y) + w_importance CV(Importance)^2 + w_load CV(Load)^2
// with the kept set held fixed.
//
// "Mixture of Experts: Outrageously Large Neural Networks" (intuitivepapers.ai),
// "Implementation notes": each expert gets gradient only from the rows routed to it,
// scaled by their gate values; W_g from the task loss through the softmax over the kept
// logits, from the importance loss by the same path, and from the load loss through the
// numerator of eq (9), also for experts that were not kept; W_noise through the noise
// term inside the kept logits and through the denominator of eq (9); the selection
// passes no gradient.  The load threshold kth_excluding(H, k, i) is the noisy logit of
// the expert at the k-th or (k+1)-th place, so its gradient reaches that expert's clean
// logit and noise std.  ReLU'(u) is taken as [hidden > 0] on the stored hidden layer.
//
// Kernels here: the CV^2 gradients, the combine's backward (gate gradients and the
// expert output gradients), the gate's elementwise backward (dclean, dnz, and their exact
// two-term bf16 split for the tensor cores), the gather of the expert input gradients
// into dx, the fixed-order reductions of the gate's weight-gradient partials, and a
// grouped CUDA-core GEMM with strided operands for the contractions the SM-pair kernels
// of ffn_pair.cu do not take (fp32 layers, shapes off their 256 grid, and the gate's
// share of dx).
#include <stdint.h>

#include "common.cuh"
#include "launch.h"
#include "reduce.cuh"

namespace moe {
namespace {

__device__ __forceinline__ float load_as_float(const float* p) { return *p; }
__device__ __forceinline__ float load_as_float(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ float load_as_float(const __half* p) { return __half2float(*p); }

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}
__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// g[i] = w * d CV(v)^2 / d v_i = w (2 / (n mean^2)) (v_i - mean - var / mean) (eq (7)),
// 0 when the mean is 0 or n = 1.  Warp 0: importance, warp 1: load; fp64 sums.
__global__ void __launch_bounds__(64)
cv2_grad_kernel(const float* __restrict__ importance, const float* __restrict__ load, int n,
                float w_imp, float w_load, float* __restrict__ g_imp, float* __restrict__ g_load) {
    griddep_wait();
    griddep_launch_dependents();
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float* v = w == 0 ? importance : load;
    float* g = w == 0 ? g_imp : g_load;
    const double wt = w == 0 ? w_imp : w_load;
    double s = 0.0;
    for (int i = lane; i < n; i += 32) s += (double)v[i];
    const double mu = warp_sum_d(s) / n;
    double q = 0.0;
    for (int i = lane; i < n; i += 32) {
        const double dv = (double)v[i] - mu;
        q += dv * dv;
    }
    const double var = warp_sum_d(q) / n;
    const bool zero = n <= 1 || mu == 0.0;
    const double c = zero ? 0.0 : wt * 2.0 / (n * mu * mu);
    for (int i = lane; i < n; i += 32)
        g[i] = zero ? 0.0f : (float)(c * ((double)v[i] - mu - var / mu));
}

// One warp per token: dG[t,j] = <dy_t, y_perm[p]> (the expert output's share of the
// gate's gradient, eq (1)) and dE[p] = gates[t,j] dy_t, p = inv[t*k+j].
__device__ __forceinline__ void store_as(float* p, float v) { *p = v; }
__device__ __forceinline__ void store_as(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

template <typename TY, typename TE>
__global__ void __launch_bounds__(256)
combine_backward_kernel(const float* __restrict__ dy, const TY* __restrict__ y_perm,
                        const int32_t* __restrict__ inv, const float* __restrict__ gates, int T,
                        int k, int d, long long R, float* __restrict__ dG, TE* __restrict__ dE) {
    griddep_wait();
    griddep_launch_dependents();
    const int lane = threadIdx.x & 31;
    const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
    for (long long t = warp; t < T; t += nwarps) {
        const float* dyt = dy + (size_t)t * d;
        for (int j = 0; j < k; ++j) {
            const int32_t p = inv[t * k + j];
            const float g = gates[t * k + j];
            float acc = 0.0f;
            if (p >= 0 && p < R) {
                for (int c = lane; c < d; c += 32) {
                    const float v = dyt[c];
                    acc = fmaf(v, load_as_float(y_perm + (size_t)p * d + c), acc);
                    store_as(dE + (size_t)p * d + c, g * v);
                }
            }
            acc = warp_sum_f(acc);
            if (lane == 0) dG[t * k + j] = acc;
        }
    }
}

// One warp per token: the gate's backward.  With G the kept gates, dG' = dG + g_imp[e],
// dH[idx_j] += G_j (dG'_j - sum_l G_l dG'_l)  (softmax over the kept logits);
// for every expert i, z = (clean_i - thr_i) / std_i, a_i = g_load[i] phi(z) / std_i:
// dclean_i += a_i, dstd_i -= a_i z, and the threshold's expert m (the (k+1)-th for a
// kept i, the k-th otherwise) gets dH_m -= a_i; then dclean += dH, dstd += eps dH and
// dnz = dstd sigmoid(nz) with sigmoid(nz) = 1 - exp(-(std - floor)) (eq (4)).
__global__ void __launch_bounds__(256)
gate_backward_kernel(const float* __restrict__ clean, const float* __restrict__ stdv,
                     const float* __restrict__ eps, const int32_t* __restrict__ idx,
                     const float* __restrict__ gates, const float* __restrict__ dG,
                     const float* __restrict__ thr, const int32_t* __restrict__ next_idx,
                     const float* __restrict__ g_imp, const float* __restrict__ g_load, int T,
                     int n, int k, float std_floor, float* __restrict__ dclean,
                     float* __restrict__ dnz, __nv_bfloat16* __restrict__ split) {
    griddep_wait();
    griddep_launch_dependents();
    const int lane = threadIdx.x & 31;
    const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
    constexpr float kInvSqrt2Pi = 0.3989422804014327f;
    for (long long t = warp; t < T; t += nwarps) {
        int ix[8];
        float dh[8];
        float s = 0.0f;
        for (int j = 0; j < k; ++j) {
            ix[j] = idx[t * k + j];
            const float dgp = dG[t * k + j] + g_imp[ix[j]];
            dh[j] = dgp;
            s = fmaf(gates[t * k + j], dgp, s);
        }
        for (int j = 0; j < k; ++j) dh[j] = gates[t * k + j] * (dh[j] - s);
        const float th_in = thr[2 * t], th_out = thr[2 * t + 1];
        const int m_in = next_idx[t], m_out = ix[k - 1];
        const float* cl = clean + (size_t)t * n;
        const float* sd = stdv + (size_t)t * n;
        // pass 1: the load terms summed per threshold expert
        float to_in = 0.0f, to_out = 0.0f;
        for (int i = lane; i < n; i += 32) {
            bool kept = false;
            for (int j = 0; j < k; ++j) kept |= ix[j] == i;
            const float th = kept ? th_in : th_out;
            if (!(th > -INFINITY)) continue;              // k = n: P = 1
            const float z = (cl[i] - th) / sd[i];
            const float a = g_load[i] * kInvSqrt2Pi * expf(-0.5f * z * z) / sd[i];
            if (kept) to_in += a; else to_out += a;
        }
        to_in = warp_sum_f(to_in);
        to_out = warp_sum_f(to_out);
        // pass 2: dclean and dnz of every expert
        for (int i = lane; i < n; i += 32) {
            bool kept = false;
            float dhi = 0.0f;
            for (int j = 0; j < k; ++j) {
                const bool hit = ix[j] == i;
                kept |= hit;
                dhi += hit ? dh[j] : 0.0f;
            }
            if (i == m_in) dhi -= to_in;
            if (i == m_out) dhi -= to_out;
            const float th = kept ? th_in : th_out;
            float dc = 0.0f, ds = 0.0f;
            if (th > -INFINITY) {
                const float z = (cl[i] - th) / sd[i];
                const float a = g_load[i] * kInvSqrt2Pi * expf(-0.5f * z * z) / sd[i];
                dc = a;
                ds = -a * z;
            }
            dc += dhi;
            if (eps != nullptr) ds = fmaf(eps[(size_t)t * n + i], dhi, ds);
            const float sig = -expm1f(std_floor - sd[i]);
            const float dn = ds * sig;
            dclean[(size_t)t * n + i] = dc;
            dnz[(size_t)t * n + i] = dn;
            if (split != nullptr) {   // exact two-term bf16 split: hi + lo, for the tensor cores
                __nv_bfloat16* row = split + (size_t)t * 4 * n;
                const __nv_bfloat16 ch = __float2bfloat16_rn(dc), nh = __float2bfloat16_rn(dn);
                row[i] = ch;
                row[n + i] = __float2bfloat16_rn(dc - __bfloat162float(ch));
                row[2 * n + i] = nh;
                row[3 * n + i] = __float2bfloat16_rn(dn - __bfloat162float(nh));
            }
        }
    }
}

// dx[t] += sum_j dX_perm[inv[t*k+j]] (one warp per token, slot order).
template <typename TX>
__global__ void __launch_bounds__(256)
gather_dx_kernel(const TX* __restrict__ dxp, const int32_t* __restrict__ inv, int T, int k,
                 int d, long long R, float* __restrict__ dx) {
    griddep_wait();
    griddep_launch_dependents();
    const int lane = threadIdx.x & 31;
    const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
    for (long long t = warp; t < T; t += nwarps) {
        for (int c = lane; c < d; c += 32) {
            float acc = 0.0f;
            for (int j = 0; j < k; ++j) {
                const int32_t p = inv[t * k + j];
                if (p >= 0 && p < R) acc += load_as_float(dxp + (size_t)p * d + c);
            }
            dx[(size_t)t * d + c] = acc;
        }
    }
}

// Column sums in two fixed-order stages (db_g): column_chunk_kernel sums rows
// [c COLSUM_ROWS, (c+1) COLSUM_ROWS) of column i into part[c][i] (compensated fp32,
// ascending t, eight rows' loads in flight), then the chunks are added in tile_sums_512's
// order (launch_partial_reduce).  B300 issues fp64 adds at a small fraction of its fp32
// rate, and one CTA walking all T rows left the loads one at a time.
constexpr int COLSUM_ROWS = 256;
__global__ void __launch_bounds__(256)
column_chunk_kernel(const float* __restrict__ v, int T, int n, float* __restrict__ part) {
    griddep_wait();
    griddep_launch_dependents();
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    const int c = blockIdx.y;
    if (i >= n) return;
    const int t0 = c * COLSUM_ROWS, t1 = min(T, t0 + COLSUM_ROWS);
    CSum s = {0.0f, 0.0f};
    for (int tb = t0; tb < t1; tb += 8) {
        float x[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) x[q] = tb + q < t1 ? v[(size_t)(tb + q) * n + i] : 0.0f;
#pragma unroll
        for (int q = 0; q < 8; ++q)
            if (tb + q < t1) s = cadd(s, x[q]);
    }
    part[(size_t)c * n + i] = s.s + s.c;
}

// ---- grouped GEMM on the CUDA cores --------------------------------------------------
//
// C(m, n) (+)= sum_k A(m, k) B(k, n), A(m, k) = A[a_base + m sam + k sak],
// B(k, n) = B[b_base + k sbk + n sbn], fp32 accumulation, 64 x 64 tiles, 16-deep k
// steps through shared memory, 4 x 4 outputs a thread.  Three ways to form groups:
//   ROWS:  one tile row block of 64 routed rows of one expert from the unit table
//          (e, first row, end of rows); A rows and C rows are those rows, B = expert e's
//          matrix (b_base = e * b_group); optional mask: C(m, n) *= [mask(m, n) > 0];
//   WGRAD: group e = blockIdx.z; k runs over expert e's rows [offsets[e], offsets[e+1]);
//          C = expert e's [M, N] block (c_base = e * c_group), written even when empty;
//   PLAIN: one group, M, N, K given.
//   SPLITK: PLAIN with the k range split over grid z; CTA z writes its partial sums to
//          C + z * c_group (reduced afterwards in a fixed order by splitk_reduce_kernel).
enum GemmMode { GEMM_ROWS = 0, GEMM_WGRAD = 1, GEMM_PLAIN = 2, GEMM_SPLITK = 3 };

struct GemmArgs {
    long long sam, sak, sbk, sbn, ldc;
    long long b_group, c_group;
    int M, N, K;
    const int4* units;          // ROWS
    const int32_t* blk;         // ROWS: blk[n] = unit count
    const int32_t* offsets;     // WGRAD
    int n_groups;
    float beta;                 // C = beta C + A B
};

constexpr int GT = 64, GK = 16, GTHREADS = 256;

template <typename TA, typename TB, typename TM, int MODE>
__global__ void __launch_bounds__(GTHREADS)
grouped_gemm_kernel(const TA* __restrict__ A, const TB* __restrict__ B, float* __restrict__ C,
                    const TM* __restrict__ mask, const GemmArgs g) {
    griddep_wait();
    griddep_launch_dependents();
    __shared__ float As[GK][GT + 4];
    __shared__ float Bs[GK][GT + 4];
    const int tid = threadIdx.x;
    const int tx = tid % 16, ty = tid / 16;
    long long a_base = 0, b_base = 0, c_base = 0;
    int m0 = 0, m_end = 0, K = 0;
    long long k_row0 = 0;     // WGRAD: first row of the group
    const int n0 = blockIdx.x * GT;
    if (MODE == GEMM_ROWS) {
        if ((int)blockIdx.y >= g.blk[g.n_groups]) return;
        const int4 u = g.units[blockIdx.y];
        m0 = u.y;
        m_end = u.z < u.y + GT ? u.z : u.y + GT;
        b_base = (long long)u.x * g.b_group;
        K = g.K;
    } else if (MODE == GEMM_WGRAD) {
        const int e = blockIdx.z;
        m0 = blockIdx.y * GT;
        m_end = g.M < m0 + GT ? g.M : m0 + GT;
        k_row0 = g.offsets[e];
        K = g.offsets[e + 1] - g.offsets[e];
        c_base = (long long)e * g.c_group;
    } else if (MODE == GEMM_SPLITK) {
        m0 = blockIdx.y * GT;
        m_end = g.M < m0 + GT ? g.M : m0 + GT;
        const int chunk = (g.K + (int)gridDim.z - 1) / (int)gridDim.z;
        k_row0 = (long long)blockIdx.z * chunk;
        K = g.K - (int)k_row0 < chunk ? g.K - (int)k_row0 : chunk;
        if (K < 0) K = 0;
        c_base = (long long)blockIdx.z * g.c_group;
    } else {
        m0 = blockIdx.y * GT;
        m_end = g.M < m0 + GT ? g.M : m0 + GT;
        K = g.K;
    }
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;
    // consecutive threads walk the operand's contiguous dimension
    const bool a_k_fast = g.sak == 1, b_k_fast = g.sbk == 1 && g.sbn != 1;
    for (int k0 = 0; k0 < K; k0 += GK) {
        // A tile [64 m][16 k], B tile [16 k][64 n]: four elements a thread each
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int l = tid + q * GTHREADS;
            const int am = a_k_fast ? l / GK : l % GT, ak = a_k_fast ? l % GK : l / GT;
            const int m = m0 + am, kk = k0 + ak;
            float av = 0.0f;
            if (m < m_end && kk < K) {
                const long long kr = (MODE == GEMM_WGRAD || MODE == GEMM_SPLITK) ? k_row0 + kk : kk;
                av = load_as_float(A + a_base + (long long)m * g.sam + kr * g.sak);
            }
            As[ak][am] = av;
            const int bn = b_k_fast ? l / GK : l % GT, bk = b_k_fast ? l % GK : l / GT;
            const int n = n0 + bn, kb = k0 + bk;
            float bv = 0.0f;
            if (n < g.N && kb < K) {
                const long long kr = (MODE == GEMM_WGRAD || MODE == GEMM_SPLITK) ? k_row0 + kb : kb;
                bv = load_as_float(B + b_base + kr * g.sbk + (long long)n * g.sbn);
            }
            Bs[bk][bn] = bv;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < GK; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int m = m0 + ty * 4 + i;
        if (m >= m_end) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = n0 + tx * 4 + j;
            if (n >= g.N) continue;
            float v = acc[i][j];
            const long long o = c_base + (long long)m * g.ldc + n;
            if (mask != nullptr && !(load_as_float(mask + (long long)m * g.N + n) > 0.0f)) v = 0.0f;
            C[o] = g.beta != 0.0f ? fmaf(g.beta, C[o], v) : v;
        }
    }
}

// The gate's weight gradients from the tensor-core partials part [chunks][d][4n] (x^T
// times the split [dclean_hi | dclean_lo | dnz_hi | dnz_lo] over each 1024-token chunk):
// dW_g[i][j] = sum over chunks, ascending, of hi then lo; dW_noise likewise; compensated
// fp32 (a two-sum per add carries each rounding error; B300's fp64 rate is a small
// fraction of its fp32 rate), four chunks' loads in flight.
__global__ void __launch_bounds__(256)
gate_split_reduce_kernel(const float* __restrict__ part, int chunks, int d, int n,
                         float* __restrict__ dW_g, float* __restrict__ dW_noise) {
    griddep_wait();
    griddep_launch_dependents();
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long long)d * n) return;
    const long long r = i / n, j = i % n;
    CSum sg = {0.0f, 0.0f}, sn = {0.0f, 0.0f};
    for (int cb = 0; cb < chunks; cb += 4) {
        float x[4][4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float* p = part + ((size_t)(cb + q) * d + r) * 4 * n;
            const bool in = cb + q < chunks;
#pragma unroll
            for (int u = 0; u < 4; ++u) x[q][u] = in ? p[u * n + j] : 0.0f;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (cb + q < chunks) {
                sg = cadd(cadd(sg, x[q][0]), x[q][1]);
                sn = cadd(cadd(sn, x[q][2]), x[q][3]);
            }
        }
    }
    dW_g[i] = sg.s + sg.c;
    dW_noise[i] = sn.s + sn.c;
}

// offsets[c] = min(c * chunk, T): the token chunks of the gate's split contraction.
__global__ void chunk_offsets_kernel(int T, int chunk, int chunks, int32_t* __restrict__ offsets) {
    griddep_wait();
    griddep_launch_dependents();
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c <= chunks) offsets[c] = c * chunk < T ? c * chunk : T;
}

// out[i] = sum over z = 0..splits-1 of part[z * count + i], in ascending z, compensated
// fp32.
__global__ void __launch_bounds__(256)
splitk_reduce_kernel(const float* __restrict__ part, int splits, long long count,
                     float* __restrict__ out) {
    griddep_wait();
    griddep_launch_dependents();
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= count) return;
    CSum s = {0.0f, 0.0f};
    for (int z = 0; z < splits; ++z) s = cadd(s, part[(size_t)z * count + i]);
    out[i] = s.s + s.c;
}

template <typename TA, typename TB, typename TM, int MODE>
cudaError_t launch_gemm(const TA* A, const TB* B, float* C, const TM* mask, const GemmArgs& g,
                        dim3 grid, cudaStream_t s) {
    const cudaError_t e = launch_pdl(grouped_gemm_kernel<TA, TB, TM, MODE>, grid, dim3(GTHREADS),
                                     0, s, 1, A, B, C, mask, g);
    note_launch();
    return e;
}

int token_blocks(long long T) {
    long long b = (T + 7) / 8;
    if (b > 148 * 16) b = 148 * 16;
    return (int)(b < 1 ? 1 : b);
}

}  // namespace

int backward_row_block() { return GT; }

int gate_splitk(int T) {
    const int s = (T + 1023) / 1024;     // about 1024 rows a layer
    return s < 1 ? 1 : (s > 64 ? 64 : s);
}

cudaError_t launch_cv2_grad(const float* importance, const float* load, int n, float w_imp,
                            float w_load, float* g_imp, float* g_load, cudaStream_t s) {
    const cudaError_t e = launch_pdl(cv2_grad_kernel, dim3(1), dim3(64), 0, s, 1, importance,
                                     load, n, w_imp, w_load, g_imp, g_load);
    note_launch();
    return e;
}

cudaError_t launch_combine_backward(const float* dy, const void* y_perm, bool half_rows,
                                    const int32_t* inv, const float* gates, int T, int k, int d,
                                    float* dG, void* dE, bool dE_bf16, cudaStream_t s) {
    const long long R = (long long)T * k;
    const dim3 grid(token_blocks(T));
    cudaError_t e;
    if (half_rows && dE_bf16)
        e = launch_pdl(combine_backward_kernel<__half, __nv_bfloat16>, grid, dim3(256), 0, s, 1,
                       dy, static_cast<const __half*>(y_perm), inv, gates, T, k, d, R, dG,
                       static_cast<__nv_bfloat16*>(dE));
    else if (half_rows)
        e = launch_pdl(combine_backward_kernel<__half, float>, grid, dim3(256), 0, s, 1, dy,
                       static_cast<const __half*>(y_perm), inv, gates, T, k, d, R, dG,
                       static_cast<float*>(dE));
    else
        e = launch_pdl(combine_backward_kernel<float, float>, grid, dim3(256), 0, s, 1, dy,
                       static_cast<const float*>(y_perm), inv, gates, T, k, d, R, dG,
                       static_cast<float*>(dE));
    note_launch();
    return e;
}

cudaError_t launch_gate_backward(const float* clean, const float* stdv, const float* eps,
                                 const int32_t* idx, const float* gates, const float* dG,
                                 const float* thr, const int32_t* next_idx, const float* g_imp,
                                 const float* g_load, int T, int n, int k, float std_floor,
                                 float* dclean, float* dnz, void* split, cudaStream_t s) {
    const cudaError_t e =
        launch_pdl(gate_backward_kernel, dim3(token_blocks(T)), dim3(256), 0, s, 1, clean, stdv,
                   eps, idx, gates, dG, thr, next_idx, g_imp, g_load, T, n, k, std_floor, dclean,
                   dnz, static_cast<__nv_bfloat16*>(split));
    note_launch();
    return e;
}

cudaError_t launch_gather_dx(const void* dxp, bool half_rows, const int32_t* inv, int T, int k,
                             int d, float* dx, cudaStream_t s) {
    const long long R = (long long)T * k;
    const cudaError_t e =
        half_rows ? launch_pdl(gather_dx_kernel<__half>, dim3(token_blocks(T)), dim3(256), 0, s, 1,
                               static_cast<const __half*>(dxp), inv, T, k, d, R, dx)
                  : launch_pdl(gather_dx_kernel<float>, dim3(token_blocks(T)), dim3(256), 0, s, 1,
                               static_cast<const float*>(dxp), inv, T, k, d, R, dx);
    note_launch();
    return e;
}

size_t column_sum_scratch_floats(int T, int n) {
    return (size_t)((T + COLSUM_ROWS - 1) / COLSUM_ROWS) * n;
}

cudaError_t launch_column_sum(const float* v, int T, int n, float* out, float* part,
                              cudaStream_t s) {
    const int chunks = (T + COLSUM_ROWS - 1) / COLSUM_ROWS;
    const cudaError_t e = launch_pdl(column_chunk_kernel, dim3((n + 255) / 256, chunks),
                                     dim3(256), 0, s, 1, v, T, n, part);
    note_launch();
    if (e != cudaSuccess) return e;
    return launch_partial_reduce(part, nullptr, chunks, n, out, nullptr, s);
}

// Expert data gradients, one 64-row block of one expert per CTA row (unit table of
// launch_row_block_prefix with block 64): dU = (dE W_out[e]^T) [hidden > 0] [R,h] and
// dX_perm = dU W_in[e]^T [R,d].
template <typename TW, typename TH>
cudaError_t expert_dgrad(const float* dE, const TW* W_in, const TW* W_out, const TH* hidden,
                         const int4* units, const int32_t* blk, long long R, int d, int h, int n,
                         float* dU, float* dXp, cudaStream_t s) {
    const long long max_units = (R + GT - 1) / GT + n;
    GemmArgs g{};
    g.units = units;
    g.blk = blk;
    g.n_groups = n;
    // dU[r, j] = sum_c dE[r, c] W_out[e][j, c]
    g.sam = d; g.sak = 1; g.sbk = 1; g.sbn = d; g.ldc = h; g.b_group = (long long)h * d;
    g.N = h; g.K = d; g.beta = 0.0f;
    cudaError_t e = launch_gemm<float, TW, TH, GEMM_ROWS>(dE, W_out, dU, hidden, g,
                                                          dim3((h + GT - 1) / GT, max_units), s);
    if (e != cudaSuccess) return e;
    // dX_perm[r, c] = sum_j dU[r, j] W_in[e][c, j]
    g.sam = h; g.sak = 1; g.sbk = 1; g.sbn = h; g.ldc = d; g.b_group = (long long)d * h;
    g.N = d; g.K = h;
    return launch_gemm<float, TW, TH, GEMM_ROWS>(dU, W_in, dXp, nullptr, g,
                                                 dim3((d + GT - 1) / GT, max_units), s);
}

// Expert weight gradients: dW_out[e] = hidden_e^T dE_e [h,d], dW_in[e] = x_perm_e^T dU_e [d,h].
template <typename TX, typename TH, typename TG>
cudaError_t expert_wgrad(const TX* x_perm, const TH* hidden, const TG* dE, const TG* dU,
                         const int32_t* offsets, int d, int h, int n, float* dW_in,
                         float* dW_out, cudaStream_t s) {
    GemmArgs g{};
    g.offsets = offsets;
    g.beta = 0.0f;
    g.sam = 1; g.sak = h; g.sbk = d; g.sbn = 1; g.ldc = d; g.c_group = (long long)h * d;
    g.M = h; g.N = d;
    cudaError_t e = launch_gemm<TH, TG, float, GEMM_WGRAD>(
        hidden, dE, dW_out, nullptr, g, dim3((d + GT - 1) / GT, (h + GT - 1) / GT, n), s);
    if (e != cudaSuccess) return e;
    g.sam = 1; g.sak = d; g.sbk = h; g.sbn = 1; g.ldc = h; g.c_group = (long long)d * h;
    g.M = d; g.N = h;
    return launch_gemm<TX, TG, float, GEMM_WGRAD>(
        x_perm, dU, dW_in, nullptr, g, dim3((h + GT - 1) / GT, (d + GT - 1) / GT, n), s);
}

// The gate's weight gradients and its share of dx:
// dW_g = x^T dclean, dW_noise = x^T dnz [d,n]; dx += dclean W_g^T + dnz W_noise^T.
template <typename TX>
cudaError_t gate_weight_grads(const TX* x, const float* W_g, const float* W_noise,
                              const float* dclean, const float* dnz, int T, int d, int n,
                              float* dW_g, float* dW_noise, float* dx, float* part,
                              cudaStream_t s) {
    // the T-long contraction split over gate_splitk(T) CTA layers, then a fixed-order sum
    const int splits = gate_splitk(T);
    GemmArgs g{};
    g.sam = 1; g.sak = d; g.sbk = n; g.sbn = 1; g.ldc = n; g.M = d; g.N = n; g.K = T;
    g.c_group = (long long)d * n;
    g.beta = 0.0f;
    const dim3 gw((n + GT - 1) / GT, (d + GT - 1) / GT, splits);
    const long long count = (long long)d * n;
    const unsigned rb = (unsigned)((count + 255) / 256);
    cudaError_t e = launch_gemm<TX, float, float, GEMM_SPLITK>(x, dclean, part, nullptr, g, gw, s);
    if (e != cudaSuccess) return e;
    e = launch_pdl(splitk_reduce_kernel, dim3(rb), dim3(256), 0, s, 1,
                   static_cast<const float*>(part), splits, count, dW_g);
    note_launch();
    if (e != cudaSuccess) return e;
    e = launch_gemm<TX, float, float, GEMM_SPLITK>(x, dnz, part, nullptr, g, gw, s);
    if (e != cudaSuccess) return e;
    e = launch_pdl(splitk_reduce_kernel, dim3(rb), dim3(256), 0, s, 1,
                   static_cast<const float*>(part), splits, count, dW_noise);
    note_launch();
    if (e != cudaSuccess) return e;
    GemmArgs q{};
    q.sam = n; q.sak = 1; q.sbk = 1; q.sbn = n; q.ldc = d; q.M = T; q.N = d; q.K = n;
    q.beta = 1.0f;
    const dim3 gx((d + GT - 1) / GT, (T + GT - 1) / GT);
    e = launch_gemm<float, float, float, GEMM_PLAIN>(dclean, W_g, dx, nullptr, q, gx, s);
    if (e != cudaSuccess) return e;
    return launch_gemm<float, float, float, GEMM_PLAIN>(dnz, W_noise, dx, nullptr, q, gx, s);
}

int gate_tc_chunk() { return 1024; }

cudaError_t launch_gate_tc_weight_grads(const void* x, const void* split, int T, int d, int n,
                                        int32_t* chunk_offsets, void* btail, float* part,
                                        float* dW_g, float* dW_noise, int* err, cudaStream_t s) {
    const int chunk = gate_tc_chunk();
    const int chunks = (T + chunk - 1) / chunk;
    cudaError_t e = launch_pdl(chunk_offsets_kernel, dim3((chunks + 256) / 256), dim3(256), 0, s,
                               1, T, chunk, chunks, chunk_offsets);
    note_launch();
    if (e != cudaSuccess) return e;
    e = launch_ffn_wgrad(x, split, btail, chunk_offsets, T, d, 4 * n, chunks, part, err, s);
    if (e != cudaSuccess) return e;
    const long long count = (long long)d * n;
    e = launch_pdl(gate_split_reduce_kernel, dim3((unsigned)((count + 255) / 256)), dim3(256), 0,
                   s, 1, static_cast<const float*>(part), chunks, d, n, dW_g, dW_noise);
    note_launch();
    return e;
}

cudaError_t launch_gate_dx(const float* W_g, const float* W_noise, const float* dclean,
                           const float* dnz, int T, int d, int n, float* dx, cudaStream_t s) {
    GemmArgs q{};
    q.sam = n; q.sak = 1; q.sbk = 1; q.sbn = n; q.ldc = d; q.M = T; q.N = d; q.K = n;
    q.beta = 1.0f;
    const dim3 gx((d + GT - 1) / GT, (T + GT - 1) / GT);
    cudaError_t e = launch_gemm<float, float, float, GEMM_PLAIN>(dclean, W_g, dx, nullptr, q, gx, s);
    if (e != cudaSuccess) return e;
    return launch_gemm<float, float, float, GEMM_PLAIN>(dnz, W_noise, dx, nullptr, q, gx, s);
}

cudaError_t launch_expert_dgrad(const float* dE, const void* W_in, const void* W_out,
                                const void* hidden, bool bf16, const void* units,
                                const int32_t* blk, long long R, int d, int h, int n, float* dU,
                                float* dXp, cudaStream_t s) {
    const int4* u = static_cast<const int4*>(units);
    if (bf16)
        return expert_dgrad(dE, static_cast<const __nv_bfloat16*>(W_in),
                            static_cast<const __nv_bfloat16*>(W_out),
                            static_cast<const __nv_bfloat16*>(hidden), u, blk, R, d, h, n, dU,
                            dXp, s);
    return expert_dgrad(dE, static_cast<const float*>(W_in), static_cast<const float*>(W_out),
                        static_cast<const float*>(hidden), u, blk, R, d, h, n, dU, dXp, s);
}

cudaError_t launch_expert_wgrad(const void* x_perm, const void* hidden, bool bf16, const void* dE,
                                const void* dU, bool grads_bf16, const int32_t* offsets, int d,
                                int h, int n, float* dW_in, float* dW_out, cudaStream_t s) {
    if (bf16 && grads_bf16)
        return expert_wgrad(static_cast<const __nv_bfloat16*>(x_perm),
                            static_cast<const __nv_bfloat16*>(hidden),
                            static_cast<const __nv_bfloat16*>(dE),
                            static_cast<const __nv_bfloat16*>(dU), offsets, d, h, n, dW_in,
                            dW_out, s);
    if (bf16)
        return expert_wgrad(static_cast<const __nv_bfloat16*>(x_perm),
                            static_cast<const __nv_bfloat16*>(hidden),
                            static_cast<const float*>(dE), static_cast<const float*>(dU), offsets,
                            d, h, n, dW_in, dW_out, s);
    return expert_wgrad(static_cast<const float*>(x_perm), static_cast<const float*>(hidden),
                        static_cast<const float*>(dE), static_cast<const float*>(dU), offsets, d,
                        h, n, dW_in, dW_out, s);
}

cudaError_t launch_gate_weight_grads(const void* x, bool x_bf16, const float* W_g,
                                     const float* W_noise, const float* dclean, const float* dnz,
                                     int T, int d, int n, float* dW_g, float* dW_noise, float* dx,
                                     float* part, cudaStream_t s) {
    if (x_bf16)
        return gate_weight_grads(static_cast<const __nv_bfloat16*>(x), W_g, W_noise, dclean, dnz,
                                 T, d, n, dW_g, dW_noise, dx, part, s);
    return gate_weight_grads(static_cast<const float*>(x), W_g, W_noise, dclean, dnz, T, d, n,
                             dW_g, dW_noise, dx, part, s);
}

}  // namespace moe
