// Noisy top-k gate on the CUDA cores (fp32 FFMA), for any x dtype.
//
// "Mixture of Experts: Outrageously Large Neural Networks" (intuitivepapers.ai):
//   section "Noisy top-k gating", eq (4):  H_i = (x W_g)_i + eps_i * Softplus((x W_noise)_i)
//   eqs (3)/(5): keep the k largest H, softmax over them;
//   section "A differentiable count of examples", eqs (8)-(10):
//   P(x,i) = Phi(((x W_g)_i - kth_excluding(H,k,i)) / std_i), Load_i = sum_x P(x,i).
// The forward-pass listing in "Implementation notes" takes the top k+1 logits: the
// (k+1)-th is the threshold for kept experts, the k-th for the others.
#include <math.h>
#include <stdint.h>

#include "common.cuh"
#include "launch.h"

namespace moe {
namespace {

constexpr int GT = 64;    // tokens per tile
constexpr int GE = 64;    // experts per tile
constexpr int GK = 16;    // reduction slice
constexpr int GTHREADS = 256;

template <typename TX>
__device__ __forceinline__ void load_x4(const TX* p, float out[4]);

template <>
__device__ __forceinline__ void load_x4<float>(const float* p, float out[4]) {
    float4 v = *reinterpret_cast<const float4*>(p);
    out[0] = v.x; out[1] = v.y; out[2] = v.z; out[3] = v.w;
}

template <>
__device__ __forceinline__ void load_x4<__nv_bfloat16>(const __nv_bfloat16* p, float out[4]) {
    uint2 v = *reinterpret_cast<const uint2*>(p);
    __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162*>(&v.x);
    __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&v.y);
    out[0] = __low2float(a); out[1] = __high2float(a);
    out[2] = __low2float(b); out[3] = __high2float(b);
}

// clean = x W_g (+ b_g), std = Softplus(x W_noise) + floor, H = clean + eps * std.
// One CTA computes a 64-token x 64-expert tile of both products; each thread
// holds 4 tokens x 4 experts of each.  d must be a multiple of 16.
template <typename TX>
__global__ void __launch_bounds__(GTHREADS)
gate_logits_kernel(const TX* __restrict__ x, const float* __restrict__ W_g,
                   const float* __restrict__ W_noise, const float* __restrict__ eps,
                   const float* __restrict__ b_g, int T, int d, int n, float std_floor,
                   float* __restrict__ clean_out, float* __restrict__ std_out,
                   float* __restrict__ H_out) {
    __shared__ float xs[GK][GT + 4];
    __shared__ float wg[GK][GE];
    __shared__ float wn[GK][GE];

    const int tid = threadIdx.x;
    const int tx = tid % 16, ty = tid / 16;
    const int t0 = blockIdx.y * GT, e0 = blockIdx.x * GE;

    float ac[4][4], ar[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) ac[i][j] = ar[i][j] = 0.0f;

    // loader coordinates
    const int lx_tok = tid / 4, lx_k = (tid % 4) * 4;      // x: 64 tokens x 16 k
    const int lw_k = tid / 16, lw_e = (tid % 16) * 4;      // W: 16 k x 64 experts

    for (int k0 = 0; k0 < d; k0 += GK) {
        float xv[4] = {0.f, 0.f, 0.f, 0.f};
        const int tok = t0 + lx_tok;
        if (tok < T) load_x4<TX>(x + (size_t)tok * d + k0 + lx_k, xv);
#pragma unroll
        for (int q = 0; q < 4; ++q) xs[lx_k + q][lx_tok] = xv[q];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int e = e0 + lw_e + q;
            const size_t off = (size_t)(k0 + lw_k) * n + e;
            wg[lw_k][lw_e + q] = e < n ? W_g[off] : 0.0f;
            wn[lw_k][lw_e + q] = e < n ? W_noise[off] : 0.0f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < GK; ++kk) {
            float a[4], bg[4], bn[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = xs[kk][ty + 16 * i];
#pragma unroll
            for (int j = 0; j < 4; ++j) { bg[j] = wg[kk][tx + 16 * j]; bn[j] = wn[kk][tx + 16 * j]; }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    ac[i][j] = fmaf(a[i], bg[j], ac[i][j]);
                    ar[i][j] = fmaf(a[i], bn[j], ar[i][j]);
                }
        }
        __syncthreads();
    }

#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int t = t0 + ty + 16 * i;
        if (t >= T) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int e = e0 + tx + 16 * j;
            if (e >= n) continue;
            const size_t o = (size_t)t * n + e;
            const float c = ac[i][j] + (b_g != nullptr ? b_g[e] : 0.0f);
            const float sd = softplus_f32(ar[i][j]) + std_floor;
            clean_out[o] = c;
            std_out[o] = sd;
            H_out[o] = eps != nullptr ? fmaf(eps[o], sd, c) : c;
        }
    }
}

// Per-token top-(k+1) of H with one warp per token.  Order: larger H first,
// equal H -> lower expert index first.  Each lane keeps a sorted list of its
// K1 best (it visits experts in ascending index, so a later equal value never
// displaces an earlier one); K1 rounds of a warp arg-max then merge the lists.
// SWITCH: the gates are the softmax over all n of H at the kept experts ("From LSTMs to
// Switch and Mixtral"), and thr[t] = (max H, 1 / sum over all n of exp(H - max)).
// next_idx (nullable): the expert at the (k+1)-th place (-1 when k = n).
template <int K1, bool SWITCH>
__global__ void __launch_bounds__(256)
gate_select_kernel(const float* __restrict__ H, int T, int n, int32_t* __restrict__ idx,
                   float* __restrict__ gates, uint8_t* __restrict__ tie, float* __restrict__ thr,
                   int32_t* __restrict__ next_idx) {
    griddep_wait();
    griddep_launch_dependents();
    constexpr int K = K1 - 1;
    const int lane = threadIdx.x & 31;
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    for (int t = warp; t < T; t += nwarps) {
        float v[K1];
        int ix[K1];
#pragma unroll
        for (int q = 0; q < K1; ++q) { v[q] = -INFINITY; ix[q] = 0x7fffffff; }
        const float* row = H + (size_t)t * n;
        for (int e = lane; e < n; e += 32) {
            const float hv = row[e];
            if (hv > v[K1 - 1]) {
                // Descending q: v[q - 1] and v[q] are still the old values here.
#pragma unroll
                for (int q = K1 - 1; q > 0; --q) {
                    if (hv > v[q - 1]) { v[q] = v[q - 1]; ix[q] = ix[q - 1]; }
                    else if (hv > v[q]) { v[q] = hv; ix[q] = e; }
                }
                if (hv > v[0]) { v[0] = hv; ix[0] = e; }
            }
        }
        float tv[K1];
        int ti[K1];
#pragma unroll
        for (int r = 0; r < K1; ++r) {
            float bv = v[0];
            int bi = ix[0];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
                if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
            }
            tv[r] = bv;
            ti[r] = bi;
            if (ix[0] == bi) {   // the owning lane pops its head
#pragma unroll
                for (int q = 0; q < K1 - 1; ++q) { v[q] = v[q + 1]; ix[q] = ix[q + 1]; }
                v[K1 - 1] = -INFINITY;
                ix[K1 - 1] = 0x7fffffff;
            }
        }
        float inv_all = 0.0f;
        if (SWITCH) {       // every lane holds tv[0]: lane-strided sum, fixed butterfly
            float ps = 0.0f;
            for (int e = lane; e < n; e += 32) ps += expf(row[e] - tv[0]);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
            inv_all = 1.0f / ps;
        }
        if (lane == 0) {
            float s = 0.0f;
            float ex[K];
#pragma unroll
            for (int j = 0; j < K; ++j) { ex[j] = expf(tv[j] - tv[0]); s += ex[j]; }
            const float inv = SWITCH ? inv_all : 1.0f / s;
#pragma unroll
            for (int j = 0; j < K; ++j) {
                idx[(size_t)t * K + j] = ti[j];
                gates[(size_t)t * K + j] = ex[j] * inv;
            }
            // k = n: tv[K] is the -inf sentinel, so the gap is +inf and no tie.
            if (tie != nullptr) tie[t] = (tv[K - 1] - tv[K]) < 1e-5f ? 1 : 0;
            if (next_idx != nullptr) next_idx[t] = ti[K] < n ? ti[K] : -1;
            thr[2 * (size_t)t + 0] = SWITCH ? tv[0] : tv[K];        // kth_excluding for a kept expert
            thr[2 * (size_t)t + 1] = SWITCH ? inv_all : tv[K - 1];  // ... for an expert not kept
        }
    }
}

constexpr int LOAD_CHUNK = 64;   // tokens summed in fp32 before the fp64 sum over chunks

// part[c, e] = sum over the chunk's tokens of P(t, e), in ascending token order;
// with imp_part, also the sum of the gates the chunk's tokens keep for e (eq (6)).
__global__ void __launch_bounds__(256)
gate_load_partial_kernel(const float* __restrict__ clean, const float* __restrict__ stdv,
                         const int32_t* __restrict__ idx, const float* __restrict__ gates,
                         const float* __restrict__ thr, int T, int n, int k,
                         float* __restrict__ part, float* __restrict__ imp_part) {
    griddep_wait();
    griddep_launch_dependents();
    __shared__ int32_t s_idx[LOAD_CHUNK * 8];
    __shared__ float s_gate[LOAD_CHUNK * 8];
    __shared__ float s_thr[LOAD_CHUNK * 2];
    const int c = blockIdx.y;
    const int t0 = c * LOAD_CHUNK;
    const int nt = min(LOAD_CHUNK, T - t0);
    for (int i = threadIdx.x; i < nt * k; i += blockDim.x) {
        s_idx[i] = idx[(size_t)t0 * k + i];
        s_gate[i] = imp_part != nullptr ? gates[(size_t)t0 * k + i] : 0.0f;
    }
    for (int i = threadIdx.x; i < nt * 2; i += blockDim.x) s_thr[i] = thr[(size_t)t0 * 2 + i];
    __syncthreads();
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= n) return;
    float acc = 0.0f, imp = 0.0f;
#pragma unroll 4
    for (int tt = 0; tt < nt; ++tt) {
        bool kept = false;
        float g = 0.0f;
        for (int j = 0; j < k; ++j) {
            const bool hit = s_idx[tt * k + j] == e;
            kept |= hit;
            g = hit ? s_gate[tt * k + j] : g;
        }
        imp += g;
        const float th = kept ? s_thr[2 * tt] : s_thr[2 * tt + 1];
        const size_t o = (size_t)(t0 + tt) * n + e;
        acc += normal_cdf_f32((clean[o] - th) / stdv[o]);
    }
    part[(size_t)c * n + e] = acc;
    if (imp_part != nullptr) imp_part[(size_t)c * n + e] = imp;
}

// The Switch gate's per-chunk sums: part[c, e] = how many of the chunk's routed rows
// went to e, imp_part[c, e] = sum over the chunk's tokens of the probability
// exp(H - max) / sum (thr from gate_select_kernel<.., true>), ascending token order.
__global__ void __launch_bounds__(256)
gate_switch_partial_kernel(const float* __restrict__ H, const int32_t* __restrict__ idx,
                           const float* __restrict__ thr, int T, int n, int k,
                           float* __restrict__ part, float* __restrict__ imp_part) {
    griddep_wait();
    griddep_launch_dependents();
    __shared__ int32_t s_idx[LOAD_CHUNK * 8];
    __shared__ float s_thr[LOAD_CHUNK * 2];
    const int c = blockIdx.y;
    const int t0 = c * LOAD_CHUNK;
    const int nt = min(LOAD_CHUNK, T - t0);
    for (int i = threadIdx.x; i < nt * k; i += blockDim.x) s_idx[i] = idx[(size_t)t0 * k + i];
    for (int i = threadIdx.x; i < nt * 2; i += blockDim.x) s_thr[i] = thr[(size_t)t0 * 2 + i];
    __syncthreads();
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= n) return;
    float cnt = 0.0f, imp = 0.0f;
#pragma unroll 4
    for (int tt = 0; tt < nt; ++tt) {
        for (int j = 0; j < k; ++j) cnt += s_idx[tt * k + j] == e ? 1.0f : 0.0f;
        imp += expf(H[(size_t)(t0 + tt) * n + e] - s_thr[2 * tt]) * s_thr[2 * tt + 1];
    }
    part[(size_t)c * n + e] = cnt;
    imp_part[(size_t)c * n + e] = imp;
}

}  // namespace

cudaError_t launch_gate_logits(const void* x, bool x_bf16, const float* W_g, const float* W_noise,
                               const float* eps, const float* b_g, int T, int d, int n,
                               float std_floor, float* clean, float* stdv, float* H,
                               cudaStream_t s) {
    dim3 grid((n + GE - 1) / GE, (T + GT - 1) / GT);
    if (x_bf16)
        gate_logits_kernel<__nv_bfloat16><<<grid, GTHREADS, 0, s>>>(
            static_cast<const __nv_bfloat16*>(x), W_g, W_noise, eps, b_g, T, d, n, std_floor,
            clean, stdv, H);
    else
        gate_logits_kernel<float><<<grid, GTHREADS, 0, s>>>(
            static_cast<const float*>(x), W_g, W_noise, eps, b_g, T, d, n, std_floor, clean,
            stdv, H);
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_gate_select(const float* H, int T, int n, int k, int32_t* idx, float* gates,
                               uint8_t* tie, float* thr, cudaStream_t s, bool sw,
                               int32_t* next_idx) {
    const int threads = 256;
    long long want = ((long long)T * 32 + threads - 1) / threads;
    const int blocks = (int)(want < 148 * 16 ? want : 148 * 16);
    cudaError_t e = cudaSuccess;
    switch (k + 1) {
#define MOE_SELECT_CASE(K1) \
    case K1:                                                                                \
        e = sw ? launch_pdl(gate_select_kernel<K1, true>, dim3(blocks), dim3(threads), 0, s, 1, \
                            H, T, n, idx, gates, tie, thr, next_idx)                        \
               : launch_pdl(gate_select_kernel<K1, false>, dim3(blocks), dim3(threads), 0, s, \
                            1, H, T, n, idx, gates, tie, thr, next_idx);                    \
        note_launch();                                                                      \
        break;
        MOE_SELECT_CASE(2) MOE_SELECT_CASE(3) MOE_SELECT_CASE(4) MOE_SELECT_CASE(5)
        MOE_SELECT_CASE(6) MOE_SELECT_CASE(7) MOE_SELECT_CASE(8) MOE_SELECT_CASE(9)
#undef MOE_SELECT_CASE
        default: return cudaErrorInvalidValue;
    }
    return e;
}

int gate_load_chunks(int T) { return (T + LOAD_CHUNK - 1) / LOAD_CHUNK; }

cudaError_t launch_gate_switch_sums(const float* H, const int32_t* idx, const float* thr, int T,
                                    int n, int k, float* part, float* load, float* imp_part,
                                    float* importance, cudaStream_t s) {
    const int chunks = gate_load_chunks(T);
    cudaError_t e = launch_pdl(gate_switch_partial_kernel, dim3((n + 255) / 256, chunks), dim3(256),
                               0, s, 1, H, idx, thr, T, n, k, part, imp_part);
    note_launch();
    if (e != cudaSuccess) return e;
    return launch_partial_reduce(part, importance != nullptr ? imp_part : nullptr, chunks, n, load,
                                 importance, s);
}

cudaError_t launch_gate_load(const float* clean, const float* stdv, const int32_t* idx,
                             const float* gates, const float* thr, int T, int n, int k, float* part,
                             float* load, float* imp_part, float* importance, cudaStream_t s) {
    const int chunks = gate_load_chunks(T);
    dim3 grid((n + 255) / 256, chunks);
    float* ip = importance != nullptr ? imp_part : nullptr;
    cudaError_t e = launch_pdl(gate_load_partial_kernel, grid, dim3(256), 0, s, 1, clean, stdv, idx,
                               gates, thr, T, n, k, part, ip);
    note_launch();
    if (e != cudaSuccess) return e;
    return launch_partial_reduce(part, ip, chunks, n, load, importance, s);
}

}  // namespace moe
