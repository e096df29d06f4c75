// Grouped expert FFN on the CUDA cores (fp32 FFMA): the fp32-expert path.
//
// "Mixture of Experts: Outrageously Large Neural Networks" (intuitivepapers.ai),
// "How a mixture-of-experts layer works": every expert is an input layer, one
// hidden layer of ReLU units and an output layer with its own weights, no biases:
// E_e(x) = ReLU(x W_in[e]) W_out[e].  Expert e runs on rows [offsets[e], offsets[e+1])
// of the expert-grouped buffer; an expert without rows is never touched.
#include <stdint.h>

#include "common.cuh"
#include "launch.h"

namespace moe {
namespace {

constexpr int FM = 64, FN = 64, FK = 16, FTHREADS = 256;

__device__ __forceinline__ void load4(const float* p, float o[4]) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
}
__device__ __forceinline__ void load4(const __nv_bfloat16* p, float o[4]) {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&v.x);
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&v.y);
    o[0] = __low2float(a); o[1] = __high2float(a); o[2] = __low2float(b); o[3] = __high2float(b);
}

// C[p, :] = act(A[p, :] W[e(p)]) for the 64-row x 64-column tile (blockIdx.y, blockIdx.x).
// A tile may straddle several experts: each expert segment of the tile is computed
// in turn with that expert's weights and only its rows are stored.
template <typename TA, typename TW, typename TC, bool RELU>
__global__ void __launch_bounds__(FTHREADS)
grouped_gemm_simt_kernel(const TA* __restrict__ A, const int32_t* __restrict__ offsets,
                         const TW* __restrict__ W, TC* __restrict__ C, long long R, int K, int N,
                         int n) {
    __shared__ float as[FK][FM + 4];
    __shared__ float ws[FK][FN];
    const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
    const long long r0 = (long long)blockIdx.y * FM;
    const long long r_end = min(R, r0 + FM);
    const int c0 = blockIdx.x * FN;
    // first expert whose rows reach r0: the last e with offsets[e] <= r0
    int lo = 0, hi = n;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (offsets[mid] <= r0) lo = mid; else hi = mid - 1;
    }
    const int la_row = tid / 4, la_k = (tid % 4) * 4;
    const int lw_k = tid / 16, lw_c = (tid % 16) * 4;
    for (int e = lo; e < n && offsets[e] < r_end; ++e) {
        const long long s0 = max(r0, (long long)offsets[e]);
        const long long s1 = min(r_end, (long long)offsets[e + 1]);
        if (s0 >= s1) continue;
        const TW* We = W + (size_t)e * K * N;
        float acc[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;
        for (int k0 = 0; k0 < K; k0 += FK) {
            float av[4] = {0.f, 0.f, 0.f, 0.f};
            const long long row = r0 + la_row;
            if (row >= s0 && row < s1) load4(A + (size_t)row * K + k0 + la_k, av);
#pragma unroll
            for (int q = 0; q < 4; ++q) as[la_k + q][la_row] = av[q];
            float wv[4];
            load4(We + (size_t)(k0 + lw_k) * N + c0 + lw_c, wv);
#pragma unroll
            for (int q = 0; q < 4; ++q) ws[lw_k][lw_c + q] = wv[q];
            __syncthreads();
#pragma unroll
            for (int kk = 0; kk < FK; ++kk) {
                float a[4], b[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) a[i] = as[kk][ty + 16 * i];
#pragma unroll
                for (int j = 0; j < 4; ++j) b[j] = ws[kk][tx + 16 * j];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
            }
            __syncthreads();
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const long long row = r0 + ty + 16 * i;
            if (row < s0 || row >= s1) continue;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float v = acc[i][j];
                if (RELU) v = fmaxf(v, 0.0f);
                C[(size_t)row * N + c0 + tx + 16 * j] = from_f32<TC>(v);
            }
        }
    }
}

}  // namespace

cudaError_t launch_ffn_simt(const float* x_perm, const int32_t* offsets, const float* W_in,
                            const float* W_out, float* y_perm, float* hidden, long long R, int d,
                            int h, int n, cudaStream_t s) {
    if (R == 0) return cudaSuccess;
    const unsigned mt = (unsigned)((R + FM - 1) / FM);
    grouped_gemm_simt_kernel<float, float, float, true>
        <<<dim3(h / FN, mt), FTHREADS, 0, s>>>(x_perm, offsets, W_in, hidden, R, d, h, n);
    note_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    grouped_gemm_simt_kernel<float, float, float, false>
        <<<dim3(d / FN, mt), FTHREADS, 0, s>>>(hidden, offsets, W_out, y_perm, R, h, d, n);
    note_launch();
    return cudaGetLastError();
}

}  // namespace moe
