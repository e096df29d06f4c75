// Gate logits on the 5th-generation tensor cores for bf16 inputs.
//
// "Mixture of Experts: Outrageously Large Neural Networks" (intuitivepapers.ai),
// section "Noisy top-k gating", eq (4):
//     clean = x W_g (+ b_g),  std = Softplus(x W_noise) + floor,  H = clean + eps * std.
// W_g and W_noise are fp32 and the logits must match fp32-or-better arithmetic, so
// each weight is split exactly into three bf16 terms, W = hi + mid + lo (each the
// bf16 rounding of what the previous terms leave; the remainder after three terms
// is below 2^-24 |W|).  x is bf16 already, so x W = x hi + x mid + x lo is one bf16
// GEMM with K = 3d whose A operand is the same x tile read three times: bf16 x bf16
// products are exact in fp32 and the tensor core accumulates them in fp32 in TMEM.
// The tensor core's fp32 accumulation truncates, so the terms are accumulated in
// the order lo, mid, hi: the small terms are summed while the accumulator is still
// small, and only the hi term's steps round at full size (measured on B300: the
// logits then match an fp32 FFMA dot product's accuracy).
//
// Layout of the split weights W3 [3d][2 n_pad] (bf16, N contiguous): rows s*d + i hold
// term s of row i; columns come in chunks of 256, chunk j = [W_g columns of experts
// 128j..128j+127 | W_noise columns of the same experts], zero past n.  One tile of
// this file's kernel is 128 tokens x one chunk: TMEM columns 0..127 accumulate the
// clean logits and 128..255 the noise logits of the same 128 experts.  This kernel
// writes clean/std/H to memory (the debug copy, and the path for n > 256); the fused
// gate of gate_fused.cu keeps them on the SM.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include "common.cuh"
#include "launch.h"
#include "tc.cuh"

namespace moe {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int EPT = BN / 2;      // experts per chunk
constexpr int BK = 64;
constexpr int STAGES = 4;
constexpr int THREADS = 192;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BK * BN * 2;
constexpr int SB = A_BYTES + B_BYTES;
constexpr uint32_t TMEM_COLS = 2 * BN;
constexpr uint32_t IDESC = tc::idesc_bf16_f32(BM, BN, false, true);

struct Barriers {
    uint64_t full[STAGES], empty[STAGES], tfull[2], tempty[2], done;
    uint32_t tmem_base;
    int abort_flag;
};
constexpr size_t SMEM_BYTES = 1024 + (size_t)STAGES * SB + sizeof(Barriers);

// blockIdx.y = group: W_g, W_noise [groups][d][n] -> W3 [groups][3d][2 n_pad]
// (one group for the flat gate).
__global__ void gate_split_weights_kernel(const float* __restrict__ W_g,
                                          const float* __restrict__ W_noise, int d, int n,
                                          int n_pad, __nv_bfloat16* __restrict__ W3) {
    const long long cols = 2LL * n_pad;
    const long long total = (long long)d * cols;
    griddep_wait();
    griddep_launch_dependents();
    W_g += (size_t)blockIdx.y * d * n;
    W_noise += (size_t)blockIdx.y * d * n;
    W3 += (size_t)blockIdx.y * 3 * d * cols;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int row = (int)(i / cols);
        const int col = (int)(i % cols);
        const int c = col % BN;
        const int e = (col / BN) * EPT + (c % EPT);
        const float* src = c < EPT ? W_g : W_noise;
        const float w = e < n ? src[(size_t)row * n + e] : 0.0f;
        const __nv_bfloat16 hi = __float2bfloat16_rn(w);
        const float r1 = w - __bfloat162float(hi);          // exact in fp32
        const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
        const float r2 = r1 - __bfloat162float(mid);        // exact in fp32
        const __nv_bfloat16 lo = __float2bfloat16_rn(r2);
        W3[((size_t)0 * d + row) * cols + col] = hi;
        W3[((size_t)1 * d + row) * cols + col] = mid;
        W3[((size_t)2 * d + row) * cols + col] = lo;
    }
}

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, int* err) {
    const long long t0 = clock64();
    while (!tc::mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > tc::kWaitCycles) { raise_error(err, DEV_TIMEOUT); return; }
    }
}

__global__ void __launch_bounds__(THREADS, 1)
gate_logits_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                      const float* __restrict__ eps, const float* __restrict__ b_g, int T, int d,
                      int n, int n_pad, float std_floor, float* __restrict__ clean_out,
                      float* __restrict__ std_out, float* __restrict__ H_out, int* err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    Barriers* bar = reinterpret_cast<Barriers*>(smem + STAGES * SB);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NT = n_pad / EPT;                 // expert chunks
    const int total = ((T + BM - 1) / BM) * NT;
    const int KBX = d / BK;                     // k-blocks of one term
    const int KB = 3 * KBX;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) { tc::mbar_init(&bar->full[s], 1); tc::mbar_init(&bar->empty[s], 1); }
        for (int a = 0; a < 2; ++a) { tc::mbar_init(&bar->tfull[a], 1); tc::mbar_init(&bar->tempty[a], 4); }
        tc::mbar_init(&bar->done, 1);
        bar->abort_flag = 0;
        tc::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) { tc::tma_prefetch(&tmX); tc::tma_prefetch(&tmW); }
    if (warp == 1) tc::tmem_alloc(&bar->tmem_base, TMEM_COLS);
    griddep_wait();                    // inputs written by the previous kernel are visible
    griddep_launch_dependents();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = bar->tmem_base;
    volatile int* abort_flag = &bar->abort_flag;

    if (warp == 0) {
        if (lane == 0) {   // TMA producer
            int stage = 0;
            uint32_t phase = 0, armed = 0, armed_parity = 0;
            for (int tile = blockIdx.x; tile < total && !*abort_flag; tile += gridDim.x) {
                const int m0 = (tile / NT) * BM, col0 = (tile % NT) * BN;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!tc::mbar_wait(&bar->empty[stage], phase ^ 1, abort_flag, err)) break;
                    uint8_t* a_dst = smem + stage * SB;
                    uint8_t* b_dst = a_dst + A_BYTES;
                    const int term = 2 - kb / KBX;      // lo, mid, hi
                    tc::mbar_arrive_expect_tx(&bar->full[stage], SB);
                    tc::tma_load_2d(a_dst, &tmX, &bar->full[stage], (kb % KBX) * BK, m0);
#pragma unroll
                    for (int i = 0; i < BN / 64; ++i)
                        tc::tma_load_2d(b_dst + i * (BK * 128), &tmW, &bar->full[stage], col0 + 64 * i,
                                        term * d + (kb % KBX) * BK);
                    armed |= 1u << stage;
                    armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
            }
            for (int s = 0; s < STAGES; ++s)
                if ((armed >> s) & 1u) drain_wait(&bar->full[s], (armed_parity >> s) & 1u, err);
        }
    } else if (warp == 1) {
        if (lane == 0) {   // MMA issuer
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            for (int tile = blockIdx.x; tile < total && !*abort_flag; tile += gridDim.x) {
                if (!tc::mbar_wait(&bar->tempty[acc], acc_phase ^ 1, abort_flag, err)) break;
                tc::fence_after_sync();
                const uint32_t d_tmem = tmem + acc * BN;
                bool ok = true;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!tc::mbar_wait(&bar->full[stage], phase, abort_flag, err)) { ok = false; break; }
                    tc::fence_after_sync();
                    const uint32_t a_addr = tc::smem_u32(smem + stage * SB);
                    const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        const uint64_t ad = tc::sdesc_sw128(a_addr + kk * 32, 16, 1024);
                        const uint64_t bd = tc::sdesc_sw128(b_addr + kk * 2048, BK * 128, 1024);
                        tc::mma_bf16(d_tmem, ad, bd, IDESC, (kb | kk) != 0 ? 1u : 0u);
                    }
                    tc::mma_commit(&bar->empty[stage]);
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                tc::mma_commit(&bar->tfull[acc]);
                if (++acc == 2) { acc = 0; acc_phase ^= 1; }
            }
            tc::mma_commit(&bar->done);
            drain_wait(&bar->done, 0, err);
        }
    } else {               // epilogue: warps 2..5, one token row per thread
        const int quarter = warp & 3;
        int acc = 0;
        uint32_t acc_phase = 0;
        const bool vec = (n % 4) == 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
            int ok = 0;
            if (lane == 0) ok = tc::mbar_wait(&bar->tfull[acc], acc_phase, abort_flag, err) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc::fence_after_sync();
            const int t = (tile / NT) * BM + quarter * 32 + lane;
            const int e_base = (tile % NT) * EPT;
            const bool live = t < T;
            const uint32_t t_addr = tmem + acc * BN + ((uint32_t)(quarter * 32) << 16);
#pragma unroll 1
            for (int c = 0; c < EPT; c += 32) {
                uint32_t rc[32], rr[32];
                tc::tmem_ld32(t_addr + c, rc);
                tc::tmem_ld32(t_addr + EPT + c, rr);
                tc::tmem_ld_wait();
                const int e0 = e_base + c;
                if (!live || e0 >= n) continue;
                const size_t o = (size_t)t * n + e0;
                if (vec && e0 + 32 <= n) {
#pragma unroll
                    for (int q = 0; q < 32; q += 4) {
                        const float4 ep = eps != nullptr   // eps == nullptr: no noise
                                              ? *reinterpret_cast<const float4*>(eps + o + q)
                                              : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                        float cv[4], sv[4], hv[4];
                        const float epv[4] = {ep.x, ep.y, ep.z, ep.w};
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            cv[u] = __uint_as_float(rc[q + u]) + (b_g != nullptr ? b_g[e0 + q + u] : 0.0f);
                            sv[u] = softplus_f32(__uint_as_float(rr[q + u])) + std_floor;
                            hv[u] = fmaf(epv[u], sv[u], cv[u]);
                        }
                        *reinterpret_cast<float4*>(clean_out + o + q) = make_float4(cv[0], cv[1], cv[2], cv[3]);
                        *reinterpret_cast<float4*>(std_out + o + q) = make_float4(sv[0], sv[1], sv[2], sv[3]);
                        *reinterpret_cast<float4*>(H_out + o + q) = make_float4(hv[0], hv[1], hv[2], hv[3]);
                    }
                } else {
#pragma unroll
                    for (int q = 0; q < 32; ++q) {
                        if (e0 + q >= n) break;
                        const float cv = __uint_as_float(rc[q]) + (b_g != nullptr ? b_g[e0 + q] : 0.0f);
                        const float sv = softplus_f32(__uint_as_float(rr[q])) + std_floor;
                        clean_out[o + q] = cv;
                        std_out[o + q] = sv;
                        H_out[o + q] = eps != nullptr ? fmaf(eps[o + q], sv, cv) : cv;
                    }
                }
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&bar->tempty[acc]);
            if (++acc == 2) { acc = 0; acc_phase ^= 1; }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 1) tc::tmem_dealloc(tmem, TMEM_COLS);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (fn == nullptr) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

int sm_count() {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms > 0 ? sms : 148;
}

}  // namespace

int gate_tc_n_pad(int n) { return (n + EPT - 1) / EPT * EPT; }

bool gate_bf16_map(CUtensorMap* m, const void* base, long long rows, long long cols, int box_rows) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int gate_sm_count() { return sm_count(); }

cudaError_t launch_gate_split_weights(const float* W_g, const float* W_noise, int d, int n,
                                      void* W3, cudaStream_t s) {
    return launch_gate_split_weights_grouped(W_g, W_noise, 1, d, n, W3, s);
}

cudaError_t launch_gate_split_weights_grouped(const float* W_g, const float* W_noise, int groups,
                                              int d, int n, void* W3, cudaStream_t s) {
    if (groups < 1 || groups > 65535) return cudaErrorInvalidValue;
    int bx = 4 * sm_count() / groups;
    if (bx < 8) bx = 8;
    const cudaError_t e =
        launch_pdl(gate_split_weights_kernel, dim3(bx, groups), dim3(256), 0, s, 1, W_g, W_noise, d,
                   n, gate_tc_n_pad(n), static_cast<__nv_bfloat16*>(W3));
    note_launch();
    return e;
}

cudaError_t launch_gate_logits_tc(const void* x, const float* W_g, const float* W_noise,
                                  const float* eps, const float* b_g, int T, int d, int n,
                                  float std_floor, void* W3, float* clean, float* stdv, float* H,
                                  int* err, cudaStream_t s) {
    const int n_pad = gate_tc_n_pad(n);
    cudaError_t e = launch_gate_split_weights(W_g, W_noise, d, n, W3, s);
    if (e != cudaSuccess) return e;
    CUtensorMap mx, mw;
    if (!gate_bf16_map(&mx, x, T, d, BM) || !gate_bf16_map(&mw, W3, 3LL * d, 2LL * n_pad, BK))
        return cudaErrorInvalidValue;
    static bool configured = false;
    if (!configured) {
        e = cudaFuncSetAttribute(gate_logits_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)SMEM_BYTES);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    e = launch_pdl(gate_logits_tc_kernel, dim3(sm_count()), dim3(THREADS), SMEM_BYTES, s, 1, mx, mw,
                   eps, b_g, T, d, n, n_pad, std_floor, clean, stdv, H, err);
    note_launch();
    return e;
}

}  // namespace moe
