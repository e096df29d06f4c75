// The gate's share of the input gradient on the 5th-generation tensor cores.
//
// "Mixture of Experts: Outrageously Large Neural Networks" (intuitivepapers.ai),
// "Implementation notes": the gate's weights pass gradient back to x through both of
// its products, so dx gets dclean W_g^T + dnz W_noise^T on top of the experts' share
// (eq (4): clean = x W_g, nz = x W_noise).
//
// fp32 operands on bf16 tensor cores: the gate backward writes dclean and dnz as
// two-term bf16 splits (hi + lo, [T][4n]: clean hi, clean lo, noise hi, noise lo) and
// gate_dx_split_kernel splits W_g and W_noise the same way ([4][d][n]); the products
// hi*hi, hi*lo and lo*hi of each pair are accumulated in fp32 in TMEM (small terms
// first), leaving out lo*lo (about 2^-16 of the product), so the result keeps about
// 2^-15 relative precision.  One GEMM with M = T (tokens), N = d, K = 6 n: its
// k-blocks walk six (A plane, B plane) segments, both operands K-contiguous.
// The epilogue adds each 32 x 32 fp32 tile into dx with a TMA reduce-add (one add per
// element: the result does not depend on timing).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include "common.cuh"
#include "launch.h"
#include "tc.cuh"

namespace moe {
namespace {

constexpr int BM = 128;                  // tokens a tile
constexpr int BN = 256;                  // columns of dx a tile
constexpr int BK = 64;
constexpr int STAGES = 3;
constexpr int THREADS = 192;
constexpr int A_BYTES = BM * BK * 2;     // 16 KB
constexpr int B_BYTES = BN * BK * 2;     // 32 KB
constexpr int SB = A_BYTES + B_BYTES;
constexpr uint32_t TMEM_COLS = 2 * BN;
constexpr uint32_t IDESC = tc::idesc_bf16_f32(BM, BN, false, false);   // A and B K-major
constexpr int ST = 32;                   // reduce tiles: 32 rows x 32 fp32 columns (128 B rows)
constexpr int ST_BYTES = ST * ST * 4;
constexpr int STAGING = 4 * 2 * ST_BYTES;
constexpr int SEGS = 6;
// (A plane, B plane) of each k segment, small products first: clean lo * W_g hi,
// clean hi * W_g lo, noise lo * W_noise hi, noise hi * W_noise lo, then the two hi * hi.
__constant__ int kSegA[SEGS] = {1, 0, 3, 2, 0, 2};
__constant__ int kSegB[SEGS] = {0, 1, 2, 3, 0, 2};

struct Barriers {
    uint64_t full[STAGES], empty[STAGES], tfull[2], tempty[2], done;
    uint32_t tmem_base;
    int abort_flag;
};
constexpr size_t SMEM_BYTES = 1024 + (size_t)STAGES * SB + STAGING + sizeof(Barriers);
static_assert(SMEM_BYTES <= 232448, "shared memory of one CTA");

// W2 [4][d][n] bf16: W_g hi, W_g lo, W_noise hi, W_noise lo.
__global__ void gate_dx_split_kernel(const float* __restrict__ W_g, const float* __restrict__ W_noise,
                                     long long count, __nv_bfloat16* __restrict__ W2) {
    griddep_wait();
    griddep_launch_dependents();
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < count;
         i += (long long)gridDim.x * blockDim.x) {
        const float g = W_g[i], z = W_noise[i];
        const __nv_bfloat16 gh = __float2bfloat16_rn(g), zh = __float2bfloat16_rn(z);
        W2[i] = gh;
        W2[count + i] = __float2bfloat16_rn(g - __bfloat162float(gh));
        W2[2 * count + i] = zh;
        W2[3 * count + i] = __float2bfloat16_rn(z - __bfloat162float(zh));
    }
}

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, int* err) {
    const long long t0 = clock64();
    while (!tc::mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > tc::kWaitCycles) { raise_error(err, DEV_TIMEOUT); return; }
    }
}

__global__ void __launch_bounds__(THREADS, 1)
gate_dx_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const __grid_constant__ CUtensorMap tmDX, int T, int d, int n, int* err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* staging = smem + STAGES * SB;
    Barriers* bar = reinterpret_cast<Barriers*>(staging + STAGING);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NT = d / BN;
    const int total = ((T + BM - 1) / BM) * NT;
    const int KBX = n / BK;                     // k-blocks of one segment
    const int KB = SEGS * KBX;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) { tc::mbar_init(&bar->full[s], 1); tc::mbar_init(&bar->empty[s], 1); }
        for (int a = 0; a < 2; ++a) { tc::mbar_init(&bar->tfull[a], 1); tc::mbar_init(&bar->tempty[a], 4); }
        tc::mbar_init(&bar->done, 1);
        bar->abort_flag = 0;
        tc::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) { tc::tma_prefetch(&tmA); tc::tma_prefetch(&tmB); tc::tma_prefetch(&tmDX); }
    if (warp == 1) tc::tmem_alloc(&bar->tmem_base, TMEM_COLS);
    griddep_wait();                    // dclean / dnz and the expert share of dx are written
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
                    const int seg = kb / KBX, kk = (kb % KBX) * BK;
                    tc::mbar_arrive_expect_tx(&bar->full[stage], SB);
                    tc::tma_load_2d(a_dst, &tmA, &bar->full[stage], kSegA[seg] * n + kk, m0);
                    tc::tma_load_2d(b_dst, &tmB, &bar->full[stage], kk, kSegB[seg] * d + col0);
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
            bool ok = true;
            for (int tile = blockIdx.x; tile < total && ok && !*abort_flag; tile += gridDim.x) {
                if (!tc::mbar_wait(&bar->tempty[acc], acc_phase ^ 1, abort_flag, err)) break;
                tc::fence_after_sync();
                for (int kb = 0; kb < KB; ++kb) {
                    if (!tc::mbar_wait(&bar->full[stage], phase, abort_flag, err)) { ok = false; break; }
                    tc::fence_after_sync();
                    const uint32_t a_addr = tc::smem_u32(smem + stage * SB);
                    const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
                    for (int k2 = 0; k2 < BK / 16; ++k2) {
                        // both operands K-major: 128-byte rows, 8-row atoms 1024 B apart
                        const uint64_t ad = tc::sdesc_sw128(a_addr + k2 * 32, 16, 1024);
                        const uint64_t bd = tc::sdesc_sw128(b_addr + k2 * 32, 16, 1024);
                        tc::mma_bf16(tmem + acc * BN, ad, bd, IDESC, (kb | k2) != 0 ? 1u : 0u);
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
    } else {               // epilogue: warps 2..5, TMEM lanes 32*quarter .. +31
        const int quarter = warp & 3;
        const int ew = warp - 2;
        uint8_t* sbuf[2] = {staging + (2 * ew) * ST_BYTES, staging + (2 * ew + 1) * ST_BYTES};
        int nbuf = 0, acc = 0;
        uint32_t acc_phase = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
            const int m0 = (tile / NT) * BM, col0 = (tile % NT) * BN;
            int w = 0;
            if (lane == 0) w = tc::mbar_wait(&bar->tfull[acc], acc_phase, abort_flag, err) ? 1 : 0;
            w = __shfl_sync(0xffffffffu, w, 0);
            if (!w) break;
            tc::fence_after_sync();
            const uint32_t t_addr = tmem + acc * BN + ((uint32_t)(quarter * 32) << 16);
#pragma unroll 1
            for (int c = 0; c < BN; c += ST) {
                uint32_t r[32];
                tc::tmem_ld32(t_addr + c, r);        // this lane's row, 32 columns
                tc::tmem_ld_wait();
                if (lane == 0) tc::bulk_wait_read<1>();   // the buffer's previous reduce read it
                __syncwarp();
                uint8_t* sb = sbuf[nbuf];
#pragma unroll
                for (int q = 0; q < 8; ++q)          // 128-byte swizzle: chunk q ^ (row & 7)
                    *reinterpret_cast<uint4*>(sb + lane * 128 + ((q ^ (lane & 7)) << 4)) =
                        make_uint4(r[4 * q], r[4 * q + 1], r[4 * q + 2], r[4 * q + 3]);
                tc::fence_proxy_async_shared();
                __syncwarp();
                // a box that starts past T is left out; rows past T inside a box are
                // clipped by the map
                if (lane == 0 && m0 + quarter * 32 < T) {
                    tc::tma_reduce_add_2d(&tmDX, sb, col0 + c, m0 + quarter * 32);
                    tc::bulk_commit();
                }
                nbuf ^= 1;
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&bar->tempty[acc]);
            if (++acc == 2) { acc = 0; acc_phase ^= 1; }
        }
        if (lane == 0) tc::bulk_wait_all();  // every reduce done before the CTA exits
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

// [rows][cols] bf16, K-major boxes of 64 columns x box_rows rows, 128-byte swizzle.
bool bf16_map(CUtensorMap* m, const void* base, long long rows, long long cols, int box_rows) {
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

// dx [T][d] fp32, boxes of 32 columns x 32 rows, 128-byte swizzle (the reduce-adds).
bool f32_map(CUtensorMap* m, void* base, long long rows, long long cols) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 4};
    cuuint32_t box[2] = {ST, ST};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int dx_sm_count() {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms > 0 ? sms : 148;
}

}  // namespace

bool gate_dx_tc_supported(int d, int n) { return d % BN == 0 && n % BK == 0; }

size_t gate_dx_split_bytes(int d, int n) { return (size_t)4 * d * n * 2; }

cudaError_t launch_gate_dx_tc(const float* W_g, const float* W_noise, const void* split, int T,
                              int d, int n, void* W2, float* dx, int* err, cudaStream_t s) {
    if (!gate_dx_tc_supported(d, n) || T <= 0) return cudaErrorInvalidValue;
    const long long count = (long long)d * n;
    cudaError_t e = launch_pdl(gate_dx_split_kernel, dim3(148 * 2), dim3(256), 0, s, 1, W_g,
                               W_noise, count, static_cast<__nv_bfloat16*>(W2));
    note_launch();
    if (e != cudaSuccess) return e;
    CUtensorMap ma, mb, mdx;
    if (!bf16_map(&ma, split, T, 4LL * n, BM) || !bf16_map(&mb, W2, 4LL * d, n, BN) ||
        !f32_map(&mdx, dx, T, d))
        return cudaErrorInvalidValue;
    static bool configured = false;
    if (!configured) {
        e = cudaFuncSetAttribute(gate_dx_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)SMEM_BYTES);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    e = launch_pdl(gate_dx_tc_kernel, dim3(dx_sm_count()), dim3(THREADS), SMEM_BYTES, s, 1, ma, mb,
                   mdx, T, d, n, err);
    note_launch();
    return e;
}

}  // namespace moe
