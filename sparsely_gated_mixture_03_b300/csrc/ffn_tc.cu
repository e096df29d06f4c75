// Grouped expert FFN on the 5th-generation tensor cores (tcgen05, bf16 in,
// fp32 accumulation in TMEM), operands staged by TMA.
//
// "Mixture of Experts: Outrageously Large Neural Networks" (intuitivepapers.ai),
// "How a mixture-of-experts layer works": E_e(x) = ReLU(x W_in[e]) W_out[e]; expert e
// runs on rows [offsets[e], offsets[e+1]) of the expert-grouped buffer and an expert
// without rows is never touched.  Section "Keeping each expert's batch large"
// describes the shrinking per-expert batch that the tile schedule below has to
// live with: tiles are (expert, 128-row block, N block), only non-empty row
// blocks exist, and the schedule is read from device memory so the host never
// waits for the routing.
//
// Two launches of one persistent kernel: hidden = ReLU(x_perm W_in[e]) (bf16),
// then y_perm = hidden W_out[e] (fp16).  One CTA per SM; warp 0 issues TMA
// loads, warp 1 issues tcgen05.mma, warps 2-5 drain the double-buffered TMEM
// accumulator and store.  Tile order: expert-major, then N block, then row
// block, so CTAs that run at the same time share the same weight tile in L2.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include "common.cuh"
#include "launch.h"
#include "tc.cuh"

namespace moe {
namespace {

constexpr int BM = 128;        // rows per tile (TMEM lanes)
constexpr int BK = 64;         // K per stage: one 128-byte swizzle row of bf16
constexpr int STAGES = 4;
constexpr int THREADS = 192;   // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int A_BYTES = BM * BK * 2;

struct Barriers {
    uint64_t full[STAGES], empty[STAGES], tfull[2], tempty[2], done;
    uint32_t tmem_base;
    int abort_flag;
};

template <int BN>
constexpr int stage_bytes() { return A_BYTES + BK * BN * 2; }
template <int BN>
constexpr size_t smem_bytes() { return 1024 + (size_t)STAGES * stage_bytes<BN>() + sizeof(Barriers); }

struct Tile {
    int e, row0, row_end, n0;
};

// tile -> (expert, first row, end of the expert's rows, first column).  Tiles of
// expert e occupy [mt_prefix[e]*NT, mt_prefix[e+1]*NT), N block major, row block minor.
__device__ __forceinline__ Tile decode_tile(int tile, const int32_t* __restrict__ mt_prefix,
                                            const int32_t* __restrict__ offsets, int n, int NT,
                                            int BN) {
    int lo = 0, hi = n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (mt_prefix[mid] * NT <= tile) lo = mid; else hi = mid - 1;
    }
    const int mt_e = mt_prefix[lo + 1] - mt_prefix[lo];
    const int local = tile - mt_prefix[lo] * NT;
    Tile t;
    t.e = lo;
    t.row0 = offsets[lo] + (local % mt_e) * BM;
    t.row_end = offsets[lo + 1];
    t.n0 = (local / mt_e) * BN;
    return t;
}

// Bounded wait that ignores the abort flag: used to let copies or MMAs already
// in flight finish before the CTA releases its shared memory and TMEM.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, int* err) {
    const long long t0 = clock64();
    while (!tc::mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > tc::kWaitCycles) { raise_error(err, DEV_TIMEOUT); return; }
    }
}

template <int BN, bool RELU>
__global__ void __launch_bounds__(THREADS, 1)
ffn_gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   uint16_t* __restrict__ out, int N, int K,
                   const int32_t* __restrict__ offsets, const int32_t* __restrict__ mt_prefix, int n,
                   int* err) {
    constexpr int SB = stage_bytes<BN>();
    constexpr uint32_t TMEM_COLS = 2 * BN;
    constexpr uint32_t IDESC = tc::idesc_bf16_f32(BM, BN, false, true);
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    Barriers* bar = reinterpret_cast<Barriers*>(smem + STAGES * SB);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NT = N / BN;
    const int total = mt_prefix[n] * NT;
    const int KB = K / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) { tc::mbar_init(&bar->full[s], 1); tc::mbar_init(&bar->empty[s], 1); }
        for (int a = 0; a < 2; ++a) { tc::mbar_init(&bar->tfull[a], 1); tc::mbar_init(&bar->tempty[a], 4); }
        tc::mbar_init(&bar->done, 1);
        bar->abort_flag = 0;
        tc::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) { tc::tma_prefetch(&tmA); tc::tma_prefetch(&tmB); }
    if (warp == 1) tc::tmem_alloc(&bar->tmem_base, TMEM_COLS);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = bar->tmem_base;
    volatile int* abort_flag = &bar->abort_flag;

    if (warp == 0) {
        if (lane == 0) {   // ---------------- TMA producer
            int stage = 0;
            uint32_t phase = 0, armed = 0, armed_parity = 0;
            for (int tile = blockIdx.x; tile < total && !*abort_flag; tile += gridDim.x) {
                const Tile t = decode_tile(tile, mt_prefix, offsets, n, NT, BN);
                for (int kb = 0; kb < KB; ++kb) {
                    if (!tc::mbar_wait(&bar->empty[stage], phase ^ 1, abort_flag, err)) break;
                    uint8_t* a_dst = smem + stage * SB;
                    uint8_t* b_dst = a_dst + A_BYTES;
                    tc::mbar_arrive_expect_tx(&bar->full[stage], SB);
                    tc::tma_load_2d(a_dst, &tmA, &bar->full[stage], kb * BK, t.row0);
#pragma unroll
                    for (int i = 0; i < BN / 64; ++i)
                        tc::tma_load_3d(b_dst + i * (BK * 128), &tmB, &bar->full[stage],
                                        t.n0 + 64 * i, kb * BK, t.e);
                    armed |= 1u << stage;
                    armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
            }
            for (int s = 0; s < STAGES; ++s)     // copies in flight land before exit
                if ((armed >> s) & 1u) drain_wait(&bar->full[s], (armed_parity >> s) & 1u, err);
        }
    } else if (warp == 1) {
        if (lane == 0) {   // ---------------- MMA issuer
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
                        // A: K-major rows of 128 B, 8-row atoms 1024 B apart; +32 B per K=16.
                        const uint64_t ad = tc::sdesc_sw128(a_addr + kk * 32, 16, 1024);
                        // B: N-major; a K row of 64 N values is 128 B, 8-row atoms 1024 B
                        // apart (SBO), 64-wide N blocks BK*128 B apart (LBO); +2048 B per K=16.
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
            tc::mma_commit(&bar->done);          // every MMA done before TMEM is freed
            drain_wait(&bar->done, 0, err);
        }
    } else {               // ---------------- epilogue: warps 2..5
        const int quarter = warp & 3;            // TMEM lanes 32*quarter .. +31
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
            const Tile t = decode_tile(tile, mt_prefix, offsets, n, NT, BN);
            // lane 0 waits and the warp follows its verdict, so the warp-collective
            // TMEM loads below are always executed by all 32 lanes or by none
            int ok = 0;
            if (lane == 0) ok = tc::mbar_wait(&bar->tfull[acc], acc_phase, abort_flag, err) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc::fence_after_sync();
            const int row = t.row0 + quarter * 32 + lane;
            const bool live = row < t.row_end;
            uint16_t* dst = out + (size_t)(live ? row : 0) * N + t.n0;
            const uint32_t t_addr = tmem + acc * BN + ((uint32_t)(quarter * 32) << 16);
#pragma unroll 1
            for (int col = 0; col < BN; col += 32) {
                uint32_t r[32];
                tc::tmem_ld32(t_addr + col, r);
                tc::tmem_ld_wait();
                if (live) {
                    uint4 pk[4];
                    uint32_t* pw = reinterpret_cast<uint32_t*>(pk);
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        float v0 = __uint_as_float(r[2 * q]), v1 = __uint_as_float(r[2 * q + 1]);
                        if (RELU) {      // hidden layer: ReLU, bf16 (the next product's operand)
                            const __nv_bfloat162 b2 =
                                __floats2bfloat162_rn(fmaxf(v0, 0.0f), fmaxf(v1, 0.0f));
                            pw[q] = *reinterpret_cast<const uint32_t*>(&b2);
                        } else {         // expert output: fp16
                            const __half2 h2 = __floats2half2_rn(v0, v1);
                            pw[q] = *reinterpret_cast<const uint32_t*>(&h2);
                        }
                    }
                    uint4* d4 = reinterpret_cast<uint4*>(dst + col);
#pragma unroll
                    for (int q = 0; q < 4; ++q) d4[q] = pk[q];
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

// Row-major [rows, cols] bf16, boxes of 64 columns x 128 rows, 128-byte swizzle.
bool make_rows_map(CUtensorMap* m, const void* base, long long rows, int cols) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {64, BM};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Expert weights [n][K][N] bf16 (N contiguous), boxes of 64 N x 64 K x 1 expert.
bool make_weight_map(CUtensorMap* m, const void* base, int n, int K, int N) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[3] = {(cuuint64_t)N, (cuuint64_t)K, (cuuint64_t)n};
    cuuint64_t strides[2] = {(cuuint64_t)N * 2, (cuuint64_t)K * N * 2};
    cuuint32_t box[3] = {64, BK, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms > 0 ? sms : 148;
}

template <int BN, bool RELU>
cudaError_t launch_gemm(const CUtensorMap& a, const CUtensorMap& b, void* out, int N, int K,
                        const int32_t* offsets, const int32_t* mt_prefix, int n, int* err,
                        cudaStream_t s) {
    static bool configured = false;
    const size_t smem = smem_bytes<BN>();
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(ffn_gemm_tc_kernel<BN, RELU>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    ffn_gemm_tc_kernel<BN, RELU><<<sm_count(), THREADS, smem, s>>>(
        a, b, static_cast<uint16_t*>(out), N, K, offsets, mt_prefix, n, err);
    note_launch();
    return cudaGetLastError();
}

template <bool RELU>
cudaError_t launch_gemm_n(const CUtensorMap& a, const CUtensorMap& b, void* out, int N, int K,
                          const int32_t* offsets, const int32_t* mt_prefix, int n, int* err,
                          cudaStream_t s) {
    if (N % 256 == 0) return launch_gemm<256, RELU>(a, b, out, N, K, offsets, mt_prefix, n, err, s);
    if (N % 128 == 0) return launch_gemm<128, RELU>(a, b, out, N, K, offsets, mt_prefix, n, err, s);
    return launch_gemm<64, RELU>(a, b, out, N, K, offsets, mt_prefix, n, err, s);
}

}  // namespace

size_t ffn_tc_prefix_entries(int n) { return (size_t)n + 1; }

cudaError_t launch_ffn_tc(const void* x_perm, const int32_t* offsets, const void* W_in,
                          const void* W_out, void* y_perm, void* hidden, int32_t* mt_prefix,
                          long long R, int d, int h, int n, int* err, cudaStream_t s) {
    if (R == 0) return cudaSuccess;
    CUtensorMap a1, b1, a2, b2;
    if (!make_rows_map(&a1, x_perm, R, d) || !make_weight_map(&b1, W_in, n, d, h) ||
        !make_rows_map(&a2, hidden, R, h) || !make_weight_map(&b2, W_out, n, h, d))
        return cudaErrorInvalidValue;
    // mt_prefix[e] = sum over e' < e of ceil(rows(e') / BM); mt_prefix[n] = all row blocks
    cudaError_t e = launch_row_block_prefix(offsets, n, BM, mt_prefix, s);
    if (e != cudaSuccess) return e;
    e = launch_gemm_n<true>(a1, b1, hidden, h, d, offsets, mt_prefix, n, err, s);
    if (e != cudaSuccess) return e;
    return launch_gemm_n<false>(a2, b2, y_perm, d, h, offsets, mt_prefix, n, err, s);
}

}  // namespace moe
