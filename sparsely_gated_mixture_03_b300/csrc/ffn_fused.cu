// Expert FFN as one persistent tcgen05 kernel that runs both products, with the
// hidden layer kept in L2 between them.
//
// "Mixture of Experts: Outrageously Large Neural Networks" (intuitivepapers.ai),
// "How a mixture-of-experts layer works": E_e(x) = ReLU(x W_in[e]) W_out[e]; expert e
// runs on rows [offsets[e], offsets[e+1]) of the expert-grouped buffer and an expert
// without rows is never touched.
//
// Work items (one CTA per SM, each CTA takes items i = blockIdx.x, + gridDim.x, ...
// in increasing order):
//   phase 1 (q, j): hidden[rows of q, block j] = ReLU(x_perm[rows] W_in[e]) as bf16,
//   phase 2 (q, j): y_perm[rows of q, block j] = hidden[rows] W_out[e] as fp16,
// for every 128-row block q of every expert e (blocks never mix experts).  The item
// list interleaves the phases with a lag: slot s holds the phase-1 items of block s,
// then the phase-2 items of block s - lag.  A phase-2 item waits (bounded) until the
// NT1 phase-1 items of its block have stored their hidden rows and counted them in
// done[q]; with the lag those rows were written a few microseconds earlier and are
// still in L2, so the hidden layer is written once and read back from L2 instead of
// DRAM.  Every dependency points to an earlier item, and the kernel is launched
// cooperatively (all CTAs resident), so the earliest unfinished item can always run.
//
// Roles: warp 0 issues TMA loads (A K-major, weights N-major, 128-byte swizzle,
// 4 stages), warp 1 issues tcgen05.mma (128 x BN x 16, fp32 accumulation in TMEM),
// warps 2-5 drain a double-buffered TMEM accumulator, apply ReLU / convert, store.
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
    int vote[4];
};

template <int BN>
constexpr int stage_bytes() { return A_BYTES + BK * BN * 2; }
template <int BN>
constexpr size_t smem_bytes() { return 1024 + (size_t)STAGES * stage_bytes<BN>() + sizeof(Barriers); }

struct Schedule {
    const int32_t* offsets;    // [n+1] rows of each expert
    const int32_t* blk;        // [n+1] prefix of 128-row blocks over the experts
    int32_t* done;             // [max blocks] phase-1 items finished per block (zeroed)
    int n, NT1, NT2, lag;
};

struct Item {
    int phase;                 // 1 or 2
    int q, j;                  // row block, N block
    int e, row0, row_end;      // expert and its rows
};

// Items before slot s: NT1 per slot below Q, NT2 per slot in [lag, lag + Q).
__device__ __forceinline__ long long items_before(int s, int Q, const Schedule& S) {
    const int p1 = min(s, Q);
    const int p2 = min(max(s - S.lag, 0), Q);
    return (long long)S.NT1 * p1 + (long long)S.NT2 * p2;
}

__device__ __forceinline__ Item decode_item(int i, int Q, const Schedule& S) {
    int lo = 0, hi = Q + S.lag - 1;              // last slot s with items_before(s) <= i
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (items_before(mid, Q, S) <= i) lo = mid; else hi = mid - 1;
    }
    const int s = lo;
    int r = i - (int)items_before(s, Q, S);
    Item it;
    const int n1 = s < Q ? S.NT1 : 0;
    if (r < n1) { it.phase = 1; it.q = s; it.j = r; }
    else { it.phase = 2; it.q = s - S.lag; it.j = r - n1; }
    int a = 0, b = S.n - 1;                      // expert of block q
    while (a < b) {
        const int mid = (a + b + 1) >> 1;
        if (S.blk[mid] <= it.q) a = mid; else b = mid - 1;
    }
    it.e = a;
    it.row0 = S.offsets[a] + (it.q - S.blk[a]) * BM;
    it.row_end = S.offsets[a + 1];
    return it;
}

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, int* err) {
    const long long t0 = clock64();
    while (!tc::mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > tc::kWaitCycles) { raise_error(err, DEV_TIMEOUT); return; }
    }
}

__device__ __forceinline__ int ld_acquire(const int32_t* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Waits until done[q] reaches `want`; false after kWaitCycles or on abort.
__device__ __forceinline__ bool wait_count(const int32_t* p, int want, volatile int* abort_flag,
                                           int* err) {
    if (ld_acquire(p) >= want) return true;
    const long long t0 = clock64();
    while (ld_acquire(p) < want) {
        if (*abort_flag) return false;
        if (clock64() - t0 > tc::kWaitCycles) {
            *abort_flag = 1;
            raise_error(err, DEV_TIMEOUT);
            return false;
        }
        __nanosleep(64);
    }
    return true;
}

template <int BN>
__global__ void __launch_bounds__(THREADS, 1)
ffn_fused_tc_kernel(const __grid_constant__ CUtensorMap tmA1, const __grid_constant__ CUtensorMap tmB1,
                    const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmB2,
                    uint16_t* __restrict__ hidden, uint16_t* __restrict__ out, int d, int h,
                    const Schedule S, int* err) {
    constexpr int SB = stage_bytes<BN>();
    constexpr uint32_t TMEM_COLS = 2 * BN;
    constexpr uint32_t IDESC = tc::idesc_bf16_f32(BM, BN, false, true);
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    Barriers* bar = reinterpret_cast<Barriers*>(smem + STAGES * SB);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Q = S.blk[S.n];
    const int total = (int)items_before(Q + S.lag, Q, S);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) { tc::mbar_init(&bar->full[s], 1); tc::mbar_init(&bar->empty[s], 1); }
        for (int a = 0; a < 2; ++a) { tc::mbar_init(&bar->tfull[a], 1); tc::mbar_init(&bar->tempty[a], 4); }
        tc::mbar_init(&bar->done, 1);
        bar->abort_flag = 0;
        tc::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tc::tma_prefetch(&tmA1); tc::tma_prefetch(&tmB1);
        tc::tma_prefetch(&tmA2); tc::tma_prefetch(&tmB2);
    }
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
            for (int i = blockIdx.x; i < total && !*abort_flag; i += gridDim.x) {
                const Item it = decode_item(i, Q, S);
                const CUtensorMap* ta = it.phase == 1 ? &tmA1 : &tmA2;
                const CUtensorMap* tb = it.phase == 1 ? &tmB1 : &tmB2;
                const int KB = (it.phase == 1 ? d : h) / BK;
                if (it.phase == 2) {
                    // the hidden rows of block q: written by NT1 phase-1 items (generic
                    // stores, released with their count), read here through TMA
                    if (!wait_count(S.done + it.q, S.NT1, abort_flag, err)) break;
                    fence_proxy_async_global();
                }
                for (int kb = 0; kb < KB; ++kb) {
                    if (!tc::mbar_wait(&bar->empty[stage], phase ^ 1, abort_flag, err)) break;
                    uint8_t* a_dst = smem + stage * SB;
                    uint8_t* b_dst = a_dst + A_BYTES;
                    tc::mbar_arrive_expect_tx(&bar->full[stage], SB);
                    tc::tma_load_2d(a_dst, ta, &bar->full[stage], kb * BK, it.row0);
#pragma unroll
                    for (int c = 0; c < BN / 64; ++c)
                        tc::tma_load_3d(b_dst + c * (BK * 128), tb, &bar->full[stage],
                                        it.j * BN + 64 * c, kb * BK, it.e);
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
            for (int i = blockIdx.x; i < total && !*abort_flag; i += gridDim.x) {
                const Item it = decode_item(i, Q, S);
                const int KB = (it.phase == 1 ? d : h) / BK;
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
        for (int i = blockIdx.x; i < total; i += gridDim.x) {
            const Item it = decode_item(i, Q, S);
            // the four warps vote, so all of them take the same branch (the named
            // barrier below must see all four or none)
            if (lane == 0)
                bar->vote[quarter] = tc::mbar_wait(&bar->tfull[acc], acc_phase, abort_flag, err) ? 1 : 0;
            epi_bar();
            const int ok = bar->vote[0] & bar->vote[1] & bar->vote[2] & bar->vote[3];
            epi_bar();                           // votes read before the next item's votes
            if (!ok) break;
            tc::fence_after_sync();
            const int N = it.phase == 1 ? h : d;
            uint16_t* base = it.phase == 1 ? hidden : out;
            const int row = it.row0 + quarter * 32 + lane;
            const bool live = row < it.row_end;
            uint16_t* dst = base + (size_t)(live ? row : 0) * N + it.j * BN;
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
                        const float v0 = __uint_as_float(r[2 * q]), v1 = __uint_as_float(r[2 * q + 1]);
                        if (it.phase == 1) {   // hidden layer: ReLU, bf16 (the next product's operand)
                            const __nv_bfloat162 b2 =
                                __floats2bfloat162_rn(fmaxf(v0, 0.0f), fmaxf(v1, 0.0f));
                            pw[q] = *reinterpret_cast<const uint32_t*>(&b2);
                        } else {               // expert output: fp16
                            check_half_range(v0, v1, err);
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
            if (it.phase == 1) {
                // all four warps' hidden stores of this item, then one count for block q
                // (the fence after the barrier makes the count release every store)
                fence_proxy_async_global();
                epi_bar();
                if (warp == 2 && lane == 0) {
                    __threadfence();
                    atomicAdd(S.done + it.q, 1);
                }
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 1) tc::tmem_dealloc(tmem, TMEM_COLS);
}

// done[0..count) = 0 (the phase-1 counters of every possible row block).
__global__ void zero_counts_kernel(int32_t* __restrict__ done, int count) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < count; i += gridDim.x * blockDim.x)
        done[i] = 0;
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

template <int BN>
cudaError_t launch_fused(const CUtensorMap& a1, const CUtensorMap& b1, const CUtensorMap& a2,
                         const CUtensorMap& b2, void* hidden, void* out, int d, int h,
                         const Schedule& S, int* err, cudaStream_t s) {
    static bool configured = false;
    const size_t smem = smem_bytes<BN>();
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(ffn_fused_tc_kernel<BN>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    // cooperative: every CTA is resident, which the cross-CTA waits rely on
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(sm_count());
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    uint16_t* hp = static_cast<uint16_t*>(hidden);
    uint16_t* op = static_cast<uint16_t*>(out);
    cudaError_t e = cudaLaunchKernelEx(&cfg, ffn_fused_tc_kernel<BN>, a1, b1, a2, b2, hp, op, d, h,
                                       S, err);
    note_launch();
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

int ffn_fused_count_entries(long long R, int n) { return (int)((R + BM - 1) / BM) + n; }

cudaError_t launch_ffn_fused(const void* x_perm, const int32_t* offsets, const void* W_in,
                             const void* W_out, void* y_perm, void* hidden, int32_t* blk,
                             int32_t* done, long long R, int d, int h, int n, int* err,
                             cudaStream_t s) {
    if (R == 0) return cudaSuccess;
    const int BN = (d % 256 == 0 && h % 256 == 0) ? 256 : (d % 128 == 0 && h % 128 == 0) ? 128 : 64;
    CUtensorMap a1, b1, a2, b2;
    if (!make_rows_map(&a1, x_perm, R, d) || !make_weight_map(&b1, W_in, n, d, h) ||
        !make_rows_map(&a2, hidden, R, h) || !make_weight_map(&b2, W_out, n, h, d))
        return cudaErrorInvalidValue;
    cudaError_t e = launch_row_block_prefix(offsets, n, BM, blk, s);
    if (e != cudaSuccess) return e;
    const int counts = ffn_fused_count_entries(R, n);
    zero_counts_kernel<<<(counts + 255) / 256 < 148 ? (counts + 255) / 256 : 148, 256, 0, s>>>(
        done, counts);
    note_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    Schedule S;
    S.offsets = offsets;
    S.blk = blk;
    S.done = done;
    S.n = n;
    S.NT1 = h / BN;
    S.NT2 = d / BN;
    // a phase-2 item trails its phase-1 items by about two rounds of the grid
    S.lag = (2 * sm_count() + S.NT1 + S.NT2 - 1) / (S.NT1 + S.NT2);
    if (S.lag < 2) S.lag = 2;
    if (BN == 256) return launch_fused<256>(a1, b1, a2, b2, hidden, y_perm, d, h, S, err, s);
    if (BN == 128) return launch_fused<128>(a1, b1, a2, b2, hidden, y_perm, d, h, S, err, s);
    return launch_fused<64>(a1, b1, a2, b2, hidden, y_perm, d, h, S, err, s);
}

}  // namespace moe
