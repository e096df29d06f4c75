// Expert FFN on pairs of SMs: tcgen05.mma with cta_group::2 (M = 256 rows per pair,
// 128 in each CTA's TMEM), both products in one persistent launch.
//
// "Mixture of Experts: Outrageously Large Neural Networks" (intuitivepapers.ai),
// "How a mixture-of-experts layer works": E_e(x) = ReLU(x W_in[e]) W_out[e]; expert e
// runs on rows [offsets[e], offsets[e+1]) of the expert-grouped buffer and an expert
// without rows is never touched.
//
// A cluster of two CTAs computes a 256-row x 256-column tile: each CTA loads its own
// 128 rows of A and half (128 columns) of B, and one thread of the leader (rank 0)
// issues the pair MMA, which reads B from both CTAs' shared memory.  Per SM this
// moves half the B bytes of a one-CTA 128 x 256 tile, so a stage is 32 KB and six
// stages fit.  The leader's full barrier of a stage expects both CTAs' bytes and is
// armed by the leader alone (no cluster-scope release per stage).  Work units are
// 256-row blocks of one expert, handed to the clusters
// round robin; a cluster runs, per unit, the phase-1 items hidden = ReLU(x W_in[e])
// (one per 256-column block j of h, hidden stored as bf16), then the phase-2 items
// y = hidden W_out[e] (one per 256-column block of d, fp16).  A CTA's phase-2 A
// operand is its own 128 hidden rows, written by its own epilogue: the k-blocks of
// hidden block j wait only on hready[j], an mbarrier of the same CTA that the four
// epilogue warps arrive on after storing block j, so phase 2 starts on the first
// blocks while the last phase-1 item drains, and a unit's 512 KB of hidden rows is
// read back from L2 a few microseconds after it was written.
//
// The same file holds the backward's SM-pair kernels: this kernel's DGRAD instance
// (the expert data gradients) and ffn_wgrad_tc_kernel (the weight gradients), and the
// swap-AB variant with tiles sized to the rows.
//
// Roles in each CTA: warp 0 issues TMA loads (completion counted on the leader's
// full barrier), warp 1 of the leader issues the MMAs and commits (multicast to both
// CTAs), warps 2-5 drain the double-buffered TMEM accumulator, convert, and write
// 32-row x 64-column tiles through swizzled shared memory with TMA stores (whole
// 128-byte rows instead of 16-byte pieces of 32 rows).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include "common.cuh"
#include "launch.h"
#include "tc.cuh"

namespace moe {
namespace {

constexpr int BM = 128;                    // rows per CTA (TMEM lanes)
constexpr int PAIR_ROWS = 2 * BM;          // rows per pair tile (one work unit)
constexpr int BN = 256;                    // columns per tile; each CTA holds BN/2 of B
constexpr int BK = 64;                     // K per stage: one 128-byte swizzle row of bf16
constexpr int STAGES = 6;
constexpr int THREADS = 192;
constexpr int A_BYTES = BM * BK * 2;       // 16 KB
constexpr int B_BYTES = BK * (BN / 2) * 2; // 16 KB
constexpr int SB = A_BYTES + B_BYTES;
constexpr uint32_t TMEM_COLS = 2 * BN;
constexpr uint32_t IDESC = tc::idesc_bf16_f32(PAIR_ROWS, BN, false, true);
constexpr uint32_t IDESC_KB = tc::idesc_bf16_f32(PAIR_ROWS, BN, false, false);   // B K-major
constexpr int MAX_NT1 = 16;                // h <= 4096
constexpr int kZeroRow = 1 << 30;          // a row coordinate past every tensor: zero fill

struct Barriers {
    uint64_t full[STAGES];     // leader: both CTAs' loads of a stage (leader's arrival + bytes)
    uint64_t empty[STAGES];    // each CTA: the stage has been consumed (leader's commit)
    uint64_t tfull[2];         // each CTA: accumulator ready (leader's commit)
    uint64_t tempty[2];        // leader: accumulator drained by both CTAs' epilogues
    uint64_t hready[MAX_NT1];  // each CTA: its hidden block j of the current unit is stored
    uint64_t done;
    uint32_t tmem_base;
    int abort_flag;
};
// Epilogue staging: per epilogue warp two 32-row x 64-column 2-byte tiles (4 KB each,
// 128-byte swizzle) that TMA stores write out as whole 128-byte rows.
constexpr int ST_ROWS = 32, ST_COLS = 64;
constexpr int ST_BYTES = ST_ROWS * ST_COLS * 2;
constexpr int STAGING = 4 * 2 * ST_BYTES;
constexpr size_t SMEM_BYTES = 1024 + (size_t)STAGES * SB + STAGING + sizeof(Barriers);
static_assert(SMEM_BYTES <= 232448, "shared memory of one CTA");

struct Unit {
    int e, row0, row_end;      // expert, first row of the 256-row block, end of e's rows
};

// Work unit u from the table the row-block prefix kernel wrote (one 16-byte load; each
// role loads the next unit's entry while it works on the current one).
__device__ __forceinline__ Unit load_unit(const int4* __restrict__ units, int u) {
    const int4 v = __ldg(units + u);
    Unit r;
    r.e = v.x;
    r.row0 = v.y;
    r.row_end = v.z;
    return r;
}

// Bounded wait that ignores the abort flag (draining work already in flight).
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, int* err) {
    const long long t0 = clock64();
    while (!tc::mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > tc::kWaitCycles) { raise_error(err, DEV_TIMEOUT); return; }
    }
}

__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// DGRAD: the same two products for the expert data gradients of the backward pass,
// dU = (dE W_out[e]^T) [hidden > 0] (phase 1, N = h, K = d, bf16 into `hidden`) and
// dX = dU W_in[e]^T (phase 2, N = d, K = h, fp16 into `out`): B is read K-contiguous
// from W_out [n][h][d] and W_in [n][d][h] (one 128-row x 64-column box a CTA a stage,
// the K-major layout A uses), and phase 1's epilogue multiplies by [mask > 0] (the
// forward's hidden layer at the same rows) instead of applying ReLU.
template <bool DGRAD>
__global__ void __launch_bounds__(THREADS, 1)
ffn_pair_tc_kernel(const __grid_constant__ CUtensorMap tmA1, const __grid_constant__ CUtensorMap tmB1,
                   const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmB2,
                   const __grid_constant__ CUtensorMap tmH, const __grid_constant__ CUtensorMap tmY,
                   uint16_t* __restrict__ hidden, uint16_t* __restrict__ out, int d, int h,
                   const int4* __restrict__ units, const int32_t* __restrict__ blk, int n,
                   int* err, const uint16_t* __restrict__ mask) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* staging = smem + STAGES * SB;               // 1024-byte aligned
    Barriers* bar = reinterpret_cast<Barriers*>(staging + STAGING);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = tc::cluster_ctarank();
    const int cluster = blockIdx.x >> 1, clusters = gridDim.x >> 1;
    const int NT1 = h / BN, NT2 = d / BN;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) { tc::mbar_init(&bar->full[s], 1); tc::mbar_init(&bar->empty[s], 1); }
        for (int a = 0; a < 2; ++a) {
            tc::mbar_init(&bar->tfull[a], 1);
            tc::mbar_init(&bar->tempty[a], 8);
        }
        for (int j = 0; j < MAX_NT1; ++j) tc::mbar_init(&bar->hready[j], 4);
        tc::mbar_init(&bar->done, 1);
        bar->abort_flag = 0;
        tc::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tc::tma_prefetch(&tmA1); tc::tma_prefetch(&tmB1);
        tc::tma_prefetch(&tmA2); tc::tma_prefetch(&tmB2);
    }
    if (warp == 1) tc::tmem_alloc_pair(&bar->tmem_base, TMEM_COLS);
    griddep_wait();                           // routing written by the previous kernels is visible
    griddep_launch_dependents();
    tc::fence_before_sync();
    __syncthreads();
    tc::cluster_sync();                       // both CTAs' barriers exist before any remote use
    tc::fence_after_sync();
    const int Q = blk[n];                                   // 256-row units
    const int M = cluster < Q ? (Q - cluster + clusters - 1) / clusters : 0;
    const uint32_t tmem = bar->tmem_base;
    volatile int* abort_flag = &bar->abort_flag;

    if (warp == 0) {
        if (lane == 0) {   // ---------------- TMA producer (both CTAs)
            int stage = 0;
            uint32_t phase = 0, armed = 0, armed_parity = 0;
            bool ok = true;
            Unit nxt = M > 0 ? load_unit(units, cluster) : Unit{};
            for (int m = 0; m < M && ok && !*abort_flag; ++m) {
                const Unit un = nxt;
                if (m + 1 < M) nxt = load_unit(units, cluster + (m + 1) * clusters);
                const bool upper_live = un.row0 + BM < un.row_end;   // the peer holds live rows
                for (int ph = 1; ph <= 2 && ok; ++ph) {
                    const CUtensorMap* ta = ph == 1 ? &tmA1 : &tmA2;
                    const CUtensorMap* tb = ph == 1 ? &tmB1 : &tmB2;
                    const int KB = (ph == 1 ? d : h) / BK, NT = ph == 1 ? NT1 : NT2;
                    for (int j = 0; j < NT && ok; ++j) {
                        for (int kb = 0; kb < KB; ++kb) {
                            if (ph == 2 && kb % (BN / BK) == 0) {
                                // this CTA's hidden block kb / 4 of unit m, stored by its
                                // own epilogue (one phase of hready per unit)
                                if (!tc::mbar_wait(&bar->hready[kb / (BN / BK)], m & 1, abort_flag,
                                                   err)) {
                                    ok = false;
                                    break;
                                }
                                fence_proxy_async_global();
                            }
                            if (!tc::mbar_wait(&bar->empty[stage], phase ^ 1, abort_flag, err)) {
                                ok = false;
                                break;
                            }
                            const uint32_t full_c = tc::mapa(tc::smem_u32(&bar->full[stage]), 0);
                            uint8_t* a_dst = smem + stage * SB;
                            uint8_t* b_dst = a_dst + A_BYTES;
                            // the leader expects both CTAs' bytes; the peer's copies only
                            // complete on the leader's barrier (the peer fills stage s again
                            // only after the MMA has consumed it, so it cannot run a phase ahead)
                            // a unit whose rows all fall in the leader's half leaves the
                            // peer's A rows unread: its accumulator rows are never stored
                            // (the peer of such a unit copies a tile from past the end of
                            // the rows instead: the TMA fills it with zeros, which the MMA
                            // multiplies at less power than stale rows)
                            if (rank == 0) tc::mbar_arrive_expect_tx(&bar->full[stage], 2 * SB);
                            tc::tma_load_2d_pair(a_dst, ta, full_c, kb * BK,
                                                 upper_live || rank == 0
                                                     ? un.row0 + (int)rank * BM
                                                     : kZeroRow);
                            if (DGRAD) {        // [128 N rows][64 K], K-contiguous
                                tc::tma_load_3d_pair(b_dst, tb, full_c, kb * BK,
                                                     j * BN + (int)rank * (BN / 2), un.e);
                            } else {
#pragma unroll
                                for (int c = 0; c < BN / 128; ++c)
                                    tc::tma_load_3d_pair(b_dst + c * (BK * 128), tb, full_c,
                                                         j * BN + (int)rank * (BN / 2) + 64 * c,
                                                         kb * BK, un.e);
                            }
                            armed |= 1u << stage;
                            armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                            if (++stage == STAGES) { stage = 0; phase ^= 1; }
                        }
                    }
                }
            }
            // every armed stage consumed by the pair MMA before the CTA can exit
            for (int s = 0; s < STAGES; ++s)
                if ((armed >> s) & 1u) drain_wait(&bar->empty[s], (armed_parity >> s) & 1u, err);
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {   // ---------------- MMA issuer (leader only)
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int m = 0; m < M && ok && !*abort_flag; ++m) {
                for (int ph = 1; ph <= 2 && ok; ++ph) {
                    const int KB = (ph == 1 ? d : h) / BK, NT = ph == 1 ? NT1 : NT2;
                    for (int j = 0; j < NT && ok; ++j) {
                        if (!tc::mbar_wait(&bar->tempty[acc], acc_phase ^ 1, abort_flag, err)) {
                            ok = false;
                            break;
                        }
                        tc::fence_after_sync();
                        const uint32_t d_tmem = tmem + acc * BN;
                        for (int kb = 0; kb < KB; ++kb) {
                            if (!tc::mbar_wait(&bar->full[stage], phase, abort_flag, err)) {
                                ok = false;
                                break;
                            }
                            tc::fence_after_sync();
                            const uint32_t a_addr = tc::smem_u32(smem + stage * SB);
                            const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
                            for (int kk = 0; kk < BK / 16; ++kk) {
                                // A: K-major rows of 128 B, 8-row atoms 1024 B apart.
                                const uint64_t ad = tc::sdesc_sw128(a_addr + kk * 32, 16, 1024);
                                // B: N-major, this CTA's 128 columns as two 64-column
                                // blocks BK*128 B apart (LBO), 8-row atoms 1024 B apart.
                                // DGRAD: B K-major like A.
                                const uint64_t bd =
                                    DGRAD ? tc::sdesc_sw128(b_addr + kk * 32, 16, 1024)
                                          : tc::sdesc_sw128(b_addr + kk * 2048, BK * 128, 1024);
                                tc::mma_bf16_pair(d_tmem, ad, bd, DGRAD ? IDESC_KB : IDESC,
                                                  (kb | kk) != 0 ? 1u : 0u);
                            }
                            tc::mma_commit_pair(&bar->empty[stage], 0x3);
                            if (++stage == STAGES) { stage = 0; phase ^= 1; }
                        }
                        if (!ok) break;
                        tc::mma_commit_pair(&bar->tfull[acc], 0x3);
                        if (++acc == 2) { acc = 0; acc_phase ^= 1; }
                    }
                }
            }
            tc::mma_commit_pair(&bar->done, 0x1);   // every MMA done before TMEM is freed
            drain_wait(&bar->done, 0, err);
        }
    } else {               // ---------------- epilogue: warps 2..5 (both CTAs)
        const int quarter = warp & 3;            // TMEM lanes 32*quarter .. +31
        const uint32_t tempty_c[2] = {tc::mapa(tc::smem_u32(&bar->tempty[0]), 0),
                                      tc::mapa(tc::smem_u32(&bar->tempty[1]), 0)};
        int acc = 0;
        uint32_t acc_phase = 0;
        bool ok = true;
        const int ew = warp - 2;
        uint8_t* sbuf[2] = {staging + (2 * ew) * ST_BYTES, staging + (2 * ew + 1) * ST_BYTES};
        int nbuf = 0;
        Unit nxt = M > 0 ? load_unit(units, cluster) : Unit{};
        for (int m = 0; m < M && ok; ++m) {
            const Unit un = nxt;
            if (m + 1 < M) nxt = load_unit(units, cluster + (m + 1) * clusters);
            const int row_base = un.row0 + (int)rank * BM + quarter * 32;
            const int row = row_base + lane;
            const bool live = row < un.row_end;
            // a warp whose 32 rows all belong to the expert stores whole tiles by TMA;
            // a warp at the end of the expert stores its live rows one by one
            const bool whole = row_base + 32 <= un.row_end;
            for (int ph = 1; ph <= 2 && ok; ++ph) {
                const int NT = ph == 1 ? NT1 : NT2;
                const int N = ph == 1 ? h : d;
                uint16_t* base = ph == 1 ? hidden : out;
                const CUtensorMap* tms = ph == 1 ? &tmH : &tmY;
                for (int j = 0; j < NT; ++j) {
                    // lane 0 waits and the warp follows its verdict, so the warp-collective
                    // TMEM loads below are executed by all 32 lanes or by none
                    int w = 0;
                    if (lane == 0)
                        w = tc::mbar_wait(&bar->tfull[acc], acc_phase, abort_flag, err) ? 1 : 0;
                    w = __shfl_sync(0xffffffffu, w, 0);
                    if (!w) { ok = false; break; }
                    tc::fence_after_sync();
                    uint16_t* dst = base + (size_t)(live ? row : 0) * N + j * BN;
                    const uint32_t t_addr = tmem + acc * BN + ((uint32_t)(quarter * 32) << 16);
#pragma unroll 1
                    for (int col = 0; col < BN; col += 64) {
                        uint4 pk[8];
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            uint32_t r[32];
                            tc::tmem_ld32(t_addr + col + 32 * hh, r);
                            uint32_t mk[16];     // DGRAD phase 1: the forward's hidden values
                            if (DGRAD && ph == 1) {
                                const uint4* mp = reinterpret_cast<const uint4*>(
                                    mask + (size_t)(live ? row : 0) * h + j * BN + col + 32 * hh);
#pragma unroll
                                for (int q = 0; q < 4; ++q) {
                                    const uint4 m4 = live ? mp[q] : make_uint4(0u, 0u, 0u, 0u);
                                    mk[4 * q] = m4.x; mk[4 * q + 1] = m4.y;
                                    mk[4 * q + 2] = m4.z; mk[4 * q + 3] = m4.w;
                                }
                            }
                            tc::tmem_ld_wait();
                            uint32_t* pw = reinterpret_cast<uint32_t*>(pk + 4 * hh);
#pragma unroll
                            for (int q = 0; q < 16; ++q) {
                                float v0 = __uint_as_float(r[2 * q]);
                                float v1 = __uint_as_float(r[2 * q + 1]);
                                if (DGRAD && ph == 1) {   // ReLU'(u) = [hidden > 0], bf16
                                    const __nv_bfloat162 m2 =
                                        *reinterpret_cast<const __nv_bfloat162*>(&mk[q]);
                                    v0 = __bfloat162float(m2.x) > 0.0f ? v0 : 0.0f;
                                    v1 = __bfloat162float(m2.y) > 0.0f ? v1 : 0.0f;
                                    const __nv_bfloat162 b2 = __floats2bfloat162_rn(v0, v1);
                                    pw[q] = *reinterpret_cast<const uint32_t*>(&b2);
                                } else if (ph == 1) {   // hidden layer: ReLU, bf16 (next operand)
                                    const __nv_bfloat162 b2 =
                                        __floats2bfloat162_rn(fmaxf(v0, 0.0f), fmaxf(v1, 0.0f));
                                    pw[q] = *reinterpret_cast<const uint32_t*>(&b2);
                                } else {         // expert output: fp16
                                    if (live) check_half_range(v0, v1, err);
                                    const __half2 h2 = __floats2half2_rn(v0, v1);
                                    pw[q] = *reinterpret_cast<const uint32_t*>(&h2);
                                }
                            }
                        }
                        if (whole) {
                            // staging buffer free once its previous store has read it
                            if (lane == 0) tc::bulk_wait_read<1>();
                            __syncwarp();
                            uint8_t* sb = sbuf[nbuf];
#pragma unroll
                            for (int q = 0; q < 8; ++q)   // 128-byte swizzle: chunk q ^ (row & 7)
                                *reinterpret_cast<uint4*>(sb + lane * 128 + ((q ^ (lane & 7)) << 4)) =
                                    pk[q];
                            tc::fence_proxy_async_shared();
                            __syncwarp();
                            if (lane == 0) {
                                tc::tma_store_2d(tms, sb, j * BN + col, row_base);
                                tc::bulk_commit();
                            }
                            nbuf ^= 1;
                        } else if (live) {
                            uint4* d4 = reinterpret_cast<uint4*>(dst + col);
#pragma unroll
                            for (int q = 0; q < 8; ++q) d4[q] = pk[q];
                        }
                    }
                    // the accumulator goes back to the MMA (TMEM reads are complete)
                    tc::fence_before_sync();
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive_cluster_relaxed(tempty_c[acc]);
                    if (++acc == 2) { acc = 0; acc_phase ^= 1; }
                    if (ph == 1) {
                        // hidden block j of this warp's rows is written (TMA stores complete,
                        // plain stores released) before the producer's copies read it
                        if (lane == 0) tc::bulk_wait_all();
                        fence_proxy_async_global();
                        __syncwarp();
                        if (lane == 0) tc::mbar_arrive(&bar->hready[j]);
                    }
                }
            }
        }
        if (lane == 0) tc::bulk_wait_all();      // stores complete before the CTA exits
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::cluster_sync();                       // no remote arrive or copy targets an exited CTA
    tc::fence_after_sync();
    if (warp == 1) tc::tmem_dealloc_pair(tmem, TMEM_COLS);
}

// ---- swap-AB variant: a tile's row count follows the expert's rows -----------------
//
// The same per-unit work (one expert, up to 256 of its rows, all six items) with the
// operands exchanged: D^T = W^T x^T.  The pair MMA's M = 256 is the tile's output
// columns (each CTA holds 128 of them, the weight tile read N-contiguous exactly as
// B above) and its N is the unit's row count rounded up to 32 (each CTA holds half of
// the rows, K-contiguous, exactly as A above).  So an expert with 520 rows costs two
// full tiles plus a 32-row tile instead of three 256-row tiles, and an expert with 16
// rows streams its weights once with a 32-wide MMA.  The accumulator holds a column
// per TMEM lane and the rows along TMEM columns; the epilogue transposes 64-row x
// 32-column pieces through shared memory and stores them by TMA.  A unit's hidden block j is
// written half by each CTA, so both CTAs' epilogue warps arrive on hready[m & 1][j]
// of both CTAs (release / acquire at cluster scope) before either producer reads it.
constexpr int SW_ST = 32;                          // columns of a transposed store tile
constexpr int SW_ST_ROWS = 64;                     // rows of a transposed store tile
constexpr int SW_ST_BYTES = SW_ST_ROWS * SW_ST * 2;   // 4 KB
constexpr int SW_STAGING = 4 * 2 * SW_ST_BYTES;
constexpr int SW_SMALL_BOX = 16;                   // rows per copy when a CTA takes < 128 rows

struct SwapBarriers {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t hready[2][MAX_NT1];   // [unit parity][hidden block]: 4 warps x 2 CTAs
    uint64_t done;
    uint32_t tmem_base;
    int abort_flag;
};
constexpr size_t SW_SMEM_BYTES = 1024 + (size_t)STAGES * SB + SW_STAGING + sizeof(SwapBarriers);
static_assert(SW_SMEM_BYTES <= 232448, "shared memory of one CTA");

// Rows of the unit's tile (N of the MMA): the live rows rounded up to 32.
__device__ __forceinline__ int swap_tile_rows(const Unit& un) {
    const int rows = min(PAIR_ROWS, un.row_end - un.row0);
    return max(32, (rows + 31) & ~31);
}

__global__ void __launch_bounds__(THREADS, 1)
ffn_swap_tc_kernel(const __grid_constant__ CUtensorMap tmX1, const __grid_constant__ CUtensorMap tmX1s,
                   const __grid_constant__ CUtensorMap tmW1, const __grid_constant__ CUtensorMap tmX2,
                   const __grid_constant__ CUtensorMap tmX2s, const __grid_constant__ CUtensorMap tmW2,
                   const __grid_constant__ CUtensorMap tmH, const __grid_constant__ CUtensorMap tmY,
                   uint16_t* __restrict__ hidden, uint16_t* __restrict__ out, int d, int h,
                   const int4* __restrict__ units, const int32_t* __restrict__ blk, int n,
                   int* err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* staging = smem + STAGES * SB;
    SwapBarriers* bar = reinterpret_cast<SwapBarriers*>(staging + SW_STAGING);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = tc::cluster_ctarank();
    const int cluster = blockIdx.x >> 1, clusters = gridDim.x >> 1;
    const int NT1 = h / BN, NT2 = d / BN;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) { tc::mbar_init(&bar->full[s], 1); tc::mbar_init(&bar->empty[s], 1); }
        for (int a = 0; a < 2; ++a) {
            tc::mbar_init(&bar->tfull[a], 1);
            tc::mbar_init(&bar->tempty[a], 8);
            for (int j = 0; j < MAX_NT1; ++j) tc::mbar_init(&bar->hready[a][j], 8);
        }
        tc::mbar_init(&bar->done, 1);
        bar->abort_flag = 0;
        tc::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tc::tma_prefetch(&tmX1); tc::tma_prefetch(&tmX1s); tc::tma_prefetch(&tmW1);
        tc::tma_prefetch(&tmX2); tc::tma_prefetch(&tmX2s); tc::tma_prefetch(&tmW2);
    }
    if (warp == 1) tc::tmem_alloc_pair(&bar->tmem_base, TMEM_COLS);
    griddep_wait();
    griddep_launch_dependents();
    tc::fence_before_sync();
    __syncthreads();
    tc::cluster_sync();
    tc::fence_after_sync();
    const int Q = blk[n];
    const int M = cluster < Q ? (Q - cluster + clusters - 1) / clusters : 0;
    const uint32_t tmem = bar->tmem_base;
    volatile int* abort_flag = &bar->abort_flag;

    if (warp == 0) {
        if (lane == 0) {   // ---------------- TMA producer (both CTAs)
            int stage = 0;
            uint32_t phase = 0, armed = 0, armed_parity = 0;
            bool ok = true;
            Unit nxt = M > 0 ? load_unit(units, cluster) : Unit{};
            for (int m = 0; m < M && ok && !*abort_flag; ++m) {
                const Unit un = nxt;
                if (m + 1 < M) nxt = load_unit(units, cluster + (m + 1) * clusters);
                const int NH = swap_tile_rows(un) / 2;           // rows this CTA holds
                const int r_start = un.row0 + (int)rank * NH;
                const uint32_t tx = 2u * (uint32_t)(A_BYTES + NH * BK * 2);
                for (int ph = 1; ph <= 2 && ok; ++ph) {
                    const CUtensorMap* tx_big = ph == 1 ? &tmX1 : &tmX2;
                    const CUtensorMap* tx_small = ph == 1 ? &tmX1s : &tmX2s;
                    const CUtensorMap* tw = ph == 1 ? &tmW1 : &tmW2;
                    const int KB = (ph == 1 ? d : h) / BK, NT = ph == 1 ? NT1 : NT2;
                    for (int j = 0; j < NT && ok; ++j) {
                        for (int kb = 0; kb < KB; ++kb) {
                            if (ph == 2 && kb % (BN / BK) == 0) {
                                // hidden block kb / 4 of unit m, stored half by each CTA
                                if (!tc::mbar_wait_cluster(&bar->hready[m & 1][kb / (BN / BK)],
                                                           (m >> 1) & 1, abort_flag, err)) {
                                    ok = false;
                                    break;
                                }
                                fence_proxy_async_global();
                            }
                            if (!tc::mbar_wait(&bar->empty[stage], phase ^ 1, abort_flag, err)) {
                                ok = false;
                                break;
                            }
                            const uint32_t full_c = tc::mapa(tc::smem_u32(&bar->full[stage]), 0);
                            uint8_t* w_dst = smem + stage * SB;
                            uint8_t* x_dst = w_dst + A_BYTES;
                            if (rank == 0) tc::mbar_arrive_expect_tx(&bar->full[stage], tx);
#pragma unroll
                            for (int c = 0; c < 2; ++c)
                                tc::tma_load_3d_pair(w_dst + c * (BK * 128), tw, full_c,
                                                     j * BN + (int)rank * (BN / 2) + 64 * c, kb * BK,
                                                     un.e);
                            if (NH == BM) {
                                tc::tma_load_2d_pair(x_dst, tx_big, full_c, kb * BK, r_start);
                            } else {
                                for (int i = 0; i < NH / SW_SMALL_BOX; ++i)
                                    tc::tma_load_2d_pair(x_dst + i * (SW_SMALL_BOX * 128), tx_small,
                                                         full_c, kb * BK, r_start + SW_SMALL_BOX * i);
                            }
                            armed |= 1u << stage;
                            armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                            if (++stage == STAGES) { stage = 0; phase ^= 1; }
                        }
                    }
                }
            }
            for (int s = 0; s < STAGES; ++s)
                if ((armed >> s) & 1u) drain_wait(&bar->empty[s], (armed_parity >> s) & 1u, err);
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {   // ---------------- MMA issuer (leader only)
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            Unit nxt = M > 0 ? load_unit(units, cluster) : Unit{};
            for (int m = 0; m < M && ok && !*abort_flag; ++m) {
                const Unit un = nxt;
                if (m + 1 < M) nxt = load_unit(units, cluster + (m + 1) * clusters);
                // A = weights (N-contiguous, "MN-major"), B = rows (K-contiguous)
                const uint32_t idesc = tc::idesc_bf16_f32(PAIR_ROWS, swap_tile_rows(un), true, false);
                for (int ph = 1; ph <= 2 && ok; ++ph) {
                    const int KB = (ph == 1 ? d : h) / BK, NT = ph == 1 ? NT1 : NT2;
                    for (int j = 0; j < NT && ok; ++j) {
                        if (!tc::mbar_wait(&bar->tempty[acc], acc_phase ^ 1, abort_flag, err)) {
                            ok = false;
                            break;
                        }
                        tc::fence_after_sync();
                        const uint32_t d_tmem = tmem + acc * BN;
                        for (int kb = 0; kb < KB; ++kb) {
                            if (!tc::mbar_wait(&bar->full[stage], phase, abort_flag, err)) {
                                ok = false;
                                break;
                            }
                            tc::fence_after_sync();
                            const uint32_t w_addr = tc::smem_u32(smem + stage * SB);
                            const uint32_t x_addr = w_addr + A_BYTES;
#pragma unroll
                            for (int kk = 0; kk < BK / 16; ++kk) {
                                // weights: this CTA's 128 columns as two 64-column blocks
                                // BK*128 B apart (LBO), 8-row atoms 1024 B apart
                                const uint64_t ad =
                                    tc::sdesc_sw128(w_addr + kk * 2048, BK * 128, 1024);
                                // rows: K-major rows of 128 B, 8-row atoms 1024 B apart
                                const uint64_t bd = tc::sdesc_sw128(x_addr + kk * 32, 16, 1024);
                                tc::mma_bf16_pair(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
                            }
                            tc::mma_commit_pair(&bar->empty[stage], 0x3);
                            if (++stage == STAGES) { stage = 0; phase ^= 1; }
                        }
                        if (!ok) break;
                        tc::mma_commit_pair(&bar->tfull[acc], 0x3);
                        if (++acc == 2) { acc = 0; acc_phase ^= 1; }
                    }
                }
            }
            tc::mma_commit_pair(&bar->done, 0x1);
            drain_wait(&bar->done, 0, err);
        }
    } else {               // ---------------- epilogue: warps 2..5 (both CTAs)
        const int quarter = warp & 3;            // TMEM lanes = this warp's 32 output columns
        const uint32_t tempty_c[2] = {tc::mapa(tc::smem_u32(&bar->tempty[0]), 0),
                                      tc::mapa(tc::smem_u32(&bar->tempty[1]), 0)};
        int acc = 0;
        uint32_t acc_phase = 0;
        bool ok = true;
        const int ew = warp - 2;
        uint8_t* sbuf[2] = {staging + (2 * ew) * SW_ST_BYTES, staging + (2 * ew + 1) * SW_ST_BYTES};
        int nbuf = 0;
        Unit nxt = M > 0 ? load_unit(units, cluster) : Unit{};
        for (int m = 0; m < M && ok; ++m) {
            const Unit un = nxt;
            if (m + 1 < M) nxt = load_unit(units, cluster + (m + 1) * clusters);
            const int rows = min(PAIR_ROWS, un.row_end - un.row0);
            for (int ph = 1; ph <= 2 && ok; ++ph) {
                const int NT = ph == 1 ? NT1 : NT2;
                const int N = ph == 1 ? h : d;
                uint16_t* base = ph == 1 ? hidden : out;
                const CUtensorMap* tms = ph == 1 ? &tmH : &tmY;
                for (int j = 0; j < NT; ++j) {
                    int w = 0;
                    if (lane == 0)
                        w = tc::mbar_wait(&bar->tfull[acc], acc_phase, abort_flag, err) ? 1 : 0;
                    w = __shfl_sync(0xffffffffu, w, 0);
                    if (!w) { ok = false; break; }
                    tc::fence_after_sync();
                    const int col0 = j * BN + (int)rank * (BN / 2) + quarter * 32;
                    const uint32_t t_addr = tmem + acc * BN + ((uint32_t)(quarter * 32) << 16);
#pragma unroll 1
                    for (int rc = 0; rc < rows; rc += SW_ST_ROWS) {
                        if (lane == 0) tc::bulk_wait_read<1>();
                        __syncwarp();
                        uint8_t* sb = sbuf[nbuf];
                        const int live = min(SW_ST_ROWS, rows - rc);
#pragma unroll 1
                        for (int hh = 0; hh < SW_ST_ROWS / 32 && 32 * hh < live; ++hh) {
                            uint32_t r[32];
                            // r[i] = column (col0 + lane), row rc + 32 hh + i
                            tc::tmem_ld32(t_addr + rc + 32 * hh, r);
                            tc::tmem_ld_wait();
#pragma unroll
                            for (int i = 0; i < 32; ++i) {
                                const float v = __uint_as_float(r[i]);
                                uint16_t bits;
                                if (ph == 1) {
                                    const __nv_bfloat16 b = __float2bfloat16_rn(fmaxf(v, 0.0f));
                                    bits = *reinterpret_cast<const uint16_t*>(&b);
                                } else {
                                    if (32 * hh + i < live) check_half_range(v, 0.0f, err);
                                    const __half hv = __float2half_rn(v);
                                    bits = *reinterpret_cast<const uint16_t*>(&hv);
                                }
                                *reinterpret_cast<uint16_t*>(sb + (32 * hh + i) * (SW_ST * 2) +
                                                             lane * 2) = bits;
                            }
                        }
                        if (live == SW_ST_ROWS) {
                            tc::fence_proxy_async_shared();
                            __syncwarp();
                            if (lane == 0) {
                                tc::tma_store_2d(tms, sb, col0, un.row0 + rc);
                                tc::bulk_commit();
                            }
                        } else {
                            __syncwarp();
                            // the expert's last rows: lanes 0-15 store two columns of a row
                            for (int i = 0; i < live; ++i)
                                if (lane < 16)
                                    *reinterpret_cast<uint32_t*>(
                                        base + (size_t)(un.row0 + rc + i) * N + col0 + 2 * lane) =
                                        *reinterpret_cast<const uint32_t*>(sb + i * (SW_ST * 2) +
                                                                           lane * 4);
                            __syncwarp();
                        }
                        nbuf ^= 1;
                    }
                    tc::fence_before_sync();
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive_cluster_relaxed(tempty_c[acc]);
                    if (++acc == 2) { acc = 0; acc_phase ^= 1; }
                    if (ph == 1) {
                        // this CTA's half of hidden block j is written before either
                        // producer's copies read the block
                        if (lane == 0) tc::bulk_wait_all();
                        fence_proxy_async_global();
                        __syncwarp();
                        if (lane == 0) {
                            const uint32_t hb = tc::smem_u32(&bar->hready[m & 1][j]);
                            tc::mbar_arrive_cluster(tc::mapa(hb, 0));
                            tc::mbar_arrive_cluster(tc::mapa(hb, 1));
                        }
                    }
                }
            }
        }
        if (lane == 0) tc::bulk_wait_all();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::cluster_sync();
    tc::fence_after_sync();
    if (warp == 1) tc::tmem_dealloc_pair(tmem, TMEM_COLS);
}

// ---- expert weight gradients on SM pairs (the backward pass) ------------------------
//
// dW[e] = A_e^T B_e, A_e and B_e expert e's routed rows of A [R,M] and B [R,N] (bf16):
// dW_out[e] = hidden_e^T dE_e and dW_in[e] = x_perm_e^T dU_e.  The pair MMA computes
// 256 (M) x 256 (N) tiles with K running over the expert's rows in 64-row blocks; A is
// read M-contiguous (each CTA's [64 rows][128 M columns], the layout of the swap
// kernel's weight tile) and B N-contiguous (the layout of the forward's weight tile).
// The expert's last, partial block of B comes from a zero-padded copy (btail, 64 rows
// an expert), so rows past the expert's end add nothing whatever A holds there.  Units
// are (expert, 256-row block of M, 256-column block of N) for every expert, one
// without rows writing zeros; fp32 results go out through swizzled shared memory by
// TMA (32 x 32 tiles of 128-byte rows).
constexpr int WG_ST = 32;                                 // fp32 staging tile 32 x 32
constexpr int WG_ST_BYTES = WG_ST * WG_ST * 4;            // 4 KB
constexpr int WG_STAGING = 4 * 2 * WG_ST_BYTES;
struct WgBarriers {
    uint64_t full[STAGES], empty[STAGES], tfull[2], tempty[2], done;
    uint32_t tmem_base;
    int abort_flag;
};
constexpr size_t WG_SMEM_BYTES = 1024 + (size_t)STAGES * SB + WG_STAGING + sizeof(WgBarriers);
static_assert(WG_SMEM_BYTES <= 232448, "shared memory of one CTA");
constexpr uint32_t IDESC_WG = tc::idesc_bf16_f32(PAIR_ROWS, BN, true, true);

struct WgUnit {
    int e, mb, nb, row0, rows;
};
__device__ __forceinline__ WgUnit wg_unit(int u, int MB, int NB, const int32_t* __restrict__ offsets) {
    WgUnit w;
    w.e = u / (MB * NB);
    const int r = u % (MB * NB);
    w.mb = r / NB;
    w.nb = r % NB;
    w.row0 = offsets[w.e];
    w.rows = offsets[w.e + 1] - w.row0;
    return w;
}

__global__ void __launch_bounds__(THREADS, 1)
ffn_wgrad_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmBt, const __grid_constant__ CUtensorMap tmC,
                    const int32_t* __restrict__ offsets, int M, int N, int n, int* err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* staging = smem + STAGES * SB;
    WgBarriers* bar = reinterpret_cast<WgBarriers*>(staging + WG_STAGING);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = tc::cluster_ctarank();
    const int cluster = blockIdx.x >> 1, clusters = gridDim.x >> 1;
    const int MB = M / PAIR_ROWS, NB = N / BN;
    const int Q = n * MB * NB;
    const int MU = cluster < Q ? (Q - cluster + clusters - 1) / clusters : 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) { tc::mbar_init(&bar->full[s], 1); tc::mbar_init(&bar->empty[s], 1); }
        for (int a = 0; a < 2; ++a) {
            tc::mbar_init(&bar->tfull[a], 1);
            tc::mbar_init(&bar->tempty[a], 8);
        }
        tc::mbar_init(&bar->done, 1);
        bar->abort_flag = 0;
        tc::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tc::tma_prefetch(&tmA); tc::tma_prefetch(&tmB); tc::tma_prefetch(&tmBt);
    }
    if (warp == 1) tc::tmem_alloc_pair(&bar->tmem_base, TMEM_COLS);
    griddep_wait();
    griddep_launch_dependents();
    tc::fence_before_sync();
    __syncthreads();
    tc::cluster_sync();
    tc::fence_after_sync();
    const uint32_t tmem = bar->tmem_base;
    volatile int* abort_flag = &bar->abort_flag;

    if (warp == 0) {
        if (lane == 0) {   // ---------------- TMA producer (both CTAs)
            int stage = 0;
            uint32_t phase = 0, armed = 0, armed_parity = 0;
            bool ok = true;
            for (int m = 0; m < MU && ok && !*abort_flag; ++m) {
                const WgUnit w = wg_unit(cluster + m * clusters, MB, NB, offsets);
                const int KB = (w.rows + BK - 1) / BK;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!tc::mbar_wait(&bar->empty[stage], phase ^ 1, abort_flag, err)) {
                        ok = false;
                        break;
                    }
                    const uint32_t full_c = tc::mapa(tc::smem_u32(&bar->full[stage]), 0);
                    uint8_t* a_dst = smem + stage * SB;
                    uint8_t* b_dst = a_dst + A_BYTES;
                    if (rank == 0) tc::mbar_arrive_expect_tx(&bar->full[stage], 2 * SB);
                    const bool whole = (kb + 1) * BK <= w.rows;
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        tc::tma_load_2d_pair(a_dst + c * (BK * 128), &tmA, full_c,
                                             w.mb * PAIR_ROWS + (int)rank * BM + 64 * c,
                                             w.row0 + kb * BK);
                        if (whole)
                            tc::tma_load_2d_pair(b_dst + c * (BK * 128), &tmB, full_c,
                                                 w.nb * BN + (int)rank * (BN / 2) + 64 * c,
                                                 w.row0 + kb * BK);
                        else        // the expert's last rows, zero-padded to 64
                            tc::tma_load_2d_pair(b_dst + c * (BK * 128), &tmBt, full_c,
                                                 w.nb * BN + (int)rank * (BN / 2) + 64 * c,
                                                 w.e * BK);
                    }
                    armed |= 1u << stage;
                    armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
            }
            for (int s = 0; s < STAGES; ++s)
                if ((armed >> s) & 1u) drain_wait(&bar->empty[s], (armed_parity >> s) & 1u, err);
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {   // ---------------- MMA issuer (leader only)
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int m = 0; m < MU && ok && !*abort_flag; ++m) {
                const WgUnit w = wg_unit(cluster + m * clusters, MB, NB, offsets);
                const int KB = (w.rows + BK - 1) / BK;
                if (!tc::mbar_wait(&bar->tempty[acc], acc_phase ^ 1, abort_flag, err)) break;
                tc::fence_after_sync();
                const uint32_t d_tmem = tmem + acc * BN;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!tc::mbar_wait(&bar->full[stage], phase, abort_flag, err)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after_sync();
                    const uint32_t a_addr = tc::smem_u32(smem + stage * SB);
                    const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        // both operands MN-contiguous: two 64-column blocks BK*128 B apart
                        // (LBO), 8-row atoms 1024 B apart; 16 rows of K per step
                        const uint64_t ad = tc::sdesc_sw128(a_addr + kk * 2048, BK * 128, 1024);
                        const uint64_t bd = tc::sdesc_sw128(b_addr + kk * 2048, BK * 128, 1024);
                        tc::mma_bf16_pair(d_tmem, ad, bd, IDESC_WG, (kb | kk) != 0 ? 1u : 0u);
                    }
                    tc::mma_commit_pair(&bar->empty[stage], 0x3);
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                tc::mma_commit_pair(&bar->tfull[acc], 0x3);
                if (++acc == 2) { acc = 0; acc_phase ^= 1; }
            }
            tc::mma_commit_pair(&bar->done, 0x1);
            drain_wait(&bar->done, 0, err);
        }
    } else {               // ---------------- epilogue: warps 2..5 (both CTAs)
        const int quarter = warp & 3;
        const uint32_t tempty_c[2] = {tc::mapa(tc::smem_u32(&bar->tempty[0]), 0),
                                      tc::mapa(tc::smem_u32(&bar->tempty[1]), 0)};
        int acc = 0;
        uint32_t acc_phase = 0;
        const int ew = warp - 2;
        uint8_t* sbuf[2] = {staging + (2 * ew) * WG_ST_BYTES, staging + (2 * ew + 1) * WG_ST_BYTES};
        int nbuf = 0;
        for (int m = 0; m < MU; ++m) {
            const WgUnit w = wg_unit(cluster + m * clusters, MB, NB, offsets);
            int ok = 0;
            if (lane == 0) ok = tc::mbar_wait(&bar->tfull[acc], acc_phase, abort_flag, err) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc::fence_after_sync();
            const int row_g = w.e * M + w.mb * PAIR_ROWS + (int)rank * BM + quarter * 32;
            const uint32_t t_addr = tmem + acc * BN + ((uint32_t)(quarter * 32) << 16);
#pragma unroll 1
            for (int col = 0; col < BN; col += WG_ST) {
                uint32_t r[32];
                if (w.rows > 0) {
                    tc::tmem_ld32(t_addr + col, r);
                    tc::tmem_ld_wait();
                } else {
#pragma unroll
                    for (int q = 0; q < 32; ++q) r[q] = 0u;     // an expert without rows
                }
                if (lane == 0) tc::bulk_wait_read<1>();
                __syncwarp();
                uint8_t* sb = sbuf[nbuf];
#pragma unroll
                for (int q = 0; q < 8; ++q)   // 128-byte swizzle: chunk q ^ (row & 7)
                    *reinterpret_cast<uint4*>(sb + lane * 128 + ((q ^ (lane & 7)) << 4)) =
                        make_uint4(r[4 * q], r[4 * q + 1], r[4 * q + 2], r[4 * q + 3]);
                tc::fence_proxy_async_shared();
                __syncwarp();
                if (lane == 0) {
                    tc::tma_store_2d(&tmC, sb, w.nb * BN + col, row_g);
                    tc::bulk_commit();
                }
                nbuf ^= 1;
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive_cluster_relaxed(tempty_c[acc]);
            if (++acc == 2) { acc = 0; acc_phase ^= 1; }
        }
        if (lane == 0) tc::bulk_wait_all();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::cluster_sync();
    tc::fence_after_sync();
    if (warp == 1) tc::tmem_dealloc_pair(tmem, TMEM_COLS);
}

// btail[e*64 + i] = B[offsets[e] + 64 (blocks - 1) + i] for the i < rows % 64 of expert
// e's last partial block, 0 for the rest of its 64 rows (one CTA an expert).
__global__ void __launch_bounds__(256)
wgrad_tail_kernel(const uint4* __restrict__ B, const int32_t* __restrict__ offsets, int vecs,
                  uint4* __restrict__ tail) {
    griddep_wait();
    griddep_launch_dependents();
    const int e = blockIdx.x;
    const int row0 = offsets[e], rows = offsets[e + 1] - row0;
    const int rem = rows % BK;
    const int first = row0 + (rows / BK) * BK;        // start of the partial block
    for (int i = threadIdx.x; i < BK * vecs; i += blockDim.x) {
        const int rr = i / vecs, v = i % vecs;
        tail[((size_t)e * BK + rr) * vecs + v] =
            rr < rem ? B[(size_t)(first + rr) * vecs + v] : make_uint4(0u, 0u, 0u, 0u);
    }
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

bool make_rows_map(CUtensorMap* m, const void* base, long long rows, int cols, int box_rows = BM) {
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

// Row-major [rows, cols] 2-byte output, boxes of 64 columns x 32 rows, 128-byte swizzle
// (the epilogue's TMA stores).
bool make_store_map(CUtensorMap* m, void* base, long long rows, int cols, bool fp16) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {ST_COLS, ST_ROWS};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base,
              dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Row-major [rows, cols] fp32 output, boxes of 32 columns x 32 rows (128-byte rows),
// 128-byte swizzle (the weight-gradient epilogue's TMA stores).
bool make_store_map_f32(CUtensorMap* m, void* base, long long rows, int cols) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 4};
    cuuint32_t box[2] = {WG_ST, WG_ST};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Row-major [rows, cols] 2-byte output, boxes of 32 columns x 64 rows, no swizzle (the
// swap-AB epilogue's transposed tiles, 64-byte rows in shared memory).
bool make_store_map_plain(CUtensorMap* m, void* base, long long rows, int cols, bool fp16) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {SW_ST, SW_ST_ROWS};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base,
              dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

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

// Weights [n][N rows][K cols] (K contiguous, read as B^T): boxes of 64 K-columns x 128
// N-rows, 128-byte swizzle (the K-major B of the backward's data gradients).
bool make_weight_map_kmajor(CUtensorMap* m, const void* base, int n, int N, int K) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)N, (cuuint64_t)n};
    cuuint64_t strides[2] = {(cuuint64_t)K * 2, (cuuint64_t)N * K * 2};
    cuuint32_t box[3] = {64, BN / 2, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Clusters of two that can be resident at once (one CTA per SM), cached per device.
template <typename Kernel>
int pair_grid(Kernel kernel, size_t smem_bytes, int* cached, cudaError_t* e) {
    int dev = 0;
    *e = cudaGetDevice(&dev);
    if (*e != cudaSuccess) return 0;
    if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(sms > 0 ? sms & ~1 : 2);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = smem_bytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    *e = cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg);
    if (*e != cudaSuccess || clusters < 1) {
        if (*e == cudaSuccess) *e = cudaErrorInvalidConfiguration;
        return 0;
    }
    if (dev >= 0 && dev < 64) cached[dev] = 2 * clusters;
    return 2 * clusters;
}

}  // namespace

bool ffn_pair_supported(int d, int h) { return d % BN == 0 && h % BN == 0 && h / BN <= MAX_NT1; }

int ffn_pair_block() { return PAIR_ROWS; }

cudaError_t launch_ffn_pair(const void* x_perm, const int32_t* offsets, const void* W_in,
                            const void* W_out, void* y_perm, void* hidden, int32_t* blk,
                            void* units, long long R, int d, int h, int n, int* err,
                            cudaStream_t s, bool prefix_done) {
    if (R == 0) return cudaSuccess;
    if (!ffn_pair_supported(d, h)) return cudaErrorInvalidValue;
    CUtensorMap a1, b1, a2, b2, sh, sy;
    if (!make_rows_map(&a1, x_perm, R, d) || !make_weight_map(&b1, W_in, n, d, h) ||
        !make_rows_map(&a2, hidden, R, h) || !make_weight_map(&b2, W_out, n, h, d) ||
        !make_store_map(&sh, hidden, R, h, false) || !make_store_map(&sy, y_perm, R, d, true))
        return cudaErrorInvalidValue;
    static bool configured = false;
    cudaError_t e;
    if (!configured) {
        e = cudaFuncSetAttribute(ffn_pair_tc_kernel<false>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    static int cached[64] = {};
    const int grid = pair_grid(ffn_pair_tc_kernel<false>, SMEM_BYTES, cached, &e);
    if (grid == 0) return e;
    if (!prefix_done) {
        e = launch_row_block_prefix(offsets, n, PAIR_ROWS, blk, s, units);
        if (e != cudaSuccess) return e;
    }
    e = launch_pdl(ffn_pair_tc_kernel<false>, dim3(grid), dim3(THREADS), SMEM_BYTES, s, 2, a1, b1,
                   a2, b2, sh, sy, static_cast<uint16_t*>(hidden), static_cast<uint16_t*>(y_perm),
                   d, h, static_cast<const int4*>(units), static_cast<const int32_t*>(blk), n, err,
                   static_cast<const uint16_t*>(nullptr));
    note_launch();
    return e;
}

cudaError_t launch_ffn_pair_dgrad(const void* dE, const int32_t* offsets, const void* W_in,
                                  const void* W_out, const void* hidden_fwd, void* dU, void* dX,
                                  int32_t* blk, void* units, long long R, int d, int h, int n,
                                  int* err, cudaStream_t s) {
    if (R == 0) return cudaSuccess;
    if (!ffn_pair_supported(d, h)) return cudaErrorInvalidValue;
    CUtensorMap a1, b1, a2, b2, sh, sy;
    if (!make_rows_map(&a1, dE, R, d) || !make_weight_map_kmajor(&b1, W_out, n, h, d) ||
        !make_rows_map(&a2, dU, R, h) || !make_weight_map_kmajor(&b2, W_in, n, d, h) ||
        !make_store_map(&sh, dU, R, h, false) || !make_store_map(&sy, dX, R, d, true))
        return cudaErrorInvalidValue;
    static bool configured = false;
    cudaError_t e;
    if (!configured) {
        e = cudaFuncSetAttribute(ffn_pair_tc_kernel<true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    static int cached[64] = {};
    const int grid = pair_grid(ffn_pair_tc_kernel<true>, SMEM_BYTES, cached, &e);
    if (grid == 0) return e;
    e = launch_row_block_prefix(offsets, n, PAIR_ROWS, blk, s, units);
    if (e != cudaSuccess) return e;
    e = launch_pdl(ffn_pair_tc_kernel<true>, dim3(grid), dim3(THREADS), SMEM_BYTES, s, 2, a1, b1,
                   a2, b2, sh, sy, static_cast<uint16_t*>(dU), static_cast<uint16_t*>(dX), d, h,
                   static_cast<const int4*>(units), static_cast<const int32_t*>(blk), n, err,
                   static_cast<const uint16_t*>(hidden_fwd));
    note_launch();
    return e;
}

cudaError_t launch_ffn_swap(const void* x_perm, const int32_t* offsets, const void* W_in,
                            const void* W_out, void* y_perm, void* hidden, int32_t* blk,
                            void* units, long long R, int d, int h, int n, int* err,
                            cudaStream_t s) {
    if (R == 0) return cudaSuccess;
    if (!ffn_pair_supported(d, h)) return cudaErrorInvalidValue;
    CUtensorMap x1, x1s, w1, x2, x2s, w2, sh, sy;
    if (!make_rows_map(&x1, x_perm, R, d) || !make_rows_map(&x1s, x_perm, R, d, SW_SMALL_BOX) ||
        !make_weight_map(&w1, W_in, n, d, h) || !make_rows_map(&x2, hidden, R, h) ||
        !make_rows_map(&x2s, hidden, R, h, SW_SMALL_BOX) || !make_weight_map(&w2, W_out, n, h, d) ||
        !make_store_map_plain(&sh, hidden, R, h, false) ||
        !make_store_map_plain(&sy, y_perm, R, d, true))
        return cudaErrorInvalidValue;
    static bool configured = false;
    cudaError_t e;
    if (!configured) {
        e = cudaFuncSetAttribute(ffn_swap_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)SW_SMEM_BYTES);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    static int cached[64] = {};
    const int grid = pair_grid(ffn_swap_tc_kernel, SW_SMEM_BYTES, cached, &e);
    if (grid == 0) return e;
    e = launch_row_block_prefix(offsets, n, PAIR_ROWS, blk, s, units);
    if (e != cudaSuccess) return e;
    e = launch_pdl(ffn_swap_tc_kernel, dim3(grid), dim3(THREADS), SW_SMEM_BYTES, s, 2, x1, x1s, w1,
                   x2, x2s, w2, sh, sy, static_cast<uint16_t*>(hidden),
                   static_cast<uint16_t*>(y_perm), d, h, static_cast<const int4*>(units),
                   static_cast<const int32_t*>(blk), n, err);
    note_launch();
    return e;
}

size_t wgrad_tail_bytes(int n, int cols) { return (size_t)n * BK * cols * 2; }

cudaError_t launch_ffn_wgrad(const void* A, const void* B, void* btail, const int32_t* offsets,
                             long long R, int M, int N, int n, float* dW, int* err,
                             cudaStream_t s) {
    if (M % PAIR_ROWS != 0 || N % BN != 0) return cudaErrorInvalidValue;
    cudaError_t e = launch_pdl(wgrad_tail_kernel, dim3(n), dim3(256), 0, s, 1,
                               static_cast<const uint4*>(B), offsets, N / 8,
                               static_cast<uint4*>(btail));
    note_launch();
    if (e != cudaSuccess) return e;
    CUtensorMap ta, tb, tt, tcm;
    if (!make_rows_map(&ta, A, R > 0 ? R : 1, M, BK) || !make_rows_map(&tb, B, R > 0 ? R : 1, N, BK) ||
        !make_rows_map(&tt, btail, (long long)n * BK, N, BK) ||
        !make_store_map_f32(&tcm, dW, (long long)n * M, N))
        return cudaErrorInvalidValue;
    static bool configured = false;
    if (!configured) {
        e = cudaFuncSetAttribute(ffn_wgrad_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)WG_SMEM_BYTES);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    static int cached[64] = {};
    const int grid = pair_grid(ffn_wgrad_tc_kernel, WG_SMEM_BYTES, cached, &e);
    if (grid == 0) return e;
    e = launch_pdl(ffn_wgrad_tc_kernel, dim3(grid), dim3(THREADS), WG_SMEM_BYTES, s, 2, ta, tb, tt,
                   tcm, offsets, M, N, n, err);
    note_launch();
    return e;
}

}  // namespace moe
