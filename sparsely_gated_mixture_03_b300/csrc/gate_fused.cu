// The whole noisy top-k gate in one tcgen05 kernel, for n <= 256 experts.
//
// "Mixture of Experts: Outrageously Large Neural Networks" (intuitivepapers.ai):
//   "Noisy top-k gating", eq (4): H = x W_g (+ b_g) + eps * (Softplus(x W_noise) + floor);
//   eqs (3)/(5): keep the k largest H, softmax over them;
//   "A differentiable count of examples", eqs (8)-(10): P(x,i) = Phi((clean_i -
//   kth_excluding(H,k,i)) / std_i), the threshold being the (k+1)-th largest H when i is
//   kept and the k-th largest otherwise; Load_i = sum_x P(x,i).
//   "Why experts collapse, and the balancing losses", eq (6): Importance_i = sum_x G(x)_i.
//
// The logits are the exact three-term bf16 split GEMM of gate_tc.cu (same W3 layout and
// lo, mid, hi accumulation order).  A tile is 128 tokens x every expert: chunk c of 128
// experts accumulates in TMEM columns 256c .. 256c+255 (clean, then noise), so a token's
// whole logit row stays on the SM.  Eight epilogue warps, two per TMEM lane quarter,
// each own one token row and half of the experts:
//   pass 1: H, 1/std (written back over the noise columns), running top-(k+1);
//   merge:  the two halves' lists through shared memory (larger H first, equal H ->
//           lower index), softmax over the k kept, the near-tie flag;
//   pass 2: P and the kept gate for every (row, expert), summed over each warp's 32 rows
//           by a fixed warp reduce-scatter, then over the 4 quarters in a fixed order
//           -> load_part / imp_part [token block][n] (summed over blocks elsewhere).
// One accumulator fills TMEM, so a tile's MMAs wait for the previous epilogue.
//
// Grouped mode (the secondary gates of "Hierarchical MoE"): the rows are the
// group-dispatched routed rows of the primary gate, rows [offsets[g], offsets[g+1]) of
// group g use that group's own split weights W3[g], and a tile never mixes groups
// (tiles are (group, 128-row block), read from a device-side prefix of row blocks).
// Routed row r = perm[p] = t*k1 + s draws its noise from eps row r, and its kept
// experts are written at r as flat ids g*n + j with the product gate
// gate_scale[r] * G_g(x)_j; the tile sums (P and product gates) then belong to group g.
#include <cuda.h>
#include <stdint.h>

#include "common.cuh"
#include "launch.h"
#include "tc.cuh"

namespace moe {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int EPT = 128;                 // experts per TMEM chunk
constexpr int BK = 64;
constexpr int STAGES = 3;
constexpr int EPI_WARPS = 8;
constexpr int THREADS = 64 + 32 * EPI_WARPS;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BK * BN * 2;
constexpr int SB = A_BYTES + B_BYTES;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t IDESC = tc::idesc_bf16_f32(BM, BN, false, true);
constexpr int KMAX1 = 9;

struct Smem {
    float red_p[4][2 * EPT];
    float red_g[4][2 * EPT];
    float mv[2][BM][KMAX1];
    int mi[2][BM][KMAX1];
    int vote[EPI_WARPS];
};
struct Barriers {
    uint64_t full[STAGES], empty[STAGES], tfull, tempty, done;
    uint32_t tmem_base;
    int abort_flag;
};
constexpr size_t SMEM_BYTES = 1024 + (size_t)STAGES * SB + sizeof(Smem) + sizeof(Barriers);

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, int* err) {
    const long long t0 = clock64();
    while (!tc::mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > tc::kWaitCycles) { raise_error(err, DEV_TIMEOUT); return; }
    }
}

// Rows of one tile: [row0, row_end) clipped to the tile by the caller, and the group.
struct TileRows {
    int row0, row_end, g;
};

// Grouped-mode arguments (unused in the flat mode).
struct GroupArgs {
    const int32_t* offsets;      // [groups+1] routed-row ranges of the groups
    const int32_t* blk_prefix;   // [groups+1] prefix of ceil(rows/BM) over the groups
    const int32_t* perm;         // [rows] routed row of each grouped position
    const float* gate_scale;     // [routed rows] primary gate of each routed row
    int groups;
};

template <bool GROUPED>
__device__ __forceinline__ int tile_count(int T, const GroupArgs& ga) {
    return GROUPED ? ga.blk_prefix[ga.groups] : (T + BM - 1) / BM;
}

template <bool GROUPED>
__device__ __forceinline__ TileRows tile_rows(int tile, int T, const GroupArgs& ga) {
    TileRows r;
    if (!GROUPED) {
        r.row0 = tile * BM;
        r.row_end = T;
        r.g = 0;
        return r;
    }
    int lo = 0, hi = ga.groups - 1;          // last group whose first block is <= tile
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (ga.blk_prefix[mid] <= tile) lo = mid; else hi = mid - 1;
    }
    r.g = lo;
    r.row0 = ga.offsets[lo] + (tile - ga.blk_prefix[lo]) * BM;
    r.row_end = ga.offsets[lo + 1];
    return r;
}

template <int K1, bool GROUPED>
__global__ void __launch_bounds__(THREADS, 1)
gate_fused_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                  const float* __restrict__ eps, const float* __restrict__ b_g, int T, int d, int n,
                  int n_pad, float std_floor, int32_t* __restrict__ idx_out,
                  float* __restrict__ gates_out, uint8_t* __restrict__ tie_out,
                  float* __restrict__ load_part, float* __restrict__ imp_part, int* err,
                  const GroupArgs ga) {
    constexpr int K = K1 - 1;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    Smem* fs = reinterpret_cast<Smem*>(smem + STAGES * SB);
    Barriers* bar = reinterpret_cast<Barriers*>(smem + STAGES * SB + sizeof(Smem));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int CPT = n_pad / EPT;
    const int total = tile_count<GROUPED>(T, ga);
    const int KBX = d / BK;
    const int KB = 3 * KBX;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) { tc::mbar_init(&bar->full[s], 1); tc::mbar_init(&bar->empty[s], 1); }
        tc::mbar_init(&bar->tfull, 1);
        tc::mbar_init(&bar->tempty, EPI_WARPS);
        tc::mbar_init(&bar->done, 1);
        bar->abort_flag = 0;
        tc::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) { tc::tma_prefetch(&tmX); tc::tma_prefetch(&tmW); }
    if (warp == 1) tc::tmem_alloc(&bar->tmem_base, TMEM_COLS);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = bar->tmem_base;
    volatile int* abort_flag = &bar->abort_flag;

    if (warp == 0) {
        if (lane == 0) {   // TMA producer: chunk-major, terms lo, mid, hi (see gate_tc.cu)
            int stage = 0;
            uint32_t phase = 0, armed = 0, armed_parity = 0;
            for (int tile = blockIdx.x; tile < total && !*abort_flag; tile += gridDim.x) {
                const TileRows tr = tile_rows<GROUPED>(tile, T, ga);
                const int w_row0 = tr.g * 3 * d;         // group g's split weights
                for (int cc = 0; cc < CPT; ++cc) {
                    for (int kb = 0; kb < KB; ++kb) {
                        if (!tc::mbar_wait(&bar->empty[stage], phase ^ 1, abort_flag, err)) break;
                        uint8_t* a_dst = smem + stage * SB;
                        uint8_t* b_dst = a_dst + A_BYTES;
                        const int term = 2 - kb / KBX;
                        tc::mbar_arrive_expect_tx(&bar->full[stage], SB);
                        tc::tma_load_2d(a_dst, &tmX, &bar->full[stage], (kb % KBX) * BK, tr.row0);
#pragma unroll
                        for (int i = 0; i < BN / 64; ++i)
                            tc::tma_load_2d(b_dst + i * (BK * 128), &tmW, &bar->full[stage],
                                            cc * BN + 64 * i, w_row0 + term * d + (kb % KBX) * BK);
                        armed |= 1u << stage;
                        armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                        if (++stage == STAGES) { stage = 0; phase ^= 1; }
                    }
                }
            }
            for (int s = 0; s < STAGES; ++s)
                if ((armed >> s) & 1u) drain_wait(&bar->full[s], (armed_parity >> s) & 1u, err);
        }
    } else if (warp == 1) {
        if (lane == 0) {   // MMA issuer
            int stage = 0;
            uint32_t phase = 0, acc_phase = 0;
            for (int tile = blockIdx.x; tile < total && !*abort_flag; tile += gridDim.x) {
                if (!tc::mbar_wait(&bar->tempty, acc_phase ^ 1, abort_flag, err)) break;
                tc::fence_after_sync();
                bool ok = true;
                for (int cc = 0; cc < CPT && ok; ++cc) {
                    for (int kb = 0; kb < KB; ++kb) {
                        if (!tc::mbar_wait(&bar->full[stage], phase, abort_flag, err)) { ok = false; break; }
                        tc::fence_after_sync();
                        const uint32_t a_addr = tc::smem_u32(smem + stage * SB);
                        const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk) {
                            const uint64_t ad = tc::sdesc_sw128(a_addr + kk * 32, 16, 1024);
                            const uint64_t bd = tc::sdesc_sw128(b_addr + kk * 2048, BK * 128, 1024);
                            tc::mma_bf16(tmem + cc * BN, ad, bd, IDESC, (kb | kk) != 0 ? 1u : 0u);
                        }
                        tc::mma_commit(&bar->empty[stage]);
                        if (++stage == STAGES) { stage = 0; phase ^= 1; }
                    }
                }
                if (!ok) break;
                tc::mma_commit(&bar->tfull);
                acc_phase ^= 1;
            }
            tc::mma_commit(&bar->done);
            drain_wait(&bar->done, 0, err);
        }
    } else {               // epilogue: warps 2..9
        const int ew = warp - 2;
        const int quarter = warp & 3;            // TMEM lanes 32*quarter .. +31
        const int half = ew >> 2;                // which half of the experts
        const int row = quarter * 32 + lane;     // token row inside the tile
        const int etid = threadIdx.x - 64;       // 0..255
        const int ne = n_pad / 2;                // experts per half: 64 or 128
        const int e_begin = half * ne;
        const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
        const bool vec = (n % 4) == 0;
        uint32_t acc_phase = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
            // all eight warps vote, so none reaches a named barrier alone
            if (lane == 0)
                fs->vote[ew] = tc::mbar_wait(&bar->tfull, acc_phase, abort_flag, err) ? 1 : 0;
            epi_bar();
            int ok = 1;
#pragma unroll
            for (int w = 0; w < EPI_WARPS; ++w) ok &= fs->vote[w];
            if (!ok) break;
            tc::fence_after_sync();
            acc_phase ^= 1;
            const TileRows tr = tile_rows<GROUPED>(tile, T, ga);
            const int p = tr.row0 + row;
            const bool live = p < tr.row_end;
            // t: the row whose noise is read and whose outputs are written (the token
            // in the flat mode, the routed row in the grouped mode)
            const int t = !live ? 0 : (GROUPED ? ga.perm[p] : p);

            // ---- pass 1: H, 1/std back into TMEM, running top-(k+1) of this half
            float v[K1];
            int ix[K1];
#pragma unroll
            for (int q = 0; q < K1; ++q) { v[q] = -INFINITY; ix[q] = 0x7fffffff; }
#pragma unroll 1
            for (int c = 0; c < ne; c += 32) {
                const int e0 = e_begin + c;
                const uint32_t col = (uint32_t)((e0 / EPT) * BN + (e0 % EPT));
                uint32_t rc[32], rr[32];
                tc::tmem_ld32(t_lane + col, rc);
                tc::tmem_ld32(t_lane + col + EPT, rr);
                tc::tmem_ld_wait();
                float ep[32];
                const float* erow = eps + (size_t)(live ? t : 0) * n + e0;
                if (live && vec && e0 + 32 <= n) {
#pragma unroll
                    for (int q = 0; q < 32; q += 4) {
                        const float4 f = *reinterpret_cast<const float4*>(erow + q);
                        ep[q] = f.x; ep[q + 1] = f.y; ep[q + 2] = f.z; ep[q + 3] = f.w;
                    }
                } else {
#pragma unroll
                    for (int q = 0; q < 32; ++q) ep[q] = (live && e0 + q < n) ? erow[q] : 0.0f;
                }
#pragma unroll
                for (int q = 0; q < 32; ++q) {
                    const int e = e0 + q;
                    const float cl =
                        __uint_as_float(rc[q]) + ((b_g != nullptr && e < n) ? b_g[e] : 0.0f);
                    const float sd = softplus_f32(__uint_as_float(rr[q])) + std_floor;
                    rr[q] = __float_as_uint(1.0f / sd);
                    const float hv = fmaf(ep[q], sd, cl);
                    if (live && e < n && hv > v[K1 - 1]) {
#pragma unroll
                        for (int u = K1 - 1; u > 0; --u) {
                            if (hv > v[u - 1]) { v[u] = v[u - 1]; ix[u] = ix[u - 1]; }
                            else if (hv > v[u]) { v[u] = hv; ix[u] = e; }
                        }
                        if (hv > v[0]) { v[0] = hv; ix[0] = e; }
                    }
                }
                tc::tmem_st32(t_lane + col + EPT, rr);
            }
            tc::tmem_st_wait();

            // ---- merge the two halves' lists (both threads of a row get the same result)
#pragma unroll
            for (int q = 0; q < K1; ++q) { fs->mv[half][row][q] = v[q]; fs->mi[half][row][q] = ix[q]; }
            epi_bar();
            {
                int ia = 0, ib = 0;
#pragma unroll
                for (int q = 0; q < K1; ++q) {
                    const float va = fs->mv[0][row][ia], vb = fs->mv[1][row][ib];
                    const int xa = fs->mi[0][row][ia], xb = fs->mi[1][row][ib];
                    const bool take_a = va > vb || (va == vb && xa < xb);
                    v[q] = take_a ? va : vb;
                    ix[q] = take_a ? xa : xb;
                    ia += take_a ? 1 : 0;
                    ib += take_a ? 0 : 1;
                }
            }
            float gk[K];
            {
                float s = 0.0f;
#pragma unroll
                for (int j = 0; j < K; ++j) { gk[j] = expf(v[j] - v[0]); s += gk[j]; }
                const float inv = 1.0f / s;
#pragma unroll
                for (int j = 0; j < K; ++j) gk[j] *= inv;
                if (GROUPED) {             // the product with the primary gate
                    const float sc = live ? ga.gate_scale[t] : 0.0f;
#pragma unroll
                    for (int j = 0; j < K; ++j) gk[j] *= sc;
                }
            }
            if (live && half == 0) {
                const int id0 = tr.g * n;  // flat id of the group's first expert
#pragma unroll
                for (int j = 0; j < K; ++j) {
                    idx_out[(size_t)t * K + j] = id0 + ix[j];
                    gates_out[(size_t)t * K + j] = gk[j];
                }
                // k = n: v[K] is the -inf sentinel, the gap is +inf, no tie
                if (tie_out != nullptr) tie_out[t] = (v[K - 1] - v[K]) < 1e-5f ? 1 : 0;
            }
            const float thr_in = v[K], thr_out = v[K - 1];

            // ---- pass 2: P and the kept gates, summed over rows
#pragma unroll 1
            for (int c = 0; c < ne; c += 32) {
                const int e0 = e_begin + c;
                const uint32_t col = (uint32_t)((e0 / EPT) * BN + (e0 % EPT));
                uint32_t rc[32], rr[32];
                tc::tmem_ld32(t_lane + col, rc);
                tc::tmem_ld32(t_lane + col + EPT, rr);     // 1/std from pass 1
                tc::tmem_ld_wait();
                if (c + 32 >= ne) {        // this warp's last TMEM read of the tile
                    tc::fence_before_sync();
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(&bar->tempty);
                }
                uint32_t kmask = 0;
#pragma unroll
                for (int j = 0; j < K; ++j) {
                    const unsigned off = (unsigned)(ix[j] - e0);
                    if (off < 32u) kmask |= 1u << off;
                }
                float p[32], g[32];
#pragma unroll
                for (int q = 0; q < 32; ++q) {
                    const int e = e0 + q;
                    const bool kept = (kmask >> q) & 1u;
                    float pv = 0.0f, gv = 0.0f;
                    if (live && e < n) {
                        const float cl =
                            __uint_as_float(rc[q]) + (b_g != nullptr ? b_g[e] : 0.0f);
                        pv = normcdff((cl - (kept ? thr_in : thr_out)) * __uint_as_float(rr[q]));
                    }
                    if (kept) {
#pragma unroll
                        for (int j = 0; j < K; ++j) gv = ix[j] == e ? gk[j] : gv;
                    }
                    p[q] = pv;
                    g[q] = gv;
                }
                const float sp = tc::reduce_scatter32(p, lane);
                const float sg = tc::reduce_scatter32(g, lane);
                fs->red_p[quarter][e0 + lane] = sp;
                fs->red_g[quarter][e0 + lane] = sg;
            }
            epi_bar();
            if (etid < n) {
                const size_t o = (size_t)tile * n + etid;
                load_part[o] = ((fs->red_p[0][etid] + fs->red_p[1][etid]) + fs->red_p[2][etid]) +
                               fs->red_p[3][etid];
                imp_part[o] = ((fs->red_g[0][etid] + fs->red_g[1][etid]) + fs->red_g[2][etid]) +
                              fs->red_g[3][etid];
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 1) tc::tmem_dealloc(tmem, TMEM_COLS);
}

template <int K1, bool GROUPED>
cudaError_t launch_k(const CUtensorMap& mx, const CUtensorMap& mw, const float* eps,
                     const float* b_g, int T, int d, int n, int n_pad, float std_floor,
                     int32_t* idx, float* gates, uint8_t* tie, float* load_part, float* imp_part,
                     int* err, const GroupArgs& ga, cudaStream_t s) {
    static bool configured = false;
    if (!configured) {
        const cudaError_t e =
            cudaFuncSetAttribute(gate_fused_kernel<K1, GROUPED>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    gate_fused_kernel<K1, GROUPED><<<gate_sm_count(), THREADS, SMEM_BYTES, s>>>(
        mx, mw, eps, b_g, T, d, n, n_pad, std_floor, idx, gates, tie, load_part, imp_part, err,
        ga);
    note_launch();
    return cudaGetLastError();
}

template <bool GROUPED>
cudaError_t launch_by_k(int k, const CUtensorMap& mx, const CUtensorMap& mw, const float* eps,
                        const float* b_g, int T, int d, int n, int n_pad, float std_floor,
                        int32_t* idx, float* gates, uint8_t* tie, float* load_part,
                        float* imp_part, int* err, const GroupArgs& ga, cudaStream_t s) {
    switch (k + 1) {
#define MOE_FUSED_CASE(K1)                                                                  \
    case K1:                                                                                \
        return launch_k<K1, GROUPED>(mx, mw, eps, b_g, T, d, n, n_pad, std_floor, idx,     \
                                     gates, tie, load_part, imp_part, err, ga, s);
        MOE_FUSED_CASE(2) MOE_FUSED_CASE(3) MOE_FUSED_CASE(4) MOE_FUSED_CASE(5)
        MOE_FUSED_CASE(6) MOE_FUSED_CASE(7) MOE_FUSED_CASE(8) MOE_FUSED_CASE(9)
#undef MOE_FUSED_CASE
        default: return cudaErrorInvalidValue;
    }
}

// out[g*n + i] = fp64 sum over the tiles of group g, in tile order, of part[tile*n + i]
// (and likewise imp); a group without rows gets 0.
__global__ void __launch_bounds__(256)
group_tile_reduce_kernel(const float* __restrict__ part, const float* __restrict__ imp_part,
                         const int32_t* __restrict__ blk_prefix, int groups, int n,
                         float* __restrict__ out, float* __restrict__ imp_out) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long long)groups * n) return;
    const int g = (int)(i / n), e = (int)(i % n);
    double s = 0.0, si = 0.0;
    for (int tile = blk_prefix[g]; tile < blk_prefix[g + 1]; ++tile) {
        s += (double)part[(size_t)tile * n + e];
        si += (double)imp_part[(size_t)tile * n + e];
    }
    out[i] = (float)s;
    imp_out[i] = (float)si;
}

}  // namespace

bool gate_tc_fusable(int n) { return gate_tc_n_pad(n) <= 2 * EPT; }

cudaError_t launch_gate_fused_tc(const void* x, const float* W_g, const float* W_noise,
                                 const float* eps, const float* b_g, int T, int d, int n, int k,
                                 float std_floor, void* W3, int32_t* idx, float* gates,
                                 uint8_t* tie, float* load_part, float* imp_part, float* load,
                                 float* importance, int* err, cudaStream_t s) {
    const int n_pad = gate_tc_n_pad(n);
    if (n_pad > 2 * EPT) return cudaErrorInvalidValue;
    cudaError_t e = launch_gate_split_weights(W_g, W_noise, d, n, W3, s);
    if (e != cudaSuccess) return e;
    CUtensorMap mx, mw;
    if (!gate_bf16_map(&mx, x, T, d, BM) || !gate_bf16_map(&mw, W3, 3LL * d, 2LL * n_pad, BK))
        return cudaErrorInvalidValue;
    const GroupArgs none{nullptr, nullptr, nullptr, nullptr, 0};
    e = launch_by_k<false>(k, mx, mw, eps, b_g, T, d, n, n_pad, std_floor, idx, gates, tie,
                           load_part, imp_part, err, none, s);
    if (e != cudaSuccess) return e;
    return launch_partial_reduce(load_part, importance != nullptr ? imp_part : nullptr,
                                 (T + BM - 1) / BM, n, load, importance, s);
}

int gate_grouped_max_tiles(long long rows, int groups) {
    return (int)((rows + BM - 1) / BM) + groups;
}

cudaError_t launch_gate_grouped_tc(const void* x_rows, long long rows, const int32_t* offsets,
                                   const int32_t* blk_prefix, const int32_t* perm, int groups,
                                   const float* W_g, const float* W_noise, const float* eps,
                                   const float* gate_scale, int d, int n, int k, float std_floor,
                                   void* W3, int32_t* idx, float* gates, uint8_t* tie,
                                   float* load_part, float* imp_part, float* load,
                                   float* importance, int* err, cudaStream_t s) {
    const int n_pad = gate_tc_n_pad(n);
    if (n_pad > 2 * EPT || rows <= 0) return cudaErrorInvalidValue;
    cudaError_t e = launch_gate_split_weights_grouped(W_g, W_noise, groups, d, n, W3, s);
    if (e != cudaSuccess) return e;
    CUtensorMap mx, mw;
    if (!gate_bf16_map(&mx, x_rows, rows, d, BM) ||
        !gate_bf16_map(&mw, W3, 3LL * d * groups, 2LL * n_pad, BK))
        return cudaErrorInvalidValue;
    const GroupArgs ga{offsets, blk_prefix, perm, gate_scale, groups};
    e = launch_by_k<true>(k, mx, mw, eps, nullptr, 0, d, n, n_pad, std_floor, idx, gates, tie,
                          load_part, imp_part, err, ga, s);
    if (e != cudaSuccess) return e;
    const long long outs = (long long)groups * n;
    group_tile_reduce_kernel<<<(int)((outs + 255) / 256), 256, 0, s>>>(
        load_part, imp_part, blk_prefix, groups, n, load, importance);
    note_launch();
    return cudaGetLastError();
}

}  // namespace moe
