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
// whole logit row stays on the SM.  Sixteen epilogue warps, four per TMEM lane quarter;
// a thread owns one token row and 32 experts of every chunk:
//   pass 1: H, 1/std (written back over the noise columns) and clean + b_g (over the
//           clean columns), running top-(k+1);
//   merge:  the four partial lists through shared memory (larger H first, equal H ->
//           lower index), softmax over the k kept, the near-tie flag; each kept gate
//           is added to its expert's tile sum in 2^-40 fixed point by an integer
//           shared-memory atomic (exact, so the order of the adds does not matter);
//   pass 2: P for every (row, expert), summed over each warp's 32 rows by a fixed warp
//           reduce-scatter, then over the 4 quarters in a fixed order
//           -> load_part / imp_part [token block][n] (summed over blocks elsewhere).
// The chunks have their own full/empty barriers: pass 1 of chunk 0 overlaps the MMAs of
// chunk 1, and the next tile's MMAs into chunk c start as soon as pass 2 has read c.
//
// The flat gate runs on SM pairs: a cluster of two CTAs takes 256 tokens, each CTA its
// own 128 token rows (A) and 128 of a chunk's 256 columns of the split weights (B), and
// the leader issues tcgen05.mma.cta_group::2 (M = 256): each SM then streams half the
// split weights per token (the one-CTA kernel re-read all 1.5 MB of them from L2 for
// every 128 tokens, which bounded its MMA rate).  Each CTA's TMEM holds its own rows'
// logits, so the epilogue is the one-CTA kernel's; its releases of a chunk go to the
// leader's barrier, which counts both CTAs' epilogue warps.
//
// Switch mode ("From LSTMs to Switch and Mixtral": the softmax runs over all n logits
// first and a kept expert's gate is its probability): pass 1 keeps H instead of 1/std in
// TMEM; after the merge each thread sums exp(H - max) over its experts, the four sums of
// a row meet in shared memory, the gates are exp(H_j - max) / sum, and pass 2 sums each
// expert's probability and its kept count over the tile's rows (imp_part, load_part).
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
constexpr int EPI_WARPS = 16;            // four per TMEM lane quarter
constexpr int THREADS = 64 + 32 * EPI_WARPS;
constexpr int A_BYTES = BM * BK * 2;
constexpr uint32_t TMEM_COLS = 512;
constexpr int KMAX1 = 9;
constexpr int MAX_CHUNKS = 2;

// One CTA a 128-token tile (3 stages of A + all 256 columns of B), or (PAIR) SM pairs:
// a cluster of two CTAs computes a 256-token tile with tcgen05.mma.cta_group::2, each CTA
// loading its own 128 token rows and half (128 columns) of B, so every SM streams half
// the split weights per token and a stage is 32 KB (four fit).
template <bool PAIR> struct Cfg {
    static constexpr int B_BYTES = BK * (PAIR ? BN / 2 : BN) * 2;
    static constexpr int SB = A_BYTES + B_BYTES;
    static constexpr int STAGES = PAIR ? 4 : 3;
    static constexpr uint32_t IDESC = tc::idesc_bf16_f32(PAIR ? 2 * BM : BM, BN, false, true);
};

struct Smem {
    float red_p[4][2 * EPT];
    float red_g[4][2 * EPT];             // Switch mode: probability sums of the quarters
    unsigned long long imp_fx[2 * EPT];  // kept gates of the tile, fixed point (2^-40)
    float mv[4][BM][KMAX1];
    int mi[4][BM][KMAX1];
    float bias[2 * EPT];
    float ssum[4][BM];                   // Switch mode: partial softmax sums of a row
    int hist[2 * EPT];                   // routed rows of the tile per expert (dispatch counts)
    int vote[EPI_WARPS];
};
constexpr int MAX_STAGES = 4;
struct Barriers {
    uint64_t full[MAX_STAGES], empty[MAX_STAGES], tfull[MAX_CHUNKS], tempty[MAX_CHUNKS], done;
    uint32_t tmem_base;
    int abort_flag;
};
template <bool PAIR>
constexpr size_t smem_bytes() {
    return 1024 + (size_t)Cfg<PAIR>::STAGES * Cfg<PAIR>::SB + sizeof(Smem) + sizeof(Barriers);
}
static_assert(smem_bytes<true>() <= 232448 && smem_bytes<false>() <= 232448, "shared memory");

__device__ __forceinline__ void epi_bar() {
    asm volatile("bar.sync 1, %0;" ::"n"(32 * EPI_WARPS) : "memory");
}

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

// Insert (hv, e) into the descending list v/ix of length K1 (strictly larger values
// move ahead, so among equal values the one inserted first, the lower index, stays
// ahead).  Branch-free: one compare and four selects per slot.
template <int K1>
__device__ __forceinline__ void topk_insert(float (&v)[K1], int (&ix)[K1], float hv, int e) {
    float cv = hv;
    int ci = e;
#pragma unroll
    for (int u = 0; u < K1; ++u) {
        const bool sw = cv > v[u];
        const float tv = v[u];
        const int ti = ix[u];
        v[u] = sw ? cv : tv;
        ix[u] = sw ? ci : ti;
        cv = sw ? tv : cv;
        ci = sw ? ti : ci;
    }
}

// 18 warps: the SM's four register files take five, five, four and four of them, so a
// thread gets at most 96 registers; the epilogue works on 16 columns at a time.
template <int K1, bool GROUPED, bool SWITCH, bool PAIR>
__global__ void __launch_bounds__(THREADS, 1)
gate_fused_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                  const float* __restrict__ eps, const float* __restrict__ b_g, int T, int d, int n,
                  int n_pad, float std_floor, int32_t* __restrict__ idx_out,
                  float* __restrict__ gates_out, uint8_t* __restrict__ tie_out,
                  float* __restrict__ load_part, float* __restrict__ imp_part, int* err,
                  const GroupArgs ga, int32_t* __restrict__ tile_counts) {
    static_assert(!(PAIR && GROUPED), "the grouped mode runs one CTA a tile");
    constexpr int K = K1 - 1;
    constexpr int STAGES = Cfg<PAIR>::STAGES;
    constexpr int SB = Cfg<PAIR>::SB;
    constexpr uint32_t IDESC = Cfg<PAIR>::IDESC;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    Smem* fs = reinterpret_cast<Smem*>(smem + STAGES * SB);
    Barriers* bar = reinterpret_cast<Barriers*>(smem + STAGES * SB + sizeof(Smem));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int CPT = n_pad / EPT;              // TMEM chunks: 1 or 2
    const int KBX = d / BK;
    const int KB = 3 * KBX;
    // PAIR: this CTA's rank in its pair, the pair index and the number of pairs
    const uint32_t rank = PAIR ? tc::cluster_ctarank() : 0u;
    const int unit0 = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
    const int units = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) { tc::mbar_init(&bar->full[s], 1); tc::mbar_init(&bar->empty[s], 1); }
        for (int c = 0; c < MAX_CHUNKS; ++c) {
            tc::mbar_init(&bar->tfull[c], 1);
            // PAIR: the leader's release barrier counts both CTAs' epilogue warps
            tc::mbar_init(&bar->tempty[c], PAIR ? 2 * EPI_WARPS : EPI_WARPS);
        }
        tc::mbar_init(&bar->done, 1);
        bar->abort_flag = 0;
        tc::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) { tc::tma_prefetch(&tmX); tc::tma_prefetch(&tmW); }
    if (warp == 1) {
        if (PAIR) tc::tmem_alloc_pair(&bar->tmem_base, TMEM_COLS);
        else tc::tmem_alloc(&bar->tmem_base, TMEM_COLS);
    }
    griddep_wait();                    // inputs written by the previous kernel are visible
    griddep_launch_dependents();
    for (int e = (int)threadIdx.x - 64; e >= 0 && e < 2 * EPT; e += 32 * EPI_WARPS) {
        fs->bias[e] = (b_g != nullptr && e < n) ? b_g[e] : 0.0f;
        fs->hist[e] = 0;
        fs->imp_fx[e] = 0ull;
    }
    tc::fence_before_sync();
    __syncthreads();
    if (PAIR) tc::cluster_sync();      // both CTAs' barriers exist before any remote use
    tc::fence_after_sync();
    const uint32_t tmem = bar->tmem_base;
    volatile int* abort_flag = &bar->abort_flag;
    // work units: 128-row tiles, or (PAIR) 256-row pair tiles
    const int total = PAIR ? (T + 2 * BM - 1) / (2 * BM) : tile_count<GROUPED>(T, ga);
    const int tiles128 = (T + BM - 1) / BM;

    if (warp == 0) {
        if (lane == 0) {   // TMA producer: chunk-major, terms lo, mid, hi (see gate_tc.cu)
            int stage = 0;
            uint32_t phase = 0, armed = 0, armed_parity = 0;
            for (int tile = unit0; tile < total && !*abort_flag; tile += units) {
                TileRows tr;
                if (PAIR) { tr.row0 = tile * 2 * BM + (int)rank * BM; tr.row_end = T; tr.g = 0; }
                else tr = tile_rows<GROUPED>(tile, T, ga);
                const int w_row0 = tr.g * 3 * d;         // group g's split weights
                for (int cc = 0; cc < CPT; ++cc) {
                    for (int kb = 0; kb < KB; ++kb) {
                        if (!tc::mbar_wait(&bar->empty[stage], phase ^ 1, abort_flag, err)) break;
                        uint8_t* a_dst = smem + stage * SB;
                        uint8_t* b_dst = a_dst + A_BYTES;
                        const int term = 2 - kb / KBX;
                        const int wrow = w_row0 + term * d + (kb % KBX) * BK;
                        if (PAIR) {
                            // both CTAs' copies complete on the leader's barrier, which the
                            // leader arms for both; the peer refills a stage only after the
                            // pair MMA has consumed it (its empty barrier)
                            // a pair tile whose upper half lies past T leaves the peer's A rows
                            // unread (its rows are all dead: nothing of them is stored)
                            const bool upper_live = tile * 2 * BM + BM < T;
                            const uint32_t full_c = tc::mapa(tc::smem_u32(&bar->full[stage]), 0);
                            if (rank == 0)
                                tc::mbar_arrive_expect_tx(&bar->full[stage],
                                                          upper_live ? 2 * SB : 2 * SB - A_BYTES);
                            if (rank == 0 || upper_live)
                                tc::tma_load_2d_pair(a_dst, &tmX, full_c, (kb % KBX) * BK, tr.row0);
#pragma unroll
                            for (int i = 0; i < BN / 128; ++i)
                                tc::tma_load_2d_pair(b_dst + i * (BK * 128), &tmW, full_c,
                                                     cc * BN + (int)rank * (BN / 2) + 64 * i, wrow);
                        } else {
                            tc::mbar_arrive_expect_tx(&bar->full[stage], SB);
                            tc::tma_load_2d(a_dst, &tmX, &bar->full[stage], (kb % KBX) * BK,
                                            tr.row0);
#pragma unroll
                            for (int i = 0; i < BN / 64; ++i)
                                tc::tma_load_2d(b_dst + i * (BK * 128), &tmW, &bar->full[stage],
                                                cc * BN + 64 * i, wrow);
                        }
                        armed |= 1u << stage;
                        armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                        if (++stage == STAGES) { stage = 0; phase ^= 1; }
                    }
                }
            }
            // every armed stage landed (one CTA) or was consumed by the pair MMA (PAIR:
            // the peer's copies complete on the leader's barrier) before the CTA exits
            for (int s = 0; s < STAGES; ++s)
                if ((armed >> s) & 1u)
                    drain_wait(PAIR ? &bar->empty[s] : &bar->full[s], (armed_parity >> s) & 1u,
                               err);
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {   // MMA issuer (PAIR: the leader's, for both CTAs):
                                        // chunk c of a tile waits only for chunk c's release
            int stage = 0;
            uint32_t phase = 0, tphase = 0;
            bool ok = true;
            for (int tile = unit0; tile < total && ok && !*abort_flag; tile += units) {
                for (int cc = 0; cc < CPT && ok; ++cc) {
                    if (!tc::mbar_wait(&bar->tempty[cc], tphase ^ 1, abort_flag, err)) { ok = false; break; }
                    tc::fence_after_sync();
                    for (int kb = 0; kb < KB; ++kb) {
                        if (!tc::mbar_wait(&bar->full[stage], phase, abort_flag, err)) { ok = false; break; }
                        tc::fence_after_sync();
                        const uint32_t a_addr = tc::smem_u32(smem + stage * SB);
                        const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk) {
                            const uint64_t ad = tc::sdesc_sw128(a_addr + kk * 32, 16, 1024);
                            // B N-major: 64-column blocks BK*128 B apart (LBO), 8-row atoms
                            const uint64_t bd = tc::sdesc_sw128(b_addr + kk * 2048, BK * 128, 1024);
                            if (PAIR)
                                tc::mma_bf16_pair(tmem + cc * BN, ad, bd, IDESC,
                                                  (kb | kk) != 0 ? 1u : 0u);
                            else
                                tc::mma_bf16(tmem + cc * BN, ad, bd, IDESC, (kb | kk) != 0 ? 1u : 0u);
                        }
                        if (PAIR) tc::mma_commit_pair(&bar->empty[stage], 0x3);
                        else tc::mma_commit(&bar->empty[stage]);
                        if (++stage == STAGES) { stage = 0; phase ^= 1; }
                    }
                    if (ok) {
                        if (PAIR) tc::mma_commit_pair(&bar->tfull[cc], 0x3);
                        else tc::mma_commit(&bar->tfull[cc]);
                    }
                }
                tphase ^= 1;
            }
            if (PAIR) tc::mma_commit_pair(&bar->done, 0x1);   // every MMA done before TMEM is freed
            else tc::mma_commit(&bar->done);
            drain_wait(&bar->done, 0, err);
        }
    } else {               // epilogue: warps 2..17
        const int ew = warp - 2;
        const int quarter = warp & 3;            // TMEM lanes 32*quarter .. +31
        const int sub = ew >> 2;                 // 32 experts of every chunk
        const int row = quarter * 32 + lane;     // token row inside the tile
        const int etid = threadIdx.x - 64;       // 0..511
        const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
        const bool vec = (n % 4) == 0;
        uint32_t tphase = 0;
        // PAIR: the releases go to the leader's barriers
        const uint32_t tempty_c[MAX_CHUNKS] = {tc::mapa(tc::smem_u32(&bar->tempty[0]), 0),
                                               tc::mapa(tc::smem_u32(&bar->tempty[1]), 0)};
        for (int tile = unit0; tile < total; tile += units) {
            TileRows tr;
            if (PAIR) { tr.row0 = tile * 2 * BM + (int)rank * BM; tr.row_end = T; tr.g = 0; }
            else tr = tile_rows<GROUPED>(tile, T, ga);
            // this CTA's 128-row tile (the index of its partial sums)
            const int ctile = PAIR ? 2 * tile + (int)rank : tile;
            const int p = tr.row0 + row;
            const bool live = p < tr.row_end;
            // t: the row whose noise is read and whose outputs are written (the token
            // in the flat mode, the routed row in the grouped mode)
            const int t = !live ? 0 : (GROUPED ? ga.perm[p] : p);
            const float* erow = eps != nullptr ? eps + (size_t)t * n : nullptr;
            const bool noisy = live && eps != nullptr;    // eps == nullptr: no noise

            // ---- pass 1 over this warp's 32 experts of each chunk: H, 1/std back
            //      into TMEM, running top-(k+1)
            float v[K1];
            int ix[K1];
#pragma unroll
            for (int q = 0; q < K1; ++q) { v[q] = -INFINITY; ix[q] = 0x7fffffff; }
            int ok = 1;
            for (int c = 0; c < CPT; ++c) {
                const int e0c = c * EPT + sub * 32;
                const uint32_t col = (uint32_t)(c * BN + sub * 32);
#pragma unroll 1
                for (int h = 0; h < 32; h += 16) {
                    const int e0 = e0c + h;
                    // noise values first: they do not depend on the MMA
                    float ep[16];
                    if (noisy && vec && e0 + 16 <= n) {
#pragma unroll
                        for (int q = 0; q < 16; q += 4) {
                            const float4 f = *reinterpret_cast<const float4*>(erow + e0 + q);
                            ep[q] = f.x; ep[q + 1] = f.y; ep[q + 2] = f.z; ep[q + 3] = f.w;
                        }
                    } else {
#pragma unroll
                        for (int q = 0; q < 16; ++q) ep[q] = (noisy && e0 + q < n) ? erow[e0 + q] : 0.0f;
                    }
                    if (h == 0) {
                        int okc = 0;
                        if (lane == 0)
                            okc = tc::mbar_wait(&bar->tfull[c], tphase, abort_flag, err) ? 1 : 0;
                        okc = __shfl_sync(0xffffffffu, okc, 0);
                        if (!okc) { ok = 0; break; }
                        tc::fence_after_sync();
                    }
                    uint32_t rc[16], rr[16];
                    tc::tmem_ld16(t_lane + col + h, rc);
                    tc::tmem_ld16(t_lane + col + EPT + h, rr);
                    tc::tmem_ld_wait();
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        const int e = e0 + q;
                        const float cl = __uint_as_float(rc[q]) + fs->bias[e];
                        const float sd = softplus_f32(__uint_as_float(rr[q])) + std_floor;
                        const float hv = fmaf(ep[q], sd, cl);
                        rr[q] = __float_as_uint(SWITCH ? hv : rcp_approx(sd));
                        rc[q] = __float_as_uint(cl);
                        if (live && e < n) topk_insert<K1>(v, ix, hv, e);
                    }
                    tc::tmem_st16(t_lane + col + EPT + h, rr);
                    if (!SWITCH) tc::tmem_st16(t_lane + col + h, rc);   // clean with the bias
                }
                if (!ok) break;
            }
            tc::tmem_st_wait();

            // ---- merge the four lists of a row (all four threads of the row get the
            //      same result: larger H first, equal H -> lower index)
#pragma unroll
            for (int q = 0; q < K1; ++q) { fs->mv[sub][row][q] = v[q]; fs->mi[sub][row][q] = ix[q]; }
            if (lane == 0) fs->vote[ew] = ok;
            epi_bar();
            {
                int all = 1;
#pragma unroll
                for (int w = 0; w < EPI_WARPS; ++w) all &= fs->vote[w];
                if (!all) break;
            }
            {
                int head[4] = {0, 0, 0, 0};
#pragma unroll
                for (int q = 0; q < K1; ++q) {
                    float bv = fs->mv[0][row][head[0]];
                    int bx = fs->mi[0][row][head[0]], bs = 0;
#pragma unroll
                    for (int s2 = 1; s2 < 4; ++s2) {
                        const float cv = fs->mv[s2][row][head[s2]];
                        const int cx = fs->mi[s2][row][head[s2]];
                        const bool take = cv > bv || (cv == bv && cx < bx);
                        bv = take ? cv : bv;
                        bx = take ? cx : bx;
                        bs = take ? s2 : bs;
                    }
                    v[q] = bv;
                    ix[q] = bx;
#pragma unroll
                    for (int s2 = 0; s2 < 4; ++s2) head[s2] += (bs == s2) ? 1 : 0;
                }
            }
            float gk[K];
            float inv_sum = 0.0f;       // Switch mode: 1 / sum over all n of exp(H - max)
            if (SWITCH) {
                float ps = 0.0f;
                for (int c = 0; c < CPT; ++c) {
                    const int e0c = c * EPT + sub * 32;
                    const uint32_t col = (uint32_t)(c * BN + EPT + sub * 32);
#pragma unroll
                    for (int h = 0; h < 32; h += 16) {
                        uint32_t rh[16];
                        tc::tmem_ld16(t_lane + col + h, rh);
                        tc::tmem_ld_wait();
#pragma unroll
                        for (int q = 0; q < 16; ++q)
                            if (live && e0c + h + q < n) ps += expf(__uint_as_float(rh[q]) - v[0]);
                    }
                }
                fs->ssum[sub][row] = ps;
                epi_bar();
                inv_sum = 1.0f / (((fs->ssum[0][row] + fs->ssum[1][row]) + fs->ssum[2][row]) +
                                  fs->ssum[3][row]);
            }
            {
                float s = 0.0f;
#pragma unroll
                for (int j = 0; j < K; ++j) { gk[j] = expf(v[j] - v[0]); s += gk[j]; }
                const float inv = SWITCH ? inv_sum : 1.0f / s;
#pragma unroll
                for (int j = 0; j < K; ++j) gk[j] *= inv;
                if (GROUPED) {             // the product with the primary gate
                    const float sc = live ? ga.gate_scale[t] : 0.0f;
#pragma unroll
                    for (int j = 0; j < K; ++j) gk[j] *= sc;
                }
            }
            if (live && sub == 0) {
                const int id0 = tr.g * n;  // flat id of the group's first expert
#pragma unroll
                for (int j = 0; j < K; ++j) {
                    idx_out[(size_t)t * K + j] = id0 + ix[j];
                    gates_out[(size_t)t * K + j] = gk[j];
                }
                // k = n: v[K] is the -inf sentinel, the gap is +inf, no tie
                if (tie_out != nullptr) tie_out[t] = (v[K - 1] - v[K]) < 1e-5f ? 1 : 0;
                if (tile_counts != nullptr) {     // integer counts: order-independent
#pragma unroll
                    for (int j = 0; j < K; ++j) atomicAdd(&fs->hist[ix[j]], 1);
                }
                if (!SWITCH) {
                    // the tile's Importance: each kept gate in fixed point with 2^-40
                    // steps (a gate is at most 1, a tile at most 128 rows, so the sums
                    // stay below 2^47), added as integers: exact and order-independent
#pragma unroll
                    for (int j = 0; j < K; ++j)
                        atomicAdd(&fs->imp_fx[ix[j]], __float2ull_rn(gk[j] * 1099511627776.0f));
                }
            }
            const float thr_in = v[K], thr_out = v[K - 1];

            // ---- pass 2: P and the kept gates of this warp's experts, summed over rows
            for (int c = 0; c < CPT; ++c) {
                const int e0 = c * EPT + sub * 32;
                const uint32_t col = (uint32_t)(c * BN + sub * 32);
                uint32_t kmask = 0;
#pragma unroll
                for (int j = 0; j < K; ++j) {
                    const unsigned off = (unsigned)(ix[j] - e0);
                    if (off < 32u) kmask |= 1u << off;
                }
                float pz[32];
                float pg[SWITCH ? 32 : 1];
#pragma unroll
                for (int h = 0; h < 32; h += 16) {
                    uint32_t rc[16], rr[16];
                    tc::tmem_ld16(t_lane + col + h, rc);
                    tc::tmem_ld16(t_lane + col + EPT + h, rr);     // 1/std from pass 1
                    tc::tmem_ld_wait();
                    if (h == 16) {                                 // chunk c may be overwritten now
                        tc::fence_before_sync();
                        __syncwarp();
                        if (lane == 0) {
                            if (PAIR) tc::mbar_arrive_cluster_relaxed(tempty_c[c]);
                            else tc::mbar_arrive(&bar->tempty[c]);
                        }
                    }
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        const int e = e0 + h + q;
                        const bool kept = (kmask >> (h + q)) & 1u;
                        float pv = 0.0f;
                        if (SWITCH) {                // kept count (the Switch load)
                            pv = live && kept ? 1.0f : 0.0f;
                        } else if (live && e < n) {
                            const float cl = __uint_as_float(rc[q]);   // clean + b_g (pass 1)
                            pv = normal_cdf_f32((cl - (kept ? thr_in : thr_out)) * __uint_as_float(rr[q]));
                        }
                        pz[h + q] = pv;
                        if (SWITCH)                  // the probability, summed as importance
                            rc[q] = __float_as_uint(live && e < n
                                                        ? expf(__uint_as_float(rr[q]) - v[0]) * inv_sum
                                                        : 0.0f);
                    }
                    if (SWITCH) {
#pragma unroll
                        for (int q = 0; q < 16; ++q) pg[h + q] = __uint_as_float(rc[q]);
                    }
                }
                const float sp = tc::reduce_scatter32(pz, lane);
                fs->red_p[quarter][e0 + lane] = sp;
                if constexpr (SWITCH) {
                    const float sg = tc::reduce_scatter32(pg, lane);
                    fs->red_g[quarter][e0 + lane] = sg;
                }
            }
            tphase ^= 1;
            epi_bar();
            if (etid < n && ctile < (GROUPED ? total : tiles128)) {   // PAIR: a dead half tile
                const size_t o = (size_t)ctile * n + etid;
                load_part[o] = ((fs->red_p[0][etid] + fs->red_p[1][etid]) + fs->red_p[2][etid]) +
                               fs->red_p[3][etid];
                if (SWITCH) {
                    imp_part[o] = ((fs->red_g[0][etid] + fs->red_g[1][etid]) + fs->red_g[2][etid]) +
                                  fs->red_g[3][etid];
                } else {
                    imp_part[o] = __ull2float_rn(fs->imp_fx[etid]) * 9.094947017729282e-13f;
                    fs->imp_fx[etid] = 0ull;     // the next tile adds after its merge barrier
                }
                if (tile_counts != nullptr) {
                    tile_counts[o] = fs->hist[etid];
                    fs->hist[etid] = 0;          // the next tile adds after its merge barrier
                }
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (PAIR) tc::cluster_sync();      // no remote arrive or copy targets an exited CTA
    tc::fence_after_sync();
    if (warp == 1) {
        if (PAIR) tc::tmem_dealloc_pair(tmem, TMEM_COLS);
        else tc::tmem_dealloc(tmem, TMEM_COLS);
    }
}

template <int K1, bool GROUPED, bool SWITCH, bool PAIR>
cudaError_t launch_k(const CUtensorMap& mx, const CUtensorMap& mw, const float* eps,
                     const float* b_g, int T, int d, int n, int n_pad, float std_floor,
                     int32_t* idx, float* gates, uint8_t* tie, float* load_part, float* imp_part,
                     int* err, const GroupArgs& ga, int32_t* tile_counts,
                     cudaStream_t s) {
    static bool configured = false;
    if (!configured) {
        const cudaError_t e =
            cudaFuncSetAttribute(gate_fused_kernel<K1, GROUPED, SWITCH, PAIR>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem_bytes<PAIR>());
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const int sms = gate_sm_count();
    const int grid = PAIR ? (sms / 2) * 2 : sms;
    const cudaError_t e =
        launch_pdl(gate_fused_kernel<K1, GROUPED, SWITCH, PAIR>, dim3(grid), dim3(THREADS),
                   smem_bytes<PAIR>(), s, PAIR ? 2 : 1, mx, mw, eps, b_g, T, d, n, n_pad,
                   std_floor, idx, gates, tie, load_part, imp_part, err, ga, tile_counts);
    note_launch();
    return e;
}

template <bool GROUPED, bool SWITCH, bool PAIR>
cudaError_t launch_by_k(int k, const CUtensorMap& mx, const CUtensorMap& mw, const float* eps,
                        const float* b_g, int T, int d, int n, int n_pad, float std_floor,
                        int32_t* idx, float* gates, uint8_t* tie, float* load_part,
                        float* imp_part, int* err, const GroupArgs& ga, int32_t* tile_counts,
                        cudaStream_t s) {
    switch (k + 1) {
#define MOE_FUSED_CASE(K1)                                                                  \
    case K1:                                                                                \
        return launch_k<K1, GROUPED, SWITCH, PAIR>(mx, mw, eps, b_g, T, d, n, n_pad,         \
                                                   std_floor, idx, gates, tie, load_part,    \
                                                   imp_part, err, ga, tile_counts, s);
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
    griddep_wait();
    griddep_launch_dependents();
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

int gate_fused_tile_tokens() { return BM; }

cudaError_t launch_gate_fused_tc(const void* x, const float* W_g, const float* W_noise,
                                 const float* eps, const float* b_g, int T, int d, int n, int k,
                                 float std_floor, void* W3, int32_t* idx, float* gates,
                                 uint8_t* tie, float* load_part, float* imp_part, float* load,
                                 float* importance, int* err, cudaStream_t s,
                                 int32_t* tile_counts, bool sw) {
    const int n_pad = gate_tc_n_pad(n);
    if (n_pad > 2 * EPT) return cudaErrorInvalidValue;
    cudaError_t e = launch_gate_split_weights(W_g, W_noise, d, n, W3, s);
    if (e != cudaSuccess) return e;
    CUtensorMap mx, mw;
    if (!gate_bf16_map(&mx, x, T, d, BM) || !gate_bf16_map(&mw, W3, 3LL * d, 2LL * n_pad, BK))
        return cudaErrorInvalidValue;
    const GroupArgs none{nullptr, nullptr, nullptr, nullptr, 0};
    e = sw ? launch_by_k<false, true, true>(k, mx, mw, eps, b_g, T, d, n, n_pad, std_floor, idx,
                                            gates, tie, load_part, imp_part, err, none,
                                            tile_counts, s)
           : launch_by_k<false, false, true>(k, mx, mw, eps, b_g, T, d, n, n_pad, std_floor, idx,
                                             gates, tie, load_part, imp_part, err, none,
                                             tile_counts, s);
    if (e != cudaSuccess) return e;
    if (load == nullptr) return cudaSuccess;     // the caller reduces the partials later
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
    e = launch_by_k<true, false, false>(k, mx, mw, eps, nullptr, 0, d, n, n_pad, std_floor, idx,
                                        gates, tie, load_part, imp_part, err, ga, nullptr, s);
    if (e != cudaSuccess) return e;
    const long long outs = (long long)groups * n;
    e = launch_pdl(group_tile_reduce_kernel, dim3((unsigned)((outs + 255) / 256)), dim3(256), 0, s,
                   1, static_cast<const float*>(load_part), static_cast<const float*>(imp_part),
                   blk_prefix, groups, n, load, importance);
    note_launch();
    return e;
}

}  // namespace moe
