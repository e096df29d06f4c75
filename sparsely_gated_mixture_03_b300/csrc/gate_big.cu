// Noisy top-k gate for more than 256 experts on the tensor cores: logits in TMEM,
// selection in the epilogue, clean logits and noise std written once for the Load.
//
// "Mixture of Experts: Outrageously Large Neural Networks" (intuitivepapers.ai):
//   "Noisy top-k gating", eq (4): H = x W_g (+ b_g) + eps * (Softplus(x W_noise) + floor);
//   eqs (3)/(5): keep the k largest H, softmax over them; the forward-pass listing
//   takes the top k+1 (the (k+1)-th and k-th values are the two thresholds of the load
//   probability, "A differentiable count of examples", eqs (8)-(10)).
//
// The whole logit row of a token does not fit in TMEM for n > 256, so a 128-token tile
// walks the experts in chunks of 128 (the exact three-term bf16 split GEMM of
// gate_tc.cu, same W3 layout): chunk c's clean and noise logits land in one of two
// 256-column TMEM buffers while the sixteen epilogue warps work on the other.  A
// thread owns one token row and 32 experts of every chunk: it forms H and std, writes
// the clean logit (with the bias) and 1/std to memory for the Load pass, keeps a running
// top-(k+1) over all its chunks, and after the last chunk the four lists of a row are
// merged through shared memory (larger H first, equal H -> lower index) into the kept
// experts, their softmax, the near-tie flag and the two thresholds.  The noisy logits
// H never reach memory.
//
// clean and 1/std are written in a blocked layout that matches the epilogue's registers:
// element (t, e) at (((tile(t) * G + e / 16) * 4 + (e % 16) / 4) * 128 + t % 128) * 4
// + e % 4, G = n_pad / 16: a warp (32 consecutive rows, the same 16 experts) writes each
// group of four experts as 512 contiguous bytes with one 16-byte store a lane (2 KB in
// four fully used stores, where row-major rows would be 32 scattered 64-byte pieces);
// gate_load_blocked_kernel reads them back the same way and forms the per-tile Load and
// Importance sums.
#include <cuda.h>
#include <stdint.h>

#include "common.cuh"
#include "launch.h"
#include "tc.cuh"

namespace moe {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;                  // one chunk: 128 clean + 128 noise columns
constexpr int EPT = 128;                 // experts per chunk
constexpr int BK = 64;
constexpr int EPI_WARPS = 16;            // four per TMEM lane quarter
constexpr int THREADS = 64 + 32 * EPI_WARPS;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BK * (BN / 2) * 2;   // this CTA's half of a chunk's columns
constexpr int A_SLOTS = 8;               // k-blocks of x held at once: d <= 512 stays resident
constexpr int MAX_STAGES = 4;
constexpr uint32_t TMEM_COLS = 2 * BN;   // two chunk buffers
constexpr uint32_t IDESC = tc::idesc_bf16_f32(2 * BM, BN, false, true);   // pair MMA, M = 256

// The merge lists of a row: K1 entries a list, rows an odd number of words apart (no
// bank conflicts across a warp's rows); the B ring takes what shared memory is left.
template <int K1> struct Smem {
    static constexpr int KP = K1 | 1;
    float mv[4][BM][KP];
    int mi[4][BM][KP];
    int vote[EPI_WARPS];
};
template <int K1> constexpr int stages() { return K1 <= 5 ? 4 : 3; }
struct Barriers {
    uint64_t full[MAX_STAGES], empty[MAX_STAGES], afull[A_SLOTS], aempty[A_SLOTS], tfull[2],
        tempty[2], done;
    uint32_t tmem_base;
    int abort_flag;
};
template <int K1> constexpr size_t smem_bytes() {
    return 1024 + (size_t)A_SLOTS * A_BYTES + (size_t)stages<K1>() * B_BYTES + sizeof(Smem<K1>) +
           sizeof(Barriers);
}
static_assert(smem_bytes<9>() <= 232448 && smem_bytes<5>() <= 232448 &&
              smem_bytes<4>() <= 232448, "shared memory");

__device__ __forceinline__ void epi_bar() {
    asm volatile("bar.sync 1, %0;" ::"n"(32 * EPI_WARPS) : "memory");
}

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, int* err) {
    const long long t0 = clock64();
    while (!tc::mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > tc::kWaitCycles) { raise_error(err, DEV_TIMEOUT); return; }
    }
}

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

// 18 warps: at most 96 registers a thread (the SM's four register files take 5/5/4/4).
template <int K1>
__global__ void __launch_bounds__(THREADS, 1)
gate_big_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                const float* __restrict__ eps, const float* __restrict__ b_g, int T, int d, int n,
                int n_pad, float std_floor, float* __restrict__ clean_out,
                float* __restrict__ std_out, int32_t* __restrict__ idx_out,
                float* __restrict__ gates_out, uint8_t* __restrict__ tie_out,
                float* __restrict__ thr_out, int* err) {
    constexpr int K = K1 - 1;
    constexpr int STAGES = stages<K1>();
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* a_smem = smem;                                   // A_SLOTS x-tile k-blocks
    uint8_t* b_smem = smem + A_SLOTS * A_BYTES;               // the B ring
    Smem<K1>* fs = reinterpret_cast<Smem<K1>*>(b_smem + STAGES * B_BYTES);
    Barriers* bar = reinterpret_cast<Barriers*>(b_smem + STAGES * B_BYTES + sizeof(Smem<K1>));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int C = n_pad / EPT;                // chunks per tile
    // SM pairs: a cluster of two CTAs takes 256-token pair tiles, each CTA its own 128
    // token rows and 128 of a chunk's 256 split-weight columns
    const uint32_t rank = tc::cluster_ctarank();
    const int unit0 = (int)(blockIdx.x >> 1), units = (int)(gridDim.x >> 1);
    const int total = (T + 2 * BM - 1) / (2 * BM);
    const int KBX = d / BK;
    const int KB = 3 * KBX;
    // d <= 512: a tile's x rows are loaded once and serve every chunk and term (slot kx
    // holds k-block kx); else x streams with B, slot `stage` beside B stage `stage`
    const bool resident = KBX <= A_SLOTS;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) { tc::mbar_init(&bar->full[s], 1); tc::mbar_init(&bar->empty[s], 1); }
        for (int s = 0; s < A_SLOTS; ++s) { tc::mbar_init(&bar->afull[s], 1); tc::mbar_init(&bar->aempty[s], 1); }
        for (int a = 0; a < 2; ++a) {
            tc::mbar_init(&bar->tfull[a], 1);
            // the leader's release barrier counts both CTAs' epilogue warps
            tc::mbar_init(&bar->tempty[a], 2 * EPI_WARPS);
        }
        tc::mbar_init(&bar->done, 1);
        bar->abort_flag = 0;
        tc::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) { tc::tma_prefetch(&tmX); tc::tma_prefetch(&tmW); }
    if (warp == 1) tc::tmem_alloc_pair(&bar->tmem_base, TMEM_COLS);
    griddep_wait();                    // inputs written by the previous kernel are visible
    griddep_launch_dependents();
    tc::fence_before_sync();
    __syncthreads();
    tc::cluster_sync();                // both CTAs' barriers exist before any remote use
    tc::fence_after_sync();
    const uint32_t tmem = bar->tmem_base;
    volatile int* abort_flag = &bar->abort_flag;

    if (warp == 0) {
        if (lane == 0) {   // TMA producer: per tile, chunk-major, terms lo, mid, hi
            int stage = 0, jt = 0;
            uint32_t phase = 0, armed = 0, armed_parity = 0;
            bool ok = true;
            for (int tile = unit0; tile < total && ok && !*abort_flag; tile += units, ++jt) {
                // a pair tile whose upper half lies past T leaves the peer's A rows unread
                const bool upper_live = tile * 2 * BM + BM < T;
                const bool load_a = rank == 0 || upper_live;
                const int row0 = tile * 2 * BM + (int)rank * BM;
                for (int cc = 0; cc < C && ok; ++cc) {
                    for (int kb = 0; kb < KB; ++kb) {
                        const int kx = kb % KBX;
                        const int term = 2 - kb / KBX;
                        if (resident && cc == 0 && kb < KBX) {
                            // slot kx gets this tile's k-block once the previous tile's
                            // last MMA on it (chunk C-1, term hi) has completed
                            if (load_a && !tc::mbar_wait(&bar->aempty[kx], (jt & 1) ^ 1,
                                                         abort_flag, err)) {
                                ok = false;
                                break;
                            }
                            const uint32_t afull_c = tc::mapa(tc::smem_u32(&bar->afull[kx]), 0);
                            if (rank == 0)
                                tc::mbar_arrive_expect_tx(&bar->afull[kx],
                                                          upper_live ? 2 * A_BYTES : A_BYTES);
                            if (load_a)
                                tc::tma_load_2d_pair(a_smem + kx * A_BYTES, &tmX, afull_c,
                                                     kx * BK, row0);
                        }
                        if (!tc::mbar_wait(&bar->empty[stage], phase ^ 1, abort_flag, err)) {
                            ok = false;
                            break;
                        }
                        uint8_t* b_dst = b_smem + stage * B_BYTES;
                        // both CTAs' copies complete on the leader's barrier, armed by it
                        const uint32_t full_c = tc::mapa(tc::smem_u32(&bar->full[stage]), 0);
                        if (rank == 0) {
                            const int a_tx = resident ? 0 : (upper_live ? 2 * A_BYTES : A_BYTES);
                            tc::mbar_arrive_expect_tx(&bar->full[stage], 2 * B_BYTES + a_tx);
                        }
                        if (!resident && load_a)
                            tc::tma_load_2d_pair(a_smem + stage * A_BYTES, &tmX, full_c, kx * BK,
                                                 row0);
#pragma unroll
                        for (int i = 0; i < BN / 128; ++i)
                            tc::tma_load_2d_pair(b_dst + i * (BK * 128), &tmW, full_c,
                                                 cc * BN + (int)rank * (BN / 2) + 64 * i,
                                                 term * d + kx * BK);
                        armed |= 1u << stage;
                        armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                        if (++stage == STAGES) { stage = 0; phase ^= 1; }
                    }
                }
            }
            // every armed stage consumed by the pair MMA (the peer's copies complete on
            // the leader's barrier) before the CTA exits; resident x slots likewise
            for (int s = 0; s < STAGES; ++s)
                if ((armed >> s) & 1u) drain_wait(&bar->empty[s], (armed_parity >> s) & 1u, err);
            if (resident && jt > 0)
                for (int kx = 0; kx < KBX; ++kx) drain_wait(&bar->aempty[kx], (jt - 1) & 1, err);
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {   // MMA issuer (the leader's, for both CTAs): chunk
                                        // after chunk into the two TMEM buffers
            int stage = 0, buf = 0, jt = 0;
            uint32_t phase = 0, buf_phase = 0;
            bool ok = true;
            for (int tile = unit0; tile < total && ok && !*abort_flag; tile += units, ++jt) {
                for (int cc = 0; cc < C && ok; ++cc) {
                    if (!tc::mbar_wait(&bar->tempty[buf], buf_phase ^ 1, abort_flag, err)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after_sync();
                    for (int kb = 0; kb < KB; ++kb) {
                        const int kx = kb % KBX;
                        if (resident && cc == 0 && kb < KBX &&
                            !tc::mbar_wait(&bar->afull[kx], jt & 1, abort_flag, err)) {
                            ok = false;
                            break;
                        }
                        if (!tc::mbar_wait(&bar->full[stage], phase, abort_flag, err)) {
                            ok = false;
                            break;
                        }
                        tc::fence_after_sync();
                        const uint32_t a_addr =
                            tc::smem_u32(a_smem + (resident ? kx : stage) * A_BYTES);
                        const uint32_t b_addr = tc::smem_u32(b_smem + stage * B_BYTES);
#pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk) {
                            const uint64_t ad = tc::sdesc_sw128(a_addr + kk * 32, 16, 1024);
                            const uint64_t bd = tc::sdesc_sw128(b_addr + kk * 2048, BK * 128, 1024);
                            tc::mma_bf16_pair(tmem + buf * BN, ad, bd, IDESC,
                                              (kb | kk) != 0 ? 1u : 0u);
                        }
                        tc::mma_commit_pair(&bar->empty[stage], 0x3);
                        // the tile's last MMA on x slot kx: both CTAs may refill it
                        if (resident && cc == C - 1 && kb >= 2 * KBX)
                            tc::mma_commit_pair(&bar->aempty[kx], 0x3);
                        if (++stage == STAGES) { stage = 0; phase ^= 1; }
                    }
                    if (!ok) break;
                    tc::mma_commit_pair(&bar->tfull[buf], 0x3);
                    if (++buf == 2) { buf = 0; buf_phase ^= 1; }
                }
            }
            tc::mma_commit_pair(&bar->done, 0x1);   // every MMA done before TMEM is freed
            drain_wait(&bar->done, 0, err);
        }
    } else {               // epilogue: warps 2..17
        const int ew = warp - 2;
        const int quarter = warp & 3;            // TMEM lanes 32*quarter .. +31
        const int sub = ew >> 2;                 // 32 experts of every chunk
        const int row = quarter * 32 + lane;     // token row inside the tile
        const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
        const bool vec = (n % 4) == 0;
        int buf = 0;
        uint32_t buf_phase = 0;
        const uint32_t tempty_c[2] = {tc::mapa(tc::smem_u32(&bar->tempty[0]), 0),
                                      tc::mapa(tc::smem_u32(&bar->tempty[1]), 0)};
        for (int ptile = unit0; ptile < total; ptile += units) {
            const int tile = 2 * ptile + (int)rank;       // this CTA's 128-row tile
            const int t = tile * BM + row;
            const bool live = t < T;
            const bool tile_live = tile * BM < T;         // not the dead half of a pair tile
            const float* erow = eps != nullptr ? eps + (size_t)(live ? t : 0) * n : nullptr;
            const bool noisy = live && eps != nullptr;    // eps == nullptr: no noise
            const int G = n_pad / 16;
            float v[K1];
            int ix[K1];
#pragma unroll
            for (int q = 0; q < K1; ++q) { v[q] = -INFINITY; ix[q] = 0x7fffffff; }
            int ok = 1;
            for (int cc = 0; cc < C; ++cc) {
                const int e0c = cc * EPT + sub * 32;
                const uint32_t col = (uint32_t)(buf * BN + sub * 32);
#pragma unroll 1
                for (int h = 0; h < 32; h += 16) {
                    const int e0 = e0c + h;
                    float ep[16];          // noise values first: they do not depend on the MMA
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
                            okc = tc::mbar_wait(&bar->tfull[buf], buf_phase, abort_flag, err) ? 1 : 0;
                        okc = __shfl_sync(0xffffffffu, okc, 0);
                        if (!okc) { ok = 0; break; }
                        tc::fence_after_sync();
                    }
                    uint32_t rc[16], rr[16];
                    tc::tmem_ld16(t_lane + col + h, rc);
                    tc::tmem_ld16(t_lane + col + EPT + h, rr);
                    tc::tmem_ld_wait();
                    if (h == 16) {         // this warp is done with the buffer
                        tc::fence_before_sync();
                        __syncwarp();
                        if (lane == 0) tc::mbar_arrive_cluster_relaxed(tempty_c[buf]);
                    }
                    float cv[16], sv[16];
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        const int e = e0 + q;
                        cv[q] = __uint_as_float(rc[q]) + ((b_g != nullptr && e < n) ? b_g[e] : 0.0f);
                        sv[q] = softplus_f32(__uint_as_float(rr[q])) + std_floor;
                        const float hv = fmaf(ep[q], sv[q], cv[q]);
                        if (live && e < n) topk_insert<K1>(v, ix, hv, e);
                        sv[q] = rcp_approx(sv[q]);   // the Load pass multiplies by 1/std
                    }
                    if (tile_live) {   // the blocked layout: four 512-byte warp stores each
                        const size_t o = ((size_t)tile * G + e0 / 16) * (BM * 16) + row * 4;
#pragma unroll
                        for (int q = 0; q < 16; q += 4) {
                            *reinterpret_cast<float4*>(clean_out + o + q * BM) =
                                make_float4(cv[q], cv[q + 1], cv[q + 2], cv[q + 3]);
                            *reinterpret_cast<float4*>(std_out + o + q * BM) =
                                make_float4(sv[q], sv[q + 1], sv[q + 2], sv[q + 3]);
                        }
                    }
                }
                if (!ok) break;
                if (++buf == 2) { buf = 0; buf_phase ^= 1; }
            }

            // ---- merge the four lists of a row (all four threads of the row agree)
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
                        const float c2 = fs->mv[s2][row][head[s2]];
                        const int x2 = fs->mi[s2][row][head[s2]];
                        const bool take = c2 > bv || (c2 == bv && x2 < bx);
                        bv = take ? c2 : bv;
                        bx = take ? x2 : bx;
                        bs = take ? s2 : bs;
                    }
                    v[q] = bv;
                    ix[q] = bx;
#pragma unroll
                    for (int s2 = 0; s2 < 4; ++s2) head[s2] += (bs == s2) ? 1 : 0;
                }
            }
            if (live && sub == 0) {
                float gk[K];
                float s = 0.0f;
#pragma unroll
                for (int j = 0; j < K; ++j) { gk[j] = expf(v[j] - v[0]); s += gk[j]; }
                const float inv = 1.0f / s;
#pragma unroll
                for (int j = 0; j < K; ++j) {
                    idx_out[(size_t)t * K + j] = ix[j];
                    gates_out[(size_t)t * K + j] = gk[j] * inv;
                }
                // k = n: v[K] is the -inf sentinel, the gap is +inf, no tie
                if (tie_out != nullptr) tie_out[t] = (v[K - 1] - v[K]) < 1e-5f ? 1 : 0;
                thr_out[2 * (size_t)t + 0] = v[K];       // kth_excluding for a kept expert
                thr_out[2 * (size_t)t + 1] = v[K - 1];   // ... for an expert not kept
            }
            epi_bar();                                   // the lists are read before reuse
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::cluster_sync();                // no remote arrive or copy targets an exited CTA
    tc::fence_after_sync();
    if (warp == 1) tc::tmem_dealloc_pair(tmem, TMEM_COLS);
}

// Sums over the warp's 32 lanes of v[0..15]; lanes l and l ^ 16 end with the sum of
// v[l % 16].  Four halving exchanges (offsets 8, 4, 2, 1: a lane keeps the half of its
// values that its lane bit selects and adds the partner's copy of that half), then the
// two half-warps added: 16 shuffles instead of the 80 of a butterfly per value.  The
// order of every sum is fixed.
__device__ __forceinline__ float reduce_scatter16(float (&v)[16], int lane) {
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int q = 0; q < o; ++q) {
            const float send = up ? v[q] : v[q + o];
            const float keep = up ? v[q + o] : v[q];
            v[q] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 16);
}

// Per-tile Load and Importance from the blocked clean / (1/std): CTA (tile, 8 groups of
// 16 experts), warp w one group; lane l takes rows l, l+32, l+64, l+96 of the tile in
// that order (each a 16-byte piece of four 512-byte warp loads of clean and of 1/std),
// forms P = Phi((clean - thr) * (1/std)) with thr the (k+1)-th largest H for a kept
// expert and the k-th otherwise (the kept experts of the row as a 16-bit mask), and the
// kept gate; the four rows are added in fp32, then the 32 lanes by reduce_scatter16.
// Three CTAs an SM (at most 85 registers a thread) keep loads in flight while others
// compute.
template <int K>
__global__ void __launch_bounds__(256, 3)
gate_load_blocked_kernel(const float* __restrict__ clean, const float* __restrict__ stdv,
                         const int32_t* __restrict__ idx, const float* __restrict__ gates,
                         const float* __restrict__ thr, int T, int n, int G,
                         float* __restrict__ load_part, float* __restrict__ imp_part) {
    griddep_wait();
    griddep_launch_dependents();
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int tile = blockIdx.x;
    const int g = blockIdx.y * 8 + w;
    if (g >= G) return;
    const int e0 = g * 16;
    float sp[16], sg[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) { sp[j] = 0.0f; sg[j] = 0.0f; }
#pragma unroll 1
    for (int rr = 0; rr < BM; rr += 32) {
        const int row = rr + lane;
        const int t = tile * BM + row;
        if (t >= T) continue;
        const size_t o = ((size_t)tile * G + g) * (BM * 16) + row * 4;
        float cl[16], sd[16];
#pragma unroll
        for (int q = 0; q < 16; q += 4) {
            const float4 a = *reinterpret_cast<const float4*>(clean + o + q * BM);
            const float4 b = *reinterpret_cast<const float4*>(stdv + o + q * BM);
            cl[q] = a.x; cl[q + 1] = a.y; cl[q + 2] = a.z; cl[q + 3] = a.w;
            sd[q] = b.x; sd[q + 1] = b.y; sd[q + 2] = b.z; sd[q + 3] = b.w;
        }
        const float thr_in = thr[2 * (size_t)t], thr_not = thr[2 * (size_t)t + 1];
        unsigned kmask = 0u;                     // the row's kept experts among these 16
#pragma unroll
        for (int j = 0; j < K; ++j) {
            const unsigned o = (unsigned)(idx[(size_t)t * K + j] - e0);
            if (o < 16u) kmask |= 1u << o;
        }
#pragma unroll
        for (int q = 0; q < 16; ++q) {
            if (e0 + q >= n) continue;
            const bool kept = (kmask >> q) & 1u;
            sp[q] += normal_cdf_f32((cl[q] - (kept ? thr_in : thr_not)) * sd[q]);
        }
        if (kmask != 0u) {                       // a gate only where an expert is kept
#pragma unroll
            for (int j = 0; j < K; ++j) {
                const int o = idx[(size_t)t * K + j] - e0;
                const float gj = gates[(size_t)t * K + j];
#pragma unroll
                for (int q = 0; q < 16; ++q) sg[q] += o == q ? gj : 0.0f;
            }
        }
    }
    const float vp = reduce_scatter16(sp, lane);
    const float vg = reduce_scatter16(sg, lane);
    if (lane < 16 && e0 + lane < n) {
        load_part[(size_t)tile * n + e0 + lane] = vp;
        imp_part[(size_t)tile * n + e0 + lane] = vg;
    }
}

template <int K1>
cudaError_t launch_big(const CUtensorMap& mx, const CUtensorMap& mw, const float* eps,
                       const float* b_g, int T, int d, int n, int n_pad, float std_floor,
                       float* clean, float* stdv, int32_t* idx, float* gates, uint8_t* tie,
                       float* thr, int* err, cudaStream_t s) {
    static bool configured = false;
    if (!configured) {
        const cudaError_t e = cudaFuncSetAttribute(
            gate_big_kernel<K1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes<K1>());
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const cudaError_t e =
        launch_pdl(gate_big_kernel<K1>, dim3((gate_sm_count() / 2) * 2), dim3(THREADS),
                   smem_bytes<K1>(), s, 2,
                   mx, mw, eps, b_g, T, d, n, n_pad, std_floor, clean, stdv, idx, gates, tie, thr,
                   err);
    note_launch();
    return e;
}

}  // namespace

int gate_big_tiles(int T) { return (T + BM - 1) / BM; }

size_t gate_big_blocked_floats(int T, int n) {
    return (size_t)gate_big_tiles(T) * BM * gate_tc_n_pad(n);
}

cudaError_t launch_gate_load_blocked(const float* clean, const float* stdv, const int32_t* idx,
                                     const float* gates, const float* thr, int T, int n, int k,
                                     float* load_part, float* imp_part, float* load,
                                     float* importance, cudaStream_t s) {
    const int tiles = gate_big_tiles(T);
    const int G = gate_tc_n_pad(n) / 16;
    const dim3 grid(tiles, (G + 7) / 8);
    cudaError_t e;
    switch (k) {
#define MOE_LOAD_CASE(K)                                                                    \
    case K:                                                                                 \
        e = launch_pdl(gate_load_blocked_kernel<K>, grid, dim3(256), 0, s, 1, clean, stdv, idx, \
                       gates, thr, T, n, G, load_part, imp_part);                            \
        break;
        MOE_LOAD_CASE(1) MOE_LOAD_CASE(2) MOE_LOAD_CASE(3) MOE_LOAD_CASE(4)
        MOE_LOAD_CASE(5) MOE_LOAD_CASE(6) MOE_LOAD_CASE(7) MOE_LOAD_CASE(8)
#undef MOE_LOAD_CASE
        default: return cudaErrorInvalidValue;
    }
    note_launch();
    if (e != cudaSuccess) return e;
    return launch_partial_reduce(load_part, importance != nullptr ? imp_part : nullptr, tiles, n,
                                 load, importance, s);
}

cudaError_t launch_gate_big_tc(const void* x, const float* W_g, const float* W_noise,
                               const float* eps, const float* b_g, int T, int d, int n, int k,
                               float std_floor, void* W3, float* clean, float* stdv, int32_t* idx,
                               float* gates, uint8_t* tie, float* thr, int* err, cudaStream_t s) {
    const int n_pad = gate_tc_n_pad(n);
    cudaError_t e = launch_gate_split_weights(W_g, W_noise, d, n, W3, s);
    if (e != cudaSuccess) return e;
    CUtensorMap mx, mw;
    if (!gate_bf16_map(&mx, x, T, d, BM) || !gate_bf16_map(&mw, W3, 3LL * d, 2LL * n_pad, BK))
        return cudaErrorInvalidValue;
    switch (k + 1) {
#define MOE_BIG_CASE(K1)                                                                    \
    case K1:                                                                                \
        return launch_big<K1>(mx, mw, eps, b_g, T, d, n, n_pad, std_floor, clean, stdv, idx,  \
                              gates, tie, thr, err, s);
        MOE_BIG_CASE(2) MOE_BIG_CASE(3) MOE_BIG_CASE(4) MOE_BIG_CASE(5)
        MOE_BIG_CASE(6) MOE_BIG_CASE(7) MOE_BIG_CASE(8) MOE_BIG_CASE(9)
#undef MOE_BIG_CASE
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace moe
