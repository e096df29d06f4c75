// Dispatch: group routed rows by expert with a stable counting sort, then copy
// each routed row's input vector into the expert-grouped buffer.
//
// "Mixture of Experts: Outrageously Large Neural Networks" (intuitivepapers.ai),
// "Implementation notes": the forward pass runs each expert on the rows where its
// gate is nonzero.  Routed row r = t*k + j (token t, kept slot j); rows of one
// expert keep ascending r, so the order is reproducible without atomics on the
// positions (integer counts only).
#include <stdint.h>

#include "common.cuh"
#include "launch.h"
#include "reduce.cuh"
#include "tc.cuh"

namespace moe {
namespace {

// Rows expert e keeps: all of them, or at most `cap` (the first in routed-row order).
__device__ __forceinline__ int32_t kept_rows(int32_t count, int cap) {
    return cap > 0 && count > cap ? cap : count;
}

// 1) per tile, per expert: how many routed rows of the tile go to the expert.
__global__ void __launch_bounds__(256)
dispatch_count_kernel(const int32_t* __restrict__ idx, long long R, int n, int chunk,
                      int32_t* __restrict__ tile_counts, int* err) {
    griddep_wait();
    griddep_launch_dependents();
    extern __shared__ int32_t hist[];
    for (int e = threadIdx.x; e < n; e += blockDim.x) hist[e] = 0;
    __syncthreads();
    const long long r0 = (long long)blockIdx.x * chunk;
    const long long r1 = min(R, r0 + chunk);
    for (long long r = r0 + threadIdx.x; r < r1; r += blockDim.x) {
        const int e = idx[r];
        if (e < 0 || e >= n) { raise_error(err, DEV_BAD_INDEX); continue; }
        atomicAdd(&hist[e], 1);
    }
    __syncthreads();
    int32_t* out = tile_counts + (size_t)blockIdx.x * n;
    for (int e = threadIdx.x; e < n; e += blockDim.x) out[e] = hist[e];
}

// 2) one warp per expert: exclusive running sum over tiles (in place) and the
// total, 32 tiles per step with a warp scan.
__global__ void __launch_bounds__(256)
dispatch_column_scan_kernel(int32_t* __restrict__ tile_counts, int tiles, int n,
                            int32_t* __restrict__ totals) {
    griddep_wait();
    griddep_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int e = (int)(((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    if (e >= n) return;
    int32_t carry = 0;
    for (int t0 = 0; t0 < tiles; t0 += 32) {
        const int t = t0 + lane;
        const int32_t c = t < tiles ? tile_counts[(size_t)t * n + e] : 0;
        int32_t incl = c;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int32_t v = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += v;
        }
        if (t < tiles) tile_counts[(size_t)t * n + e] = carry + incl - c;
        carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) totals[e] = carry;
}

// 3) one CTA: offsets = exclusive scan of the per-expert totals (offsets[n] = R).
__global__ void __launch_bounds__(1024)
dispatch_offsets_kernel(const int32_t* __restrict__ totals, int n, int cap,
                        int32_t* __restrict__ offsets) {
    griddep_wait();
    griddep_launch_dependents();
    __shared__ int32_t warp_sums[32];
    const int tid = threadIdx.x;
    const int per = (n + blockDim.x - 1) / blockDim.x;      // experts per thread, contiguous
    const int e0 = tid * per;
    int32_t local = 0;
    for (int i = 0; i < per; ++i)
        if (e0 + i < n) local += kept_rows(totals[e0 + i], cap);
    // block exclusive scan of `local`
    const int lane = tid & 31, wid = tid >> 5;
    int32_t incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int32_t v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
    }
    if (lane == 31) warp_sums[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        int32_t w = lane < (int)(blockDim.x >> 5) ? warp_sums[lane] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int32_t v = __shfl_up_sync(0xffffffffu, w, off);
            if (lane >= off) w += v;
        }
        warp_sums[lane] = w;    // inclusive over warps
    }
    __syncthreads();
    int32_t run = incl - local + (wid > 0 ? warp_sums[wid - 1] : 0);
    for (int i = 0; i < per; ++i) {
        if (e0 + i < n) {
            offsets[e0 + i] = run;
            run += kept_rows(totals[e0 + i], cap);
        }
    }
    if (tid == blockDim.x - 1) offsets[n] = run;
}

// out[g] = sum over g' < g of ceil(rows(g') / block), out[n] = the total: the
// first tile of each group in a tile schedule of `block`-row tiles that never
// mixes groups; with units, the table of those tiles (group, first row, end of the
// group's rows, 0).  The whole CTA (any multiple of 32 threads up to 1024), contiguous
// groups per thread, a block-wide scan.
__device__ __forceinline__ void block_prefix_body(const int32_t* __restrict__ offsets, int n,
                                                  int block, int32_t* __restrict__ out,
                                                  int4* __restrict__ units) {
    __shared__ int32_t warp_sums[32];
    const int tid = threadIdx.x;
    const int per = (n + blockDim.x - 1) / blockDim.x;
    const int g0 = tid * per;
    int32_t local = 0;
    for (int i = 0; i < per; ++i)
        if (g0 + i < n) local += (offsets[g0 + i + 1] - offsets[g0 + i] + block - 1) / block;
    const int lane = tid & 31, wid = tid >> 5;
    int32_t incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int32_t v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
    }
    if (lane == 31) warp_sums[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        int32_t w = lane < (int)(blockDim.x >> 5) ? warp_sums[lane] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int32_t v = __shfl_up_sync(0xffffffffu, w, off);
            if (lane >= off) w += v;
        }
        warp_sums[lane] = w;
    }
    __syncthreads();
    int32_t run = incl - local + (wid > 0 ? warp_sums[wid - 1] : 0);
    for (int i = 0; i < per; ++i) {
        if (g0 + i < n) {
            const int32_t a = offsets[g0 + i], b = offsets[g0 + i + 1];
            const int32_t cnt = (b - a + block - 1) / block;
            out[g0 + i] = run;
            if (units != nullptr)
                for (int32_t u = 0; u < cnt; ++u)
                    units[run + u] = make_int4(g0 + i, a + u * block, b, 0);
            run += cnt;
        }
    }
    if (tid == blockDim.x - 1) out[n] = run;
}

// 2+3 in one launch (n <= 256, one cluster): a CTA takes 32 experts (lane = expert, so
// every load is one 128-byte row piece) and its 16 warps contiguous ranges of tiles;
// pass 1 sums each warp's range (16 tiles at a time, the forward pass's Load and
// Importance partials in the same loads), the warps' sums are scanned in shared memory,
// pass 2 writes the range as exclusive running sums (in place; from registers when a
// range is at most 16 tiles) and the last warp records the totals.
constexpr int SCAN_THREADS = 512;
constexpr int SCAN_WARPS = SCAN_THREADS / 32;
constexpr int SCAN_REG_TILES = 16;
constexpr int SCAN_CLUSTER_MAX = 8;           // CTAs of the one-cluster scan (n <= 256)

static_assert(SCAN_THREADS == 32 * RED_WARPS, "the scan's CTAs run the loss reductions");

// The CTAs (at most eight, 32 experts each) form ONE cluster and meet in distributed
// shared memory.  Each CTA publishes its experts' kept rows and row blocks; each then writes
// the offsets, row-block prefix and unit-table entries of its own experts from the
// lower CTAs' published counts.  The losses follow losses_512's order exactly: CTA c's
// warp 0 holds experts 32c .. 32c+31, which are warp c of the 512-thread reduction, so
// its butterfly is that warp's, and CTA 0 merges the CTAs' results in rank order (the
// warps past the last CTA would add exact zeros), once for the means and once for the
// squared deviations.
__device__ __forceinline__ CSum warp_csum(CSum v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const CSum o = {__shfl_xor_sync(0xffffffffu, v.s, off),
                        __shfl_xor_sync(0xffffffffu, v.c, off)};
        v = (lane & off) ? cmerge(o, v) : cmerge(v, o);   // lower lane first
    }
    return v;
}

__global__ void __launch_bounds__(SCAN_THREADS)
dispatch_scan_cluster_kernel(int32_t* __restrict__ tile_counts, int tiles, int n, int cap,
                             int32_t* __restrict__ totals, int32_t* __restrict__ offsets,
                             const DispatchTail tail) {
    griddep_wait();
    griddep_launch_dependents();
    __shared__ int32_t part[SCAN_WARPS][32];
    __shared__ float part_l[SCAN_WARPS][33], part_i[SCAN_WARPS][33];
    __shared__ int32_t ctot[32], cblk[32];     // published: kept rows, row blocks
    __shared__ float cs[4];                    // published: the CTA's two warp sums (s, c)
    __shared__ float cmean[2];                 // CTA 0: the two means
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const uint32_t rank = tc::cluster_ctarank();
    const int ncta = (int)gridDim.x;           // the grid is one cluster
    const int e = (int)rank * 32 + lane;
    const int span = (tiles + SCAN_WARPS - 1) / SCAN_WARPS;
    const int t0 = wid * span < tiles ? wid * span : tiles;
    const int t1 = t0 + span < tiles ? t0 + span : tiles;
    const bool sums = tail.load_part != nullptr;
    const bool imp = sums && tail.imp_part != nullptr;
    const int block = tail.block > 0 ? tail.block : 1;
    int32_t c[SCAN_REG_TILES];
    int32_t sum = 0;
    float sl = 0.0f, si = 0.0f;
    if (e < n) {
        for (int tb = t0; tb < t1; tb += SCAN_REG_TILES) {
            float lp[SCAN_REG_TILES], ip[SCAN_REG_TILES];
#pragma unroll
            for (int q = 0; q < SCAN_REG_TILES; ++q) {
                const bool in = tb + q < t1;
                const size_t o = (size_t)(tb + q) * n + e;
                c[q] = in ? tile_counts[o] : 0;
                lp[q] = sums && in ? tail.load_part[o] : 0.0f;
                ip[q] = imp && in ? tail.imp_part[o] : 0.0f;
            }
#pragma unroll
            for (int q = 0; q < SCAN_REG_TILES; ++q) {
                sum += c[q];
                if (tb + q < t1) { sl += lp[q]; si += ip[q]; }
            }
        }
    }
    part[wid][lane] = sum;
    part_l[wid][lane] = sl;
    part_i[wid][lane] = si;
    if (sums)
        tile_sums_tree(part_l, part_i, n, (int)rank * 32, tail.load,
                       imp ? tail.importance : nullptr);
    else
        __syncthreads();
    int32_t run = 0;
    for (int w = 0; w < wid; ++w) run += part[w][lane];
    if (e < n) {
        if (span <= SCAN_REG_TILES) {
#pragma unroll
            for (int q = 0; q < SCAN_REG_TILES; ++q) {
                if (t0 + q < t1) {
                    tile_counts[(size_t)(t0 + q) * n + e] = run;
                    run += c[q];
                }
            }
        } else {
            for (int tb = t0; tb < t1; tb += 8) {
                int32_t cc[8];
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    cc[q] = tb + q < t1 ? tile_counts[(size_t)(tb + q) * n + e] : 0;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    if (tb + q < t1) tile_counts[(size_t)(tb + q) * n + e] = run;
                    run += cc[q];
                }
            }
        }
        if (wid == SCAN_WARPS - 1) totals[e] = run;
    }
    if (wid == SCAN_WARPS - 1) {
        const int32_t kr = e < n ? kept_rows(run, cap) : 0;
        ctot[lane] = kr;
        cblk[lane] = (kr + block - 1) / block;
    }
    tc::cluster_sync();                        // every CTA's counts published
    if (wid == 0) {
        const int32_t kr = ctot[lane], nbk = cblk[lane];
        int32_t before = 0, before_b = 0;      // the lower CTAs' experts
        for (int q = 0; q < (int)rank; ++q) {
            before += (int32_t)tc::ld_cluster_u32(tc::mapa(tc::smem_u32(&ctot[lane]), q));
            before_b += (int32_t)tc::ld_cluster_u32(tc::mapa(tc::smem_u32(&cblk[lane]), q));
        }
        int32_t incl = kr, incl_b = nbk;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int32_t v = __shfl_up_sync(0xffffffffu, incl, off);
            const int32_t vb = __shfl_up_sync(0xffffffffu, incl_b, off);
            if (lane >= off) { incl += v; incl_b += vb; }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            before += __shfl_xor_sync(0xffffffffu, before, off);
            before_b += __shfl_xor_sync(0xffffffffu, before_b, off);
        }
        const int32_t pos = before + incl - kr, pos_b = before_b + incl_b - nbk;
        if (e < n) {
            offsets[e] = pos;
            if (tail.blk != nullptr) {
                tail.blk[e] = pos_b;
                int4* units = static_cast<int4*>(tail.units);
                if (units != nullptr)            // (expert, first row, end row) of every unit
                    for (int32_t u = 0; u < nbk; ++u)
                        units[pos_b + u] = make_int4(e, pos + u * block, pos + kr, 0);
            }
        }
        if ((int)rank == ncta - 1 && lane == 31) {
            offsets[n] = before + incl;
            if (tail.blk != nullptr) tail.blk[n] = before_b + incl_b;
        }
    }
    if (sums) {
        const bool sw = tail.switch_scale > 0.0;
        const bool in = e < n;
        float vi = 0.0f, vl = 0.0f;
        if (wid == 0 && in) { vi = tail.importance[e]; vl = tail.load[e]; }   // written above
        if (wid == 0) {                        // the sums: warp rank of losses_512
            CSum a = {0.0f, 0.0f}, b = {0.0f, 0.0f};
            if (in) { a = cadd(a, sw ? vi * vl : vi); b = cadd(b, vl); }
            a = warp_csum(a);
            b = warp_csum(b);
            if (lane == 0) { cs[0] = a.s; cs[1] = a.c; cs[2] = b.s; cs[3] = b.c; }
        }
        tc::cluster_sync();
        if (rank == 0 && threadIdx.x == 0) {
            CSum a = {cs[0], cs[1]}, b = {cs[2], cs[3]};
            for (int q = 1; q < ncta; ++q) {
                const uint32_t base = tc::mapa(tc::smem_u32(&cs[0]), q);
                a = cmerge(a, {__uint_as_float(tc::ld_cluster_u32(base)),
                               __uint_as_float(tc::ld_cluster_u32(base + 4))});
                b = cmerge(b, {__uint_as_float(tc::ld_cluster_u32(base + 8)),
                               __uint_as_float(tc::ld_cluster_u32(base + 12))});
            }
            cmean[0] = a.s + a.c;              // the totals (Switch: the product sum)
            cmean[1] = b.s + b.c;
        }
        tc::cluster_sync();
        const float tot_i = __uint_as_float(tc::ld_cluster_u32(tc::mapa(tc::smem_u32(&cmean[0]), 0)));
        const float tot_l = __uint_as_float(tc::ld_cluster_u32(tc::mapa(tc::smem_u32(&cmean[1]), 0)));
        const float mean_i = tot_i / (float)n, mean_l = tot_l / (float)n;
        tc::cluster_sync();                    // the totals read before cs is reused
        if (!sw && wid == 0) {                 // the squared deviations
            CSum a = {0.0f, 0.0f}, b = {0.0f, 0.0f};
            if (in) {
                const float di = vi - mean_i, dl = vl - mean_l;
                a = cadd(a, di * di);
                b = cadd(b, dl * dl);
            }
            a = warp_csum(a);
            b = warp_csum(b);
            if (lane == 0) { cs[0] = a.s; cs[1] = a.c; cs[2] = b.s; cs[3] = b.c; }
        }
        tc::cluster_sync();
        if (rank == 0 && threadIdx.x == 0) {
            float c0, c1;
            if (sw) {
                c0 = (float)((double)tot_i * tail.switch_scale);
                c1 = 0.0f;
            } else {
                CSum a = {cs[0], cs[1]}, b = {cs[2], cs[3]};
                for (int q = 1; q < ncta; ++q) {
                    const uint32_t base = tc::mapa(tc::smem_u32(&cs[0]), q);
                    a = cmerge(a, {__uint_as_float(tc::ld_cluster_u32(base)),
                                   __uint_as_float(tc::ld_cluster_u32(base + 4))});
                    b = cmerge(b, {__uint_as_float(tc::ld_cluster_u32(base + 8)),
                                   __uint_as_float(tc::ld_cluster_u32(base + 12))});
                }
                const float qi = a.s + a.c, ql = b.s + b.c;
                c0 = (n <= 1 || mean_i == 0.0f) ? 0.0f : (qi / (float)n) / (mean_i * mean_i);
                c1 = (n <= 1 || mean_l == 0.0f) ? 0.0f : (ql / (float)n) / (mean_l * mean_l);
            }
            tail.losses[0] = c0;
            tail.losses[1] = c1;
            tail.losses[2] = weighted_losses(tail.w_imp, c0, tail.w_load, c1);
        }
    }
    tc::cluster_sync();                        // no CTA exits while its shared memory is read
}

// 4+5 in one launch: the stable scatter of one tile by its first warp, 256 rows at a
// time (rows taken 32 at a time in ascending r; lanes holding the same expert get
// consecutive slots in lane order, after everything the tile placed before them), each
// row's source token and destination
// recorded in shared memory; then all 16 warps copy those 256 input rows into
// x_perm (16 rows a warp, four rows and up to eight 16-byte vectors a lane in flight).
constexpr int SG_THREADS = 512;
constexpr int SG_BATCH = 256;

__global__ void __launch_bounds__(SG_THREADS)
dispatch_scatter_gather_kernel(const int32_t* __restrict__ idx, long long R, int n, int chunk,
                               int cap, const int32_t* __restrict__ tile_base,
                               const int32_t* __restrict__ offsets, int32_t* __restrict__ perm,
                               int32_t* __restrict__ inv, const uint4* __restrict__ x, int k,
                               int T, int row_vecs, uint4* __restrict__ out) {
    griddep_wait();
    griddep_launch_dependents();
    extern __shared__ int32_t next[];
    __shared__ int32_t s_src[SG_BATCH], s_dst[SG_BATCH];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int32_t* base = tile_base + (size_t)blockIdx.x * n;
    for (int e = threadIdx.x; e < n; e += SG_THREADS)
        next[e] = (cap > 0 ? 0 : offsets[e]) + base[e];   // position, or rank under a capacity
    __syncthreads();
    const long long r0 = (long long)blockIdx.x * chunk;
    const long long r1 = min(R, r0 + chunk);
    const unsigned lt = lanemask_lt();
    for (long long rb = r0; rb < r1; rb += SG_BATCH) {
        if (wid == 0) {
            constexpr int ROUNDS = SG_BATCH / 32;
            int ev[ROUNDS];
#pragma unroll
            for (int u = 0; u < ROUNDS; ++u) {
                const long long r = rb + u * 32 + lane;
                int e = -1;
                if (r < r1) {
                    e = idx[r];
                    if (e < 0 || e >= n) e = -1;   // reported by the count pass
                }
                ev[u] = e;
            }
#pragma unroll
            for (int u = 0; u < ROUNDS; ++u) {
                const long long r = rb + u * 32 + lane;
                const int e = ev[u];
                const unsigned peers = __match_any_sync(0xffffffffu, e);
                const int leader = __ffs(peers) - 1;
                int32_t slot = 0;
                if (e >= 0) slot = next[e];
                __syncwarp();
                if (e >= 0 && lane == leader) next[e] = slot + __popc(peers);
                __syncwarp();
                int32_t src = -1, dst = -1;
                if (e >= 0) {
                    int32_t p = slot + __popc(peers & lt);
                    if (cap > 0) p = p < cap ? __ldg(offsets + e) + p : -1;   // beyond capacity
                    if (p >= 0) perm[p] = (int32_t)r;
                    inv[r] = p;
                    if (p >= 0 && r / k < T) { src = (int32_t)(r / k); dst = p; }
                }
                s_src[u * 32 + lane] = src;
                s_dst[u * 32 + lane] = dst;
            }
        }
        __syncthreads();
        constexpr int ROWS_PER_WARP = SG_BATCH / (SG_THREADS / 32);
#pragma unroll 1
        for (int i0 = wid * ROWS_PER_WARP; i0 < (wid + 1) * ROWS_PER_WARP; i0 += 4) {
            int32_t src[4], dst[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) { src[q] = s_src[i0 + q]; dst[q] = s_dst[i0 + q]; }
            for (int v = lane; v < row_vecs; v += 64) {
                const bool two = v + 32 < row_vecs;
                uint4 b0[4], b1[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    if (src[q] >= 0) {
                        b0[q] = x[(size_t)src[q] * row_vecs + v];
                        if (two) b1[q] = x[(size_t)src[q] * row_vecs + v + 32];
                    }
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    if (src[q] >= 0) {
                        out[(size_t)dst[q] * row_vecs + v] = b0[q];
                        if (two) out[(size_t)dst[q] * row_vecs + v + 32] = b1[q];
                    }
                }
            }
        }
        __syncthreads();
    }
}

// The same stable scatter with the rows moved by the bulk-copy (TMA) engine through
// shared memory.  Two warps: warp 0 places the routed rows of a batch exactly as
// dispatch_scatter_gather_kernel does (perm, inv, and each row's source token and
// destination in shared memory); warp 1 copies each source token's input row once into
// a staging buffer (cp.async.bulk global -> shared, completion on an mbarrier) and then
// writes it to every destination of the batch (cp.async.bulk shared -> global, one
// per routed row).  A batch is 32 tokens' worth of rows (32 k); the staging buffers,
// the batch's rows and the placement are double-buffered, so batch b + 1's loads and
// placement overlap batch b's stores.  A tile's batches may be split over `parts` CTAs
// (consecutive runs of batches): part s starts each expert's slot after the tile's
// rows of parts 0 .. s-1, which it counts first (integer shared-memory adds, so the
// placement is the same as with one CTA a tile).
constexpr int BK_TOK = 32;                  // tokens a batch
constexpr int BK_MAX_ROWS = BK_TOK * 8;     // k <= 8
constexpr size_t BK_MAX_ROW_BYTES = 2048;   // two staging buffers of 33 rows: 132 KB

struct BulkShared {
    uint64_t full[2];
    int32_t src[2][BK_MAX_ROWS], dst[2][BK_MAX_ROWS];
    int abort_flag;
};

__global__ void __launch_bounds__(64)
dispatch_scatter_bulk_kernel(const int32_t* __restrict__ idx, long long R, int n, int chunk,
                             int parts, int cap, const int32_t* __restrict__ tile_base,
                             const int32_t* __restrict__ offsets, int32_t* __restrict__ perm,
                             int32_t* __restrict__ inv, const uint8_t* __restrict__ x, int k,
                             int T, int row_bytes, uint8_t* __restrict__ out, int* err) {
    extern __shared__ __align__(128) uint8_t dyn[];
    uint8_t* stage[2] = {dyn, dyn + (size_t)(BK_TOK + 1) * row_bytes};
    int32_t* next = reinterpret_cast<int32_t*>(dyn + (size_t)2 * (BK_TOK + 1) * row_bytes);
    __shared__ BulkShared sh;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        tc::mbar_init(&sh.full[0], 1);
        tc::mbar_init(&sh.full[1], 1);
        sh.abort_flag = 0;
        tc::fence_mbar_init();
    }
    griddep_wait();
    griddep_launch_dependents();
    const int tile = (int)blockIdx.x / parts, part = (int)blockIdx.x % parts;
    const int32_t* base = tile_base + (size_t)tile * n;
    for (int e = threadIdx.x; e < n; e += 64)
        next[e] = (cap > 0 ? 0 : offsets[e]) + base[e];   // position, or rank under a capacity
    const long long t0r = (long long)tile * chunk;
    const long long t1r = min(R, t0r + chunk);
    const int B = BK_TOK * k;                  // rows a batch, a multiple of 32
    const int nb_tile = (int)((t1r - t0r + B - 1) / B);
    const int per = (nb_tile + parts - 1) / parts;
    const long long r0 = min(t1r, t0r + (long long)part * per * B);
    const long long r1 = min(t1r, r0 + (long long)per * B);
    __syncthreads();
    for (long long r = t0r + threadIdx.x; r < r0; r += 64) {   // the earlier parts' rows
        const int e = idx[r];
        if (e >= 0 && e < n) atomicAdd(&next[e], 1);
    }
    __syncthreads();
    const int nb = (int)((r1 - r0 + B - 1) / B);
    // tokens [t_lo, t_hi] of batch i (the tokens of its rows, clipped to T)
    auto tok_lo = [&](int i) { return (int)((r0 + (long long)i * B) / k); };
    auto tok_hi = [&](int i) {
        const long long last = min(r1, r0 + (long long)(i + 1) * B) - 1;
        return (int)min((long long)T - 1, last / k);
    };
    volatile int* abort_flag = &sh.abort_flag;
    if (wid == 1) {
        auto issue_loads = [&](int i) {
            if (lane == 0) {
                const int lo = tok_lo(i), hi = tok_hi(i);
                uint64_t* bar = &sh.full[i & 1];
                tc::mbar_arrive_expect_tx(bar, (uint32_t)((hi - lo + 1) * row_bytes));
                for (int t = lo; t <= hi; ++t)
                    tc::bulk_load_1d(stage[i & 1] + (size_t)(t - lo) * row_bytes,
                                     x + (size_t)t * row_bytes, (uint32_t)row_bytes, bar);
            }
        };
        bool alive = true;
        // loads of batches [first_pending, last_issued] are in flight and not awaited
        int first_pending = 0, last_issued = -1;
        if (nb > 0) { issue_loads(0); last_issued = 0; }
        for (int i = 0; i < nb; ++i) {
            __syncthreads();                        // batch i placed by warp 0
            if (alive && i + 1 < nb) {
                // batch i + 1's buffer held batch i - 1, whose stores have read it: its
                // loads go out now, so their latency overlaps batch i's wait and stores
                tc::bulk_wait_read<0>();
                __syncwarp();
                issue_loads(i + 1);
                last_issued = i + 1;
            }
            int ok = 0;
            if (alive && lane == 0)
                ok = tc::mbar_wait(&sh.full[i & 1], (i >> 1) & 1, abort_flag, err) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (ok) {
                first_pending = i + 1;
                const int lo = tok_lo(i);
                const int rows = (int)min((long long)B, r1 - r0 - (long long)i * B);
                for (int q = lane; q < rows; q += 32) {
                    const int32_t src = sh.src[i & 1][q], dst = sh.dst[i & 1][q];
                    if (dst >= 0)
                        tc::bulk_store_1d(out + (size_t)dst * row_bytes,
                                          stage[i & 1] + (size_t)(src - lo) * row_bytes,
                                          (uint32_t)row_bytes);
                }
            } else {
                alive = false;                      // keep meeting warp 0's barriers only
            }
            tc::bulk_commit();
        }
        // loads left in flight by an abort complete before the CTA exits (bounded)
        if (lane == 0) {
            for (int j = first_pending; j <= last_issued; ++j) {
                const long long t0 = clock64();
                while (!tc::mbar_try_wait(&sh.full[j & 1], (j >> 1) & 1))
                    if (clock64() - t0 > tc::kWaitCycles) { raise_error(err, DEV_TIMEOUT); break; }
            }
        }
        tc::bulk_wait_all();                        // every row written before the CTA exits
    } else {
        const unsigned lt = lanemask_lt();
        // batch i's expert ids in registers (B / 32 <= 8 a lane), batch i + 1's loads
        // issued before batch i is placed, so no placement step waits on a global load
        constexpr int MAXQ = BK_MAX_ROWS / 32;
        auto load_ids = [&](int i, int (&ids)[MAXQ]) {
            const long long rb = r0 + (long long)i * B;
            const long long re = min(r1, rb + B);
#pragma unroll
            for (int q = 0; q < MAXQ; ++q) {
                const long long r = rb + 32 * q + lane;
                ids[q] = (32 * q < B && r < re) ? idx[r] : -1;
            }
        };
        int cur[MAXQ], nxt[MAXQ];
        if (nb > 0) load_ids(0, cur);
        for (int i = 0; i < nb; ++i) {
            const long long rb = r0 + (long long)i * B;
            const long long re = min(r1, rb + B);
            if (i + 1 < nb) load_ids(i + 1, nxt);
#pragma unroll
            for (int q = 0; q < MAXQ; ++q) {
                const int u = 32 * q;
                if (u >= B) break;
                const long long r = rb + u + lane;
                int e = -1;
                if (r < re) {
                    e = cur[q];
                    if (e < 0 || e >= n) e = -1;   // reported by the count pass
                }
                const unsigned peers = __match_any_sync(0xffffffffu, e);
                const int leader = __ffs(peers) - 1;
                int32_t slot = 0;
                if (e >= 0) slot = next[e];
                __syncwarp();
                if (e >= 0 && lane == leader) next[e] = slot + __popc(peers);
                __syncwarp();
                int32_t src = -1, dst = -1;
                if (e >= 0) {
                    int32_t p = slot + __popc(peers & lt);
                    if (cap > 0) p = p < cap ? __ldg(offsets + e) + p : -1;   // beyond capacity
                    if (p >= 0) perm[p] = (int32_t)r;
                    inv[r] = p;
                    if (p >= 0 && r / k < T) { src = (int32_t)(r / k); dst = p; }
                }
                sh.src[i & 1][u + lane] = src;
                sh.dst[i & 1][u + lane] = dst;
            }
#pragma unroll
            for (int q = 0; q < MAXQ; ++q) cur[q] = nxt[q];
            __syncthreads();                        // batch i placed
        }
    }
}

__global__ void __launch_bounds__(1024)
row_block_prefix_kernel(const int32_t* __restrict__ offsets, int n, int block,
                        int32_t* __restrict__ out, int4* __restrict__ units) {
    griddep_wait();
    griddep_launch_dependents();
    block_prefix_body(offsets, n, block, out, units);
}

}  // namespace

cudaError_t launch_row_block_prefix(const int32_t* offsets, int n, int block, int32_t* out,
                                    cudaStream_t s, void* units) {
    const cudaError_t e = launch_pdl(row_block_prefix_kernel, dim3(1), dim3(1024), 0, s, 1, offsets,
                                     n, block, out, static_cast<int4*>(units));
    note_launch();
    return e;
}

DispatchPlan dispatch_plan(long long R) {
    DispatchPlan p;
    long long tiles = (R + 1023) / 1024;
    if (tiles < 1) tiles = 1;
    if (tiles > 256) tiles = 256;
    long long chunk = (R + tiles - 1) / tiles;
    chunk = (chunk + 31) / 32 * 32;
    if (chunk < 32) chunk = 32;
    p.chunk = (int)chunk;
    p.tiles = (int)((R + chunk - 1) / chunk);
    if (p.tiles < 1) p.tiles = 1;
    return p;
}

namespace {

// The stable scatter with the row copy into x_perm.
cudaError_t launch_scatter_stage(const int32_t* idx, long long R, int n, int tiles, int chunk,
                                 int cap, const int32_t* tile_base, const int32_t* offsets,
                                 int32_t* perm, int32_t* inv, const void* x, int k, int T,
                                 size_t row_bytes, void* x_perm, int* err, cudaStream_t s) {
    const size_t hist_bytes = (size_t)n * sizeof(int32_t);
    if (x == nullptr || x_perm == nullptr) return cudaErrorInvalidValue;
    if (row_bytes <= BK_MAX_ROW_BYTES && k <= 8) {
        const size_t smem = 2 * (BK_TOK + 1) * row_bytes + hist_bytes;
        cudaError_t e = cudaFuncSetAttribute(dispatch_scatter_bulk_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
        // fewer tiles than SMs: a tile's batches split over `parts` CTAs, about two an SM
        // (measured at 128 tiles: 45.9 -> 39.4 us for the dispatch stage; at 256 tiles
        // on 148 SMs the split was slower, 57.3 -> 61.4 us, so it stays one CTA a tile)
        const int sms = gate_sm_count();
        const int batches = (int)((chunk + (long long)BK_TOK * k - 1) / ((long long)BK_TOK * k));
        int parts = tiles >= sms ? 1 : (2 * sms + tiles - 1) / tiles;
        parts = parts < 1 ? 1 : (parts > batches ? batches : parts);
        e = launch_pdl(dispatch_scatter_bulk_kernel, dim3(tiles * parts), dim3(64), smem, s, 1, idx,
                       R, n, chunk, parts, cap, tile_base, offsets, perm, inv,
                       static_cast<const uint8_t*>(x), k, T, (int)row_bytes,
                       static_cast<uint8_t*>(x_perm), err);
        note_launch();
        return e;
    }
    if (hist_bytes > 40 * 1024)
        cudaFuncSetAttribute(dispatch_scatter_gather_kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)hist_bytes);
    const cudaError_t e =
        launch_pdl(dispatch_scatter_gather_kernel, dim3(tiles), dim3(SG_THREADS), hist_bytes, s, 1,
                   idx, R, n, chunk, cap, tile_base, offsets, perm, inv,
                   static_cast<const uint4*>(x), k, T, (int)(row_bytes / 16),
                   static_cast<uint4*>(x_perm));
    note_launch();
    return e;
}

}  // namespace

// tile_counts needs tiles*n + n int32 (the last n hold the per-expert totals).
cudaError_t launch_dispatch(const int32_t* idx, int T, int k, int n, int32_t* tile_counts,
                            int32_t* offsets, int32_t* perm, int32_t* inv, int* err,
                            cudaStream_t s, const void* x, size_t row_bytes, void* x_perm,
                            int cap) {
    const long long R = (long long)T * k;
    const DispatchPlan p = dispatch_plan(R);
    int32_t* totals = tile_counts + (size_t)p.tiles * n;
    const size_t hist_bytes = (size_t)n * sizeof(int32_t);
    if (hist_bytes > 48 * 1024)
        cudaFuncSetAttribute(dispatch_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)hist_bytes);
    cudaError_t e = launch_pdl(dispatch_count_kernel, dim3(p.tiles), dim3(256), hist_bytes, s, 1,
                               idx, R, n, p.chunk, tile_counts, err);
    note_launch();
    if (e != cudaSuccess) return e;
    e = launch_pdl(dispatch_column_scan_kernel, dim3((n + 7) / 8), dim3(256), 0, s, 1, tile_counts,
                   p.tiles, n, totals);
    note_launch();
    if (e != cudaSuccess) return e;
    e = launch_pdl(dispatch_offsets_kernel, dim3(1), dim3(1024), 0, s, 1,
                   static_cast<const int32_t*>(totals), n, cap, offsets);
    note_launch();
    if (e != cudaSuccess) return e;
    return launch_scatter_stage(idx, R, n, p.tiles, p.chunk, cap, tile_counts, offsets, perm, inv,
                                x, k, T, row_bytes, x_perm, err, s);
}

cudaError_t launch_dispatch_counted(const int32_t* idx, long long R, int n, int tiles, int chunk,
                                    int32_t* tile_counts, int32_t* offsets, int32_t* perm,
                                    int32_t* inv, cudaStream_t s, const void* x, int k, int T,
                                    size_t row_bytes, void* x_perm, int cap, int* err,
                                    const DispatchTail* tail) {
    int32_t* totals = tile_counts + (size_t)tiles * n;
    const DispatchTail none{};
    const int ctas = (n + 31) / 32;
    if (ctas > SCAN_CLUSTER_MAX) return cudaErrorInvalidValue;
    // one cluster meeting in distributed shared memory (measured on one B300: the dispatch
    // stage, scan and scatter, 60.5 -> 57.5 us at 256 experts and 39.8 -> 34.2 us at 32
    // against a scan whose last CTA, found by a ticket, read the totals back from memory)
    cudaError_t e = launch_pdl(dispatch_scan_cluster_kernel, dim3(ctas), dim3(SCAN_THREADS), 0,
                               s, ctas, tile_counts, tiles, n, cap, totals, offsets,
                               tail != nullptr ? *tail : none);
    note_launch();
    if (e != cudaSuccess) return e;
    return launch_scatter_stage(idx, R, n, tiles, chunk, cap, tile_counts, offsets, perm, inv, x,
                                k, T, row_bytes, x_perm, err, s);
}


}  // namespace moe
