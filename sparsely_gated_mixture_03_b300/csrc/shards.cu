// Sharding the layer over several GPUs ("Mixture of Experts: Outrageously Large Neural
// Networks" (intuitivepapers.ai), section "Keeping each expert's batch large": standard
// layers and the gate replicated data-parallel, the experts spread over the devices,
// and every routed row sent to the device that holds its expert).
//
// ep_plan_host: the exchange plan of one rank, host-only integer work on every rank's
// dispatch offsets.  ep_regroup_kernel: the row permutation between the order rows
// arrive in (source rank major) and the order the grouped expert FFN reads (local
// expert major), in either direction.
#include <stdint.h>

#include "common.cuh"
#include "launch.h"

namespace moe {
namespace {

// One warp per row of the expert-major order: a binary search over the block starts
// finds its (expert, source) block; the row moves with 16-byte vector copies.
__global__ void __launch_bounds__(256)
ep_regroup_kernel(const int32_t* __restrict__ plan, int blocks, const uint4* __restrict__ in,
                  uint4* __restrict__ out, int row_vecs, int to_expert_major) {
    griddep_wait();
    griddep_launch_dependents();
    const int32_t* src_start = plan;             // [blocks] source-major start of block q
    const int32_t* dst_start = plan + blocks;    // [blocks + 1] expert-major starts, then total
    const int total = __ldg(dst_start + blocks);
    const int lane = threadIdx.x & 31;
    const int warps = gridDim.x * (blockDim.x >> 5);
    for (int p = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); p < total; p += warps) {
        int lo = 0, hi = blocks - 1;             // the last block q with dst_start[q] <= p
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (__ldg(dst_start + mid) <= p) lo = mid; else hi = mid - 1;
        }
        const int s = __ldg(src_start + lo) + (p - __ldg(dst_start + lo));
        const uint4* a = in + (size_t)(to_expert_major ? s : p) * row_vecs;
        uint4* b = out + (size_t)(to_expert_major ? p : s) * row_vecs;
        for (int v = lane; v < row_vecs; v += 32) b[v] = a[v];
    }
}

}  // namespace

int ep_plan_host(int world, int rank, int n, const int32_t* offs, int32_t* send_rows,
                 int32_t* recv_rows, int32_t* plan) {
    const int nl = n / world;
    for (int s = 0; s < world; ++s) {
        const int32_t* o = offs + (size_t)s * (n + 1);
        if (o[0] != 0) return 1;
        for (int e = 0; e < n; ++e)
            if (o[e + 1] < o[e]) return 1;
    }
    auto cnt = [&](int s, int g) -> long long {
        const int32_t* o = offs + (size_t)s * (n + 1);
        return (long long)o[g + 1] - o[g];
    };
    const int32_t* mine = offs + (size_t)rank * (n + 1);
    for (int r = 0; r < world; ++r) send_rows[r] = mine[(r + 1) * nl] - mine[r * nl];
    long long total = 0;
    for (int s = 0; s < world; ++s) {
        const int32_t* o = offs + (size_t)s * (n + 1);
        recv_rows[s] = o[(rank + 1) * nl] - o[rank * nl];
        total += recv_rows[s];
    }
    if (total >= (1LL << 31)) return 2;
    const int blocks = world * nl;
    int32_t* src_start = plan;
    int32_t* dst_start = plan + blocks;
    int32_t* local_offsets = plan + 2 * blocks + 1;
    long long a = 0;                              // arrival order: source, then its experts
    for (int s = 0; s < world; ++s)
        for (int e = 0; e < nl; ++e) {
            src_start[e * world + s] = (int32_t)a;
            a += cnt(s, rank * nl + e);
        }
    long long b = 0;                              // FFN order: expert, then the sources
    for (int e = 0; e < nl; ++e) {
        local_offsets[e] = (int32_t)b;
        for (int s = 0; s < world; ++s) {
            dst_start[e * world + s] = (int32_t)b;
            b += cnt(s, rank * nl + e);
        }
    }
    dst_start[blocks] = (int32_t)b;
    local_offsets[nl] = (int32_t)b;
    return 0;
}

cudaError_t launch_ep_regroup(int world, int n_local, const int32_t* plan, const void* in,
                              void* out, size_t row_bytes, int to_expert_major, int sms,
                              cudaStream_t s) {
    const cudaError_t e = launch_pdl(ep_regroup_kernel, dim3(sms * 8), dim3(256), 0, s, 1, plan,
                                     world * n_local, static_cast<const uint4*>(in),
                                     static_cast<uint4*>(out), (int)(row_bytes / 16),
                                     to_expert_major);
    note_launch();
    return e;
}

}  // namespace moe
