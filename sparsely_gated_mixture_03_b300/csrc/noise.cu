// The noise of the noisy top-k gate drawn on the device.
//
// "Mixture of Experts: Outrageously Large Neural Networks" (intuitivepapers.ai),
// "Noisy top-k gating", eq (4): H = x W_g + StandardNormal() * Softplus(x W_noise): one
// standard normal draw per (token, expert).  With MOE_FLAG_DEVICE_NOISE the layer draws
// them itself instead of reading a caller's eps, so a batch's noise never crosses the
// host link.  The draws are counter-based (element i of the call, a 64-bit seed), so
// any element can be reproduced on its own; elements 2j and 2j + 1 are the two normals
// of one Box-Muller pair j:
//   z  = seed + (j + 1) * 0x9E3779B97F4A7C15 (mod 2^64), then the SplitMix64 finaliser
//        (Steele, Lea and Flood, "Fast splittable pseudorandom number generators",
//        OOPSLA 2014): z ^= z >> 30; z *= 0xBF58476D1CE4E5B9; z ^= z >> 27;
//        z *= 0x94D049BB133111EB; z ^= z >> 31;
//   u1 = (top 24 bits of z + 1) / 2^24 in (0, 1],  u2 = (low 24 bits of z) / 2^24 in [0, 1);
//   eps[2j] = r cos(2 pi u2), eps[2j+1] = r sin(2 pi u2), r = sqrt(-2 ln u1)
//   (Box and Muller, 1958; |eps| <= 5.77).
#include <stdint.h>

#include "common.cuh"
#include "launch.h"

namespace moe {
namespace {

// The Box-Muller pair j: (eps[2j], eps[2j+1]).
__device__ __forceinline__ float2 draw_pair(uint64_t seed, uint64_t j) {
    uint64_t z = seed + (j + 1ull) * 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    z ^= z >> 31;
    const float u1 = (float)((z >> 40) + 1ull) * 5.9604644775390625e-8f;   // 2^-24
    const float u2 = (float)(z & 0xFFFFFFull) * 5.9604644775390625e-8f;
    const float r = sqrtf(-2.0f * logf(u1));
    float sn, cs;
    sincospif(2.0f * u2, &sn, &cs);
    return make_float2(r * cs, r * sn);
}

// Two pairs (four consecutive elements, one 16-byte store) a thread, grid-stride.
// WAIT = false (the layer's own draw into its workspace, the first kernel of a call):
// the kernel reads nothing and writes only the workspace's noise region, so it does not
// wait for the previous kernel on the stream and runs beside its tail.  That is safe
// because every kernel of this library lets its successor start only after its own
// wait, i.e. once every earlier kernel has finished, and the only kernels that read the
// noise region (the gate's) are never the last kernel of a call.  moe_draw_noise writes
// a caller's buffer, which the previous kernel may still read: WAIT = true.
template <bool WAIT>
__global__ void __launch_bounds__(256)
noise_kernel(uint64_t seed, long long count, float* __restrict__ eps) {
    if (WAIT) griddep_wait();
    griddep_launch_dependents();
    const long long stride = (long long)gridDim.x * blockDim.x * 4;
    for (long long i = ((long long)blockIdx.x * blockDim.x + threadIdx.x) * 4; i < count;
         i += stride) {
        const float2 a = draw_pair(seed, (uint64_t)i >> 1);
        const float2 b = draw_pair(seed, ((uint64_t)i >> 1) + 1);
        if (i + 4 <= count) {
            *reinterpret_cast<float4*>(eps + i) = make_float4(a.x, a.y, b.x, b.y);
        } else {
            const float v[4] = {a.x, a.y, b.x, b.y};
            for (long long j = i; j < count; ++j) eps[j] = v[j - i];
        }
    }
}

}  // namespace

cudaError_t launch_noise(unsigned long long seed, long long count, float* eps, cudaStream_t s,
                         bool wait) {
    if (count <= 0) return cudaSuccess;
    long long blocks = (count + 1023) / 1024;
    const long long cap = (long long)gate_sm_count() * 8;
    if (blocks > cap) blocks = cap;
    const cudaError_t e =
        wait ? launch_pdl(noise_kernel<true>, dim3((unsigned)blocks), dim3(256), 0, s, 1,
                          (uint64_t)seed, count, eps)
             : launch_pdl(noise_kernel<false>, dim3((unsigned)blocks), dim3(256), 0, s, 1,
                          (uint64_t)seed, count, eps);
    note_launch();
    return e;
}

}  // namespace moe
