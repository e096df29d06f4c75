// Failure-detection self-test: the bounded-wait path of the kernels, exercised
// without faulting or hanging the GPU.
//
// One CTA: thread 0 waits for a phase of an mbarrier that nothing ever completes,
// with a small cycle budget; the wait gives up, records DEV_TIMEOUT in the device
// error word and sets the CTA's abort flag.  Thread 32 waits on a second barrier that
// nothing completes either, with the full budget of the real kernels; it sees the
// abort flag and returns, as the other roles of a kernel do when one role gives up.
// Both reach the final barrier and the CTA exits normally, so the context stays usable.
#include <stdint.h>

#include "common.cuh"
#include "launch.h"
#include "tc.cuh"

namespace moe {
namespace {

__global__ void timeout_probe_kernel(long long budget, int* err) {
    __shared__ uint64_t bar[2];
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        tc::mbar_init(&bar[0], 1);
        tc::mbar_init(&bar[1], 1);
        abort_flag = 0;
        tc::fence_mbar_init();
    }
    __syncthreads();
    volatile int* abort = &abort_flag;
    if (threadIdx.x == 0) tc::mbar_wait(&bar[0], 0, abort, err, budget);
    if (threadIdx.x == 32) tc::mbar_wait(&bar[1], 0, abort, err);
    __syncthreads();
}

}  // namespace

cudaError_t launch_timeout_probe(long long budget_cycles, int* err, cudaStream_t s) {
    timeout_probe_kernel<<<1, 64, 0, s>>>(budget_cycles, err);
    note_launch();
    return cudaGetLastError();
}

}  // namespace moe
