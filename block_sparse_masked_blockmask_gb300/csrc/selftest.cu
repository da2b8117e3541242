// Check of the failure path: one CTA waits on an mbarrier that no thread ever
// arrives at, with the same bounded wait the attention kernel uses but a short
// limit.  The wait gives up, the kernel records the timeout in the device
// status word and returns normally, so the context stays usable.  Nothing
// here faults, traps or hangs the GPU.
#include "flex_internal.h"
#include "ptx.cuh"

namespace flex {
namespace {

__global__ void wait_timeout_kernel(int *status, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    // phase 0 of `bar` never completes: nobody arrives
    const bool ok = mbar_wait(&bar, 0, &abort_flag, limit_ns);
    if (!ok && threadIdx.x == 0) atomicCAS(status, 0, kDeviceTimeout);
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(int *status, uint64_t limit_ns, cudaStream_t stream) {
    wait_timeout_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
    return cudaGetLastError();
}

}  // namespace flex
