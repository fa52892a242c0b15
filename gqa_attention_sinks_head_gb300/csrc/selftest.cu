// selftest.cu -- a check of the failure path that every kernel's pipeline
// waits share: a wait that nothing will complete must give up after its limit,
// set SA_DEVICE_TIMEOUT in the device status word and let the kernel return,
// leaving the context usable.  No fault, trap or unbounded spin is involved.
#include "sa_internal.h"
#include "sa_ptx.cuh"

namespace sa {
namespace {

__global__ void wait_timeout_kernel(uint32_t *status)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);  // one arrival expected; none will come
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && mbar_wait(&bar, 0, status))
        atomicOr(status, 0x80000000u);  // completed: must not happen (reported as a failure)
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(uint32_t *status, cudaStream_t stream)
{
    wait_timeout_kernel<<<2, 32, 0, stream>>>(status);
    return cudaGetLastError();
}

}  // namespace sa
