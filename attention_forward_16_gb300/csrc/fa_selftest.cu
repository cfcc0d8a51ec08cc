// Watchdog self-test: one thread waits on an mbarrier that nothing ever
// arrives at, bounded by a time limit, then records a timeout in the device
// status word -- the same bounded-wait-and-report path the attention kernels
// take, exercised without touching them.
#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

__global__ void selftest_wait_kernel(int* status, unsigned long long limit_ns) {
    __shared__ uint64_t bar;
    const uint32_t b = ptx::smem_u32(&bar);
    if (threadIdx.x == 0) {
        ptx::mbar_init(b, 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint64_t t0 = ptx::globaltimer_ns();
        while (!ptx::mbar_try_wait(b, 0)) {
            if (ptx::globaltimer_ns() - t0 > limit_ns) {
                atomicExch(status, DEV_TIMEOUT);
                break;
            }
        }
    }
}

}  // namespace

cudaError_t launch_selftest_timeout(int* status, unsigned long long limit_ns, cudaStream_t s) {
    selftest_wait_kernel<<<1, 32, 0, s>>>(status, limit_ns);
    return cudaGetLastError();
}

}  // namespace fa
