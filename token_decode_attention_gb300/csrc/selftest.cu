// selftest.cu -- self-test of the library's failure detection.
//
// Every pipeline wait in the library's kernels is bounded: after
// kWaitLimitNs of global time it gives up, records a code in the device error
// word and lets the kernel return, so the CUDA context stays usable and the
// host learns of it through dattn_device_error().  This kernel exercises that
// path on purpose and without any fault: one CTA waits, through the same
// bounded-wait primitive the decode kernel uses, on an mbarrier that nothing
// ever arrives on.
#include <cuda_runtime.h>

#include "dattn_internal.h"
#include "ptx.cuh"

namespace dattn {
namespace {

__global__ void wait_timeout_selftest_kernel(unsigned *err) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);  // expects one arrival; none will come
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !mbar_wait_bounded(&bar, 0, kWaitLimitNs)) atomicOr(err, kErrSelftestWait);
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(unsigned *err, cudaStream_t stream) {
    void *args[] = {&err};
    return cudaLaunchKernel(reinterpret_cast<const void *>(wait_timeout_selftest_kernel), dim3(1),
                            dim3(32), args, 0, stream);
}

}  // namespace dattn
