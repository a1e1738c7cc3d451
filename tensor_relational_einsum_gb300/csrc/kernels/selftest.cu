// selftest.cu -- a wait that nothing ends, to show that the bounded
// mbarrier wait the tcgen05 kernels use gives up, raises the device error
// word and returns, leaving the context usable (failure detection without a
// GPU fault: no trap, no bad address, no endless loop).
#include "../ea_internal.h"
#include "tc_common.cuh"

namespace ea {

namespace {

__global__ void wait_timeout_kernel(int *err, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        tc::mbar_init(&bar, 1);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // phase 0 of `bar` never completes: no thread arrives on it
    if (threadIdx.x == 0) (void)tc::mbar_wait(&bar, 0, &abort_flag, err, kDevTimeoutSelftest, limit_ns);
    __syncthreads();
}

}  // namespace

cudaError_t launch_wait_timeout(int *err, uint64_t limit_ns, cudaStream_t st) {
    wait_timeout_kernel<<<1, 32, 0, st>>>(err, limit_ns);
    return cudaGetLastError();
}

}  // namespace ea
