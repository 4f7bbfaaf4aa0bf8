// Failure-path self-test.  Every pipeline in this library waits on mbarriers
// through mbar_wait, which gives up after about a second and lets the caller
// record kPipelineFailureBit in err_count and unwind, so that a defect is
// reported instead of hanging the GPU.  This kernel exercises exactly that
// path: one thread waits on a barrier that nothing arrives on, the wait runs
// out, the bit is recorded, and the kernel exits normally.
#include "common.cuh"
#include "internal.h"

namespace nvattn {

__global__ void wait_timeout_selftest_kernel(int *err_count) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbarrier_init();
    }
    __syncthreads();
    // Phase 0 of a fresh barrier with one expected arrival: it never completes.
    if (threadIdx.x == 0 && !mbar_wait(&bar, 0)) flag_pipeline_failure(err_count);
}

cudaError_t launch_wait_timeout_selftest(int *err_count, cudaStream_t s) {
    wait_timeout_selftest_kernel<<<1, 32, 0, s>>>(err_count);
    return cudaGetLastError();
}

}  // namespace nvattn
