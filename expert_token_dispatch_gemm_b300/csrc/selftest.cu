// Check of the device-side failure path: one warp waits, with the same bounded mbarrier
// wait every tensor-core kernel uses, on a barrier that nothing arrives at. After the
// wait limit (about 2 s) the wait gives up, records MOE_DEV_TIMEOUT in the status word
// and the kernel returns normally, so the context stays usable and the host reads the
// status. No fault, trap or unbounded loop is involved.
#include "sm100.cuh"

namespace moe {
namespace {

__global__ void __launch_bounds__(32) wait_timeout_kernel(int32_t *status) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        tc::mbar_init(&bar, 1);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    if (threadIdx.x == 0) {
        volatile int *abort_s = &abort_flag;
        tc::mbar_wait(&bar, 0, abort_s, status);   // phase 0 never completes
    }
}

}  // namespace

cudaError_t launch_wait_timeout_check(int32_t *status, cudaStream_t s) {
    wait_timeout_kernel<<<1, 32, 0, s>>>(status);
    return cudaGetLastError();
}

}  // namespace moe
