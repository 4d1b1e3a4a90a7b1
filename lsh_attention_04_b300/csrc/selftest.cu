// selftest.cu -- exercises the bounded wait that every tensor-core kernel relies on.
//
// One warp waits, through the same sm100::wait as the kernels, on an mbarrier that
// nothing ever arrives on.  After the wait limit (1 s) the wait records its code in the
// workspace status block, raises the CTA's abort flag and returns false, and the kernel
// ends: no trap, no fault, no hang, and the context stays usable.  Tests use it to check
// that a stuck pipeline reports LSH_ERR_DEVICE_CHECK instead of hanging the GPU.
#include "sm100.cuh"

namespace lsh {
namespace {

using namespace sm100;

__global__ void __launch_bounds__(32, 1) selftest_wait_kernel(StatusBlock *status)
{
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();
    volatile int *ab = &abort_flag;
    // phase 0 never completes: the wait gives up after its limit and reports
    wait(&bar, 0, ab, status, kSelftestWaitCode);
}

}  // namespace

cudaError_t selftest_wait_launch(StatusBlock *status, cudaStream_t st)
{
    selftest_wait_kernel<<<1, 32, 0, st>>>(status);
    return cudaGetLastError();
}

}  // namespace lsh
