// selftest.cu -- failure-detection self-test of the bounded device waits.
//
// One CTA of one warp initialises an mbarrier that nothing will ever complete
// and waits on it with the given limit through the same wait helpers the main
// kernel uses.  The wait runs out, records kErrTimeout in the error word and
// the kernel returns: the host sees FA_ERR_TIMEOUT from fa_check_device and the
// CUDA context stays usable.  No fault, trap or unbounded loop is involved.
#include "bounded_wait.cuh"
#include "fa_internal.cuh"

namespace fa {
namespace {

__global__ void __launch_bounds__(32) wait_selftest_kernel(unsigned int* err, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t never;
    __shared__ int abort_flag;
    const uint32_t bar = ptx::smem_u32(&never);
    if (threadIdx.x == 0) {
        abort_flag = 0;
        ptx::mbar_init(bar, 1);  // count 1, and nobody arrives
        ptx::fence_mbar_init();
    }
    __syncwarp();
    wait_bar_warp(bar, 0, &abort_flag, err, limit_ns);
}

}  // namespace

cudaError_t launch_wait_selftest(unsigned int* err, uint64_t limit_ns, cudaStream_t st) {
    wait_selftest_kernel<<<1, 32, 0, st>>>(err, limit_ns);
    return cudaGetLastError();
}

}  // namespace fa
