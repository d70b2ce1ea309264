// kda_selftest.cu -- failure-detection self-test of the bounded waits in the tensor-core kernels.
//
// Every mbarrier wait in the prefill's tensor-core kernels gives up after a fixed number of polls,
// records device error 3 (timeout), lets the tensor core finish the work it was given (commit to
// a spare mbarrier, bounded wait), frees its TMEM and returns, so that the context stays usable
// and the host learns of it through kda_check_device_errors.  This kernel runs that exact
// sequence with a wait that cannot succeed: one warp allocates TMEM, waits on an mbarrier that
// nothing arrives on, records the timeout, drains, frees and exits.  No fault, trap or unbounded
// loop is involved.

#include "kda_internal.cuh"
#include "kda_tc.cuh"

namespace kda {

__device__ int32_t g_selftest_error = 0;

namespace {

__global__ void __launch_bounds__(32, 1) wait_timeout_selftest_kernel(uint32_t polls, int32_t* result)
{
    __shared__ __align__(8) uint64_t bar[2];
    __shared__ uint32_t s_tmem;
    const int lane = threadIdx.x;
    tc::tmem_alloc(&s_tmem, 32);        // warp-wide
    tc::tmem_relinquish();
    if (lane == 0) {
        tc::mbar_init(bar, 1);          // the wait that cannot complete: nothing arrives on it
        tc::mbar_init(bar + 1, 1);      // the drain
        tc::fence_mbar_init();
    }
    tc::tc_fence_before();
    __syncwarp();
    tc::tc_fence_after();
    const uint32_t tmem = s_tmem;
    if (lane == 0) {
        const bool done = tc::mbar_wait(bar, 0, polls);
        bool drained = true;
        if (!done) {
            atomicCAS(&g_selftest_error, 0, (int32_t)kDevErrTimeout);
            tc::mma_commit(bar + 1);    // arrives once this thread's tensor-core work (none) is done
            drained = tc::mbar_wait(bar + 1, 0, polls);
        }
        if (result) {
            result[0] = done ? 1 : 0;
            result[1] = drained ? 1 : 0;
        }
    }
    tc::tc_fence_before();
    __syncwarp();
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 32);
}

}  // namespace

cudaError_t launch_wait_selftest(uint32_t polls, int32_t* result, cudaStream_t stream)
{
    wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(polls, result);
    return cudaGetLastError();
}

cudaError_t selftest_read_and_clear_error(int32_t* code)
{
    int32_t zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(code, g_selftest_error, sizeof(int32_t));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_selftest_error, &zero, sizeof(int32_t));
}

}  // namespace kda
