// Self-test of the failure-detection path that every tensor-core kernel here
// uses: a bounded mbarrier wait that gives up, records a site code in a device
// error word and returns, leaving the context usable.  One CTA waits on a
// barrier phase that nothing completes, with a caller-chosen limit; a second
// wait, on a phase that does complete, must succeed.  Nothing faults, traps
// or hangs: the wait ends by itself after the limit.
#include "tc_common.cuh"

namespace dsa {

__device__ int g_selftest_error = 0;

namespace {

constexpr int SELFTEST_SITE = 90;

__global__ void bounded_wait_selftest_kernel(long long limit_cycles, int *completed_ok) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x != 0) return;
    tc::mbar_init(&bar, 1);
    abort_flag = 0;
    tc::fence_mbar_init();
    // phase 0 has one pending arrival that never comes: the wait runs out and reports
    const bool gave_up = !tc::mbar_wait(&bar, 0, (volatile int *)&abort_flag, &g_selftest_error, SELFTEST_SITE,
                                        limit_cycles);
    // the same barrier, completed this time: the wait must succeed (the abort flag is cleared first)
    abort_flag = 0;
    tc::mbar_arrive(&bar);
    const bool completed = tc::mbar_wait(&bar, 0, (volatile int *)&abort_flag, &g_selftest_error, SELFTEST_SITE + 1,
                                         limit_cycles);
    if (completed_ok) *completed_ok = (gave_up && completed) ? 1 : 0;
}

}  // namespace

cudaError_t launch_bounded_wait_selftest(long long limit_cycles, int *completed_ok, cudaStream_t s) {
    bounded_wait_selftest_kernel<<<1, 32, 0, s>>>(limit_cycles, completed_ok);
    note_launch(DSA_KERNEL_SELFTEST);
    return cudaGetLastError();
}

int selftest_read_error(int *site) {
    int v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_selftest_error, sizeof(int));
    if (e != cudaSuccess) return fail_cuda(e);
    if (v) {
        e = cudaMemcpyToSymbol(g_selftest_error, &zero, sizeof(int));
        if (e != cudaSuccess) return fail_cuda(e);
        if (site) *site = v;
        return DSA_ERR_TIMEOUT;
    }
    return DSA_OK;
}

}  // namespace dsa
