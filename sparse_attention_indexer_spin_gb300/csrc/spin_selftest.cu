// spin_selftest.cu -- self-test of the bounded wait every pipelined kernel of the library uses.
//
// The score kernels stage data through shared-memory rings whose stages are handed between
// warps by mbarriers.  Every such wait is bounded: after a limit of GPU global time (or when
// another warp has raised the kernel's abort flag) it gives up, and the kernel reports
// SPIN_STATUS_TIMEOUT, drains its own copies and returns instead of spinning forever.  This
// kernel runs that same wait on a barrier whose arrival is controlled by the test: nobody
// arrives (the limit must end the wait), the abort flag is raised first (the wait must end
// at once), or a second warp arrives (the wait must succeed).
#include "spin_common.cuh"
#include "spin_internal.h"

namespace spin {

__global__ void __launch_bounds__(64) wait_selftest_kernel(int mode, uint64_t limit_ns, uint32_t* status,
                                                           unsigned long long* elapsed_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = mode == 1 ? 1 : 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (mode == 2 && threadIdx.x == 32) mbar_arrive(&bar);  // the positive control
    if (threadIdx.x == 0) {
        const uint64_t t0 = global_ns();
        const bool ok = mbar_wait(&bar, 0u, &abort_flag, limit_ns);
        *elapsed_ns = (unsigned long long)(global_ns() - t0);
        if (!ok) set_status(status, SPIN_STATUS_TIMEOUT);
    }
}

cudaError_t launch_wait_selftest(int mode, uint64_t limit_ns, uint32_t* status, unsigned long long* elapsed_ns,
                                 cudaStream_t s) {
    wait_selftest_kernel<<<1, 64, 0, s>>>(mode, limit_ns, status, elapsed_ns);
    return cudaGetLastError();
}

}  // namespace spin
