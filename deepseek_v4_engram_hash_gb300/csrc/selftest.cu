// selftest.cu -- a check of the bounded wait that every copy ring and GEMM
// of this library uses (mbar_wait): one thread waits on an mbarrier that
// nothing arrives at, with a short limit, and must give up, raise the abort
// flag and ENGRAM_E_TIMEOUT, and return; the CTA's other warp leaves when it
// sees the flag, as the other roles of a ring do.  Nothing faults or hangs:
// every wait here ends by itself.
#include "common.cuh"

namespace {

__global__ void __launch_bounds__(64) wait_timeout_kernel(int *err, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        engram::mbar_init(engram::smem_u32(&bar), 1);
        abort_flag = 0;
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();
    volatile int *flag = &abort_flag;
    if (threadIdx.x == 0) {
        engram::mbar_wait(engram::smem_u32(&bar), 0, flag, err, limit_ns);   // phase 0 never completes
    } else if (threadIdx.x == 32) {
        const uint64_t t0 = engram::now_ns();                               // bounded as well
        while (!*flag && engram::now_ns() - t0 < 2 * limit_ns + 1000000ull) {
        }
    }
}

}  // namespace

namespace engram {
cudaError_t launch_wait_timeout(int *err, uint64_t limit_ns, cudaStream_t s) {
    wait_timeout_kernel<<<1, 64, 0, s>>>(err, limit_ns);
    return cudaGetLastError();
}
}  // namespace engram
