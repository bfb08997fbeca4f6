// k_selftest.cu -- exercises the bounded in-kernel wait that every kernel of
// the library uses (mbar_wait): one thread waits on an mbarrier that nothing
// ever arrives at.  The wait gives up after the time limit, raises the CTA's
// abort flag and writes the timeout code into the device status word, and the
// kernel returns; the context stays usable.  No fault, trap or unbounded
// loop is involved.
#include "ra_device.cuh"

namespace ra {
namespace {

__global__ void __launch_bounds__(32) wait_selftest_kernel(int *status, uint64_t timeout_ns,
                                                           int *gave_up)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const WaitCtx ctx{&abort_flag, status, timeout_ns};
        // phase 0 of `bar` needs one arrival that never comes
        const bool ok = mbar_wait(&bar, 0, ctx);
        *gave_up = ok ? 0 : 1;
    }
}

} // namespace

cudaError_t launch_wait_selftest(int *status, uint64_t timeout_ns, int *gave_up, cudaStream_t s)
{
    wait_selftest_kernel<<<1, 32, 0, s>>>(status, timeout_ns, gave_up);
    return cudaGetLastError();
}

} // namespace ra
