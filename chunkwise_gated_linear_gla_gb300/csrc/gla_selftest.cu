// A check of the failure path of the library's bounded waits that faults
// nothing: one warp waits, with the same bounded mbarrier wait the pipelined
// kernels use, on a shared-memory barrier that nothing arrives on. When the
// limit runs out the kernel records a timeout in the device status word and
// returns, exactly as a pipelined kernel's role does before it winds down.
// The kernel allocates no tensor memory and issues no asynchronous copy, so
// nothing is left in flight when it returns.
#include "gla_internal.h"
#include "sm100.cuh"

namespace gla {
namespace {

constexpr int ERR_SELFTEST = 0x701;

__global__ void __launch_bounds__(32) gla_wait_selftest_kernel(int* status, uint64_t timeout_ns, int arrive)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        sm100::mbar_init(&bar, 1);
        sm100::mbar_fence_init();
    }
    __syncwarp();
    if (threadIdx.x == 0) {
        if (arrive) sm100::mbar_arrive(&bar);
        if (!sm100::mbar_wait(&bar, 0, timeout_ns)) atomicExch(status, ERR_SELFTEST);
    }
}

}  // namespace

cudaError_t launch_wait_selftest(int* status, unsigned limit_us, bool arrive, cudaStream_t s)
{
    gla_wait_selftest_kernel<<<1, 32, 0, s>>>(status, (uint64_t)limit_us * 1000ull, arrive ? 1 : 0);
    return cudaGetLastError();
}

}  // namespace gla
