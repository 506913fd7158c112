// Self-test of the bounded waits: a barrier that nothing ever arrives on,
// waited for with the decode kernel's wait primitive and a short limit. The
// wait gives up, the kernel records PA_DEV_TIMEOUT_BIT in the status word and
// returns; the GPU context stays usable. This exercises the failure path of
// every pipeline wait without a fault or a hang.
#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {
namespace {

__global__ void wait_selftest_kernel(int32_t *dev_status, uint64_t limit_ns)
{
    __shared__ alignas(8) uint64_t bar;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1); // one arrival expected; none is ever made
        fence_barrier_init();
    }
    __syncthreads();
    const bool ok = mbar_wait(b, 0, limit_ns);
    if (!__all_sync(0xffffffffu, ok) && threadIdx.x == 0 && dev_status)
        atomicOr(dev_status, PA_DEV_TIMEOUT_BIT);
}

} // namespace

cudaError_t launch_wait_selftest(int32_t *dev_status, uint64_t limit_ns, cudaStream_t stream)
{
    wait_selftest_kernel<<<1, 32, 0, stream>>>(dev_status, limit_ns);
    return cudaGetLastError();
}

} // namespace pa
