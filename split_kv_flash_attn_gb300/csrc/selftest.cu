// selftest.cu -- the failure path of a bounded device-side wait, on demand.
//
// One thread waits on an mbarrier that nothing arrives on, with the wall-clock
// budget the caller gives; tc::mbar_wait gives up, and the thread sets bit 0
// of the handle's status word exactly as the tensor-core kernels do when a
// pipeline barrier never completes.
#include "internal.h"
#include "ptx.cuh"
#include "tc.cuh"

namespace skv {
namespace {

__global__ void __launch_bounds__(32) wait_timeout_kernel(uint64_t budget_ns, int *status)
{
    __shared__ __align__(8) uint64_t never;
    if (threadIdx.x == 0) {
        tc::mbar_init(smem_addr(&never), 1);
        tc::fence_barrier_init();
    }
    __syncwarp();
    if (threadIdx.x == 0 && !tc::mbar_wait(smem_addr(&never), 0, nullptr, budget_ns)) atomicOr(status, 1);
}

}  // namespace
}  // namespace skv

extern "C" int skv_selftest_wait_timeout(skv_handle *h, int64_t budget_ns, void *stream)
{
    if (!h) return SKV_EINVAL;
    h->err[0] = 0;
    if (budget_ns < 1000 || budget_ns > 1000000000) return skv::fail(h, SKV_EINVAL, "budget %lld ns outside [1e3, 1e9]",
                                                                    static_cast<long long>(budget_ns));
    skv::wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<uint64_t>(budget_ns),
                                                                             h->status);
    return skv::cuda_fail(h, cudaGetLastError(), "self-test launch");
}
