// Self-test of the bounded device waits that every TMA / tensor-core kernel relies on: one CTA
// waits, through the same helper the kernels use, on an mbarrier that nothing ever arrives on.
// The wait must give up after `limit_ns`, record OSF_ERR_TIMEOUT in the device status word and
// let the kernel exit normally, so the context stays usable (no trap, no hang).
#include "osf_internal.cuh"
#include "sm100_ptx.cuh"
#include "selftest.cuh"

namespace osf {
namespace {

__global__ void bounded_wait_selftest_kernel(unsigned long long limit_ns, int *status) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        ptx::mbar_init(ptx::smem_u32(&bar), 1);
        ptx::mbar_init_fence();
    }
    __syncthreads();
    // every thread of the warp waits on phase 0, which never completes
    const bool ok = ptx::mbar_wait(ptx::smem_u32(&bar), 0, nullptr, limit_ns);
    if (!__all_sync(0xffffffffu, ok) && threadIdx.x == 0) atomicExch(status, kStatusTimeout);
}

}  // namespace

cudaError_t launch_bounded_wait_selftest(unsigned long long limit_ns, int *status, cudaStream_t s) {
    bounded_wait_selftest_kernel<<<1, 32, 0, s>>>(limit_ns, status);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace osf
