// selftest.cu - proves that a device-side wait gives up: one thread waits on an
// mbarrier that nothing will ever complete and must leave after `limit_ns`,
// setting the timeout bit of the error word instead of hanging.
#include "kernels.h"
#include "ptx.cuh"

namespace moe {
namespace {

__global__ void wait_selftest_kernel(int* err, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = ptx::smem_u32(&bar);
    if (threadIdx.x == 0) {
        ptx::mbar_init(b, 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !ptx::mbar_wait(b, 0, limit_ns, nullptr)) atomicOr(err, kErrTimeout);
}

}  // namespace

cudaError_t launch_wait_selftest(int* err, uint64_t limit_ns, cudaStream_t s) {
    wait_selftest_kernel<<<1, 32, 0, s>>>(err, limit_ns);
    return cudaGetLastError();
}

}  // namespace moe
