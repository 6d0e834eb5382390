// Self-test of the device-side wait limit: one warp waits on a shared-memory
// barrier that nothing ever arrives at.  The bounded wait gives up after the
// configured limit, records a timeout in the device error word and the block
// exits normally, leaving the context usable.
#include "ptx_sm103.cuh"
#include "rsa_internal.h"

namespace rsa {
namespace {

__global__ void wait_never_kernel(uint64_t limit_ns, unsigned int *err)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        ptx::mbar_init(ptx::smem_u32(&bar), 1);
        abort_flag = 0;
        ptx::fence_barrier_init();
    }
    __syncthreads();
    ptx::mbar_wait(ptx::smem_u32(&bar), 0, limit_ns, &abort_flag, err, 0x7f);
}

}  // namespace

cudaError_t launch_selftest_wait(uint64_t limit_ns, unsigned int *err, cudaStream_t s)
{
    wait_never_kernel<<<1, 32, 0, s>>>(limit_ns, err);
    return cudaGetLastError();
}

}  // namespace rsa
