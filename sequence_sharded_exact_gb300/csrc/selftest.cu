// selftest.cu -- exercises the failure path of the kernels' bounded waits on the GPU, without a
// fault: one thread waits on an mbarrier that nothing will complete, through the same bounded-wait
// routine the tensor-core kernels use.  The wait runs out after `limit_ns`, sets the timeout bit
// of the device status word and the kernel returns, leaving the context usable.
#include "ra_internal.h"
#include "ra_ptx.cuh"

namespace ra {
namespace {

__global__ void bounded_wait_kernel(unsigned int* status, unsigned long long limit_ns, unsigned int* returned)
{
    __shared__ __align__(8) unsigned long long bar_storage;
    __shared__ int abort_flag;
    const uint32_t bar = smem_u32(&bar_storage);
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);  // one arrival expected; none will come
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const WaitCtl ctl{&abort_flag, status, limit_ns};
        const bool completed = mbar_wait(bar, 0, ctl);
        *returned = completed ? 2u : 1u;  // 1: the wait gave up, as it must
    }
}

}  // namespace

cudaError_t launch_bounded_wait_selftest(unsigned int* status, unsigned long long limit_ns, unsigned int* returned,
                                         cudaStream_t s)
{
    bounded_wait_kernel<<<1, 32, 0, s>>>(status, limit_ns, returned);
    return cudaGetLastError();
}

}  // namespace ra
