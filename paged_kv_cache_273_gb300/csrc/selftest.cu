// pkv_selftest_wait_timeout: one thread waits, with the library's bounded
// mbarrier wait, on a phase that nothing completes.  The wait gives up after
// its time limit and the kernel records PKV_EBIT_TIMEOUT in the pool's error
// word and returns, so the failure path of every bounded wait in the
// library's kernels (report, return, context still usable) can be checked
// without faulting or hanging the device.

#include <cuda_runtime.h>

#include "device_common.cuh"

namespace pkv {
namespace {

using namespace dev;

__global__ void wait_timeout_kernel(unsigned int *err)
{
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);                        // one arrival expected, none comes
        abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !mbar_wait_bounded(&bar, 0u, &abort_flag))
        atomicOr(err, PKV_EBIT_TIMEOUT);
}

}  // namespace

int launch_selftest_wait_timeout(const pkv_pool *pool, pkv_stream_t stream)
{
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    wait_timeout_kernel<<<1, 32, 0, s>>>(pool->d_err);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace pkv
