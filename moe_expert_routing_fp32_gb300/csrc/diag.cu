// diag.cu -- moe_selftest_wait_timeout: a check of the bounded waits.
//
// Every pipeline wait in this library (TMA stages, tensor-memory
// accumulators, the router's copy ring) goes through mbar_wait_bounded, which
// gives up after kWaitLimitNs, records MOE_DEV_TIMEOUT and lets the kernel
// unwind instead of hanging the GPU.  This kernel waits through that same
// helper on a barrier phase that nothing ever completes, so a caller can
// observe the mechanism end to end: the call returns after about one limit
// with the bit set, and the context stays usable.
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

__global__ void wait_timeout_kernel(int32_t *dev_status) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(&bar, 1);      // expects one arrival; none will come
        fence_barrier_init();
    }
    __syncthreads();
    mbar_wait_bounded(&bar, 0, &abort_flag, dev_status);
}

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_selftest_wait_timeout(int32_t *dev_status, moe_stream_t stream) {
    if (!dev_status) return MOE_ERR_INVALID_ARG;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_NO_DEVICE;
    }
    moe::wait_timeout_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(dev_status);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
