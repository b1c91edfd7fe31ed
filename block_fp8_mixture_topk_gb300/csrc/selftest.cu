// Check of the pipelines' bounded wait.  Every wait of the GEMM and decode pipelines goes
// through mbar_wait (common.cuh), which gives up after kWaitLimitNs, sets
// MOE_STATUS_WAIT_TIMEOUT and returns, so that a stalled pipeline ends its kernel with a status
// the host reads instead of hanging the GPU.  This kernel makes one such wait expire on purpose:
// it waits on an mbarrier phase that no thread completes (expire != 0), or on one completed
// first (expire == 0, which returns at once).  Nothing faults and the context stays usable.
#include "kernels.cuh"

namespace mfp8 {

namespace {

__global__ void bounded_wait_kernel(int expire, uint32_t* status) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_addr(&bar), 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (!expire) mbar_arrive(smem_addr(&bar));
        mbar_wait(smem_addr(&bar), 0, &abort_flag, status);
    }
    __syncthreads();
}

}  // namespace

cudaError_t launch_bounded_wait_check(int expire, uint32_t* status, cudaStream_t stream) {
    bounded_wait_kernel<<<1, 32, 0, stream>>>(expire, status);
    return cudaGetLastError();
}

}  // namespace mfp8
