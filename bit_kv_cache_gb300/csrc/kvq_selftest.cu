// kvq_selftest.cu -- self-test of the kernels' bounded waits (kvq_selftest_wait_timeout,
// declared in include/kvq.h).  It has no counterpart on the pages: it lets a test make
// a wait run out on a GPU without faulting, hanging or trapping it.
#include <cuda_runtime.h>
#include <stdint.h>

#include "kvq.h"
#include "kvq_device.cuh"

namespace {

// One warp waits on an mbarrier that nothing completes, through the same bounded wait
// the decode kernels use (mbar_wait, kWaitLimitCycles): it runs out, ORs the timeout
// bit into *status and returns.
__global__ void wait_selftest_kernel(int32_t *status) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        kvq::mbar_init(&bar, 1);
        kvq::fence_barrier_init();
    }
    __syncwarp();
    kvq::mbar_wait(&bar, 0u, status);
}

}  // namespace

extern "C" int kvq_selftest_wait_timeout(int32_t *status, void *stream) {
    if (!status || ((uintptr_t)status & 3)) return KVQ_ERR_INVALID_ARG;
    wait_selftest_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(status);
    return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}
