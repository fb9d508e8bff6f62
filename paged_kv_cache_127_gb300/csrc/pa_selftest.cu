// pa_selftest.cu -- a device-side check of the kernels' failure path.
//
// Every wait of the library's kernels on an mbarrier gives up after a bounded
// number of polls, records PA_DEVERR_TIMEOUT and lets the kernel return,
// instead of spinning forever on a copy or a peer that never arrives.  This
// entry point runs exactly that bounded wait on an mbarrier nothing ever
// arrives at, so a test can watch it give up and then check that the context
// still runs kernels.  It makes no GPU fault and no hang: the wait ends after
// `limit` polls, each of which the hardware bounds in time.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/pa.h"
#include "pa_device.cuh"

namespace {

__global__ void bounded_wait_selftest_kernel(uint32_t limit, uint32_t *status) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = pa::smem_addr(&bar);
    if (threadIdx.x == 0) {
        pa::mbar_init(b, 1);  // expects one arrival, which never comes
        pa::fence_mbar_init();
    }
    __syncthreads();
    const bool arrived = pa::mbar_wait_bounded(b, 0u, limit);
    if (threadIdx.x == 0) *status = arrived ? 0u : PA_DEVERR_TIMEOUT;
}

}  // namespace

extern "C" PA_API int32_t pa_selftest_bounded_wait(uint32_t limit, uint32_t *status, void *stream) {
    if (!status || limit == 0 || limit > (1u << 20)) return PA_ERR_INVALID;
    bounded_wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(limit, status);
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
