// Self-test of the failure path every kernel shares: a bounded mbarrier
// wait that runs out sets the timeout flag in the workspace's status word
// and returns, so that uw_check_status reports UW_ERR_TIMEOUT and the
// context stays usable.  The kernel waits on a barrier that nothing ever
// arrives on (no copy, no other thread), with the same wait routine the
// matmul and decode kernels use and a caller-chosen number of tries.
#include <cuda_runtime.h>

#include "decode.cuh"
#include "tc.cuh"
#include "uw.h"

namespace uw {
namespace {

__global__ void withheld_arrival_kernel(uint32_t *status, uint32_t tries) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_addr(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        mbar_init_fence();
    }
    __syncthreads();
    if (threadIdx.x == 0)
        mbar_wait_tries(b, 0u, status, kStatusTimeout, tries);  // phase 0 never completes
}

}  // namespace
}  // namespace uw

extern "C" uw_status uw_selftest_bounded_wait(void *ws, size_t ws_bytes, uint32_t tries, void *stream) {
    if (!ws || tries == 0 || tries > uw::kWaitTries)
        return UW_ERR_INVALID_ARG;
    if (ws_bytes < 256)
        return UW_ERR_BUFFER_TOO_SMALL;
    uw::withheld_arrival_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<uint32_t *>(ws), tries);
    return cudaGetLastError() == cudaSuccess ? UW_OK : UW_ERR_CUDA;
}
