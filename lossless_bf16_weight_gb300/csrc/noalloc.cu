// uw_matmul_noalloc: the fused matmul for callers that cannot allocate.
//
// Its scratch (the device error word, the split-K arrival counters and the
// split-K partial sums that uw_matmul otherwise takes from the caller's
// workspace) lives in one file-scope device array of kNoAllocScratchBytes.
// Every GPU that loads the library holds that array until the process
// exits.  The call itself allocates nothing: no cudaMalloc, no cudaFree.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "desc_check.h"
#include "uw.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;  // 1 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch, looked up once per device with that
// device current.  In host code the array's name is only a host-side
// stand-in, so kernels must be given this address, never the name.
void *scratch_address(int device, uw_status *err) {
    static std::mutex mu;
    static void *addr[kMaxDevices] = {};
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[device]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            *err = UW_ERR_CUDA;
            return nullptr;
        }
        addr[device] = p;
    }
    return addr[device];
}

}  // namespace

extern "C" uw_status uw_matmul_noalloc(const uw_desc *d, const void *blob_dev, const uint16_t *x_dev,
                                       int64_t batch, uint16_t *y_dev, void *stream) {
    if (!d || !blob_dev || !x_dev || !y_dev || batch <= 0)
        return UW_ERR_INVALID_ARG;
    // the checks uw_matmul makes, before any size is worked out from the
    // descriptor and before anything is queued on the stream
    if (!uw::desc_ok(*d) || (reinterpret_cast<uintptr_t>(x_dev) & 15u) != 0)
        return UW_ERR_INVALID_ARG;
    size_t need = 0;
    uw_status s = uw_workspace_size(d, batch, nullptr, &need);
    if (s != UW_OK)
        return s;
    if (need > kNoAllocScratchBytes)
        return UW_ERR_UNSUPPORTED;  // more scratch than the fixed array holds
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= kMaxDevices)
        return UW_ERR_CUDA;
    uw_status err = UW_OK;
    void *scratch = scratch_address(device, &err);
    if (!scratch)
        return err;
    // The array keeps whatever the previous call left: clear the part this
    // call uses (error word, arrival counters, partial sums).
    if (cudaMemsetAsync(scratch, 0, need, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return UW_ERR_CUDA;
    return uw_matmul(d, blob_dev, x_dev, batch, y_dev, nullptr, scratch, kNoAllocScratchBytes, stream);
}
