// Autotuner: for each batch size, time every (strategy, variant) candidate
// on the caller's stream and keep the fastest.  Mirrors the Unweight blog's
// autotuner, which picks the pipeline per weight matrix and batch size from
// measured throughput rather than heuristics (paragraphs on the autotuner
// and on small vs large batches).
//
// Timing: CUDA events around each call; the L2 cache is overwritten before
// every timed call (a memset of twice the L2 size inside the workspace), so
// each candidate reads its weights from HBM as it would inside a model whose
// weights are far larger than L2.  The median of kReps calls is kept.
#include <cuda_runtime.h>

#include <algorithm>
#include <vector>

#include "format.h"
#include "desc_check.h"
#include "kernels.h"
#include "uw.h"

namespace {

constexpr int kReps = 5;
constexpr int kWarm = 2;

size_t l2_flush_bytes() {
    int dev = 0, l2 = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess)
        return size_t(256) << 20;
    return uw::align_up(2 * size_t(l2), 256);
}

struct TuneLayout {
    size_t run, x, y, flush, total;
};

TuneLayout tune_layout(const uw_desc *d, int64_t max_batch) {
    TuneLayout t{};
    size_t need = 0;
    for (int strategy : {UW_STRATEGY_FUSED, UW_STRATEGY_DECOMPRESS_GEMM, UW_STRATEGY_PALETTE4, UW_STRATEGY_EXPONENT})
        for (int v = 0; v < uw_variant_count(strategy); v++) {
            uw_plan p{strategy, v, max_batch, 0.f};
            size_t b = 0;
            if (uw_workspace_size(d, max_batch, &p, &b) == UW_OK)
                need = std::max(need, b);
        }
    t.run = 0;
    t.x = uw::align_up(need, 256);
    t.y = uw::align_up(t.x + 2 * size_t(max_batch) * size_t(d->cols), 256);
    t.flush = uw::align_up(t.y + 2 * size_t(max_batch) * size_t(d->rows), 256);
    t.total = t.flush + l2_flush_bytes();
    return t;
}

}  // namespace

extern "C" uw_status uw_autotune_workspace_size(const uw_desc *d, const int64_t *batches, int32_t n,
                                                size_t *bytes) {
    if (!d || !batches || n <= 0 || !bytes)
        return UW_ERR_INVALID_ARG;
    int64_t mb = 1;
    for (int i = 0; i < n; i++) {
        if (batches[i] <= 0)
            return UW_ERR_INVALID_ARG;
        mb = std::max(mb, batches[i]);
    }
    *bytes = tune_layout(d, mb).total;
    return UW_OK;
}

extern "C" uw_status uw_autotune(const uw_desc *d, const void *blob_dev, const int64_t *batches, int32_t n,
                                 uw_plan *plans_out, void *ws, size_t ws_bytes, void *stream) {
    if (!d || !blob_dev || !batches || n <= 0 || !plans_out || !ws || !uw::desc_ok(*d))
        return UW_ERR_INVALID_ARG;
    size_t need = 0;
    uw_status s = uw_autotune_workspace_size(d, batches, n, &need);
    if (s != UW_OK)
        return s;
    if (ws_bytes < need)
        return UW_ERR_BUFFER_TOO_SMALL;
    int64_t mb = 1;
    for (int i = 0; i < n; i++)
        mb = std::max(mb, batches[i]);
    const TuneLayout L = tune_layout(d, mb);
    uint8_t *base = static_cast<uint8_t *>(ws);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(base, 0, L.flush, st) != cudaSuccess)
        return UW_ERR_CUDA;
    const uint16_t *x = reinterpret_cast<const uint16_t *>(base + L.x);
    uint16_t *y = reinterpret_cast<uint16_t *>(base + L.y);
    const size_t run_bytes = L.x - L.run;

    cudaEvent_t e0, e1;
    if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess)
        return UW_ERR_CUDA;
    uw_status result = UW_OK;
    for (int i = 0; i < n && result == UW_OK; i++) {
        uw_plan best{UW_STRATEGY_FUSED, -1, batches[i], -1.f};
        for (int strategy : {UW_STRATEGY_FUSED, UW_STRATEGY_DECOMPRESS_GEMM, UW_STRATEGY_PALETTE4, UW_STRATEGY_EXPONENT}) {
            for (int v = 0; v < uw_variant_count(strategy) && result == UW_OK; v++) {
                uw_plan p{strategy, v, batches[i], 0.f};
                std::vector<float> times;
                bool ok = true;
                for (int r = 0; r < kWarm + kReps && ok; r++) {
                    cudaMemsetAsync(base + L.flush, r & 0xFF, L.total - L.flush, st);
                    cudaEventRecord(e0, st);
                    const uw_status cs = uw_matmul(d, blob_dev, x, batches[i], y, &p, base, run_bytes, stream);
                    cudaEventRecord(e1, st);
                    if (cs != UW_OK) {
                        ok = false;  // variant not runnable for this shape (e.g. shared memory)
                        if (cs == UW_ERR_CUDA)
                            result = cs;
                        break;
                    }
                    if (cudaEventSynchronize(e1) != cudaSuccess) {
                        result = UW_ERR_CUDA;
                        break;
                    }
                    float ms = 0.f;
                    cudaEventElapsedTime(&ms, e0, e1);
                    if (r >= kWarm)
                        times.push_back(ms * 1000.f);
                    // a candidate 4x slower than the best so far cannot win: stop timing it
                    if (best.us > 0.f && ms * 1000.f > 4.f * best.us && r + 1 >= kWarm) {
                        times.clear();
                        break;
                    }
                }
                if (!ok || times.empty())
                    continue;
                std::sort(times.begin(), times.end());
                const float med = times[times.size() / 2];
                if (best.us < 0.f || med < best.us) {
                    best = p;
                    best.us = med;
                }
            }
        }
        plans_out[i] = best;
        if (best.variant < 0 && result == UW_OK)
            result = UW_ERR_UNSUPPORTED;
    }
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (result == UW_OK) {
        // leave the run region ready for the next user of the workspace
        if (cudaMemsetAsync(base, 0, L.x, st) != cudaSuccess)
            return UW_ERR_CUDA;
    }
    return result;
}
