// Host-side interface between the C ABI entry points and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstddef>
#include <mutex>
#include <vector>
#include <cstdint>

#include "decode.cuh"
#include "uw.h"

namespace uw {

constexpr int kMaxSmemPerBlock = 227 * 1024;

// Where a matmul kernel gets its weights: uncompressed BF16 rows (the twin),
// the Huffman-coded blob, or the palette-4 form (4-bit palette indices) next
// to the blob's sign+mantissa bytes.
constexpr int kSrcBf16 = 0;
constexpr int kSrcHuffman = 1;
constexpr int kSrcPalette4 = 2;
constexpr int kSrcExponent = 3;  // the exponent bytes next to the blob's sign+mantissa bytes
constexpr int kP4TableBytes = 256 * 32 * 4;  // palette-4 pair table, 32 lane-private copies
constexpr int kSmemPerSm = 228 * 1024 - 3 * 1024;  // minus the per-CTA reservation of 3 CTAs

struct GemvParams {
    BlobView v;            // compressed weights (fused kernel)
    const uint16_t *w;     // uncompressed weights (twin kernel)
    const uint8_t *p4;     // palette-4 indices or exponent bytes (sign+mantissa etc. from v)
    const uint16_t *x;     // [batch, cols]
    uint16_t *y;           // [batch, rows]
    float *partial;        // [row blocks * splits][bp][32] split partial sums
    uint32_t *counters;    // [row blocks] arrival counters, left at zero
    uint32_t *status;      // device error word
    int64_t rows, cols, batch;
    int splits;
};

size_t gemv_smem_bytes(int64_t cols, int warps, int splits, int bp, bool compressed, uint32_t tbuf);
uw_status launch_gemv(const GemvParams &p, int warps, int bp, bool compressed, cudaStream_t stream);

// Batch-1 GEMV on column-range CTAs: W warps splitting all 64-column groups,
// rb_per_cta row blocks per CTA, one CTA per SM.
size_t gemv_kg_smem_bytes(int warps, int rb_per_cta, bool compressed, uint32_t tdata, int gpr);
uw_status launch_gemv_kg(const GemvParams &p, int warps, int rb_per_cta, int src, cudaStream_t stream);

// Tensor-core matmul (gemm_tc.cu): persistent CTAs of 4G producer warps, an
// MMA warp and an x loader, stream-K over (128-row block, 64-column group)
// units on every SM; batches above kTcMaxBatch run as several launches.
constexpr int kTcMaxBatch = 256;
struct TcParams {
    BlobView v;            // compressed weights (fused kernel)
    const uint16_t *w;     // uncompressed weights (twin kernel)
    const uint8_t *p4;     // palette-4 indices or exponent bytes (sign+mantissa etc. from v)
    const uint16_t *x;     // [batch, cols]
    uint16_t *y;           // [batch, rows]
    float *partial;        // [128-row blocks][maxseg][Np][128] segment partial sums
    uint32_t *counters;    // [128-row blocks] arrival counters, left at zero
    uint32_t *status;      // device error word
    int64_t rows, cols, batch;
    // set by the launcher
    uint32_t T, V, nk, maxseg;  // units, workers, K steps per block, segments per block at most
    int SX, Np;            // x stages (shared memory), padded batch
    uint32_t a0col;        // first tensor-memory column of the A stages
    CUtensorMap xmap;      // x as a 2-D tensor (cols x batch rows), 64 x Np boxes, 128-byte swizzle
    CUtensorMap wmap;      // uncompressed W (cols x rows), 64 x 128 boxes, 128-byte swizzle
    CUtensorMap ymap;      // y (rows x batch rows), 128 x 32 boxes, when ystage
    int ystage;            // whole segments store y through shared memory and ymap
    uint32_t ybuf_off;     // the y buffers' offset from the 1024-aligned shared base
};
// Whether G producer groups, batch rows Np and weights from `src` (tile
// data bytes tdata for the Huffman source) fit one CTA.
bool gemm_tc_fits(int G, int Np, int src, uint32_t tdata);
// Workspace floats of the segment partials.
int64_t gemm_tc_partial_floats(int64_t rows, int64_t cols, int64_t batch);
// max_ctas > 0: launch at most that many CTAs (the result does not change).
uw_status launch_gemm_tc(const TcParams &p, int G, int src, cudaStream_t stream, int max_ctas = 0);
// W [rows, cols] BF16 as a tensor map of 32-row x 64-column tiles, 128-byte
// swizzle (the batch-1 uncompressed GEMV's stages).
bool encode_w_tile_map(CUtensorMap *m, const uint16_t *w, int64_t rows, int64_t cols);

// Preprocess kernels.  max_ctas > 0 caps the grid (the SM split of a
// preprocess kernel running beside a matmul on another stream) and leaves
// the other SMs whole.  Decompress: over the whole matrix, 8-warp CTAs two
// per SM with one shared pair table; capped, persistent CTAs that each ask
// for kExclusiveSmem of shared memory so that each holds an SM by itself.
// Transcode: always persistent CTAs, one per SM, each holding 32
// lane-private copies of the pair table (more than half of an SM's shared
// memory, so a CTA always has its SM to itself).
constexpr size_t kExclusiveSmem = 116 * 1024;
uw_status launch_decompress(const BlobView &v, uint16_t *w_out, uint32_t *status, cudaStream_t stream,
                            int max_ctas = 0);
// Palette-4 form (rows*cols/2 bytes) or exponent form (rows*cols bytes) of a
// blob at out (16-byte aligned).
uw_status launch_transcode(const BlobView &v, uint8_t *out, bool palette4, uint32_t *status, cudaStream_t stream,
                           int max_ctas = 0);
uw_status launch_swiglu(const uint16_t *g, const uint16_t *u, uint16_t *h, int64_t n, cudaStream_t stream);
// dst[r, k] = k < cols ? src[r, k] : 0 for rows of cp (a multiple of 64)
// values; dst 16-byte aligned.
uw_status launch_pad_rows(const uint16_t *src, int64_t rows, int64_t cols, uint16_t *dst, int64_t cp,
                          cudaStream_t stream);

// SMs of the current device (152 if the query fails).
int sm_count();

// Raise a kernel's dynamic shared-memory limit once per (kernel, device);
// later launches skip the call, so they stay capturable in CUDA graphs.
bool ensure_smem_limit(const void *kernel, size_t bytes);
template <class Kernel>
inline bool ensure_smem(Kernel *kern, size_t bytes) {
    return ensure_smem_limit(reinterpret_cast<const void *>(kern), bytes);
}

// Launch with programmatic dependent launch allowed: the kernel may begin
// while the kernel before it in the stream drains.  Only for kernels that
// execute grid_dep_wait() before reading anything an earlier kernel wrote and
// before writing anything an earlier kernel may still read; their prologue
// (tables, first copies of the constant blob) then overlaps the earlier
// kernel's tail.
template <class... KArgs, class... Args>
inline cudaError_t launch_overlapped(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                     Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Tile buffer stride assumed where no blob is at hand (the largest possible).
constexpr uint32_t kWorstTileBuf = kMaxTileData + kTileSlack;

// Host helpers (api.cu).
void canonical_code_values(const uint8_t len[16], uint16_t code[16]);
void fill_blob_view(const uw_desc &d, const void *blob_dev, BlobView *v);
uint32_t tile_data_bytes(const uw_desc &d);  // a blob's tile buffer capacity

// Workspace layout: [status word | counters | split partials | weights].
struct WsLayout {
    size_t status = 0, counters = 0, partial = 0, weights = 0, xpad = 0, wpad = 0, total = 0;
};

// Plan resolution and matmul dispatch (api.cu), shared by the MLP chain.
//   plan_resolve       the strategy and variant a plan (or NULL) runs with.
//   run_layout         where a matmul's status word, split counters and
//                      partials sit in its workspace (`weights` = their end).
//   run_matmul         one matmul; p.status/counters/partial laid out as
//                      run_layout says, p.w / p.p4 / p.v by `src`.
uw_status plan_resolve(const uw_plan *plan, const uw_desc &d, int64_t batch, int *strategy, int *variant);
WsLayout run_layout(int64_t rows, int64_t cols, int64_t batch, int variant);
uw_status run_matmul(const GemvParams &p, int variant, int src, cudaStream_t stream, int max_ctas = 0);

}  // namespace uw
