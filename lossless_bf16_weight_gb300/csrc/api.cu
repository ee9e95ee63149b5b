// C ABI entry points: blob validation, workspace layout, dispatch to the
// kernels.  No device memory is allocated here; everything comes from the
// caller's buffers.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <vector>

#include "format.h"
#include "desc_check.h"
#include "kernels.h"
#include "uw.h"

namespace uw {

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        n <= 0)
        return 152;
    return n;
}

namespace {

uint32_t rd32(const uint8_t *p) {
    uint32_t v;
    std::memcpy(&v, p, 4);
    return v;
}
uint64_t rd64(const uint8_t *p) {
    uint64_t v;
    std::memcpy(&v, p, 8);
    return v;
}

cudaStream_t as_stream(void *s) { return static_cast<cudaStream_t>(s); }

// Kernel variants.
//   0..14  row-block CTAs (gemv.cu): warps per CTA x split count
//   15..26 column CTAs, batch 1 only (gemv_kg.cu): warps per CTA x grid
//          size in full waves (1..4) of the GPU; the row blocks per CTA
//          follow from the matrix and the SM count
//   27..29 tensor-core CTAs (gemm_tc.cu): producer groups G (2, 3, 4),
//          stream-K over every SM
constexpr int kWarpChoices[3] = {4, 8, 16};
constexpr int kSplitChoices = 5;  // 1, 2, 4, 8, 16
constexpr int kRowVariants = 3 * kSplitChoices;
constexpr int kColWaves = 4;
constexpr int kColVariants = 3 * kColWaves;
constexpr int kTcGroups[3] = {2, 3, 4};
constexpr int kTcVariants = 3;
constexpr int kTcFirst = kRowVariants + kColVariants;
constexpr int kGemvVariants = kTcFirst + kTcVariants;
constexpr int kMaxBatchChunk = 8;

enum class Kind { kRow, kColumn, kTensor };

struct GemvVariant {
    Kind kind;
    int warps, splits, rb;  // warps: CTA warps (row, column) or producer groups G (tensor)
};


// `src`: the weights' source; only the Huffman stages constrain the row
// blocks per column CTA (the other sources keep a few KB of shared memory).
GemvVariant gemv_variant(int v, int64_t rows, int64_t cols, uint32_t tbuf = kWorstTileBuf, int src = kSrcHuffman) {
    const int64_t gpr = cols / kGroup;
    if (v < kRowVariants)
        return {Kind::kRow, kWarpChoices[v % 3], 1 << (v / 3), 0};
    if (v >= kTcFirst)
        return {Kind::kTensor, kTcGroups[v - kTcFirst], 1, 0};
    const int i = v - kRowVariants;
    const int w = kWarpChoices[i % 3];
    const int waves = 1 + i / 3;
    const int64_t nrb = (rows + kTileRows - 1) / kTileRows;
    const int64_t slots = int64_t(sm_count()) * waves;  // one CTA per SM per wave
    int64_t rb = (nrb + slots - 1) / slots;
    // keep the CTA within one SM's shared memory
    while (rb > 1 && src == kSrcHuffman &&
           gemv_kg_smem_bytes(w, int(rb), true, tbuf - kTileSlack, int(gpr)) > size_t(kMaxSmemPerBlock) - 1024)
        rb--;
    return {Kind::kColumn, w, 1, int(rb)};
}

// Tile data bytes assumed for a Huffman blob that is not at hand.
constexpr uint32_t kWorstTileData = kWorstTileBuf - kTileSlack;

// Tensor-core default: three producer groups when their stages fit this
// weight source and batch (measured on the gate matrix: the fastest at 16 and
// 64 batch rows, within 2% of two groups at 256; four groups leave the
// producers 96 registers and spill), else two.  The result does not depend on
// the number of groups (the MMAs accumulate in K order over the same cut), so
// the choice only changes the speed.
int default_tc_variant(int64_t rows, int64_t cols, int64_t batch, int src, uint32_t tdata) {
    (void)rows;
    (void)cols;
    const int np = int(std::min<int64_t>((batch + 15) / 16 * 16, kTcMaxBatch));
    return gemm_tc_fits(kTcGroups[1], np, src, tdata) ? kTcFirst + 1 : kTcFirst;
}

int pad_batch(int64_t b) {
    const int c = int(std::min<int64_t>(b, kMaxBatchChunk));
    return c <= 1 ? 1 : c <= 2 ? 2 : c <= 4 ? 4 : 8;
}

// Default variant.  Batch 1: column CTAs of 16 warps, one wave of the GPU.
// Batch 16 and up: tensor-core CTAs (sized for `src`, with the blob's tile
// data bytes for the Huffman source).  Otherwise row-block CTAs of 8 warps,
// split along K when the matrix has few row blocks.
int default_gemv_variant(int64_t rows, int64_t cols, int64_t batch, int src = kSrcHuffman,
                         uint32_t tdata = kWorstTileData) {
    const int64_t nrb = (rows + kTileRows - 1) / kTileRows;
    const int64_t gpr = cols / kGroup;
    if (batch == 1)
        return kRowVariants + 2;  // 16 warps, one wave
    if (batch >= 16)
        return default_tc_variant(rows, cols, batch, src, tdata);
    const int bp = pad_batch(batch);
    int si = 0;
    while (si + 1 < kSplitChoices && nrb * (int64_t(1) << si) < 2 * 152 &&
           gpr / (int64_t(1) << (si + 1)) >= 8)
        si++;
    while (si + 1 < kSplitChoices && gemv_smem_bytes(cols, 8, 1 << si, bp, true, kWorstTileBuf) > size_t(kMaxSmemPerBlock))
        si++;
    return 1 + 3 * si;
}

// cols: the matrix's own columns.  Ragged rows (cols % 64 != 0) run on the
// stored width with x (and, for the uncompressed matmul, W) copied into
// zero-extended rows at the end of the workspace.
WsLayout layout_for(int64_t rows, int64_t cols_true, int64_t batch, int strategy, int variant, bool pad_w = false) {
    WsLayout L;
    const int64_t cols = stored_cols(cols_true);
    const int64_t nrb = (rows + kTileRows - 1) / kTileRows;
    const GemvVariant gv = gemv_variant(variant, rows, cols);
    const int bp = gv.kind == Kind::kColumn ? 1 : pad_batch(batch);
    const uint64_t partial_floats = gv.kind == Kind::kTensor
                                        ? uint64_t(gemm_tc_partial_floats(rows, cols, batch))
                                        : uint64_t(nrb) * gv.splits * bp * 32;
    L.status = 0;
    L.counters = 256;
    L.partial = align_up(L.counters + 4 * uint64_t(nrb), 256);
    L.weights = align_up(L.partial + 4 * partial_floats, 256);
    L.total = L.weights;
    if (strategy == UW_STRATEGY_DECOMPRESS_GEMM)
        L.total = align_up(L.weights + 2 * uint64_t(rows) * uint64_t(cols), 256);
    else if (strategy == UW_STRATEGY_PALETTE4)  // the palette-4 form, 4 bits per weight
        L.total = align_up(L.weights + uint64_t(rows) * uint64_t(cols) / 2, 256);
    else if (strategy == UW_STRATEGY_EXPONENT)  // the exponent form, a byte per weight
        L.total = align_up(L.weights + uint64_t(rows) * uint64_t(cols), 256);
    L.xpad = L.wpad = L.total;
    if (cols != cols_true) {
        L.total = align_up(L.xpad + 2 * uint64_t(batch) * uint64_t(cols), 256);
        L.wpad = L.total;
        if (pad_w)
            L.total = align_up(L.wpad + 2 * uint64_t(rows) * uint64_t(cols), 256);
    }
    return L;
}

struct ResolvedPlan {
    int strategy, variant;
};

// Default variant of the palette-4 kernels: the column GEMV at batch 1, the
// tensor cores otherwise (there is no palette-4 row kernel).
int default_p4_variant(int64_t rows, int64_t cols, int64_t batch, int src) {
    return batch == 1 ? default_gemv_variant(rows, cols, 1) : default_tc_variant(rows, cols, batch, src, 0);
}

// tdata: the blob's tile data bytes (sizes the Huffman stages of the default).
uw_status resolve_plan(const uw_plan *plan, int64_t rows, int64_t cols_true, int64_t batch, ResolvedPlan *out,
                       uint32_t tdata = kWorstTileData) {
    const int64_t cols = stored_cols(cols_true);
    out->strategy = UW_STRATEGY_FUSED;
    out->variant = -1;
    if (plan) {
        if (plan->strategy != UW_STRATEGY_DEFAULT) {
            if (plan->strategy != UW_STRATEGY_FUSED && plan->strategy != UW_STRATEGY_DECOMPRESS_GEMM &&
                plan->strategy != UW_STRATEGY_PALETTE4 && plan->strategy != UW_STRATEGY_EXPONENT)
                return UW_ERR_INVALID_ARG;
            out->strategy = plan->strategy;
        }
        if (plan->variant >= 0) {
            if (plan->variant >= kGemvVariants)
                return UW_ERR_INVALID_ARG;
            out->variant = plan->variant;
        }
    }
    if (out->variant < 0) {
        switch (out->strategy) {
            case UW_STRATEGY_PALETTE4: out->variant = default_p4_variant(rows, cols, batch, kSrcPalette4); break;
            case UW_STRATEGY_EXPONENT: out->variant = default_p4_variant(rows, cols, batch, kSrcExponent); break;
            case UW_STRATEGY_DECOMPRESS_GEMM: out->variant = default_gemv_variant(rows, cols, batch, kSrcBf16); break;
            default: out->variant = default_gemv_variant(rows, cols, batch, kSrcHuffman, tdata); break;
        }
    }
    return UW_OK;
}

// A ragged matrix's activations, copied into zero-extended rows of the
// stored width (p.cols) at dst; p.x then points there.
uw_status pad_x(GemvParams &p, const uint16_t *x, int64_t cols_true, uint8_t *dst, cudaStream_t stream) {
    if (p.cols == cols_true)
        return UW_OK;
    uint16_t *xp = reinterpret_cast<uint16_t *>(dst);
    const uw_status s = launch_pad_rows(x, p.batch, cols_true, xp, p.cols, stream);
    if (s == UW_OK)
        p.x = xp;
    return s;
}

// Batch rows go through the CUDA-core row kernels in chunks of at most 8;
// the column kernels take batch 1 only; the tensor-core kernels take any
// batch (chunks of 256 inside the launcher).
uw_status run_gemv(GemvParams p, int variant, int src, cudaStream_t stream, int max_ctas = 0) {
    const bool compressed = src == kSrcHuffman;
    const GemvVariant gv = gemv_variant(variant, p.rows, p.cols, compressed ? p.v.tbuf : kWorstTileBuf, src);
    if (gv.kind == Kind::kTensor) {
        TcParams t{};
        t.v = p.v;
        t.w = p.w;
        t.p4 = p.p4;
        t.x = p.x;
        t.y = p.y;
        t.partial = p.partial;
        t.counters = p.counters;
        t.status = p.status;
        t.rows = p.rows;
        t.cols = p.cols;
        t.batch = p.batch;
        return launch_gemm_tc(t, gv.warps, src, stream, max_ctas);
    }
    if (gv.kind == Kind::kColumn) {
        if (p.batch != 1)
            return UW_ERR_UNSUPPORTED;
        p.splits = gv.splits;
        return launch_gemv_kg(p, gv.warps, gv.rb, src, stream);
    }
    if (src == kSrcPalette4 || src == kSrcExponent)
        return UW_ERR_UNSUPPORTED;  // no row kernel for the intermediate forms
    p.splits = gv.splits;
    const int64_t total = p.batch;
    for (int64_t b0 = 0; b0 < total; b0 += kMaxBatchChunk) {
        GemvParams q = p;
        q.batch = std::min<int64_t>(kMaxBatchChunk, total - b0);
        q.x = p.x + b0 * p.cols;
        q.y = p.y + b0 * p.rows;
        const uw_status s = launch_gemv(q, gv.warps, pad_batch(q.batch), compressed, stream);
        if (s != UW_OK)
            return s;
    }
    return UW_OK;
}

}  // namespace

uw_status plan_resolve(const uw_plan *plan, const uw_desc &d, int64_t batch, int *strategy, int *variant) {
    ResolvedPlan rp;
    const uw_status s = resolve_plan(plan, d.rows, d.cols, batch, &rp, tile_data_bytes(d));
    *strategy = rp.strategy;
    *variant = rp.variant;
    return s;
}

WsLayout run_layout(int64_t rows, int64_t cols, int64_t batch, int variant) {
    return layout_for(rows, cols, batch, UW_STRATEGY_FUSED, variant);
}

uw_status run_matmul(const GemvParams &p, int variant, int src, cudaStream_t stream, int max_ctas) {
    return run_gemv(p, variant, src, stream, max_ctas);
}

bool ensure_smem_limit(const void *kernel, size_t bytes) {
    struct Entry {
        const void *kernel;
        int device;
        size_t bytes;
    };
    static std::mutex mu;
    static std::vector<Entry> done;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return false;
    std::lock_guard<std::mutex> lock(mu);
    for (Entry &e : done)
        if (e.kernel == kernel && e.device == dev) {
            if (e.bytes >= bytes)
                return true;
            if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(bytes)) != cudaSuccess)
                return false;
            e.bytes = bytes;
            return true;
        }
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(bytes)) != cudaSuccess)
        return false;
    done.push_back({kernel, dev, bytes});
    return true;
}

void canonical_code_values(const uint8_t len[16], uint16_t code[16]) {
    int per_len[kLmax + 2] = {};
    for (int s = 0; s < 16; s++)
        if (len[s] <= kLmax)
            per_len[len[s]]++;
    per_len[0] = 0;
    uint32_t next[kLmax + 2] = {};
    uint32_t c = 0;
    for (int l = 1; l <= kLmax; l++) {
        c = (c + per_len[l - 1]) << 1;
        next[l] = c;
    }
    for (int s = 0; s < 16; s++)
        code[s] = (len[s] && len[s] <= kLmax) ? uint16_t(next[len[s]]++) : 0;
}

uint32_t tile_data_bytes(const uw_desc &d) {
    const uint64_t t = (std::max<uint64_t>(d.max_tile_bytes, 16) + 15) / 16 * 16;
    return uint32_t(std::min<uint64_t>(t, kMaxTileData));
}

void fill_blob_view(const uw_desc &d, const void *blob_dev, BlobView *v) {
    const uint8_t *b = static_cast<const uint8_t *>(blob_dev);
    v->sm = b + d.off_sm;
    v->glen = b + d.off_glen;
    v->tcode = reinterpret_cast<const uint32_t *>(b + d.off_tcode);
    v->tesc = reinterpret_cast<const uint32_t *>(b + d.off_tesc);
    v->code = b + d.off_code;
    v->esc = b + d.off_esc;
    v->code_bytes = d.off_esc - d.off_code;
    v->n_escaped = d.n_escaped;
    v->code16 = uint32_t((d.off_esc - d.off_code) / 16 > 0xFFFFFFFFull ? 0xFFFFFFFFull : (d.off_esc - d.off_code) / 16);
    v->n_esc32 = uint32_t(d.n_escaped);
    v->gpr = uint32_t(stored_cols(d.cols) / kGroup);
    v->nfull = uint32_t(d.rows / kTileRows);
    v->tail_rows = uint32_t(d.rows % kTileRows);
    v->ntiles = uint32_t(std::min<uint64_t>(d.n_tiles, 0xFFFFFFFFull));
    v->tdata = tile_data_bytes(d);
    v->tbuf = v->tdata + kTileSlack;
    v->rows = d.rows;
    v->cols = stored_cols(d.cols);
    v->ocols = d.cols;
    uint16_t code[16];
    canonical_code_values(d.code_len, code);
    std::memcpy(v->palette, d.palette, sizeof v->palette);
    for (int s = d.n_palette; s < 16; s++)
        v->palette[s] = 0;
    std::memset(v->prefix, 0, sizeof v->prefix);
    for (int s = 0; s < d.n_palette; s++) {
        const int l = d.code_len[s];
        if (!l)
            continue;
        const int lo = code[s] << (kLmax - l), hi = (code[s] + 1) << (kLmax - l);
        for (int p = lo; p < hi && p < kPrefixEntries; p++)
            v->prefix[p] = uint16_t((d.palette[s] << 4) | l);
    }
}

}  // namespace uw

using namespace uw;

extern "C" const char *uw_status_string(uw_status s) {
    switch (s) {
        case UW_OK: return "ok";
        case UW_ERR_INVALID_ARG: return "invalid argument";
        case UW_ERR_SHAPE: return "unsupported shape (rows and cols must be positive)";
        case UW_ERR_BUFFER_TOO_SMALL: return "buffer too small";
        case UW_ERR_CORRUPT: return "corrupt blob";
        case UW_ERR_CUDA: return "CUDA error";
        case UW_ERR_TIMEOUT: return "device wait timed out";
        case UW_ERR_UNSUPPORTED: return "unsupported request";
        case UW_ERR_INTERNAL: return "internal error";
    }
    return "unknown status";
}

namespace uw {

// The checks on a blob's header that need nothing but the header: sizes, the
// counts they imply, the sections in order inside blob_bytes, and a prefix
// code on the palette.  Sizes stay small enough that no section size wraps
// and every tile and escape index fits the kernels' 32-bit arithmetic.
bool desc_ok(const uw_desc &d) {
    if (d.lmax != kLmax || d.n_palette < 0 || d.n_palette > kPalette)
        return false;
    if (d.rows <= 0 || d.cols <= 0 || d.rows > (int64_t(1) << 31) || d.cols > (int64_t(1) << 31))
        return false;
    const uint64_t rows = uint64_t(d.rows), cols = uint64_t(stored_cols(d.cols));
    const uint64_t gpr = cols / kGroup;
    const uint64_t ntiles = (rows + kTileRows - 1) / kTileRows * gpr;
    if (d.n_groups != rows * gpr || d.n_tiles != ntiles || d.n_escaped > d.n_groups ||
        ntiles >= (uint64_t(1) << 32) || d.n_escaped >= (uint64_t(1) << 32))
        return false;
    const uint64_t sec[6] = {d.off_sm, d.off_glen, d.off_tcode, d.off_tesc, d.off_code, d.off_esc};
    if (d.blob_bytes >= (uint64_t(1) << 62))
        return false;
    for (uint64_t o : sec)
        if (o % kSectionAlign || o > d.blob_bytes)
            return false;
    if (d.off_sm != uint64_t(kHeaderBytes) || d.off_glen < d.off_sm + rows * cols ||
        d.off_tcode < d.off_glen + d.n_groups || d.off_tesc < d.off_tcode + 4 * (ntiles + 1) ||
        d.off_code < d.off_tesc + 4 * (ntiles + 1) || d.off_esc < d.off_code ||
        d.off_esc + 64 * d.n_escaped > d.blob_bytes)
        return false;
    double kraft = 0.0;
    for (int s = 0; s < kPalette; s++) {
        if (d.code_len[s] > kLmax || (s >= d.n_palette && d.code_len[s]))
            return false;
        if (d.code_len[s])
            kraft += 1.0 / double(1u << d.code_len[s]);
        for (int t = 0; t < s && s < d.n_palette; t++)
            if (d.palette[t] == d.palette[s])
                return false;
    }
    return kraft <= 1.0;
}

}  // namespace uw

extern "C" uw_status uw_blob_info(const void *blob_host, size_t bytes, uw_desc *out) {
    if (!blob_host || !out)
        return UW_ERR_INVALID_ARG;
    const uint8_t *b = static_cast<const uint8_t *>(blob_host);
    if (bytes < size_t(kHeaderBytes) || rd32(b + hdr::magic) != kMagic || rd32(b + hdr::version) != kVersion)
        return UW_ERR_CORRUPT;
    uw_desc d;
    std::memset(&d, 0, sizeof d);
    d.rows = int64_t(rd64(b + hdr::rows));
    d.cols = int64_t(rd64(b + hdr::cols));
    d.lmax = int32_t(rd32(b + hdr::lmax));
    d.n_palette = int32_t(rd32(b + hdr::n_palette));
    std::memcpy(d.palette, b + hdr::palette, 16);
    std::memcpy(d.code_len, b + hdr::code_len, 16);
    d.n_groups = rd64(b + hdr::n_groups);
    d.n_escaped = rd64(b + hdr::n_escaped);
    d.n_tiles = rd64(b + hdr::n_tiles);
    d.code_bits = rd64(b + hdr::code_bits);
    d.off_sm = rd64(b + hdr::off_sm);
    d.off_glen = rd64(b + hdr::off_glen);
    d.off_tcode = rd64(b + hdr::off_tcode);
    d.off_tesc = rd64(b + hdr::off_tesc);
    d.off_code = rd64(b + hdr::off_code);
    d.off_esc = rd64(b + hdr::off_esc);
    d.blob_bytes = rd64(b + hdr::blob_bytes);
    if (rd32(b + hdr::group) != uint32_t(kGroup) || rd32(b + hdr::tile_rows) != uint32_t(kTileRows) ||
        !desc_ok(d) || d.blob_bytes > bytes)
        return UW_ERR_CORRUPT;
    const uint64_t rows = uint64_t(d.rows), cols = uint64_t(stored_cols(d.cols));
    const uint64_t gpr = cols / kGroup;
    const uint64_t ntiles = (rows + kTileRows - 1) / kTileRows * gpr;
    // tile tables against the group lengths
    const uint32_t *tcode = reinterpret_cast<const uint32_t *>(b + d.off_tcode);
    const uint32_t *tesc = reinterpret_cast<const uint32_t *>(b + d.off_tesc);
    const uint8_t *glen = b + d.off_glen;
    if (tcode[0] != 0 || tesc[0] != 0 || tesc[ntiles] != d.n_escaped ||
        uint64_t(tcode[ntiles]) * 16 > d.off_esc - d.off_code)
        return UW_ERR_CORRUPT;
    uint64_t bits_hint = 0, max_tile = 0;
    for (uint64_t t = 0; t < ntiles; t++) {
        const uint64_t rb = t / gpr, kg = t % gpr;
        const uint64_t R = std::min<uint64_t>(kTileRows, rows - rb * kTileRows);
        const uint64_t q0 = kTileRows * rb * gpr + R * kg;
        uint64_t sum = 0, nz = 0;
        for (uint64_t j = 0; j < R; j++) {
            const unsigned g = glen[q0 + j];
            if (g > unsigned(kMaxGroupCodeBytes))
                return UW_ERR_CORRUPT;
            sum += g;
            nz += g == 0;
        }
        if (tcode[t + 1] < tcode[t] || uint64_t(tcode[t + 1] - tcode[t]) != (sum + 15) / 16 ||
            tesc[t + 1] < tesc[t] || tesc[t + 1] - tesc[t] != nz)
            return UW_ERR_CORRUPT;
        bits_hint += sum;
        max_tile = std::max<uint64_t>(max_tile, 16 * uint64_t(tcode[t + 1] - tcode[t]) + 64 * nz);
    }
    d.max_tile_bytes = max_tile;
    if (d.code_bits > 8 * bits_hint || d.code_bits + 8 * (d.n_groups - d.n_escaped) < 8 * bits_hint)
        return UW_ERR_CORRUPT;
    *out = d;
    return UW_OK;
}

extern "C" uw_status uw_workspace_size(const uw_desc *d, int64_t batch, const uw_plan *plan, size_t *bytes) {
    if (!d || !bytes || batch < 0)
        return UW_ERR_INVALID_ARG;
    ResolvedPlan rp;
    const uw_status s = resolve_plan(plan, d->rows, d->cols, std::max<int64_t>(batch, 1), &rp, tile_data_bytes(*d));
    if (s != UW_OK)
        return s;
    *bytes = layout_for(d->rows, d->cols, std::max<int64_t>(batch, 1), rp.strategy, rp.variant).total;
    return UW_OK;
}

extern "C" uw_status uw_workspace_init(void *ws, size_t ws_bytes, void *stream) {
    if (!ws)
        return UW_ERR_INVALID_ARG;
    return cudaMemsetAsync(ws, 0, ws_bytes, as_stream(stream)) == cudaSuccess ? UW_OK : UW_ERR_CUDA;
}

extern "C" uw_status uw_check_status(void *ws, void *stream) {
    if (!ws)
        return UW_ERR_INVALID_ARG;
    uint32_t word = 0;
    cudaStream_t st = as_stream(stream);
    if (cudaMemcpyAsync(&word, ws, 4, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return UW_ERR_CUDA;
    if (!word)
        return UW_OK;
    if (cudaMemsetAsync(ws, 0, 4, st) != cudaSuccess || cudaStreamSynchronize(st) != cudaSuccess)
        return UW_ERR_CUDA;
    return (word & kStatusTimeout) ? UW_ERR_TIMEOUT : UW_ERR_CORRUPT;
}

extern "C" uw_status uw_decompress(const uw_desc *d, const void *blob_dev, uint16_t *w_dev, void *ws,
                                   size_t ws_bytes, void *stream) {
    if (!d || !blob_dev || !w_dev || !ws || (reinterpret_cast<uintptr_t>(w_dev) & 15) || !desc_ok(*d))
        return UW_ERR_INVALID_ARG;
    if (ws_bytes < 256)
        return UW_ERR_BUFFER_TOO_SMALL;
    BlobView v;
    fill_blob_view(*d, blob_dev, &v);
    return launch_decompress(v, w_dev, static_cast<uint32_t *>(ws), as_stream(stream));
}

extern "C" uw_status uw_matmul(const uw_desc *d, const void *blob_dev, const uint16_t *x, int64_t batch,
                               uint16_t *y, const uw_plan *plan, void *ws, size_t ws_bytes, void *stream) {
    if (!d || !blob_dev || !x || !y || !ws || batch <= 0 || (reinterpret_cast<uintptr_t>(x) & 15) || !desc_ok(*d))
        return UW_ERR_INVALID_ARG;
    ResolvedPlan rp;
    uw_status s = resolve_plan(plan, d->rows, d->cols, batch, &rp, tile_data_bytes(*d));
    if (s != UW_OK)
        return s;
    const WsLayout L = layout_for(d->rows, d->cols, batch, rp.strategy, rp.variant);
    if (ws_bytes < L.total)
        return UW_ERR_BUFFER_TOO_SMALL;
    uint8_t *wsb = static_cast<uint8_t *>(ws);
    GemvParams p{};
    fill_blob_view(*d, blob_dev, &p.v);
    p.x = x;
    p.y = y;
    p.partial = reinterpret_cast<float *>(wsb + L.partial);
    p.counters = reinterpret_cast<uint32_t *>(wsb + L.counters);
    p.status = reinterpret_cast<uint32_t *>(wsb + L.status);
    p.rows = d->rows;
    p.cols = p.v.cols;
    p.batch = batch;
    if (rp.strategy == UW_STRATEGY_DECOMPRESS_GEMM) {
        uint16_t *w = reinterpret_cast<uint16_t *>(wsb + L.weights);
        BlobView stored = p.v;  // the stored width, filler columns included
        stored.ocols = stored.cols;
        s = launch_decompress(stored, w, p.status, as_stream(stream));
        if (s == UW_OK)
            s = pad_x(p, x, d->cols, wsb + L.xpad, as_stream(stream));
        if (s != UW_OK)
            return s;
        p.w = w;
        return run_gemv(p, rp.variant, kSrcBf16, as_stream(stream));
    }
    if (rp.strategy == UW_STRATEGY_PALETTE4 || rp.strategy == UW_STRATEGY_EXPONENT) {
        const bool pal = rp.strategy == UW_STRATEGY_PALETTE4;
        uint8_t *form = wsb + L.weights;
        s = launch_transcode(p.v, form, pal, p.status, as_stream(stream));
        if (s == UW_OK)
            s = pad_x(p, x, d->cols, wsb + L.xpad, as_stream(stream));
        if (s != UW_OK)
            return s;
        p.p4 = form;
        return run_gemv(p, rp.variant, pal ? kSrcPalette4 : kSrcExponent, as_stream(stream));
    }
    s = pad_x(p, x, d->cols, wsb + L.xpad, as_stream(stream));
    return s != UW_OK ? s : run_gemv(p, rp.variant, kSrcHuffman, as_stream(stream));
}

extern "C" uw_status uw_palette4_bytes(const uw_desc *d, size_t *bytes) {
    if (!d || !bytes)
        return UW_ERR_INVALID_ARG;
    *bytes = size_t(uint64_t(d->rows) * uint64_t(stored_cols(d->cols)) / 2);
    return UW_OK;
}

extern "C" uw_status uw_transcode_palette4(const uw_desc *d, const void *blob_dev, void *p4_dev, void *ws,
                                           size_t ws_bytes, void *stream) {
    if (!d || !blob_dev || !p4_dev || !ws || (reinterpret_cast<uintptr_t>(p4_dev) & 15) || !desc_ok(*d))
        return UW_ERR_INVALID_ARG;
    if (ws_bytes < 256)
        return UW_ERR_BUFFER_TOO_SMALL;
    BlobView v;
    fill_blob_view(*d, blob_dev, &v);
    return launch_transcode(v, static_cast<uint8_t *>(p4_dev), true, static_cast<uint32_t *>(ws), as_stream(stream));
}

namespace uw {
namespace {
uw_status matmul_formed(const uw_desc *d, const void *blob_dev, const void *form_dev, const uint16_t *x, int64_t batch,
                        uint16_t *y, int32_t variant, void *ws, size_t ws_bytes, void *stream, int src) {
    if (!d || !blob_dev || !form_dev || !x || !y || !ws || batch <= 0 || (reinterpret_cast<uintptr_t>(x) & 15) ||
        (reinterpret_cast<uintptr_t>(form_dev) & 15) || !desc_ok(*d))
        return UW_ERR_INVALID_ARG;
    if (variant >= kGemvVariants)
        return UW_ERR_INVALID_ARG;
    const int v = variant < 0 ? default_p4_variant(d->rows, stored_cols(d->cols), batch, src) : variant;
    const WsLayout L = layout_for(d->rows, d->cols, batch, UW_STRATEGY_FUSED, v);
    if (ws_bytes < L.total)
        return UW_ERR_BUFFER_TOO_SMALL;
    uint8_t *wsb = static_cast<uint8_t *>(ws);
    GemvParams p{};
    fill_blob_view(*d, blob_dev, &p.v);
    p.p4 = static_cast<const uint8_t *>(form_dev);
    p.x = x;
    p.y = y;
    p.partial = reinterpret_cast<float *>(wsb + L.partial);
    p.counters = reinterpret_cast<uint32_t *>(wsb + L.counters);
    p.status = reinterpret_cast<uint32_t *>(wsb + L.status);
    p.rows = d->rows;
    p.cols = p.v.cols;
    p.batch = batch;
    const uw_status s = pad_x(p, x, d->cols, wsb + L.xpad, as_stream(stream));
    return s != UW_OK ? s : run_gemv(p, v, src, as_stream(stream));
}
}  // namespace
}  // namespace uw

extern "C" uw_status uw_matmul_palette4(const uw_desc *d, const void *blob_dev, const void *p4_dev,
                                        const uint16_t *x, int64_t batch, uint16_t *y, int32_t variant, void *ws,
                                        size_t ws_bytes, void *stream) {
    return uw::matmul_formed(d, blob_dev, p4_dev, x, batch, y, variant, ws, ws_bytes, stream, uw::kSrcPalette4);
}

extern "C" uw_status uw_exponent_bytes(const uw_desc *d, size_t *bytes) {
    if (!d || !bytes)
        return UW_ERR_INVALID_ARG;
    *bytes = size_t(uint64_t(d->rows) * uint64_t(uw::stored_cols(d->cols)));
    return UW_OK;
}

extern "C" uw_status uw_decode_exponents(const uw_desc *d, const void *blob_dev, void *e_dev, void *ws,
                                         size_t ws_bytes, void *stream) {
    if (!d || !blob_dev || !e_dev || !ws || (reinterpret_cast<uintptr_t>(e_dev) & 15) || !uw::desc_ok(*d))
        return UW_ERR_INVALID_ARG;
    if (ws_bytes < 256)
        return UW_ERR_BUFFER_TOO_SMALL;
    uw::BlobView v;
    uw::fill_blob_view(*d, blob_dev, &v);
    return uw::launch_transcode(v, static_cast<uint8_t *>(e_dev), false, static_cast<uint32_t *>(ws),
                                uw::as_stream(stream));
}

extern "C" uw_status uw_matmul_exponents(const uw_desc *d, const void *blob_dev, const void *e_dev,
                                         const uint16_t *x, int64_t batch, uint16_t *y, int32_t variant, void *ws,
                                         size_t ws_bytes, void *stream) {
    return uw::matmul_formed(d, blob_dev, e_dev, x, batch, y, variant, ws, ws_bytes, stream, uw::kSrcExponent);
}

extern "C" uw_status uw_matmul_bf16(const uint16_t *w, int64_t rows, int64_t cols, const uint16_t *x,
                                    int64_t batch, uint16_t *y, int32_t variant, void *ws, size_t ws_bytes,
                                    void *stream) {
    if (!w || !x || !y || !ws || batch <= 0 || (reinterpret_cast<uintptr_t>(x) & 15) ||
        (reinterpret_cast<uintptr_t>(w) & 15))
        return UW_ERR_INVALID_ARG;
    if (rows <= 0 || cols <= 0)
        return UW_ERR_SHAPE;
    if (rows > (int64_t(1) << 31) || cols > (int64_t(1) << 31))
        return UW_ERR_UNSUPPORTED;  // the same limit as compressed matrices
    if (variant >= kGemvVariants)
        return UW_ERR_INVALID_ARG;
    const int64_t cp = stored_cols(cols);
    const int v = variant < 0 ? default_gemv_variant(rows, cp, batch, kSrcBf16) : variant;
    const WsLayout L = layout_for(rows, cols, batch, UW_STRATEGY_FUSED, v, true);
    if (ws_bytes < L.total)
        return UW_ERR_BUFFER_TOO_SMALL;
    uint8_t *wsb = static_cast<uint8_t *>(ws);
    GemvParams p{};
    p.w = w;
    p.x = x;
    p.y = y;
    p.partial = reinterpret_cast<float *>(wsb + L.partial);
    p.counters = reinterpret_cast<uint32_t *>(wsb + L.counters);
    p.status = reinterpret_cast<uint32_t *>(wsb + L.status);
    p.rows = rows;
    p.cols = cp;
    p.batch = batch;
    if (cp != cols) {  // ragged rows: W and x copied into zero-extended rows
        uint16_t *wp = reinterpret_cast<uint16_t *>(wsb + L.wpad);
        const uw_status s = launch_pad_rows(w, rows, cols, wp, cp, as_stream(stream));
        if (s != UW_OK)
            return s;
        p.w = wp;
    }
    const uw_status s = pad_x(p, x, cols, wsb + L.xpad, as_stream(stream));
    return s != UW_OK ? s : run_gemv(p, v, kSrcBf16, as_stream(stream));
}

extern "C" uw_status uw_workspace_size_bf16(int64_t rows, int64_t cols, int64_t batch, int32_t variant,
                                          size_t *bytes) {
    if (!bytes || batch < 0)
        return UW_ERR_INVALID_ARG;
    if (rows <= 0 || cols <= 0)
        return UW_ERR_SHAPE;
    if (rows > (int64_t(1) << 31) || cols > (int64_t(1) << 31))
        return UW_ERR_UNSUPPORTED;
    if (variant >= kGemvVariants)
        return UW_ERR_INVALID_ARG;
    const int64_t b = std::max<int64_t>(batch, 1);
    const int v = variant < 0 ? default_gemv_variant(rows, stored_cols(cols), b, kSrcBf16) : variant;
    *bytes = layout_for(rows, cols, b, UW_STRATEGY_FUSED, v, true).total;
    return UW_OK;
}

extern "C" uw_status uw_swiglu(const uint16_t *g, const uint16_t *u, uint16_t *h, int64_t n, void *stream) {
    if (!g || !u || !h || n < 0)
        return UW_ERR_INVALID_ARG;
    return launch_swiglu(g, u, h, n, as_stream(stream));
}

extern "C" int32_t uw_variant_count(int32_t strategy) {
    return (strategy == UW_STRATEGY_FUSED || strategy == UW_STRATEGY_DECOMPRESS_GEMM ||
            strategy == UW_STRATEGY_PALETTE4 || strategy == UW_STRATEGY_EXPONENT)
               ? kGemvVariants
               : 0;
}

extern "C" const char *uw_variant_name(int32_t strategy, int32_t variant) {
    static const char *names[kGemvVariants] = {
        "w4s1", "w8s1", "w16s1", "w4s2", "w8s2", "w16s2", "w4s4", "w8s4", "w16s4",
        "w4s8", "w8s8", "w16s8", "w4s16", "w8s16", "w16s16",
        "col_w4x1", "col_w8x1", "col_w16x1", "col_w4x2", "col_w8x2", "col_w16x2",
        "col_w4x3", "col_w8x3", "col_w16x3", "col_w4x4", "col_w8x4", "col_w16x4",
        "tc_g2", "tc_g3", "tc_g4"};
    if (uw_variant_count(strategy) == 0 || variant < 0 || variant >= kGemvVariants)
        return nullptr;
    return names[variant];
}
