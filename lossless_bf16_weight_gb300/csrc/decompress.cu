// Decompress a blob back to BF16 weights in HBM (the Unweight blog's "full
// decode" pipeline: the restored matrix can then go to any GEMM).
//
// Each warp decodes consecutive tiles with the shared tile decoder
// (decode.cuh).  Lane j produces the 64 BF16 weights of row j; they pass
// through a per-warp 4 KB shared-memory buffer (16-byte chunks XOR-swizzled
// by row, conflict-free both ways) so that the global stores are coalesced
// 128-byte row segments.
#include "decode.cuh"
#include "kernels.h"

namespace uw {

namespace {

constexpr int kDecompWarps = 8;
constexpr int kTilesPerWarp = 4;
constexpr int kOutBufBytes = kTileRows * kGroup * 2;  // 4096

__global__ void __launch_bounds__(kDecompWarps * 32, 2)
    decompress_kernel(const BlobView v, uint16_t *__restrict__ out, uint32_t *status) {
    extern __shared__ __align__(16) unsigned char smem[];
    grid_dep_launch();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const DecodeShared ds = carve_common(smem);
    const uint32_t lut = smem_addr(ds.lut);
    const uint32_t tbuf = v.tbuf;
    uint32_t *wbuf = reinterpret_cast<uint32_t *>(smem + kCommonSmemBytes + size_t(warp) * 2 * tbuf);
    uint4 *obuf = reinterpret_cast<uint4 *>(smem + kCommonSmemBytes + size_t(kDecompWarps) * 2 * tbuf +
                                            size_t(warp) * kOutBufBytes);

    const int64_t gpr = v.cols / kGroup;
    const int64_t ntiles = (v.rows + kTileRows - 1) / kTileRows * gpr;
    const int64_t t_lo = (int64_t(blockIdx.x) * kDecompWarps + warp) * kTilesPerWarp;
    const int64_t t_hi = t_lo + kTilesPerWarp < ntiles ? t_lo + kTilesPerWarp : ntiles;

    // this warp's tiles t_lo .. t_hi-1, walked as (row block, group column)
    int64_t rb = t_lo / gpr, kg = t_lo - (t_lo / gpr) * gpr;
    TileMeta meta{};
    uint4 smn[4];
    uint32_t offs_next = 0;
    const uint32_t cbuf0 = smem_addr(wbuf);
    if (t_lo < t_hi) {
        tile_fetch(v, tile_loc(v, rb, kg, gpr), tile_offsets_load(v, t_lo), cbuf0, meta, smn);
        if (t_lo + 1 < t_hi)
            offs_next = tile_offsets_load(v, t_lo + 1);
    }
    build_tables(ds, v);
    __syncthreads();
    grid_dep_wait();  // the output may still be read by the kernel before

    for (int64_t t = t_lo; t < t_hi; t++) {
        const int R = tile_rows(v, rb);
        const int64_t rb_cur = rb, kg_cur = kg;
        if (++kg == gpr) {
            kg = 0;
            rb++;
        }
        const uint32_t cbuf = cbuf0 + uint32_t((t - t_lo) & 1) * tbuf;
        uint4 sm[4];
#pragma unroll
        for (int c = 0; c < 4; c++)
            sm[c] = smn[c];
        LaneStream ls;
        const uint32_t esc_mask = tile_begin(ds, meta, R, cbuf, ls, status);
        const uint32_t ebase = escape_base(meta, cbuf);
        if (t + 1 < t_hi) {
            tile_fetch(v, tile_loc(v, rb, kg, gpr), offs_next, cbuf0 + uint32_t((t + 1 - t_lo) & 1) * tbuf,
                       meta, smn);
            if (t + 2 < t_hi)
                offs_next = tile_offsets_load(v, t + 2);
        }
        uint32_t q[4];
#pragma unroll
        for (int I = 0; I < 32; I++) {
            q[I & 3] = decode_pair(ls, lut, I, sm_word(sm, I >> 1));
            if ((I & 3) == 3) {
                const int c = I >> 2;  // 16-byte chunk of the row segment
                obuf[lane * 8 + (c ^ (lane & 7))] = make_uint4(q[0], q[1], q[2], q[3]);
            }
        }
        tile_check(ls, status);
        if (esc_mask) {  // escaped groups: redo those lanes from raw exponents
            if ((esc_mask >> lane) & 1u) {
                uint4 e[4];
                escape_read(ebase, esc_mask, e);
#pragma unroll
                for (int I = 0; I < 32; I += 4) {
                    uint32_t q2[4];
#pragma unroll
                    for (int k = 0; k < 4; k++)
                        q2[k] = escape_pair(e, I + k, sm_word(sm, (I + k) >> 1));
                    const int c = I >> 2;
                    obuf[lane * 8 + (c ^ (lane & 7))] = make_uint4(q2[0], q2[1], q2[2], q2[3]);
                }
            }
        }
        __syncwarp();
        // coalesced stores: 4 rows x 128 bytes per instruction
        const int c = lane & 7;
#pragma unroll
        for (int it = 0; it < 8; it++) {
            const int r = it * 4 + (lane >> 3);
            if (r < R) {
                const uint4 val = obuf[r * 8 + (c ^ (r & 7))];
                uint16_t *dst = out + (rb_cur * kTileRows + r) * v.cols + kg_cur * kGroup + c * 8;
                *reinterpret_cast<uint4 *>(dst) = val;
            }
        }
        __syncwarp();
    }
}

}  // namespace

uw_status launch_decompress(const BlobView &v, uint16_t *w_out, uint32_t *status, cudaStream_t stream) {
    const int64_t gpr = v.cols / kGroup;
    const int64_t ntiles = (v.rows + kTileRows - 1) / kTileRows * gpr;
    const int64_t per_cta = int64_t(kDecompWarps) * kTilesPerWarp;
    const int64_t grid = (ntiles + per_cta - 1) / per_cta;
    const size_t smem = size_t(kCommonSmemBytes) + size_t(kDecompWarps) * (2 * size_t(v.tbuf) + kOutBufBytes);
    if (!ensure_smem(decompress_kernel, smem))
        return UW_ERR_CUDA;
    return launch_overlapped(decompress_kernel, dim3(unsigned(grid)), dim3(kDecompWarps * 32), smem, stream, v, w_out,
                             status) == cudaSuccess
               ? UW_OK
               : UW_ERR_CUDA;
}

}  // namespace uw
