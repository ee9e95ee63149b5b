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

constexpr int kDecompWarps = 8;        // warps of a CTA launched over the whole matrix (two CTAs per SM)
constexpr int kDecompWarpsSplit = 16;  // warps of a CTA of a capped, persistent grid (one CTA per SM)
constexpr int kTilesPerWarp = 4;
constexpr int kOutBufBytes = kTileRows * kGroup * 2;  // 4096

template <int W>
__global__ void __launch_bounds__(W * 32, 16 / W)
    decompress_kernel(const BlobView v, uint16_t *__restrict__ out, uint32_t *status) {
    extern __shared__ __align__(16) unsigned char smem[];
    grid_dep_launch();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const DecodeShared ds = carve_common(smem);
    const uint32_t lut = smem_addr(ds.lut);
    const uint32_t tbuf = v.tbuf;
    uint32_t *wbuf = reinterpret_cast<uint32_t *>(smem + kCommonSmemBytes + size_t(warp) * 2 * tbuf);
    uint4 *obuf = reinterpret_cast<uint4 *>(smem + kCommonSmemBytes + size_t(W) * 2 * tbuf +
                                            size_t(warp) * kOutBufBytes);

    const uint32_t gpr = v.gpr, ntiles = v.ntiles;
    const uint32_t step = gridDim.x * uint32_t(W * kTilesPerWarp);
    const uint64_t first = (uint64_t(blockIdx.x) * W + warp) * kTilesPerWarp;
    TileWalk cur, nxt;
    walk_seek(cur, first < ntiles ? uint32_t(first) : ntiles, gpr);
    nxt = cur;
    walk_next(nxt, kTilesPerWarp, step, ntiles, gpr);
    TileMeta meta{};
    uint4 smn[4];
    uint32_t offs_next = 0;
    const uint32_t cbuf0 = smem_addr(wbuf);
    if (cur.t < ntiles) {
        tile_fetch(v, tile_loc32(v, cur.rb, cur.kg, cur.t), tile_offsets_load32(v, cur.t), cbuf0, meta, smn);
        if (nxt.t < ntiles)
            offs_next = tile_offsets_load32(v, nxt.t);
    }
    build_tables(ds, v);
    __syncthreads();
    grid_dep_wait();  // the output may still be read by the kernel before

    for (uint32_t i = 0; cur.t < ntiles; i++) {
        const int R = tile_rows32(v, cur.rb);
        const uint32_t cbuf = cbuf0 + (i & 1u) * tbuf;
        uint4 sm[4];
#pragma unroll
        for (int c = 0; c < 4; c++)
            sm[c] = smn[c];
        LaneStream ls;
        const uint32_t esc_mask = tile_begin(ds, meta, R, cbuf, ls, status);
        const uint32_t ebase = escape_base(meta, cbuf);
        TileWalk n2 = nxt;
        if (nxt.t < ntiles) {
            tile_fetch(v, tile_loc32(v, nxt.rb, nxt.kg, nxt.t), offs_next, cbuf0 + ((i + 1) & 1u) * tbuf, meta, smn);
            walk_next(n2, kTilesPerWarp, step, ntiles, gpr);
            if (n2.t < ntiles)
                offs_next = tile_offsets_load32(v, n2.t);
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
                uint16_t *dst = out + (int64_t(cur.rb) * kTileRows + r) * v.cols + int64_t(cur.kg) * kGroup + c * 8;
                *reinterpret_cast<uint4 *>(dst) = val;
            }
        }
        __syncwarp();
        cur = nxt;
        nxt = n2;
    }
}

template <int W>
uw_status launch_decompress_w(const BlobView &v, uint16_t *w_out, uint32_t *status, int64_t grid, size_t min_smem,
                              cudaStream_t stream) {
    size_t smem = size_t(kCommonSmemBytes) + size_t(W) * (2 * size_t(v.tbuf) + kOutBufBytes);
    smem = smem < min_smem ? min_smem : smem;
    if (!ensure_smem(decompress_kernel<W>, smem))
        return UW_ERR_CUDA;
    return launch_overlapped(decompress_kernel<W>, dim3(unsigned(grid)), dim3(W * 32), smem, stream, v, w_out,
                             status) == cudaSuccess
               ? UW_OK
               : UW_ERR_CUDA;
}

}  // namespace

uw_status launch_decompress(const BlobView &v, uint16_t *w_out, uint32_t *status, cudaStream_t stream, int max_ctas) {
    const int64_t per_cta = int64_t(kDecompWarps) * kTilesPerWarp;
    const int64_t grid = (int64_t(v.ntiles) + per_cta - 1) / per_cta;
    if (max_ctas <= 0 || max_ctas >= grid)
        return launch_decompress_w<kDecompWarps>(v, w_out, status, grid, 0, stream);
    // capped: persistent CTAs of 16 warps, each holding an SM to itself
    const int64_t per_split = int64_t(kDecompWarpsSplit) * kTilesPerWarp;
    const int64_t g = std::min<int64_t>(max_ctas, (int64_t(v.ntiles) + per_split - 1) / per_split);
    return launch_decompress_w<kDecompWarpsSplit>(v, w_out, status, g, kExclusiveSmem, stream);
}

}  // namespace uw
