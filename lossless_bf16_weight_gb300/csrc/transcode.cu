// Transcode a blob's Huffman-coded exponents into one of two intermediate
// forms (the Unweight blog's paragraph on the four execution pipelines):
//   * palette-4: the 4-bit palette index of every weight (the palette
//     pipelines: at run time, a quarter of the bytes a full decode writes, or
//     once when the model is loaded; paragraph on the palette format at model
//     load);
//   * exponents: the exponent byte of every weight, escaped groups included
//     (the exponent-only pipeline: half the bytes a full decode writes),
//     laid out like the sign+mantissa section: chunk c (weights 16c..16c+15)
//     of group q at byte 64*q0 + (c*R + j)*16.
//
// Palette-4 layout (half the width of the sign+mantissa section): group q = 32*rb*gpr
// + R*kg + j (row j of row block rb, R rows in the block) owns 32 bytes in
// two 16-byte chunks; chunk c (weights 32c .. 32c+31) sits at byte
// 32*q0 + (c*R + j)*16, q0 = 32*rb*gpr + R*kg the tile's first group, and
// weight 32c + 2i + b is nibble b (0 = low) of byte i.  Escaped groups hold
// index 0: their exponents stay in the blob's escape section.
//
// Persistent CTAs, one per SM, each with the pair table (whose entries carry
// palette indices or exponents) replicated into 32 lane-private copies, so
// that every lookup is one shared-memory wavefront.  Each warp walks runs of
// consecutive tiles with the shared tile decoder (decode.cuh); lane j packs
// row j's 64 indices into 32 bytes (or its 64 exponents into 64 bytes) and
// stores its chunks (32 lanes x 16 bytes = 512 contiguous bytes per store).
#include "decode.cuh"
#include "kernels.h"

namespace uw {

namespace {

constexpr int kTcdWarps = 16;
constexpr int kTcdTilesPerWarp = 4;

// Shared memory: [32 private table copies][common tables][W x 2 tile buffers].
size_t transcode_smem(uint32_t tbuf) {
    return size_t(kPrivateLutBytes) + size_t(kCommonSmemBytes) + size_t(kTcdWarps) * 2 * size_t(tbuf);
}

template <bool kP4>
__global__ void __launch_bounds__(kTcdWarps * 32, 1)
    transcode_kernel(const BlobView v, uint8_t *__restrict__ out, uint32_t *status) {
    constexpr int W = kTcdWarps;
    extern __shared__ __align__(16) unsigned char smem[];
    grid_dep_launch();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t priv = smem_addr(smem);
    unsigned char *common = smem + kPrivateLutBytes;
    const DecodeShared ds = carve_common(common);
    const uint32_t lut = priv + 4u * uint32_t(lane);  // this lane's copy
    const uint32_t tbuf = v.tbuf;
    const uint32_t cbuf0 = smem_addr(common + kCommonSmemBytes + size_t(warp) * 2 * tbuf);

    const uint32_t gpr = v.gpr, ntiles = v.ntiles;
    const uint32_t step = gridDim.x * uint32_t(W * kTcdTilesPerWarp);
    const uint64_t first = (uint64_t(blockIdx.x) * W + warp) * kTcdTilesPerWarp;
    TileWalk cur, nxt;
    walk_seek(cur, first < ntiles ? uint32_t(first) : ntiles, gpr);
    nxt = cur;
    walk_next(nxt, kTcdTilesPerWarp, step, ntiles, gpr);
    TileMeta meta{};
    uint32_t offs_next = 0;
    if (cur.t < ntiles) {
        tile_fetch_codes(v, tile_loc32(v, cur.rb, cur.kg, cur.t), tile_offsets_load32(v, cur.t), cbuf0, meta);
        if (nxt.t < ntiles)
            offs_next = tile_offsets_load32(v, nxt.t);
    }
    if constexpr (kP4)
        build_tables_palette_index(ds, v);
    else
        build_tables(ds, v);
    __syncthreads();
    replicate_private(ds, priv);  // while the first tiles' copies fly
    __syncthreads();
    grid_dep_wait();  // the output may still be read by the kernel before

    for (uint32_t i = 0; cur.t < ntiles; i++) {
        const int R = tile_rows32(v, cur.rb);
        const uint32_t cbuf = cbuf0 + (i & 1u) * tbuf;
        LaneStream ls;
        const uint32_t esc_mask = tile_begin(ds, meta, R, cbuf, ls, status);
        const uint32_t ebase = escape_base(meta, cbuf);  // before meta is reused for the next tile
        TileWalk n2 = nxt;
        if (nxt.t < ntiles) {
            tile_fetch_codes(v, tile_loc32(v, nxt.rb, nxt.kg, nxt.t), offs_next, cbuf0 + ((i + 1) & 1u) * tbuf, meta);
            walk_next(n2, kTcdTilesPerWarp, step, ntiles, gpr);
            if (n2.t < ntiles)
                offs_next = tile_offsets_load32(v, n2.t);
        }
        const uint64_t q0 = uint64_t(kTileRows) * cur.rb * gpr + uint64_t(R) * cur.kg;
        if constexpr (kP4) {
            uint32_t wd[8];
#pragma unroll
            for (int k = 0; k < 8; k++)
                wd[k] = 0u;
#pragma unroll
            for (int I = 0; I < 32; I++) {
                const uint32_t ent = decode_entry<kStridePrivate>(ls, lut, I);
                const uint32_t byte = ((ent >> 7) & 15u) | ((ent >> 19) & 0xF0u);  // weights 2I (low), 2I+1
                wd[I >> 2] |= byte << (8 * (I & 3));
            }
            tile_check(ls, status);
            if ((esc_mask >> lane) & 1u) {
#pragma unroll
                for (int k = 0; k < 8; k++)
                    wd[k] = 0u;
            }
            if (lane < R) {
                uint8_t *dst = out + 32 * q0 + 16 * lane;
                *reinterpret_cast<uint4 *>(dst) = make_uint4(wd[0], wd[1], wd[2], wd[3]);
                *reinterpret_cast<uint4 *>(dst + 16 * R) = make_uint4(wd[4], wd[5], wd[6], wd[7]);
            }
        } else {
            uint32_t wd[16];
#pragma unroll
            for (int k = 0; k < 16; k++)
                wd[k] = 0u;
#pragma unroll
            for (int I = 0; I < 32; I++) {
                const uint32_t ent = decode_entry<kStridePrivate>(ls, lut, I);
                const uint32_t two = ((ent >> 7) & 0xFFu) | ((ent >> 15) & 0xFF00u);  // exponents of 2I, 2I+1
                wd[I >> 1] |= two << (16 * (I & 1));
            }
            tile_check(ls, status);
            uint4 q[4];
#pragma unroll
            for (int c = 0; c < 4; c++)
                q[c] = make_uint4(wd[4 * c], wd[4 * c + 1], wd[4 * c + 2], wd[4 * c + 3]);
            if ((esc_mask >> lane) & 1u)  // the raw exponents, already in weight order
                escape_read(ebase, esc_mask, q);
            if (lane < R) {
                uint8_t *dst = out + 64 * q0 + 16 * lane;
#pragma unroll
                for (int c = 0; c < 4; c++)
                    *reinterpret_cast<uint4 *>(dst + 16 * c * R) = q[c];
            }
        }
        cur = nxt;
        nxt = n2;
    }
}

}  // namespace

uw_status launch_transcode(const BlobView &v, uint8_t *out, bool palette4, uint32_t *status, cudaStream_t stream,
                           int max_ctas) {
    const size_t smem = transcode_smem(v.tbuf);  // tile buffers are at most 2112 bytes: 198 KB at most
    if (smem > size_t(kMaxSmemPerBlock))
        return UW_ERR_INTERNAL;
    const int64_t per_cta = int64_t(kTcdWarps) * kTcdTilesPerWarp;
    int64_t grid = std::min<int64_t>(sm_count(), (int64_t(v.ntiles) + per_cta - 1) / per_cta);
    if (max_ctas > 0)  // capped: the SM share of a transcode running beside a matmul
        grid = std::min<int64_t>(grid, max_ctas);
    grid = std::max<int64_t>(grid, 1);
    // more than half of an SM's shared memory: every CTA holds an SM alone
    auto kern = palette4 ? transcode_kernel<true> : transcode_kernel<false>;
    if (!ensure_smem(kern, smem))
        return UW_ERR_CUDA;
    return launch_overlapped(kern, dim3(unsigned(grid)), dim3(kTcdWarps * 32), smem, stream, v, out, status) ==
                   cudaSuccess
               ? UW_OK
               : UW_ERR_CUDA;
}

}  // namespace uw
