// Decompress a blob back to BF16 weights in HBM (the Unweight blog's "full
// decode" pipeline: the restored matrix can then go to any GEMM).
//
// Persistent CTAs, one per SM: each CTA builds the pair table once and
// replicates it into 32 lane-private copies (entry w of copy l at word
// 32*w + l), so every lookup of the decode loop is one shared-memory
// wavefront whatever the 32 lanes' windows are.  Each warp then walks runs
// of consecutive tiles with the shared tile decoder (decode.cuh); a tile's
// sign+mantissa bytes are prefetched into L2 two tiles ahead and loaded
// into registers one tile ahead.  Lane j produces the 64 BF16 weights of
// row j; they pass through a per-warp 4 KB shared-memory buffer (16-byte
// chunks XOR-swizzled by row, conflict-free both ways) so that the global
// stores are coalesced 128-byte row segments.
#include "decode.cuh"
#include "kernels.h"

namespace uw {

namespace {

constexpr int kDecompMaxWarps = 16;
constexpr int kTilesPerWarp = 4;
constexpr int kOutBufBytes = kTileRows * kGroup * 2;  // 4096

// Shared memory of a CTA of nw warps: [32 private table copies][common
// tables][nw x 2 tile buffers][nw x output buffer].
size_t decompress_smem(int nw, uint32_t tbuf) {
    return size_t(kPrivateLutBytes) + size_t(kCommonSmemBytes) + size_t(nw) * (2 * size_t(tbuf) + kOutBufBytes);
}

__global__ void __launch_bounds__(kDecompMaxWarps * 32, 1)
    decompress_kernel(const BlobView v, uint16_t *__restrict__ out, uint32_t *status) {
    extern __shared__ __align__(16) unsigned char smem[];
    grid_dep_launch();
    const uint32_t nw = blockDim.x >> 5;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t priv = smem_addr(smem);
    unsigned char *common = smem + kPrivateLutBytes;
    const DecodeShared ds = carve_common(common);
    const uint32_t lut = priv + 4u * uint32_t(lane);  // this lane's copy
    const uint32_t tbuf = v.tbuf;
    uint4 *obuf = reinterpret_cast<uint4 *>(common + kCommonSmemBytes + size_t(nw) * 2 * tbuf +
                                            size_t(warp) * kOutBufBytes);

    const uint32_t gpr = v.gpr, ntiles = v.ntiles;
    const uint32_t step = gridDim.x * nw * uint32_t(kTilesPerWarp);
    const uint64_t first = (uint64_t(blockIdx.x) * nw + warp) * kTilesPerWarp;
    TileWalk cur, nxt;
    walk_seek(cur, first < ntiles ? uint32_t(first) : ntiles, gpr);
    nxt = cur;
    walk_next(nxt, kTilesPerWarp, step, ntiles, gpr);
    TileMeta meta{};
    uint4 smn[4];
    uint32_t offs_next = 0;
    const uint32_t cbuf0 = smem_addr(common + kCommonSmemBytes + size_t(warp) * 2 * tbuf);
    if (cur.t < ntiles) {
        tile_fetch(v, tile_loc32(v, cur.rb, cur.kg, cur.t), tile_offsets_load32(v, cur.t), cbuf0, meta, smn);
        if (nxt.t < ntiles) {
            offs_next = tile_offsets_load32(v, nxt.t);
            tile_prefetch_sm_l2(tile_loc32(v, nxt.rb, nxt.kg, nxt.t));
        }
    }
    build_tables(ds, v);
    __syncthreads();
    replicate_private(ds, priv);  // while the first tiles' copies fly
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
        const uint32_t esc_mask = tile_begin<kShiftPrivate>(ds, meta, R, cbuf, ls, status);
        const uint32_t ebase = escape_base(meta, cbuf);
        TileWalk n2 = nxt;
        if (nxt.t < ntiles) {
            tile_fetch(v, tile_loc32(v, nxt.rb, nxt.kg, nxt.t), offs_next, cbuf0 + ((i + 1) & 1u) * tbuf, meta, smn);
            walk_next(n2, kTilesPerWarp, step, ntiles, gpr);
            if (n2.t < ntiles) {
                offs_next = tile_offsets_load32(v, n2.t);
                // its sign+mantissa bytes go to registers one tile from now:
                // have L2 hold them by then
                tile_prefetch_sm_l2(tile_loc32(v, n2.rb, n2.kg, n2.t));
            }
        }
        uint32_t q[4];
#pragma unroll
        for (int I = 0; I < 32; I++) {
            q[I & 3] = decode_pair<kShiftPrivate>(ls, lut, I, sm_word(sm, I >> 1));
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

}  // namespace

uw_status launch_decompress(const BlobView &v, uint16_t *w_out, uint32_t *status, cudaStream_t stream, int max_ctas) {
    // as many warps as the shared memory holds beside the private tables
    // (tile buffers are at most 2112 bytes, so at least 11)
    int nw = kDecompMaxWarps;
    while (nw > 1 && decompress_smem(nw, v.tbuf) > size_t(kMaxSmemPerBlock))
        nw--;
    const size_t smem = decompress_smem(nw, v.tbuf);
    if (smem > size_t(kMaxSmemPerBlock))
        return UW_ERR_INTERNAL;
    const int64_t per_cta = int64_t(nw) * kTilesPerWarp;
    int64_t grid = std::min<int64_t>(sm_count(), (int64_t(v.ntiles) + per_cta - 1) / per_cta);
    if (max_ctas > 0)  // capped: the SM share of a decode running beside a matmul
        grid = std::min<int64_t>(grid, max_ctas);
    grid = std::max<int64_t>(grid, 1);
    // more than half of an SM's shared memory: every CTA holds an SM alone
    if (!ensure_smem(decompress_kernel, smem))
        return UW_ERR_CUDA;
    return launch_overlapped(decompress_kernel, dim3(unsigned(grid)), dim3(unsigned(nw) * 32u), smem, stream, v,
                             w_out, status) == cudaSuccess
               ? UW_OK
               : UW_ERR_CUDA;
}

}  // namespace uw
