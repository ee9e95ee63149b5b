// CUDA-core GEMV / small-batch GEMM, y = x W^T, fp32 accumulation.
//
// Two weight sources share one kernel body and therefore one accumulation
// order, so that the results are bit-identical:
//   * compressed: each warp decodes tiles of the blob on chip (decode.cuh)
//     and multiplies the BF16 pairs straight from registers -- the weights
//     never exist in memory (Unweight blog, paragraphs on the reconstructive
//     matmul and on decompressing into fast on-chip memory);
//   * bf16: the same warps load the uncompressed weights.
//
// Work split: a CTA owns one block of 32 rows (lane j = row j) and one of
// `splits` contiguous ranges of 64-column groups; its W warps take
// contiguous sub-ranges.  Each lane keeps two fp32 accumulators per batch
// row (even and odd k, one packed FFMA2 per weight pair).  Order of the
// final sum for output (b, n):
//   warp partial  = acc_even + acc_odd
//   CTA partial   = ((warp0 + warp1) + warp2) + ...
//   y             = ((split0 + split1) + split2) + ...   (last CTA sums)
// then round to nearest even BF16.
#include <cuda_bf16.h>

#include "decode.cuh"
#include "kernels.h"

namespace uw {

namespace {

__device__ __forceinline__ float2 pair_to_float2(uint32_t pair) {
    return make_float2(__uint_as_float(pair << 16), __uint_as_float(pair & 0xFFFF0000u));
}

// Pair I (weights 2I, 2I+1 of the lane's group) times the x slab, BP rows.
template <int BP>
__device__ __forceinline__ void fma_pair(uint32_t pair, int I, const float *xk, float4 (&x4)[BP],
                                         float2 (&acc)[BP]) {
    const float2 wv = pair_to_float2(pair);
    if ((I & 1) == 0) {
#pragma unroll
        for (int b = 0; b < BP; b++)
            x4[b] = *reinterpret_cast<const float4 *>(xk + ((I >> 1) * BP + b) * 4);
    }
#pragma unroll
    for (int b = 0; b < BP; b++) {
        const float2 xv = (I & 1) ? make_float2(x4[b].z, x4[b].w) : make_float2(x4[b].x, x4[b].y);
        acc[b] = __ffma2_rn(wv, xv, acc[b]);
    }
}

template <int W, int BP, bool kCompressed>
__device__ __forceinline__ void gemv_body(const GemvParams &p) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t gpr = p.cols / kGroup;
    const int64_t rb = blockIdx.x / p.splits;
    const int split = int(blockIdx.x - rb * p.splits);
    const int64_t kg_lo = gpr * split / p.splits, kg_hi = gpr * (split + 1) / p.splits;
    const int64_t nk = kg_hi - kg_lo;
    const int64_t w_lo = kg_lo + nk * warp / W, w_hi = kg_lo + nk * (warp + 1) / W;
    const int64_t left = p.rows - rb * kTileRows;
    const int R = left < kTileRows ? int(left) : kTileRows;

    size_t off = 0;
    DecodeShared ds{};
    uint32_t *wbuf = nullptr;
    if (kCompressed) {
        ds = carve_common(smem);
        off = kCommonSmemBytes;
        wbuf = reinterpret_cast<uint32_t *>(smem + off + size_t(warp) * 2 * p.v.tbuf);
        off += size_t(W) * 2 * p.v.tbuf;
    }
    float *xs = reinterpret_cast<float *>(smem + off);
    off += size_t(nk) * kGroup * BP * 4;
    float *red = reinterpret_cast<float *>(smem + off);

    // Start the first tile's loads before the shared tables are built.
    TileMeta meta{};
    uint4 smn[4];
    uint32_t offs_next = 0;
    uint4 wcur[8], wnext[8];
    const uint32_t cbuf0 = kCompressed ? smem_addr(wbuf) : 0u;
    if (kCompressed) {
        if (w_lo < w_hi) {
            tile_fetch(p.v, tile_loc(p.v, rb, w_lo, gpr), tile_offsets_load(p.v, rb * gpr + w_lo), cbuf0, meta,
                       smn);
            if (w_lo + 1 < w_hi)
                offs_next = tile_offsets_load(p.v, rb * gpr + w_lo + 1);
        }
    } else {
        grid_dep_wait();  // the weights may come from the kernel before (decompress)
        const uint16_t *src = p.w + (rb * kTileRows + lane) * p.cols + w_lo * kGroup;
#pragma unroll
        for (int c = 0; c < 8; c++)
            wnext[c] = (lane < R && w_lo < w_hi) ? __ldg(reinterpret_cast<const uint4 *>(src) + c)
                                                 : make_uint4(0, 0, 0, 0);
    }

    if (kCompressed) {
        build_tables(ds, p.v);
        grid_dep_wait();  // x may come from the kernel before
    }
    // x slab: xs[((kk >> 2) * BP + b) * 4 + (kk & 3)] = x[b, 64*kg_lo + kk]
    const int64_t nkk = nk * kGroup;
    for (int64_t i = threadIdx.x; i < nkk * BP; i += blockDim.x) {
        const int b = int(i / nkk);
        const int64_t kk = i - b * nkk;
        float xv = 0.f;
        if (b < p.batch) {
            const uint16_t bits = p.x[b * p.cols + kg_lo * kGroup + kk];
            xv = __uint_as_float(uint32_t(bits) << 16);
        }
        xs[((kk >> 2) * BP + b) * 4 + (kk & 3)] = xv;
    }
    __syncthreads();
    const uint32_t lut = kCompressed ? smem_addr(ds.lut) : 0u;

    float2 acc[BP];
#pragma unroll
    for (int b = 0; b < BP; b++)
        acc[b] = make_float2(0.f, 0.f);

    for (int64_t kg = w_lo; kg < w_hi; kg++) {
        const int64_t t = rb * gpr + kg;
        const float *xk = xs + (kg - kg_lo) * kGroup * BP;
        float4 x4[BP];
        if (kCompressed) {
            const uint32_t cbuf = cbuf0 + uint32_t((kg - w_lo) & 1) * p.v.tbuf;
            uint4 sm[4];
#pragma unroll
            for (int c = 0; c < 4; c++)
                sm[c] = smn[c];
            LaneStream ls;
            const uint32_t esc_mask = tile_begin(ds, meta, R, cbuf, ls, p.status);
            const uint32_t ebase = escape_base(meta, cbuf);
            if (kg + 1 < w_hi) {
                tile_fetch(p.v, tile_loc(p.v, rb, kg + 1, gpr), offs_next,
                           cbuf0 + uint32_t((kg + 1 - w_lo) & 1) * p.v.tbuf, meta, smn);
                if (kg + 2 < w_hi)
                    offs_next = tile_offsets_load(p.v, t + 2);
            }
            float2 saved[BP];
#pragma unroll
            for (int b = 0; b < BP; b++)
                saved[b] = acc[b];
#pragma unroll
            for (int I = 0; I < 32; I++) {
                const uint32_t pair = decode_pair(ls, lut, I, sm_word(sm, I >> 1));
                fma_pair<BP>(pair, I, xk, x4, acc);
            }
            tile_check(ls, p.status);
            if (esc_mask) {  // escaped groups: redo those lanes from raw exponents
                if ((esc_mask >> lane) & 1u) {
                    uint4 e[4];
                    escape_read(ebase, esc_mask, e);
#pragma unroll
                    for (int b = 0; b < BP; b++)
                        acc[b] = saved[b];
#pragma unroll
                    for (int I = 0; I < 32; I++)
                        fma_pair<BP>(escape_pair(e, I, sm_word(sm, I >> 1)), I, xk, x4, acc);
                }
            }
        } else {
#pragma unroll
            for (int c = 0; c < 8; c++)
                wcur[c] = wnext[c];
            if (kg + 1 < w_hi) {
                const uint16_t *src = p.w + (rb * kTileRows + lane) * p.cols + (kg + 1) * kGroup;
#pragma unroll
                for (int c = 0; c < 8; c++)
                    wnext[c] = lane < R ? __ldg(reinterpret_cast<const uint4 *>(src) + c) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int I = 0; I < 32; I++) {
                const uint4 &q = wcur[I >> 2];
                const uint32_t pair = (I & 3) == 0 ? q.x : (I & 3) == 1 ? q.y : (I & 3) == 2 ? q.z : q.w;
                fma_pair<BP>(pair, I, xk, x4, acc);
            }
        }
    }

    // Reduction in a fixed order (see file comment).
#pragma unroll
    for (int b = 0; b < BP; b++)
        red[(warp * BP + b) * 32 + lane] = acc[b].x + acc[b].y;
    __syncthreads();
    const int tid = threadIdx.x;
    const int b = tid >> 5, j = tid & 31;
    float s = 0.f;
    if (tid < BP * 32) {
        s = red[b * 32 + j];
#pragma unroll
        for (int w = 1; w < W; w++)
            s += red[(w * BP + b) * 32 + j];
    }
    const int64_t n = rb * kTileRows + j;
    if (p.splits == 1) {
        if (tid < BP * 32 && b < p.batch && j < R)
            p.y[b * p.rows + n] = __bfloat16_as_ushort(__float2bfloat16_rn(s));
        return;
    }
    if (tid < BP * 32)
        p.partial[((rb * p.splits + split) * BP + b) * 32 + j] = s;
    __threadfence();
    __syncthreads();
    __shared__ int last;
    if (tid == 0)
        last = atomicAdd(p.counters + rb, 1u) == uint32_t(p.splits - 1);
    __syncthreads();
    if (!last)
        return;
    __threadfence();
    if (tid < BP * 32) {
        float tot = __ldcg(p.partial + (rb * p.splits * BP + b) * 32 + j);
        for (int sp = 1; sp < p.splits; sp++)
            tot += __ldcg(p.partial + ((rb * p.splits + sp) * BP + b) * 32 + j);
        if (b < p.batch && j < R)
            p.y[b * p.rows + n] = __bfloat16_as_ushort(__float2bfloat16_rn(tot));
    }
    if (tid == 0)
        p.counters[rb] = 0;
}

template <int W>
struct Occupancy;
template <>
struct Occupancy<4> { static constexpr int kMinBlocks = 4; };
template <>
struct Occupancy<8> { static constexpr int kMinBlocks = 2; };
template <>
struct Occupancy<16> { static constexpr int kMinBlocks = 1; };

template <int W, int BP, bool kCompressed>
__global__ void __launch_bounds__(W * 32, Occupancy<W>::kMinBlocks) gemv_kernel(const GemvParams p) {
    grid_dep_launch();
    gemv_body<W, BP, kCompressed>(p);
}

template <int W, int BP, bool kCompressed>
uw_status launch_one(const GemvParams &p, size_t smem, cudaStream_t stream) {
    auto kern = gemv_kernel<W, BP, kCompressed>;
    if (!ensure_smem(kern, smem))
        return UW_ERR_CUDA;
    const int64_t nrb = (p.rows + kTileRows - 1) / kTileRows;
    return launch_overlapped(kern, dim3(unsigned(nrb * p.splits)), dim3(W * 32), smem, stream, p) == cudaSuccess
               ? UW_OK
               : UW_ERR_CUDA;
}

template <int W, bool kCompressed>
uw_status launch_bp(const GemvParams &p, int bp, size_t smem, cudaStream_t stream) {
    switch (bp) {
        case 1: return launch_one<W, 1, kCompressed>(p, smem, stream);
        case 2: return launch_one<W, 2, kCompressed>(p, smem, stream);
        case 4: return launch_one<W, 4, kCompressed>(p, smem, stream);
        case 8: return launch_one<W, 8, kCompressed>(p, smem, stream);
        default: return UW_ERR_UNSUPPORTED;
    }
}

}  // namespace

size_t gemv_smem_bytes(int64_t cols, int warps, int splits, int bp, bool compressed, uint32_t tbuf) {
    const int64_t gpr = cols / kGroup;
    const int64_t nk_max = (gpr + splits - 1) / splits;
    size_t s = compressed ? size_t(kCommonSmemBytes) + size_t(warps) * 2 * tbuf : 0;
    s += size_t(nk_max) * kGroup * bp * 4;
    s += size_t(warps) * bp * 32 * 4;
    return s;
}

uw_status launch_gemv(const GemvParams &p, int warps, int bp, bool compressed, cudaStream_t stream) {
    const size_t smem = gemv_smem_bytes(p.cols, warps, p.splits, bp, compressed, p.v.tbuf);
    if (smem > size_t(kMaxSmemPerBlock))
        return UW_ERR_UNSUPPORTED;
    if (compressed) {
        switch (warps) {
            case 4: return launch_bp<4, true>(p, bp, smem, stream);
            case 8: return launch_bp<8, true>(p, bp, smem, stream);
            case 16: return launch_bp<16, true>(p, bp, smem, stream);
        }
    } else {
        switch (warps) {
            case 4: return launch_bp<4, false>(p, bp, smem, stream);
            case 8: return launch_bp<8, false>(p, bp, smem, stream);
            case 16: return launch_bp<16, false>(p, bp, smem, stream);
        }
    }
    return UW_ERR_UNSUPPORTED;
}

}  // namespace uw
