// Batch-1 GEMV with the activation vector held in registers ("column" CTAs),
// y = x W^T, fp32 accumulation.
//
// A CTA of W warps covers W consecutive 64-column groups (warp w owns group
// kg0 + w) of a range of 32-row blocks.  The CTA's x values sit in shared
// memory as BF16 pairs (one broadcast load per step serves both tiles).
// Each warp walks down its column two tiles at a time (row blocks rb and
// rb+1), interleaving the two tiles step by step so that every lane runs two
// independent dependency chains:
//   * compressed source: each tile is decoded on chip (decode.cuh) and each
//     BF16 weight pair is multiplied straight from the register it was
//     rebuilt in -- the weights never exist in memory (Unweight blog,
//     paragraphs on the reconstructive matmul and on decompressing into
//     fast on-chip memory);
//   * bf16 source: the same warps load the uncompressed weights.
// Both share this body, so the results are bit-identical.  Products use the
// mixed-precision fma.rn.f32.bf16 (BF16 x BF16 is exact in fp32, so each
// step is one correctly rounded fp32 add of the exact product).
//
// Loads run one tile pair ahead: code regions and escaped groups' raw
// exponents by cp.async into the warp's second pair of shared buffers; glen
// and the sign+mantissa bytes into registers.
//
// Order of the sum for output n (row j of block rb):
//   tile partial  = acc_even + acc_odd       (k even / odd within the group)
//   CTA partial   = ((p(kg0) + p(kg0+1)) + p(kg0+2)) + ...   over its W groups
//   y             = ((split0 + split1) + split2) + ...       split s = CTA column s
// then round to nearest even BF16.
#include <cuda_bf16.h>

#include "decode.cuh"
#include "kernels.h"

namespace uw {

namespace {

__device__ __forceinline__ void fma_bf16x2(float &a0, float &a1, uint32_t w, uint32_t x) {
    asm("{\n\t.reg .b16 wl, wh, xl, xh;\n\t"
        "mov.b32 {wl, wh}, %2;\n\t"
        "mov.b32 {xl, xh}, %3;\n\t"
        "fma.rn.f32.bf16 %0, wl, xl, %0;\n\t"
        "fma.rn.f32.bf16 %1, wh, xh, %1;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "r"(w), "r"(x));
}

__device__ __forceinline__ void prefetch_bf16_row(const GemvParams &p, int64_t rb, int64_t kg) {
    const int lane = threadIdx.x & 31;
    const int64_t n = rb * kTileRows + lane;
    if (n < p.rows)
        asm volatile("prefetch.global.L2 [%0];" :: "l"(p.w + n * p.cols + kg * kGroup));
}

// The two accumulators of an escaped group's lane, rebuilt from its raw
// exponent bytes (rare; kept out of line so that it costs the hot loop no
// registers, so the sign+mantissa bytes are loaded again).
__device__ __noinline__ float2 escaped_tile_sum(uint32_t ebase, uint32_t em, const TileLoc &L, uint32_t xw) {
    uint4 e[4], sm[4];
    escape_read(ebase, em, e);
    tile_sm_load(L, sm);
    float b0 = 0.f, b1 = 0.f;
#pragma unroll
    for (int I = 0; I < 32; I++)
        fma_bf16x2(b0, b1, escape_pair(e, I, sm_word(sm, I >> 1)), lds32(xw + 4 * I));
    return make_float2(b0, b1);
}

template <int W, bool kCompressed>
__device__ __forceinline__ void gemv_col_body(const GemvParams &p, int rb_per_cta) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t gpr = p.cols / kGroup;
    const int64_t nrb = (p.rows + kTileRows - 1) / kTileRows;
    const int64_t rb0 = int64_t(blockIdx.x) * rb_per_cta;
    const int64_t rb1 = rb0 + rb_per_cta < nrb ? rb0 + rb_per_cta : nrb;
    const int split = blockIdx.y;
    const int64_t kg = int64_t(split) * W + warp;
    const bool active = kg < gpr;
    const TileMeta empty = {0u, 0u, 0u};

    // shared memory: [common tables][x slab W x 32 pairs][per warp 4 code buffers]
    // [tile partials rb_per_cta x W x 32]
    size_t off = 0;
    DecodeShared ds{};
    if (kCompressed) {
        ds = carve_common(smem);
        off = kCommonSmemBytes;
    }
    uint32_t *xs = reinterpret_cast<uint32_t *>(smem + off);
    off += size_t(W) * 32 * 4;
    const uint32_t xw = smem_addr(xs + warp * 32);
    uint32_t cb0 = 0;  // warp's four code buffers: pair parity x (A, B)
    if (kCompressed) {
        cb0 = smem_addr(smem + off + size_t(warp) * 4 * kCodeBufBytes);
        off += size_t(W) * 4 * kCodeBufBytes;
    }
    float *red = reinterpret_cast<float *>(smem + off);  // [rb_per_cta][W][32]

    for (int i = threadIdx.x; i < W * 32; i += blockDim.x) {
        const int64_t g = int64_t(split) * W + (i >> 5);
        const uint16_t *xp = p.x + g * kGroup + 2 * (i & 31);
        xs[i] = g < gpr ? (uint32_t(xp[0]) | (uint32_t(xp[1]) << 16)) : 0u;
    }

    const int64_t ntile = active ? rb1 - rb0 : 0;
    const int64_t npair = (ntile + 1) / 2;
    TileMeta mA = empty, mB = empty;
    uint32_t offA = 0, offB = 0;  // offsets of the next pair to fetch
    uint4 nsmA[4], nsmB[4];  // sign+mantissa bytes of the next pair
#pragma unroll
    for (int c = 0; c < 4; c++) {
        nsmA[c] = make_uint4(0, 0, 0, 0);
        nsmB[c] = make_uint4(0, 0, 0, 0);
    }
    if (kCompressed && npair > 0) {
        tile_fetch(p.v, tile_loc(p.v, rb0, kg, gpr), tile_offsets_load(p.v, rb0 * gpr + kg), cb0, mA, nsmA);
        if (ntile > 1)
            tile_fetch(p.v, tile_loc(p.v, rb0 + 1, kg, gpr), tile_offsets_load(p.v, (rb0 + 1) * gpr + kg),
                       cb0 + kCodeBufBytes, mB, nsmB);
        if (ntile > 2)
            offA = tile_offsets_load(p.v, (rb0 + 2) * gpr + kg);
        if (ntile > 3)
            offB = tile_offsets_load(p.v, (rb0 + 3) * gpr + kg);
    } else if (!kCompressed && npair > 0) {
        prefetch_bf16_row(p, rb0, kg);
        if (ntile > 1)
            prefetch_bf16_row(p, rb0 + 1, kg);
    }
    if (kCompressed)
        build_tables(ds, p.v);
    __syncthreads();

#pragma unroll 1
    for (int64_t i = 0; i < npair; i++) {
        const int64_t rbA = rb0 + 2 * i, rbB = rbA + 1;
        const bool hasB = rbB < rb1;
        float aA0 = 0.f, aA1 = 0.f, aB0 = 0.f, aB1 = 0.f;
        if (kCompressed) {
            const int RA = tile_rows(p.v, rbA);
            const int RB = hasB ? tile_rows(p.v, rbB) : 0;  // no tile B: every lane decodes zeros
            const uint32_t bufA = cb0 + uint32_t(i & 1) * 2 * kCodeBufBytes, bufB = bufA + kCodeBufBytes;
            uint4 smA[4], smB[4];  // this pair's sign+mantissa bytes, loaded during the previous pair
#pragma unroll
            for (int c = 0; c < 4; c++) {
                smA[c] = nsmA[c];
                smB[c] = nsmB[c];
            }
            LaneStream la, lb;
            const uint32_t emA = tile_begin(ds, mA, RA, bufA, la, p.status);
            const uint32_t emB = tile_begin(ds, mB, RB, bufB, lb, p.status);
            const uint32_t ebA = escape_base(mA, bufA), ebB = escape_base(mB, bufB);
            // fetch the next pair while this one is decoded
            if (i + 1 < npair) {
                const uint32_t nA = cb0 + uint32_t((i + 1) & 1) * 2 * kCodeBufBytes;
                tile_fetch(p.v, tile_loc(p.v, rbA + 2, kg, gpr), offA, nA, mA, nsmA);
                if (rbB + 2 < rb1) {
                    tile_fetch(p.v, tile_loc(p.v, rbB + 2, kg, gpr), offB, nA + kCodeBufBytes, mB, nsmB);
                } else {
                    mB = empty;
#pragma unroll
                    for (int c = 0; c < 4; c++)
                        nsmB[c] = make_uint4(0, 0, 0, 0);
                }
                if (rbA + 4 < rb1)
                    offA = tile_offsets_load(p.v, (rbA + 4) * gpr + kg);
                if (rbB + 4 < rb1)
                    offB = tile_offsets_load(p.v, (rbB + 4) * gpr + kg);
            }
#pragma unroll
            for (int I = 0; I < 32; I++) {
                const uint32_t x2 = lds32(xw + 4 * I);
                fma_bf16x2(aA0, aA1, decode_pair(la, I, sm_word(smA, I >> 1)), x2);
                fma_bf16x2(aB0, aB1, decode_pair(lb, I, sm_word(smB, I >> 1)), x2);
            }
            tile_check(la, p.status);
            tile_check(lb, p.status);
            if (emA | emB) {  // escaped groups: redo those lanes from raw exponents
                if ((emA >> lane) & 1u) {
                    const float2 r = escaped_tile_sum(ebA, emA, tile_loc(p.v, rbA, kg, gpr), xw);
                    aA0 = r.x;
                    aA1 = r.y;
                }
                if ((emB >> lane) & 1u) {
                    const float2 r = escaped_tile_sum(ebB, emB, tile_loc(p.v, rbB, kg, gpr), xw);
                    aB0 = r.x;
                    aB1 = r.y;
                }
            }
        } else {
            if (rbA + 2 < rb1)
                prefetch_bf16_row(p, rbA + 2, kg);
            if (rbB + 2 < rb1)
                prefetch_bf16_row(p, rbB + 2, kg);
            const int64_t nA = rbA * kTileRows + lane, nB = rbB * kTileRows + lane;
            const uint4 *srcA = reinterpret_cast<const uint4 *>(p.w + nA * p.cols + kg * kGroup);
            const uint4 *srcB = reinterpret_cast<const uint4 *>(p.w + (hasB ? nB : nA) * p.cols + kg * kGroup);
            const bool okA = nA < p.rows, okB = hasB && nB < p.rows;
#pragma unroll 1
            for (int q = 0; q < 4; q++) {
                const uint4 wA0 = okA ? __ldg(srcA + 2 * q) : make_uint4(0, 0, 0, 0);
                const uint4 wA1 = okA ? __ldg(srcA + 2 * q + 1) : make_uint4(0, 0, 0, 0);
                const uint4 wB0 = okB ? __ldg(srcB + 2 * q) : make_uint4(0, 0, 0, 0);
                const uint4 wB1 = okB ? __ldg(srcB + 2 * q + 1) : make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int k = 0; k < 8; k++) {
                    const uint32_t x2 = lds32(xw + 4 * (8 * q + k));
                    fma_bf16x2(aA0, aA1, word4(k < 4 ? wA0 : wA1, k & 3), x2);
                    fma_bf16x2(aB0, aB1, word4(k < 4 ? wB0 : wB1, k & 3), x2);
                }
            }
        }
        red[(int(rbA - rb0) * W + warp) * 32 + lane] = aA0 + aA1;
        if (hasB)
            red[(int(rbB - rb0) * W + warp) * 32 + lane] = aB0 + aB1;
    }
    if (!active)
        for (int64_t rb = rb0; rb < rb1; rb++)
            red[(int(rb - rb0) * W + warp) * 32 + lane] = 0.f;
    __syncthreads();

    // CTA partial per (row block, row): sum over the W groups in order.
    const int nsplit = gridDim.y;
    const int nrows_cta = int(rb1 - rb0) * 32;
    for (int t = threadIdx.x; t < nrows_cta; t += blockDim.x) {
        const int rl = t >> 5, j = t & 31;
        float s = red[(rl * W) * 32 + j];
#pragma unroll
        for (int w = 1; w < W; w++)
            s += red[(rl * W + w) * 32 + j];
        const int64_t n = (rb0 + rl) * kTileRows + j;
        if (nsplit == 1) {
            if (n < p.rows)
                p.y[n] = __bfloat16_as_ushort(__float2bfloat16_rn(s));
        } else {
            p.partial[(rb0 + rl) * kTileRows * nsplit + int64_t(split) * kTileRows + j] = s;
        }
    }
    if (nsplit == 1)
        return;
    __threadfence();
    __syncthreads();
    __shared__ int last;
    if (threadIdx.x == 0)
        last = atomicAdd(p.counters + blockIdx.x, 1u) == uint32_t(nsplit - 1);
    __syncthreads();
    if (!last)
        return;
    __threadfence();
    for (int t = threadIdx.x; t < nrows_cta; t += blockDim.x) {
        const int rl = t >> 5, j = t & 31;
        const float *ps = p.partial + (rb0 + rl) * kTileRows * nsplit + j;
        float tot = __ldcg(ps);
        for (int sp = 1; sp < nsplit; sp++)
            tot += __ldcg(ps + sp * kTileRows);
        const int64_t n = (rb0 + rl) * kTileRows + j;
        if (n < p.rows)
            p.y[n] = __bfloat16_as_ushort(__float2bfloat16_rn(tot));
    }
    if (threadIdx.x == 0)
        p.counters[blockIdx.x] = 0;
}

template <int W, bool kCompressed>
__global__ void __launch_bounds__(W * 32, col_blocks_per_sm(W)) gemv_kg_kernel(const GemvParams p, int rb_per_cta) {
    gemv_col_body<W, kCompressed>(p, rb_per_cta);
}

template <int W, bool kCompressed>
uw_status launch_kg_one(const GemvParams &p, int rb_per_cta, cudaStream_t stream) {
    const size_t smem = gemv_kg_smem_bytes(W, rb_per_cta, kCompressed);
    auto kern = gemv_kg_kernel<W, kCompressed>;
    if (!ensure_smem(kern, smem))
        return UW_ERR_CUDA;
    const int64_t nrb = (p.rows + kTileRows - 1) / kTileRows;
    const int64_t gpr = p.cols / kGroup;
    const dim3 grid(unsigned((nrb + rb_per_cta - 1) / rb_per_cta), unsigned((gpr + W - 1) / W));
    kern<<<grid, dim3(W * 32), smem, stream>>>(p, rb_per_cta);
    return cudaGetLastError() == cudaSuccess ? UW_OK : UW_ERR_CUDA;
}

}  // namespace

size_t gemv_kg_smem_bytes(int warps, int rb_per_cta, bool compressed) {
    size_t s = compressed ? size_t(kCommonSmemBytes) + size_t(warps) * 4 * kCodeBufBytes : 0;
    return s + size_t(warps) * 32 * 4 + size_t(rb_per_cta) * warps * 32 * 4;
}

uw_status launch_gemv_kg(const GemvParams &p, int warps, int rb_per_cta, bool compressed, cudaStream_t stream) {
    if (p.batch != 1 || rb_per_cta < 1)
        return UW_ERR_UNSUPPORTED;
    if (gemv_kg_smem_bytes(warps, rb_per_cta, compressed) > size_t(kMaxSmemPerBlock))
        return UW_ERR_UNSUPPORTED;
    switch (warps) {
        case 4: return compressed ? launch_kg_one<4, true>(p, rb_per_cta, stream)
                                  : launch_kg_one<4, false>(p, rb_per_cta, stream);
        case 8: return compressed ? launch_kg_one<8, true>(p, rb_per_cta, stream)
                                  : launch_kg_one<8, false>(p, rb_per_cta, stream);
        case 16: return compressed ? launch_kg_one<16, true>(p, rb_per_cta, stream)
                                   : launch_kg_one<16, false>(p, rb_per_cta, stream);
    }
    return UW_ERR_UNSUPPORTED;
}

}  // namespace uw
