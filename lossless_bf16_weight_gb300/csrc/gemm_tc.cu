// Tensor-core matmul for batches that make it a real contraction,
// y = x W^T with W [rows, cols], x [batch, cols], fp32 accumulation in
// tensor memory, BF16 out.
//
// D = W x^T is computed as tcgen05.mma tiles with M = 128 rows of W (the A
// operand) and N = the batch padded to a multiple of 16 (the B operand),
// K = 16 per instruction.  A CTA owns 128 rows and one of `splits` ranges
// of 64-column groups (one group = one pipeline stage, four MMAs).
//
// Warp roles (CTA of 4G + 1 warps):
//   producers  warps 0 .. 4G-1: warp w fills the A rows 32*(w%4) .. +31 of
//              the stages of K steps i = w/4, w/4 + G, ...  and a quarter of
//              the stage's B rows (x, by cp.async; rows past the batch are
//              zero-filled);
//                * compressed source: each warp decodes its 32 x 64 tile on
//                  chip (decode.cuh) into registers and stores the BF16 rows
//                  into the swizzled stage -- the weights go from the blob to
//                  the tensor cores without touching HBM (Unweight blog,
//                  paragraphs on the reconstructive matmul and on decoding
//                  into shared memory);
//                * bf16 source: the same warps copy the uncompressed rows.
//   MMA warp   warp 4G: one thread waits for each stage, issues its four
//              MMAs and commits them to the stage's "empty" barrier.
//   epilogue   warps 0..3 read the accumulator (tensor-memory lane quarter
//              = warp index) and write y, or fp32 split partials; the last
//              CTA of a row block adds the splits in order.
// Both sources feed the same MMA sequence, so their outputs are
// bit-identical.  Stage s holds A (16 KB) and B (Np x 128 bytes) in the
// 128-byte-swizzled K-major layout of tc.cuh.
#include <cuda_bf16.h>

#include <algorithm>

#include "decode.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace uw {

namespace {

constexpr int kTcM = 128;
constexpr int kTcMaxStages = 8;
constexpr uint32_t kAStageBytes = kTcM * kGroup * 2;  // 16384

// The quarter `qtr` of the stage's x rows: Np/4 rows x 8 chunks of 16 bytes.
__device__ __forceinline__ void load_x_quarter(const TcParams &p, uint32_t b_st, int64_t kg, int qtr, int lane) {
    const int per = p.Np >> 2;
    const int nchunk = per * 8;  // a multiple of 32: Np is a multiple of 16
    for (int t = lane; t < nchunk; t += 32) {
        const int b = qtr * per + (t >> 3), c = t & 7;
        const bool ok = b < p.batch;
        const uint16_t *src = ok ? p.x + int64_t(b) * p.cols + kg * kGroup + 8 * c : p.x;
        cp_async16_zfill(b_st + sw128_offset(uint32_t(b), uint32_t(c)), src, ok ? 16u : 0u);
    }
}

template <int G, bool kCompressed>
__global__ void __launch_bounds__((4 * G + 1) * 32, 1) gemm_tc_kernel(const TcParams p) {
    constexpr int P = 4 * G;  // producer warps
    extern __shared__ unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t bars[2 * kTcMaxStages + 1];
    __shared__ uint32_t tmem_slot;
    __shared__ int last_cta;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = p.S, Np = p.Np;
    const int64_t gpr = p.cols / kGroup;
    const int64_t nrb = (p.rows + kTileRows - 1) / kTileRows;
    const int64_t mb = blockIdx.x;
    const int split = blockIdx.y;
    const int64_t kg_lo = gpr * split / p.splits, kg_hi = gpr * (split + 1) / p.splits;
    const int nk = int(kg_hi - kg_lo);

    // shared memory: [pad to 1024][A stages][B stages][decode tables][code buffers]
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
    const uint32_t a0 = raw + pad;
    const uint32_t bstage = uint32_t(Np) * 128u;
    const uint32_t b0 = a0 + uint32_t(S) * kAStageBytes;
    unsigned char *dec = smem_raw + pad + size_t(S) * (kAStageBytes + bstage);
    const uint32_t full0 = smem_addr(&bars[0]), empty0 = smem_addr(&bars[kTcMaxStages]);
    const uint32_t done = smem_addr(&bars[2 * kTcMaxStages]);

    if (warp == P)
        tmem_alloc(smem_addr(&tmem_slot), p.tmem_cols);
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; s++) {
            mbar_init(full0 + 8u * s, 4);
            mbar_init(empty0 + 8u * s, 1);
        }
        mbar_init(done, 1);
        mbar_init_fence();
    }

    // producer identity: row block rb (of 32 rows), K steps grp, grp + G, ...
    const int rbl = warp & 3, grp = warp >> 2;
    const int64_t rb = mb * 4 + rbl;
    const bool producer = warp < P;
    const bool rb_ok = producer && rb < nrb;
    DecodeShared ds{};
    uint32_t cbuf0 = 0;
    TileMeta meta{0u, 0u, 0u};
    uint4 smn[4];
#pragma unroll
    for (int c = 0; c < 4; c++)
        smn[c] = make_uint4(0, 0, 0, 0);
    uint32_t offs_next = 0;
    if (kCompressed) {
        ds = carve_common(dec);
        cbuf0 = smem_addr(dec + kCommonSmemBytes + size_t(warp) * 2 * p.v.tbuf);
        if (rb_ok && grp < nk) {
            tile_fetch(p.v, tile_loc(p.v, rb, kg_lo + grp, gpr), tile_offsets_load(p.v, rb * gpr + kg_lo + grp),
                       cbuf0, meta, smn);
            if (grp + G < nk)
                offs_next = tile_offsets_load(p.v, rb * gpr + kg_lo + grp + G);
        }
        build_tables(ds, p.v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    const uint32_t lut = kCompressed ? smem_addr(ds.lut) : 0u;

    if (producer) {
        const int64_t left = p.rows - rb * kTileRows;  // rows of this row block (p.v is unset for bf16)
        const int R = !rb_ok ? 0 : left < kTileRows ? int(left) : kTileRows;
        const uint32_t arow = uint32_t(32 * rbl + lane);
        int it = 0;
#pragma unroll 1
        for (int i = grp; i < nk; i += G, it++) {
            const int s = i % S, u = i / S;
            const uint32_t a_st = a0 + uint32_t(s) * kAStageBytes, b_st = b0 + uint32_t(s) * bstage;
            const int64_t kg = kg_lo + i;
            if (kCompressed) {
                uint32_t q[32];
                if (rb_ok) {
                    const uint32_t cbuf = cbuf0 + uint32_t(it & 1) * p.v.tbuf;
                    uint4 sm[4];
#pragma unroll
                    for (int c = 0; c < 4; c++)
                        sm[c] = smn[c];
                    LaneStream ls;
                    const uint32_t em = tile_begin(ds, meta, R, cbuf, ls, p.status);
                    const uint32_t eb = escape_base(meta, cbuf);
                    if (i + G < nk) {
                        tile_fetch(p.v, tile_loc(p.v, rb, kg + G, gpr), offs_next,
                                   cbuf0 + uint32_t((it + 1) & 1) * p.v.tbuf, meta, smn);
                        if (i + 2 * G < nk)
                            offs_next = tile_offsets_load(p.v, rb * gpr + kg + 2 * G);
                    }
#pragma unroll
                    for (int I = 0; I < 32; I++)
                        q[I] = decode_pair(ls, lut, I, sm_word(sm, I >> 1));
                    tile_check(ls, p.status);
                    if ((em >> lane) & 1u) {  // escaped group: rebuild from its raw exponents
                        uint4 e[4];
                        escape_read(eb, em, e);
#pragma unroll
                        for (int I = 0; I < 32; I++)
                            q[I] = escape_pair(e, I, sm_word(sm, I >> 1));
                    }
                } else {
#pragma unroll
                    for (int I = 0; I < 32; I++)
                        q[I] = 0u;
                }
                if (u > 0)
                    mbar_wait(empty0 + 8u * s, uint32_t(u - 1) & 1u, p.status, kStatusTimeout);
                load_x_quarter(p, b_st, kg, rbl, lane);
                cp_async_commit();
#pragma unroll
                for (int c = 0; c < 8; c++)
                    sts128(a_st + sw128_offset(arow, uint32_t(c)), q[4 * c], q[4 * c + 1], q[4 * c + 2],
                           q[4 * c + 3]);
            } else {
                if (u > 0)
                    mbar_wait(empty0 + 8u * s, uint32_t(u - 1) & 1u, p.status, kStatusTimeout);
                load_x_quarter(p, b_st, kg, rbl, lane);
                const int64_t n = rb * kTileRows + lane;
                const bool ok = rb_ok && lane < R;
                const uint16_t *src = ok ? p.w + n * p.cols + kg * kGroup : p.w;
#pragma unroll
                for (int c = 0; c < 8; c++)
                    cp_async16_zfill(a_st + sw128_offset(arow, uint32_t(c)), ok ? src + 8 * c : src, ok ? 16u : 0u);
                cp_async_commit();
            }
            cp_async_wait_all();
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(full0 + 8u * s);
        }
    } else if (lane == 0) {  // the MMA warp
        const uint32_t idesc = idesc_bf16_f32(kTcM, Np);
#pragma unroll 1
        for (int i = 0; i < nk; i++) {
            const int s = i % S;
            mbar_wait(full0 + 8u * s, uint32_t(i / S) & 1u, p.status, kStatusTimeout);
            tc_fence_after();
            const uint32_t a_st = a0 + uint32_t(s) * kAStageBytes, b_st = b0 + uint32_t(s) * bstage;
#pragma unroll
            for (int k = 0; k < 4; k++)
                mma_bf16(tmem, sdesc_sw128(a_st + 32u * k), sdesc_sw128(b_st + 32u * k), idesc, (i | k) != 0);
            mma_commit(empty0 + 8u * s);
        }
        mma_commit(done);
    }
    __syncwarp();

    // epilogue: TMEM lane quarter `warp` holds rows n0 + 32*warp + lane
    const int64_t n = mb * kTcM + 32 * warp + lane;
    if (warp < 4) {
        mbar_wait(done, 0u, p.status, kStatusTimeout);
        tc_fence_after();
#pragma unroll 1
        for (int c0 = 0; c0 < Np; c0 += 16) {
            uint32_t v[16];
            tmem_ld16(tmem + (uint32_t(32 * warp) << 16) + uint32_t(c0), v);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; j++) {
                const int b = c0 + j;
                if (b < p.batch && n < p.rows) {
                    const float f = __uint_as_float(v[j]);
                    if (p.splits == 1)
                        p.y[int64_t(b) * p.rows + n] = __bfloat16_as_ushort(__float2bfloat16_rn(f));
                    else
                        p.partial[((mb * p.splits + split) * Np + b) * kTcM + 32 * warp + lane] = f;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == P)
        tmem_dealloc(tmem, p.tmem_cols);
    if (p.splits == 1)
        return;

    // split-K: the last CTA of this row block adds the splits in order
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0)
        last_cta = atomicAdd(p.counters + mb, 1u) == uint32_t(p.splits - 1);
    __syncthreads();
    if (!last_cta)
        return;
    __threadfence();
    if (warp < 4 && n < p.rows) {
        for (int b = 0; b < p.batch; b++) {
            const float *ps = p.partial + (mb * p.splits * Np + b) * kTcM + 32 * warp + lane;
            float tot = __ldcg(ps);
            for (int sp = 1; sp < p.splits; sp++)
                tot += __ldcg(ps + int64_t(sp) * Np * kTcM);
            p.y[int64_t(b) * p.rows + n] = __bfloat16_as_ushort(__float2bfloat16_rn(tot));
        }
    }
    if (threadIdx.x == 0)
        p.counters[mb] = 0;
}

template <int G, bool kCompressed>
uw_status launch_tc_one(const TcParams &p, size_t smem, cudaStream_t stream) {
    auto kern = gemm_tc_kernel<G, kCompressed>;
    if (!ensure_smem(kern, smem))
        return UW_ERR_CUDA;
    const dim3 grid(unsigned((p.rows + kTcM - 1) / kTcM), unsigned(p.splits));
    kern<<<grid, dim3((4 * G + 1) * 32), smem, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? UW_OK : UW_ERR_CUDA;
}

}  // namespace

size_t gemm_tc_smem_bytes(int G, int S, int Np, bool compressed, uint32_t tbuf) {
    size_t s = 1024 + size_t(S) * (kAStageBytes + size_t(Np) * 128);
    if (compressed)
        s += size_t(kCommonSmemBytes) + size_t(4 * G) * 2 * tbuf;
    return s;
}

int gemm_tc_stages(int G, int Np, bool compressed, uint32_t tbuf) {
    int S = kTcMaxStages;
    while (S > 1 && gemm_tc_smem_bytes(G, S, Np, compressed, tbuf) > size_t(kMaxSmemPerBlock - 1024))
        S--;
    return S;
}

int64_t gemm_tc_partial_floats(int64_t rows, int64_t batch, int splits) {
    if (splits <= 1)
        return 0;
    const int64_t np = std::min<int64_t>((batch + 15) / 16 * 16, kTcMaxBatch);
    return (rows + kTcM - 1) / kTcM * splits * np * kTcM;
}

uw_status launch_gemm_tc(const TcParams &base, int G, bool compressed, cudaStream_t stream) {
    const int64_t gpr = base.cols / kGroup;
    if (base.splits < 1 || base.splits > gpr || (G != 2 && G != 4))
        return UW_ERR_UNSUPPORTED;
    for (int64_t b0 = 0; b0 < base.batch; b0 += kTcMaxBatch) {
        TcParams p = base;
        p.batch = std::min<int64_t>(kTcMaxBatch, base.batch - b0);
        p.x = base.x + b0 * base.cols;
        p.y = base.y + b0 * base.rows;
        p.Np = int((p.batch + 15) / 16 * 16);
        p.tmem_cols = 32;
        while (p.tmem_cols < uint32_t(p.Np))
            p.tmem_cols <<= 1;
        p.S = gemm_tc_stages(G, p.Np, compressed, p.v.tbuf);
        if (p.S < G)
            return UW_ERR_UNSUPPORTED;
        const size_t smem = gemm_tc_smem_bytes(G, p.S, p.Np, compressed, p.v.tbuf);
        uw_status s;
        if (G == 2)
            s = compressed ? launch_tc_one<2, true>(p, smem, stream) : launch_tc_one<2, false>(p, smem, stream);
        else
            s = compressed ? launch_tc_one<4, true>(p, smem, stream) : launch_tc_one<4, false>(p, smem, stream);
        if (s != UW_OK)
            return s;
    }
    return UW_OK;
}

}  // namespace uw
