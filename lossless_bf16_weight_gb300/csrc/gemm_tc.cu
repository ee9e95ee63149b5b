// Tensor-core matmul for batches that make it a real contraction,
// y = x W^T with W [rows, cols], x [batch, cols], fp32 accumulation in
// tensor memory, BF16 out.
//
// D = W x^T is computed as tcgen05.mma tiles with M = 128 rows of W (the A
// operand, in tensor memory) and N = the batch padded to a multiple of 16
// (the B operand, x, in shared memory), K = 16 per instruction.  A "unit" is
// one 128-row block mb and one 64-column group k: a K step of four MMAs.
//
// Stream-K over every SM.  The units, block after block (u = mb * nk + k),
// are cut into V contiguous ranges of equal length ("workers"; V is the SM
// count unless the matrix has fewer than four units per SM).  One
// persistent CTA per SM runs worker blockIdx.x (and blockIdx.x + gridDim.x,
// ... when the launch is given fewer CTAs).  A worker's range falls into a
// few segments (mb, K steps [ks, ke)); a segment that covers the whole K
// range writes y from the accumulator; otherwise its fp32 accumulator goes
// to the workspace, and the block's last segment to finish adds the block's
// segments in segment order and writes y.  The cut depends only on the shape
// and the SM count, so every weight source (compressed or not) and every
// number of CTAs give the same sums in the same order: bit-identical y.
//
// Warp roles (CTA of 4G + 2 warps):
//   producers  warp w < 4G: rows 32*(w%4) .. +31 of each block, and the K
//              step pairs p = w/4, w/4 + G, ... of each segment (steps
//              ks + 2p, ks + 2p + 1); it rebuilds the pair's two 32 x 64 tiles
//              in registers (lane = row) and writes each with one tcgen05.st
//              into an A stage (32 tensor-memory columns, two BF16 per
//              column):
//                * Huffman source: the copy engine stages each pair's codes
//                  (pair_stage.cuh) two pairs ahead and the warp decodes the
//                  two tiles side by side (decode.cuh); the sign+mantissa
//                  bytes come from L2 after a bulk prefetch.  The weights go
//                  from the blob to the tensor cores without touching HBM
//                  (Unweight blog, paragraphs on the reconstructive matmul and
//                  on decoding on chip);
//                * palette-4 / exponent forms: the form and sign+mantissa
//                  bytes of the lane's row, merged through a 256-entry table
//                  (palette-4) or directly (exponents);
//                * uncompressed BF16: the rows themselves.
//              After its last pair of a segment each producer reads 16-column
//              chunks of its lane quarter of the accumulator (the epilogue).
//   MMA warp   warp 4G: one thread waits for each unit's A and x stages,
//              issues its four MMAs and commits them to both stages' "empty"
//              barriers, and the segment's last to the "accumulator full"
//              barrier; it starts a segment once the producers have read the
//              previous one's accumulator.
//   x loader   warp 4G + 1: one thread brings each unit's x rows (64 columns
//              x Np rows, 128-byte swizzled) into an x stage with one
//              tensor-map copy; rows past the batch are zero-filled.
#include <cuda_bf16.h>

#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "decode.cuh"
#include "kernels.h"
#include "pair_stage.cuh"
#include "tc.cuh"

namespace uw {

namespace {

constexpr int kTcM = 128;
constexpr int kStagesA = 8;        // A stages: 32 tensor-memory columns each (a power of two)
constexpr int kMaxX = 8;           // x stages in shared memory
constexpr int kMaxProducers = 16;  // 4G, G <= 4
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kMinUnits = 4;  // K steps per worker at least
constexpr uint32_t kYBufBytes = 32 * kTcM * 2;  // a producer group's y chunk: 32 columns x 128 rows BF16

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
        :: "r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
           "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]),
           "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]),
           "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};"
        :: "r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
           "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// D[tmem] (+)= A[tmem] * B[smem]^T for one K slice of 16; issued by one thread.
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                       bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
        :: "r"(d_tmem), "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(uint32_t(accumulate)) : "memory");
}

// Barrier 1 over the producer warps only (barrier 0 is __syncthreads).
__device__ __forceinline__ void producers_sync(int nthreads) {
    asm volatile("bar.sync 1, %0;" :: "r"(nthreads) : "memory");
}

// Barrier 2 + g over the four producer warps of group g.
__device__ __forceinline__ void group_sync(int g) {
    asm volatile("bar.sync %0, 128;" :: "r"(2 + g) : "memory");
}

__device__ __forceinline__ void sts16(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.u16 [%0], %1;" :: "r"(addr), "h"(uint16_t(v)) : "memory");
}

// An escaped group's 32 BF16 pairs, from its raw exponents (in the pair
// stage) and its four sign+mantissa chunks.
__device__ __forceinline__ void escaped_pairs(uint32_t ebase, uint32_t em, const uint4 (&sm)[4], uint32_t (&q)[32]) {
    uint4 e[4];
    escape_read(ebase, em, e);
#pragma unroll
    for (int I = 0; I < 32; I++)
        q[I] = escape_pair(e, I, sm_word(sm, I >> 1));
}

// The same for the 16 pairs of half h (pairs 16h .. 16h + 15).
__device__ __forceinline__ void escaped_half(uint32_t ebase, uint32_t em, const uint4 (&sm)[4], int h,
                                             uint32_t (&q)[16]) {
    uint4 e[4];
    escape_read(ebase, em, e);
#pragma unroll
    for (int i = 0; i < 16; i++)
        q[i] = escape_pair(e, 16 * h + i, sm_word(sm, (16 * h + i) >> 1));
}

__device__ __forceinline__ void sm_chunks(const uint8_t *g_lane, uint32_t stride, uint4 (&sm)[4]) {
#pragma unroll
    for (int c = 0; c < 4; c++)
        sm[c] = __ldg(reinterpret_cast<const uint4 *>(g_lane + c * stride));
}

// ---------------------------------------------------------------------------
// The stream-K cut: worker c owns units [start(c), start(c + 1)); worker_of(u)
// is the worker whose range holds unit u (the last c with start(c) <= u).
__host__ __device__ __forceinline__ uint32_t sk_start(uint32_t T, uint32_t V, uint32_t c) {
    return uint32_t(uint64_t(T) * c / V);
}
__host__ __device__ __forceinline__ uint32_t sk_worker(uint32_t T, uint32_t V, uint32_t u) {
    return uint32_t((uint64_t(u + 1) * V - 1) / T);
}

// One segment of a worker: block mb, K steps [ks, ke).
struct SkSeg {
    uint32_t mb, ks, ke;
    uint32_t j, nseg;  // index of the segment among the block's, and their number
    uint32_t i0;       // units of the CTA before this segment (stage and phase bookkeeping)
    uint32_t n;        // segments of the CTA before this one
};

// The CTA's segments in order (every role walks the same sequence).
struct SkWalk {
    uint32_t T, V, nk, c, u, u1, icum, ncum;
    __device__ __forceinline__ void init(const TcParams &p) {
        T = p.T;
        V = p.V;
        nk = p.nk;
        c = blockIdx.x;
        icum = ncum = 0;
        u = c < V ? sk_start(T, V, c) : 0u;
        u1 = c < V ? sk_start(T, V, c + 1) : 0u;
    }
    __device__ __forceinline__ bool next(SkSeg &s) {
        while (u >= u1) {
            c += gridDim.x;
            if (c >= V)
                return false;
            u = sk_start(T, V, c);
            u1 = sk_start(T, V, c + 1);
        }
        const uint32_t mb = u / nk, base = mb * nk;
        const uint32_t end = u1 < base + nk ? u1 : base + nk;
        s.mb = mb;
        s.ks = u - base;
        s.ke = end - base;
        const uint32_t w0 = sk_worker(T, V, base);
        s.j = c - w0;
        s.nseg = sk_worker(T, V, base + nk - 1) - w0 + 1;
        s.i0 = icum;
        s.n = ncum;
        icum += s.ke - s.ks;
        ncum++;
        u = end;
        return true;
    }
};

// A producer warp's pairs in order: segment after segment, pairs g, g + G, ...
// of each (used to start the pairs' copies ahead of their decode).
struct PairWalk {
    SkWalk w;
    SkSeg s;
    uint32_t p;
    bool ok;
    __device__ __forceinline__ void skip(uint32_t g) {
        while (ok && 2u * p >= s.ke - s.ks) {
            ok = w.next(s);
            p = g;
        }
    }
    __device__ __forceinline__ void init(const TcParams &tp, uint32_t g) {
        w.init(tp);
        ok = w.next(s);
        p = g;
        skip(g);
    }
    __device__ __forceinline__ void advance(uint32_t g, uint32_t G) {
        p += G;
        skip(g);
    }
};

// y of block mb from its nseg segment partials ([seg][Np][128] fp32 each),
// added in segment order; the nthreads threads from 0 share the block as
// float4s (four rows of one batch column), four of them at a time so that
// their loads are in flight together.
__device__ __forceinline__ void fixup_block(const TcParams &p, uint32_t mb, uint32_t nseg, int Np, int nthreads) {
    const float4 *ps = reinterpret_cast<const float4 *>(p.partial + uint64_t(mb) * p.maxseg * uint64_t(Np) * kTcM);
    const uint32_t seg4 = uint32_t(Np) * (kTcM / 4);  // float4s of one segment
    const uint32_t step = uint32_t(nthreads);
    constexpr int kU = 4;
#pragma unroll 1
    for (uint32_t e0 = threadIdx.x; e0 < seg4; e0 += kU * step) {
        float4 tot[kU];
#pragma unroll
        for (int u = 0; u < kU; u++) {
            const uint32_t e = e0 + u * step;
            tot[u] = e < seg4 ? __ldcg(ps + e) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll 1
        for (uint32_t sj = 1; sj < nseg; sj++) {
            float4 add[kU];
#pragma unroll
            for (int u = 0; u < kU; u++) {
                const uint32_t e = e0 + u * step;
                add[u] = e < seg4 ? __ldcg(ps + uint64_t(sj) * seg4 + e) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < kU; u++) {
                tot[u].x += add[u].x;
                tot[u].y += add[u].y;
                tot[u].z += add[u].z;
                tot[u].w += add[u].w;
            }
        }
#pragma unroll
        for (int u = 0; u < kU; u++) {
            const uint32_t e = e0 + u * step;
            const int b = int(e / (kTcM / 4));
            if (e >= seg4 || b >= p.batch)
                continue;
            const int64_t n0 = int64_t(mb) * kTcM + 4 * (e % (kTcM / 4));
            uint16_t *yb = p.y + int64_t(b) * p.rows;
            const float t4[4] = {tot[u].x, tot[u].y, tot[u].z, tot[u].w};
#pragma unroll
            for (int k = 0; k < 4; k++)
                if (n0 + k < p.rows)
                    yb[n0 + k] = __bfloat16_as_ushort(__float2bfloat16_rn(t4[k]));
        }
    }
}

// One 32-column chunk of a whole segment's y: the group's four warps write
// their rows into the group's shared buffer ([32 columns][128 rows] BF16),
// then one tensor-map store sends whole 256-byte rows of y.
__device__ __forceinline__ void y_chunk_store(const TcParams &p, uint32_t ybuf, int g, int q, uint32_t mb, int c0,
                                              bool two, const uint32_t (&va)[16], const uint32_t (&vb)[16]) {
    const int lane = threadIdx.x & 31;
    if (q == 0 && lane == 0)
        tma_store_wait_read();  // the previous chunk's store has read the buffer
    group_sync(g);
    const uint32_t row = ybuf + 2u * uint32_t(32 * q + lane);
#pragma unroll
    for (int jj = 0; jj < 16; jj++)
        sts16(row + 256u * uint32_t(jj), __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(va[jj]))));
    if (two) {
#pragma unroll
        for (int jj = 0; jj < 16; jj++)
            sts16(row + 256u * uint32_t(16 + jj), __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(vb[jj]))));
    }
    fence_proxy_async_smem();
    group_sync(g);
    if (q == 0 && lane == 0) {
        tma_store_2d(&p.ymap, int(mb * kTcM), c0, ybuf);
        tma_store_commit();
    }
}

__device__ __noinline__ void y_chunk_store_call(const TcParams &p, uint32_t ybuf, int g, int q, uint32_t mb, int c0,
                                                bool two, const uint32_t (&va)[16], const uint32_t (&vb)[16]) {
    y_chunk_store(p, ybuf, g, q, mb, c0, two, va, vb);
}

// kTab (Huffman source): the pair table as 32 lane-private copies (2: every
// lookup one shared-memory wavefront, as in the batch-1 GEMV; fits beside
// the x stages up to batch ~64), as 16 copies shared by lane pairs (1: one or
// two wavefronts, 64 KB; wider batches) or as one table (0).
template <int G, int kSrc, int kTab>
__global__ void __launch_bounds__((4 * G + 2) * 32, 1) gemm_tc_kernel(const __grid_constant__ TcParams p) {
    constexpr int P = 4 * G;  // producer warps
    constexpr bool kCompressed = kSrc == kSrcHuffman;
    constexpr bool kP4 = kSrc == kSrcPalette4;
    constexpr bool kExp = kSrc == kSrcExponent;
    constexpr bool kTma = kSrc == kSrcBf16;  // A tiles by tensor-map copies into the x stages
    static_assert(kTab == 0 || kCompressed, "table copies: Huffman source");
    static_assert(P <= kMaxProducers, "producer warps");
    constexpr int kStride = kTab == 2 ? kStridePrivate : kTab == 1 ? kStrideHalf : kStrideShared;
    constexpr size_t kTabBytes = kTab == 2 ? kPrivateLutBytes : kTab == 1 ? kHalfLutBytes : 0;
    extern __shared__ unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t bars[2 * kStagesA + 2 * kMaxX + 2];
    __shared__ __align__(8) uint64_t pbars[P * kPairStages];
    __shared__ PairMeta metas[P * kPairStages];
    __shared__ uint32_t tmem_slot;
    __shared__ uint32_t last_seg;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const BlobView &v = p.v;
    const int Np = p.Np, SX = p.SX;
    const uint32_t gpr = p.nk;
    const uint32_t nrb = uint32_t((p.rows + kTileRows - 1) / kTileRows);
    const uint32_t xbytes = uint32_t(Np) * 128u;
    // a stage: [A tile, 128 rows x 64 columns (uncompressed source only)][x rows]
    const uint32_t abytes = kTma ? uint32_t(kTcM) * 128u : 0u;
    const uint32_t xstage = abytes + xbytes;
    const uint32_t a0col = p.a0col;  // first tensor-memory column of the A stages

    // shared memory: [pad to 1024][x stages][table copies (kTab)][decode
    // tables, or the palette-4 pair table][per producer warp kPairStages code stages]
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
    const uint32_t xs0 = raw + pad;
    const uint32_t priv = xs0 + uint32_t(SX) * xstage;
    unsigned char *dec = smem_raw + pad + size_t(SX) * xstage + kTabBytes;
    const uint32_t sbytes = code_stage_bytes(v.tdata);
    const uint32_t pst0 = (smem_addr(dec + kCommonSmemBytes) + 127u) & ~127u;
    const uint32_t afull0 = smem_addr(&bars[0]), aempty0 = smem_addr(&bars[kStagesA]);
    const uint32_t xfull0 = smem_addr(&bars[2 * kStagesA]), xempty0 = smem_addr(&bars[2 * kStagesA + kMaxX]);
    const uint32_t dfull = smem_addr(&bars[2 * kStagesA + 2 * kMaxX]), dfree = dfull + 8u;

    if (warp == P)
        tmem_alloc(smem_addr(&tmem_slot), kTmemCols);
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStagesA; s++) {
            mbar_init(afull0 + 8u * s, 4);  // the four producer warps of the unit's group
            mbar_init(aempty0 + 8u * s, 1);
        }
        for (int s = 0; s < SX; s++) {
            mbar_init(xfull0 + 8u * s, 1);
            mbar_init(xempty0 + 8u * s, 1);
        }
        mbar_init(dfull, 1);
        mbar_init(dfree, P);
        for (int i = 0; i < P * kPairStages; i++)
            mbar_init(smem_addr(&pbars[i]), 1);
        mbar_init_fence();
    }
    __syncthreads();

    // producer identity: lane quarter q (rows 32q .. 32q + 31 of each block),
    // group g (pairs g, g + G, ... of each segment)
    const int q = warp & 3, g = warp >> 2;
    const bool producer = warp < P;
    const uint32_t st0 = pst0 + uint32_t(warp) * kPairStages * sbytes;
    const uint32_t pbar0 = smem_addr(&pbars[producer ? warp * kPairStages : 0]);
    PairMeta *meta = &metas[producer ? warp * kPairStages : 0];
    DecodeShared ds{};
    // palette-4 source: one 256-entry pair table (entry b = palette[b >> 4] << 23 |
    // palette[b & 15] << 7) where the decode tables would be
    const uint32_t ptab = smem_addr(dec);
    if constexpr (kP4) {
        for (int b = threadIdx.x; b < 256; b += blockDim.x)
            reinterpret_cast<uint32_t *>(dec)[b] =
                (uint32_t(v.palette[b >> 4]) << 23) | (uint32_t(v.palette[b & 15]) << 7);
    }
    // Huffman source: the copies of this warp's pairs run kPairStages ahead of
    // their decode (`iss` walks the same pairs), each pair's tile offsets one
    // pair ahead of its copies
    PairWalk iss;
    uint32_t nissued = 0, o_next = 0;
    auto walk_rb = [&](const PairWalk &it) { return 4u * it.s.mb + uint32_t(q); };
    auto walk_tile = [&](const PairWalk &it) { return walk_rb(it) * gpr + it.s.ks + 2u * it.p; };
    auto issue = [&](uint32_t o, uint32_t s) {
        const uint32_t rb = walk_rb(iss), kA = iss.s.ks + 2u * iss.p;
        const bool hasB = kA + 1 < iss.s.ke;
        const uint32_t st = st0 + s * sbytes, bar = pbar0 + 8u * s;
        if (rb < nrb) {
            pair_issue_codes(v, o, rb, kA, hasB, rb * gpr + kA, st, bar, meta + s);
        } else if (lane == 0) {  // rows past the matrix: nothing to copy
            meta[s] = PairMeta{};
            mbar_arrive(bar);
        }
        __syncwarp();
    };
    if constexpr (kCompressed) {
        ds = carve_common(dec);
        if (producer) {
            iss.init(p, uint32_t(g));
            PairWalk i2 = iss;
            if (i2.ok)
                i2.advance(uint32_t(g), G);
            const uint32_t t0 = iss.ok && walk_rb(iss) < nrb ? walk_tile(iss) : 0u;
            const uint32_t t1 = i2.ok && walk_rb(i2) < nrb ? walk_tile(i2) : 0u;
            o_next = pair_offsets_load2(v, t0, t1);
        }
        build_tables(ds, v);
        if (producer) {
            for (int s = 0; s < kPairStages && iss.ok; s++) {
                issue(o_next, uint32_t(s));
                nissued++;
                iss.advance(uint32_t(g), G);
                o_next = pair_offsets_shift(o_next);
            }
            if (iss.ok && walk_rb(iss) < nrb)
                o_next = pair_offsets_load(v, walk_tile(iss));
        }
    }
    if constexpr (kTab != 0) {
        __syncthreads();
        if constexpr (kTab == 2)
            replicate_private(ds, priv);
        else
            replicate_half(ds, priv);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // Let the next kernel launch only now that this CTA holds its tensor
    // memory: a later CTA on this SM then waits in its own allocation for
    // this one to finish, never the other way round.
    grid_dep_launch();
    grid_dep_wait();  // x (and the uncompressed weights) may come from the kernel before; the partials are reused
    const uint32_t tmem = tmem_slot;
    const uint32_t lut = !kCompressed ? 0u
                         : kTab == 2  ? priv + 4u * uint32_t(lane)
                         : kTab == 1  ? priv + 4u * uint32_t(lane & 15)
                                      : smem_addr(ds.lut);

    if (producer) {
        const uint32_t trow = tmem + (uint32_t(32 * q) << 16) + a0col;
        uint32_t bad = 0;
        uint32_t j = 0;  // this warp's pairs so far: stage index and parity
        // chunk 0 of the current pair's sign+mantissa bytes, loaded during the
        // previous pair when that one knew it
        uint4 c0A = make_uint4(0, 0, 0, 0), c0B = c0A;
        bool c0_ok = false;
        SkWalk wk;
        wk.init(p);
        SkSeg s;
        while (wk.next(s)) {
            const uint32_t rb = 4u * s.mb + uint32_t(q);
            const bool rb_ok = rb < nrb;
            const uint32_t npairs = kTma ? 0u : (s.ke - s.ks + 1) / 2;  // uncompressed: epilogue only
#pragma unroll 1
            for (uint32_t pp = uint32_t(g); pp < npairs; pp += G, j++) {
                const uint32_t kgA = s.ks + 2u * pp;
                const bool hasB = kgA + 1 < s.ke;
                // A stages of the pair's two units (unit i reuses the stage of unit i - kStagesA)
                const uint32_t iA = s.i0 + 2u * pp;
                const uint32_t sA_ = iA % kStagesA, sB_ = (iA + 1) % kStagesA;
                const uint32_t uA = iA / kStagesA, uB = (iA + 1) / kStagesA;
                auto stages_free = [&]() {
                    if (uA > 0)
                        mbar_wait(aempty0 + 8u * sA_, (uA - 1) & 1u, p.status, kStatusTimeout);
                    if (hasB && uB > 0)
                        mbar_wait(aempty0 + 8u * sB_, (uB - 1) & 1u, p.status, kStatusTimeout);
                    tc_fence_after();
                };
                auto stages_full = [&]() {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(afull0 + 8u * sA_);
                        if (hasB)
                            mbar_arrive(afull0 + 8u * sB_);
                    }
                };
                if constexpr (kCompressed) {
                    // each tile is stored in two 16-column halves as it is decoded
                    const uint32_t si = j % kPairStages;
                    const uint32_t st = st0 + si * sbytes, pb = pbar0 + 8u * si;
                    mbar_wait(pb, (j / kPairStages) & 1u, p.status, kStatusTimeout);
                    const PairMeta m = meta[si];
                    const uint32_t R = m.R & 0xFFu;
                    if (rb_ok && R != 0u) {
                        const uint8_t *sm_cur = reinterpret_cast<const uint8_t *>((uint64_t(m.sm_hi) << 32) | m.sm_lo);
                        const bool full = rb < v.nfull;
                        uint32_t gA, gB;
                        if (full) {
                            gA = lds_u8(st + uint32_t(lane));
                            gB = lds_u8(st + 32u + uint32_t(lane));
                        } else {
                            const uint64_t q0 = uint64_t(rb * gpr + kgA) * kTileRows - uint64_t(kTileRows - R) * kgA;
                            const uint32_t l = uint32_t(lane) < R ? uint32_t(lane) : 0u;
                            gA = __ldg(v.glen + q0 + l);
                            gB = hasB ? __ldg(v.glen + q0 + R + l) : 0u;
                        }
                        LaneStream la, lb;
                        const uint32_t cA = st + 64u, cB = cA + 16u * m.n16A;
                        uint32_t emA, emB;
                        pair_begin_ready(ds, gA, gB, m.pkA, m.pkB, int(R), hasB ? int(R) : 0, cA, cB, la, lb,
                                         p.status, emA, emB);
                        const uint32_t ebA = cA + 16u * (m.n16A + m.n16B), ebB = ebA + 64u * m.nescA;
                        // sign+mantissa bytes straight from L2 (prefetched there with the codes), one
                        // 16-byte chunk ahead; chunk 0 of the next pair during this one
                        const uint32_t stride = 16u * R;
                        const uint32_t lc = uint32_t(lane) < R ? uint32_t(lane) : 0u;
                        const uint8_t *gA_sm = sm_cur + 16u * lc, *gB_sm = hasB ? gA_sm + 64u * R : gA_sm;
                        if (!c0_ok) {
                            c0A = __ldg(reinterpret_cast<const uint4 *>(gA_sm));
                            c0B = __ldg(reinterpret_cast<const uint4 *>(gB_sm));
                        }
                        const PairMeta mn = meta[(j + 1) % kPairStages];
                        const uint32_t Rn = mn.R & 0xFFu;
                        const bool more = j + 1 < nissued && Rn != 0u;
                        const uint8_t *sm_nxt = reinterpret_cast<const uint8_t *>((uint64_t(mn.sm_hi) << 32) | mn.sm_lo);
                        const uint32_t lcn = uint32_t(lane) < Rn ? uint32_t(lane) : 0u;
                        const uint32_t offBn = (mn.R & 0x100u) ? 64u * Rn : 0u;
                        const bool escA = (emA >> lane) & 1u, escB = (emB >> lane) & 1u;
                        uint4 sA = c0A, sB = c0B, nA = sA, nB = sB;
#pragma unroll
                        for (int h = 0; h < 2; h++) {
                            uint32_t qA[16], qB[16];
#pragma unroll
                            for (int i = 0; i < 16; i++) {
                                const int I = 16 * h + i;
                                if ((I & 7) == 0) {
                                    if (I < 24) {
                                        nA = __ldg(reinterpret_cast<const uint4 *>(gA_sm + uint32_t((I >> 3) + 1) * stride));
                                        nB = __ldg(reinterpret_cast<const uint4 *>(gB_sm + uint32_t((I >> 3) + 1) * stride));
                                    } else if (more) {
                                        const uint8_t *a = sm_nxt + 16u * lcn;
                                        nA = __ldg(reinterpret_cast<const uint4 *>(a));
                                        nB = __ldg(reinterpret_cast<const uint4 *>(a + offBn));
                                    }
                                }
                                qA[i] = decode_pair<kStride>(la, lut, I, word4(sA, (I >> 1) & 3));
                                qB[i] = decode_pair<kStride>(lb, lut, I, word4(sB, (I >> 1) & 3));
                                if ((I & 7) == 7) {
                                    sA = nA;
                                    sB = nB;
                                }
                            }
                            if (escA | escB) {  // escaped groups: this half again from the raw exponents
                                uint4 smc[4];
                                if (escA) {
                                    sm_chunks(gA_sm, stride, smc);
                                    escaped_half(ebA, emA, smc, h, qA);
                                }
                                if (escB) {
                                    sm_chunks(gB_sm, stride, smc);
                                    escaped_half(ebB, emB, smc, h, qB);
                                }
                            }
                            if (h == 0)
                                stages_free();
                            tmem_st16(trow + 32u * sA_ + 16u * uint32_t(h), qA);
                            if (hasB)
                                tmem_st16(trow + 32u * sB_ + 16u * uint32_t(h), qB);
                            tmem_st_wait();
                        }
                        bad |= tile_check_bits(la) | tile_check_bits(lb);
                        c0A = sA;  // chunk 0 of the next pair
                        c0B = sB;
                        c0_ok = more;
                    } else {  // rows past the matrix
                        uint32_t z[16];
#pragma unroll
                        for (int i = 0; i < 16; i++)
                            z[i] = 0u;
                        stages_free();
#pragma unroll
                        for (int h = 0; h < 2; h++) {
                            tmem_st16(trow + 32u * sA_ + 16u * uint32_t(h), z);
                            if (hasB)
                                tmem_st16(trow + 32u * sB_ + 16u * uint32_t(h), z);
                        }
                        tmem_st_wait();
                        c0_ok = false;
                    }
                    stages_full();
                    // the pair stage is free: start the pair kPairStages ahead
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (iss.ok) {
                        issue(o_next, si);
                        nissued++;
                        iss.advance(uint32_t(g), G);
                        if (iss.ok && walk_rb(iss) < nrb)
                            o_next = pair_offsets_load(v, walk_tile(iss));
                    }
                } else if constexpr (kP4 || kExp) {
                    // the intermediate form (4-bit palette indices rebuilt through the
                    // pair table, or exponent bytes) and the sign+mantissa bytes of the
                    // lane's row, one tile after the other; palette-4 escaped groups from
                    // their raw exponents
                    const int R = !rb_ok ? 0 : int(std::min<int64_t>(kTileRows, p.rows - int64_t(rb) * kTileRows));
                    const bool ok = rb_ok && lane < R;
                    const uint32_t lc = ok ? uint32_t(lane) : 0u;
                    constexpr int NI = kP4 ? 2 : 4;  // 16-byte chunks of the form per row
                    auto rebuild = [&](uint32_t kg, bool has, uint32_t (&qq)[32]) {
                        const uint64_t q0 = uint64_t(kTileRows) * rb * gpr + uint64_t(R) * kg;
                        uint4 ix[NI], sx[4];
#pragma unroll
                        for (int c = 0; c < NI; c++)
                            ix[c] = ok && has ? __ldg(reinterpret_cast<const uint4 *>(p.p4 + 16 * NI * q0 + 16 * lc + c * 16 * R))
                                              : make_uint4(0, 0, 0, 0);
#pragma unroll
                        for (int c = 0; c < 4; c++)
                            sx[c] = ok && has ? __ldg(reinterpret_cast<const uint4 *>(v.sm + 64 * q0 + 16 * lc + c * 16 * R))
                                              : make_uint4(0, 0, 0, 0);
                        const uint32_t gl = kP4 && ok && has ? __ldg(v.glen + q0 + lc) : 1u;
#pragma unroll
                        for (int I = 0; I < 32; I++) {
                            if constexpr (kP4) {
                                const uint32_t b = (word4(ix[I >> 4], (I >> 2) & 3) >> (8 * (I & 3))) & 0xFFu;
                                qq[I] = lop3_merge(prmt(sm_word(sx, I >> 1), 0u, (I & 1) ? 0xB3A2u : 0x9180u),
                                                   lds32(ptab + 4u * b));
                            } else {
                                qq[I] = escape_pair(ix, I, sm_word(sx, I >> 1));
                            }
                        }
                        const uint32_t em = __ballot_sync(0xffffffffu, ok && has && gl == 0u);
                        if ((em >> lane) & 1u) {
                            const uint32_t t = rb * gpr + kg;
                            const uint4 *ep = reinterpret_cast<const uint4 *>(
                                v.esc + 64 * uint64_t(__ldg(v.tesc + t) + __popc(em & ((1u << lane) - 1u))));
                            uint4 e[4];
#pragma unroll
                            for (int c = 0; c < 4; c++)
                                e[c] = __ldg(ep + c);
#pragma unroll
                            for (int I = 0; I < 32; I++)
                                qq[I] = escape_pair(e, I, sm_word(sx, I >> 1));
                        }
                        if (!(ok && has)) {
#pragma unroll
                            for (int I = 0; I < 32; I++)
                                qq[I] = 0u;
                        }
                    };
                    // the next pair of this segment's form and sign+mantissa bytes into L2
                    if (lane == 0 && rb_ok && pp + G < npairs) {
                        const uint32_t kgN = kgA + 2u * G;
                        const uint32_t nt = kgN + 1 < s.ke ? 2u : 1u;
                        const uint64_t q0 = uint64_t(kTileRows) * rb * gpr + uint64_t(R) * kgN;
                        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(p.p4 + 16 * NI * q0),
                                     "r"(16u * NI * uint32_t(R) * nt) : "memory");
                        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(v.sm + 64 * q0),
                                     "r"(64u * uint32_t(R) * nt) : "memory");
                    }
                    // one tile after the other into its A stage
                    uint32_t qq[32];
                    rebuild(kgA, true, qq);
                    stages_free();
                    tmem_st32(trow + 32u * sA_, qq);
                    tmem_st_wait();
                    if (hasB) {
                        rebuild(kgA + 1, true, qq);
                        tmem_st32(trow + 32u * sB_, qq);
                        tmem_st_wait();
                    }
                    stages_full();
                }
            }

            // epilogue of the segment: this warp's 32-column chunks of its lane
            // quarter (two loads, one wait), to y (a segment over the whole K
            // range) or to the segment's partial
            mbar_wait(dfull, s.n & 1u, p.status, kStatusTimeout);
            tc_fence_after();
            const int64_t n = int64_t(s.mb) * kTcM + 32 * q + lane;
            const bool whole = s.nseg == 1;
            float *part = p.partial + (uint64_t(s.mb) * p.maxseg + s.j) * uint64_t(Np) * kTcM + 32 * q + lane;
            // y of a whole segment through the group's shared buffer ([32 columns][128 rows]
            // BF16) and one tensor-map store per chunk, whole 256-byte rows of y
            const bool ytma = whole && p.ystage != 0;
            const uint32_t ybuf = xs0 + p.ybuf_off + uint32_t(g) * kYBufBytes;
#pragma unroll 1
            for (int c0 = 32 * g; c0 < Np; c0 += 32 * G) {
                uint32_t va[16], vb[16];
                tmem_ld16(tmem + (uint32_t(32 * q) << 16) + uint32_t(c0), va);
                if (c0 + 16 < Np)
                    tmem_ld16(tmem + (uint32_t(32 * q) << 16) + uint32_t(c0 + 16), vb);
                tmem_ld_wait();
                if (ytma) {
                    // out of line beside producers, so that it does not weigh on their registers
                    if constexpr (kTma)
                        y_chunk_store(p, ybuf, g, q, s.mb, c0, c0 + 16 < Np, va, vb);
                    else
                        y_chunk_store_call(p, ybuf, g, q, s.mb, c0, c0 + 16 < Np, va, vb);
                    continue;
                }
                auto put = [&](int b, uint32_t bits) {
                    if (b < p.batch) {
                        const float f = __uint_as_float(bits);
                        if (!whole)
                            part[int64_t(b) * kTcM] = f;
                        else if (n < p.rows)
                            p.y[int64_t(b) * p.rows + n] = __bfloat16_as_ushort(__float2bfloat16_rn(f));
                    }
                };
#pragma unroll
                for (int jj = 0; jj < 16; jj++)
                    put(c0 + jj, va[jj]);
                if (c0 + 16 < Np) {
#pragma unroll
                    for (int jj = 0; jj < 16; jj++)
                        put(c0 + 16 + jj, vb[jj]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(dfree);  // the MMA warp may start the next segment
            if (!whole) {
                // the block's last segment to finish adds all of them in order
                __threadfence();
                producers_sync(P * 32);
                if (threadIdx.x == 0) {
                    const uint32_t done = atomicAdd(p.counters + s.mb, 1u) + 1u;
                    last_seg = done == s.nseg;
                    if (done == s.nseg)
                        p.counters[s.mb] = 0;
                }
                producers_sync(P * 32);
                if (last_seg) {
                    __threadfence();
                    fixup_block(p, s.mb, s.nseg, Np, P * 32);
                }
            }
        }
        if (p.ystage != 0 && q == 0 && lane == 0)
            tma_store_wait_all();
        tile_check_flush(bad, p.status);
    } else if (warp == P) {
        if (lane == 0) {  // the MMA warp
            const uint32_t idesc = idesc_bf16_f32(kTcM, Np);
            SkWalk wk;
            wk.init(p);
            SkSeg s;
            uint32_t i = 0, sx = 0, xph = 0;  // unit, its x stage and that stage's phase parity
            while (wk.next(s)) {
                if (s.n > 0)  // the producers have read the previous segment's accumulator
                    mbar_wait(dfree, (s.n - 1) & 1u, p.status, kStatusTimeout);
                tc_fence_after();
#pragma unroll 1
                for (uint32_t k = s.ks; k < s.ke; k++, i++) {
                    const uint32_t sa = i % kStagesA;
                    if (!kTma)
                        mbar_wait(afull0 + 8u * sa, (i / kStagesA) & 1u, p.status, kStatusTimeout);
                    mbar_wait(xfull0 + 8u * sx, xph, p.status, kStatusTimeout);
                    tc_fence_after();
                    const uint32_t a_st = xs0 + sx * xstage, b_st = a_st + abytes;
#pragma unroll
                    for (int kk = 0; kk < 4; kk++) {
                        if constexpr (kTma)
                            mma_bf16(tmem, sdesc_sw128(a_st + 32u * kk), sdesc_sw128(b_st + 32u * kk), idesc,
                                     k != s.ks || kk != 0);
                        else
                            mma_ts(tmem, tmem + a0col + 32u * sa + 8u * kk, sdesc_sw128(b_st + 32u * kk), idesc,
                                   k != s.ks || kk != 0);
                    }
                    if (!kTma)
                        mma_commit(aempty0 + 8u * sa);
                    mma_commit(xempty0 + 8u * sx);
                    if (++sx == uint32_t(SX)) {
                        sx = 0;
                        xph ^= 1u;
                    }
                }
                mma_commit(dfull);
            }
        }
    } else if (lane == 0) {  // the x loader
        SkWalk wk;
        wk.init(p);
        SkSeg s;
        uint32_t sx = 0, xph = 0;  // x stage and the parity of its next phase
        bool wrapped = false;      // every stage used once: wait for the MMAs to free it
        while (wk.next(s)) {
#pragma unroll 1
            for (uint32_t k = s.ks; k < s.ke; k++) {
                if (wrapped)
                    mbar_wait(xempty0 + 8u * sx, xph ^ 1u, p.status, kStatusTimeout);
                mbar_expect_tx(xfull0 + 8u * sx, xstage);
                if (kTma)
                    tma_load_2d(xs0 + sx * xstage, &p.wmap, int(k * kGroup), int(s.mb * kTcM), xfull0 + 8u * sx);
                tma_load_2d(xs0 + sx * xstage + abytes, &p.xmap, int(k * kGroup), 0, xfull0 + 8u * sx);
                if (++sx == uint32_t(SX)) {
                    sx = 0;
                    xph ^= 1u;
                    wrapped = true;
                }
            }
        }
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == P)
        tmem_dealloc(tmem, kTmemCols);
}

template <int G, int kSrc, int kTab>
uw_status launch_tc_one(const TcParams &p, size_t smem, int grid, cudaStream_t stream) {
    auto kern = gemm_tc_kernel<G, kSrc, kTab>;
    if (!ensure_smem(kern, smem))
        return UW_ERR_CUDA;
    return launch_overlapped(kern, dim3(unsigned(grid)), dim3((4 * G + 2) * 32), smem, stream, p) == cudaSuccess
               ? UW_OK
               : UW_ERR_CUDA;
}

template <int kSrc, int kTab = 0>
uw_status launch_tc_g(const TcParams &p, int G, size_t smem, int grid, cudaStream_t stream) {
    if constexpr (kSrc == kSrcBf16)  // no producers: the warps that would be run the epilogue
        return launch_tc_one<3, kSrc, 0>(p, smem, grid, stream);
    else
        return G == 2 ? launch_tc_one<2, kSrc, kTab>(p, smem, grid, stream)
               : G == 3 ? launch_tc_one<3, kSrc, kTab>(p, smem, grid, stream)
                        : launch_tc_one<4, kSrc, kTab>(p, smem, grid, stream);
}

// Tensor-memory columns before the A stages (the accumulator's Np, rounded up to 32).
uint32_t a0_col(int Np) { return (uint32_t(Np) + 31u) & ~31u; }

// Shared memory of a launch with SX x stages; `tab`: copies of the pair
// table (Huffman source: 2 = 32 lane-private, 1 = 16, 0 = one table).
size_t tc_smem(int G, int SX, int Np, int src, uint32_t tdata, int tab) {
    const size_t stage = size_t(Np) * 128 + (src == kSrcBf16 ? size_t(kTcM) * 128 : 0);  // [A tile][x rows]
    size_t s = 1024 + size_t(SX) * stage + (tab == 2 ? size_t(kPrivateLutBytes) : tab == 1 ? size_t(kHalfLutBytes) : 0);
    if (src == kSrcHuffman)
        s += size_t(kCommonSmemBytes) + 128 + size_t(4 * G) * kPairStages * code_stage_bytes(tdata);
    else if (src == kSrcPalette4)
        s += 256 * 4;  // the pair table
    return s;
}

struct TcConfig {
    int SX;
    int tab;  // table copies (Huffman source)
    size_t smem;
    uint32_t ybuf_off;  // offset of the y buffers from the 1024-aligned base, when they fit
    bool ystage;
    size_t smem_base;   // without the y buffers
};

// Stages for G producer groups and Np batch rows: A stages in the tensor
// memory the accumulator leaves; x stages in shared memory (with the A tile
// for the uncompressed source), the most that fit up to kMaxX (for the
// Huffman source the most table copies that leave three x stages, else one
// table and at least two).
bool tc_config(int G, int Np, int src, uint32_t tdata, TcConfig &c) {
    if (a0_col(Np) + 32u * kStagesA > kTmemCols)
        return false;
    const size_t lim = size_t(kMaxSmemPerBlock) - 1024;
    for (int tab = 2; tab >= 0; tab--) {
        if (tab != 0 && src != kSrcHuffman)
            continue;
        for (int sx = kMaxX; sx >= (tab != 0 ? 3 : 2); sx--)
            if (tc_smem(G, sx, Np, src, tdata, tab) <= lim) {
                c.SX = sx;
                c.tab = tab;
                const size_t base = tc_smem(G, sx, Np, src, tdata, tab);
                const int groups = src == kSrcBf16 ? 3 : G;  // the uncompressed form runs three groups
                c.ybuf_off = uint32_t((base - 1024 + 127) / 128 * 128);
                c.ystage = 1024 + size_t(c.ybuf_off) + size_t(groups) * kYBufBytes <= lim;
                c.smem = std::max(c.ystage ? 1024 + size_t(c.ybuf_off) + size_t(groups) * kYBufBytes : base,
                                  kExclusiveSmem);
                c.smem_base = base;
                return true;
            }
    }
    return false;
}

// The cut of a rows x cols matrix (cols a multiple of 64) for Np batch
// rows: units, workers, K steps per block and the most segments a block can
// have.  Stream-K over every SM, unless one whole block per worker costs no
// more: a split block's partials cost about Np / 16 units to write, read and
// add, so wide batches on a matrix of at most one block per SM keep whole
// blocks.
bool tc_partition(int64_t rows, int64_t cols, int Np, uint32_t &T, uint32_t &V, uint32_t &nk, uint32_t &maxseg) {
    const uint64_t nmb = uint64_t(rows + kTcM - 1) / kTcM, k = uint64_t(cols) / kGroup;
    if (nmb == 0 || k == 0 || nmb * k >= (uint64_t(1) << 32) / 2)
        return false;
    const uint64_t sms = uint64_t(sm_count());
    nk = uint32_t(k);
    T = uint32_t(nmb * k);
    V = uint32_t(std::min<uint64_t>(sms, (uint64_t(T) + kMinUnits - 1) / kMinUnits));
    V = std::max<uint32_t>(V, 1u);
    const uint64_t sk_cost = (uint64_t(T) + V - 1) / V + (T % V != 0 || V > nmb ? uint64_t(Np) / 16 : 0u);
    if (nmb <= sms && uint64_t(nk) <= sk_cost)
        V = uint32_t(nmb);  // whole blocks
    const uint32_t L = T / V;  // shortest worker range
    maxseg = std::min<uint32_t>(V, (nk + L - 1) / L + 1);
    return true;
}

}  // namespace

bool gemm_tc_fits(int G, int Np, int src, uint32_t tdata) {
    TcConfig c;
    return G >= 2 && G <= 4 && tc_config(G, Np, src, tdata, c);
}

int64_t gemm_tc_partial_floats(int64_t rows, int64_t cols, int64_t batch) {
    // the largest of the launches' needs (batches above kTcMaxBatch run as
    // several launches: full ones and the remainder)
    int64_t most = 0;
    for (int64_t b : {std::min<int64_t>(batch, kTcMaxBatch), batch % kTcMaxBatch}) {
        if (b <= 0)
            continue;
        const int np = int((b + 15) / 16 * 16);
        uint32_t T, V, nk, maxseg;
        if (!tc_partition(rows, cols, np, T, V, nk, maxseg))
            continue;
        most = std::max<int64_t>(most, (rows + kTcM - 1) / kTcM * int64_t(maxseg) * np * kTcM);
    }
    return most;
}

// The driver's tensor-map encoder, looked up once through the runtime.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// x rows b0 .. b0+batch-1 as a 2-D tensor (cols inner), boxes of 64 columns x
// Np rows with the 128-byte swizzle of the B stages; rows past the batch read
// as zeros.
bool encode_x_map(CUtensorMap *m, const uint16_t *x, int64_t cols, int64_t batch, int Np) {
    const auto enc = tensor_map_encoder();
    if (!enc)
        return false;
    const cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(batch)};
    const cuuint64_t strides[1] = {cuuint64_t(cols) * 2};
    const cuuint32_t box[2] = {cuuint32_t(kGroup), cuuint32_t(Np)};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(x), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// y [batch, rows] as a 2-D tensor (rows inner), boxes of 128 rows x 32 batch
// rows, no swizzle (the epilogue's shared buffer is [32][128] BF16).
bool encode_y_map(CUtensorMap *m, const uint16_t *y, int64_t rows, int64_t batch) {
    const auto enc = tensor_map_encoder();
    if (!enc)
        return false;
    const cuuint64_t dims[2] = {cuuint64_t(rows), cuuint64_t(batch)};
    const cuuint64_t strides[1] = {cuuint64_t(rows) * 2};
    const cuuint32_t box[2] = {cuuint32_t(kTcM), 32u};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(y), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// W [rows, cols] as a 2-D tensor (cols inner), boxes of a 128-row block x
// 64 columns with the 128-byte swizzle (the tensor-core A operand's layout);
// rows past the end read as zeros.
bool encode_w_block_map(CUtensorMap *m, const uint16_t *w, int64_t rows, int64_t cols) {
    const auto enc = tensor_map_encoder();
    if (!enc)
        return false;
    const cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
    const cuuint64_t strides[1] = {cuuint64_t(cols) * 2};
    const cuuint32_t box[2] = {cuuint32_t(kGroup), cuuint32_t(kTcM)};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(w), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// W [rows, cols] as a 2-D tensor (cols inner), boxes of one 32-row x
// 64-column tile with the 128-byte swizzle; rows past the end read as zeros.
bool encode_w_tile_map(CUtensorMap *m, const uint16_t *w, int64_t rows, int64_t cols) {
    const auto enc = tensor_map_encoder();
    if (!enc)
        return false;
    const cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
    const cuuint64_t strides[1] = {cuuint64_t(cols) * 2};
    const cuuint32_t box[2] = {cuuint32_t(kGroup), cuuint32_t(kTileRows)};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(w), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

uw_status launch_gemm_tc(const TcParams &base, int G, int src, cudaStream_t stream, int max_ctas) {
    if (G < 2 || G > 4)
        return UW_ERR_UNSUPPORTED;
    if (uint64_t(base.rows / kTileRows + 1) * uint64_t(base.cols / kGroup) >= (uint64_t(1) << 32))
        return UW_ERR_UNSUPPORTED;  // tile indices are 32-bit
    TcParams p = base;
    for (int64_t b0 = 0; b0 < base.batch; b0 += kTcMaxBatch) {
        p.batch = std::min<int64_t>(kTcMaxBatch, base.batch - b0);
        p.x = base.x + b0 * base.cols;
        p.y = base.y + b0 * base.rows;
        p.Np = int((p.batch + 15) / 16 * 16);
        if (!tc_partition(p.rows, p.cols, p.Np, p.T, p.V, p.nk, p.maxseg))
            return UW_ERR_UNSUPPORTED;
        const int grid = int(max_ctas > 0 ? std::min<uint32_t>(p.V, uint32_t(max_ctas)) : p.V);
        p.a0col = a0_col(p.Np);
        TcConfig c;
        if (!tc_config(G, p.Np, src, p.v.tdata, c))
            return UW_ERR_UNSUPPORTED;
        p.SX = c.SX;
        if (!encode_x_map(&p.xmap, p.x, p.cols, p.batch, p.Np))
            return UW_ERR_CUDA;
        if (src == kSrcBf16 && !encode_w_block_map(&p.wmap, p.w, p.rows, p.cols))
            return UW_ERR_CUDA;
        // y by tensor-map stores when every block is whole (wide batches; a stream-K cut
        // writes y only for the rare whole segment, and the buffers would cost L1) and its
        // rows are whole 16-byte units
        const uint64_t nmb = uint64_t(p.rows + kTcM - 1) / kTcM;
        p.ystage = c.ystage && p.V == nmb && p.T == nmb * p.nk && p.rows % 8 == 0 &&
                   (reinterpret_cast<uintptr_t>(p.y) & 15u) == 0 && encode_y_map(&p.ymap, p.y, p.rows, p.batch);
        const size_t smem = p.ystage ? c.smem : std::max(c.smem_base, kExclusiveSmem);
        p.ybuf_off = c.ybuf_off;
        uw_status s;
        if (src == kSrcBf16)
            s = launch_tc_g<kSrcBf16>(p, G, smem, grid, stream);
        else if (src == kSrcPalette4)
            s = launch_tc_g<kSrcPalette4>(p, G, smem, grid, stream);
        else if (src == kSrcExponent)
            s = launch_tc_g<kSrcExponent>(p, G, smem, grid, stream);
        else if (c.tab == 2)
            s = launch_tc_g<kSrcHuffman, 2>(p, G, smem, grid, stream);
        else if (c.tab == 1)
            s = launch_tc_g<kSrcHuffman, 1>(p, G, smem, grid, stream);
        else
            s = launch_tc_g<kSrcHuffman, 0>(p, G, smem, grid, stream);
        if (s != UW_OK)
            return s;
    }
    return UW_OK;
}

}  // namespace uw
