// Tensor-core matmul for batches that make it a real contraction,
// y = x W^T with W [rows, cols], x [batch, cols], fp32 accumulation in
// tensor memory, BF16 out.
//
// D = W x^T is computed as tcgen05.mma tiles with M = 128 rows of W (the A
// operand) and N = the batch padded to a multiple of 16 (the B operand),
// K = 16 per instruction.  A CTA owns 128 rows (four 32-row blocks) and one
// of `splits` ranges of 64-column groups; each group is one pipeline stage
// (K step) of four MMAs.
//
// The A operand lives in tensor memory: a producer warp holds the 64 BF16
// weights of its 32 rows of a K step in registers (lane = row) and writes
// them with one tcgen05.st into the stage's 32 tensor-memory columns (two
// BF16 per column); the MMA reads A from there and B (x) from shared memory.
//
// Warp roles (CTA of 4G + 2 warps):
//   producers  warp w < 4G owns row block w % 4 and the group pairs
//              p = w/4, w/4 + G, ... (K steps 2p, 2p+1):
//                * compressed source: the copy engine stages each pair
//                  (pair_stage.cuh) and the warp decodes its two tiles side
//                  by side (decode.cuh) into registers -- the weights go from
//                  the blob to the tensor cores without touching HBM or
//                  shared memory (Unweight blog, paragraphs on the
//                  reconstructive matmul and on decoding on chip);
//                * bf16 source: the same warps load the uncompressed rows.
//   MMA warp   warp 4G: one thread waits for each stage, issues its four
//              MMAs and commits them to the stage's "empty" barrier.
//   x loader   warp 4G+1: one thread brings each K step's B rows (x, 64
//              columns x Np rows, 128-byte swizzled) into the stage with one
//              tensor-map bulk copy as soon as the stage is free; rows past the
//              batch are zero-filled by the copy.  A stage is full when its four
//              producer warps have arrived and the copy has landed.
//   epilogue   warps 0..3 read the accumulator (tensor-memory lane quarter
//              = warp index) and write y, or fp32 split partials; the last
//              CTA of a row block adds the splits in order.
// Both sources feed the same MMA sequence, so their outputs are
// bit-identical.
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
constexpr int kTcMaxStages = 12;
constexpr uint32_t kTmemCols = 512;

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

// An escaped group's 32 BF16 pairs, from its raw exponents (in the pair
// stage) and its four sign+mantissa chunks.
__device__ __forceinline__ void escaped_pairs(uint32_t ebase, uint32_t em, const uint4 (&sm)[4], uint32_t (&q)[32]) {
    uint4 e[4];
    escape_read(ebase, em, e);
#pragma unroll
    for (int I = 0; I < 32; I++)
        q[I] = escape_pair(e, I, sm_word(sm, I >> 1));
}

// The four sign+mantissa chunks of a lane's row: from the pair stage in
// shared memory, or from global memory.
__device__ __forceinline__ void sm_chunks(uint32_t s_lane, uint32_t stride, uint4 (&sm)[4]) {
#pragma unroll
    for (int c = 0; c < 4; c++)
        sm[c] = lds128(s_lane + uint32_t(c) * stride);
}
__device__ __forceinline__ void sm_chunks(const uint8_t *g_lane, uint32_t stride, uint4 (&sm)[4]) {
#pragma unroll
    for (int c = 0; c < 4; c++)
        sm[c] = __ldg(reinterpret_cast<const uint4 *>(g_lane + c * stride));
}

// kPrivate (Huffman source, codes-only stages): the pair table as 32
// lane-private copies, every lookup one shared-memory wavefront, as in the
// batch-1 GEMV; it fits beside the x stages up to batch ~64.
template <int G, int kSrc, bool kSmStaged, bool kPrivate>
__global__ void __launch_bounds__((4 * G + 2) * 32, 1) gemm_tc_kernel(const __grid_constant__ TcParams p) {
    constexpr int P = 4 * G;  // producer warps
    constexpr bool kCompressed = kSrc == kSrcHuffman;
    constexpr bool kP4 = kSrc == kSrcPalette4;
    constexpr bool kExp = kSrc == kSrcExponent;
    static_assert(!kPrivate || (kSrc == kSrcHuffman && !kSmStaged), "private tables: Huffman codes-only stages");
    constexpr int kStride = kPrivate ? kStridePrivate : kStrideShared;
    extern __shared__ unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t bars[2 * kTcMaxStages + 1];
    __shared__ __align__(8) uint64_t pbars[P * kPairStages];
    __shared__ PairMeta metas[P * kPairStages];
    __shared__ uint32_t tmem_slot;
    __shared__ int last_cta;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const BlobView &v = p.v;
    const int S = p.S, Np = p.Np;
    const uint32_t gpr = uint32_t(p.cols / kGroup);
    const uint32_t nrb = uint32_t((p.rows + kTileRows - 1) / kTileRows);
    const uint32_t mb = blockIdx.x;
    const int split = blockIdx.y;
    const uint32_t kg_lo = uint32_t(uint64_t(gpr) * split / p.splits);
    const uint32_t kg_hi = uint32_t(uint64_t(gpr) * (split + 1) / p.splits);
    const uint32_t nk = kg_hi - kg_lo, npr = (nk + 1) / 2;
    const uint32_t a0col = p.a0col;  // first tensor-memory column of the A stages

    // shared memory: [pad to 1024][B stages][private tables (kPrivate)][decode
    // tables][per producer warp kPairStages pair stages]
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
    const uint32_t bstage = uint32_t(Np) * 128u;
    const uint32_t b0 = raw + pad;
    const uint32_t priv = b0 + uint32_t(S) * bstage;
    unsigned char *dec = smem_raw + pad + size_t(S) * bstage + (kPrivate ? size_t(kPrivateLutBytes) : 0);
    const uint32_t full0 = smem_addr(&bars[0]), empty0 = smem_addr(&bars[kTcMaxStages]);
    const uint32_t done = smem_addr(&bars[2 * kTcMaxStages]);
    // pair stages: with the sign+mantissa bytes (kSmStaged) or codes only
    const uint32_t sbytes = kSmStaged ? pair_stage_bytes(v.tdata) : code_stage_bytes(v.tdata);
    const uint32_t smoff = pair_stage_smoff(v.tdata);
    const uint32_t pst0 = (smem_addr(dec + kCommonSmemBytes) + 127u) & ~127u;

    if (warp == P)
        tmem_alloc(smem_addr(&tmem_slot), kTmemCols);
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; s++) {
            mbar_init(full0 + 8u * s, 5);  // four producer warps + the x copy's expect_tx
            mbar_init(empty0 + 8u * s, 1);
        }
        mbar_init(done, 1);
        for (int i = 0; i < P * kPairStages; i++)
            mbar_init(smem_addr(&pbars[i]), 1);
        mbar_init_fence();
    }
    __syncthreads();

    // producer identity: row block rb, pairs g, g + G, ...
    const int rbl = warp & 3, grp = warp >> 2;
    const uint32_t rb = mb * 4 + uint32_t(rbl);
    const bool producer = warp < P;
    const bool rb_ok = producer && rb < nrb;
    const uint32_t my_pairs = producer && uint32_t(grp) < npr ? (npr - uint32_t(grp) + G - 1) / G : 0u;
    const uint32_t st0 = pst0 + uint32_t(warp) * kPairStages * sbytes;
    const uint32_t pbar0 = smem_addr(&pbars[producer ? warp * kPairStages : 0]);
    PairMeta *meta = &metas[producer ? warp * kPairStages : 0];
    DecodeShared ds{};
    uint32_t nissued = 0, o_next = 0;
    // palette-4 source: one 256-entry pair table (entry b = palette[b >> 4] << 23 |
    // palette[b & 15] << 7) where the decode tables would be
    const uint32_t ptab = smem_addr(dec);
    if constexpr (kP4) {
        for (int b = threadIdx.x; b < 256; b += blockDim.x)
            reinterpret_cast<uint32_t *>(dec)[b] =
                (uint32_t(v.palette[b >> 4]) << 23) | (uint32_t(v.palette[b & 15]) << 7);
    }
    if (kCompressed) {
        ds = carve_common(dec);
        // the first two pairs' offsets in one round trip, the tables built
        // while they arrive, then the pairs' copies started
        if (rb_ok && my_pairs > 0)
            o_next = pair_offsets_load2(v, rb * gpr + kg_lo + 2u * uint32_t(grp),
                                        rb * gpr + kg_lo + 2u * (uint32_t(grp) + G));
        build_tables(ds, v);
        if (rb_ok && my_pairs > 0) {
            for (int s = 0; s < kPairStages && nissued < my_pairs; s++) {
                const uint32_t kgA = kg_lo + 2u * (uint32_t(grp) + nissued * G);
                if constexpr (kSmStaged)
                    pair_issue(v, o_next, rb, kgA, kgA + 1 < kg_hi, rb * gpr + kgA, st0 + uint32_t(s) * sbytes, smoff,
                               pbar0 + 8u * s, meta + s);
                else
                    pair_issue_codes(v, o_next, rb, kgA, kgA + 1 < kg_hi, rb * gpr + kgA, st0 + uint32_t(s) * sbytes,
                                     pbar0 + 8u * s, meta + s);
                nissued++;
                o_next = pair_offsets_shift(o_next);
            }
            if (nissued < my_pairs)
                o_next = pair_offsets_load(v, rb * gpr + kg_lo + 2u * (uint32_t(grp) + nissued * G));
        }
    }
    if constexpr (kPrivate) {
        __syncthreads();
        replicate_private(ds, priv);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // Let the next kernel launch only now that this CTA holds its tensor
    // memory: a later CTA on this SM then waits in its own allocation for
    // this one to finish, never the other way round.
    grid_dep_launch();
    grid_dep_wait();  // x (and the twin's weights) may come from the kernel before; the split partials are reused
    const uint32_t tmem = tmem_slot;
    const uint32_t lut = !kCompressed ? 0u : kPrivate ? priv + 4u * uint32_t(lane) : smem_addr(ds.lut);

    if (producer) {
        const int R = !rb_ok ? 0 : rb < v.nfull || !kCompressed ? int(std::min<int64_t>(kTileRows, p.rows - int64_t(rb) * kTileRows))
                                                                  : int(v.tail_rows);
        const uint32_t trow = tmem + (uint32_t(32 * rbl) << 16) + a0col;
        uint32_t bad = 0;
        // sign+mantissa bytes of the current pair, and its chunk 0 in registers
        const uint8_t *sm_cur = nullptr;
        uint4 c0A = make_uint4(0, 0, 0, 0), c0B = c0A;
        if (kCompressed && !kSmStaged && rb_ok && my_pairs > 0) {
            uint32_t R0;
            const uint32_t kg0 = kg_lo + 2u * uint32_t(grp);
            sm_cur = pair_sm_base(v, rb, kg0, rb * gpr + kg0, R0);
            const uint8_t *a = sm_cur + 16u * (uint32_t(lane) < R0 ? uint32_t(lane) : 0u);
            c0A = __ldg(reinterpret_cast<const uint4 *>(a));
            c0B = __ldg(reinterpret_cast<const uint4 *>(kg0 + 1 < kg_hi ? a + 64u * R0 : a));
        }
#pragma unroll 1
        for (uint32_t j = 0; j < my_pairs; j++) {
            const uint32_t pi = uint32_t(grp) + j * G;  // pair index in the CTA's K range
            const uint32_t i0 = 2u * pi, kgA = kg_lo + i0;
            const bool hasB = kgA + 1 < kg_hi;
            uint32_t qA[32], qB[32];
            if (kCompressed) {
                if (rb_ok) {
                    const uint32_t s = j % kPairStages;
                    const uint32_t st = st0 + s * sbytes, pb = pbar0 + 8u * s;
                    mbar_wait(pb, (j / kPairStages) & 1u, p.status, kStatusTimeout);
                    const PairMeta m = meta[s];
                    const bool full = rb < v.nfull;
                    uint32_t gA, gB;
                    if (full) {
                        gA = lds_u8(st + uint32_t(lane));
                        gB = lds_u8(st + 32u + uint32_t(lane));
                    } else {
                        const uint64_t q0 = uint64_t(rb * gpr + kgA) * kTileRows - uint64_t(kTileRows - R) * kgA;
                        const uint32_t l = uint32_t(lane) < uint32_t(R) ? uint32_t(lane) : 0u;
                        gA = __ldg(v.glen + q0 + l);
                        gB = hasB ? __ldg(v.glen + q0 + uint32_t(R) + l) : 0u;
                    }
                    LaneStream la, lb;
                    const uint32_t cA = st + 64u, cB = cA + 16u * m.n16A;
                    uint32_t emA, emB;
                    pair_begin_ready(ds, gA, gB, m.pkA, m.pkB, R, hasB ? R : 0, cA, cB, la, lb, p.status, emA,
                                             emB);
                    const uint32_t ebA = cA + 16u * (m.n16A + m.n16B), ebB = ebA + 64u * m.nescA;
                    // sign+mantissa bytes straight from L2 (prefetched there with the codes), one
                    // 16-byte chunk ahead; chunk 0 of this pair was loaded during the previous one
                    const uint32_t stride = 16u * uint32_t(R);
                    const uint32_t lc = uint32_t(lane) < uint32_t(R) ? uint32_t(lane) : 0u;
                    const uint8_t *gA_sm = sm_cur + 16u * lc, *gB_sm = hasB ? gA_sm + 64u * uint32_t(R) : gA_sm;
                    const bool more = j + 1 < my_pairs;
                    uint32_t Rn = 0;
                    const uint32_t kgN1 = kgA + 2u * G;
                    const uint8_t *sm_nxt = !kSmStaged && more ? pair_sm_base(v, rb, kgN1, rb * gpr + kgN1, Rn) : sm_cur;
                    const uint32_t smA = st + smoff + 16u * uint32_t(lane), smB = smA + 64u * uint32_t(R);
                    uint4 sA = c0A, sB = c0B;
                    if constexpr (kSmStaged) {
                        sA = lds128(smA);
                        sB = lds128(smB);
                    }
                    uint4 nA = sA, nB = sB;
#pragma unroll
                    for (int I = 0; I < 32; I++) {
                        if ((I & 7) == 0) {
                            if constexpr (kSmStaged) {
                                if (I < 24) {
                                    nA = lds128(smA + uint32_t((I >> 3) + 1) * stride);
                                    nB = lds128(smB + uint32_t((I >> 3) + 1) * stride);
                                }
                            } else if (I < 24) {
                                nA = __ldg(reinterpret_cast<const uint4 *>(gA_sm + uint32_t((I >> 3) + 1) * stride));
                                nB = __ldg(reinterpret_cast<const uint4 *>(gB_sm + uint32_t((I >> 3) + 1) * stride));
                            } else if (more) {
                                const uint8_t *a = sm_nxt + 16u * lc;
                                nA = __ldg(reinterpret_cast<const uint4 *>(a));
                                nB = __ldg(reinterpret_cast<const uint4 *>(kgN1 + 1 < kg_hi ? a + 64u * Rn : a));
                            }
                        }
                        qA[I] = decode_pair<kStride>(la, lut, I, word4(sA, (I >> 1) & 3));
                        qB[I] = decode_pair<kStride>(lb, lut, I, word4(sB, (I >> 1) & 3));
                        if ((I & 7) == 7) {
                            sA = nA;
                            sB = nB;
                        }
                    }
                    bad |= tile_check_bits(la) | tile_check_bits(lb);
                    if ((emA | emB) & (1u << lane)) {
                        uint4 smc[4];
                        if ((emA >> lane) & 1u) {
                            if constexpr (kSmStaged)
                                sm_chunks(smA, stride, smc);
                            else
                                sm_chunks(gA_sm, stride, smc);
                            escaped_pairs(ebA, emA, smc, qA);
                        }
                        if ((emB >> lane) & 1u) {
                            if constexpr (kSmStaged)
                                sm_chunks(smB, stride, smc);
                            else
                                sm_chunks(gB_sm, stride, smc);
                            escaped_pairs(ebB, emB, smc, qB);
                        }
                    }
                    c0A = sA;  // chunk 0 of the next pair
                    c0B = sB;
                    sm_cur = sm_nxt;
                    // the pair stage is free: start the pair kPairStages ahead
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (nissued < my_pairs) {
                        const uint32_t kgN = kg_lo + 2u * (uint32_t(grp) + nissued * G);
                        if constexpr (kSmStaged)
                            pair_issue(v, o_next, rb, kgN, kgN + 1 < kg_hi, rb * gpr + kgN, st, smoff, pb, meta + s);
                        else
                            pair_issue_codes(v, o_next, rb, kgN, kgN + 1 < kg_hi, rb * gpr + kgN, st, pb, meta + s);
                        nissued++;
                        if (nissued < my_pairs)
                            o_next = pair_offsets_load(v, rb * gpr + kg_lo + 2u * (uint32_t(grp) + nissued * G));
                    }
                    __syncwarp();
                } else {
#pragma unroll
                    for (int I = 0; I < 32; I++) {
                        qA[I] = 0u;
                        qB[I] = 0u;
                    }
                }
            } else if constexpr (kP4 || kExp) {
                // the intermediate form (4-bit palette indices rebuilt through the
                // pair table, or exponent bytes) and the sign+mantissa bytes of the
                // lane's row, one tile after the other; palette-4 escaped groups from
                // their raw exponents
                const bool ok = rb_ok && lane < R;
                const uint32_t lc = ok ? uint32_t(lane) : 0u;
                constexpr int NI = kP4 ? 2 : 4;  // 16-byte chunks of the form per row
                auto rebuild = [&](uint32_t kg, bool has, uint32_t (&q)[32]) {
                    const uint64_t q0 = uint64_t(kTileRows) * rb * gpr + uint64_t(R) * kg;
                    uint4 ix[NI], sx[4];
#pragma unroll
                    for (int c = 0; c < NI; c++)
                        ix[c] = __ldg(reinterpret_cast<const uint4 *>(p.p4 + 16 * NI * q0 + 16 * lc + c * 16 * R));
#pragma unroll
                    for (int c = 0; c < 4; c++)
                        sx[c] = __ldg(reinterpret_cast<const uint4 *>(v.sm + 64 * q0 + 16 * lc + c * 16 * R));
                    const uint32_t g = kP4 ? __ldg(v.glen + q0 + lc) : 1u;
#pragma unroll
                    for (int I = 0; I < 32; I++) {
                        if constexpr (kP4) {
                            const uint32_t b = (word4(ix[I >> 4], (I >> 2) & 3) >> (8 * (I & 3))) & 0xFFu;
                            q[I] = lop3_merge(prmt(sm_word(sx, I >> 1), 0u, (I & 1) ? 0xB3A2u : 0x9180u),
                                              lds32(ptab + 4u * b));
                        } else {
                            q[I] = escape_pair(ix, I, sm_word(sx, I >> 1));
                        }
                    }
                    const uint32_t em = __ballot_sync(0xffffffffu, ok && has && g == 0u);
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
                            q[I] = escape_pair(e, I, sm_word(sx, I >> 1));
                    }
                    if (!(ok && has)) {
#pragma unroll
                        for (int I = 0; I < 32; I++)
                            q[I] = 0u;
                    }
                };
                // the next pair's form and sign+mantissa bytes (both tiles contiguous) into L2
                if (lane == 0 && rb_ok && j + 1 < my_pairs) {
                    const uint32_t kgN = kgA + 2u * G;
                    const uint32_t nt = kgN + 1 < kg_hi ? 2u : 1u;
                    const uint64_t q0 = uint64_t(kTileRows) * rb * gpr + uint64_t(R) * kgN;
                    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(p.p4 + 16 * NI * q0),
                                 "r"(16u * NI * uint32_t(R) * nt) : "memory");
                    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(v.sm + 64 * q0),
                                 "r"(64u * uint32_t(R) * nt) : "memory");
                }
                rebuild(kgA, true, qA);
                rebuild(hasB ? kgA + 1 : kgA, hasB, qB);
            } else {
                const int64_t n = int64_t(rb) * kTileRows + lane;
                const bool ok = rb_ok && n < p.rows;
                const uint4 *row = reinterpret_cast<const uint4 *>(p.w + (ok ? n : 0) * p.cols) + size_t(kgA) * 8;
#pragma unroll
                for (int c = 0; c < 8; c++) {
                    const uint4 a = ok ? __ldg(row + c) : make_uint4(0, 0, 0, 0);
                    const uint4 b = ok && hasB ? __ldg(row + 8 + c) : make_uint4(0, 0, 0, 0);
                    qA[4 * c] = a.x, qA[4 * c + 1] = a.y, qA[4 * c + 2] = a.z, qA[4 * c + 3] = a.w;
                    qB[4 * c] = b.x, qB[4 * c + 1] = b.y, qB[4 * c + 2] = b.z, qB[4 * c + 3] = b.w;
                }
            }
            // hand the two K steps to the MMA warp once their stages are free
            const uint32_t sA_ = i0 % uint32_t(S), sB_ = (i0 + 1) % uint32_t(S);
            const uint32_t uA = i0 / uint32_t(S), uB = (i0 + 1) / uint32_t(S);
            if (uA > 0)
                mbar_wait(empty0 + 8u * sA_, (uA - 1) & 1u, p.status, kStatusTimeout);
            if (hasB && uB > 0)
                mbar_wait(empty0 + 8u * sB_, (uB - 1) & 1u, p.status, kStatusTimeout);
            tc_fence_after();
            tmem_st32(trow + 32u * sA_, qA);
            if (hasB)
                tmem_st32(trow + 32u * sB_, qB);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(full0 + 8u * sA_);
                if (hasB)
                    mbar_arrive(full0 + 8u * sB_);
            }
        }
        tile_check_flush(bad, p.status);
    } else if (warp == P) {
        if (lane == 0) {  // the MMA warp
            const uint32_t idesc = idesc_bf16_f32(kTcM, Np);
#pragma unroll 1
            for (uint32_t i = 0; i < nk; i++) {
                const uint32_t s = i % uint32_t(S);
                mbar_wait(full0 + 8u * s, (i / uint32_t(S)) & 1u, p.status, kStatusTimeout);
                tc_fence_after();
                const uint32_t b_st = b0 + s * bstage;
#pragma unroll
                for (int k = 0; k < 4; k++)
                    mma_ts(tmem, tmem + a0col + 32u * s + 8u * k, sdesc_sw128(b_st + 32u * k), idesc, (i | k) != 0);
                mma_commit(empty0 + 8u * s);
            }
            mma_commit(done);
        }
    } else if (lane == 0) {  // the x loader
#pragma unroll 1
        for (uint32_t i = 0; i < nk; i++) {
            const uint32_t s = i % uint32_t(S), u = i / uint32_t(S);
            if (u > 0)
                mbar_wait(empty0 + 8u * s, (u - 1) & 1u, p.status, kStatusTimeout);
            mbar_expect_tx(full0 + 8u * s, bstage);
            tma_load_2d(b0 + s * bstage, &p.xmap, int((kg_lo + i) * kGroup), 0, full0 + 8u * s);
        }
    }
    __syncwarp();

    // epilogue: tensor-memory lane quarter `warp` holds rows n0 + 32*warp + lane
    const int64_t n = int64_t(mb) * kTcM + 32 * warp + lane;
    if (warp < 4) {
        mbar_wait(done, 0u, p.status, kStatusTimeout);
        tc_fence_after();
#pragma unroll 1
        for (int c0 = 0; c0 < Np; c0 += 16) {
            uint32_t vv[16];
            tmem_ld16(tmem + (uint32_t(32 * warp) << 16) + uint32_t(c0), vv);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; j++) {
                const int b = c0 + j;
                if (b < p.batch && n < p.rows) {
                    const float f = __uint_as_float(vv[j]);
                    if (p.splits == 1)
                        p.y[int64_t(b) * p.rows + n] = __bfloat16_as_ushort(__float2bfloat16_rn(f));
                    else
                        p.partial[((int64_t(mb) * p.splits + split) * Np + b) * kTcM + 32 * warp + lane] = f;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == P)
        tmem_dealloc(tmem, kTmemCols);
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
    for (int t = threadIdx.x; t < p.batch * kTcM; t += blockDim.x) {
        const int b = t / kTcM, r = t % kTcM;
        const int64_t nn = int64_t(mb) * kTcM + r;
        if (nn >= p.rows)
            continue;
        const float *ps = p.partial + (int64_t(mb) * p.splits * Np + b) * kTcM + r;
        float tot = __ldcg(ps);
        for (int sp = 1; sp < p.splits; sp++)
            tot += __ldcg(ps + int64_t(sp) * Np * kTcM);
        p.y[int64_t(b) * p.rows + nn] = __bfloat16_as_ushort(__float2bfloat16_rn(tot));
    }
    if (threadIdx.x == 0)
        p.counters[mb] = 0;
}

template <int G, int kSrc, bool kSmStaged, bool kPrivate>
uw_status launch_tc_one(const TcParams &p, size_t smem, cudaStream_t stream) {
    auto kern = gemm_tc_kernel<G, kSrc, kSmStaged, kPrivate>;
    if (!ensure_smem(kern, smem))
        return UW_ERR_CUDA;
    const dim3 grid(unsigned((p.rows + kTcM - 1) / kTcM), unsigned(p.splits));
    return launch_overlapped(kern, grid, dim3((4 * G + 2) * 32), smem, stream, p) == cudaSuccess ? UW_OK : UW_ERR_CUDA;
}

template <int kSrc, bool kSmStaged, bool kPrivate = false>
uw_status launch_tc_g(const TcParams &p, int G, size_t smem, cudaStream_t stream) {
    return G == 1 ? launch_tc_one<1, kSrc, kSmStaged, kPrivate>(p, smem, stream)
           : G == 2 ? launch_tc_one<2, kSrc, kSmStaged, kPrivate>(p, smem, stream)
                    : launch_tc_one<3, kSrc, kSmStaged, kPrivate>(p, smem, stream);
}

// Tensor-memory columns before the A stages (the accumulator's Np, rounded up to 32).
uint32_t a0_col(int Np) { return (uint32_t(Np) + 31u) & ~31u; }

// Shared memory of a launch; `staged` (Huffman source): the producers' pair
// stages hold the sign+mantissa bytes too (otherwise the producers read
// those from L2); `priv`: 32 lane-private copies of the pair table.
size_t tc_smem(int G, int S, int Np, int src, bool staged, uint32_t tdata, bool priv = false) {
    size_t s = 1024 + size_t(S) * size_t(Np) * 128 + (priv ? size_t(kPrivateLutBytes) : 0);
    if (src == kSrcHuffman)
        s += size_t(kCommonSmemBytes) + 128 +
             size_t(4 * G) * kPairStages * (staged ? pair_stage_bytes(tdata) : code_stage_bytes(tdata));
    else if (src == kSrcPalette4 || src == kSrcExponent)
        s += 256 * 4;  // the pair table (palette-4)
    return s;
}

int tc_stages(int G, int Np, int src, bool staged, uint32_t tdata, bool priv = false) {
    int S = std::min<int>(kTcMaxStages, int((kTmemCols - a0_col(Np)) / 32));
    while (S > 1 && tc_smem(G, S, Np, src, staged, tdata, priv) > size_t(kMaxSmemPerBlock - 1024))
        S--;
    return S;
}

}  // namespace

int gemm_tc_stages(int G, int Np, int src, uint32_t tdata) { return tc_stages(G, Np, src, false, tdata); }

int64_t gemm_tc_partial_floats(int64_t rows, int64_t batch, int splits) {
    if (splits <= 1)
        return 0;
    const int64_t np = std::min<int64_t>((batch + 15) / 16 * 16, kTcMaxBatch);
    return (rows + kTcM - 1) / kTcM * splits * np * kTcM;
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

uw_status launch_gemm_tc(const TcParams &base, int G, int src, cudaStream_t stream) {
    const int64_t gpr = base.cols / kGroup;
    if (base.splits < 1 || base.splits > gpr || G < 1 || G > 3)
        return UW_ERR_UNSUPPORTED;
    if (uint64_t(base.rows / kTileRows + 1) * uint64_t(gpr) >= (uint64_t(1) << 32))
        return UW_ERR_UNSUPPORTED;  // tile indices are 32-bit
    for (int64_t b0 = 0; b0 < base.batch; b0 += kTcMaxBatch) {
        TcParams p = base;
        p.batch = std::min<int64_t>(kTcMaxBatch, base.batch - b0);
        p.x = base.x + b0 * base.cols;
        p.y = base.y + b0 * base.rows;
        p.Np = int((p.batch + 15) / 16 * 16);
        p.a0col = a0_col(p.Np);
        p.tmem_cols = kTmemCols;
        if (!encode_x_map(&p.xmap, p.x, p.cols, p.batch, p.Np))
            return UW_ERR_CUDA;
        // Huffman source: stage the sign+mantissa bytes in shared memory when that
        // leaves each producer group its two K steps (and some slack); read them
        // from L2 otherwise
        // Huffman source, first choice: lane-private tables (conflict-free
        // lookups) with codes-only stages, when they leave each producer group
        // its two K steps and some slack
        const bool priv = src == kSrcHuffman && tc_stages(G, p.Np, kSrcHuffman, false, p.v.tdata, true) >= 2 * G + 2;
        const bool staged =
            !priv && src == kSrcHuffman && tc_stages(G, p.Np, kSrcHuffman, true, p.v.tdata) >= 2 * G + 2;
        p.S = tc_stages(G, p.Np, src, staged, p.v.tdata, priv);
        if (p.S < 2 * G)
            return UW_ERR_UNSUPPORTED;  // each producer group works on two K steps at once
        const size_t smem = tc_smem(G, p.S, p.Np, src, staged, p.v.tdata, priv);
        uw_status s;
        if (src == kSrcBf16)
            s = launch_tc_g<kSrcBf16, false>(p, G, smem, stream);
        else if (src == kSrcPalette4)
            s = launch_tc_g<kSrcPalette4, false>(p, G, smem, stream);
        else if (src == kSrcExponent)
            s = launch_tc_g<kSrcExponent, false>(p, G, smem, stream);
        else if (priv)
            s = launch_tc_g<kSrcHuffman, false, true>(p, G, smem, stream);
        else if (staged)
            s = launch_tc_g<kSrcHuffman, true>(p, G, smem, stream);
        else
            s = launch_tc_g<kSrcHuffman, false>(p, G, smem, stream);
        if (s != UW_OK)
            return s;
    }
    return UW_OK;
}

}  // namespace uw
