// Batch-1 GEMV on "column range" CTAs, y = x W^T, fp32 accumulation.
//
// A CTA owns `rb_per_cta` consecutive 32-row blocks and every column.  Its W
// warps split the 64-column groups into W contiguous ranges (warp w: groups
// k0(w) .. k1(w)-1).  A warp walks its row blocks and, within one, its groups
// two at a time: a "pair" is the tiles (rb, kg) and (rb, kg+1), which sit
// next to each other in every section of the blob.
//   * compressed source: the copy engine brings each pair's glen, code
//     region, escaped exponents and sign+mantissa bytes into one of the
//     warp's two shared-memory stages (bulk copies completing on an
//     mbarrier), one pair ahead of the decode.  The two tiles of a pair are
//     decoded side by side (two dependency chains per lane, decode.cuh) and
//     each BF16 weight pair is multiplied straight from the register it was
//     rebuilt in -- the weights never exist in memory (Unweight blog,
//     paragraphs on the reconstructive matmul and on decompressing into fast
//     on-chip memory);
//   * bf16 source: the same warps load the uncompressed rows.
// Both compute every tile partial and every sum below in the same order, so
// the results are bit-identical.  Products use the mixed-precision
// fma.rn.f32.bf16 (BF16 x BF16 is exact in fp32, so each step is one
// correctly rounded fp32 add of the exact product).
//
// Order of the sum for output n (row j of block rb):
//   tile partial  p(kg) = acc_even + acc_odd     (k even / odd within the group)
//   warp partial  s_w   = ((0 + p(k0)) + p(k0+1)) + ...   over the warp's groups
//   y                   = ((s_0 + s_1) + s_2) + ...        over the warps
// then round to nearest even BF16.
#include <cuda_bf16.h>

#include "decode.cuh"
#include "kernels.h"
#include "pair_stage.cuh"
#include "tc.cuh"

namespace uw {

namespace {

constexpr int kMaxColWarps = 32;

// A 16-byte read-only load that does not allocate in L1: the sign+mantissa
// chunks are read once, and beside 224 KB of shared memory L1 is small
// enough that they would evict x.
__device__ __forceinline__ uint4 ldg_stream(const void *p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

__device__ __forceinline__ void fma_bf16x2(float &a0, float &a1, uint32_t w, uint32_t x) {
    asm("{\n\t.reg .b16 wl, wh, xl, xh;\n\t"
        "mov.b32 {wl, wh}, %2;\n\t"
        "mov.b32 {xl, xh}, %3;\n\t"
        "fma.rn.f32.bf16 %0, wl, xl, %0;\n\t"
        "fma.rn.f32.bf16 %1, wh, xh, %1;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "r"(w), "r"(x));
}

// Group range of warp w out of W over gpr groups.
__device__ __forceinline__ void warp_cols(uint32_t gpr, int w, int W, uint32_t &k0, uint32_t &k1) {
    k0 = uint32_t(uint64_t(gpr) * uint32_t(w) / uint32_t(W));
    k1 = uint32_t(uint64_t(gpr) * uint32_t(w + 1) / uint32_t(W));
}

// Fill the CTA's x slab: gpr groups x 32 BF16 pairs.
__device__ __forceinline__ void load_x_all(const GemvParams &p, uint32_t *xs, uint32_t gpr) {
    const uint32_t *x32 = reinterpret_cast<const uint32_t *>(p.x);
    for (uint32_t i = threadIdx.x; i < gpr * 32u; i += blockDim.x)
        xs[i] = __ldg(x32 + i);
}

// y for the CTA's rows: the warp partials in order.
template <int W>
__device__ __forceinline__ void cta_reduce(const GemvParams &p, const float *red, uint32_t rb0, uint32_t nrbc) {
    for (uint32_t t = threadIdx.x; t < nrbc * 32u; t += blockDim.x) {
        const uint32_t rl = t >> 5, j = t & 31;
        float s = red[(rl * W) * 32 + j];
#pragma unroll
        for (int w = 1; w < W; w++)
            s += red[(rl * W + w) * 32 + j];
        const int64_t n = int64_t(rb0 + rl) * kTileRows + j;
        if (n < p.rows)
            p.y[n] = __bfloat16_as_ushort(__float2bfloat16_rn(s));
    }
}

// An escaped group's two accumulators, from its raw exponents (in the
// stage) and its sign+mantissa bytes: in the stage (shared address) or in
// global memory (rare; out of line).
__device__ __noinline__ float2 escaped_sum(uint32_t ebase, uint32_t em, uint32_t sm_lane, uint32_t stride,
                                           const uint32_t *x) {
    uint4 e[4], sm[4];
    escape_read(ebase, em, e);
#pragma unroll
    for (int c = 0; c < 4; c++)
        sm[c] = lds128(sm_lane + uint32_t(c) * stride);
    float b0 = 0.f, b1 = 0.f;
#pragma unroll
    for (int I = 0; I < 32; I++)
        fma_bf16x2(b0, b1, escape_pair(e, I, sm_word(sm, I >> 1)), __ldg(x + I));
    return make_float2(b0, b1);
}

__device__ __noinline__ float2 escaped_sum_global(uint32_t ebase, uint32_t em, const uint8_t *sm_lane,
                                                  uint32_t stride, const uint32_t *x) {
    uint4 e[4], sm[4];
    escape_read(ebase, em, e);
#pragma unroll
    for (int c = 0; c < 4; c++)
        sm[c] = __ldg(reinterpret_cast<const uint4 *>(sm_lane + c * stride));
    float b0 = 0.f, b1 = 0.f;
#pragma unroll
    for (int I = 0; I < 32; I++)
        fma_bf16x2(b0, b1, escape_pair(e, I, sm_word(sm, I >> 1)), __ldg(x + I));
    return make_float2(b0, b1);
}

// kPrivate: the pair table as 32 lane-private copies (every lookup one
// shared-memory wavefront); the stages then hold only the codes and the
// sign+mantissa bytes are read from L2, where the copy engine prefetches
// them when the pair is issued.  Otherwise one shared table and stages that
// hold the sign+mantissa bytes too.
template <int W, bool kPrivate>
__device__ __forceinline__ void gemv_col_compressed(const GemvParams &p, int rb_per_cta) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) uint64_t bars[kMaxColWarps * kPairStages];
    constexpr int kStride = kPrivate ? kStridePrivate : kStrideShared;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const BlobView &v = p.v;
    const uint32_t gpr = v.gpr;
    const uint32_t nrb = v.nfull + (v.tail_rows ? 1u : 0u);
    const uint32_t rb0 = blockIdx.x * uint32_t(rb_per_cta);
    const uint32_t rb1 = rb0 + uint32_t(rb_per_cta) < nrb ? rb0 + uint32_t(rb_per_cta) : nrb;
    const uint32_t nrbc = rb1 - rb0;
    uint32_t k0, k1;
    warp_cols(gpr, warp, W, k0, k1);
    const uint32_t np = (k1 - k0 + 1) / 2;  // pairs per row block
    const uint32_t npairs = np * nrbc;
    const uint32_t sbytes = kPrivate ? code_stage_bytes(v.tdata) : pair_stage_bytes(v.tdata);
    const uint32_t smoff = pair_stage_smoff(v.tdata);

    // shared memory: [private tables (kPrivate)][common tables][warp partials
    // rb_per_cta x W x 32][pad to 128][per warp kPairStages stages][per warp
    // kRecRing pair records]
    const uint32_t priv = smem_addr(smem);
    unsigned char *common = smem + (kPrivate ? kPrivateLutBytes : 0);
    const DecodeShared ds = carve_common(common);
    float *red = reinterpret_cast<float *>(common + kCommonSmemBytes);
    const uint32_t cbase = smem_addr(common);
    const uint32_t stage_lo = (cbase + uint32_t(kCommonSmemBytes) + uint32_t(rb_per_cta) * W * 128u + 127u) & ~127u;
    const uint32_t st0 = stage_lo + uint32_t(warp) * kPairStages * sbytes;
    const uint32_t bar0 = smem_addr(&bars[warp * kPairStages]);
    const uint32_t ring = stage_lo + uint32_t(W) * kPairStages * sbytes + uint32_t(warp) * kRecRing * kRecBytes;
    const PairRecSpan span{npairs, rb0, k0, k1, np};

    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < kPairStages; s++)
            mbar_init(bar0 + 8u * s, 1);
        mbar_init_fence();
    }
    __syncwarp();

    // Prologue, ordered so that the memory round trips overlap the table
    // build: the first kRecRound pairs' offsets (one round trip); the 1024
    // table entries; their records and the first two pairs' copies as soon
    // as the offsets are in; chunk 0 of the first pair's sign+mantissa bytes;
    // then the private copies of the table while the copies fly.
    uint32_t nissued = 0;
    const RecLoad first = pair_recs_load(v, span, 0);
    build_tables(ds, v);
    pair_recs_store(v, ring, span, 0, first);
#pragma unroll
    for (int s = 0; s < kPairStages; s++) {
        if (nissued < npairs) {
            pair_issue_rec<!kPrivate>(v, ring + kRecBytes * nissued, st0 + uint32_t(s) * sbytes, smoff,
                                      bar0 + 8u * s);
            nissued++;
        }
    }
    // kPrivate: sign+mantissa bytes of the current pair, and its chunk 0 in
    // registers (loaded during the previous pair)
    const uint8_t *sm_cur = nullptr;
    uint4 c0A = make_uint4(0, 0, 0, 0), c0B = c0A;
    if (kPrivate && npairs > 0) {
        const uint32_t R0 = rb0 < v.nfull ? uint32_t(kTileRows) : v.tail_rows;
        sm_cur = rec_sm(v, ring);
        const uint8_t *a = sm_cur + 16u * (uint32_t(lane) < R0 ? uint32_t(lane) : 0u);
        c0A = __ldg(reinterpret_cast<const uint4 *>(a));
        c0B = __ldg(reinterpret_cast<const uint4 *>(k0 + 1 < k1 ? a + 64u * R0 : a));
    }
    if constexpr (kPrivate) {
        __syncthreads();
        replicate_private(ds, priv);
    }
    __syncthreads();
    grid_dep_wait();  // x may come from the kernel before
    const uint32_t lut = kPrivate ? priv + 4u * uint32_t(lane) : smem_addr(ds.lut);

    PairCursor cur{rb0, k0};
    float s_w = 0.f;  // this warp's partial for row `lane` of row block cur.rb
    uint32_t bad = 0;
    if (npairs == 0)
        for (uint32_t rl = 0; rl < nrbc; rl++)
            red[(rl * W + warp) * 32 + lane] = 0.f;

#pragma unroll 1
    for (uint32_t j = 0; j < npairs; j++) {
        const uint32_t s = j % kPairStages;
        const uint32_t st = st0 + s * sbytes, bar = bar0 + 8u * s;
        mbar_wait(bar, (j / kPairStages) & 1u, p.status, kStatusTimeout);
        const uint32_t rec = ring + kRecBytes * (j % uint32_t(kRecRing));
        const uint4 ra = lds128(rec), rbk = lds128(rec + 16u);
        const uint32_t n16A = ra.w & 0xFFu, n16B = (ra.w >> 8) & 0xFFu, nescA = (ra.w >> 16) & 0x3Fu;
        const bool hasB = cur.kgA + 1 < k1;
        const bool full = cur.rb < v.nfull;
        const int R = full ? kTileRows : int(v.tail_rows);
        // glen: from the stage, or (partial row block) straight from the blob
        uint32_t gA, gB;
        if (full) {
            gA = lds_u8(st + uint32_t(lane));
            gB = lds_u8(st + 32u + uint32_t(lane));
        } else {
            const uint64_t q0 = uint64_t(cur.rb * gpr + cur.kgA) * kTileRows - uint64_t(kTileRows - R) * cur.kgA;
            const uint32_t l = uint32_t(lane) < uint32_t(R) ? uint32_t(lane) : 0u;
            gA = __ldg(v.glen + q0 + l);
            gB = hasB ? __ldg(v.glen + q0 + uint32_t(R) + l) : 0u;
        }
        LaneStream la, lb;
        const uint32_t cA = st + 64u, cB = cA + 16u * n16A;
        uint32_t emA, emB;
        pair_begin_ready(ds, gA, gB, rbk.x, rbk.y, R, hasB ? R : 0, cA, cB, la, lb, p.status, emA, emB);
        const uint32_t ebA = cA + 16u * (n16A + n16B), ebB = ebA + 64u * nescA;
        const uint32_t stride = 16u * uint32_t(R);
        const uint32_t smA = st + smoff + 16u * uint32_t(lane), smB = smA + 64u * uint32_t(R);
        // kPrivate: the pair's bytes in global memory, and the next pair's
        const uint32_t lc = uint32_t(lane) < uint32_t(R) ? uint32_t(lane) : 0u;
        const uint8_t *gA_sm = sm_cur + 16u * lc, *gB_sm = hasB ? gA_sm + 64u * uint32_t(R) : gA_sm;
        const bool more = j + 1 < npairs;
        PairCursor nxt = cur;
        nxt.next(k0, k1);
        const uint32_t Rn = nxt.rb < v.nfull ? uint32_t(kTileRows) : v.tail_rows;
        const uint8_t *sm_nxt =
            kPrivate && more ? rec_sm(v, ring + kRecBytes * ((j + 1) % uint32_t(kRecRing))) : sm_cur;
        // an escaped group is redone after the loop from its sign+mantissa
        // bytes in global memory: have them in L1 by then
        if (kPrivate && ((emA | emB) >> lane) & 1u) {
            const uint8_t *e = ((emA >> lane) & 1u) ? gA_sm : gB_sm;
#pragma unroll
            for (int c = 0; c < 4; c++)
                asm volatile("prefetch.global.L1 [%0];" :: "l"(e + c * stride));
        }
        // x of the two groups, 4 pairs per load, one load ahead (broadcast, L1-resident)
        const uint4 *xA = reinterpret_cast<const uint4 *>(p.x) + size_t(cur.kgA) * 8;
        const uint4 *xB = xA + (hasB ? 8 : 0);
        float aA0 = 0.f, aA1 = 0.f, aB0 = 0.f, aB1 = 0.f;
        uint4 sA = c0A, sB = c0B;
        if constexpr (!kPrivate) {
            sA = lds128(smA);
            sB = lds128(smB);
        }
        uint4 nA = sA, nB = sB;
        uint4 x4A = __ldg(xA), x4B = __ldg(xB), nxA = x4A, nxB = x4B;
#pragma unroll
        for (int I = 0; I < 32; I++) {
            if ((I & 7) == 0) {  // next chunk of sign+mantissa bytes
                if constexpr (!kPrivate) {
                    if (I < 24) {
                        nA = lds128(smA + uint32_t((I >> 3) + 1) * stride);
                        nB = lds128(smB + uint32_t((I >> 3) + 1) * stride);
                    }
                } else if (I < 24) {
                    nA = __ldg(reinterpret_cast<const uint4 *>(gA_sm + uint32_t((I >> 3) + 1) * stride));
                    nB = __ldg(reinterpret_cast<const uint4 *>(gB_sm + uint32_t((I >> 3) + 1) * stride));
                } else if (more) {  // chunk 0 of the next pair
                    const uint8_t *a = sm_nxt + 16u * (uint32_t(lane) < Rn ? uint32_t(lane) : 0u);
                    nA = __ldg(reinterpret_cast<const uint4 *>(a));
                    nB = __ldg(reinterpret_cast<const uint4 *>(nxt.kgA + 1 < k1 ? a + 64u * Rn : a));
                }
            }
            if ((I & 3) == 0) {
                if (I > 0) {
                    x4A = nxA;
                    x4B = nxB;
                }
                if (I < 28) {
                    nxA = __ldg(xA + (I >> 2) + 1);
                    nxB = __ldg(xB + (I >> 2) + 1);
                }
            }
            fma_bf16x2(aA0, aA1, decode_pair<kStride>(la, lut, I, word4(sA, (I >> 1) & 3)), word4(x4A, I));
            fma_bf16x2(aB0, aB1, decode_pair<kStride>(lb, lut, I, word4(sB, (I >> 1) & 3)), word4(x4B, I));
            if ((I & 7) == 7) {
                sA = nA;
                sB = nB;
            }
        }
        bad |= tile_check_bits(la) | tile_check_bits(lb);
        if ((emA >> lane) & 1u) {
            const float2 r = kPrivate ? escaped_sum_global(ebA, emA, gA_sm, stride, reinterpret_cast<const uint32_t *>(xA))
                                      : escaped_sum(ebA, emA, smA, stride, reinterpret_cast<const uint32_t *>(xA));
            aA0 = r.x;
            aA1 = r.y;
        }
        if ((emB >> lane) & 1u) {
            const float2 r = kPrivate ? escaped_sum_global(ebB, emB, gB_sm, stride, reinterpret_cast<const uint32_t *>(xB))
                                      : escaped_sum(ebB, emB, smB, stride, reinterpret_cast<const uint32_t *>(xB));
            aB0 = r.x;
            aB1 = r.y;
        }
        c0A = sA;  // kPrivate: chunk 0 of the next pair
        c0B = sB;
        sm_cur = sm_nxt;
        s_w = s_w + (aA0 + aA1);
        if (hasB)
            s_w = s_w + (aB0 + aB1);
        const uint32_t rb_done = cur.rb;
        cur = nxt;
        if (cur.rb != rb_done) {  // the warp's last pair of this row block
            red[((rb_done - rb0) * W + warp) * 32 + lane] = s_w;
            s_w = 0.f;
        }
        // the stage is free: start the pair kPairStages ahead (the reads above
        // come before the copy engine's writes)
        fence_proxy_async_smem();
        __syncwarp();
        if (nissued < npairs) {
            pair_issue_rec<!kPrivate>(v, ring + kRecBytes * (nissued % uint32_t(kRecRing)), st, smoff, bar);
            // the next round's records, kRecRound - 2 pairs before the first is
            // issued (its ring slots belong to pairs already decoded)
            if (nissued % uint32_t(kRecRound) == 2u && nissued - 2u + uint32_t(kRecRound) < npairs)
                pair_recs_store(v, ring, span, nissued - 2u + uint32_t(kRecRound),
                                pair_recs_load(v, span, nissued - 2u + uint32_t(kRecRound)));
            nissued++;
        }
        __syncwarp();
    }
    tile_check_flush(bad, p.status);
    __syncthreads();
    cta_reduce<W>(p, red, rb0, nrbc);
}

// Batch 1 with 32 lane-private copies of the pair table (taken whenever they
// fit, as for every matrix measured): the pair loop above, trimmed for the
// instruction budget of the decode, plus escaped groups decoded inside the
// main loop.  An escaped group's raw exponents are expanded once into 32
// table-entry words (both exponents of a weight pair in BF16 position, bit
// count 10) in a per-warp slot; the lane then runs the same 32 steps over a
// constant "counting" stream whose 10-bit windows are 0, 1, ..., 31, with
// the slot as its table and stride 4, so step I reads entry I.  The steps,
// the products and their order are exactly those of any other lane, hence
// bit-identical results with no second pass.  More than kEscSlots escaped
// groups in one pair (rare outside heavy-tailed matrices) fall back to the
// second pass from raw exponents.
// (kEscSlots, expand_escapes and the counting stream: pair_stage.cuh)

// Per-warp constants of the batch-1 private-table GEMV.
struct PrivCtx {
    uint32_t lut;    // the lane's column of the private table copies
    uint32_t zero;   // zero stream
    uint32_t cnt;    // counting stream (escaped groups)
    uint32_t slots;  // the warp's escape slots
    uint32_t below;  // lanes below this one
    uint32_t one;    // 1, held in a register
};

// A pair's group lengths reduced over the warp: the lane's own (A | B << 16;
// zero for rows past a partial block and without tile B), their exclusive
// prefix sums and totals (16-bit halves) and the masks of escaped groups.
struct PairScan {
    uint32_t g2, off2, tot2, emA, emB;
};

// The scan of the pair staged at `st` (full row block: glen in the stage;
// partial block of R rows: glen read at group q0).
template <bool kFull>
__device__ __forceinline__ PairScan pair_scan(const BlobView &v, uint32_t st, uint64_t q0, uint32_t R, bool hasB) {
    const int lane = threadIdx.x & 31;
    uint32_t gA, gB;
    if (kFull) {
        gA = lds_u8(st + uint32_t(lane));
        gB = lds_u8(st + 32u + uint32_t(lane));
    } else {
        const uint32_t l = uint32_t(lane) < R ? uint32_t(lane) : 0u;
        gA = __ldg(v.glen + q0 + l);
        gB = hasB ? __ldg(v.glen + q0 + R + l) : 0u;
    }
    const bool vA = kFull || uint32_t(lane) < R, vB = hasB && vA;
    const uint32_t ga = vA ? gA : 0u, gb = vB ? gB : 0u;
    PairScan s;
    s.g2 = ga | (gb << 16);
    uint32_t incl = s.g2;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1)
        asm("{\n\t.reg .b32 u;\n\t.reg .pred q;\n\t"
            "shfl.sync.up.b32 u|q, %0, %1, 0, -1;\n\t"
            "@q add.u32 %0, %0, u;\n\t}"
            : "+r"(incl) : "r"(d));
    s.off2 = incl - s.g2;
    s.tot2 = __shfl_sync(0xffffffffu, incl, 31);
    s.emA = __ballot_sync(0xffffffffu, vA && ga == 0u);
    s.emB = __ballot_sync(0xffffffffu, vB && gb == 0u);
    return s;
}

// The pair after the current one, scanned halfway through the current
// pair's decode so that the scan's round trips overlap the decode.
struct NextPair {
    uint32_t st, bar, parity, R;
    uint64_t q0;
    bool hasB, full;
};

// One pair (tiles A = (rb, kgA), B = (rb, kgA + 1) when hasB) staged at `st`
// and scanned (`sc`): returns the two tiles' partials pA = acc_even + acc_odd
// of A, pB of B.  kFull: a full row block (32 rows: constant strides).  sm:
// the pair's first sign+mantissa byte; chunk 0 of each tile arrives in c0A /
// c0B and chunk 0 of the next pair (at sm_nxt, Rn rows, B when nhasB) leaves
// in them; when `more`, the next pair's stage is waited for and scanned into
// `nsc` after the 16th step.
template <bool kFull>
__device__ __forceinline__ void priv_pair(const GemvParams &p, const PrivCtx &k, uint32_t st, uint32_t pkA,
                                          uint32_t pkB, const PairScan &sc, const NextPair &nb, PairScan &nsc,
                                          uint32_t Rr, bool hasB, const uint8_t *sm, const uint4 *xA, bool more,
                                          const uint8_t *sm_nxt, uint32_t Rn, bool nhasB, uint4 &c0A, uint4 &c0B,
                                          uint32_t &bad, float &pA, float &pB) {
    const BlobView &v = p.v;
    const int lane = threadIdx.x & 31;
    const uint32_t R = kFull ? uint32_t(kTileRows) : Rr;
    const uint32_t n16A = pkA & 0xFFu, n16B = pkB & 0xFFu;
    const uint32_t nescA = (pkA >> 8) & 0xFFu, nescB = (pkB >> 8) & 0xFFu;
    uint32_t ga = sc.g2 & 0xFFFFu, gb = sc.g2 >> 16;
    const uint32_t off2 = sc.off2, tot2 = sc.tot2;
    uint32_t emA = sc.emA, emB = sc.emB;
    // A pair whose tables or group lengths do not add up (a device copy
    // damaged after its header was checked) is flagged and decodes the zero
    // stream in every lane, so no read leaves the stage.
    if (((pkA | pkB) >> 16) != 0u || (tot2 & 0xFFFFu) > 16u * n16A || (tot2 >> 16) > 16u * n16B ||
        uint32_t(__popc(emA)) != nescA || uint32_t(__popc(emB)) != nescB) {
        if (lane == 0)
            atomicOr(p.status, uint32_t(kStatusBadTile));
        ga = 0u;
        gb = 0u;
        emA = 0u;
        emB = 0u;
    }
    const uint32_t cA = st + 64u, cB = cA + 16u * n16A;
    const uint32_t ebA = cB + 16u * n16B, ebB = ebA + 64u * nescA;
    // escaped groups: slots 0.. for A's, then B's, at most kEscSlots
    uint32_t wzA = k.zero, wzB = k.zero, lutA = k.lut, lutB = k.lut, sA_ = kStridePrivate, sB_ = kStridePrivate;
    bool xa = false, xb = false;
    if ((emA | emB) != 0u) {
        const uint32_t pa = __popc(emA), pb = __popc(emB);
        const uint32_t nA = pa < uint32_t(kEscSlots) ? pa : uint32_t(kEscSlots);
        const uint32_t nB = pb < uint32_t(kEscSlots) - nA ? pb : uint32_t(kEscSlots) - nA;
        expand_escapes(nA, ebA, k.slots, 0u);
        expand_escapes(nB, ebB, k.slots, nA);
        __syncwarp();
        const uint32_t rA = __popc(emA & k.below), rB = nA + __popc(emB & k.below);
        xa = (emA >> lane) & 1u;
        xb = (emB >> lane) & 1u;
        if (xa && rA < nA) {
            wzA = k.cnt;
            lutA = k.slots + kEscSlotBytes * rA;
            sA_ = 4u;
            xa = false;  // decoded in the main loop
        }
        if (xb && rB < nA + nB) {
            wzB = k.cnt;
            lutB = k.slots + kEscSlotBytes * rB;
            sB_ = 4u;
            xb = false;
        }
    }
    LaneStream la, lb;
    {
        const uint32_t offA = off2 & 0xFFFFu, offB = off2 >> 16;
        const uint32_t wA = ga != 0u ? ((cA + offA) & ~3u) : wzA;
        const uint32_t wB = gb != 0u ? ((cB + offB) & ~3u) : wzB;
        la.lo = lds32(wA);
        la.hi = lds32(wA + 4);
        la.nx = lds32(wA + 8);
        la.wp = wA + 12;
        la.c = ga != 0u ? 8u * (offA & 3u) : 0u;
        la.expect = ga != 0u ? 8u * (la.wp + ga) + la.c : 0u;
        lb.lo = lds32(wB);
        lb.hi = lds32(wB + 4);
        lb.nx = lds32(wB + 8);
        lb.wp = wB + 12;
        lb.c = gb != 0u ? 8u * (offB & 3u) : 0u;
        lb.expect = gb != 0u ? 8u * (lb.wp + gb) + lb.c : 0u;
    }
    const uint32_t stride = 16u * R;
    const uint32_t lc = (kFull || uint32_t(lane) < R) ? uint32_t(lane) : 0u;
    const uint8_t *gA_sm = sm + 16u * lc, *gB_sm = hasB ? gA_sm + 64u * R : gA_sm;
    const uint4 *xB = xA + (hasB ? 8 : 0);
    float aA0 = 0.f, aA1 = 0.f, aB0 = 0.f, aB1 = 0.f;
    uint4 sA = c0A, sB = c0B, nA = sA, nB = sB;
    uint4 x4A = __ldg(xA), x4B = __ldg(xB), nxA = x4A, nxB = x4B;
#pragma unroll
    for (int I = 0; I < 32; I++) {
        if ((I & 7) == 0) {  // next chunk of sign+mantissa bytes
            if (I < 24) {
                nA = ldg_stream(gA_sm + uint32_t((I >> 3) + 1) * stride);
                nB = ldg_stream(gB_sm + uint32_t((I >> 3) + 1) * stride);
            } else if (more) {  // chunk 0 of the next pair
                const uint8_t *a = sm_nxt + 16u * (uint32_t(lane) < Rn ? uint32_t(lane) : 0u);
                nA = ldg_stream(a);
                nB = ldg_stream(nhasB ? a + 64u * Rn : a);
            }
        }
        if ((I & 3) == 0) {
            if (I > 0) {
                x4A = nxA;
                x4B = nxB;
            }
            if (I < 28) {
                nxA = __ldg(xA + (I >> 2) + 1);
                nxB = __ldg(xB + (I >> 2) + 1);
            }
        }
        if (I == 16 && more) {  // the next pair: its stage and scan
            mbar_wait(nb.bar, nb.parity, p.status, kStatusTimeout);
            nsc = nb.full ? pair_scan<true>(v, nb.st, nb.q0, kTileRows, nb.hasB)
                          : pair_scan<false>(v, nb.st, nb.q0, nb.R, nb.hasB);
        }
        const uint32_t eA = decode_entry_rs(la, lutA, sA_, k.one, I);
        const uint32_t eB = decode_entry_rs(lb, lutB, sB_, k.one, I);
        const uint32_t sel = (I & 1) ? 0xB3A2u : 0x9180u;
        fma_bf16x2(aA0, aA1, lop3_merge(prmt(word4(sA, (I >> 1) & 3), 0u, sel), eA), word4(x4A, I));
        fma_bf16x2(aB0, aB1, lop3_merge(prmt(word4(sB, (I >> 1) & 3), 0u, sel), eB), word4(x4B, I));
        if ((I & 7) == 7) {
            sA = nA;
            sB = nB;
        }
    }
    bad |= tile_check_bits(la) | tile_check_bits(lb);
    if (xa | xb) {  // escaped groups beyond the slots: second pass
        if (xa) {
            const float2 r = escaped_sum_global(ebA, emA, gA_sm, stride, reinterpret_cast<const uint32_t *>(xA));
            aA0 = r.x;
            aA1 = r.y;
        }
        if (xb) {
            const float2 r = escaped_sum_global(ebB, emB, gB_sm, stride, reinterpret_cast<const uint32_t *>(xB));
            aB0 = r.x;
            aB1 = r.y;
        }
    }
    c0A = sA;  // chunk 0 of the next pair
    c0B = sB;
    pA = aA0 + aA1;
    pB = aB0 + aB1;
}

// The batch-1 Huffman GEMV with 32 lane-private copies of the pair table
// (taken whenever they fit, as for every matrix measured): one CTA per SM of
// whole row blocks, the pair loop of gemv_col_compressed with escaped groups
// decoded inside the main loop (see expand_escapes above) and full row
// blocks on a path with constant strides.
template <int W>
__device__ __forceinline__ void gemv_private(const GemvParams &p, int rb_per_cta) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) uint64_t bars[kMaxColWarps * kPairStages];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const BlobView &v = p.v;
    const uint32_t gpr = v.gpr;
    const uint32_t nrb = v.nfull + (v.tail_rows ? 1u : 0u);
    const uint32_t rb0 = blockIdx.x * uint32_t(rb_per_cta);
    const uint32_t rb1 = rb0 + uint32_t(rb_per_cta) < nrb ? rb0 + uint32_t(rb_per_cta) : nrb;
    const uint32_t nrbc = rb1 - rb0;
    uint32_t k0, k1;
    warp_cols(gpr, warp, W, k0, k1);
    const uint32_t np = (k1 - k0 + 1) / 2;  // pairs per row block
    const uint32_t npairs = np * nrbc;
    const uint32_t sbytes = code_stage_bytes(v.tdata);

    // shared memory: [private tables][common tables][counting stream][warp
    // partials nrbc x W x 32][pad to 128][per warp kPairStages stages]
    // [per warp kRecRing pair records][per warp kEscSlots escape slots]
    const uint32_t priv = smem_addr(smem);
    unsigned char *common = smem + kPrivateLutBytes;
    const DecodeShared ds = carve_common(common);
    const uint32_t cnt = smem_addr(common) + uint32_t(kCommonSmemBytes);
    float *red = reinterpret_cast<float *>(common + kCommonSmemBytes + kCountWords * 4);
    const uint32_t stage_lo = (smem_addr(red) + uint32_t(rb_per_cta) * W * 128u + 127u) & ~127u;
    const uint32_t st0 = stage_lo + uint32_t(warp) * kPairStages * sbytes;
    const uint32_t bar0 = smem_addr(&bars[warp * kPairStages]);
    const uint32_t ring = stage_lo + uint32_t(W) * kPairStages * sbytes + uint32_t(warp) * kRecRing * kRecBytes;
    const uint32_t slots = stage_lo + uint32_t(W) * (kPairStages * sbytes + kRecRing * kRecBytes) +
                           uint32_t(warp) * kEscSlots * kEscSlotBytes;
    const PairRecSpan span{npairs, rb0, k0, k1, np};

    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < kPairStages; s++)
            mbar_init(bar0 + 8u * s, 1);
        mbar_init_fence();
    }
    __syncwarp();

    // Prologue: offsets of the first pairs (one round trip, under the table
    // build), the private table copies, the first pair's copies and chunk 0
    // of its sign+mantissa bytes, the counting stream.  The second pair is
    // issued after the dependency wait, so that every warp's first copies
    // are queued before any second ones.
    uint32_t nissued = 0;
    const RecLoad first = pair_recs_load(v, span, 0);
    build_prefix_zero(ds, v);
    build_private(ds, priv);
    pair_recs_store(v, ring, span, 0, first);
    if (npairs > 0) {
        pair_issue_rec<false>(v, ring, st0, 0u, bar0);
        nissued = 1;
    }
    const uint8_t *sm_cur = nullptr;
    uint4 c0A = make_uint4(0, 0, 0, 0), c0B = c0A;
    if (npairs > 0) {
        const uint32_t R0 = rb0 < v.nfull ? uint32_t(kTileRows) : v.tail_rows;
        sm_cur = rec_sm(v, ring);
        const uint8_t *a = sm_cur + 16u * (uint32_t(lane) < R0 ? uint32_t(lane) : 0u);
        c0A = __ldg(reinterpret_cast<const uint4 *>(a));
        c0B = __ldg(reinterpret_cast<const uint4 *>(k0 + 1 < k1 ? a + 64u * R0 : a));
    }
    build_count_stream(cnt);
    __syncthreads();
    grid_dep_wait();  // x may come from the kernel before
    PrivCtx kc;
    kc.lut = priv + 4u * uint32_t(lane);
    kc.zero = smem_addr(ds.zero);
    kc.cnt = cnt;
    kc.slots = slots;
    kc.below = (1u << lane) - 1u;
    kc.one = gpr != 0u ? 1u : 0u;

    PairCursor cur{rb0, k0};
    float s_w = 0.f;  // this warp's partial for row `lane` of row block cur.rb
    uint32_t bad = 0;
    if (npairs == 0)
        for (uint32_t rl = 0; rl < nrbc; rl++)
            red[(rl * W + warp) * 32 + lane] = 0.f;
    // the second pair (see the prologue), then the first pair's stage and scan;
    // every later pair is waited for and scanned halfway through the one before
    PairScan sc{};
    if (npairs > 0) {
        if (nissued < npairs) {
            pair_issue_rec<false>(v, ring + kRecBytes, st0 + sbytes, 0u, bar0 + 8u);
            nissued++;
        }
        mbar_wait(bar0, 0u, p.status, kStatusTimeout);
        const uint4 r0 = lds128(ring + 16u);
        const uint64_t q00 = (uint64_t(r0.w) << 32) | r0.z;
        sc = rb0 < v.nfull ? pair_scan<true>(v, st0, q00, kTileRows, k0 + 1 < k1)
                           : pair_scan<false>(v, st0, q00, v.tail_rows, k0 + 1 < k1);
    }

#pragma unroll 1
    for (uint32_t j = 0; j < npairs; j++) {
        const uint32_t st = st0 + (j & 1u) * sbytes, bar = bar0 + 8u * (j & 1u);
        const uint4 rbk = lds128(ring + kRecBytes * (j % uint32_t(kRecRing)) + 16u);  // pkA, pkB, q0
        const bool hasB = cur.kgA + 1 < k1;
        const bool full = cur.rb < v.nfull;
        const bool more = j + 1 < npairs;
        PairCursor nxt = cur;
        nxt.next(k0, k1);
        const uint32_t Rn = nxt.rb < v.nfull ? uint32_t(kTileRows) : v.tail_rows;
        NextPair nb{};
        const uint8_t *sm_nxt = sm_cur;
        if (more) {
            const uint4 rn = lds128(ring + kRecBytes * ((j + 1) % uint32_t(kRecRing)) + 16u);
            nb.q0 = (uint64_t(rn.w) << 32) | rn.z;
            sm_nxt = v.sm + nb.q0 * kGroup;
            nb.st = st0 + ((j + 1) & 1u) * sbytes;
            nb.bar = bar0 + 8u * ((j + 1) & 1u);
            nb.parity = ((j + 1) >> 1) & 1u;
            nb.R = Rn;
            nb.hasB = nxt.kgA + 1 < k1;
            nb.full = nxt.rb < v.nfull;
        }
        const uint4 *xA = reinterpret_cast<const uint4 *>(p.x) + size_t(cur.kgA) * 8;
        float pA, pB;
        PairScan nsc = sc;
        if (full)
            priv_pair<true>(p, kc, st, rbk.x, rbk.y, sc, nb, nsc, kTileRows, hasB, sm_cur, xA, more, sm_nxt, Rn,
                            nxt.kgA + 1 < k1, c0A, c0B, bad, pA, pB);
        else
            priv_pair<false>(p, kc, st, rbk.x, rbk.y, sc, nb, nsc, v.tail_rows, hasB, sm_cur, xA, more, sm_nxt, Rn,
                             nxt.kgA + 1 < k1, c0A, c0B, bad, pA, pB);
        sc = nsc;
        sm_cur = sm_nxt;
        s_w = s_w + pA;
        if (hasB)
            s_w = s_w + pB;
        const uint32_t rb_done = cur.rb;
        cur = nxt;
        if (cur.rb != rb_done) {  // the warp's last pair of this row block
            red[((rb_done - rb0) * W + warp) * 32 + lane] = s_w;
            s_w = 0.f;
        }
        // the stage is free: start the pair kPairStages ahead (the reads above
        // come before the copy engine's writes)
        fence_proxy_async_smem();
        __syncwarp();
        if (nissued < npairs) {
            pair_issue_rec<false>(v, ring + kRecBytes * (nissued % uint32_t(kRecRing)), st, 0u, bar);
            if (nissued % uint32_t(kRecRound) == 2u && nissued - 2u + uint32_t(kRecRound) < npairs)
                pair_recs_store(v, ring, span, nissued - 2u + uint32_t(kRecRound),
                                pair_recs_load(v, span, nissued - 2u + uint32_t(kRecRound)));
            nissued++;
        }
        __syncwarp();
    }
    tile_check_flush(bad, p.status);
    __syncthreads();
    cta_reduce<W>(p, red, rb0, nrbc);
}

template <int W>
__device__ __forceinline__ void gemv_col_bf16(const GemvParams &p, int rb_per_cta) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t gpr = uint32_t(p.cols / kGroup);
    const uint32_t nrb = uint32_t((p.rows + kTileRows - 1) / kTileRows);
    const uint32_t rb0 = blockIdx.x * uint32_t(rb_per_cta);
    const uint32_t rb1 = rb0 + uint32_t(rb_per_cta) < nrb ? rb0 + uint32_t(rb_per_cta) : nrb;
    const uint32_t nrbc = rb1 - rb0;
    uint32_t k0, k1;
    warp_cols(gpr, warp, W, k0, k1);

    // shared memory: [x slab gpr x 32 pairs][warp partials rb_per_cta x W x 32]
    uint32_t *xs = reinterpret_cast<uint32_t *>(smem);
    float *red = reinterpret_cast<float *>(smem + size_t(gpr) * 128);
    grid_dep_wait();  // x may come from the kernel before
    load_x_all(p, xs, gpr);
    __syncthreads();

#pragma unroll 1
    for (uint32_t rl = 0; rl < nrbc; rl++) {
        const int64_t n = int64_t(rb0 + rl) * kTileRows + lane;
        const bool ok = n < p.rows;
        const uint4 *row = reinterpret_cast<const uint4 *>(p.w + (ok ? n : 0) * p.cols);
        float s_w = 0.f;
        uint4 cur[8], nxt[8];
#pragma unroll
        for (int c = 0; c < 8; c++)
            nxt[c] = (ok && k0 < k1) ? __ldg(row + size_t(k0) * 8 + c) : make_uint4(0, 0, 0, 0);
#pragma unroll 1
        for (uint32_t kg = k0; kg < k1; kg++) {
#pragma unroll
            for (int c = 0; c < 8; c++)
                cur[c] = nxt[c];
            if (kg + 1 < k1) {
#pragma unroll
                for (int c = 0; c < 8; c++)
                    nxt[c] = ok ? __ldg(row + size_t(kg + 1) * 8 + c) : make_uint4(0, 0, 0, 0);
            }
            const uint32_t xaddr = smem_addr(xs) + kg * 128u;
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int I = 0; I < 32; I++)
                fma_bf16x2(a0, a1, word4(cur[I >> 2], I & 3), lds32(xaddr + 4u * I));
            s_w = s_w + (a0 + a1);
        }
        red[(rl * W + warp) * 32 + lane] = s_w;
    }
    __syncthreads();
    cta_reduce<W>(p, red, rb0, nrbc);
}

// The uncompressed twin with its tiles brought by the copy engine: one
// 32-row x 64-column tile of W per 2-D tensor-map copy (128-byte swizzle:
// 16-byte chunk c of tile row r at chunk position c ^ (r % 8), so the 32
// lanes' 16-byte reads of one chunk hit distinct banks), kTwinStages tiles in
// flight per warp.  Same warps, groups and order of every sum as
// gemv_col_bf16 (and the compressed paths), so the same bits.
constexpr uint32_t kTwinTileBytes = kTileRows * kGroup * 2;  // 4 KB

size_t twin_tma_smem(int warps, int rb_per_cta, int gpr, int stages) {
    return size_t(gpr) * 128 + size_t(rb_per_cta) * warps * 128 + 1024 + size_t(warps) * stages * kTwinTileBytes;
}

template <int W, int kS>
__global__ void __launch_bounds__(W * 32, 1)
    gemv_kg_twin_tma_kernel(const __grid_constant__ GemvParams p, const __grid_constant__ CUtensorMap wmap,
                            int rb_per_cta) {
    grid_dep_launch();
    extern __shared__ __align__(1024) unsigned char smem[];
    __shared__ __align__(8) uint64_t bars[kMaxColWarps * kS];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t gpr = uint32_t(p.cols / kGroup);
    const uint32_t nrb = uint32_t((p.rows + kTileRows - 1) / kTileRows);
    const uint32_t rb0 = blockIdx.x * uint32_t(rb_per_cta);
    const uint32_t rb1 = rb0 + uint32_t(rb_per_cta) < nrb ? rb0 + uint32_t(rb_per_cta) : nrb;
    const uint32_t nrbc = rb1 - rb0;
    uint32_t k0, k1;
    warp_cols(gpr, warp, W, k0, k1);
    const uint32_t per = k1 - k0, ntile = per * nrbc;
    // shared memory: [x slab gpr x 32 pairs][warp partials][pad to 1024][per warp kS tiles]
    uint32_t *xs = reinterpret_cast<uint32_t *>(smem);
    float *red = reinterpret_cast<float *>(smem + size_t(gpr) * 128);
    const uint32_t tiles0 = (smem_addr(red) + uint32_t(rb_per_cta) * W * 128u + 1023u) & ~1023u;
    const uint32_t st0 = tiles0 + uint32_t(warp) * kS * kTwinTileBytes;
    const uint32_t bar0 = smem_addr(&bars[warp * kS]);
    auto issue = [&](uint32_t i) {  // tile i of the warp: row block rb0 + i / per, group k0 + i % per
        const uint32_t s = i % uint32_t(kS);
        mbar_expect_tx(bar0 + 8u * s, kTwinTileBytes);
        tma_load_2d(st0 + s * kTwinTileBytes, &wmap, int((k0 + i % per) * kGroup), int((rb0 + i / per) * kTileRows),
                    bar0 + 8u * s);
    };
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < kS; s++)
            mbar_init(bar0 + 8u * s, 1);
        mbar_init_fence();
    }
    __syncwarp();
    grid_dep_wait();  // x and W may come from the kernel before (W from a decompress)
    if (lane == 0)
        for (uint32_t i = 0; i < uint32_t(kS) && i < ntile; i++)
            issue(i);
    load_x_all(p, xs, gpr);
    __syncthreads();
    float s_w = 0.f;
    if (ntile == 0)
        for (uint32_t rl = 0; rl < nrbc; rl++)
            red[(rl * W + warp) * 32 + lane] = 0.f;
#pragma unroll 1
    for (uint32_t i = 0; i < ntile; i++) {
        const uint32_t s = i % uint32_t(kS);
        mbar_wait(bar0 + 8u * s, (i / uint32_t(kS)) & 1u, p.status, kStatusTimeout);
        const uint32_t kg = k0 + i % per;
        const uint32_t row = st0 + s * kTwinTileBytes + uint32_t(lane) * 128u;
        const uint32_t xaddr = smem_addr(xs) + kg * 128u;
        uint4 wv[8];
#pragma unroll
        for (int c = 0; c < 8; c++)
            wv[c] = lds128(row + 16u * (uint32_t(c) ^ (uint32_t(lane) & 7u)));
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int I = 0; I < 32; I++)
            fma_bf16x2(a0, a1, word4(wv[I >> 2], I & 3), lds32(xaddr + 4u * I));
        s_w = s_w + (a0 + a1);
        if (i % per == per - 1) {  // the warp's last group of this row block
            red[((i / per) * W + warp) * 32 + lane] = s_w;
            s_w = 0.f;
        }
        // the stage is free once every lane has read it: refill it
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && i + kS < ntile)
            issue(i + kS);
        __syncwarp();
    }
    __syncthreads();
    cta_reduce<W>(p, red, rb0, nrbc);
}

// Palette-4 and exponent sources (the blog's palette and exponent-only
// pipelines): the twin's loop -- same warps, groups and order of every sum,
// so the results are bit-identical -- with each group's BF16 pairs rebuilt
// from an intermediate form and its sign+mantissa bytes.
//   * palette-4: a byte of two 4-bit indices is looked up in a 256-entry
//     pair table (entry b = palette[b >> 4] << 23 | palette[b & 15] << 7,
//     both exponents in BF16 position) kept as 32 lane-private copies at a
//     32 KB-aligned shared address, so that one three-input logic op both
//     masks the byte out of the index word and adds the lane's column, and
//     every lookup is one shared-memory wavefront.  Escaped groups (glen 0)
//     take their exponents from the blob's escape section instead.
//   * exponents: the group's 64 exponent bytes, merged like raw escaped
//     exponents (escaped groups need nothing else).
template <int W, int kSrc>
__device__ __forceinline__ void gemv_col_formed(const GemvParams &p, int rb_per_cta) {
    constexpr bool kP4 = kSrc == kSrcPalette4;
    extern __shared__ __align__(128) unsigned char smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const BlobView &v = p.v;
    const uint32_t gpr = v.gpr;
    const uint32_t nrb = v.nfull + (v.tail_rows ? 1u : 0u);
    const uint32_t rb0 = blockIdx.x * uint32_t(rb_per_cta);
    const uint32_t rb1 = rb0 + uint32_t(rb_per_cta) < nrb ? rb0 + uint32_t(rb_per_cta) : nrb;
    const uint32_t nrbc = rb1 - rb0;
    uint32_t k0, k1;
    warp_cols(gpr, warp, W, k0, k1);

    // shared memory: [pad to 32 KB][pair table 256 x 32 lanes][x slab gpr x 32 pairs]
    // [warp partials rb_per_cta x W x 32]
    const uint32_t base = smem_addr(smem);
    const uint32_t tab = (base + 32767u) & ~32767u;
    unsigned char *after = smem + (tab - base) + kP4TableBytes;
    uint32_t *xs = reinterpret_cast<uint32_t *>(after);
    float *red = reinterpret_cast<float *>(after + size_t(gpr) * 128);
    if constexpr (kP4) {
        for (int i = threadIdx.x; i < 256 * 8; i += blockDim.x) {
            const uint32_t b = uint32_t(i) >> 3;
            const uint32_t e = (uint32_t(v.palette[b >> 4]) << 23) | (uint32_t(v.palette[b & 15u]) << 7);
            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" :: "r"(tab + 16u * uint32_t(i)), "r"(e)
                         : "memory");
        }
    }
    grid_dep_wait();  // x may come from the kernel before
    load_x_all(p, xs, gpr);
    __syncthreads();
    const uint32_t lbase = tab + 4u * uint32_t(lane);  // bits 7..14 clear

#pragma unroll 1
    for (uint32_t rl = 0; rl < nrbc; rl++) {
        const uint32_t rb = rb0 + rl;
        const uint32_t R = rb < v.nfull ? uint32_t(kTileRows) : v.tail_rows;
        const bool ok = uint32_t(lane) < R;
        const uint32_t lc = ok ? uint32_t(lane) : 0u;
        const uint64_t qrb = uint64_t(kTileRows) * rb * gpr;  // first group of the row block
        float s_w = 0.f;
        constexpr int NI = kP4 ? 2 : 4;  // 16-byte chunks of the intermediate form per row
        uint4 ic[NI], sc[4], in_[NI], sn[4];
        uint32_t gc = 0, gn = 0;
        auto fetch = [&](uint32_t kg, uint4 (&ix)[NI], uint4 (&sx)[4], uint32_t &g) {
            const uint64_t q0 = qrb + uint64_t(R) * kg;
            const uint8_t *ip = p.p4 + 16 * NI * q0 + 16 * lc;
            const uint8_t *sp = v.sm + 64 * q0 + 16 * lc;
#pragma unroll
            for (int c = 0; c < NI; c++)
                ix[c] = __ldg(reinterpret_cast<const uint4 *>(ip + c * 16 * R));
#pragma unroll
            for (int c = 0; c < 4; c++)
                sx[c] = __ldg(reinterpret_cast<const uint4 *>(sp + c * 16 * R));
            if constexpr (kP4)
                g = __ldg(v.glen + q0 + lc);
        };
        if (k0 < k1)
            fetch(k0, in_, sn, gn);
#pragma unroll 1
        for (uint32_t kg = k0; kg < k1; kg++) {
#pragma unroll
            for (int c = 0; c < NI; c++)
                ic[c] = in_[c];
#pragma unroll
            for (int c = 0; c < 4; c++)
                sc[c] = sn[c];
            gc = gn;
            if (kg + 1 < k1)
                fetch(kg + 1, in_, sn, gn);
            const uint32_t xaddr = smem_addr(xs) + kg * 128u;
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int I = 0; I < 32; I++) {
                if constexpr (kP4) {
                    const uint32_t iw = word4(ic[I >> 4], (I >> 2) & 3);
                    const int sh = 8 * (I & 3) - 7;  // byte I&3 of the word, times 128
                    const uint32_t moved = sh < 0 ? iw << -sh : iw >> sh;
                    uint32_t off;
                    asm("lop3.b32 %0, %1, 0x7F80, %2, 0xEA;" : "=r"(off) : "r"(moved), "r"(lbase));  // (a & b) | c
                    const uint32_t y = prmt(sm_word(sc, I >> 1), 0u, (I & 1) ? 0xB3A2u : 0x9180u);
                    fma_bf16x2(a0, a1, lop3_merge(y, lds32(off)), lds32(xaddr + 4u * I));
                } else {
                    fma_bf16x2(a0, a1, escape_pair(ic, I, sm_word(sc, I >> 1)), lds32(xaddr + 4u * I));
                }
            }
            // palette-4, escaped groups: exponents from the escape section
            const uint32_t em = kP4 ? __ballot_sync(0xffffffffu, ok && gc == 0u) : 0u;
            if ((em >> lane) & 1u) {
                const uint32_t rank = __popc(em & ((1u << lane) - 1u));
                const uint32_t t = rb * gpr + kg;
                const uint4 *ep = reinterpret_cast<const uint4 *>(v.esc + 64 * uint64_t(__ldg(v.tesc + t) + rank));
                uint4 e[4];
#pragma unroll
                for (int c = 0; c < 4; c++)
                    e[c] = __ldg(ep + c);
                a0 = 0.f;
                a1 = 0.f;
#pragma unroll
                for (int I = 0; I < 32; I++)
                    fma_bf16x2(a0, a1, escape_pair(e, I, sm_word(sc, I >> 1)), lds32(xaddr + 4u * I));
            }
            s_w = s_w + (a0 + a1);
        }
        red[(rl * W + warp) * 32 + lane] = s_w;
    }
    __syncthreads();
    cta_reduce<W>(p, red, rb0, nrbc);
}

template <int W, int kSrc, bool kPrivate>
__global__ void __launch_bounds__(W * 32, 1) gemv_kg_kernel(const GemvParams p, int rb_per_cta) {
    grid_dep_launch();
    if constexpr (kSrc == kSrcHuffman && kPrivate)
        gemv_private<W>(p, rb_per_cta);
    else if constexpr (kSrc == kSrcHuffman)
        gemv_col_compressed<W, false>(p, rb_per_cta);
    else if constexpr (kSrc == kSrcPalette4 || kSrc == kSrcExponent)
        gemv_col_formed<W, kSrc>(p, rb_per_cta);
    else
        gemv_col_bf16<W>(p, rb_per_cta);
}

size_t kg_smem(int warps, int rb_per_cta, int src, bool priv, uint32_t tdata, int gpr) {
    const size_t red = size_t(rb_per_cta) * warps * 128;
    if (src == kSrcBf16)
        return size_t(gpr) * 128 + red;
    if (src == kSrcPalette4 || src == kSrcExponent)  // worst-case pad to 32 KB, the table, x, partials
        return 32768 + size_t(kP4TableBytes) + size_t(gpr) * 128 + red;
    if (priv)
        return size_t(kPrivateLutBytes) + size_t(kCommonSmemBytes) + kCountWords * 4 + red + 128 +
               size_t(warps) * (kPairStages * code_stage_bytes(tdata) + size_t(kRecRing) * kRecBytes +
                                kEscSlots * kEscSlotBytes);
    return size_t(kCommonSmemBytes) + red + 128 +
           size_t(warps) * (kPairStages * pair_stage_bytes(tdata) + size_t(kRecRing) * kRecBytes);
}

template <int W, int kSrc, bool kPrivate>
uw_status launch_kg_one(const GemvParams &p, int rb_per_cta, cudaStream_t stream) {
    const size_t smem = kg_smem(W, rb_per_cta, kSrc, kPrivate, p.v.tdata, int(p.cols / kGroup));
    if (smem > size_t(kMaxSmemPerBlock) - 1024)
        return UW_ERR_UNSUPPORTED;
    auto kern = gemv_kg_kernel<W, kSrc, kPrivate>;
    if (!ensure_smem(kern, smem))
        return UW_ERR_CUDA;
    const int64_t nrb = (p.rows + kTileRows - 1) / kTileRows;
    const dim3 grid(unsigned((nrb + rb_per_cta - 1) / rb_per_cta));
    return launch_overlapped(kern, grid, dim3(W * 32), smem, stream, p, rb_per_cta) == cudaSuccess ? UW_OK
                                                                                             : UW_ERR_CUDA;
}

// Huffman source: the private-table form when its shared memory fits, else
// one shared table.  Both decode the same weights, so the results are
// identical.
template <int W, int kS>
uw_status launch_twin_tma(const GemvParams &p, const CUtensorMap &m, int rb_per_cta, size_t smem, cudaStream_t stream) {
    auto kern = gemv_kg_twin_tma_kernel<W, kS>;
    if (!ensure_smem(kern, smem))
        return UW_ERR_CUDA;
    const int64_t nrb = (p.rows + kTileRows - 1) / kTileRows;
    const dim3 grid(unsigned((nrb + rb_per_cta - 1) / rb_per_cta));
    return launch_overlapped(kern, grid, dim3(W * 32), smem, stream, p, m, rb_per_cta) == cudaSuccess ? UW_OK
                                                                                                  : UW_ERR_CUDA;
}

// The uncompressed twin: tiles by tensor-map copies when W can be described
// by a tensor map and three (else two) stages per warp fit; otherwise the
// per-lane loads of gemv_col_bf16.  All give the same bits.
template <int W>
uw_status launch_twin(const GemvParams &p, int rb_per_cta, cudaStream_t stream) {
    const int gpr = int(p.cols / kGroup);
    CUtensorMap m;
    if (encode_w_tile_map(&m, p.w, p.rows, p.cols)) {
        if (twin_tma_smem(W, rb_per_cta, gpr, 3) <= size_t(kMaxSmemPerBlock) - 1024)
            return launch_twin_tma<W, 3>(p, m, rb_per_cta, twin_tma_smem(W, rb_per_cta, gpr, 3), stream);
        if (twin_tma_smem(W, rb_per_cta, gpr, 2) <= size_t(kMaxSmemPerBlock) - 1024)
            return launch_twin_tma<W, 2>(p, m, rb_per_cta, twin_tma_smem(W, rb_per_cta, gpr, 2), stream);
    }
    return launch_kg_one<W, kSrcBf16, false>(p, rb_per_cta, stream);
}

template <int W>
uw_status launch_kg_src(const GemvParams &p, int rb_per_cta, int src, cudaStream_t stream) {
    if (src == kSrcBf16)
        return launch_twin<W>(p, rb_per_cta, stream);
    if (src == kSrcPalette4)
        return launch_kg_one<W, kSrcPalette4, false>(p, rb_per_cta, stream);
    if (src == kSrcExponent)
        return launch_kg_one<W, kSrcExponent, false>(p, rb_per_cta, stream);
    if (kg_smem(W, rb_per_cta, kSrcHuffman, true, p.v.tdata, int(p.cols / kGroup)) <= size_t(kMaxSmemPerBlock) - 1024)
        return launch_kg_one<W, kSrcHuffman, true>(p, rb_per_cta, stream);
    return launch_kg_one<W, kSrcHuffman, false>(p, rb_per_cta, stream);
}

}  // namespace

size_t gemv_kg_smem_bytes(int warps, int rb_per_cta, bool compressed, uint32_t tdata, int gpr) {
    return kg_smem(warps, rb_per_cta, compressed ? kSrcHuffman : kSrcBf16, false, tdata, gpr);
}

uw_status launch_gemv_kg(const GemvParams &p, int warps, int rb_per_cta, int src, cudaStream_t stream) {
    if (p.batch != 1 || rb_per_cta < 1)
        return UW_ERR_UNSUPPORTED;
    if (uint64_t(p.rows / kTileRows + 1) * (p.cols / kGroup) >= (uint64_t(1) << 32))
        return UW_ERR_UNSUPPORTED;  // tile indices are 32-bit
    switch (warps) {
        case 4: return launch_kg_src<4>(p, rb_per_cta, src, stream);
        case 8: return launch_kg_src<8>(p, rb_per_cta, src, stream);
        case 16: return launch_kg_src<16>(p, rb_per_cta, src, stream);
    }
    return UW_ERR_UNSUPPORTED;
}

}  // namespace uw
