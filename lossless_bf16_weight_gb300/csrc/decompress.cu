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
#include "pair_stage.cuh"
#include "tc.cuh"

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
            const int64_t col = int64_t(cur.kg) * kGroup + c * 8;
            if (r < R && col < v.ocols) {
                const uint4 val = obuf[r * 8 + (c ^ (r & 7))];
                uint16_t *dst = out + (int64_t(cur.rb) * kTileRows + r) * v.ocols + col;
                if ((v.ocols & 7) == 0) {
                    *reinterpret_cast<uint4 *>(dst) = val;
                } else {  // ragged rows not 16-byte aligned: the true columns one by one
                    const uint16_t *h = reinterpret_cast<const uint16_t *>(&val);
                    const int n = v.ocols - col < 8 ? int(v.ocols - col) : 8;
                    for (int k = 0; k < n; k++)
                        dst[k] = h[k];
                }
            }
        }
        __syncwarp();
        cur = nxt;
        nxt = n2;
    }
}

// ---------------------------------------------------------------------------
// The batch-1 GEMV's pipeline applied to the decompress: one CTA of
// kPrivWarps per SM owning whole row blocks, warp w the groups [k0(w),
// k1(w)) of each, two tiles (a pair) decoded side by side from bulk-copied
// code stages issued two pairs ahead, escaped groups in the main loop through
// the counting stream (pair_stage.cuh), the sign+mantissa bytes read from L2
// after a bulk prefetch.  The pair table is one shared copy (4 KB): the
// shared memory goes to an 8 KB output buffer per warp instead, into which
// lane j writes row j of both tiles (128-byte swizzle, conflict-free), sent
// to the output by two tensor-map stores per pair (whole 128-byte lines).
constexpr int kPrivWarps = 16;
constexpr uint32_t kOutPairBytes = 2 * kTileRows * kGroup * 2;  // 8 KB

__device__ __forceinline__ void priv_warp_cols(uint32_t gpr, int w, int W, uint32_t &k0, uint32_t &k1) {
    k0 = uint32_t(uint64_t(gpr) * uint32_t(w) / uint32_t(W));
    k1 = uint32_t(uint64_t(gpr) * uint32_t(w + 1) / uint32_t(W));
}

__device__ __forceinline__ void sts128(uint32_t a, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" :: "r"(a), "r"(x), "r"(y), "r"(z), "r"(w) : "memory");
}

template <bool kFull>
__device__ __forceinline__ void dec_pair(const BlobView &v, uint32_t *status, uint32_t obuf, uint32_t lut,
                                         uint32_t zero, uint32_t cnt, uint32_t slots, uint32_t below, uint32_t one,
                                         uint32_t st, uint32_t pkA, uint32_t pkB, uint64_t q0, uint32_t Rr,
                                         uint32_t rb, uint32_t kgA, bool hasB, const uint8_t *sm, bool more,
                                         const uint8_t *sm_nxt, uint32_t Rn, bool nhasB, uint4 &c0A, uint4 &c0B,
                                         uint32_t &bad) {
    const int lane = threadIdx.x & 31;
    const uint32_t R = kFull ? uint32_t(kTileRows) : Rr;
    const uint32_t n16A = pkA & 0xFFu, n16B = pkB & 0xFFu;
    const uint32_t nescA = (pkA >> 8) & 0xFFu, nescB = (pkB >> 8) & 0xFFu;
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
    uint32_t ga = vA ? gA : 0u, gb = vB ? gB : 0u;
    const uint32_t g2 = ga | (gb << 16);
    uint32_t incl = g2;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1)
        asm("{\n\t.reg .b32 u;\n\t.reg .pred q;\n\t"
            "shfl.sync.up.b32 u|q, %0, %1, 0, -1;\n\t"
            "@q add.u32 %0, %0, u;\n\t}"
            : "+r"(incl) : "r"(d));
    const uint32_t off2 = incl - g2;
    const uint32_t tot2 = __shfl_sync(0xffffffffu, incl, 31);
    uint32_t emA = __ballot_sync(0xffffffffu, vA && ga == 0u);
    uint32_t emB = __ballot_sync(0xffffffffu, vB && gb == 0u);
    if (((pkA | pkB) >> 16) != 0u || (tot2 & 0xFFFFu) > 16u * n16A || (tot2 >> 16) > 16u * n16B ||
        uint32_t(__popc(emA)) != nescA || uint32_t(__popc(emB)) != nescB) {
        if (lane == 0)
            atomicOr(status, uint32_t(kStatusBadTile));
        ga = 0u;
        gb = 0u;
        emA = 0u;
        emB = 0u;
    }
    const uint32_t cA = st + 64u, cB = cA + 16u * n16A;
    const uint32_t ebA = cB + 16u * n16B, ebB = ebA + 64u * nescA;
    uint32_t wzA = zero, wzB = zero, lutA = lut, lutB = lut, sA_ = kStrideShared, sB_ = kStrideShared;
    bool xa = false, xb = false;
    if ((emA | emB) != 0u) {
        const uint32_t pa = __popc(emA), pb = __popc(emB);
        const uint32_t nA = pa < uint32_t(kEscSlots) ? pa : uint32_t(kEscSlots);
        const uint32_t nB = pb < uint32_t(kEscSlots) - nA ? pb : uint32_t(kEscSlots) - nA;
        expand_escapes(nA, ebA, slots, 0u);
        expand_escapes(nB, ebB, slots, nA);
        __syncwarp();
        const uint32_t rA = __popc(emA & below), rB = nA + __popc(emB & below);
        xa = (emA >> lane) & 1u;
        xb = (emB >> lane) & 1u;
        if (xa && rA < nA) {
            wzA = cnt;
            lutA = slots + kEscSlotBytes * rA;
            sA_ = 4u;
            xa = false;
        }
        if (xb && rB < nA + nB) {
            wzB = cnt;
            lutB = slots + kEscSlotBytes * rB;
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
    // row `lane` of tile A at obuf + 128 lane, of tile B 4 KB further; chunk c
    // at position c ^ (lane % 8)
    const uint32_t rowA = obuf + 128u * uint32_t(lane), rowB = rowA + kTileRows * kGroup * 2u;
    const uint32_t sw = uint32_t(lane) & 7u;
    uint4 sA = c0A, sB = c0B, nA = sA, nB = sB;
    uint32_t qA[4], qB[4];
#pragma unroll
    for (int I = 0; I < 32; I++) {
        if ((I & 7) == 0) {  // next chunk of sign+mantissa bytes
            if (I < 24) {
                nA = __ldg(reinterpret_cast<const uint4 *>(gA_sm + uint32_t((I >> 3) + 1) * stride));
                nB = __ldg(reinterpret_cast<const uint4 *>(gB_sm + uint32_t((I >> 3) + 1) * stride));
            } else if (more) {  // chunk 0 of the next pair
                const uint8_t *a = sm_nxt + 16u * (uint32_t(lane) < Rn ? uint32_t(lane) : 0u);
                nA = __ldg(reinterpret_cast<const uint4 *>(a));
                nB = __ldg(reinterpret_cast<const uint4 *>(nhasB ? a + 64u * Rn : a));
            }
        }
        const uint32_t eA = decode_entry_rs(la, lutA, sA_, one, I);
        const uint32_t eB = decode_entry_rs(lb, lutB, sB_, one, I);
        const uint32_t sel = (I & 1) ? 0xB3A2u : 0x9180u;
        qA[I & 3] = lop3_merge(prmt(word4(sA, (I >> 1) & 3), 0u, sel), eA);
        qB[I & 3] = lop3_merge(prmt(word4(sB, (I >> 1) & 3), 0u, sel), eB);
        if ((I & 3) == 3) {
            const uint32_t c = ((uint32_t(I) >> 2) ^ sw) << 4;
            sts128(rowA + c, qA[0], qA[1], qA[2], qA[3]);
            sts128(rowB + c, qB[0], qB[1], qB[2], qB[3]);
        }
        if ((I & 7) == 7) {
            sA = nA;
            sB = nB;
        }
    }
    bad |= tile_check_bits(la) | tile_check_bits(lb);
    if (xa | xb) {  // escaped groups beyond the slots: second pass from their raw exponents
        uint4 e[4], smv[4];
        for (int pass = 0; pass < 2; pass++) {  // tile A, then tile B
            const bool mine = pass == 0 ? xa : xb;
            if (!mine)
                continue;
            escape_read(pass == 0 ? ebA : ebB, pass == 0 ? emA : emB, e);
            const uint8_t *g = pass == 0 ? gA_sm : gB_sm;
#pragma unroll
            for (int c = 0; c < 4; c++)
                smv[c] = __ldg(reinterpret_cast<const uint4 *>(g + c * stride));
            const uint32_t row = pass == 0 ? rowA : rowB;
#pragma unroll
            for (int I = 0; I < 32; I += 4) {
                uint32_t q2[4];
#pragma unroll
                for (int k = 0; k < 4; k++)
                    q2[k] = escape_pair(e, I + k, sm_word(smv, (I + k) >> 1));
                sts128(row + ((uint32_t(I >> 2) ^ sw) << 4), q2[0], q2[1], q2[2], q2[3]);
            }
        }
    }
    c0A = sA;
    c0B = sB;
}

__global__ void __launch_bounds__(kPrivWarps * 32, 1)
    decompress_priv_kernel(const __grid_constant__ BlobView v, const __grid_constant__ CUtensorMap omap,
                           uint32_t *status, int rb_per_cta) {
    constexpr int W = kPrivWarps;
    extern __shared__ __align__(1024) unsigned char smem[];
    __shared__ __align__(8) uint64_t bars[W * kPairStages];
    grid_dep_launch();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t gpr = v.gpr;
    const uint32_t nrb = v.nfull + (v.tail_rows ? 1u : 0u);
    const uint32_t rb0 = blockIdx.x * uint32_t(rb_per_cta);
    const uint32_t rb1 = rb0 + uint32_t(rb_per_cta) < nrb ? rb0 + uint32_t(rb_per_cta) : nrb;
    const uint32_t nrbc = rb1 > rb0 ? rb1 - rb0 : 0u;
    uint32_t k0, k1;
    priv_warp_cols(gpr, warp, W, k0, k1);
    const uint32_t np = (k1 - k0 + 1) / 2;
    const uint32_t npairs = np * nrbc;
    const uint32_t sbytes = code_stage_bytes(v.tdata);
    // shared memory: [pad to 1024][per warp an 8 KB output buffer][common
    // tables][counting stream][pad to 128][per warp kPairStages stages][per
    // warp kRecRing records][per warp kEscSlots escape slots]
    const uint32_t base = (smem_addr(smem) + 1023u) & ~1023u;
    const uint32_t obuf = base + uint32_t(warp) * kOutPairBytes;
    unsigned char *common = smem + (base - smem_addr(smem)) + W * kOutPairBytes;
    const DecodeShared ds = carve_common(common);
    const uint32_t cnt = smem_addr(common) + uint32_t(kCommonSmemBytes);
    const uint32_t stage_lo = (cnt + kCountWords * 4u + 127u) & ~127u;
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
    uint32_t nissued = 0;
    const RecLoad first = pair_recs_load(v, span, 0);
    build_tables(ds, v);
    pair_recs_store(v, ring, span, 0, first);
#pragma unroll
    for (int s = 0; s < kPairStages; s++) {
        if (nissued < npairs) {
            pair_issue_rec<false>(v, ring + kRecBytes * nissued, st0 + uint32_t(s) * sbytes, 0u, bar0 + 8u * s);
            nissued++;
        }
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
    grid_dep_wait();  // the output may still be read by the kernel before
    const uint32_t lut = smem_addr(ds.lut);
    const uint32_t zero = smem_addr(ds.zero);
    const uint32_t one = gpr != 0u ? 1u : 0u;
    const uint32_t below = (1u << lane) - 1u;
    PairCursor cur{rb0, k0};
    uint32_t bad = 0;
#pragma unroll 1
    for (uint32_t j = 0; j < npairs; j++) {
        const uint32_t st = st0 + (j & 1u) * sbytes, bar = bar0 + 8u * (j & 1u);
        mbar_wait(bar, (j >> 1) & 1u, status, kStatusTimeout);
        const uint4 rbk = lds128(ring + kRecBytes * (j % uint32_t(kRecRing)) + 16u);
        const bool hasB = cur.kgA + 1 < k1;
        const bool full = cur.rb < v.nfull;
        const bool more = j + 1 < npairs;
        PairCursor nxt = cur;
        nxt.next(k0, k1);
        const uint32_t Rn = nxt.rb < v.nfull ? uint32_t(kTileRows) : v.tail_rows;
        const uint8_t *sm_nxt = more ? rec_sm(v, ring + kRecBytes * ((j + 1) % uint32_t(kRecRing))) : sm_cur;
        const uint64_t q0 = (uint64_t(rbk.w) << 32) | rbk.z;
        // the output buffer is free once the previous pair's stores have read it
        if (lane == 0)
            tma_store_wait_read();
        __syncwarp();
        if (full)
            dec_pair<true>(v, status, obuf, lut, zero, cnt, slots, below, one, st, rbk.x, rbk.y, q0, kTileRows, cur.rb,
                           cur.kgA, hasB, sm_cur, more, sm_nxt, Rn, nxt.kgA + 1 < k1, c0A, c0B, bad);
        else
            dec_pair<false>(v, status, obuf, lut, zero, cnt, slots, below, one, st, rbk.x, rbk.y, q0, v.tail_rows,
                            cur.rb, cur.kgA, hasB, sm_cur, more, sm_nxt, Rn, nxt.kgA + 1 < k1, c0A, c0B, bad);
        // the pair's rows to the output (rows past the matrix are not written),
        // and the code stage back to the copy engine
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(&omap, int(cur.kgA * kGroup), int(cur.rb * kTileRows), obuf);
            if (hasB)
                tma_store_2d(&omap, int((cur.kgA + 1) * kGroup), int(cur.rb * kTileRows),
                             obuf + kTileRows * kGroup * 2u);
            tma_store_commit();
        }
        sm_cur = sm_nxt;
        cur = nxt;
        if (nissued < npairs) {
            pair_issue_rec<false>(v, ring + kRecBytes * (nissued % uint32_t(kRecRing)), st, 0u, bar);
            if (nissued % uint32_t(kRecRound) == 2u && nissued - 2u + uint32_t(kRecRound) < npairs)
                pair_recs_store(v, ring, span, nissued - 2u + uint32_t(kRecRound),
                                pair_recs_load(v, span, nissued - 2u + uint32_t(kRecRound)));
            nissued++;
        }
        __syncwarp();
    }
    if (lane == 0)
        tma_store_wait_all();
    tile_check_flush(bad, status);
}

size_t priv_smem(uint32_t tdata) {
    return 1024 + size_t(kPrivWarps) * kOutPairBytes + size_t(kCommonSmemBytes) + kCountWords * 4 + 128 +
           size_t(kPrivWarps) * (kPairStages * code_stage_bytes(tdata) + size_t(kRecRing) * kRecBytes +
                                 kEscSlots * kEscSlotBytes);
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
    // lane-private tables when they fit: one CTA per SM (or per allowed SM)
    // with whole row blocks.  The output map has the matrix's own width, so
    // the tensor-map stores drop the filler columns of ragged rows; a row
    // pitch that is not a multiple of 16 bytes (no tensor map) goes to the
    // tile kernel, which stores the true columns one by one.
    const size_t psmem = priv_smem(v.tdata);
    CUtensorMap omap;
    if (psmem <= size_t(kMaxSmemPerBlock) - 1024 && v.gpr >= 1 && (v.ocols & 7) == 0 &&
        encode_w_tile_map(&omap, w_out, v.rows, v.ocols)) {
        const int64_t nrb = int64_t(v.nfull) + (v.tail_rows ? 1 : 0);
        int64_t ctas = sm_count();
        if (max_ctas > 0 && max_ctas < ctas)
            ctas = max_ctas;
        const int64_t rbc = (nrb + ctas - 1) / ctas;
        const int64_t grid = (nrb + rbc - 1) / rbc;
        if (!ensure_smem(decompress_priv_kernel, psmem))
            return UW_ERR_CUDA;
        return launch_overlapped(decompress_priv_kernel, dim3(unsigned(grid)), dim3(kPrivWarps * 32), psmem, stream, v,
                                 omap, status, int(rbc)) == cudaSuccess
                   ? UW_OK
                   : UW_ERR_CUDA;
    }
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
