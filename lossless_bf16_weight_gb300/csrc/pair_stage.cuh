// Staging of tile pairs by the copy engine, shared by the batch-1 GEMV and
// the tensor-core matmul.
//
// A "pair" is the tiles (rb, kg) and (rb, kg+1): they sit next to each other
// in every section of the blob, so one bulk copy per section brings both --
// their glen, their code regions followed by their escaped groups' raw
// exponents, and their sign+mantissa bytes -- into one shared-memory stage,
// completing on an mbarrier.  A warp keeps kPairStages stages and works one
// pair ahead.
#pragma once
#include <cstdint>

#include "decode.cuh"
#include "tc.cuh"

namespace uw {

constexpr int kPairStages = 2;

__device__ __forceinline__ uint32_t lds_u8(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

// Bytes of one pair stage, and the offset of its sign+mantissa bytes.
__host__ __device__ constexpr uint32_t pair_stage_bytes(uint32_t tdata) {
    return (64u + 2u * tdata + 64u + 4096u + 127u) & ~127u;
}
__host__ __device__ constexpr uint32_t pair_stage_smoff(uint32_t tdata) { return 64u + 2u * tdata + 64u; }

// Offsets of the pair at tile t (lanes 0..2: tcode[t..t+2], lanes 3..5:
// tesc[t..t+2]; indices past the table end read its last entry).
__device__ __forceinline__ uint32_t pair_offsets_load(const BlobView &v, uint32_t t) {
    const int lane = threadIdx.x & 31;
    const int l = lane < 6 ? lane : 0;
    const uint32_t k = t + uint32_t(l % 3);
    return __ldg((l < 3 ? v.tcode : v.tesc) + (k < v.ntiles ? k : v.ntiles));
}

// The same for two pairs in one round trip: t0 into lanes 0..5, t1 into
// lanes 8..13 (read the second with pair_offsets_shift).
__device__ __forceinline__ uint32_t pair_offsets_load2(const BlobView &v, uint32_t t0, uint32_t t1) {
    const int lane = threadIdx.x & 31;
    const int l = (lane & 7) < 6 ? (lane & 7) : 0;
    const uint32_t k = (lane < 8 ? t0 : t1) + uint32_t(l % 3);
    return __ldg((l < 3 ? v.tcode : v.tesc) + (k < v.ntiles ? k : v.ntiles));
}

// Move lanes 8..13 of a pair_offsets_load2 result down to lanes 0..5.
__device__ __forceinline__ uint32_t pair_offsets_shift(uint32_t o) { return __shfl_down_sync(0xffffffffu, o, 8); }

// What the decode needs to know about a staged pair (warp-uniform; kept in
// shared memory next to the stage so that the loop body is not duplicated).
struct PairMeta {
    uint32_t pkA, pkB;   // n16 | nesc << 8 | bad << 16 of each tile
    uint32_t n16A, n16B, nescA;
    uint32_t R;          // rows of the pair's tiles | 0x100 when tile B is present (0: no pair)
    uint32_t sm_lo, sm_hi;  // address of the pair's sign+mantissa bytes (tile A's; B's follow 64 * R later)
};

// Code stage of a pair without its sign+mantissa bytes:
//   [0, 64)                      glen of A and B (full row blocks only)
//   [64, 64 + 2*tdata)           code regions of A then B, then escaped exponents of A then B
//   then 64 bytes of read slack
__host__ __device__ constexpr uint32_t code_stage_bytes(uint32_t tdata) {
    return (64u + 2u * tdata + 64u + 127u) & ~127u;
}

// First byte of the pair's sign+mantissa bytes (tile A's; tile B's follow
// 64 * R bytes later) and R.
__device__ __forceinline__ const uint8_t *pair_sm_base(const BlobView &v, uint32_t rb, uint32_t kgA, uint32_t t,
                                                       uint32_t &R) {
    const bool full = rb < v.nfull;
    R = full ? uint32_t(kTileRows) : v.tail_rows;
    const uint64_t q0 = uint64_t(t) * kTileRows - (full ? 0u : (kTileRows - R) * kgA);
    return v.sm + q0 * kGroup;
}

// Validate the pair's offsets `o` (pair_offsets_load) and start its bulk
// copies into stage `st`:
//   [0, 64)                      glen of A and B (full row blocks only)
//   [64, 64 + 2*tdata)           code regions of A then B, then escaped exponents of A then B
// plus an L2 prefetch of the pair's sign+mantissa bytes, which the caller
// reads from global memory.  A pair with bad offsets copies no codes and is
// decoded as zeros (the error is recorded when it is decoded).
__device__ __forceinline__ void pair_issue_codes(const BlobView &v, uint32_t o, uint32_t rb, uint32_t kgA, bool hasB,
                                                 uint32_t t, uint32_t st, uint32_t bar, PairMeta *meta) {
    const int lane = threadIdx.x & 31;
    const uint32_t c0 = __shfl_sync(0xffffffffu, o, 0), c1 = __shfl_sync(0xffffffffu, o, 1);
    const uint32_t c2r = __shfl_sync(0xffffffffu, o, 2), e0 = __shfl_sync(0xffffffffu, o, 3);
    const uint32_t e1 = __shfl_sync(0xffffffffu, o, 4), e2r = __shfl_sync(0xffffffffu, o, 5);
    const uint32_t c2 = hasB ? c2r : c1, e2 = hasB ? e2r : e1;
    uint32_t R;
    const uint8_t *sm = pair_sm_base(v, rb, kgA, t, R);
    const bool full = rb < v.nfull;
    const uint32_t n16A = c1 - c0, n16B = c2 - c1, nescA = e1 - e0, nescB = e2 - e1;
    const uint32_t lim16 = uint32_t(kMaxTileCodeBytes / 16);
    const bool bad = n16A > lim16 || n16B > lim16 || nescA > R || nescB > R || n16A * 16u + nescA * 64u > v.tdata ||
                     n16B * 16u + nescB * 64u > v.tdata || c2 > v.code16 || e2 > v.n_esc32;
    const uint32_t ntile = hasB ? 2u : 1u;
    const uint64_t q0 = uint64_t(sm - v.sm) / kGroup;
    const uint32_t code_bytes = bad ? 0u : (c2 - c0) * 16u;
    const uint32_t esc_bytes = bad ? 0u : (e2 - e0) * 64u;
    const uint32_t glen_bytes = full ? uint32_t(kTileRows) * ntile : 0u;
    if (lane == 0) {
        meta->pkA = bad ? (1u << 16) : (n16A | (nescA << 8));
        meta->pkB = !hasB ? 0u : bad ? (1u << 16) : (n16B | (nescB << 8));
        meta->n16A = bad ? 0u : n16A;
        meta->n16B = bad ? 0u : n16B;
        meta->nescA = bad ? 0u : nescA;
        meta->R = R | (hasB ? 0x100u : 0u);
        meta->sm_lo = uint32_t(reinterpret_cast<uint64_t>(sm));
        meta->sm_hi = uint32_t(reinterpret_cast<uint64_t>(sm) >> 32);
        mbar_expect_tx(bar, code_bytes + esc_bytes + glen_bytes);
        if (glen_bytes)
            bulk_g2s(st, v.glen + q0, glen_bytes, bar);
        if (code_bytes)
            bulk_g2s(st + 64u, v.code + size_t(c0) * 16, code_bytes, bar);
        if (esc_bytes)
            bulk_g2s(st + 64u + code_bytes, v.esc + size_t(e0) * 64, esc_bytes, bar);
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(sm), "r"(uint32_t(kGroup) * R * ntile)
                     : "memory");
    }
}

// What issuing a pair and decoding it need from the tile tables, worked out
// for kRecRound pairs at a time (lane i: the round's pair i, all offsets in
// one round trip) and kept in a ring of kRecRing records per warp, so that
// issuing a pair is two shared-memory loads and the copies.
constexpr int kRecRound = 8;
constexpr int kRecRing = 2 * kRecRound;
constexpr uint32_t kRecBytes = 32;

// Record layout (8 words):
//   0 c0      first 16-byte unit of tile A's codes
//   1 bytes   code bytes | escape bytes << 16 (both 0 for a bad pair)
//   2 e0      first escaped group of tile A
//   3 sizes   n16A | n16B << 8 | nescA << 16 | (glen bytes / 32) << 22 | (R * tiles) << 24
//   4 pkA     n16 | nesc << 8 | bad << 16 of tile A (as TileMeta.pk)
//   5 pkB     the same for tile B (0 without B)
//   6, 7      q0, the pair's first group (64-bit)
// Lanes 0..kRecRound-1 fill the records of pairs base .. base+kRecRound-1
// (pair j: row block rb0 + j / ppr, group kA = k0 + 2 (j % ppr), B present
// when kA + 1 < k1): pair_recs_load issues the table loads, pair_recs_store
// (after other work, if any) writes the records.
struct PairRecSpan {
    uint32_t npairs, rb0, k0, k1, ppr;
};
struct RecLoad {
    uint32_t c0, c1, c2, e0, e1, e2;
};

__device__ __forceinline__ void rec_pair(const PairRecSpan &sp, uint32_t j, uint32_t gpr, uint32_t &rb, uint32_t &kgA,
                                         bool &hasB) {
    rb = sp.rb0 + j / sp.ppr;
    kgA = sp.k0 + 2u * (j % sp.ppr);
    hasB = kgA + 1 < sp.k1;
}

__device__ __forceinline__ RecLoad pair_recs_load(const BlobView &v, const PairRecSpan &sp, uint32_t base) {
    const uint32_t lane = threadIdx.x & 31, j = base + lane;
    RecLoad r{};
    if (lane < uint32_t(kRecRound) && j < sp.npairs) {
        uint32_t rb, kgA;
        bool hasB;
        rec_pair(sp, j, v.gpr, rb, kgA, hasB);
        const uint32_t t = rb * v.gpr + kgA;
        auto at = [&](const uint32_t *tab, uint32_t k) { return __ldg(tab + (k < v.ntiles ? k : v.ntiles)); };
        r.c0 = at(v.tcode, t);
        r.c1 = at(v.tcode, t + 1);
        r.c2 = at(v.tcode, t + (hasB ? 2u : 1u));
        r.e0 = at(v.tesc, t);
        r.e1 = at(v.tesc, t + 1);
        r.e2 = at(v.tesc, t + (hasB ? 2u : 1u));
    }
    return r;
}

__device__ __forceinline__ void pair_recs_store(const BlobView &v, uint32_t ring, const PairRecSpan &sp, uint32_t base,
                                                const RecLoad &r) {
    const uint32_t lane = threadIdx.x & 31, j = base + lane;
    if (lane < uint32_t(kRecRound) && j < sp.npairs) {
        uint32_t rb, kgA;
        bool hasB;
        rec_pair(sp, j, v.gpr, rb, kgA, hasB);
        const uint32_t t = rb * v.gpr + kgA;
        const bool full = rb < v.nfull;
        const uint32_t R = full ? uint32_t(kTileRows) : v.tail_rows;
        const uint32_t n16A = r.c1 - r.c0, n16B = r.c2 - r.c1, nescA = r.e1 - r.e0, nescB = r.e2 - r.e1;
        const uint32_t lim16 = uint32_t(kMaxTileCodeBytes / 16);
        const bool bad = n16A > lim16 || n16B > lim16 || nescA > R || nescB > R || n16A * 16u + nescA * 64u > v.tdata ||
                         n16B * 16u + nescB * 64u > v.tdata || r.c2 > v.code16 || r.e2 > v.n_esc32;
        const uint32_t ntile = hasB ? 2u : 1u;
        const uint64_t q0 = uint64_t(t) * kTileRows - (full ? 0u : (kTileRows - R) * kgA);
        const uint32_t bytes = bad ? 0u : ((r.c2 - r.c0) * 16u) | (((r.e2 - r.e0) * 64u) << 16);
        const uint32_t sizes = (bad ? 0u : (n16A | (n16B << 8) | (nescA << 16))) | ((full ? ntile : 0u) << 22) |
                               ((R * ntile) << 24);
        const uint32_t pkA = bad ? (1u << 16) : (n16A | (nescA << 8));
        const uint32_t pkB = !hasB ? 0u : bad ? (1u << 16) : (n16B | (nescB << 8));
        const uint32_t a = ring + kRecBytes * (j % uint32_t(kRecRing));
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" :: "r"(a), "r"(r.c0), "r"(bytes), "r"(r.e0),
                     "r"(sizes) : "memory");
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" :: "r"(a + 16u), "r"(pkA), "r"(pkB),
                     "r"(uint32_t(q0)), "r"(uint32_t(q0 >> 32)) : "memory");
    }
    __syncwarp();
}

// The pair's sign+mantissa bytes (tile A's first; B's follow 64 * R later).
__device__ __forceinline__ const uint8_t *rec_sm(const BlobView &v, uint32_t rec) {
    const uint4 b = lds128(rec + 16u);
    return v.sm + ((uint64_t(b.w) << 32) | b.z) * kGroup;
}

// Start the bulk copies of a pair from its record (one lane issues):
//   [0, 64)                  glen of A and B (full row blocks only)
//   [64, 64 + 2*tdata)       code regions of A then B, then escaped exponents of A then B
//   [smoff, smoff + 128*R)   kStageSm: sign+mantissa bytes of A then B;
//                            otherwise they are only prefetched into L2
template <bool kStageSm>
__device__ __forceinline__ void pair_issue_rec(const BlobView &v, uint32_t rec, uint32_t st, uint32_t smoff,
                                               uint32_t bar) {
    if ((threadIdx.x & 31) == 0) {
        const uint4 a = lds128(rec), b = lds128(rec + 16u);
        const uint32_t code_bytes = a.y & 0xFFFFu, esc_bytes = a.y >> 16;
        const uint32_t glen_bytes = ((a.w >> 22) & 3u) * 32u, sm_bytes = (a.w >> 24) * uint32_t(kGroup);
        const uint64_t q0 = (uint64_t(b.w) << 32) | b.z;
        mbar_expect_tx(bar, code_bytes + esc_bytes + glen_bytes + (kStageSm ? sm_bytes : 0u));
        if (glen_bytes)
            bulk_g2s(st, v.glen + q0, glen_bytes, bar);
        if (code_bytes)
            bulk_g2s(st + 64u, v.code + size_t(a.x) * 16, code_bytes, bar);
        if (esc_bytes)
            bulk_g2s(st + 64u + code_bytes, v.esc + size_t(a.z) * 64, esc_bytes, bar);
        if constexpr (kStageSm)
            bulk_g2s(st + smoff, v.sm + q0 * kGroup, sm_bytes, bar);
        else
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(v.sm + q0 * kGroup), "r"(sm_bytes)
                         : "memory");
    }
}

// The warp's pairs in order: row block by row block, group pairs within
// [k0, k1).
struct PairCursor {
    uint32_t rb, kgA;
    __device__ __forceinline__ void next(uint32_t k0, uint32_t k1) {
        kgA += 2;
        if (kgA >= k1) {
            kgA = k0;
            rb++;
        }
    }
};

// Escaped groups decoded in the main loop of the private-table kernels.  An
// escaped group's raw exponents are expanded once into 32 table-entry words
// (both exponents of a weight pair in BF16 position, bit count 10) in a
// per-warp slot; the lane then runs the same 32 steps as every other lane
// over a constant "counting" stream whose 10-bit windows are 0, 1, ..., 31,
// with the slot as its table and stride 4, so step I reads entry I.  More
// than kEscSlots escaped groups in one pair (rare outside heavy-tailed
// matrices) go to a second pass from their raw exponents.
constexpr int kEscSlots = 4;             // expanded escaped groups per warp and pair
constexpr uint32_t kEscSlotBytes = 128;  // 32 entry words
constexpr int kCountWords = 16;          // counting stream (320 bits) and read slack

// Expand escaped groups into entry words, all 32 lanes at once (lane i
// makes word i = e[2i] << 7 | e[2i+1] << 23 | 10 of each): the first n
// escaped groups whose raw exponents start at shared address `eb` (64 bytes
// each, in lane order) go to slots s0, s0 + 1, ... at `slots`.
__device__ __forceinline__ void expand_escapes(uint32_t n, uint32_t eb, uint32_t slots, uint32_t s0) {
    const uint32_t lane = threadIdx.x & 31;
#pragma unroll 1
    for (uint32_t r = 0; r < n; r++) {
        uint32_t two;
        asm volatile("ld.shared.u16 %0, [%1];" : "=r"(two) : "r"(eb + 64u * r + 2u * lane) : "memory");
        const uint32_t e = prmt(two, 0u, 0x4140u) * 128u + 10u;
        asm volatile("st.shared.u32 [%0], %1;" :: "r"(slots + kEscSlotBytes * (s0 + r) + 4u * lane), "r"(e)
                     : "memory");
    }
}

// The counting stream at shared address `cnt` (kCountWords words; threads
// 0 .. kCountWords - 1 each write one): word k holds stream bits 32k ..
// 32k + 31 of the 10-bit values 0, 1, ..., 31 in order.  Follow with a
// __syncthreads() before use.
__device__ __forceinline__ void build_count_stream(uint32_t cnt) {
    if (threadIdx.x < uint32_t(kCountWords)) {
        const int k = int(threadIdx.x);
        uint32_t wv = 0;
        for (int i = 0; i < 32; i++) {
            const int lo = 10 * i - 32 * k;
            if (lo > -10 && lo < 32)
                wv |= lo >= 0 ? uint32_t(i) << lo : uint32_t(i) >> -lo;
        }
        asm volatile("st.shared.u32 [%0], %1;" :: "r"(cnt + 4u * uint32_t(k)), "r"(wv) : "memory");
    }
}

}  // namespace uw
