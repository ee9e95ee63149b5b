// Device-side tile decoder shared by the decompress and fused matmul kernels.
//
// One warp decodes one tile (32 rows x 64 columns): lane j owns the 64-weight
// group of row j (Unweight blog, paragraph on rows of 64).  Per tile:
//   * the group byte lengths (glen) give each lane its code offset by an
//     exclusive warp prefix sum (shuffles), and each escaped lane its rank
//     among the escaped groups by ballot + popc;
//   * the tile's code bytes are staged in the warp's shared-memory buffer
//     (byte-swapped into big-endian words so that bit 31 of a word is the
//     first code bit);
//   * every step looks up a 12-bit window in a 4096-entry table that decodes
//     two codes at once (codes are at most 6 bits).  An entry holds both
//     exponents already in BF16 position (bits 14..7 and 30..23) and the
//     number of bits the two codes take (bits 3..0);
//   * the exponent pair is merged with two raw sign+mantissa bytes by one
//     byte permute (sign-replicating) and one three-input logic op, giving
//     two BF16 weights in one 32-bit register (the blog's reconstruction:
//     exponent + sign/mantissa bytes -> BF16, paragraph on the consumer
//     warps of the reconstructive matmul).
// Escaped groups and lanes without a row use the same loop: they read a
// fixed stream of 12-bit numbers 0..31 through a private 32-entry table that
// holds their raw exponents (or zeros), so the hot loop has no branch on
// the group kind.
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

#include "format.h"

namespace uw {

enum StatusFlag : uint32_t {
    kStatusBadCode = 1u,    // a group's codes do not add up to its byte length
    kStatusBadTile = 2u,    // tile offsets / sizes out of range
    kStatusBadEscape = 4u,  // escape counts inconsistent
    kStatusTimeout = 8u,    // a bounded wait gave up
};

// Device view of a blob (pointers into the device copy) plus the small
// tables the host derives from the header.
struct BlobView {
    const uint8_t *sm;
    const uint8_t *glen;
    const uint32_t *tcode;
    const uint32_t *tesc;
    const uint8_t *code;
    const uint8_t *esc;
    uint64_t code_bytes;  // size of the code section
    uint64_t n_escaped;
    int64_t rows, cols;
    // 6-bit prefix -> (exponent << 4) | code length; 0 where no code starts
    // with that prefix.
    uint16_t prefix6[64];
};

constexpr int kLutEntries = 4096;
constexpr int kFakeWords = 16;                      // stream of 12-bit values 0..31 (+slack)
constexpr int kWarpBufBytes = 4096 + 64;            // codes + escape tables + read slack
constexpr int kCommonSmemBytes = kLutEntries * 4 + kFakeWords * 4 + 32 * 4 + 64 * 2;

// Shared memory common to every decoding CTA.
struct DecodeShared {
    uint32_t *lut;       // [4096] pair table
    uint32_t *fake;      // [16]   stream 0, 1, ..., 31 in 12-bit fields
    uint32_t *zeros;     // [32]   entries with no exponent, 12 bits each
    uint16_t *prefix6;   // [64]
};

__device__ __forceinline__ DecodeShared carve_common(unsigned char *smem) {
    DecodeShared s;
    s.lut = reinterpret_cast<uint32_t *>(smem);
    s.fake = s.lut + kLutEntries;
    s.zeros = s.fake + kFakeWords;
    s.prefix6 = reinterpret_cast<uint16_t *>(s.zeros + 32);
    return s;
}

// Fill the pair table and the fixed streams.  Must be followed by
// __syncthreads() before use.
__device__ __forceinline__ void build_tables(const DecodeShared &s, const BlobView &v) {
    const int tid = threadIdx.x, nt = blockDim.x;
    for (int i = tid; i < 64; i += nt)
        s.prefix6[i] = v.prefix6[i];
    for (int i = tid; i < 32; i += nt)
        s.zeros[i] = 12u;
    for (int wi = tid; wi < kFakeWords; wi += nt) {
        uint32_t word = 0;
        for (int b = 0; b < 32; b++) {
            const int p = wi * 32 + b;              // bit position in the stream
            const int val = p / 12;                 // 12-bit field holding it
            const uint32_t bit = val < 32 ? (uint32_t(val) >> (11 - p % 12)) & 1u : 0u;
            word |= bit << (31 - b);
        }
        s.fake[wi] = word;
    }
    __syncthreads();
    for (int w = tid; w < kLutEntries; w += nt) {
        const uint32_t a = s.prefix6[w >> 6];
        const uint32_t la = a & 15u;
        uint32_t entry = 0;
        if (la) {
            const uint32_t w2 = (uint32_t(w) << la) & 0xFFFu;
            const uint32_t b = s.prefix6[w2 >> 6];
            const uint32_t lb = b & 15u;
            if (lb)
                entry = ((b >> 4) << 23) | ((a >> 4) << 7) | (la + lb);
        }
        s.lut[w] = entry;
    }
}

// PTX prmt in its generic mode: a selector nibble with bit 3 set fills the
// target byte with the sign bit of the selected byte.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

__device__ __forceinline__ uint32_t lop3_merge(uint32_t sm_part, uint32_t exp_part) {
    // (sm_part & 0x807F807F) | (exp_part & 0x7F807F80)
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xE4;" : "=r"(r) : "r"(sm_part), "r"(exp_part), "r"(0x807F807Fu));
    return r;
}

// Per-tile, per-lane decode state set up by tile_setup().
struct LaneStream {
    const uint32_t *wp;    // next word to load
    const uint32_t *lutp;  // pair table of this lane (shared table, escape table or zeros)
    uint32_t hi, lo, c;    // 64-bit window and bit position (low 7 bits exact)
    uint32_t c0;           // starting bit offset (for the consumed-bits check)
    const uint32_t *wp0;
    int coded;             // lane holds Huffman codes (checked at the end)
    uint32_t glen;
};

// Registers holding one tile's raw inputs, loaded ahead of use.
struct TileRaw {
    uint4 sm[4];     // lane's 64 sign+mantissa bytes
    uint4 code[3];   // up to 96 16-byte chunks of the tile's code region
    uint32_t glen;   // lane's group byte length
    uint32_t beg16, n16;  // code region (16-byte units)
    uint32_t esc0, nesc;  // escape index of the tile and escaped groups in it
    int bad;              // offsets failed validation
};

// Tile coordinates.
struct TileCoord {
    int64_t rb, kg;  // row block and group column
    int R;           // rows in this block
};

__device__ __forceinline__ TileCoord tile_coord(const BlobView &v, int64_t t) {
    const int64_t gpr = v.cols / kGroup;
    TileCoord tc;
    tc.rb = t / gpr;
    tc.kg = t - tc.rb * gpr;
    const int64_t left = v.rows - tc.rb * kTileRows;
    tc.R = left < kTileRows ? int(left) : kTileRows;
    return tc;
}

// Load the offsets of tile t into lanes 0..3 (tcode[t], tcode[t+1],
// tesc[t], tesc[t+1]); issued one tile earlier than the data they locate.
__device__ __forceinline__ uint32_t tile_offsets_load(const BlobView &v, int64_t t) {
    const int lane = threadIdx.x & 31;
    uint32_t off = 0;
    if (lane < 2)
        off = __ldg(v.tcode + t + lane);
    else if (lane < 4)
        off = __ldg(v.tesc + t + (lane - 2));
    return off;
}

// Issue the global loads of tile t (no shared-memory traffic).  `offs` comes
// from tile_offsets_load(v, t).
__device__ __forceinline__ void tile_load(const BlobView &v, int64_t t, uint32_t offs, TileRaw &r) {
    const int lane = threadIdx.x & 31;
    const TileCoord tc = tile_coord(v, t);
    const int64_t gpr = v.cols / kGroup;
    const uint32_t c0 = __shfl_sync(0xffffffffu, offs, 0);
    const uint32_t c1 = __shfl_sync(0xffffffffu, offs, 1);
    const uint32_t e0 = __shfl_sync(0xffffffffu, offs, 2);
    const uint32_t e1 = __shfl_sync(0xffffffffu, offs, 3);
    r.beg16 = c0;
    r.n16 = c1 - c0;
    r.esc0 = e0;
    r.nesc = e1 - e0;
    r.bad = (c1 < c0) || (r.n16 * 16u > uint32_t(kMaxTileCodeBytes)) ||
            (uint64_t(c1) * 16u > v.code_bytes) || (e1 < e0) || (r.nesc > uint32_t(tc.R)) ||
            (uint64_t(e1) > v.n_escaped);
    const int64_t q0 = int64_t(kTileRows) * tc.rb * gpr + int64_t(tc.R) * tc.kg;
    const bool valid = lane < tc.R;
    r.glen = valid ? __ldg(v.glen + q0 + lane) : 0u;
    const uint8_t *smt = v.sm + q0 * kGroup;
#pragma unroll
    for (int c = 0; c < 4; c++)
        r.sm[c] = valid ? __ldg(reinterpret_cast<const uint4 *>(smt + (size_t(c) * tc.R + lane) * 16))
                        : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int c = 0; c < 3; c++) {
        const uint32_t idx = uint32_t(lane + 32 * c);
        r.code[c] = (!r.bad && idx < r.n16)
                        ? __ldg(reinterpret_cast<const uint4 *>(v.code + (size_t(r.beg16) + idx) * 16))
                        : make_uint4(0, 0, 0, 0);
    }
}

__device__ __forceinline__ uint32_t bswap32(uint32_t x) { return prmt(x, 0u, 0x0123u); }

// Stage the tile's codes and escape tables in the warp buffer and set up
// the lane's stream.  Returns whether the tile passed validation.
__device__ __forceinline__ bool tile_setup(const BlobView &v, const DecodeShared &s, const TileRaw &r,
                                           int R, uint32_t *wbuf, LaneStream &ls, uint32_t *status) {
    const int lane = threadIdx.x & 31;
    const bool valid = lane < R;
    // byte-swapped code words into the warp buffer
#pragma unroll
    for (int c = 0; c < 3; c++) {
        const uint32_t idx = uint32_t(lane + 32 * c);
        if (idx < r.n16 && !r.bad) {
            uint4 q = r.code[c];
            q.x = bswap32(q.x);
            q.y = bswap32(q.y);
            q.z = bswap32(q.z);
            q.w = bswap32(q.w);
            reinterpret_cast<uint4 *>(wbuf)[idx] = q;
        }
    }
    // code offsets by an exclusive warp prefix sum of the byte lengths
    const uint32_t g = r.glen;
    uint32_t incl = g;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t o = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d)
            incl += o;
    }
    const uint32_t off = incl - g;
    const uint32_t total = __shfl_sync(0xffffffffu, incl, 31);
    const uint32_t esc_mask = __ballot_sync(0xffffffffu, valid && g == 0);
    const uint32_t nesc = __popc(esc_mask);
    const uint32_t region = r.n16 * 16u;
    bool bad = r.bad || total > region || nesc != r.nesc || region + 128u * nesc > 4096u;
    if (bad && lane == 0)
        atomicOr(status, r.bad || total > region ? kStatusBadTile : kStatusBadEscape);
    // escape tables: 32 entries per escaped lane after the code region
    uint32_t *esc_tab = wbuf + region / 4;
    if (!bad) {
        uint32_t m = esc_mask;
        int rank = 0;
        while (m) {
            const uint16_t two = __ldg(reinterpret_cast<const uint16_t *>(v.esc + (uint64_t(r.esc0) + rank) * 64) + lane);
            const uint32_t e0 = two & 0xFFu, e1 = two >> 8;
            esc_tab[rank * 32 + lane] = (e1 << 23) | (e0 << 7) | 12u;
            m &= m - 1;
            rank++;
        }
    }
    __syncwarp();
    const uint32_t my_rank = __popc(esc_mask & ((1u << lane) - 1u));
    ls.coded = !bad && valid && g != 0;
    ls.glen = g;
    if (ls.coded) {
        const uint32_t *w0 = wbuf + (off >> 2);
        ls.c0 = 8u * (off & 3u);
        ls.hi = w0[0];
        ls.lo = w0[1];
        ls.wp = w0 + 2;
        ls.lutp = s.lut;
    } else {
        ls.c0 = 0;
        ls.hi = s.fake[0];
        ls.lo = s.fake[1];
        ls.wp = s.fake + 2;
        ls.lutp = (!bad && valid && g == 0) ? esc_tab + my_rank * 32 : s.zeros;
    }
    ls.wp0 = ls.wp;
    ls.c = ls.c0;
    return !bad;
}

// One step: decode the exponents of weights 2i, 2i+1 and merge them with the
// sign+mantissa bytes.  `sm4` holds the bytes of weights 4*(i/2)..+3.
// `I` is a compile-time constant once the caller's 32-step loop is unrolled.
__device__ __forceinline__ uint32_t decode_pair(LaneStream &ls, int I, uint32_t sm4) {
    const uint32_t win = __funnelshift_l(ls.lo, ls.hi, ls.c);
    const uint32_t ent = ls.lutp[win >> 20];
    const uint32_t c2 = ls.c + ent;  // bits above 6 collect junk; the low 7 stay exact
    if ((c2 ^ ls.c) & 32u) {
        ls.hi = ls.lo;
        ls.lo = *ls.wp++;
    }
    ls.c = c2;
    // sign-replicate byte permute: bytes (b0, sign(b0), b1, sign(b1)) for the
    // even pair of the word, (b2, sign(b2), b3, sign(b3)) for the odd one
    const uint32_t y = prmt(sm4, 0u, (I & 1) ? 0xB3A2u : 0x9180u);
    return lop3_merge(y, ent);
}

// After the 32 steps: a coded lane must have used exactly its byte length.
__device__ __forceinline__ void tile_check(const LaneStream &ls, uint32_t *status) {
    if (ls.coded) {
        const uint32_t used = 32u * uint32_t(ls.wp - ls.wp0) + (ls.c & 31u) - ls.c0;
        if (((used + 7u) >> 3) != ls.glen)
            atomicOr(status, uint32_t(kStatusBadCode));
    }
}

__device__ __forceinline__ uint32_t sm_word(const uint4 (&sm)[4], int w) {
    const uint4 &q = sm[w >> 2];
    switch (w & 3) {
        case 0: return q.x;
        case 1: return q.y;
        case 2: return q.z;
        default: return q.w;
    }
}

}  // namespace uw
