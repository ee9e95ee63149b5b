// Device-side tile decoder shared by the decompress and fused matmul kernels.
//
// One warp decodes one tile (32 rows x 64 columns): lane j owns the 64-weight
// group of row j (Unweight blog, paragraph on rows of 64).  Per tile:
//   * the tile's code bytes are copied with cp.async straight into one of
//     the warp's two shared-memory code buffers while the previous tile is
//     being decoded, and its sign+mantissa bytes are loaded into registers;
//   * the group byte lengths (glen) give each lane its code offset by an
//     exclusive warp prefix sum (shuffles); ballot + popc give each escaped
//     group its rank among the tile's escaped groups;
//   * read as little-endian 32-bit words, stream bit i is bit i%32 of word
//     i/32, so a funnel shift right brings the next bits to the bottom;
//   * every step looks up a 12-bit window (first stream bit = bit 0) in a
//     4096-entry table that decodes two codes at once (codes are at most 6
//     bits).  An entry holds both exponents already in BF16 position (bits
//     14..7 and 30..23) and the bits the two codes take (bits 3..0);
//   * the exponent pair is merged with two raw sign+mantissa bytes by one
//     byte permute (sign-replicating) and one three-input logic op, giving
//     two BF16 weights in one 32-bit register (the blog's reconstruction:
//     exponent + sign/mantissa bytes -> BF16, paragraph on the consumer
//     warps of the reconstructive matmul).
// Escaped groups (rare) and lanes without a row run the same loop on a
// fixed stream of 12-bit numbers 0..31 through a 32-entry table of zero
// exponents, so the hot loop has no branch on the group kind; the escaped
// groups are then redone in a short second pass from their raw exponent
// bytes.  Every lane's sum is independent of the other lanes', so the
// second pass gives exactly what a single pass would.
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
    uint32_t code16;      // code section size in 16-byte units (fits: tile offsets are u32)
    uint32_t n_esc32;     // escaped groups (fits: escape offsets are u32)
    int64_t rows, cols;
    // 6-bit prefix -> (exponent << 4) | code length; 0 where no code starts
    // with that prefix.
    uint16_t prefix6[64];
};

constexpr int kLutEntries = 4096;
constexpr int kFakeWords = 16;                             // stream of 12-bit values 0..31 (+slack)
// One tile's shared buffer: its code region, then the raw exponent bytes of
// its escaped groups ((32 - e) * 48 + 64 * e <= 2048 bytes), then read slack.
constexpr int kTileBufData = 2048;
constexpr int kCodeBufBytes = kTileBufData + 64;
constexpr int kWarpBufBytes = 2 * kCodeBufBytes;           // two buffers: decode one, fill the other
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
            const uint32_t bit = val < 32 ? (uint32_t(val) >> (p % 12)) & 1u : 0u;
            word |= bit << b;
        }
        s.fake[wi] = word;
    }
    __syncthreads();
    // Window w holds stream bits in order from bit 0; codes enter the stream
    // most significant bit first, so the code-order window is w reversed.
    for (int w = tid; w < kLutEntries; w += nt) {
        const uint32_t r = __brev(uint32_t(w)) >> 20;
        const uint32_t a = s.prefix6[r >> 6];
        const uint32_t la = a & 15u;
        uint32_t entry = 0;
        if (la) {
            const uint32_t r2 = (r << la) & 0xFFFu;
            const uint32_t b = s.prefix6[r2 >> 6];
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

// Where a tile's data lives: rows 32*rb .. 32*rb+R-1, group column kg.
struct TileLoc {
    const uint8_t *sm;    // the tile's sign+mantissa bytes (64 * R)
    const uint8_t *glen;  // the tile's group byte lengths (R)
    int R;                // rows in the tile
};

__device__ __forceinline__ TileLoc tile_loc(const BlobView &v, int64_t rb, int64_t kg, int64_t gpr) {
    TileLoc L;
    const int64_t left = v.rows - rb * kTileRows;
    L.R = left < kTileRows ? int(left) : kTileRows;
    const int64_t q0 = int64_t(kTileRows) * rb * gpr + int64_t(L.R) * kg;  // first group of the tile
    L.sm = v.sm + q0 * kGroup;
    L.glen = v.glen + q0;
    return L;
}

__device__ __forceinline__ int tile_rows(const BlobView &v, int64_t rb) {
    const int64_t left = v.rows - rb * kTileRows;
    return left < kTileRows ? int(left) : kTileRows;
}

// A tile's bookkeeping as fetched: the lane's glen, and warp-uniform
// values: first escaped group, and n16 | nesc << 8 | bad << 16.
struct TileMeta {
    uint32_t glen;
    uint32_t esc0;
    uint32_t pk;
};

// Load the offsets of tile t = rb * (cols/64) + kg into lanes 0..3
// (tcode[t], tcode[t+1], tesc[t], tesc[t+1]); issued ahead of the data.
__device__ __forceinline__ uint32_t tile_offsets_load(const BlobView &v, int64_t t) {
    const int lane = threadIdx.x & 31;
    const uint32_t *src = lane < 2 ? v.tcode + t + lane : v.tesc + t + (lane - 2);
    return lane < 4 ? __ldg(src) : 0u;
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(dst), "l"(src) : "memory");
}

// The lane's 64 sign+mantissa bytes: chunk c of row j sits at (c*R + j)*16
// inside the tile (zeros for lanes without a row).
__device__ __forceinline__ void tile_sm_load(const TileLoc &L, uint4 (&sm)[4]) {
    const int lane = threadIdx.x & 31;
    const uint8_t *smb = L.sm + 16 * lane;
    const int stride = 16 * L.R;
#pragma unroll
    for (int c = 0; c < 4; c++)
        sm[c] = lane < L.R ? __ldg(reinterpret_cast<const uint4 *>(smb + c * stride)) : make_uint4(0, 0, 0, 0);
}

// Fetch a tile: validate its offsets (`offs` from tile_offsets_load), load
// the lane's glen and 64 sign+mantissa bytes into registers, and start
// copying its code region followed by its escaped groups' raw exponents
// into the tile buffer at shared address `cbuf` (cp.async, one commit
// group).
__device__ __forceinline__ void tile_fetch(const BlobView &v, const TileLoc &L, uint32_t offs, uint32_t cbuf,
                                           TileMeta &m, uint4 (&sm)[4]) {
    const int lane = threadIdx.x & 31;
    const uint32_t c0 = __shfl_sync(0xffffffffu, offs, 0);
    const uint32_t c1 = __shfl_sync(0xffffffffu, offs, 1);
    const uint32_t e0 = __shfl_sync(0xffffffffu, offs, 2);
    const uint32_t e1 = __shfl_sync(0xffffffffu, offs, 3);
    const uint32_t n16 = c1 - c0, nesc = e1 - e0;
    const bool bad = c1 < c0 || n16 > uint32_t(kMaxTileCodeBytes / 16) || c1 > v.code16 || e1 < e0 ||
                     nesc > uint32_t(L.R) || e1 > v.n_esc32 || n16 * 16u + nesc * 64u > uint32_t(kTileBufData);
    m.pk = bad ? (1u << 16) : (n16 | (nesc << 8));
    m.esc0 = e0;
    m.glen = lane < L.R ? __ldg(L.glen + lane) : 0u;
    tile_sm_load(L, sm);
    if (!bad) {
        const uint8_t *src = v.code + size_t(c0) * 16 + 16 * lane;
        const uint32_t dst = cbuf + 16u * lane;
#pragma unroll
        for (int c = 0; c < 3; c++)
            if (uint32_t(lane + 32 * c) < n16)
                cp_async16(dst + 512u * c, src + 512 * c);
        if (nesc) {
            const uint8_t *esrc = v.esc + size_t(e0) * 64 + 16 * lane;
            const uint32_t edst = cbuf + 16u * n16 + 16u * lane;
#pragma unroll
            for (int c = 0; c < 4; c++)
                if (uint32_t(lane + 32 * c) < 4 * nesc)
                    cp_async16(edst + 512u * c, esrc + 512 * c);
        }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// Per-tile, per-lane decode state.  Addresses are 32-bit shared addresses.
struct LaneStream {
    uint32_t lo, hi, nx;   // current, next and (already loaded) following stream word
    uint32_t c;            // bit position in lo (low 5 bits); low 7 bits exact
    uint32_t wp;           // address of the next word to load
    uint32_t lut;          // pair table of this lane (codes) or the zero table
    uint32_t base;         // 8 * (first wp) + start bit: bits used = 8 * wp + (c & 31) - base
    uint32_t glen;         // bytes the lane must use (48 for lanes on the fixed stream)
};

// Wait for the tile's codes, validate, and set up every lane's stream.
// Returns the mask of lanes whose group is escaped (0 for a bad tile, whose
// lanes all decode zeros; the error is recorded in *status).
__device__ __forceinline__ uint32_t tile_begin(const DecodeShared &s, const TileMeta &m, int R, uint32_t cbuf,
                                               LaneStream &ls, uint32_t *status) {
    const int lane = threadIdx.x & 31;
    const bool valid = lane < R;
    const uint32_t n16 = m.pk & 0xFFu, nesc = (m.pk >> 8) & 0xFFu;
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncwarp();
    const uint32_t g = m.glen;
    uint32_t incl = g;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t u = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d)
            incl += u;
    }
    const uint32_t off = incl - g;
    const uint32_t total = __shfl_sync(0xffffffffu, incl, 31);
    const uint32_t esc_mask = __ballot_sync(0xffffffffu, valid && g == 0);
    const bool over = (m.pk >> 16) != 0 || total > n16 * 16u;
    const bool bad = over || uint32_t(__popc(esc_mask)) != nesc;
    if (bad && lane == 0)
        atomicOr(status, over ? kStatusBadTile : kStatusBadEscape);
    uint32_t w0, c0;
    if (!bad && valid && g != 0) {
        w0 = cbuf + (off & ~3u);
        c0 = 8u * (off & 3u);
        ls.lut = smem_addr(s.lut);
        ls.glen = g;
    } else {
        w0 = smem_addr(s.fake);
        c0 = 0;
        ls.lut = smem_addr(s.zeros);
        ls.glen = 48;  // the fixed stream is 32 fields of 12 bits
    }
    ls.lo = lds32(w0);
    ls.hi = lds32(w0 + 4);
    ls.nx = lds32(w0 + 8);
    ls.wp = w0 + 12;
    ls.c = c0;
    ls.base = 8u * ls.wp + c0;
    return bad ? 0u : esc_mask;
}

// Shared address of a fetched tile's raw escape bytes (after its codes).
__device__ __forceinline__ uint32_t escape_base(const TileMeta &m, uint32_t cbuf) {
    return cbuf + 16u * (m.pk & 0xFFu);
}

// Raw exponent bytes of the calling lane's escaped group, from the tile
// buffer (lane must be in the mask returned by tile_begin; `ebase` from
// escape_base).
__device__ __forceinline__ void escape_read(uint32_t ebase, uint32_t esc_mask, uint4 (&e)[4]) {
    const int lane = threadIdx.x & 31;
    const uint32_t rank = __popc(esc_mask & ((1u << lane) - 1u));
    const uint32_t a = ebase + 64u * rank;
#pragma unroll
    for (int c = 0; c < 4; c++)
        e[c] = lds128(a + 16u * c);
}

// One step: decode the exponents of weights 2i, 2i+1 and merge them with the
// sign+mantissa bytes.  `sm4` holds the bytes of weights 4*(i/2)..+3.
// `I` is a compile-time constant once the caller's 32-step loop is unrolled.
__device__ __forceinline__ uint32_t decode_pair(LaneStream &ls, int I, uint32_t sm4) {
    // window = next 32 stream bits (funnel right); entry = table[window & 4095];
    // c += entry (its bits above 6 only add junk above the exact low 7);
    // when bit 5 of c flips the window has moved into the next word: shift
    // the words and load the one after, predicated rather than branched.  The
    // loaded word is needed only at the following crossing, so the load is
    // off the step-to-step dependency chain.
    uint32_t ent;
    asm volatile(
        "{\n\t"
        ".reg .b32 win, addr, c2, t;\n\t"
        ".reg .pred p;\n\t"
        "shf.r.wrap.b32 win, %1, %2, %4;\n\t"
        "and.b32 win, win, 4095;\n\t"
        "mad.lo.u32 addr, win, 4, %6;\n\t"     // integer multiply-add: FMA pipe, not ALU
        "ld.shared.u32 %0, [addr];\n\t"
        "mad.lo.u32 c2, %0, 1, %4;\n\t"
        "xor.b32 t, c2, %4;\n\t"
        "and.b32 t, t, 32;\n\t"
        "setp.ne.u32 p, t, 0;\n\t"
        "@p mov.b32 %1, %2;\n\t"
        "@p mov.b32 %2, %3;\n\t"
        "@p ld.shared.u32 %3, [%5];\n\t"
        "@p mad.lo.u32 %5, 1, 4, %5;\n\t"
        "mov.b32 %4, c2;\n\t"
        "}"
        : "=r"(ent), "+r"(ls.lo), "+r"(ls.hi), "+r"(ls.nx), "+r"(ls.c), "+r"(ls.wp)
        : "r"(ls.lut)
        : "memory");
    // sign-replicate byte permute: bytes (b0, sign(b0), b1, sign(b1)) for the
    // even pair of the word, (b2, sign(b2), b3, sign(b3)) for the odd one
    const uint32_t y = prmt(sm4, 0u, (I & 1) ? 0xB3A2u : 0x9180u);
    return lop3_merge(y, ent);
}

// After the 32 steps: every lane must have used exactly its byte length.
__device__ __forceinline__ void tile_check(const LaneStream &ls, uint32_t *status) {
    const uint32_t used = 8u * ls.wp + (ls.c & 31u) - ls.base;
    if (((used + 7u) >> 3) != ls.glen)
        atomicOr(status, uint32_t(kStatusBadCode));
}

__device__ __forceinline__ uint32_t word4(const uint4 &q, int w) {
    return (w & 3) == 0 ? q.x : (w & 3) == 1 ? q.y : (w & 3) == 2 ? q.z : q.w;
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

// Pair I of an escaped group: its two raw exponents (bytes 2I, 2I+1 of `e`)
// moved to BF16 position, merged with the sign+mantissa bytes as in
// decode_pair.
__device__ __forceinline__ uint32_t escape_pair(const uint4 (&e)[4], int I, uint32_t sm4) {
    const uint32_t two = prmt(sm_word(e, I >> 1), 0u, (I & 1) ? 0x4342u : 0x4140u);  // e_lo | e_hi << 16
    const uint32_t y = prmt(sm4, 0u, (I & 1) ? 0xB3A2u : 0x9180u);
    return lop3_merge(y, two << 7);
}

}  // namespace uw
