// Device-side tile decoder shared by the decompress and matmul kernels.
//
// One warp decodes one tile (32 rows x 64 columns): lane j owns the 64-weight
// group of row j (Unweight blog, paragraph on rows of 64).  Per tile:
//   * the tile's code bytes (and the raw exponents of its escaped groups)
//     are copied with cp.async into one of the warp's shared-memory tile
//     buffers while the previous tile is being decoded, and its
//     sign+mantissa bytes are loaded into registers;
//   * the group byte lengths (glen) give each lane its code offset by an
//     exclusive warp prefix sum (shuffles); ballot + popc give each escaped
//     group its rank among the tile's escaped groups;
//   * read as little-endian 32-bit words, stream bit i is bit i%32 of word
//     i/32; a lane keeps two consecutive words as one 64-bit window and a
//     64-bit shift right brings its next bits to the bottom;
//   * every step looks up a 10-bit window in a 1024-entry table that decodes
//     two codes at once (codes are at most 5 bits).  An entry holds both
//     exponents already in BF16 position (bits 14..7 and 30..23) and the bits
//     the two codes take (bits 3..0).  The entry's address is the window
//     times a stride plus a base, one integer multiply-add (which runs on the
//     FMA pipe, leaving the half-rate ALU pipe to the shifts and masks):
//     stride 4 indexes one shared table, stride 128 indexes 32 lane-private
//     copies of it, copy l holding entry w at word 32*w + l.  Lane l then
//     always reads bank l, so a lookup is a single shared-memory wavefront
//     whatever the 32 windows are (one shared table costs about four: the
//     windows are random);
//   * two codes take at most 10 bits, so three steps from a bit offset below
//     32 stay inside the 64-bit window; the window moves on by a word (a
//     predicated refill from the word already loaded after it) only after
//     every third step, not after every step;
//   * the exponent pair is merged with two raw sign+mantissa bytes by one
//     byte permute (sign-replicating) and one three-input logic op, giving
//     two BF16 weights in one 32-bit register (the blog's reconstruction:
//     exponent + sign/mantissa bytes -> BF16, paragraph on the consumer
//     warps of the reconstructive matmul).
// Escaped groups (rare) and lanes without a row run the same loop over a
// block of zero bytes, so the hot loop has no branch on the group kind; the
// escaped groups are then redone in a short second pass from their raw
// exponent bytes.  Every lane's sum is independent of the other lanes', so
// the second pass gives exactly what a single pass would.
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

constexpr int kPrefixEntries = 1 << kLmax;

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
    uint32_t tdata;       // tile buffer capacity: the blob's largest tile, a multiple of 16
    uint32_t tbuf;        // tile buffer stride: tdata + kTileSlack
    uint32_t gpr;         // 64-column groups per row (32-bit kernels: tiles < 2^32)
    uint32_t nfull;       // full 32-row blocks
    uint32_t tail_rows;   // rows of the last, partial block (0: none)
    uint32_t ntiles;      // tiles (the tile tables hold ntiles + 1 entries)
    int64_t rows, cols;   // cols: the stored width, a multiple of 64
    int64_t ocols;        // the matrix's own columns (cols rounded up to 64 gives cols)
    // kLmax-bit prefix -> (exponent << 4) | code length; 0 where no code
    // starts with that prefix.
    uint16_t prefix[kPrefixEntries];
    uint8_t palette[16];  // exponent of each palette index (unused entries 0)
};

constexpr int kWindowBits = 2 * kLmax;                     // two codes always fit
constexpr int kLutEntries = 1 << kWindowBits;              // 1024
constexpr int kPrivateLutBytes = kLutEntries * 32 * 4;     // 32 lane-private copies: 128 KB
constexpr int kHalfLutBytes = kLutEntries * 16 * 4;        // 16 copies (lanes l, l + 16 share one): 64 KB
constexpr int kZeroWords = 32;                             // zero stream for lanes without codes
// One tile's shared buffer: its code region, then the raw exponent bytes of
// its escaped groups ((32 - e) * 48 + 64 * e <= 2048 bytes), then read
// slack.  Buffers are sized for the largest tile of the blob at hand.
constexpr uint32_t kMaxTileData = 2048;
constexpr uint32_t kTileSlack = 64;
constexpr int kCommonSmemBytes = kLutEntries * 4 + kZeroWords * 4 + kPrefixEntries * 2;

// Shared memory common to every decoding CTA.
struct DecodeShared {
    uint32_t *lut;       // [1024] pair table (or, when built private, 32 copies elsewhere)
    uint32_t *zero;      // [32]   zero bytes: the stream of lanes without codes
    uint16_t *prefix;    // [32]
};

__device__ __forceinline__ DecodeShared carve_common(unsigned char *smem) {
    DecodeShared s;
    s.lut = reinterpret_cast<uint32_t *>(smem);
    s.zero = s.lut + kLutEntries;
    s.prefix = reinterpret_cast<uint16_t *>(s.zero + kZeroWords);
    return s;
}

// Table entry of window w.  The window holds stream bits in order from bit
// 0; codes enter the stream most significant bit first, so the code-order
// window is w reversed.
__device__ __forceinline__ uint32_t pair_entry(const uint16_t *prefix, uint32_t w) {
    const uint32_t r = __brev(w) >> (32 - kWindowBits);
    const uint32_t a = prefix[r >> kLmax];
    const uint32_t la = a & 15u;
    uint32_t entry = 0;
    if (la) {
        const uint32_t r2 = (r << la) & uint32_t(kLutEntries - 1);
        const uint32_t b = prefix[r2 >> kLmax];
        const uint32_t lb = b & 15u;
        if (lb)
            entry = ((b >> 4) << 23) | ((a >> 4) << 7) | (la + lb);
    }
    return entry;
}

__device__ __forceinline__ void build_prefix_zero(const DecodeShared &s, const BlobView &v) {
    const int tid = threadIdx.x, nt = blockDim.x;
    for (int i = tid; i < kPrefixEntries; i += nt)
        s.prefix[i] = v.prefix[i];
    for (int i = tid; i < kZeroWords; i += nt)
        s.zero[i] = 0u;
    __syncthreads();
}

// Fill the pair table and the zero stream.  Must be followed by
// __syncthreads() before use.
__device__ __forceinline__ void build_tables(const DecodeShared &s, const BlobView &v) {
    build_prefix_zero(s, v);
    for (int w = threadIdx.x; w < kLutEntries; w += blockDim.x)
        s.lut[w] = pair_entry(s.prefix, uint32_t(w));
}

// The pair table with palette indices in place of exponents (index of the
// first code at bits 7..10, of the second at bits 23..26), for transcoding
// to the palette-4 form.  Must be followed by __syncthreads() before use.
__device__ __forceinline__ void build_tables_palette_index(const DecodeShared &s, const BlobView &v) {
    const int tid = threadIdx.x;
    if (tid < kPrefixEntries) {
        const uint32_t p = v.prefix[tid];
        uint32_t idx = 0;
        for (int i = 15; i >= 0; i--)  // the first palette entry with this exponent
            if (v.palette[i] == (p >> 4))
                idx = uint32_t(i);
        s.prefix[tid] = uint16_t((idx << 4) | (p & 15u));
    }
    if (tid < kZeroWords)
        s.zero[tid] = 0u;
    __syncthreads();
    for (int w = tid; w < kLutEntries; w += blockDim.x)
        s.lut[w] = pair_entry(s.prefix, uint32_t(w));
}

// Second half of a private-table build: after build_tables and a
// __syncthreads(), copy the pair table into 32 lane-private copies at shared
// address `priv` (kPrivateLutBytes, 16-byte aligned; entry w of copy l at
// word 32*w + l) for decode_pair<kStridePrivate>.  Must be followed by
// __syncthreads() before use.
__device__ __forceinline__ void replicate_private(const DecodeShared &s, uint32_t priv) {
    for (int i = threadIdx.x; i < kLutEntries * 8; i += blockDim.x) {
        const uint32_t e = s.lut[uint32_t(i) >> 3];
        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" :: "r"(priv + 16u * uint32_t(i)), "r"(e) : "memory");
    }
}

// The 32 lane-private copies made directly, without the single table in
// between (after build_prefix_zero): each warp makes 32 entries at a time,
// one per lane, and writes their rows (entry w of copy l at word 32w + l,
// as replicate_private lays them out) four rows at a time, 512 contiguous
// bytes per store instruction.  Needs no barrier between warps; follow with
// __syncthreads() before use.
__device__ __forceinline__ void build_private(const DecodeShared &s, uint32_t priv) {
    const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    for (uint32_t base = 32u * warp; base < uint32_t(kLutEntries); base += 32u * nw) {
        const uint32_t e = pair_entry(s.prefix, base + lane);
#pragma unroll
        for (uint32_t i = 0; i < 8u; i++) {
            const uint32_t r = 4u * i + (lane >> 3);
            const uint32_t er = __shfl_sync(0xffffffffu, e, int(r));
            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};"
                         :: "r"(priv + 128u * (base + r) + 16u * (lane & 7u)), "r"(er) : "memory");
        }
    }
}

// The same with 16 copies (entry w of copy c at word 16w + c), read by
// lane l from copy l % 16: a lookup is one or two wavefronts (lanes l and
// l + 16 meet in a bank when their entries' parities agree).
__device__ __forceinline__ void replicate_half(const DecodeShared &s, uint32_t tab) {
    for (int i = threadIdx.x; i < kLutEntries * 4; i += blockDim.x) {
        const uint32_t e = s.lut[uint32_t(i) >> 2];
        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" :: "r"(tab + 16u * uint32_t(i)), "r"(e) : "memory");
    }
}

constexpr int kStrideShared = 4;    // bytes between entries of one table
constexpr int kStridePrivate = 128; // bytes between rows of 32 lane-private copies
constexpr int kStrideHalf = 64;     // bytes between rows of 16 copies shared by lanes l and l + 16

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

// The same with 32-bit indices, t = rb * gpr + kg.  A partial last block
// holds R < 32 rows, so its tiles start (32 - R) * kg groups before 32 * t.
__device__ __forceinline__ TileLoc tile_loc32(const BlobView &v, uint32_t rb, uint32_t kg, uint32_t t) {
    TileLoc L;
    const bool full = rb < v.nfull;
    L.R = full ? kTileRows : int(v.tail_rows);
    const uint32_t short_by = full ? 0u : (kTileRows - v.tail_rows) * kg;
    L.sm = v.sm + uint64_t(t) * (kTileRows * kGroup) - uint64_t(short_by) * kGroup;
    L.glen = v.glen + uint64_t(t) * kTileRows - short_by;
    return L;
}

__device__ __forceinline__ int tile_rows32(const BlobView &v, uint32_t rb) {
    return rb < v.nfull ? kTileRows : int(v.tail_rows);
}

__device__ __forceinline__ int tile_rows(const BlobView &v, int64_t rb) {
    const int64_t left = v.rows - rb * kTileRows;
    return left < kTileRows ? int(left) : kTileRows;
}

// A tile's bookkeeping as fetched: the lane's glen (any value for lanes
// without a row), and warp-uniform values: first escaped group, and
// n16 | nesc << 8 | bad << 16.  The loads are consumed only by tile_begin,
// so fetching never waits for them.
struct TileMeta {
    uint32_t glen;
    uint32_t esc0;
    uint32_t pk;
};

// Load the offsets of tile t into lanes 0..3 (32-bit tile index).
__device__ __forceinline__ uint32_t tile_offsets_load32(const BlobView &v, uint32_t t) {
    const int lane = threadIdx.x & 31, l = lane & 3;
    const uint32_t *src = (l < 2 ? v.tcode + l : v.tesc + (l - 2)) + t;
    return lane < 4 ? __ldg(src) : 0u;
}

// Load the offsets of tile t = rb * (cols/64) + kg into lanes 0..3
// (tcode[t], tcode[t+1], tesc[t], tesc[t+1]); issued ahead of the data.
__device__ __forceinline__ uint32_t tile_offsets_load(const BlobView &v, int64_t t) {
    const int lane = threadIdx.x & 31;
    const uint32_t *src = lane < 2 ? v.tcode + t + lane : v.tesc + t + (lane - 2);
    return lane < 4 ? __ldg(src) : 0u;
}

// The tiles one warp of a decode kernel walks: runs of `per` consecutive
// tiles (t = rb * gpr + kg), run number (k * gridDim.x + blockIdx.x) * W +
// warp for k = 0, 1, ... while tiles remain.  A grid smaller than the number
// of runs makes the kernel persistent (the SM split of a preprocess kernel
// running beside a matmul).
struct TileWalk {
    uint32_t t, lo, rb, kg;  // current tile, first tile of its run, row block, group column
};

__device__ __forceinline__ void walk_seek(TileWalk &w, uint32_t t, uint32_t gpr) {
    w.t = t;
    w.lo = t;
    w.rb = t / gpr;
    w.kg = t - w.rb * gpr;
}

// step = gridDim.x * W * per: the distance between a warp's runs.
__device__ __forceinline__ void walk_next(TileWalk &w, uint32_t per, uint32_t step, uint32_t ntiles, uint32_t gpr) {
    w.t++;
    if (w.t - w.lo == per || w.t >= ntiles) {
        const uint32_t lo = (step < ntiles && w.lo < ntiles - step) ? w.lo + step : ntiles;
        walk_seek(w, lo, gpr);
    } else if (++w.kg == gpr) {
        w.kg = 0;
        w.rb++;
    }
}

// Programmatic dependent launch: let the next kernel in the stream start
// launching, and wait until every earlier kernel has completed and its
// writes are visible.
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

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
// inside the tile.  Lanes without a row read row 0's bytes (their results
// are never used).
__device__ __forceinline__ void tile_sm_load(const TileLoc &L, uint4 (&sm)[4]) {
    const int lane = threadIdx.x & 31;
    const uint8_t *smb = L.sm + 16 * (lane < L.R ? lane : 0);
    const int stride = 16 * L.R;
#pragma unroll
    for (int c = 0; c < 4; c++)
        sm[c] = __ldg(reinterpret_cast<const uint4 *>(smb + c * stride));
}

// Ask L2 to bring in a tile's sign+mantissa bytes (one lane issues it).
__device__ __forceinline__ void tile_prefetch_sm_l2(const TileLoc &L) {
    if ((threadIdx.x & 31) == 0 && L.R > 0)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(L.sm), "r"(uint32_t(64 * L.R)) : "memory");
}

// Load chunks c0, c0+1 of the lane's sign+mantissa bytes (see tile_sm_load).
__device__ __forceinline__ void tile_sm_load_half(const TileLoc &L, int c0, uint4 &a, uint4 &b) {
    const int lane = threadIdx.x & 31;
    const uint8_t *smb = L.sm + 16 * (lane < L.R ? lane : 0) + c0 * 16 * L.R;
    a = __ldg(reinterpret_cast<const uint4 *>(smb));
    b = __ldg(reinterpret_cast<const uint4 *>(smb + 16 * L.R));
}

// Fetch a tile's codes: validate its offsets (`offs` from
// tile_offsets_load), load the lane's glen, and start copying its code
// region followed by its escaped groups' raw exponents into the tile buffer
// at shared address `cbuf` (cp.async, one commit group).
__device__ __forceinline__ void tile_fetch_codes(const BlobView &v, const TileLoc &L, uint32_t offs, uint32_t cbuf,
                                                 TileMeta &m) {
    const int lane = threadIdx.x & 31;
    const uint32_t c0 = __shfl_sync(0xffffffffu, offs, 0);
    const uint32_t c1 = __shfl_sync(0xffffffffu, offs, 1);
    const uint32_t e0 = __shfl_sync(0xffffffffu, offs, 2);
    const uint32_t e1 = __shfl_sync(0xffffffffu, offs, 3);
    const uint32_t n16 = c1 - c0, nesc = e1 - e0;
    const bool bad = c1 < c0 || n16 > uint32_t(kMaxTileCodeBytes / 16) || c1 > v.code16 || e1 < e0 ||
                     nesc > uint32_t(L.R) || e1 > v.n_esc32 || n16 * 16u + nesc * 64u > v.tdata;
    m.pk = bad ? (1u << 16) : (n16 | (nesc << 8));
    m.esc0 = e0;
    m.glen = __ldg(L.glen + (lane < L.R ? lane : 0));  // lanes without a row: ignored by tile_begin
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

// tile_fetch_codes, plus the lane's 64 sign+mantissa bytes into registers.
__device__ __forceinline__ void tile_fetch(const BlobView &v, const TileLoc &L, uint32_t offs, uint32_t cbuf,
                                           TileMeta &m, uint4 (&sm)[4]) {
    tile_fetch_codes(v, L, offs, cbuf, m);
    tile_sm_load(L, sm);
}

// Per-tile, per-lane decode state.  Addresses are 32-bit shared addresses.
// The lane's next code bit is bit c of the 64-bit window {hi:lo}, where lo
// is the word at wp - 12 and hi the word after it; nx (the word at wp - 4)
// is already loaded.  c is below 32 at the start of every round of three
// steps.  The bit address of the next code bit is 8 * wp + c - 96 whatever
// the refills did.
struct LaneStream {
    uint32_t lo, hi, nx;   // window words and the (already loaded) following word
    uint32_t c;            // bit offset of the next code bit in {hi:lo}
    uint32_t wp;           // address of the next word to load
    uint32_t expect;       // 8 * wp + c after the lane's last code, + 0..7; 0: unchecked
};

// Set up a lane's stream at byte offset `off` of the tile buffer at `cbuf`
// (coded lanes), or at the zero stream.  The lane's group has g code bytes.
__device__ __forceinline__ void stream_setup(const DecodeShared &s, bool coded, uint32_t cbuf, uint32_t off,
                                             uint32_t g, LaneStream &ls) {
    const uint32_t w0 = coded ? cbuf + (off & ~3u) : smem_addr(s.zero);
    const uint32_t c0 = coded ? 8u * (off & 3u) : 0u;
    ls.lo = lds32(w0);
    ls.hi = lds32(w0 + 4);
    ls.nx = lds32(w0 + 8);
    ls.wp = w0 + 12;
    ls.c = c0;
    ls.expect = coded ? 8u * ls.wp + c0 + 8u * g : 0u;
}

// Wait for the tile's codes, validate, and set up every lane's stream.
// Returns the mask of lanes whose group is escaped (0 for a bad tile, whose
// lanes all decode the zero stream; the error is recorded in *status).
// tile_begin for data already in shared memory (nothing to wait for).
__device__ __forceinline__ uint32_t tile_begin_ready(const DecodeShared &s, const TileMeta &m, int R, uint32_t cbuf,
                                                     LaneStream &ls, uint32_t *status) {
    const int lane = threadIdx.x & 31;
    const bool valid = lane < R;
    const uint32_t n16 = m.pk & 0xFFu, nesc = (m.pk >> 8) & 0xFFu;
    const uint32_t g = valid ? m.glen : 0u;
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
    stream_setup(s, !bad && g != 0, cbuf, off, g, ls);
    return bad ? 0u : esc_mask;
}

// tile_begin_ready for the two tiles of a pair at once (B has RB = R or 0
// rows): one warp prefix sum over both group lengths packed into one word
// (a tile's sum is at most 32 * 255 < 2^16, so the halves never carry into
// each other), the source lane's existence taken from the shuffle's own
// predicate.  Returns both escape masks.
__device__ __forceinline__ void pair_begin_ready(const DecodeShared &s, uint32_t gA, uint32_t gB, uint32_t pkA,
                                                 uint32_t pkB, int R, int RB, uint32_t cbA, uint32_t cbB,
                                                 LaneStream &la, LaneStream &lb, uint32_t *status, uint32_t &emA,
                                                 uint32_t &emB) {
    const int lane = threadIdx.x & 31;
    const bool vA = lane < R, vB = lane < RB;
    const uint32_t ga = vA ? gA : 0u, gb = vB ? gB : 0u;  // group lengths are bytes
    const uint32_t g2 = ga | (gb << 16);
    uint32_t incl = g2;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1)
        asm("{\n\t.reg .b32 u;\n\t.reg .pred p;\n\t"
            "shfl.sync.up.b32 u|p, %0, %1, 0, -1;\n\t"
            "@p add.u32 %0, %0, u;\n\t}"
            : "+r"(incl) : "r"(d));
    const uint32_t off2 = incl - g2;
    const uint32_t tot2 = __shfl_sync(0xffffffffu, incl, 31);
    const uint32_t mA = __ballot_sync(0xffffffffu, vA && ga == 0u);
    const uint32_t mB = __ballot_sync(0xffffffffu, vB && gb == 0u);
    auto setup = [&](uint32_t g, uint32_t off, uint32_t total, uint32_t esc_mask, uint32_t pk, uint32_t cbuf,
                     LaneStream &ls) -> uint32_t {
        const uint32_t n16 = pk & 0xFFu, nesc = (pk >> 8) & 0xFFu;
        const bool over = (pk >> 16) != 0 || total > n16 * 16u;
        const bool bad = over || uint32_t(__popc(esc_mask)) != nesc;
        if (bad && lane == 0)
            atomicOr(status, over ? kStatusBadTile : kStatusBadEscape);
        stream_setup(s, !bad && g != 0, cbuf, off, g, ls);
        return bad ? 0u : esc_mask;
    };
    emA = setup(ga, off2 & 0xFFFFu, tot2 & 0xFFFFu, mA, pkA, cbA, la);
    emB = setup(gb, off2 >> 16, tot2 >> 16, mB, pkB, cbB, lb);
}

__device__ __forceinline__ uint32_t tile_begin(const DecodeShared &s, const TileMeta &m, int R, uint32_t cbuf,
                                               LaneStream &ls, uint32_t *status) {
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncwarp();
    return tile_begin_ready(s, m, R, cbuf, ls, status);
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

// One step of the lane's stream: look up the next two codes and advance past
// them; returns the table entry (both exponents in BF16 position, or both
// palette indices, and the bits taken).  `lut` is the shared address of the
// pair table (kStrideShared), or of the lane's column of the private copies,
// i.e. their base + 4 * lane (kStridePrivate).  `I` is the step's index
// within the tile (a compile-time constant once the caller's 32-step loop is
// unrolled): after steps 2, 5, ..., 29 the window moves on by a word if the
// last three steps took it past one.
template <int kStride = kStrideShared>
__device__ __forceinline__ uint32_t decode_entry(LaneStream &ls, uint32_t lut, int I) {
    // window = ({hi:lo} >> c) & 1023; entry = table[window]; c += bits taken.
    // The refill's load is needed only three steps later, so it is off the
    // step-to-step dependency chain.
    uint32_t ent;
    asm volatile(
        "{\n\t"
        ".reg .b64 b;\n\t"
        ".reg .b32 w, t;\n\t"
        "mov.b64 b, {%1, %2};\n\t"
        "shr.b64 b, b, %3;\n\t"
        "cvt.u32.u64 w, b;\n\t"
        "and.b32 w, w, 1023;\n\t"
        "mad.lo.u32 w, w, %5, %4;\n\t"
        "ld.shared.u32 %0, [w];\n\t"
        "and.b32 t, %0, 15;\n\t"
        "add.u32 %3, %3, t;\n\t"
        "}"
        : "=r"(ent), "+r"(ls.lo), "+r"(ls.hi), "+r"(ls.c)
        : "r"(lut), "n"(kStride)
        : "memory");
    if ((I % 3) == 2 && I < 30) {
        asm volatile(
            "{\n\t"
            ".reg .pred p;\n\t"
            "setp.gt.u32 p, %3, 31;\n\t"
            "@p mov.b32 %0, %1;\n\t"
            "@p mov.b32 %1, %2;\n\t"
            "@p ld.shared.u32 %2, [%4];\n\t"
            "@p add.u32 %4, %4, 4;\n\t"
            "@p sub.u32 %3, %3, 32;\n\t"
            "}"
            : "+r"(ls.lo), "+r"(ls.hi), "+r"(ls.nx), "+r"(ls.c), "+r"(ls.wp)
            :
            : "memory");
    }
    return ent;
}

// decode_entry with the entry stride in a register (a lane may walk its own
// short list of entries with stride 4 instead of the table; see the batch-1
// GEMV's escaped groups), and the bit counter advanced by a multiply-add
// with `one` (1 held in a register), which runs on the FMA pipe instead of
// the half-rate ALU pipe that the shift and the masks already load.
__device__ __forceinline__ uint32_t decode_entry_rs(LaneStream &ls, uint32_t lut, uint32_t stride, uint32_t one,
                                                    int I) {
    uint32_t ent;
    asm volatile(
        "{\n\t"
        ".reg .b64 b;\n\t"
        ".reg .b32 w, t;\n\t"
        "mov.b64 b, {%1, %2};\n\t"
        "shr.b64 b, b, %3;\n\t"
        "cvt.u32.u64 w, b;\n\t"
        "and.b32 w, w, 1023;\n\t"
        "mad.lo.u32 w, w, %5, %4;\n\t"
        "ld.shared.u32 %0, [w];\n\t"
        "and.b32 t, %0, 15;\n\t"
        "mad.lo.u32 %3, t, %6, %3;\n\t"
        "}"
        : "=r"(ent), "+r"(ls.lo), "+r"(ls.hi), "+r"(ls.c)
        : "r"(lut), "r"(stride), "r"(one)
        : "memory");
    if ((I % 3) == 2 && I < 30) {
        asm volatile(
            "{\n\t"
            ".reg .pred p;\n\t"
            "setp.gt.u32 p, %3, 31;\n\t"
            "@p mov.b32 %0, %1;\n\t"
            "@p mov.b32 %1, %2;\n\t"
            "@p ld.shared.u32 %2, [%4];\n\t"
            "@p add.u32 %4, %4, 4;\n\t"
            "@p sub.u32 %3, %3, 32;\n\t"
            "}"
            : "+r"(ls.lo), "+r"(ls.hi), "+r"(ls.nx), "+r"(ls.c), "+r"(ls.wp)
            :
            : "memory");
    }
    return ent;
}

// One step: decode the exponents of weights 2i, 2i+1 and merge them with the
// sign+mantissa bytes.  `sm4` holds the bytes of weights 4*(i/2)..+3.  `I`
// is a compile-time constant once the caller's 32-step loop is unrolled.
template <int kStride = kStrideShared>
__device__ __forceinline__ uint32_t decode_pair(LaneStream &ls, uint32_t lut, int I, uint32_t sm4) {
    const uint32_t ent = decode_entry<kStride>(ls, lut, I);
    // sign-replicate byte permute: bytes (b0, sign(b0), b1, sign(b1)) for the
    // even pair of the word, (b2, sign(b2), b3, sign(b3)) for the odd one
    const uint32_t y = prmt(sm4, 0u, (I & 1) ? 0xB3A2u : 0x9180u);
    return lop3_merge(y, ent);
}

// After the 32 steps: every lane with codes must have used its byte length
// exactly (its last code ends in the length's final byte).
__device__ __forceinline__ void tile_check(const LaneStream &ls, uint32_t *status) {
    const uint32_t pos = 8u * ls.wp + ls.c;
    if (ls.expect != 0u && ls.expect - pos >= 8u)
        atomicOr(status, uint32_t(kStatusBadCode));
}

// The same check folded into a per-lane flag (nonzero: some group was bad);
// report it once with tile_check_flush.
__device__ __forceinline__ uint32_t tile_check_bits(const LaneStream &ls) {
    const uint32_t pos = 8u * ls.wp + ls.c;
    return (ls.expect != 0u) & (ls.expect - pos >= 8u);
}

__device__ __forceinline__ void tile_check_flush(uint32_t bad, uint32_t *status) {
    if (__any_sync(0xffffffffu, bad != 0u) && (threadIdx.x & 31) == 0)
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
