// Blob layout "UWB1" shared by the library's host and device code.
//
// Rows whose length is not a multiple of 64 are stored extended to the next
// multiple (stored_cols) with filler weights; the header's `cols` is the
// matrix's own column count and every section below is laid out for the
// stored width.
//
// A blob is position independent (offsets only) so the same bytes serve as
// the on-disk bundle, the host copy and the device copy.  All integers are
// little endian; every section starts at a multiple of 256 bytes.
//
//   header (256 bytes)            see HeaderField below
//   sm     rows*cols bytes        raw sign<<7 | mantissa of every weight
//   glen   n_groups bytes         code bytes of each group, 0 = escaped
//   tcode  u32[n_tiles+1]         tile code start, in 16-byte units
//   tesc   u32[n_tiles+1]         escaped groups in all earlier tiles
//   code   per tile: the byte-aligned codes of its groups, in row order,
//          padded with zeros to 16 bytes
//   esc    64 raw exponent bytes per escaped group, in group order
//
// Tiles: 32 rows x 64 columns.  Row block rb holds rows 32*rb .. (R rows,
// R = 32 except possibly in the last block); t = rb * (cols/64) + kg.
// Group order: q = 32*rb*(cols/64) + R*kg + j for row j of the block.
// sm byte of weight (32*rb + j, 64*kg + 16*c + b) sits at
// 32*rb*cols + 64*R*kg + (c*R + j)*16 + b: one 16-byte chunk per row and
// chunk index c, so that 32 lanes loading chunk c read 512 contiguous bytes.
//
// Codes: canonical, assigned in (length, palette index) order, at most
// kLmax = 5 bits so that a 10-bit window holds two codes.  Bit order: the
// code stream fills each byte from bit 0 up (stream bit i = bit i%8 of byte
// i/8), each code entering most significant bit first; read as 32-bit
// little-endian words, stream bit i is bit i%32 of word i/32.
#pragma once
#include <cstdint>

namespace uw {

constexpr uint32_t kMagic = 0x31425755u;  // "UWB1"
constexpr uint32_t kVersion = 2;  // 2: codes of at most 5 bits
constexpr int kGroup = 64;
constexpr int kTileRows = 32;
constexpr int kLmax = 5;
constexpr int kPalette = 16;
constexpr int kHeaderBytes = 256;
constexpr int kSectionAlign = 256;
constexpr int kMaxGroupCodeBytes = kGroup * kLmax / 8;            // 40
constexpr int kMaxTileCodeBytes = kTileRows * kMaxGroupCodeBytes;  // 1280 (multiple of 16)

namespace hdr {
constexpr int magic = 0, version = 4, rows = 8, cols = 16, group = 24, tile_rows = 28,
              lmax = 32, n_palette = 36, palette = 40, code_len = 56, n_groups = 72,
              n_escaped = 80, n_tiles = 88, code_bits = 96, off_sm = 104, off_glen = 112,
              off_tcode = 120, off_tesc = 128, off_code = 136, off_esc = 144,
              blob_bytes = 152;
}  // namespace hdr

inline uint64_t align_up(uint64_t v, uint64_t a) { return (v + a - 1) / a * a; }

// Columns a blob stores for rows of `cols` weights: the next multiple of the
// group (a ragged row is extended with filler weights; the header keeps
// `cols`).
constexpr int64_t stored_cols(int64_t cols) { return (cols + kGroup - 1) / kGroup * kGroup; }

}  // namespace uw
