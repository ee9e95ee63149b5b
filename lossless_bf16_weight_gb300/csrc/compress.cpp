// Host compressor: BF16 weight matrix -> UWB1 blob.
//
// Steps (Unweight blog, paragraphs on the BF16 layout, exponent skew,
// Huffman coding of the exponent byte and rows of 64 with rare exponents):
//   1. exponent histogram over the whole matrix;
//   2. palette = the 16 most frequent exponents (ties: smaller exponent);
//   3. a 64-weight group with an exponent outside the palette is escaped;
//   4. symbol frequencies over the coded groups;
//   5. minimum-redundancy code lengths under the limit kLmax, found by a
//      dynamic program over the levels of the code tree;
//   6. canonical codes in (length, palette index) order;
//   7. blob: raw sign+mantissa bytes, group byte lengths, tile offsets,
//      byte-aligned group codes (stream bits fill each byte from bit 0 up,
//      each code enters most significant bit first), raw exponents of
//      escaped groups.
// Every pass is parallel over rows or tiles with OpenMP; the result does not
// depend on the thread count.
#include <omp.h>

#include <algorithm>
#include <cstring>
#include <vector>

#include "format.h"
#include "uw.h"

namespace uw {
namespace {

struct Codebook {
    int npal = 0;
    uint8_t pal[kPalette] = {};
    uint8_t len[kPalette] = {};
    uint16_t code[kPalette] = {};
    int8_t sym_of[256];  // palette index of an exponent, -1 if absent
};

inline unsigned exponent_of(uint16_t b) { return (b >> 7) & 0xFFu; }
inline uint8_t sign_mantissa_of(uint16_t b) { return static_cast<uint8_t>(((b >> 8) & 0x80u) | (b & 0x7Fu)); }

// Minimum of sum_r f[r] * len[r] over monotone length assignments with
// lengths in [1, L], written as levels of a binary code tree.  With
// a_l = symbols given a length <= l, the cost is S(0) + sum_{l<L} S(a_l)
// where S(a) = f[a] + ... + f[m-1]: every symbol not yet placed at level l
// pays one more bit.  State (level, placed, free nodes at this level); free
// nodes beyond the symbols left change nothing, so they are capped there.
class LevelDP {
public:
    LevelDP(const std::vector<uint64_t> &ranked, int L) : m_(static_cast<int>(ranked.size())), L_(L) {
        S_.assign(m_ + 1, 0);
        for (int a = m_ - 1; a >= 0; a--)
            S_[a] = S_[a + 1] + ranked[a];
        memo_.assign((L_ + 2) * (m_ + 1) * (m_ + 1), kUnset);
    }

    // Counts (n_1..n_L) of an optimal code; among optimal codes the
    // lexicographically largest count vector.  Empty if none exists.
    std::vector<int> best_counts() {
        std::vector<int> counts;
        if (solve(1, 0, 2) == kInf)
            return counts;
        int a = 0;
        int64_t f = 2;
        for (int l = 1; l <= L_ && a < m_; l++) {
            const uint64_t target = solve(l, a, f);
            const int64_t cap = std::min<int64_t>(f, m_ - a);
            for (int64_t n = cap; n >= 0; n--) {
                if (take(l, a, f, static_cast<int>(n)) == target) {
                    counts.push_back(static_cast<int>(n));
                    a += static_cast<int>(n);
                    f = 2 * (f - n);
                    break;
                }
            }
        }
        return counts;
    }

private:
    static constexpr uint64_t kInf = ~0ull;
    static constexpr uint64_t kUnset = ~0ull - 1;

    // Cost of levels l.. when n of the remaining symbols get length l.
    uint64_t take(int l, int a, int64_t f, int n) {
        const int a2 = a + n;
        if (l == L_)
            return a2 == m_ ? 0 : kInf;
        const uint64_t rest = solve(l + 1, a2, 2 * (f - n));
        return rest == kInf ? kInf : rest + S_[a2];
    }

    uint64_t solve(int l, int a, int64_t f) {
        if (a == m_)
            return 0;
        if (l > L_ || f <= 0)
            return kInf;
        const int fc = static_cast<int>(std::min<int64_t>(f, m_ - a));
        uint64_t &slot = memo_[(l * (m_ + 1) + a) * (m_ + 1) + fc];
        if (slot != kUnset)
            return slot;
        uint64_t best = kInf;
        for (int n = fc; n >= 0; n--)
            best = std::min(best, take(l, a, fc, n));
        slot = best;
        return best;
    }

    int m_, L_;
    std::vector<uint64_t> S_;
    std::vector<uint64_t> memo_;
};

void choose_lengths(const uint64_t freq[kPalette], int npal, uint8_t len[kPalette]) {
    std::vector<int> order;
    for (int s = 0; s < npal; s++)
        if (freq[s] > 0)
            order.push_back(s);
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return freq[a] > freq[b]; });
    std::fill(len, len + kPalette, 0);
    if (order.empty())
        return;
    std::vector<uint64_t> ranked;
    for (int s : order)
        ranked.push_back(freq[s]);
    LevelDP dp(ranked, kLmax);
    std::vector<int> counts = dp.best_counts();
    size_t r = 0;
    for (size_t l = 0; l < counts.size(); l++)
        for (int c = 0; c < counts[l]; c++)
            len[order[r++]] = static_cast<uint8_t>(l + 1);
}

// Canonical code values: count codes per length, first value per length,
// then hand out values in palette-index order within each length.
void canonical_codes(const uint8_t len[kPalette], uint16_t code[kPalette]) {
    int per_len[kLmax + 2] = {};
    for (int s = 0; s < kPalette; s++)
        per_len[len[s]]++;
    per_len[0] = 0;
    uint32_t next[kLmax + 2] = {};
    uint32_t c = 0;
    for (int l = 1; l <= kLmax; l++) {
        c = (c + per_len[l - 1]) << 1;
        next[l] = c;
    }
    for (int s = 0; s < kPalette; s++)
        code[s] = len[s] ? static_cast<uint16_t>(next[len[s]]++) : 0;
}

// Bit packer for one group: stream bit i goes to bit i%8 of byte i/8, and
// each code enters the stream most significant bit first, so the code is
// appended bit-reversed to a little-endian accumulator.  Returns the bits.
int pack_group(const uint16_t *w, const Codebook &cb, uint8_t *out /* >= 48 bytes */) {
    uint64_t acc = 0;
    int pending = 0, bits = 0, pos = 0;
    for (int i = 0; i < kGroup; i++) {
        const int s = cb.sym_of[exponent_of(w[i])];
        const int l = cb.len[s];
        uint32_t rev = 0;
        for (int b = 0; b < l; b++)
            rev |= ((cb.code[s] >> b) & 1u) << (l - 1 - b);
        acc |= uint64_t(rev) << pending;
        pending += l;
        bits += l;
        while (pending >= 8) {
            out[pos++] = static_cast<uint8_t>(acc & 0xFFu);
            acc >>= 8;
            pending -= 8;
        }
    }
    if (pending)
        out[pos++] = static_cast<uint8_t>(acc & 0xFFu);
    return bits;
}

int group_bits(const uint16_t *w, const Codebook &cb) {
    int bits = 0;
    for (int i = 0; i < kGroup; i++)
        bits += cb.len[cb.sym_of[exponent_of(w[i])]];
    return bits;
}

void put32(uint8_t *p, uint32_t v) { std::memcpy(p, &v, 4); }
void put64(uint8_t *p, uint64_t v) { std::memcpy(p, &v, 8); }

}  // namespace
}  // namespace uw

extern "C" uw_status uw_compress(const uint16_t *w, int64_t rows, int64_t cols, void *blob_out,
                                 size_t *blob_bytes) {
    using namespace uw;
    if (!w || !blob_bytes)
        return UW_ERR_INVALID_ARG;
    if (rows <= 0 || cols <= 0)
        return UW_ERR_SHAPE;
    if (rows > (int64_t(1) << 31) || cols > (int64_t(1) << 31))
        return UW_ERR_UNSUPPORTED;  // the blob descriptor's limit (no size product can wrap)
    // A row whose length is not a multiple of 64 is stored extended to the
    // next multiple with filler weights (sign and mantissa 0, exponent the
    // first palette exponent below 255, else 0); the palette is chosen from
    // the matrix's own weights and the header keeps the true column count.
    const int64_t cols_true = cols;
    cols = stored_cols(cols);
    const int64_t gpr = cols / kGroup;
    const int64_t nrb = (rows + kTileRows - 1) / kTileRows;
    const int64_t ntiles = nrb * gpr;
    const int64_t ngroups = rows * gpr;
    if (ntiles >= (1ll << 31) || rows * cols / 16 >= (1ll << 32))
        return UW_ERR_UNSUPPORTED;  // tile offsets are u32

    // 1. histogram
    uint64_t hist[256] = {};
#pragma omp parallel
    {
        uint64_t local[256] = {};
#pragma omp for schedule(static)
        for (int64_t n = 0; n < rows; n++) {
            const uint16_t *r = w + n * cols_true;
            for (int64_t k = 0; k < cols_true; k++)
                local[exponent_of(r[k])]++;
        }
#pragma omp critical
        for (int v = 0; v < 256; v++)
            hist[v] += local[v];
    }

    // 2. palette
    Codebook cb;
    {
        std::vector<int> ex(256);
        for (int v = 0; v < 256; v++)
            ex[v] = v;
        std::stable_sort(ex.begin(), ex.end(), [&](int a, int b) { return hist[a] > hist[b]; });
        std::memset(cb.sym_of, -1, sizeof cb.sym_of);
        for (int i = 0; i < kPalette && hist[ex[i]] > 0; i++) {
            cb.pal[cb.npal] = static_cast<uint8_t>(ex[i]);
            cb.sym_of[ex[i]] = static_cast<int8_t>(cb.npal);
            cb.npal++;
        }
    }

    // the extended matrix, when the rows are ragged
    std::vector<uint16_t> extended;
    if (cols != cols_true) {
        uint16_t filler = 0;
        for (int i = 0; i < cb.npal; i++)
            if (cb.pal[i] != 255) {
                filler = static_cast<uint16_t>(cb.pal[i] << 7);
                break;
            }
        extended.resize(size_t(rows) * size_t(cols));
#pragma omp parallel for schedule(static)
        for (int64_t n = 0; n < rows; n++)
            for (int64_t k = 0; k < cols; k++)
                extended[size_t(n) * cols + k] = k < cols_true ? w[n * cols_true + k] : filler;
        w = extended.data();
    }

    // 3-4. escaped groups and symbol frequencies of the coded ones
    std::vector<uint8_t> escaped(ngroups);
    uint64_t freq[kPalette] = {};
#pragma omp parallel
    {
        uint64_t local[kPalette] = {};
#pragma omp for schedule(static)
        for (int64_t g = 0; g < ngroups; g++) {
            const uint16_t *p = w + (g / gpr) * cols + (g % gpr) * kGroup;
            uint64_t cnt[kPalette] = {};
            bool esc = false;
            for (int i = 0; i < kGroup; i++) {
                const int s = cb.sym_of[exponent_of(p[i])];
                if (s < 0) {
                    esc = true;
                    break;
                }
                cnt[s]++;
            }
            escaped[g] = esc;
            if (!esc)
                for (int s = 0; s < kPalette; s++)
                    local[s] += cnt[s];
        }
#pragma omp critical
        for (int s = 0; s < kPalette; s++)
            freq[s] += local[s];
    }

    // 5-6. code
    choose_lengths(freq, cb.npal, cb.len);
    canonical_codes(cb.len, cb.code);

    // Group byte lengths and per-tile sizes.
    std::vector<uint8_t> glen(ngroups);
    std::vector<uint32_t> tile_bytes(ntiles), tile_esc(ntiles);
    std::vector<uint64_t> tile_bits(ntiles);
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < ntiles; t++) {
        const int64_t rb = t / gpr, kg = t % gpr;
        const int64_t R = std::min<int64_t>(kTileRows, rows - rb * kTileRows);
        uint32_t bytes = 0, nesc = 0;
        uint64_t bits = 0;
        for (int64_t j = 0; j < R; j++) {
            const int64_t n = rb * kTileRows + j;
            const int64_t q = kTileRows * rb * gpr + R * kg + j;
            if (escaped[n * gpr + kg]) {
                glen[q] = 0;
                nesc++;
                continue;
            }
            const int b = group_bits(w + n * cols + kg * kGroup, cb);
            bits += b;
            glen[q] = static_cast<uint8_t>((b + 7) / 8);
            bytes += glen[q];
        }
        tile_bytes[t] = (bytes + 15) / 16;
        tile_esc[t] = nesc;
        tile_bits[t] = bits;
    }
    std::vector<uint32_t> tcode(ntiles + 1), tesc(ntiles + 1);
    uint64_t code16 = 0, nesc = 0, code_bits = 0;
    for (int64_t t = 0; t < ntiles; t++) {
        tcode[t] = static_cast<uint32_t>(code16);
        tesc[t] = static_cast<uint32_t>(nesc);
        code16 += tile_bytes[t];
        nesc += tile_esc[t];
        code_bits += tile_bits[t];
    }
    if (code16 >= (1ull << 32))
        return UW_ERR_UNSUPPORTED;
    tcode[ntiles] = static_cast<uint32_t>(code16);
    tesc[ntiles] = static_cast<uint32_t>(nesc);

    const uint64_t off_sm = kHeaderBytes;
    const uint64_t off_glen = align_up(off_sm + rows * cols, kSectionAlign);
    const uint64_t off_tcode = align_up(off_glen + ngroups, kSectionAlign);
    const uint64_t off_tesc = align_up(off_tcode + 4 * (ntiles + 1), kSectionAlign);
    const uint64_t off_code = align_up(off_tesc + 4 * (ntiles + 1), kSectionAlign);
    const uint64_t off_esc = align_up(off_code + 16 * code16, kSectionAlign);
    const uint64_t total = align_up(off_esc + 64 * nesc, kSectionAlign);

    if (!blob_out || *blob_bytes < total) {
        *blob_bytes = total;
        return UW_ERR_BUFFER_TOO_SMALL;
    }
    *blob_bytes = total;
    uint8_t *blob = static_cast<uint8_t *>(blob_out);

    uint8_t *h = blob;
    std::memset(h, 0, kHeaderBytes);
    put32(h + hdr::magic, kMagic);
    put32(h + hdr::version, kVersion);
    put64(h + hdr::rows, rows);
    put64(h + hdr::cols, cols_true);
    put32(h + hdr::group, kGroup);
    put32(h + hdr::tile_rows, kTileRows);
    put32(h + hdr::lmax, kLmax);
    put32(h + hdr::n_palette, cb.npal);
    std::memcpy(h + hdr::palette, cb.pal, kPalette);
    std::memcpy(h + hdr::code_len, cb.len, kPalette);
    put64(h + hdr::n_groups, ngroups);
    put64(h + hdr::n_escaped, nesc);
    put64(h + hdr::n_tiles, ntiles);
    put64(h + hdr::code_bits, code_bits);
    put64(h + hdr::off_sm, off_sm);
    put64(h + hdr::off_glen, off_glen);
    put64(h + hdr::off_tcode, off_tcode);
    put64(h + hdr::off_tesc, off_tesc);
    put64(h + hdr::off_code, off_code);
    put64(h + hdr::off_esc, off_esc);
    put64(h + hdr::blob_bytes, total);

    // Zero the gaps between sections (padding bytes are part of the format).
    std::memset(blob + off_sm + rows * cols, 0, off_glen - off_sm - rows * cols);
    std::memset(blob + off_glen + ngroups, 0, off_tcode - off_glen - ngroups);
    std::memset(blob + off_tcode, 0, off_code - off_tcode);
    std::memset(blob + off_code + 16 * code16, 0, off_esc - off_code - 16 * code16);
    std::memset(blob + off_esc, 0, total - off_esc);
    std::memcpy(blob + off_glen, glen.data(), ngroups);
    std::memcpy(blob + off_tcode, tcode.data(), 4 * (ntiles + 1));
    std::memcpy(blob + off_tesc, tesc.data(), 4 * (ntiles + 1));

#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < ntiles; t++) {
        const int64_t rb = t / gpr, kg = t % gpr;
        const int64_t R = std::min<int64_t>(kTileRows, rows - rb * kTileRows);
        uint8_t *sm_tile = blob + off_sm + kTileRows * rb * cols + kGroup * R * kg;
        uint8_t *code = blob + off_code + 16ull * tcode[t];
        uint8_t *code_end = blob + off_code + 16ull * tcode[t + 1];
        uint8_t *esc = blob + off_esc + 64ull * tesc[t];
        for (int64_t j = 0; j < R; j++) {
            const int64_t n = rb * kTileRows + j;
            const uint16_t *g = w + n * cols + kg * kGroup;
            for (int c = 0; c < 4; c++)
                for (int b = 0; b < 16; b++)
                    sm_tile[(c * R + j) * 16 + b] = sign_mantissa_of(g[16 * c + b]);
            if (escaped[n * gpr + kg]) {
                for (int i = 0; i < kGroup; i++)
                    esc[i] = static_cast<uint8_t>(exponent_of(g[i]));
                esc += 64;
            } else {
                uint8_t buf[kMaxGroupCodeBytes + 8];
                const int bits = pack_group(g, cb, buf);
                const int nb = (bits + 7) / 8;
                std::memcpy(code, buf, nb);
                code += nb;
            }
        }
        std::memset(code, 0, code_end - code);
    }
    return UW_OK;
}
