/*
 * uw_oracle.c -- plain, slow, single-threaded reference implementation of
 * Unweight-style lossless BF16 weight compression.
 *
 * TEST INFRASTRUCTURE ONLY.  This file exists to check the CUDA library.
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load it.  It shares no code, header, table or constant generator with the
 * library; the blob layout it writes and reads is restated here from the
 * format description, not included from the library.
 *
 * Source of every step: the Unweight blog post ("Unweight: how we compressed
 * an LLM 22% without sacrificing quality", Cloudflare; the text used here is
 * its Russian translation).  The page has no headings, so citations name the
 * paragraph by its topic:
 *   [BF16]      a BF16 value is 1 sign bit, 8 exponent bits, 7 mantissa bits.
 *   [RANDOM]    sign and mantissa look random and are left uncompressed.
 *   [SKEW]      a handful of the 256 exponent values dominate; the 16 most
 *               common cover >99% of a layer, about 2.6 bits of entropy.
 *   [HUFFMAN]   only the exponent byte is Huffman coded (short codes for
 *               common values); sign and mantissa are untouched.
 *   [ROWS64]    if any weight in a row of 64 has an exponent outside the
 *               top-16 palette, the whole row is stored in original form:
 *               one decision per row, no per-element branch.
 *   [LUT16K]    the decoder keeps a ~16 KB Huffman lookup table in SMEM.
 *   [MATMUL]    the compressed weights feed y = x W^T (decode once, multiply).
 *   [EXPONENT]  the exponent-only pipeline: only the exponent bytes are
 *               decoded to memory, and the matmul merges them with the raw
 *               sign+mantissa bytes (paragraph on the four execution
 *               pipelines).
 *   [PALETTE]   the palette pipelines: Huffman-coded exponents turned into
 *               4-bit palette indices (at run time or once at model load),
 *               from which the matmul rebuilds BF16 on the fly (paragraphs
 *               on the four execution pipelines and on the palette format
 *               at model load).
 *
 * Readings taken where the page is silent:
 *   - "row of 64" = 64 consecutive weights along K inside one output row.
 *   - the Huffman alphabet is the palette (<=16 symbols); escaped groups are
 *     outside the code and keep their 64 raw exponent bytes.
 *   - palette = 16 most frequent exponents over the whole matrix, ties to the
 *     smaller exponent value; exponents with zero count are never included.
 *   - one code per matrix; code length limit LMAX = 5 so that a 10-bit window
 *     always holds two whole codes (a 1024-entry pair table; the page's own
 *     table is about 16 KB, sized for its hardware).
 *   - among equally short codes, pick the lexicographically largest count
 *     vector (n_1, ..., n_LMAX), symbols ranked by (frequency desc, palette
 *     index asc); canonical code values by (length, palette index).
 *   - bit order: the code stream fills each byte from its least significant
 *     bit up (stream bit i is bit i%8 of byte i/8, the convention of
 *     DEFLATE); each code enters the stream most significant code bit
 *     first; each group starts on a byte boundary.
 *   - a row whose length is not a multiple of 64 (the page's matrices all
 *     are) is extended to the next multiple with filler weights: sign and
 *     mantissa 0, exponent = the first palette exponent below 255 (a
 *     finite weight, in the palette, so the last group is escaped only if
 *     its own weights force it), or 0 when the palette has none.  The
 *     palette is chosen from the matrix's own weights; everything after it
 *     (escape flags, code lengths, encoding) runs on the extended matrix.
 *     The header keeps the true column count; the sections are laid out
 *     for the extended one.
 *
 * The fp64 matrix product is the plain definition y[b,n] = sum_k x[b,k] W[n,k].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define UWO_GROUP 64      /* weights per group ("row of 64")         */
#define UWO_TROWS 32      /* rows per tile (one lane per row)        */
#define UWO_LMAX 5        /* longest code                             */
#define UWO_PAL 16        /* palette size                             */
#define UWO_MAGIC 0x31425755u /* "UWB1" little endian                 */
#define UWO_VERSION 2u
#define UWO_HEADER 256

/* ------------------------------------------------------------------------
 * [BF16] field split and join.
 * sign = bit 15, exponent = bits 14..7, mantissa = bits 6..0.
 * The raw sign+mantissa byte is sign<<7 | mantissa ([RANDOM], [HUFFMAN]).
 * --------------------------------------------------------------------- */
unsigned uwo_exponent(uint16_t b) { return (b >> 7) & 0xFFu; }
unsigned uwo_sign(uint16_t b) { return (b >> 15) & 1u; }
unsigned uwo_mantissa(uint16_t b) { return b & 0x7Fu; }
unsigned uwo_sm_byte(uint16_t b) { return (uwo_sign(b) << 7) | uwo_mantissa(b); }

uint16_t uwo_join(unsigned e, unsigned sm)
{
    unsigned sign = (sm >> 7) & 1u;
    unsigned mant = sm & 0x7Fu;
    return (uint16_t)((sign << 15) | ((e & 0xFFu) << 7) | mant);
}

void uwo_split(const uint16_t *w, int64_t n, uint8_t *e, uint8_t *sm)
{
    for (int64_t i = 0; i < n; i++) {
        e[i] = (uint8_t)uwo_exponent(w[i]);
        sm[i] = (uint8_t)uwo_sm_byte(w[i]);
    }
}

/* [SKEW] exponent histogram over every weight of the matrix. */
void uwo_histogram(const uint16_t *w, int64_t n, uint64_t count[256])
{
    for (int v = 0; v < 256; v++)
        count[v] = 0;
    for (int64_t i = 0; i < n; i++)
        count[uwo_exponent(w[i])] += 1;
}

/* [SKEW], [ROWS64] palette: repeatedly take the most frequent exponent not
 * yet taken (ties: smaller exponent), at most 16, never a zero count.
 * Returns the palette size. */
int uwo_palette(const uint64_t count[256], uint8_t palette[UWO_PAL])
{
    int taken[256] = {0};
    int n = 0;
    while (n < UWO_PAL) {
        int best = -1;
        for (int v = 0; v < 256; v++) {
            if (taken[v] || count[v] == 0)
                continue;
            if (best < 0 || count[v] > count[best])
                best = v; /* strict '>' keeps the smaller value on ties */
        }
        if (best < 0)
            break;
        taken[best] = 1;
        palette[n++] = (uint8_t)best;
    }
    for (int i = n; i < UWO_PAL; i++)
        palette[i] = 0;
    return n;
}

/* Palette index of exponent e, or -1 if e is not in the palette. */
static int palette_index(const uint8_t *palette, int npal, unsigned e)
{
    for (int i = 0; i < npal; i++)
        if (palette[i] == e)
            return i;
    return -1;
}

/* [ROWS64] a group (row n, weights k = 64*kg .. 64*kg+63) is escaped iff one
 * of its exponents is outside the palette.  flags[n*(cols/64)+kg]. */
void uwo_escape_flags(const uint16_t *w, int64_t rows, int64_t cols,
                      const uint8_t *palette, int npal, uint8_t *flags)
{
    int64_t gpr = cols / UWO_GROUP;
    for (int64_t n = 0; n < rows; n++)
        for (int64_t kg = 0; kg < gpr; kg++) {
            int esc = 0;
            for (int i = 0; i < UWO_GROUP; i++) {
                unsigned e = uwo_exponent(w[n * cols + kg * UWO_GROUP + i]);
                if (palette_index(palette, npal, e) < 0)
                    esc = 1;
            }
            flags[n * gpr + kg] = (uint8_t)esc;
        }
}

/* ------------------------------------------------------------------------
 * [HUFFMAN] minimum-redundancy code lengths under the limit lmax.
 * Definition: minimise sum_s freq[s]*len[s] over 1 <= len[s] <= lmax with
 * sum_s 2^-len[s] <= 1 (Kraft), over the symbols with freq > 0.  A minimiser
 * gives longer codes only to less frequent symbols, so it is described by the
 * counts (n_1..n_lmax) handed out to the symbols in rank order (frequency
 * desc, palette index asc).  This function tries every count vector: obviously
 * correct, and cheap for 16 symbols.  Ties: the first vector met in
 * lexicographically descending order of (n_1, n_2, ...) wins.
 * Symbols with freq 0 get length 0 (no code).  Returns the number of coded
 * symbols.
 * --------------------------------------------------------------------- */
struct lsearch {
    int m, lmax;
    uint64_t f[UWO_PAL];     /* ranked frequencies               */
    int counts[16];          /* counts at levels 1..lmax (index l-1) */
    int best_counts[16];
    double best_cost;        /* exact for counts < 2^53            */
    int have_best;
};

static void lsearch_rec(struct lsearch *S, int level, int assigned, int64_t free_nodes)
{
    if (assigned == S->m) {
        /* cost of this count vector */
        double cost = 0.0;
        int r = 0;
        for (int l = 1; l < level; l++)
            for (int c = 0; c < S->counts[l - 1]; c++)
                cost += (double)S->f[r++] * l;
        if (!S->have_best || cost < S->best_cost) {
            S->have_best = 1;
            S->best_cost = cost;
            for (int l = 0; l < 16; l++)
                S->best_counts[l] = l < level - 1 ? S->counts[l] : 0;
        }
        return;
    }
    if (level > S->lmax)
        return;
    int left = S->m - assigned;
    int64_t hi = free_nodes < left ? free_nodes : left;
    for (int64_t c = hi; c >= 0; c--) {
        S->counts[level - 1] = (int)c;
        lsearch_rec(S, level + 1, assigned + (int)c, 2 * (free_nodes - c));
    }
    S->counts[level - 1] = 0;
}

int uwo_code_lengths(const uint64_t *freq, int nsym, int lmax, uint8_t *len)
{
    struct lsearch S;
    int rank[UWO_PAL];
    memset(&S, 0, sizeof S);
    S.lmax = lmax;
    /* rank symbols: frequency desc, index asc (selection, plain) */
    int used[UWO_PAL] = {0};
    for (;;) {
        int best = -1;
        for (int s = 0; s < nsym; s++) {
            if (used[s] || freq[s] == 0)
                continue;
            if (best < 0 || freq[s] > freq[best])
                best = s;
        }
        if (best < 0)
            break;
        used[best] = 1;
        rank[S.m] = best;
        S.f[S.m] = freq[best];
        S.m++;
    }
    for (int s = 0; s < nsym; s++)
        len[s] = 0;
    if (S.m == 0)
        return 0;
    lsearch_rec(&S, 1, 0, 2);
    if (!S.have_best)
        return -1; /* more symbols than 2^lmax */
    int r = 0;
    for (int l = 1; l <= lmax; l++)
        for (int c = 0; c < S.best_counts[l - 1]; c++)
            len[rank[r++]] = (uint8_t)l;
    return S.m;
}

/* Canonical code values: symbols with a code, in (length, index) order;
 * the first gets 0, each next one (previous + 1) << (length difference). */
void uwo_canonical_codes(const uint8_t *len, int nsym, uint16_t *code)
{
    uint32_t c = 0;
    int prev_len = 0, any = 0;
    for (int s = 0; s < nsym; s++)
        code[s] = 0;
    for (int l = 1; l <= 15; l++)
        for (int s = 0; s < nsym; s++) {
            if (len[s] != l)
                continue;
            if (any)
                c = (c + 1) << (l - prev_len);
            else
                c = 0;
            code[s] = (uint16_t)c;
            prev_len = l;
            any = 1;
        }
}

/* ------------------------------------------------------------------------
 * Blob layout (format UWB1; the library writes the same bytes).
 *   tiles: row block rb (32 rows, the last may be shorter: R rows),
 *          group column kg;  t = rb*(cols/64) + kg.
 *   group order q (used by glen and esc): q = 32*rb*(cols/64) + R*kg + j,
 *          j = row inside the block.
 *   sm:    byte of weight (32*rb + j, 64*kg + 16*c + b) at
 *          32*rb*cols + 64*R*kg + (c*R + j)*16 + b.
 *   glen:  u8 per group, code bytes of the group, 0 = escaped.
 *   tcode: u32[n_tiles+1], start of tile t's code bytes in 16-byte units.
 *   code:  per tile, the codes of its groups in row order, each group
 *          byte aligned, then zero padding to 16 bytes.
 *   tesc:  u32[n_tiles+1], escaped groups in tiles before t.
 *   esc:   64 raw exponent bytes per escaped group, in group order.
 *   Sections start at multiples of 256 bytes.
 * --------------------------------------------------------------------- */
static uint64_t align_up(uint64_t v, uint64_t a) { return (v + a - 1) / a * a; }

static void put_u32(uint8_t *p, uint32_t v)
{
    for (int i = 0; i < 4; i++)
        p[i] = (uint8_t)(v >> (8 * i));
}
static void put_u64(uint8_t *p, uint64_t v)
{
    for (int i = 0; i < 8; i++)
        p[i] = (uint8_t)(v >> (8 * i));
}
static uint32_t get_u32(const uint8_t *p)
{
    uint32_t v = 0;
    for (int i = 0; i < 4; i++)
        v |= (uint32_t)p[i] << (8 * i);
    return v;
}
static uint64_t get_u64(const uint8_t *p)
{
    uint64_t v = 0;
    for (int i = 0; i < 8; i++)
        v |= (uint64_t)p[i] << (8 * i);
    return v;
}

/* Code bits of one group (symbols s[0..63]) into out[48], each code most
 * significant bit first, stream bit i stored as bit i%8 of byte i/8;
 * returns the number of bits. */
static int encode_group(const int *sym, const uint8_t *len, const uint16_t *code, uint8_t *out)
{
    int bit = 0;
    memset(out, 0, 48);
    for (int i = 0; i < UWO_GROUP; i++) {
        int l = len[sym[i]];
        for (int b = l - 1; b >= 0; b--) {
            unsigned v = (code[sym[i]] >> b) & 1u;
            out[bit / 8] |= (uint8_t)(v << (bit % 8));
            bit++;
        }
    }
    return bit;
}

/* Header fields the oracle reports back to its caller. */
typedef struct {
    int64_t rows, cols;
    int64_t n_groups, n_escaped, n_tiles;
    int64_t code_bits, blob_bytes;
    int32_t n_palette, lmax;
    uint8_t palette[16], code_len[16];
    uint64_t off_sm, off_glen, off_tcode, off_tesc, off_code, off_esc;
} uwo_info;

/* Stored columns: cols rounded up to a whole number of groups. */
int64_t uwo_stored_cols(int64_t cols) { return (cols + UWO_GROUP - 1) / UWO_GROUP * UWO_GROUP; }

/* The filler weight of a matrix with this palette: sign and mantissa 0,
 * exponent the first palette entry below 255, else 0. */
uint16_t uwo_filler(const uint8_t *palette, int npal)
{
    for (int s = 0; s < npal; s++)
        if (palette[s] != 255)
            return (uint16_t)((unsigned)palette[s] << 7);
    return 0;
}

/* W [rows, cols] extended to [rows, uwo_stored_cols(cols)] with the filler
 * weight of the palette (out: rows * stored columns values). */
void uwo_pad(const uint16_t *w, int64_t rows, int64_t cols, const uint8_t *palette, int npal, uint16_t *out)
{
    int64_t cp = uwo_stored_cols(cols);
    uint16_t f = uwo_filler(palette, npal);
    for (int64_t n = 0; n < rows; n++)
        for (int64_t k = 0; k < cp; k++)
            out[n * cp + k] = k < cols ? w[n * cols + k] : f;
}

/* Compress W [rows, cols] (row-major bf16 bits).  If len_override is not
 * NULL its 16 code lengths are used instead of the optimum (the caller must
 * pass a valid prefix code).  Writes the blob when blob != NULL and
 * cap is large enough.  Returns the blob size, or a negative error:
 * -1 bad shape, -2 bad override, -3 out of memory. */
int64_t uwo_compress(const uint16_t *w, int64_t rows, int64_t cols,
                     const uint8_t *len_override, uint8_t *blob, int64_t cap,
                     uwo_info *info)
{
    if (rows <= 0 || cols <= 0)
        return -1;
    const int64_t cols_true = cols;
    uint64_t count[256];
    uint8_t palette[UWO_PAL];
    uwo_histogram(w, rows * cols, count);
    int npal = uwo_palette(count, palette);

    /* a ragged row length: the rest of the encoder runs on the extended matrix */
    uint16_t *padded = NULL;
    if (cols % UWO_GROUP != 0) {
        padded = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)(rows * uwo_stored_cols(cols)));
        if (!padded)
            return -3;
        uwo_pad(w, rows, cols, palette, npal, padded);
        w = padded;
        cols = uwo_stored_cols(cols);
    }
    int64_t gpr = cols / UWO_GROUP;
    int64_t nrb = (rows + UWO_TROWS - 1) / UWO_TROWS;
    int64_t ntiles = nrb * gpr;
    int64_t ngroups = rows * gpr;

    uint8_t *esc = (uint8_t *)malloc((size_t)ngroups);
    if (!esc) {
        free(padded);
        return -3;
    }
    uwo_escape_flags(w, rows, cols, palette, npal, esc);

    /* symbol frequencies over the groups that are coded */
    uint64_t freq[UWO_PAL] = {0};
    int64_t nesc = 0;
    for (int64_t n = 0; n < rows; n++)
        for (int64_t kg = 0; kg < gpr; kg++) {
            if (esc[n * gpr + kg]) {
                nesc++;
                continue;
            }
            for (int i = 0; i < UWO_GROUP; i++) {
                unsigned e = uwo_exponent(w[n * cols + kg * UWO_GROUP + i]);
                freq[palette_index(palette, npal, e)] += 1;
            }
        }

    uint8_t len[UWO_PAL] = {0};
    if (len_override) {
        double kraft = 0.0;
        for (int s = 0; s < UWO_PAL; s++) {
            len[s] = len_override[s];
            if (len[s] > UWO_LMAX || (s >= npal && len[s]) || (freq[s] && !len[s])) {
                free(esc);
                free(padded);
                return -2;
            }
            if (len[s])
                kraft += ldexp(1.0, -len[s]);
        }
        if (kraft > 1.0) {
            free(esc);
            free(padded);
            return -2;
        }
    } else {
        uwo_code_lengths(freq, npal, UWO_LMAX, len);
    }
    uint16_t code[UWO_PAL];
    uwo_canonical_codes(len, UWO_PAL, code);

    /* Pass 1: group byte lengths, tile code sizes. */
    uint8_t *glen = (uint8_t *)malloc((size_t)ngroups);
    uint32_t *tcode = (uint32_t *)malloc(sizeof(uint32_t) * (size_t)(ntiles + 1));
    uint32_t *tesc = (uint32_t *)malloc(sizeof(uint32_t) * (size_t)(ntiles + 1));
    if (!glen || !tcode || !tesc) {
        free(esc); free(glen); free(tcode); free(tesc); free(padded);
        return -3;
    }
    int64_t code_bits = 0, code16 = 0, escs = 0;
    int sym[UWO_GROUP];
    uint8_t gbuf[48];
    for (int64_t rb = 0; rb < nrb; rb++) {
        int64_t R = rows - rb * UWO_TROWS < UWO_TROWS ? rows - rb * UWO_TROWS : UWO_TROWS;
        for (int64_t kg = 0; kg < gpr; kg++) {
            int64_t t = rb * gpr + kg;
            int64_t tbytes = 0;
            tcode[t] = (uint32_t)code16;
            tesc[t] = (uint32_t)escs;
            for (int64_t j = 0; j < R; j++) {
                int64_t n = rb * UWO_TROWS + j;
                int64_t q = UWO_TROWS * rb * gpr + R * kg + j;
                if (esc[n * gpr + kg]) {
                    glen[q] = 0;
                    escs++;
                    continue;
                }
                for (int i = 0; i < UWO_GROUP; i++)
                    sym[i] = palette_index(palette, npal, uwo_exponent(w[n * cols + kg * UWO_GROUP + i]));
                int bits = encode_group(sym, len, code, gbuf);
                code_bits += bits;
                glen[q] = (uint8_t)((bits + 7) / 8);
                tbytes += glen[q];
            }
            code16 += (tbytes + 15) / 16;
        }
    }
    tcode[ntiles] = (uint32_t)code16;
    tesc[ntiles] = (uint32_t)escs;

    uint64_t off_sm = UWO_HEADER;
    uint64_t off_glen = align_up(off_sm + (uint64_t)(rows * cols), 256);
    uint64_t off_tcode = align_up(off_glen + (uint64_t)ngroups, 256);
    uint64_t off_tesc = align_up(off_tcode + 4 * (uint64_t)(ntiles + 1), 256);
    uint64_t off_code = align_up(off_tesc + 4 * (uint64_t)(ntiles + 1), 256);
    uint64_t off_esc = align_up(off_code + 16 * (uint64_t)code16, 256);
    uint64_t total = align_up(off_esc + 64 * (uint64_t)nesc, 256);

    if (info) {
        memset(info, 0, sizeof *info);
        info->rows = rows;
        info->cols = cols_true;
        info->n_groups = ngroups;
        info->n_escaped = nesc;
        info->n_tiles = ntiles;
        info->code_bits = code_bits;
        info->blob_bytes = (int64_t)total;
        info->n_palette = npal;
        info->lmax = UWO_LMAX;
        memcpy(info->palette, palette, 16);
        memcpy(info->code_len, len, 16);
        info->off_sm = off_sm;
        info->off_glen = off_glen;
        info->off_tcode = off_tcode;
        info->off_tesc = off_tesc;
        info->off_code = off_code;
        info->off_esc = off_esc;
    }

    if (blob && cap >= (int64_t)total) {
        memset(blob, 0, (size_t)total);
        put_u32(blob + 0, UWO_MAGIC);
        put_u32(blob + 4, UWO_VERSION);
        put_u64(blob + 8, (uint64_t)rows);
        put_u64(blob + 16, (uint64_t)cols_true);
        put_u32(blob + 24, UWO_GROUP);
        put_u32(blob + 28, UWO_TROWS);
        put_u32(blob + 32, UWO_LMAX);
        put_u32(blob + 36, (uint32_t)npal);
        memcpy(blob + 40, palette, 16);
        memcpy(blob + 56, len, 16);
        put_u64(blob + 72, (uint64_t)ngroups);
        put_u64(blob + 80, (uint64_t)nesc);
        put_u64(blob + 88, (uint64_t)ntiles);
        put_u64(blob + 96, (uint64_t)code_bits);
        put_u64(blob + 104, off_sm);
        put_u64(blob + 112, off_glen);
        put_u64(blob + 120, off_tcode);
        put_u64(blob + 128, off_tesc);
        put_u64(blob + 136, off_code);
        put_u64(blob + 144, off_esc);
        put_u64(blob + 152, total);

        for (int64_t t = 0; t <= ntiles; t++) {
            put_u32(blob + off_tcode + 4 * t, tcode[t]);
            put_u32(blob + off_tesc + 4 * t, tesc[t]);
        }
        memcpy(blob + off_glen, glen, (size_t)ngroups);

        /* Pass 2: sign+mantissa, codes, escapes. */
        for (int64_t rb = 0; rb < nrb; rb++) {
            int64_t R = rows - rb * UWO_TROWS < UWO_TROWS ? rows - rb * UWO_TROWS : UWO_TROWS;
            for (int64_t kg = 0; kg < gpr; kg++) {
                int64_t t = rb * gpr + kg;
                uint64_t cpos = off_code + 16 * (uint64_t)tcode[t];
                uint64_t epos = off_esc + 64 * (uint64_t)tesc[t];
                for (int64_t j = 0; j < R; j++) {
                    int64_t n = rb * UWO_TROWS + j;
                    int64_t q = UWO_TROWS * rb * gpr + R * kg + j;
                    const uint16_t *g = w + n * cols + kg * UWO_GROUP;
                    for (int c = 0; c < 4; c++)
                        for (int b = 0; b < 16; b++) {
                            uint64_t at = off_sm + (uint64_t)(UWO_TROWS * rb * cols + 64 * R * kg + (c * R + j) * 16 + b);
                            blob[at] = (uint8_t)uwo_sm_byte(g[16 * c + b]);
                        }
                    if (esc[n * gpr + kg]) {
                        for (int i = 0; i < UWO_GROUP; i++)
                            blob[epos + i] = (uint8_t)uwo_exponent(g[i]);
                        epos += 64;
                    } else {
                        for (int i = 0; i < UWO_GROUP; i++)
                            sym[i] = palette_index(palette, npal, uwo_exponent(g[i]));
                        encode_group(sym, len, code, gbuf);
                        memcpy(blob + cpos, gbuf, glen[q]);
                        cpos += glen[q];
                    }
                }
            }
        }
    }
    free(esc);
    free(glen);
    free(tcode);
    free(tesc);
    free(padded);
    return (int64_t)total;
}

/* Read the header.  Returns 0, or -1 if the bytes are not a well-formed
 * UWB1 header whose sections fit in `bytes`. */
int uwo_read_header(const uint8_t *blob, int64_t bytes, uwo_info *info)
{
    if (bytes < UWO_HEADER || get_u32(blob) != UWO_MAGIC || get_u32(blob + 4) != UWO_VERSION)
        return -1;
    memset(info, 0, sizeof *info);
    info->rows = (int64_t)get_u64(blob + 8);
    info->cols = (int64_t)get_u64(blob + 16);
    if (get_u32(blob + 24) != UWO_GROUP || get_u32(blob + 28) != UWO_TROWS)
        return -1;
    info->lmax = (int32_t)get_u32(blob + 32);
    info->n_palette = (int32_t)get_u32(blob + 36);
    memcpy(info->palette, blob + 40, 16);
    memcpy(info->code_len, blob + 56, 16);
    info->n_groups = (int64_t)get_u64(blob + 72);
    info->n_escaped = (int64_t)get_u64(blob + 80);
    info->n_tiles = (int64_t)get_u64(blob + 88);
    info->code_bits = (int64_t)get_u64(blob + 96);
    info->off_sm = get_u64(blob + 104);
    info->off_glen = get_u64(blob + 112);
    info->off_tcode = get_u64(blob + 120);
    info->off_tesc = get_u64(blob + 128);
    info->off_code = get_u64(blob + 136);
    info->off_esc = get_u64(blob + 144);
    info->blob_bytes = (int64_t)get_u64(blob + 152);
    if (info->rows <= 0 || info->cols <= 0)
        return -1;
    if (info->blob_bytes > bytes || info->lmax != UWO_LMAX || info->n_palette > UWO_PAL)
        return -1;
    if (info->rows > ((int64_t)1 << 31) || info->cols > ((int64_t)1 << 31))
        return -1;
    int64_t cp = uwo_stored_cols(info->cols);
    int64_t gpr = cp / UWO_GROUP;
    if (info->n_groups != info->rows * gpr ||
        info->n_tiles != (info->rows + UWO_TROWS - 1) / UWO_TROWS * gpr)
        return -1;
    /* every section inside the blob, in the order the format lays them out
     * (sizes kept below 2^62 first, so the sums cannot wrap) */
    if (info->rows > ((int64_t)1 << 31) || info->cols > ((int64_t)1 << 31) || info->n_escaped < 0 ||
        info->n_escaped > info->n_groups || info->blob_bytes < UWO_HEADER)
        return -1;
    const uint64_t end = (uint64_t)info->blob_bytes;
    const uint64_t tiles4 = 4 * ((uint64_t)info->n_tiles + 1);
    const uint64_t start[6] = {info->off_sm, info->off_glen, info->off_tcode,
                               info->off_tesc, info->off_code, info->off_esc};
    const uint64_t size[6] = {(uint64_t)(info->rows * cp), (uint64_t)info->n_groups, tiles4,
                              tiles4, 0, 64 * (uint64_t)info->n_escaped};
    uint64_t prev = UWO_HEADER;
    for (int s = 0; s < 6; s++) {
        if (start[s] < prev || start[s] > end || size[s] > end - start[s])
            return -1;
        prev = start[s] + size[s];
    }
    return 0;
}

/* Decompress a blob back to W.  The decode walks the bits one at a time and
 * compares the prefix read so far with every code of that length.
 * Returns 0, or -1 malformed header, -2 bad code, -3 a group's bit count
 * disagrees with its byte length, -4 escape or code offsets out of range. */
int uwo_decompress(const uint8_t *blob, int64_t bytes, uint16_t *w)
{
    uwo_info I;
    if (uwo_read_header(blob, bytes, &I) != 0)
        return -1;
    uint16_t code[UWO_PAL];
    uwo_canonical_codes(I.code_len, UWO_PAL, code);
    int64_t rows = I.rows, cols = uwo_stored_cols(I.cols), gpr = cols / UWO_GROUP;
    int64_t nrb = (rows + UWO_TROWS - 1) / UWO_TROWS;
    uint64_t code_end = I.off_esc; /* code section ends before esc section */
    for (int64_t rb = 0; rb < nrb; rb++) {
        int64_t R = rows - rb * UWO_TROWS < UWO_TROWS ? rows - rb * UWO_TROWS : UWO_TROWS;
        for (int64_t kg = 0; kg < gpr; kg++) {
            int64_t t = rb * gpr + kg;
            uint64_t cpos = I.off_code + 16 * (uint64_t)get_u32(blob + I.off_tcode + 4 * t);
            uint64_t eidx = get_u32(blob + I.off_tesc + 4 * t);
            for (int64_t j = 0; j < R; j++) {
                int64_t n = rb * UWO_TROWS + j;
                int64_t q = UWO_TROWS * rb * gpr + R * kg + j;
                unsigned gl = blob[I.off_glen + q];
                uint8_t e[UWO_GROUP];
                if (gl == 0) {
                    if (eidx >= (uint64_t)I.n_escaped)
                        return -4;
                    memcpy(e, blob + I.off_esc + 64 * eidx, 64);
                    eidx++;
                } else {
                    if (cpos + gl > code_end)
                        return -4;
                    int64_t bit = 0;
                    for (int i = 0; i < UWO_GROUP; i++) {
                        unsigned v = 0;
                        int l = 0, s = -1;
                        while (s < 0) {
                            if (l >= UWO_LMAX || bit >= 8 * (int64_t)gl)
                                return -2;
                            unsigned b = (blob[cpos + bit / 8] >> (bit % 8)) & 1u;
                            v = (v << 1) | b;
                            l++;
                            bit++;
                            for (int c = 0; c < I.n_palette; c++)
                                if (I.code_len[c] == l && code[c] == v)
                                    s = c;
                        }
                        e[i] = I.palette[s];
                    }
                    if ((bit + 7) / 8 != gl)
                        return -3;
                    cpos += gl;
                }
                /* the output keeps only the matrix's own columns */
                for (int c = 0; c < 4; c++)
                    for (int b = 0; b < 16; b++) {
                        uint64_t at = I.off_sm + (uint64_t)(UWO_TROWS * rb * cols + 64 * R * kg + (c * R + j) * 16 + b);
                        int64_t k = kg * UWO_GROUP + 16 * c + b;
                        if (k < I.cols)
                            w[n * I.cols + k] = uwo_join(e[16 * c + b], blob[at]);
                    }
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------
 * [EXPONENT] the exponent byte of every weight (escaped groups included),
 * laid out like the blob's sign+mantissa section: group q = 32*rb*gpr +
 * R*kg + j (row j of row block rb, R rows in the block) owns 64 bytes in four
 * 16-byte chunks; chunk c (weights 16c .. 16c+15) sits at byte
 * 64*q0 + (c*R + j)*16 of the buffer, q0 = 32*rb*gpr + R*kg, weight 16c + b
 * at byte b of the chunk.  out: rows*cols bytes, overwritten.
 */
void uwo_exponents(const uint16_t *w, int64_t rows, int64_t cols, uint8_t *out)
{
    int64_t gpr = cols / UWO_GROUP;
    for (int64_t n = 0; n < rows; n++) {
        int64_t rb = n / UWO_TROWS, j = n % UWO_TROWS;
        int64_t left = rows - rb * UWO_TROWS;
        int64_t R = left < UWO_TROWS ? left : UWO_TROWS;
        for (int64_t kg = 0; kg < gpr; kg++) {
            int64_t q0 = UWO_TROWS * rb * gpr + R * kg;
            for (int k = 0; k < UWO_GROUP; k++)
                out[64 * q0 + ((k / 16) * R + j) * 16 + k % 16] =
                    (uint8_t)((w[n * cols + kg * UWO_GROUP + k] >> 7) & 0xFFu);
        }
    }
}

/* ------------------------------------------------------------------------
 * [PALETTE] 4-bit palette index of every weight of a matrix.
 * Definition: for a weight in a group that is not escaped, its index is the
 * position of its exponent in the blob's palette (header order); escaped
 * groups get index 0 (their exponents stay in the escape section).
 * Layout (the library's palette-4 form): like the sign+mantissa section at
 * half the width.  Group q = 32*rb*gpr + R*kg + j (row j of row block rb,
 * R rows in the block) owns 32 bytes in two 16-byte chunks; chunk c holds
 * weights 32c .. 32c+31 at byte 32*q0 + (c*R + j)*16 of the buffer, q0 =
 * 32*rb*gpr + R*kg the tile's first group, and weight 32c + 2i + b is nibble
 * b (0 = low) of byte i of the chunk.  out: rows*cols/2 bytes, overwritten.
 */
void uwo_palette4(const uint16_t *w, int64_t rows, int64_t cols, const uint8_t *palette, int npal, uint8_t *out)
{
    int64_t gpr = cols / UWO_GROUP;
    memset(out, 0, (size_t)(rows * cols / 2));
    for (int64_t n = 0; n < rows; n++) {
        int64_t rb = n / UWO_TROWS, j = n % UWO_TROWS;
        int64_t left = rows - rb * UWO_TROWS;
        int64_t R = left < UWO_TROWS ? left : UWO_TROWS;
        for (int64_t kg = 0; kg < gpr; kg++) {
            int idx[UWO_GROUP], escaped = 0;
            for (int k = 0; k < UWO_GROUP; k++) {
                unsigned e = (w[n * cols + kg * UWO_GROUP + k] >> 7) & 0xFFu;
                idx[k] = palette_index(palette, npal, e);
                if (idx[k] < 0)
                    escaped = 1;
            }
            int64_t q0 = UWO_TROWS * rb * gpr + R * kg;
            for (int k = 0; k < UWO_GROUP; k++) {
                int v = escaped ? 0 : idx[k];
                int c = k / 32, i = (k % 32) / 2, b = k % 2;
                out[32 * q0 + (c * R + j) * 16 + i] |= (uint8_t)(v << (4 * b));
            }
        }
    }
}

/* ------------------------------------------------------------------------
 * [MATMUL] y[b,n] = sum_k x[b,k] * W[n,k] in fp64, and the magnitude sum
 * a[b,n] = sum_k |x[b,k] * W[n,k]| used by the error bound.
 * Rows n0 .. n0+nr-1 of W only (nr = N for all of them).
 * --------------------------------------------------------------------- */
double uwo_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

void uwo_matmul_f64(const uint16_t *x, int64_t B, const uint16_t *w, int64_t N, int64_t K,
                    int64_t n0, int64_t nr, double *y, double *absum)
{
    for (int64_t b = 0; b < B; b++)
        for (int64_t n = n0; n < n0 + nr && n < N; n++) {
            double s = 0.0, a = 0.0;
            for (int64_t k = 0; k < K; k++) {
                double p = uwo_bf16_to_double(x[b * K + k]) * uwo_bf16_to_double(w[n * K + k]);
                s += p;
                a += fabs(p);
            }
            y[b * nr + (n - n0)] = s;
            if (absum)
                absum[b * nr + (n - n0)] = a;
        }
}

/* SwiGLU glue of an MLP layer: h = silu(g) * u, silu(z) = z / (1 + e^-z),
 * in fp64 from bf16 inputs. */
void uwo_swiglu_f64(const uint16_t *g, const uint16_t *u, int64_t n, double *h)
{
    for (int64_t i = 0; i < n; i++) {
        double z = uwo_bf16_to_double(g[i]);
        h[i] = z / (1.0 + exp(-z)) * uwo_bf16_to_double(u[i]);
    }
}
