/*
 * uw.h -- C ABI of the lossless BF16 weight compression library for NVIDIA
 * GB300 (sm_103a).
 *
 * The method is the one the Unweight blog post ("Unweight: how we compressed
 * an LLM 22% without sacrificing quality", Cloudflare) describes:
 *   - a BF16 weight is 1 sign bit, 8 exponent bits and 7 mantissa bits; sign
 *     and mantissa look random and are stored raw, one byte per weight
 *     (paragraphs on the BF16 layout and on what is left uncompressed);
 *   - the exponent byte is Huffman coded over a per-matrix palette of the 16
 *     most common exponents (paragraphs on exponent skew and Huffman coding);
 *   - a row of 64 weights that holds an exponent outside the palette keeps
 *     its 64 raw exponent bytes: one decision per row (paragraph on rare
 *     exponents);
 *   - at inference the weights are either decompressed back to BF16 in HBM
 *     and multiplied, or decoded on chip and fed straight to the matrix
 *     multiply without ever being written back (paragraphs on the four
 *     execution pipelines and the reconstructive matmul);
 *   - an autotuner measures each choice per weight matrix and batch size
 *     (paragraph on the autotuner).
 *
 * Conventions for every entry point:
 *   - Weights W are [rows, cols] row-major BF16 (uint16 bit patterns), the
 *     layout of a PyTorch Linear weight (out_features x in_features).
 *     Activations x are [batch, cols] row-major BF16; outputs y are
 *     [batch, rows] row-major BF16; y = x W^T with fp32 accumulation and
 *     round-to-nearest-even to BF16.
 *   - rows and cols must be positive, otherwise UW_ERR_SHAPE.  A row whose
 *     length is not a multiple of 64 ("ragged") is stored extended to the
 *     next multiple, cp = 64 * ceil(cols / 64), with filler weights (sign
 *     and mantissa 0, exponent the first palette exponent below 255, else
 *     0); the descriptor keeps the true cols.  The blog's matrices all have
 *     whole rows of 64; this extension is the library's reading for the
 *     rest.  The matmuls run on the stored width with the activations
 *     copied into zero-extended rows in the workspace (a filler weight
 *     times zero adds nothing); uw_decompress writes the true columns only.
 *   - The caller owns all memory.  The library allocates no device memory,
 *     with one exception: the 1 MiB scratch array of uw_matmul_noalloc, a
 *     static device array that every GPU which loads the library holds until
 *     the process exits.  Pointers marked _dev are device pointers, _host
 *     host pointers.
 *     Scratch space ("workspace") is passed in by the caller; its size comes
 *     from uw_workspace_size and it must be cleared once with
 *     uw_workspace_init before first use.  Kernels leave it ready for the
 *     next call.  One workspace must not be used by two calls that may run
 *     at the same time.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Device work is enqueued on it and the call returns without
 *     waiting, except where a function says it synchronises.
 *   - Errors are returned as uw_status; nothing throws across the ABI.
 *     Errors found by the GPU while decoding (a blob corrupted after
 *     uw_blob_info checked its header) are recorded in the workspace and
 *     reported by uw_check_status.
 */
#ifndef UW_H
#define UW_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    UW_OK = 0,
    UW_ERR_INVALID_ARG = 1,      /* NULL pointer, negative size, bad plan      */
    UW_ERR_SHAPE = 2,            /* rows <= 0 or cols <= 0; the MLP chain also
                                    refuses cols % 64 != 0                     */
    UW_ERR_BUFFER_TOO_SMALL = 3, /* output or workspace buffer too small       */
    UW_ERR_CORRUPT = 4,          /* blob header or data inconsistent           */
    UW_ERR_CUDA = 5,             /* a CUDA runtime call failed                 */
    UW_ERR_TIMEOUT = 6,          /* a bounded device wait gave up              */
    UW_ERR_UNSUPPORTED = 7,      /* valid request this build cannot run        */
    UW_ERR_INTERNAL = 8
} uw_status;

/* Execution strategies (the blog's pipelines).  DECOMPRESS_GEMM restores
 * BF16 weights into the workspace, then multiplies them.  FUSED decodes in
 * registers / shared memory and never writes the weights back.  PALETTE4
 * transcodes the Huffman codes into 4-bit palette indices in the workspace
 * (a quarter of the bytes a full decode writes), then multiplies from those
 * (uw_matmul_palette4).  EXPONENT decodes only the exponent bytes into the
 * workspace (half the bytes of a full decode), then multiplies, merging them
 * with the raw sign+mantissa bytes (uw_matmul_exponents). */
enum {
    UW_STRATEGY_DEFAULT = -1,
    UW_STRATEGY_DECOMPRESS_GEMM = 0,
    UW_STRATEGY_FUSED = 1,
    UW_STRATEGY_PALETTE4 = 2,
    UW_STRATEGY_EXPONENT = 3
};

/* Description of a compressed matrix, filled by uw_blob_info from the blob
 * header (host copy).  All offsets are byte offsets from the blob start.
 * Every entry point that reads a blob re-checks the descriptor it is given
 * (sizes and counts consistent, at most 2^31 rows and columns, sections in
 * order inside blob_bytes, code lengths a prefix code of at most 5 bits) and
 * returns UW_ERR_INVALID_ARG for one that uw_blob_info could not have filled.
 * The size queries (uw_workspace_size, uw_palette4_bytes, ...) read only rows
 * and cols. */
typedef struct {
    int64_t rows, cols;
    uint64_t blob_bytes;     /* total blob size                              */
    uint64_t code_bits;      /* Huffman bits of all coded groups (no padding) */
    uint64_t n_groups;       /* rows * cp / 64 (cp: cols rounded up to 64)    */
    uint64_t n_escaped;      /* groups stored with raw exponents              */
    uint64_t n_tiles;        /* ceil(rows / 32) * cp / 64                     */
    int32_t n_palette;       /* palette entries in use (0..16)                */
    int32_t lmax;            /* longest code length (5 in format version 2)   */
    uint8_t palette[16];     /* exponent value of each symbol                 */
    uint8_t code_len[16];    /* code length of each symbol, 0 = unused        */
    uint64_t off_sm, off_glen, off_tcode, off_tesc, off_code, off_esc;
    uint64_t max_tile_bytes; /* largest code region + escaped exponents of one
                                tile (sizes the kernels' on-chip tile buffers) */
} uw_desc;

/* One tuned choice for (matrix, batch). */
typedef struct {
    int32_t strategy;        /* UW_STRATEGY_*                                  */
    int32_t variant;         /* kernel variant inside the strategy             */
    int64_t batch;           /* batch size the choice was measured at          */
    float us;                /* measured time of one call, microseconds        */
} uw_plan;

/* uw_compress -- build the compressed blob of one weight matrix on the host.
 * Follows the blog's paragraphs on exponent skew, Huffman coding of the
 * exponent byte and rows of 64 with rare exponents: exponent histogram ->
 * 16-entry palette -> escaped groups -> length-limited minimum-redundancy
 * canonical code -> blob (format UWB1, laid out in the library source csrc/format.h).
 *   w_host     [rows, cols] BF16 bits, host memory, read only.
 *   blob_out   host buffer of *blob_bytes bytes, or NULL to query the size.
 *   blob_bytes in: capacity of blob_out; out: size of the blob.
 * Returns UW_ERR_BUFFER_TOO_SMALL (with *blob_bytes set) when blob_out is
 * NULL or too small, UW_ERR_SHAPE when rows or cols is not positive,
 * UW_ERR_UNSUPPORTED beyond 2^31 rows or columns or
 * when the tile tables' 32-bit offsets would overflow.  Uses the host's cores
 * (OpenMP); deterministic. */
uw_status uw_compress(const uint16_t *w_host, int64_t rows, int64_t cols,
                      void *blob_out, size_t *blob_bytes);

/* uw_blob_info -- validate a blob's header and section table (host copy of
 * at least the first 256 bytes and its declared size) and fill *out.
 *   bytes  size of the buffer holding the blob (>= header's blob size).
 * Returns UW_ERR_CORRUPT for a bad magic, version, shape or section that
 * does not fit. */
uw_status uw_blob_info(const void *blob_host, size_t bytes, uw_desc *out);

/* uw_workspace_size -- bytes of workspace the given call needs.
 *   batch     activation rows of the uw_matmul call (0 for uw_decompress).
 *   plan      the plan the call will use, or NULL for the default plan.   */
uw_status uw_workspace_size(const uw_desc *d, int64_t batch, const uw_plan *plan,
                            size_t *bytes);

/* uw_workspace_init -- clear a freshly allocated workspace (stream ordered). */
uw_status uw_workspace_init(void *ws_dev, size_t ws_bytes, void *stream);

/* uw_decompress -- restore the exact BF16 weights into HBM (the blog's
 * "full decode" pipeline).
 *   blob_dev   device copy of the blob described by d.
 *   w_dev      [rows, cols] BF16 output, device memory, 16-byte aligned.
 *   ws_dev     workspace (error word only; >= uw_workspace_size(d, 0, NULL)). */
uw_status uw_decompress(const uw_desc *d, const void *blob_dev, uint16_t *w_dev,
                        void *ws_dev, size_t ws_bytes, void *stream);

/* uw_matmul -- y = x W^T with W still compressed (the blog's reconstructive
 * matmul, or decompress-then-multiply, as the plan says).
 *   x_dev   [batch, cols] BF16, 16-byte aligned;  y_dev  [batch, rows] BF16
 *           (written).
 *   plan    strategy/variant to run, or NULL for the library's default for
 *           this shape and batch.  A variant whose on-chip buffers do not fit
 *           this blob or batch returns UW_ERR_UNSUPPORTED without running.
 * The result is bit-identical to uw_matmul_bf16 with the same variant on the
 * original weights. */
uw_status uw_matmul(const uw_desc *d, const void *blob_dev, const uint16_t *x_dev,
                    int64_t batch, uint16_t *y_dev, const uw_plan *plan,
                    void *ws_dev, size_t ws_bytes, void *stream);

/* uw_matmul_bf16 -- the same kernels fed uncompressed BF16 weights: the
 * baseline that compression is measured against.
 *   w_dev   [rows, cols] BF16 device weights, x_dev [batch, cols]; both
 *           16-byte aligned (UW_ERR_INVALID_ARG otherwise).  variant as in
 *           uw_plan.  rows and cols positive (UW_ERR_SHAPE) and at most 2^31
 *           (UW_ERR_UNSUPPORTED), as for compressed matrices.  Ragged rows
 *           (cols % 64 != 0) are copied with x into zero-extended rows in the
 *           workspace first.
 *   ws_dev  workspace of at least uw_workspace_size_bf16 bytes. */
uw_status uw_matmul_bf16(const uint16_t *w_dev, int64_t rows, int64_t cols,
                         const uint16_t *x_dev, int64_t batch, uint16_t *y_dev,
                         int32_t variant, void *ws_dev, size_t ws_bytes, void *stream);

/* uw_workspace_size_bf16 -- bytes of workspace uw_matmul_bf16 needs for this
 * shape, batch and variant (-1: the default). */
uw_status uw_workspace_size_bf16(int64_t rows, int64_t cols, int64_t batch, int32_t variant,
                                 size_t *bytes);

/* The palette-4 form of a blob (the blog's palette pipelines: the Huffman
 * codes turned into 4-bit palette indices at run time, or once when the
 * model is loaded, from which the matmul rebuilds BF16 on the fly;
 * paragraphs on the four execution pipelines and on the palette format at
 * model load).  Every weight's 4-bit index into the blob's palette, laid out
 * like the blob's sign+mantissa section at half the width: group q (row j of
 * row block rb, column group kg; R rows in the block) owns 32 bytes in two
 * 16-byte chunks, chunk c (weights 32c..32c+31) at byte 32*q0 + (c*R + j)*16
 * with q0 = 32*rb*(cp/64) + R*kg, weight 32c + 2i + b in nibble b (0 = low)
 * of byte i.  Escaped groups hold index 0; their exponents stay in the blob.
 *
 * Ragged matrices have the form of their stored width cp.
 *
 * uw_palette4_bytes -- size of the form: rows * cp / 2 bytes. */
uw_status uw_palette4_bytes(const uw_desc *d, size_t *bytes);

/* uw_transcode_palette4 -- write the palette-4 form of the blob.
 *   blob_dev   device copy of the blob described by d.
 *   p4_dev     uw_palette4_bytes(d) bytes of device memory, 16-byte aligned
 *              (written).
 *   ws_dev     workspace (error word only; >= uw_workspace_size(d, 0, NULL)). */
uw_status uw_transcode_palette4(const uw_desc *d, const void *blob_dev, void *p4_dev,
                                void *ws_dev, size_t ws_bytes, void *stream);

/* uw_matmul_palette4 -- y = x W^T from the palette-4 form p4_dev (made by
 * uw_transcode_palette4 from blob_dev) plus the blob's sign+mantissa bytes,
 * group lengths and escaped exponents.
 *   variant  a column variant (batch 1 only) or a tensor-core variant, -1 for
 *            the default; row variants return UW_ERR_UNSUPPORTED.
 *   ws_dev   workspace of at least uw_workspace_size(d, batch, plan) for a
 *            FUSED plan with the same variant.
 * The result is bit-identical to uw_matmul_bf16 with the same variant on the
 * original weights. */
uw_status uw_matmul_palette4(const uw_desc *d, const void *blob_dev, const void *p4_dev,
                             const uint16_t *x_dev, int64_t batch, uint16_t *y_dev, int32_t variant,
                             void *ws_dev, size_t ws_bytes, void *stream);

/* The exponent form of a blob (the blog's exponent-only pipeline: only the
 * exponent bytes are decoded to memory, and the matmul merges them with the
 * raw sign+mantissa bytes; paragraph on the four execution pipelines).
 * Every weight's exponent byte, escaped groups included, laid out like the
 * blob's sign+mantissa section: group q owns 64 bytes in four 16-byte
 * chunks, chunk c (weights 16c..16c+15) at byte 64*q0 + (c*R + j)*16 with q0
 * and R as for the palette-4 form, weight 16c + b at byte b of the chunk.
 *
 * uw_exponent_bytes -- size of the form: rows * cp bytes. */
uw_status uw_exponent_bytes(const uw_desc *d, size_t *bytes);

/* uw_decode_exponents -- write the exponent form of the blob.
 *   e_dev    uw_exponent_bytes(d) bytes of device memory, 16-byte aligned
 *            (written).  Other arguments as for uw_transcode_palette4. */
uw_status uw_decode_exponents(const uw_desc *d, const void *blob_dev, void *e_dev,
                              void *ws_dev, size_t ws_bytes, void *stream);

/* uw_matmul_exponents -- y = x W^T from the exponent form e_dev (made by
 * uw_decode_exponents from blob_dev) plus the blob's sign+mantissa bytes.
 * Arguments, variants and the bit-identity guarantee as for
 * uw_matmul_palette4. */
uw_status uw_matmul_exponents(const uw_desc *d, const void *blob_dev, const void *e_dev,
                              const uint16_t *x_dev, int64_t batch, uint16_t *y_dev, int32_t variant,
                              void *ws_dev, size_t ws_bytes, void *stream);

/* uw_autotune -- measure every (strategy, variant) candidate for each batch
 * size and return the fastest per batch (the blog's autotuner, which picks a
 * pipeline per weight matrix and batch size from measured throughput).
 * Each timed call follows an overwrite of the L2 cache, so the weights are
 * read from HBM.  Synchronises `stream`.  The workspace (size from
 * uw_autotune_workspace_size) holds the run workspace, x and y scratch and
 * the L2 overwrite buffer; it is left cleared for uw_matmul.
 *   batches    n batch sizes; plans_out  n results (us = median time). */
uw_status uw_autotune(const uw_desc *d, const void *blob_dev, const int64_t *batches,
                      int32_t n, uw_plan *plans_out, void *ws_dev, size_t ws_bytes,
                      void *stream);
uw_status uw_autotune_workspace_size(const uw_desc *d, const int64_t *batches, int32_t n,
                                     size_t *bytes);

/* uw_matmul_noalloc -- uw_matmul with the default plan for callers that
 * cannot allocate device memory: code that must not call cudaMalloc (it can
 * synchronise the device or is not allowed in its context), plug-ins whose
 * host framework owns all device memory, or callers that simply have no
 * workspace buffer to hand over.  The Unweight blog has no counterpart;
 * this is a convenience of this library.
 * Scratch comes from a fixed array of 1 MiB inside the library, which every
 * GPU that loads the library keeps until the process exits.  The call
 * allocates nothing; the caller still passes x_dev [batch, cols] and
 * y_dev [batch, rows] and gets the same result as uw_matmul with plan NULL.
 * Returns UW_ERR_UNSUPPORTED when the call would need more than 1 MiB of
 * scratch (uw_workspace_size(d, batch, NULL) > 1 MiB; then use uw_matmul).
 * The first call on each device looks up the array's device address, so
 * make that first call before any stream capture.  All calls share the one
 * array: calls that may overlap on the GPU (other streams, other threads)
 * race and must not be issued.  Decode errors found on the GPU are not
 * reported here; use uw_matmul with a workspace and uw_check_status for
 * that. */
uw_status uw_matmul_noalloc(const uw_desc *d, const void *blob_dev, const uint16_t *x_dev,
                            int64_t batch, uint16_t *y_dev, void *stream);

/* uw_selftest_bounded_wait -- exercises the failure path of the kernels'
 * bounded waits.  Launches one small kernel that waits, with the same wait
 * routine the matmul and decode kernels use, on a shared-memory barrier
 * that nothing arrives on; after `tries` attempts (1 .. 2^22, the kernels'
 * own limit) the wait gives up, records a timeout in the workspace's status
 * word and the kernel returns.  uw_check_status(ws) then reports
 * UW_ERR_TIMEOUT (and clears the word); the CUDA context stays usable.
 *   ws_dev   a workspace of at least 256 bytes (only its status word is used).
 * Returns UW_ERR_INVALID_ARG for tries outside 1 .. 2^22.  Diagnostic only:
 * the Unweight blog has no counterpart. */
uw_status uw_selftest_bounded_wait(void *ws_dev, size_t ws_bytes, uint32_t tries, void *stream);

/* uw_swiglu -- h = bf16(silu(g) * u), silu(z) = z / (1 + e^-z) in fp32,
 * the glue between the gate/up and down projections of a SwiGLU MLP.
 * g_dev, u_dev, h_dev: n BF16 values each, device memory. */
uw_status uw_swiglu(const uint16_t *g_dev, const uint16_t *u_dev, uint16_t *h_dev,
                    int64_t n, void *stream);

/* ---------------------------------------------------------------------------
 * MLP chain with concurrent preprocessing.  Follows the Unweight blog's
 * paragraphs on running the preprocess kernel (Huffman decoder or palette
 * transcoder) beside the reconstructive matmul, on splitting the SMs between
 * the two, on "hard" and "easy" layers, on double-buffered preprocess slots
 * and on tuning gate, up and down in turn.
 *
 * Layer l maps x_l [batch, D] to x_{l+1} [batch, D]:
 *     g = x_l Wg^T, u = x_l Wu^T   ([batch, F_l] each)
 *     h = bf16(silu(g) * u)        (as uw_swiglu)
 *     x_{l+1} = h Wd^T
 * and the last layer writes y.  Matrices come three per layer, in the order
 * gate [F_l, D], up [F_l, D], down [D, F_l].  Each runs under its own plan:
 *   FUSED                          decoded inside the matmul (no preprocessing);
 *   PALETTE4 with form_dev         "easy": the palette-4 form made at load by
 *                                  uw_transcode_palette4 is read directly;
 *   PALETTE4 without form_dev, EXPONENT, DECOMPRESS_GEMM
 *                                  "hard": a preprocess kernel writes the
 *                                  palette-4 form, the exponent form or the
 *                                  BF16 weights into a slot of the workspace,
 *                                  and the plan's matmul reads the slot.
 * With a side stream, preprocessing runs there in the order the hard
 * matrices are used, as far ahead as the slots allow: a slot is rewritten
 * only after the matmul that read it has completed.  It waits for nothing
 * else, so it overlaps the matmuls of the layers before it.  Each
 * preprocess kernel is limited to dec_ctas SMs (one persistent CTA each,
 * holding its SM by itself), which leaves the rest to the matmul beside it.
 * Every matmul gives the same bits as under uw_matmul with its plan (and as
 * uw_matmul_bf16 with its variant on the original weights), so the chain's
 * output does not depend on the schedule. */
typedef struct {
    const uw_desc *desc;     /* host description of the blob                        */
    const void *blob_dev;    /* device copy of the blob                             */
    const void *form_dev;    /* palette-4 form made at load (16-byte aligned), or NULL */
    uw_plan plan;            /* strategy and variant (-1: default); batch, us unused */
} uw_mlp_matrix;

typedef struct {
    int32_t slots;           /* preprocess slots: 1, or 2 (double-buffered)          */
    int32_t dec_ctas;        /* SMs of each preprocess kernel; 0: as many as its work
                                needs (no split)                                      */
} uw_schedule;

/* uw_mlp_workspace_size -- bytes of workspace uw_mlp_forward needs for these
 * matrices, plans, batch and schedule (NULL: 2 slots, no split). */
uw_status uw_mlp_workspace_size(const uw_mlp_matrix *m, int32_t n_layers, int64_t batch,
                                const uw_schedule *sched, size_t *bytes);

/* uw_mlp_forward -- run the chain on `stream`, preprocessing on side_stream.
 *   m          3 * n_layers matrices (gate, up, down per layer); shapes as
 *              above with one D for all layers, D and every F multiples of
 *              64 (UW_ERR_SHAPE otherwise).
 *   x_dev      [batch, D] BF16, 16-byte aligned;  y_dev [batch, D] BF16 (written).
 *   sched      slots and SM split, or NULL (2 slots, no split).
 *   ws_dev     at least uw_mlp_workspace_size bytes, cleared once by
 *              uw_workspace_init; decode errors are recorded in its first
 *              word (read them with uw_check_status).
 *   side_stream  a stream other than `stream` (created non-blocking), or NULL:
 *              then each preprocess kernel runs on `stream` right before its
 *              matmul and nothing overlaps.
 * Stream ordered: the side stream first waits for all work already on
 * `stream`, and `stream` ends waiting for the side stream, so the next call
 * on `stream` may reuse the workspace.  Capturable in a CUDA graph when both
 * streams are captured from `stream`. */
uw_status uw_mlp_forward(const uw_mlp_matrix *m, int32_t n_layers, const uint16_t *x_dev,
                         int64_t batch, uint16_t *y_dev, const uw_schedule *sched,
                         void *ws_dev, size_t ws_bytes, void *stream, void *side_stream);

/* uw_mlp_autotune -- choose, by coordinate descent on the measured time of
 * whole uw_mlp_forward calls, one plan per role and the SM split: sweep the
 * gate's candidates with up and down held, then up's, then down's (first for
 * the matrices without a load-time form, then for those with one), then
 * dec_ctas, and repeat until a pass changes nothing (at most `passes`
 * passes).  Candidates: every strategy with its default variant, plus
 * (batch >= 16) the tensor-core variants with two or three producer groups
 * and any K split (split 1 leaves SMs free beside the matmul); matrices with
 * a form only PALETTE4.
 *   m, n_layers, x_dev, batch, y_dev, streams as for uw_mlp_forward (the
 *              plans in m are ignored; y is overwritten).
 *   plans_out  6 plans: gate, up, down of the matrices without a form, then
 *              of those with one; us = the best forward's time.
 *   sched_out  the chosen schedule (2 slots).
 *   ws_dev     at least uw_mlp_autotune_workspace_size bytes, cleared.
 * Synchronises both streams. */
uw_status uw_mlp_autotune(const uw_mlp_matrix *m, int32_t n_layers, const uint16_t *x_dev,
                          int64_t batch, uint16_t *y_dev, int32_t passes, uw_plan *plans_out,
                          uw_schedule *sched_out, void *ws_dev, size_t ws_bytes, void *stream,
                          void *side_stream);
uw_status uw_mlp_autotune_workspace_size(const uw_mlp_matrix *m, int32_t n_layers, int64_t batch,
                                         size_t *bytes);

/* uw_check_status -- synchronise `stream`, read and clear the error word the
 * kernels record in the workspace.  Returns UW_OK, UW_ERR_CORRUPT or
 * UW_ERR_TIMEOUT (or UW_ERR_CUDA if the stream itself failed). */
uw_status uw_check_status(void *ws_dev, void *stream);

/* Variant names for diagnostics; NULL for an unknown (strategy, variant). */
const char *uw_variant_name(int32_t strategy, int32_t variant);
int32_t uw_variant_count(int32_t strategy);

const char *uw_status_string(uw_status s);

#ifdef __cplusplus
}
#endif

#endif /* UW_H */
