/*
 * entropack.h -- C ABI of libentropack.so, the B300 (sm_103a) implementation
 * of EntroPack's inference hot path: on-GPU decoding of entropy-coded E8
 * lattice weights into BF16 / FP16 / FP8 / INT8 containers, plus the host
 * encoder that produces the stream.
 *
 * Method: "EntroPack: Fast and Accurate Entropy-Coded Weight Compression at
 * Arbitrary Bitrates", Abstract -- E8 lattice quantisation of rows scaled to
 * unit size, a probability model of each lattice coordinate given the coset,
 * a resolution picked from rate estimates on sampled rows, entropy coding in
 * tiles that decode independently, one GPU pass that decodes the symbols and
 * rebuilds the weights, and BF16/FP16/FP8/INT8 containers whose precision is
 * chosen apart from the storage rate.
 * API surface: "EntroPack PyTorch Guide: Lossless Weights, Bitrates and Memory
 * Checks", sections "Choose a compression contract" (lossy target bitrate vs
 * lossless tiled ANS; compress / decompress), "Start with a tensor round trip"
 * (target_bpp vs actual_bpp, which includes metadata).
 * The byte layout is stream format version 1 (header, tables, tile offsets,
 * 4-lane tile payloads).
 *
 * Conventions
 *  - Matrices are row-major; rows = out_features (M), cols = in_features (K).
 *    Any rows >= 1 and cols >= 1 with cols % 8 == 0; the stream codes the
 *    matrix padded with zeros to whole 32 x 128 tiles and the decoder writes
 *    only the rows x cols values (row stride cols).
 *  - Every pointer is owned by the caller, except the blob returned by
 *    ep_encode (release it with ep_free).
 *  - Device entry points are asynchronous on `stream`; they allocate nothing
 *    and return EP_OK once the work is enqueued.  Corruption that only the
 *    device can see (rANS end state, word counts, escape payloads, tile
 *    bounds) is reported through the caller's status word; read it with
 *    ep_sync_status.  Decoding never loops unboundedly: every loop is bounded
 *    by the tile geometry.
 *  - h_blob is a host copy of the stream (parsed and fully validated on the
 *    host before any launch); d_blob must hold the same bytes on the device,
 *    16-byte aligned.  The kernels re-check every tile's bounds, so a
 *    mismatching device copy can only produce EP_ERR_CORRUPT, never an
 *    out-of-bounds access.
 */
#ifndef ENTROPACK_H
#define ENTROPACK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream; NULL is the legacy default stream. */
typedef struct CUstream_st *ep_stream_t;

typedef enum {
    EP_OK = 0,
    EP_ERR_INVALID_ARG = 1, /* NULL pointer, misaligned pointer, bad enum, bad sizes */
    EP_ERR_SHAPE = 2,       /* empty, cols % 8 != 0, or a dimension above 2^40 */
    EP_ERR_NONFINITE = 3,   /* lossy input holds NaN or +-inf */
    EP_ERR_CORRUPT = 4,     /* stream fails validation (host) or decoding (device status) */
    EP_ERR_UNSUPPORTED = 5, /* value range outside format version 1 */
    EP_ERR_NOMEM = 6,       /* host allocation failed (ep_encode only) */
    EP_ERR_CUDA = 7         /* a CUDA runtime call failed */
} ep_status;

/* Containers of decoded weights.  Lossy streams: BF16, FP16, FP8 e4m3, INT8.
 * Lossless streams keep the input's own type: BF16, FP16, FP8 e4m3 or FP32. */
typedef enum { EP_C_BF16 = 0, EP_C_FP16 = 1, EP_C_FP8_E4M3 = 2, EP_C_INT8 = 3, EP_C_FP32 = 4 } ep_container;
typedef enum { EP_MODE_LOSSY_E8 = 0, EP_MODE_LOSSLESS_TILEANS = 1 } ep_mode;

/* Device status-word bits (OR-ed by the kernels). */
#define EP_STATUS_LANE_END 0x1u   /* a rANS lane did not end at L or did not consume exactly its words */
#define EP_STATUS_TILE_BOUNDS 0x2u /* a tile offset or word count points outside the stream */
#define EP_STATUS_ESCAPE 0x4u     /* an escape payload contradicts its coset */
#define EP_STATUS_WAIT_TIMEOUT 0x8u /* ep_batch_decode: a ring wait gave up (about 2 s); that unit was skipped */

typedef struct {
    int32_t mode;      /* ep_mode */
    float target_bpp;  /* lossy: target coded bits per parameter (> 0) */
    int32_t container; /* ep_container of the decoded weights; lossless: the input's type
                          (EP_C_BF16, EP_C_FP16, EP_C_FP8_E4M3 or EP_C_FP32) */
    float sample_frac; /* fraction of rows sampled by the rate search; <= 0 selects 0.05 */
    int32_t n_threads; /* host threads for ep_encode; <= 0 selects all hardware threads */
} ep_params;

typedef struct {
    int64_t rows, cols, n_tiles;
    int32_t mode, container;
    float target_bpp;    /* as requested (lossy) */
    int32_t j;           /* chosen resolution index: Delta = 2^(j/64) */
    double delta;        /* Delta_j */
    uint64_t total_bytes;
    uint32_t n_sample_rows;
    double actual_bpp;   /* 8 * total_bytes / (rows * cols): includes every byte of metadata */
    size_t out_elem_bytes; /* bytes per decoded element (2 for BF16/FP16, 1 for FP8/INT8, 4 for FP32) */
    int32_t has_row_scale; /* 1 when ep_decode also writes per-row output scales t_r */
} ep_info;

/* Library/format version (format 1). */
int32_t ep_version(void);
const char *ep_status_string(ep_status s);

/*
 * Host encoder.  w: rows x cols elements, row-major, in host memory: BF16
 * bit patterns for lossy streams; for lossless streams elements of the type
 * p->container names (2 bytes for BF16/FP16, 1 for FP8 e4m3, 4 for FP32).
 * Lossy (p->mode == EP_MODE_LOSSY_E8): row-normalised E8 quantisation at the
 * resolution whose sampled rate estimate is closest to p->target_bpp, then
 * 12-bit rANS in 4-lane tiles of 32 x 128.  Lossless: the exponent byte
 * (FP8: the whole element) is coded, sign and mantissa stored raw; decoding
 * restores every bit.
 * On success *blob points to *blob_bytes bytes allocated by the library
 * (release with ep_free).  Errors: EP_ERR_INVALID_ARG, EP_ERR_SHAPE,
 * EP_ERR_NONFINITE (lossy only), EP_ERR_UNSUPPORTED, EP_ERR_NOMEM.
 */
ep_status ep_encode(const void *w, int64_t rows, int64_t cols, const ep_params *p, uint8_t **blob,
                    size_t *blob_bytes);
void ep_free(void *p);

/*
 * Lossy encode at a caller-chosen resolution index j (Delta = 2^(j/64)), with
 * no rate search; otherwise as ep_encode (p->mode must be EP_MODE_LOSSY_E8;
 * p->target_bpp is only recorded in the header).  EP_ERR_INVALID_ARG when j
 * is outside [-640, 128] or below the smallest index that keeps every row's
 * peak in range (ep_estimate_bpp reports that index).
 */
ep_status ep_encode_at(const void *w, int64_t rows, int64_t cols, const ep_params *p, int32_t j, uint8_t **blob,
                       size_t *blob_bytes);

/*
 * The sampled storage estimate (Abstract: the resolution is chosen from rate
 * estimates on a sample, not by encoding the whole stream again and again)
 * of a BF16 matrix (host) at index j: coded bits per parameter on the strided
 * row sample (sample_frac <= 0 selects 0.05), the figure the rate search
 * steers.  *j_min (may be NULL) receives the smallest admissible index.
 */
ep_status ep_estimate_bpp(const uint16_t *w, int64_t rows, int64_t cols, float sample_frac, int32_t j,
                          int32_t n_threads, double *bpp, int32_t *j_min);

/* One layer of a model-level allocation: a BF16 matrix in host memory. */
typedef struct {
    const uint16_t *w;
    int64_t rows, cols; /* cols % 8 == 0 */
    float sensitivity;  /* alpha > 0: weight of this layer's squared relative error (1 = neutral) */
} ep_layer_ref;

/*
 * Per-layer bitrate allocation for a whole-model budget ("EntroPack PyTorch
 * Guide", "Separate reconstruction metrics from application metrics":
 * different bitrates across layers, with the allocation recorded).  Minimises
 * sum_l alpha_l n_l D_l subject to sum_l n_l R_l <= avg_bpp * sum_l n_l.  At
 * high resolution every row-normalised layer has D ~ Delta^2, so the optimum
 * has equal slopes, alpha_l Delta_l^2 constant:
 *   o_l = lround(32 log2 alpha_l),  j_l(t) = clamp(t - o_l, j_min_l, 128);
 *   t = the smallest shared index whose estimated total
 *       E(t) = sum_l n_l * estimate_l(j_l(t)) fits the budget, by bisection
 *       between min_l(j_min_l + o_l) and max_l(128 + o_l) (the lower end if it
 *       fits, the upper end if nothing fits).
 * Writes j_out[n_layers] (encode each layer with ep_encode_at), optionally
 * est_bpp_out[n_layers] and *t_out.  Errors: EP_ERR_INVALID_ARG (NULL, no
 * layers, sensitivity not positive and finite, bad budget), EP_ERR_SHAPE,
 * EP_ERR_NONFINITE, EP_ERR_NOMEM.
 */
ep_status ep_allocate_bits(const ep_layer_ref *layers, int64_t n_layers, float avg_bpp, float sample_frac,
                           int32_t n_threads, int32_t *j_out, double *est_bpp_out, int32_t *t_out);

/* 8 * bytes / (rows * cols) after validating the stream ("actual_bpp", metadata included). */
ep_status ep_actual_bpp(const uint8_t *blob, size_t bytes, double *bpp);
/* Parse and fully validate a host copy of a stream and report its metadata
 * (shape, mode, container, resolution, sizes).  Serves the guide's advice
 * for a failed restore: check that the settings and metadata agree before
 * and after the round trip, and that the stored object holds everything the
 * decoder reads ("EntroPack PyTorch Guide", "Diagnose compression failures
 * in the correct order").  Errors: EP_ERR_INVALID_ARG (NULL),
 * EP_ERR_CORRUPT (any inconsistent header field, table, offset or size). */
ep_status ep_query(const uint8_t *blob, size_t bytes, ep_info *out);

/*
 * Decode a stream on the GPU (Abstract: symbol decoding and the rebuilding of
 * the weight values run fused, on the GPU).
 *   d_out            rows x cols container elements, row-major, 16-byte aligned
 *   d_row_scale_out  FP8/INT8 lossy streams: rows floats t_r such that
 *                    weight[r, k] ~= t_r * d_out[r, k]; NULL allowed (and
 *                    ignored) for BF16/FP16 and lossless streams
 *   d_status         one u32, zeroed by this call (cudaMemsetAsync), then
 *                    OR-ed with EP_STATUS_* bits by the kernel
 * Returns EP_OK when the work is enqueued; host-side validation errors
 * (EP_ERR_CORRUPT, EP_ERR_INVALID_ARG) return before any launch.
 */
ep_status ep_decode(const uint8_t *h_blob, const void *d_blob, size_t bytes, void *d_out, float *d_row_scale_out,
                    uint32_t *d_status, ep_stream_t stream);

/*
 * Debug variant of ep_decode: also writes the coded symbol byte of every
 * coordinate (rows x cols bytes, row-major) to d_sym_out; used to check the
 * symbol stream against the CPU oracle bit for bit.
 */
ep_status ep_decode_symbols(const uint8_t *h_blob, const void *d_blob, size_t bytes, void *d_out,
                            float *d_row_scale_out, uint8_t *d_sym_out, uint32_t *d_status, ep_stream_t stream);

/*
 * Validated stream handles.  ep_decode and ep_compressed_linear parse and
 * validate the host copy on every call (tens of microseconds per layer).
 * A handle keeps the parsed layout so that a stream decoded many times (a
 * CompressedLinear in a denoising loop) is validated once:
 *   ep_stream_open   parse and fully validate h_blob; *out is owned by the
 *                    caller (release with ep_stream_close).  Errors as
 *                    ep_query, plus EP_ERR_NOMEM.  The handle keeps no
 *                    pointer to h_blob.
 *   ep_decode_h      ep_decode of the stream the handle describes; d_blob
 *                    must hold its bytes on the device (16-byte aligned).
 *                    The kernels re-check every tile against the stream
 *                    size, so different device bytes can only raise
 *                    EP_ERR_CORRUPT in the status word.
 *   ep_compressed_linear_h   ep_compressed_linear likewise.
 */
typedef struct ep_stream_handle ep_stream_handle;
ep_status ep_stream_open(const uint8_t *h_blob, size_t bytes, ep_stream_handle **out);
void ep_stream_close(ep_stream_handle *h);
ep_status ep_decode_h(const ep_stream_handle *h, const void *d_blob, void *d_out, float *d_row_scale_out,
                      uint32_t *d_status, ep_stream_t stream);

/*
 * Batched decode: many streams (e.g. every linear layer of a model) in one
 * persistent launch.  All items must share mode and container.  Work is cut
 * into units of 40 groups of 8 tiles (320 tiles) of one item; CTAs (one per
 * SM, 20 warps) claim units in item order, two groups per warp.
 *
 *   ring == 0  every item writes its own d_out (outputs must not overlap);
 *   ring == R  item i may reuse the output buffer of item i - R ("decode back
 *              to back into reused buffers"): a unit of item i starts only
 *              after every unit of item i - R has finished.  The wait is
 *              bounded (about 2 s); on expiry the unit is skipped and
 *              EP_STATUS_WAIT_TIMEOUT is set, so the call always returns.
 *
 * ep_batch_prepare validates every stream on the host and uploads the item
 * descriptors into the caller's device workspace (d_workspace, 256-byte
 * aligned, at least ep_batch_workspace_bytes(n_items) bytes) with a
 * synchronous copy; the plan is a plain host struct.  ep_batch_decode then
 * zeroes the workspace counters and *d_status on `stream` and launches one
 * kernel; it may be called repeatedly (and captured in a CUDA graph) while
 * the workspace, the streams and the outputs stay alive.  Calls that share a
 * workspace must not overlap on the GPU.
 */
typedef struct {
    const uint8_t *h_blob; /* host copy of the stream */
    const void *d_blob;    /* device copy, 16-byte aligned */
    size_t bytes;
    void *d_out;            /* rows x cols container elements, 16-byte aligned */
    float *d_row_scale_out; /* FP8/INT8: rows floats t_r (or NULL) */
} ep_batch_item;

typedef struct {
    int64_t n_items, total_units; /* total_units: work units (32 tile groups) of all items */
    int32_t ring, kind, n_ctx, reserved; /* reserved: set when an item's shape is not whole tiles */
    void *d_workspace;
    size_t workspace_bytes;
    uint64_t items_off, units_off, counters_off;
} ep_batch_plan;

size_t ep_batch_workspace_bytes(int64_t n_items);
ep_status ep_batch_prepare(const ep_batch_item *items, int64_t n_items, int32_t ring, void *d_workspace,
                           size_t workspace_bytes, ep_batch_plan *plan);
ep_status ep_batch_decode(const ep_batch_plan *plan, uint32_t *d_status, ep_stream_t stream);

/*
 * Linear layers ("EntroPack PyTorch Guide", "Replace one linear layer before
 * a whole model": CompressedLinear.from_linear).  Y = X * W^T (+ b) with
 * row-major BF16 X [tokens x cols], W [rows x cols], Y [tokens x rows] and an
 * optional BF16 bias b [rows] (NULL: none); the product is accumulated in
 * fp32 by tcgen05 tensor-core instructions, the bias is added in fp32, and
 * the sum is rounded to BF16 once.  Device pointers are caller-owned and
 * 16-byte aligned; tokens may be any positive count, rows and cols must be
 * multiples of 8.
 * d_status (one u32) is zeroed by the call; the kernel sets
 * EP_STATUS_WAIT_TIMEOUT if an internal pipeline wait gives up (about 2 s),
 * which never happens in a correct run.  Returns EP_OK once enqueued.
 */
typedef enum {
    EP_LINEAR_DECODE_THEN_GEMM = 0, /* decode W into d_ws (rows x cols BF16), then the GEMM */
    EP_LINEAR_FUSED = 1             /* W decoded straight into shared memory as the tensor-core operand and
                                       multiplied there: no workspace (d_ws may be NULL), W never written to
                                       global memory.  Needs cols % 128 == 0; tokens run in passes of
                                       ep_fused_tokens_per_pass(cols) (640 for cols = 3840), each decoding W
                                       again, so it serves few tokens.  EP_ERR_UNSUPPORTED for other shapes */
} ep_linear_mode;

/* Dense BF16 GEMM (uncompressed W): the tensor-core kernel used by
 * ep_compressed_linear, exported so that a compressed layer can be compared
 * with its uncompressed original on the same inputs and the same kernel (the
 * guide keeps an uncompressed baseline beside every compressed result:
 * "EntroPack PyTorch Guide", "Measure memory with clear boundaries" and
 * "Test saved artifacts and reloads before deployment").  Arguments, layout
 * and errors as ep_compressed_linear, with W given as rows x cols BF16. */
ep_status ep_linear_bf16(const uint16_t *d_x, const uint16_t *d_w, uint16_t *d_y, const uint16_t *d_bias,
                         int64_t tokens, int64_t rows, int64_t cols, uint32_t *d_status, ep_stream_t stream);

/*
 * CompressedLinear forward on a lossy BF16 stream (h_blob / d_blob as for
 * ep_decode; rows = out_features, cols = in_features; both multiples of 8).  mode
 * EP_LINEAR_DECODE_THEN_GEMM needs d_ws of at least rows * cols * 2 bytes.
 * Stream corruption found by the decoder shows up in d_status like
 * ep_decode's.  Errors before launch: EP_ERR_INVALID_ARG, EP_ERR_SHAPE,
 * EP_ERR_CORRUPT (host validation), EP_ERR_UNSUPPORTED (lossless or non-BF16
 * stream, or a mode the library does not provide: EP_LINEAR_FUSED).
 */
ep_status ep_compressed_linear(const uint8_t *h_blob, const void *d_blob, size_t bytes, const uint16_t *d_x,
                               int64_t tokens, uint16_t *d_y, const uint16_t *d_bias, int32_t mode, void *d_ws,
                               size_t ws_bytes, uint32_t *d_status, ep_stream_t stream);
ep_status ep_compressed_linear_h(const ep_stream_handle *h, const void *d_blob, const uint16_t *d_x, int64_t tokens,
                                 uint16_t *d_y, const uint16_t *d_bias, int32_t mode, void *d_ws, size_t ws_bytes,
                                 uint32_t *d_status, ep_stream_t stream);

/* Tokens that one pass of EP_LINEAR_FUSED covers for a layer with cols
 * in_features on the current device (every pass decodes W once); 0 when the
 * fused mode does not serve the shape.  The decoder's unit is whole tile rows
 * of W, as many (up to 3) as shared memory holds next to the slot tables; the
 * tensor-memory accumulators (512 columns, 32 per tile row and 128 tokens)
 * bound the tokens of a pass. */
int64_t ep_fused_tokens_per_pass(int64_t cols);

/*
 * Allocation-free variant of ep_batch_prepare + ep_batch_decode.  The pages
 * have no counterpart: this entry point exists for callers that cannot
 * allocate device memory, such as code running under another framework's
 * caching allocator or memory budget, plug-ins inside a host process that
 * owns every allocation, and latency-critical paths where cudaMalloc would
 * synchronise the device.  The batch kernel's scratch (item descriptors, unit
 * table, claim and completion counters) lives in a device array inside the
 * library, sized for EP_BATCH_STATIC_MAX_ITEMS streams (about 177 KB, held
 * on every GPU that loads the library until the process exits).  The caller
 * still passes the streams, the outputs and the status word, exactly as for
 * ep_batch_prepare; ring has the same meaning.
 *  - n_items > EP_BATCH_STATIC_MAX_ITEMS returns EP_ERR_INVALID_ARG before
 *    any work is enqueued; so do the validation errors of ep_batch_prepare.
 *  - No cudaMalloc, cudaFree or other allocating routine is called.  The
 *    descriptors are copied to the device array from host stack memory with
 *    cudaMemcpyAsync on `stream`; for pageable memory that copy may wait for
 *    the stream's earlier work.  The counters are cleared on every call.
 *  - The first call on a device looks up the array's device address with
 *    cudaGetSymbolAddress (with that device current) and caches it; make that
 *    first call before any stream capture.
 *  - Every call shares the one array.  Host threads that call at the same
 *    time are serialised inside the library from the first copy to the
 *    launch, so calls on one stream run one after another.  Calls whose work
 *    overlaps on the GPU (for example on two streams) race on the array and
 *    must be serialised by the caller.
 */
#define EP_BATCH_STATIC_MAX_ITEMS 1024
ep_status ep_batch_decode_static(const ep_batch_item *items, int64_t n_items, int32_t ring, uint32_t *d_status,
                                 ep_stream_t stream);

/* ---- Fixed-width 4-bit comparators (NF4, INT4) ----------------------------
 * The formats EntroPack is evaluated against ("EntroPack: Fast and Accurate
 * Entropy-Coded Weight Compression at Arbitrary Bitrates", Abstract: about 24%
 * lower relative L2 weight error than NF4 at a 4-bit target, with less
 * storage).  Block-absmax 4-bit codebook quantisation:
 *  - the n weights (BF16, any row-major order; n even) form blocks of `block`
 *    consecutive weights (block a multiple of 16; the last block may be short);
 *  - each block stores s = max |w| as FP32 (scales[n / block rounded up]);
 *  - each weight stores the 4-bit code k minimising |w / s - levels[k]| (FP32
 *    arithmetic, ties to the lower k; w / s = 0 when s = 0), packed two per
 *    byte, element 2j in the low nibble of codes[j] (n / 2 bytes);
 *  - reconstruction is BF16(levels[k] * s): one FP32 product, round to
 *    nearest even.  Storage: 4 + 32 / block bits per weight.
 * NF4 levels: standard-normal quantiles at 7 negative and 8 positive evenly
 * spaced probabilities from 1 - d down towards 1/2 (d = (1/32 + 1/30) / 2)
 * plus an exact zero, scaled to [-1, 1], ascending.  INT4 levels: k / 7 for
 * k = -7..7 (index k + 7) and a 16th code equal to 0 that is never chosen. */
typedef enum { EP_Q4_NF4 = 0, EP_Q4_INT4 = 1 } ep_q4_kind;

/* Host: the 16 FP32 levels of `kind` into levels[16].  EP_ERR_INVALID_ARG on a
 * bad kind or NULL. */
ep_status ep_q4_levels(int32_t kind, float *levels);

/* Host: quantise n BF16 weights w (host memory) with levels[16] into codes
 * (n / 2 bytes) and scales (FP32, ceil(n / block)); all caller-owned host
 * buffers.  n_threads <= 0 uses every hardware thread; the result does not
 * depend on it.  Errors: EP_ERR_INVALID_ARG (NULL, block not a positive
 * multiple of 16, non-finite level), EP_ERR_SHAPE (n <= 0 or odd),
 * EP_ERR_NONFINITE (a weight is NaN or +-inf). */
ep_status ep_q4_encode(const uint16_t *w, int64_t n, int64_t block, const float *levels, uint8_t *codes,
                       float *scales, int32_t n_threads);

/* Device: reconstruct the n BF16 weights into d_out (n x 2 bytes) from d_codes
 * (8-byte aligned) and d_scales (device), with levels[16] read from HOST
 * memory at the call.  Asynchronous on `stream`; allocates nothing.  Errors
 * before launch: EP_ERR_INVALID_ARG (NULL, misaligned: d_out needs 16 bytes,
 * d_scales 4; bad block), EP_ERR_SHAPE (n <= 0 or odd); EP_ERR_CUDA if the
 * launch fails. */
ep_status ep_q4_decode(const uint8_t *d_codes, const float *d_scales, int64_t n, int64_t block, const float *levels,
                       uint16_t *d_out, ep_stream_t stream);

/* Per-row-scaled FP8 comparator (8 + 32 / cols bits per weight): row r keeps
 * t_r = max_c |w[r, c]| / 448 as FP32 and each weight the E4M3 byte of
 * w / t_r (FP32 division; 0 when t_r = 0), rounded to nearest even and
 * saturated to +-448; the reconstruction is BF16(e4m3 * t_r), one FP32
 * product rounded to nearest even.
 * Host: encode rows x cols BF16 weights (cols % 8 == 0) into codes (rows *
 * cols bytes) and scales (rows floats), caller-owned host buffers.  Errors:
 * EP_ERR_INVALID_ARG (NULL), EP_ERR_SHAPE, EP_ERR_NONFINITE. */
ep_status ep_fp8_row_encode(const uint16_t *w, int64_t rows, int64_t cols, uint8_t *codes, float *scales,
                            int32_t n_threads);
/* Device: reconstruct into d_out (rows x cols BF16, 16-byte aligned) from
 * d_codes (16-byte aligned) and d_scales; asynchronous on `stream`, allocates
 * nothing.  Errors before launch: EP_ERR_INVALID_ARG, EP_ERR_SHAPE; EP_ERR_CUDA
 * if the launch fails. */
ep_status ep_fp8_row_decode(const uint8_t *d_codes, const float *d_scales, int64_t rows, int64_t cols,
                            uint16_t *d_out, ep_stream_t stream);

/* Synchronise `stream` and map the status word: 0 -> EP_OK, any bit ->
 * EP_ERR_CORRUPT.  A decode that the device found corrupt must stop with a
 * clear error rather than hand back a partly converted tensor ("EntroPack
 * PyTorch Guide", "Test saved artifacts and reloads before deployment":
 * partial failures end in a clear error).  EP_ERR_INVALID_ARG for a NULL
 * status word, EP_ERR_CUDA if the copy or the synchronisation fails. */
ep_status ep_sync_status(const uint32_t *d_status, ep_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* ENTROPACK_H */
