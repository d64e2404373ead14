/*
 * uw.h - C ABI of the lossless BF16 exponent codec with fused decode+matmul.
 *
 * Method: Cloudflare blog post "Unweight" (lossless compression of BF16 model
 * weights, decompressed on-chip inside the matrix multiply).  Each BF16 weight
 * is split into a raw sign+mantissa byte and an exponent byte; the exponent
 * byte is coded against a per-matrix palette of the 16 most frequent exponents
 * (4-bit codes) or with a length-limited canonical Huffman code; any run of 64
 * weights holding an exponent outside the palette is stored verbatim.
 *
 * Conventions for every entry point:
 *   - Every call returns a uw_status; nothing is thrown across the ABI.  On an
 *     error, uw_last_error() returns a message for the calling thread.
 *   - Device pointers are CUDA device addresses on the current device; host
 *     pointers are ordinary process memory.  The caller owns every buffer it
 *     passes (weights, blob, X, Y, workspace); the library owns only what a
 *     uw_matrix holds.
 *   - Device work is enqueued on the given stream (NULL = legacy default
 *     stream) and is asynchronous unless stated otherwise.  No entry point
 *     falls back to the CPU: without a CUDA device they return UW_ERR_CUDA.
 *   - Shapes: W is [N, K] row-major with K % 64 == 0 (a block is 64 weights of
 *     one row); X is [B, K] row-major bf16; Y is [B, N] row-major.  Device
 *     pointers to X, Y and workspaces must be 16-byte aligned.
 *   - Errors found by device kernels (a Huffman stream that overruns its
 *     chunk) are latched in a per-matrix status word and reported by uw_check
 *     and by the next uw_decode / uw_matmul on that matrix.
 */
#ifndef UW_H
#define UW_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, declared without the CUDA headers. */
typedef struct CUstream_st *uw_stream;

typedef enum {
    UW_OK = 0,
    UW_ERR_INVALID_ARG = 1,   /* null pointer, misaligned pointer, bad option value */
    UW_ERR_SHAPE = 2,         /* K % 64 != 0, negative sizes, B < 0, size overflow */
    UW_ERR_UNSUPPORTED = 3,   /* strategy not available for this matrix / batch */
    UW_ERR_CORRUPT = 4,       /* blob failed validation, or a device decoder found a bad stream */
    UW_ERR_NO_MEMORY = 5,     /* host or device allocation failed */
    UW_ERR_WORKSPACE = 6,     /* workspace smaller than uw_workspace_size reports */
    UW_ERR_CUDA = 7,          /* a CUDA runtime call failed (message in uw_last_error) */
    UW_ERR_TIMEOUT = 8,       /* a bounded device wait expired */
    UW_ERR_BUFFER_TOO_SMALL = 9 /* host output buffer too small; required size returned */
} uw_status;

typedef enum { UW_CODEC_PALETTE = 0, UW_CODEC_HUFFMAN = 1 } uw_codec;

/*
 * Execution strategies: the four pipelines of the "Unweight" post (section on
 * the four execution pipelines), and a fifth that decodes inside the GEMV:
 *   FULL_DECODE        rebuild the whole BF16 matrix into the workspace, then a
 *                      plain BF16 GEMV/GEMM (the post uses cuBLAS; here a
 *                      hand-written kernel).
 *   EXP_ONLY           a preprocess kernel writes only the exponent bytes into
 *                      the workspace; the fused kernel joins them with the raw
 *                      sign+mantissa bytes.
 *   PALETTE_TRANSCODE  a preprocess kernel turns the Huffman stream into 4-bit
 *                      palette codes in the workspace; the fused kernel rebuilds
 *                      BF16 from them.
 *   DIRECT_PALETTE     no preprocessing: the fused kernel reads resident 4-bit
 *                      codes (palette codec, or a Huffman matrix loaded with its
 *                      palette form).
 *   HUFFMAN_DIRECT     no preprocessing and no palette form: one GEMV kernel
 *                      decodes the Huffman stream itself (the lookup table in
 *                      shared memory, as in the post's section on the decode
 *                      kernels) and multiplies the rebuilt weights straight away.
 *                      Huffman codec only, code lengths <= 12, chunk_weights a
 *                      divisor of K of at most 2048, 1 <= B <= 8; runs on
 *                      UW_KERNEL_GEMV with split_k 0/1 and variant 0 (plain
 *                      loads) or 1 (each work unit also prefetched into L2 in
 *                      bulk one unit ahead).  It goes beyond the post's four
 *                      pipelines.
 *   AUTO               the autotuned choice for (matrix, B), else a default:
 *                      DIRECT_PALETTE when the palette form is resident, else
 *                      HUFFMAN_DIRECT where it applies, else PALETTE_TRANSCODE.
 */
typedef enum {
    UW_STRAT_AUTO = 0,
    UW_STRAT_FULL_DECODE = 1,
    UW_STRAT_EXP_ONLY = 2,
    UW_STRAT_PALETTE_TRANSCODE = 3,
    UW_STRAT_DIRECT_PALETTE = 4,
    UW_STRAT_HUFFMAN_DIRECT = 5
} uw_strategy;

typedef enum { UW_OUT_F32 = 0, UW_OUT_BF16 = 1 } uw_out_dtype;

/*
 * What uw_load keeps on the device for a Huffman blob (a palette blob always
 * keeps its 4-bit codes and has no stream):
 *   UW_RESIDENT_HUFFMAN  the Huffman stream alone (the smallest form; the
 *                        Huffman-fed pipelines and HUFFMAN_DIRECT run on it)
 *   UW_RESIDENT_BOTH     the stream and the 4-bit palette form
 *   UW_RESIDENT_PALETTE  the 4-bit palette form alone: the stream is transcoded
 *                        at load time (the post's direct-palette form) and then
 *                        dropped, so PALETTE_TRANSCODE and HUFFMAN_DIRECT are not
 *                        available
 * Matching the post's results section, the choice trades footprint against
 * speed: the stream is about 10.8 bits per weight on Gaussian weights, the
 * palette form about 12.1.
 */
typedef enum { UW_RESIDENT_HUFFMAN = 0, UW_RESIDENT_BOTH = 1, UW_RESIDENT_PALETTE = 2 } uw_resident;

/* Matmul kernel families. */
typedef enum {
    UW_KERNEL_AUTO = 0,
    UW_KERNEL_GEMV = 1,      /* matrix-vector kernels for small B (see uw_plan.variant) */
    UW_KERNEL_TC = 2         /* tcgen05 tensor-core GEMM, W rebuilt in shared memory, fp32 in TMEM */
} uw_kernel;

typedef struct {
    uint32_t codec;          /* uw_codec */
    uint32_t chunk_weights;  /* Huffman chunk size in weights: multiple of 64, >= 64 (default 256) */
    uint32_t max_code_len;   /* Huffman length limit, 4..15 (default 12) */
} uw_encode_opts;

/* One execution plan: what uw_matmul runs for a given (matrix, B). */
typedef struct {
    int32_t strategy;        /* uw_strategy, never AUTO inside a stored plan */
    int32_t kernel;          /* uw_kernel */
    int32_t split_k;         /* K-splits (>= 1); 0 = kernel's default */
    int32_t variant;         /* kernel-specific launch shape; 0 = default.  UW_KERNEL_GEMV:
                              *   0, 2..5: bulk-copy GEMV, fp32 FMA on CUDA cores, B <= 2 (0: 8 consumer warps,
                              *            2 CTAs/SM; 2: 16 warps, 1 CTA/SM; 3: 8 warps, 1 CTA/SM in half the
                              *            shared memory; 4, 5: as 0, 2 with 64 weights per lane)
                              *   1:       plain-load GEMV, any B (batch groups of up to 8)
                              *   6, 7:    GEMV on the tensor pipe (mma.sync, fp32 accumulate), B <= 16,
                              *            K a multiple of 256 (6: K-slices of 4096 weights up to B = 8;
                              *            7: of 2048)
                              *   8:       GEMV on the tensor pipe, B <= 64, K a multiple of 256: one CTA per
                              *            SM walks an even share of the 128-row x 256-weight units, each warp
                              *            owning 8 rows (split_k ignored)
                              * UW_KERNEL_TC: 0, 1: one CTA per 128-row tile and K-slice, rebuilt tiles in shared
                              *   memory; 4: one CTA per SM over an even share of the 128-row x 256-weight units,
                              *   each 64-weight step rebuilt into shared memory (B <= 512, K a multiple of 256,
                              *   4-bit codes, split_k ignored); other values run as 0
                              * a shape that does not fit the matrix or B runs the nearest one that does */
} uw_plan;

typedef struct {
    int64_t N, K;
    uint32_t codec;
    uint32_t n_pal;
    uint8_t palette[16];
    uint8_t code_len[16];
    uint64_t n_blocks, n_verbatim, n_chunks, total_bits;
    uint64_t blob_bytes;     /* size of the serialized blob */
    uint64_t device_bytes;   /* device memory held by the uw_matrix */
    int32_t has_palette_form;/* 4-bit codes resident (DIRECT_PALETTE available) */
    int32_t chunk_weights, max_code_len;
    int32_t has_huffman_stream; /* the Huffman stream is resident (PALETTE_TRANSCODE, HUFFMAN_DIRECT available) */
} uw_info;

typedef struct uw_matrix uw_matrix;

/*
 * uw_encode - encode W[N,K] (host bf16 bit patterns, row-major) into a blob.
 *   Passages: BF16 anatomy (sign+mantissa byte kept raw), exponent statistics
 *   (top-16 palette), Huffman coding of the exponent byte, verbatim 64-weight
 *   runs.  Host-only, pure and deterministic: the bytes are a function of
 *   (W, opts) alone.  opts == NULL means palette codec.
 *   out == NULL: only *out_size is written (required size).  out != NULL and
 *   out_cap < required: UW_ERR_BUFFER_TOO_SMALL with *out_size = required.
 *   Errors: UW_ERR_SHAPE (K % 64, negative sizes), UW_ERR_INVALID_ARG (bad
 *   options), UW_ERR_UNSUPPORTED (Huffman stream of 2^32 bits or more).
 */
uw_status uw_encode(const uint16_t *w_host, int64_t N, int64_t K, const uw_encode_opts *opts,
                    void *out, size_t out_cap, size_t *out_size);

/*
 * uw_load - validate a blob fully on the host (magic, version, sizes, section
 *   bounds and alignment, bitmap/prefix/verbatim consistency, code lengths and
 *   Kraft sum, chunk offsets) and copy it to device memory owned by the new
 *   uw_matrix.  `resident` (uw_resident) says what stays on the device for a
 *   Huffman blob; any form with the palette codes runs the post's load-time
 *   transcode of the stream into 4-bit codes.  Blocks the host until the
 *   upload on `stream` is done, so the caller may free `blob` on return.
 *   uw_get_info reports the device bytes the matrix holds.
 *   Errors: UW_ERR_INVALID_ARG (resident out of range), UW_ERR_CORRUPT
 *   (validation), UW_ERR_NO_MEMORY, UW_ERR_CUDA.
 */
uw_status uw_load(const void *blob, size_t size, int resident, uw_stream stream, uw_matrix **out);

/*
 * uw_blob_validate - the host-side checks of uw_load without any device work
 *   (usable on a machine without a GPU).  info may be NULL.
 *   Errors: UW_ERR_CORRUPT with the first failed check in uw_last_error().
 */
uw_status uw_blob_validate(const void *blob, size_t size, uw_info *info);

/* uw_free - release a uw_matrix and its device memory.  As with cudaFree (which it calls, and which waits for
 * work still running on the device), no work that reads the matrix may be enqueued after it.  NULL is a no-op. */
void uw_free(uw_matrix *m);

/* uw_get_info - header facts and memory footprint of a loaded matrix. */
uw_status uw_get_info(const uw_matrix *m, uw_info *out);

/*
 * uw_decode - rebuild W[N,K] bf16 (bit-exact, the post's lossless claim) into
 *   caller-owned device memory w_dev (N*K*2 bytes, 16-byte aligned).
 *   Asynchronous on `stream`.  Errors: UW_ERR_INVALID_ARG, UW_ERR_CORRUPT (a
 *   device error latched by an earlier call), UW_ERR_CUDA.
 */
uw_status uw_decode(const uw_matrix *m, uint16_t *w_dev, uw_stream stream);

/*
 * uw_workspace_size - device workspace bytes uw_matmul needs for (m, B,
 *   strategy) (AUTO: the plan AUTO would pick; an explicit strategy: that
 *   strategy with the kernel and launch shape AUTO would pair with it at this B).
 *   0 is a valid answer.  The workspace holds a preprocess output, an fp32
 *   accumulator [B,N] and 24 bytes per 128 rows of W; its contents need no
 *   initialisation (the tensor-core kernel tags the cells it shares between
 *   its CTAs with a per-launch epoch, and clears them before it ends, so a
 *   CUDA graph that replays the call finds them clear).  A call owns its
 *   workspace until `stream` has passed it: calls that may overlap take
 *   separate workspaces.  If a call ends with UW_ERR_TIMEOUT in uw_check, a
 *   graph replay of it on the same workspace may find stale cells.
 */
uw_status uw_workspace_size(const uw_matrix *m, int64_t B, uw_strategy strategy, size_t *bytes);

/*
 * uw_matmul - Y[B,N] = X[B,K] . W^T with W decoded on-chip (the post's
 *   reconstructive matmul; fp32 accumulation).  x_dev: [B,K] bf16 device;
 *   y_dev: [B,N] fp32 or bf16 (RNE) device; workspace: device scratch of at
 *   least uw_workspace_size bytes (may be NULL if that size is 0).  B == 0 is a
 *   no-op.  Asynchronous on `stream`.
 *   Errors: UW_ERR_INVALID_ARG, UW_ERR_SHAPE, UW_ERR_UNSUPPORTED (e.g.
 *   DIRECT_PALETTE without resident codes), UW_ERR_WORKSPACE, UW_ERR_CORRUPT,
 *   UW_ERR_CUDA.
 */
/*   AUTO runs the autotuned plan for B's bucket, else the default plan; an explicit
 *   strategy runs with the default kernel and launch shape for that strategy and B. */
uw_status uw_matmul(const uw_matrix *m, const uint16_t *x_dev, int64_t B, void *y_dev, uw_out_dtype out_dtype,
                    uw_strategy strategy, void *workspace, size_t ws_bytes, uw_stream stream);

/* uw_matmul_plan - as uw_matmul, with an explicit plan (strategy, kernel, split, variant). */
uw_status uw_matmul_plan(const uw_matrix *m, const uint16_t *x_dev, int64_t B, void *y_dev, uw_out_dtype out_dtype,
                         const uw_plan *plan, void *workspace, size_t ws_bytes, uw_stream stream);

/* uw_plan_workspace_size - workspace bytes for an explicit plan. */
uw_status uw_plan_workspace_size(const uw_matrix *m, int64_t B, const uw_plan *plan, size_t *bytes);

/* uw_plan_for - the plan AUTO runs for (m, B): the autotuned entry for B's
 *   bucket if one exists, else a default rule. */
uw_status uw_plan_for(const uw_matrix *m, int64_t B, uw_plan *out);

/*
 * uw_matmul_host - end-to-end form of uw_matmul with HOST X and Y: copies
 *   x_host ([B,K] bf16) to the device, runs the plan AUTO picks, copies Y back
 *   into y_host and synchronises `stream` before returning.  workspace must be
 *   a device buffer of at least uw_host_workspace_size bytes (it also holds
 *   the device copies of X and Y).  Pinned host memory gives the fastest copies.
 */
uw_status uw_matmul_host(const uw_matrix *m, const uint16_t *x_host, int64_t B, void *y_host,
                         uw_out_dtype out_dtype, void *workspace, size_t ws_bytes, uw_stream stream);
uw_status uw_host_workspace_size(const uw_matrix *m, int64_t B, uw_out_dtype out_dtype, size_t *bytes);

/*
 * uw_matmul_host_async - uw_matmul_host without the final synchronisation: the
 *   copy of X, the matmul and the copy of Y back are enqueued on `stream` and
 *   the call returns.  x_host must stay unchanged, and y_host unread, until
 *   the stream has passed the copy back (synchronise the stream or an event
 *   recorded after the call); the workspace belongs to the call until then.
 *   With pinned host buffers and two streams, one call's copies overlap the
 *   other's matmul.  Errors as uw_matmul_host.
 */
uw_status uw_matmul_host_async(const uw_matrix *m, const uint16_t *x_host, int64_t B, void *y_host,
                               uw_out_dtype out_dtype, void *workspace, size_t ws_bytes, uw_stream stream);

/*
 * uw_matmul_noalloc - uw_matmul with the palette-transcode pipeline
 *   (UW_STRAT_PALETTE_TRANSCODE on the GEMV kernel) that allocates nothing and
 *   takes no workspace.  The Unweight post has no counterpart to this entry
 *   point; it exists for callers that cannot call cudaMalloc - an engine whose
 *   allocator reserved all device memory at start-up, or a latency-critical
 *   path that must not take the device synchronisation cudaMalloc / cudaFree may
 *   imply.  Its scratch (the transcoded 4-bit codes, plus the fp32 accumulator a
 *   K-split may need) is a library-owned static device array of 36 MiB, held on
 *   every GPU that loads the library until the process exits.
 *   m must be a Huffman-coded matrix; x_dev, y_dev, B and out_dtype are as in
 *   uw_matmul.  The array's device address is looked up (cudaGetSymbolAddress)
 *   by the first call in each CUDA context - the device's primary context, or
 *   one a driver-API caller made current - and cached under that context's
 *   unique id, so a call after cudaDeviceReset looks it up again.  Make the
 *   first call in a context before any stream capture.  All calls share the
 *   one array and it keeps the last call's contents (the accumulator is
 *   cleared on the stream before each use): calls whose GPU work overlaps
 *   (different streams, or different threads without ordering) race on it.
 *   Errors: UW_ERR_WORKSPACE when N*K/2 plus B*N*4 plus 24 bytes per 128 rows
 *   (each rounded up to 256 bytes, with 64 bytes of padding on the codes)
 *   exceeds the 36 MiB array;
 *   UW_ERR_UNSUPPORTED for a palette-codec matrix; otherwise as uw_matmul.
 */
uw_status uw_matmul_noalloc(const uw_matrix *m, const uint16_t *x_dev, int64_t B, void *y_dev, uw_out_dtype out_dtype,
                            uw_stream stream);

/*
 * uw_autotune - for each batch size in batches[0..n_batches), time the
 *   candidate plans on this GPU (CUDA events on `stream`, several repetitions,
 *   median) by coordinate descent over strategy, kernel, split and variant (the
 *   post's autotuner: measure real throughput, vary one choice at a time until
 *   nothing improves), and store the fastest in the matrix's tune table, keyed
 *   by batch bucket.  workspace must hold uw_workspace_size for every candidate
 *   (uw_autotune_workspace_size).  Synchronous.  Writes scratch outputs only
 *   into the workspace.  It also allocates, for the duration of the call, a
 *   device buffer of twice the L2 size that it rewrites before each timed
 *   launch, so candidates are timed with their weights coming from HBM (if
 *   that allocation fails, timing proceeds without it).
 */
uw_status uw_autotune(uw_matrix *m, const int64_t *batches, int n_batches, void *workspace, size_t ws_bytes,
                      uw_stream stream);
uw_status uw_autotune_workspace_size(const uw_matrix *m, const int64_t *batches, int n_batches, size_t *bytes);

/*
 * uw_tune_save / uw_tune_load - the tune table as text, one line per batch
 *   bucket: "B strategy kernel split_k variant us".  save: buf == NULL returns
 *   the length in *len.  load replaces the table; it rejects malformed lines
 *   with UW_ERR_INVALID_ARG and leaves the table unchanged.
 */
uw_status uw_tune_save(const uw_matrix *m, char *buf, size_t cap, size_t *len);
uw_status uw_tune_load(uw_matrix *m, const char *text);

/* One matmul of a sequence: Y[B,N] = X[B,K] . W^T for the loaded matrix m; x and y are device pointers as in
 * uw_matmul, out_dtype a uw_out_dtype; flags 0 or UW_STEP_CONCURRENT. */
typedef struct {
    const uw_matrix *m;
    const uint16_t *x;
    void *y;
    int32_t out_dtype;
    int32_t flags;
} uw_step;

/* The step may run at the same time as the steps before it back to the last step without the flag: it reads
 * nothing those steps write and writes nothing they read or write (an MLP's up projection beside its gate
 * projection: both read the layer's input).  Such a run forms a group.  The flag permits overlap; a schedule
 * with UW_SEQ_GROUPS runs each group's matmuls on streams of their own (the first four members on four streams,
 * any further member after the member four places before it), any other schedule runs them in order. */
#define UW_STEP_CONCURRENT 1

/*
 * uw_sequence_run - run n matmuls in order at batch B (the post's section on scheduling hard and easy layers).
 *   A step is "hard" when its matrix holds only its Huffman stream (UW_RESIDENT_HUFFMAN): its 4-bit palette codes
 *   are transcoded on `side_stream` into one of two slots of the workspace (double buffering), as soon as the
 *   slot's previous matmul is done, so the transcode of the next hard step runs while the main stream works on
 *   the steps before it.  Its matmul on `stream` waits for that transcode and reads the codes (the direct-palette
 *   kernels).  Steps whose matrix holds its palette form run their AUTO plan.  Asynchronous: everything is enqueued
 *   at once and ordered by events; `stream` ends joined with `side_stream`, so the call can be captured into one
 *   CUDA graph from `stream`.  `side_stream` must differ from `stream` when a step is hard.  The workspace
 *   (uw_sequence_workspace_size bytes, 256-byte aligned) belongs to the sequence until `stream` has passed it.
 *   The first call in a thread on a device creates the events the calls use; make it before any stream capture.
 *   The steps' x and y must not overlap a later step's inputs unless the caller wants that chaining: steps run in
 *   order on `stream`, except that under a UW_SEQ_GROUPS schedule a group of steps joined by UW_STEP_CONCURRENT
 *   runs on `stream` and on streams the library keeps per thread and device (forked from and joined back to
 *   `stream` with events, so a graph captured from `stream` holds them).  Each member of a group has its own part
 *   of the workspace (the size covers both forms).  With the transcode schedule a hard step always waits for the
 *   steps before it (the flag is not applied to it).
 *   Errors: UW_ERR_INVALID_ARG, UW_ERR_WORKSPACE, UW_ERR_CUDA, or a step's uw_matmul error.
 */
/*   decode_sms: the post's decode-vs-matmul SM split.  0: every launch sizes its grid for all SMs.  d > 0: the
 *   main stream's persistent matmul grids are sized for the device's SMs minus d, and each transcode is a
 *   persistent grid of d SMs' worth of CTAs, so the two run side by side.  UW_SEQ_DIRECT (-1): no side-stream
 *   transcode; every step runs its own AUTO plan on `stream` (a hard step at B <= 8: the Huffman-direct GEMV;
 *   `side_stream` is not used).  Any of these plus UW_SEQ_GROUPS: the same schedule with the groups of
 *   UW_STEP_CONCURRENT steps overlapped.  Must lie in [-1, SMs) or in UW_SEQ_GROUPS + [-1, SMs).
 */
#define UW_SEQ_DIRECT (-1)
#define UW_SEQ_GROUPS 65536
uw_status uw_sequence_workspace_size(const uw_step *steps, int n, int64_t B, size_t *bytes);
uw_status uw_sequence_run(const uw_step *steps, int n, int64_t B, void *workspace, size_t ws_bytes, uw_stream stream,
                          uw_stream side_stream, int decode_sms);

/*
 * uw_sequence_tune - time uw_sequence_run over these steps (same arguments) for the direct schedule and a range of
 *   decode SM splits (UW_SEQ_DIRECT, 0, 8, 16, ..., 96; CUDA events on `stream`, median of three runs after two),
 *   each also with UW_SEQ_GROUPS when a step carries UW_STEP_CONCURRENT, and return the fastest in *decode_sms
 *   (the post's tuning of the decoder's share of the SMs).  Synchronous; runs the sequence 5 times per
 *   candidate, writing the steps' outputs.
 */
uw_status uw_sequence_tune(const uw_step *steps, int n, int64_t B, void *workspace, size_t ws_bytes, uw_stream stream,
                           uw_stream side_stream, int *decode_sms);

/* uw_check - synchronise `stream` and report (then clear) the matrix's device status word. */
uw_status uw_check(const uw_matrix *m, uw_stream stream);

/* Human-readable name of a status code (static storage). */
const char *uw_status_string(uw_status s);

/* Last error message of the calling thread ("" if none). */
const char *uw_last_error(void);

/* Library build string (version, target architecture). */
const char *uw_version(void);

#ifdef __cplusplus
}
#endif

#endif /* UW_H */
