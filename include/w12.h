/*
 * w12.h -- C ABI of the W12 library: lossless 12-bit storage of BF16 weights
 * and the skinny-M GEMM (1..256 activation rows) that decodes it on the fly on
 * one GB300 GPU (sm_103a).
 *
 * Sources (pages about "SpecPilot: Autonomous Algorithm Discovery and Systems
 * Optimization for Speculative Decoding"):
 *   [F5a] thelatestinai.com page, Figure 5(a) caption -- the format: per BF16
 *         weight three 4-bit planes A (sign + top three mantissa bits), E
 *         (exponent offset in a 16-binade window per output channel) and B
 *         (low mantissa bits); weights outside the window go to an exact
 *         escape list; A and E form the 8-bit view read by the Q pass.
 *   [F5b] same page, Figure 5(b) caption -- the GEMM decodes W12 records on
 *         the fly and feeds the tensor cores.
 *   [F7]  same page, Figure 7 caption -- the Q pass reads the 8-bit view
 *         nested in each W12 record.
 *   [MF]  ai.info "AI summary" page, Main Findings -- "W12 compression"
 *         (lossless, 12.01-12.02 bits/weight, 7.3e-5 escapes) and "W12 works
 *         beyond speculation" (the W12 GEMM against cuBLAS at 1 and 32 rows).
 *   [KC3] ai.info page, Key Contributions 3 -- the zero-copy Q pass.
 *
 * Conventions shared by every call:
 *   - W is [N][K] row-major BF16 (raw 16-bit patterns): row n = output
 *     channel n.  x is [M][K] row-major BF16, y is [M][N] row-major FP32,
 *     y = x . W^T.
 *   - Layout of an encoded matrix: AE byte = A<<4|E per weight, B packed 8 weights per little-endian 32-bit word (evens in
 *     nibble slots 0..3, odds in 4..7), window = 16 binades ending at the
 *     row's largest finite normal exponent, escapes grouped by 128 x 256 tile
 *     as (row%128)<<24 | (k%256)<<16 | bits, sorted inside each tile.
 *   - Errors are returned as w12_status; no call aborts or throws.  Device
 *     calls are asynchronous on the given stream and never synchronise,
 *     except w12_dev_status.
 *   - Streams are CUDA runtime streams (cudaStream_t); NULL = legacy default.
 *   - Host-side objects are opaque and owned by the library; free them with
 *     the matching *_free call.  Caller-provided buffers stay caller-owned.
 */
#ifndef W12_H
#define W12_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *w12_stream_t; /* same type as cudaStream_t */

typedef enum {
    W12_OK = 0,
    W12_ERR_INVALID_ARG = 1, /* NULL pointer or negative size               */
    W12_ERR_SHAPE = 2,       /* N/K disagree with the encoded matrix         */
    W12_ERR_ALIGNMENT = 3,   /* a device buffer is not 16-byte aligned       */
    W12_ERR_UNSUPPORTED = 4, /* M outside 0..256, K % 32 != 0 for the GEMM   */
    W12_ERR_OOM = 5,         /* host or device allocation failed             */
    W12_ERR_CUDA = 6,        /* a CUDA runtime/driver call failed            */
    W12_ERR_CORRUPT = 7,     /* an encoded matrix breaks a format invariant  */
    W12_ERR_TIMEOUT = 8,     /* a kernel gave up waiting (device status)     */
    W12_ERR_IO = 9           /* file could not be read or written            */
} w12_status;

typedef struct w12_host w12_host; /* encoded matrix in host memory   */
typedef struct w12_dev w12_dev;   /* encoded matrix in device memory */

typedef struct {
    int64_t N, K;
    int64_t n_escapes;
    int64_t n_tiles;              /* 128 x 256 escape tiles               */
    int64_t max_escapes_per_tile;
    double bits_per_weight;       /* 8 * blob bytes / (N K), incl. header */
    double escape_fraction;       /* n_escapes / (N K)                    */
    size_t bytes_total;           /* blob bytes (header + all arrays)     */
    size_t bytes_ae, bytes_b;     /* the two plane arrays                 */
} w12_stats;

/* Human-readable name of a status code (static string). */
const char *w12_status_string(w12_status s);

/* ---- host side ------------------------------------------------------------ */

/*
 * Encode W[N][K] (host, row-major BF16 bit patterns) into W12 [F5a], losslessly
 * [MF].  N, K >= 0 (empty matrices are valid).  n_threads: worker threads, 0 =
 * all hardware threads.  Synchronous, host-only; *out receives a new handle.
 * Errors: INVALID_ARG (NULL, negative size), OOM.
 */
w12_status w12_encode(const uint16_t *w_bf16, int64_t N, int64_t K, int n_threads,
                      w12_host **out);

/* Flags of w12_encode_ex / w12_encode_device_ex. */
enum {
    W12_ENCODE_COUNT_MAX = 1 /* count-maximising windows instead of max-anchored ones */
};

/*
 * w12_encode with flags (an unknown bit gives INVALID_ARG).
 *
 * W12_ENCODE_COUNT_MAX chooses each row's window as the 16 binades holding
 * the most of its finite normal weights -- the highest such window at or
 * below the max-anchored one -- instead of the window topped by the row's
 * largest weight [F5a].  On heavy-tailed rows this trades a few top outliers
 * for many fewer escapes (Student-t(1.5) weights: about 1e-2 -> 2e-3).  The
 * weights above the window escape too; their slot holds the saturated
 * placeholder A = s<<3 | 7, E = 15, B = 15, the window's largest magnitude
 * with the weight's sign, which is what the Q pass reads for them.  The
 * stored format, decoding and the exact GEMM are the same: the blob records
 * each row's base, and w12_validate accepts both placeholders.  (The pages'
 * encoder anchors the window at the maximum; this option is a library
 * extension.)
 */
w12_status w12_encode_ex(const uint16_t *w_bf16, int64_t N, int64_t K, int n_threads, unsigned flags,
                         w12_host **out);

void w12_host_free(w12_host *h);

/* Storage statistics of an encoded matrix [MF "W12 compression"]. */
w12_status w12_host_stats(const w12_host *h, w12_stats *out);

/*
 * Borrow the arrays of an encoded matrix (valid until w12_host_free):
 * ebase[N] (window base per row), ae[N*K] (A<<4|E bytes), b[N*brow] with
 * brow = 4*ceil(K/8), tile_ptr[T+1], esc[n_escapes].  Any output may be NULL.
 */
w12_status w12_host_view(const w12_host *h, const uint8_t **ebase, const uint8_t **ae,
                         const uint8_t **b, const uint32_t **tile_ptr, const uint32_t **esc);

/* Check every invariant of the format; W12_ERR_CORRUPT on the first breach. */
w12_status w12_validate(const w12_host *h);

/*
 * Serialise into the portable blob ("W12\0", version 1, N, K, n_esc, T, then
 * ebase, AE, B, tile_ptr, escapes; little-endian).  buf == NULL queries the
 * size into *len.  Errors: INVALID_ARG (cap too small).
 */
w12_status w12_serialize(const w12_host *h, uint8_t *buf, size_t cap, size_t *len);

/* Parse and validate a blob into a new host handle (CORRUPT if malformed). */
w12_status w12_deserialize(const uint8_t *buf, size_t len, w12_host **out);

/* Blob + CRC-32 trailer to/from a file (IO, CORRUPT on a bad checksum). */
w12_status w12_save(const w12_host *h, const char *path);
w12_status w12_load(const char *path, w12_host **out);

/* ---- device side ------------------------------------------------------------ */

/*
 * Copy an encoded matrix to the current CUDA device: one device allocation
 * holding every array (256-byte aligned), filled by asynchronous copies on
 * `stream` (the host handle must stay alive until the stream has passed
 * them).  Errors: INVALID_ARG, OOM, CUDA.
 */
w12_status w12_upload(const w12_host *h, w12_stream_t stream, w12_dev **out);

/* Free a device handle (synchronises with the device first). */
void w12_dev_free(w12_dev *d);

/*
 * Encode on the device: BF16 weights w_bf16 (device memory, [N][K] row-major,
 * caller-owned) become a device handle whose arrays are byte-identical to
 * w12_upload(w12_encode(...)) of the same weights [F5a] -- conversion of a
 * checkpoint already on the GPU without a round trip through the host.  Runs
 * on `stream` and synchronises with it (the handle's size depends on the
 * number of escapes).  N = 0 or K = 0 gives an empty handle.  Errors:
 * INVALID_ARG, UNSUPPORTED (N or K above 2^31), OOM, CUDA.
 */
w12_status w12_encode_device(const void *w_bf16, int64_t N, int64_t K, w12_stream_t stream, w12_dev **out);

/* w12_encode_device with the flags of w12_encode_ex; the arrays are
 * byte-identical to w12_encode_ex's with the same flags. */
w12_status w12_encode_device_ex(const void *w_bf16, int64_t N, int64_t K, unsigned flags, w12_stream_t stream,
                                w12_dev **out);

/*
 * Copy a device handle's arrays back into a new host handle (for
 * w12_serialize / w12_save of a matrix encoded on the device).  Synchronises
 * with `stream`.  Errors: INVALID_ARG, OOM, CUDA.
 */
w12_status w12_download(const w12_dev *d, w12_stream_t stream, w12_host **out);

/* Shape and device-byte count of a device handle. */
w12_status w12_dev_info(const w12_dev *d, int64_t *N, int64_t *K, size_t *device_bytes);

/*
 * y[M][N] = x[M][K] . W^T with W decoded to exact BF16 on the fly [F5a, F5b]
 * and FP32 accumulation.  x: device BF16 [M][K], 16-byte aligned; y: device
 * FP32 [M][N], 16-byte aligned; both caller-owned.  1 <= M <= 256 (M = 0 is
 * a no-op), N and K must equal the handle's; K % 32 == 0 (else UNSUPPORTED).
 * Kernel choice is a function of M only: M <= 2 CUDA-core FMAs with warp
 * reductions, 3..256 tcgen05 tensor cores with TMEM accumulators (one
 * launch; every weight is read once).  Uses a
 * library-owned workspace cached per (device, stream); the first call on a
 * stream allocates it (stream-ordered), so make that first call outside any
 * stream capture.  It holds the partial sums of M = 128 on every SM; a later
 * uncaptured call that needs more (M > 128) moves the stream to a larger
 * workspace, and the old one stays allocated until w12_release_workspaces, so
 * CUDA graphs captured earlier keep valid addresses (capturing a call that
 * would need to grow fails with UNSUPPORTED).  Release workspaces only when
 * no captured graph that uses them will be replayed again.  Errors:
 * INVALID_ARG, SHAPE, ALIGNMENT, UNSUPPORTED, OOM, CUDA.  Device-side
 * failures are reported by w12_dev_status.
 */
w12_status w12_gemm(const void *x_bf16, const w12_dev *w, float *y, int M, int N, int K,
                     w12_stream_t stream);

/*
 * The Q pass [F7, KC3]: the same product over the nested 8-bit view only --
 * each weight rebuilt from its A+E byte with B = 0 and escapes left as their
 * placeholders.  Reads 1 byte per weight and nothing else of the matrix.
 * Same arguments, limits and errors as w12_gemm.
 */
w12_status w12_gemm_q8view(const void *x_bf16, const w12_dev *w, float *y, int M, int N, int K,
                           w12_stream_t stream);

/*
 * The launch a GEMM of M x N x K makes on a GPU with `sm_count` SMs (0: the
 * current device's), without running it -- the same planning w12_gemm uses.
 * kernel: 1 the CUDA-core kernel (M <= 2), 2 the tensor-core kernel; 0 when
 * nothing is launched (M, N or K zero).  The weights are split into
 * row_blocks x k_steps units of block_rows x 256; split_row_blocks counts row
 * blocks shared by several CTAs, whose partial sums a split-K fix-up combines
 * (inside the GEMM, or as a second kernel when separate_fixup is 1), using
 * partial_bytes of scratch.  Errors: INVALID_ARG, UNSUPPORTED (as w12_gemm:
 * M above 256, K % 32 != 0), CUDA (no device to ask for its SM count).
 */
typedef struct {
    int kernel;
    int tile_rows;       /* activation rows per tile: 1, 2, 16, 32, 64, 128 or 256 */
    int block_rows;      /* weight rows per row block: 64 or 128 */
    int grid;            /* CTAs */
    int64_t row_blocks;
    int64_t k_steps;
    int64_t split_row_blocks;
    int separate_fixup;
    size_t partial_bytes;
} w12_gemm_plan_t;

w12_status w12_gemm_plan(int M, int64_t N, int64_t K, int sm_count, w12_gemm_plan_t *out);

/*
 * The launch w12_gemm_grouped makes for n matrices of Ns[i] rows (all with K
 * columns), M activation rows and `sm_count` SMs: the row blocks of all of
 * them end to end (row_blocks is their total), the rest as w12_gemm_plan.
 * 1 <= n <= W12_MAX_GROUP; a group of one plans as w12_gemm_plan.  Errors:
 * INVALID_ARG (no Ns, n out of range, a negative size), UNSUPPORTED and CUDA
 * as w12_gemm_plan.
 */
w12_status w12_gemm_plan_grouped(int M, const int64_t *Ns, int n, int64_t K, int sm_count, w12_gemm_plan_t *out);

/* Flags of w12_gemm_ex. */
enum {
    W12_GEMM_Q8VIEW = 1,      /* the Q pass (as w12_gemm_q8view) instead of the exact GEMM */
    W12_GEMM_INPUT_READY = 2, /* x was complete before the previous operation on the stream started */
    W12_GEMM_OUT_BF16 = 4,    /* y is BF16: each FP32 result rounded to nearest, ties to even */
    W12_GEMM_SILU_MUL = 8     /* gated-MLP product of row pairs (gate 2i, up 2i+1): y is [M][N/2] */
};

/*
 * w12_gemm / w12_gemm_q8view with flags.  Arguments, limits and errors are
 * w12_gemm's, with y's element type and row length set by the flags: FP32
 * [M][N] by default; BF16 under W12_GEMM_OUT_BF16; [M][N/2] under
 * W12_GEMM_SILU_MUL.  An unknown flag bit gives INVALID_ARG.
 *
 * Epilogues of a decode step's projections (the pages time the projections of
 * one dense layer -- q, k, v, o, gate, up, down -- and leave the work beside
 * each GEMM open; these are the plain readings of that layer):
 * - W12_GEMM_OUT_BF16 writes each FP32 result rounded to the nearest BF16,
 *   ties to even (IEEE 754), so y can feed the next GEMM as its x.
 * - W12_GEMM_SILU_MUL is for a gate and an up projection merged into one
 *   matrix by interleaving their rows (row 2i = gate row i, row 2i+1 = up row
 *   i; encode the merged BF16 matrix once): y[m][i] = silu(g) * u with g and u
 *   the FP32 results of rows 2i and 2i+1 and silu(g) = g / (1 + e^-g), in
 *   FP32.  N must be even (else SHAPE).  With W12_GEMM_OUT_BF16 as well, the
 *   product is rounded to BF16 -- the down projection's input.
 *
 * Every GEMM launch may begin (streaming its weights) while the previous
 * kernel on the stream is still finishing; by default it reads x only after
 * that kernel has completed, since that kernel may have produced x.
 * W12_GEMM_INPUT_READY is the caller's statement that x was complete before
 * the previous operation on the stream started -- for instance several
 * projections of one activation vector issued back to back, or inputs copied
 * earlier.  The launch then reads x at once and overlaps the previous kernel's
 * tail.  It still writes nothing (y, its workspace) before the previous kernel
 * has completed, so the previous kernel may read or write y.  The flag has no
 * counterpart on the pages: it is a launch-overlap mode of this library.
 */
w12_status w12_gemm_ex(const void *x_bf16, const w12_dev *w, void *y, int M, int N, int K,
                       unsigned flags, w12_stream_t stream);

/* ---- INT8 copy for the Q pass ------------------------------------------------ */

/*
 * A separate INT8 copy of a weight matrix for the Q pass (the pages keep an
 * INT6/INT8 copy on the smaller GPU, RTX PRO 6000 section; this is the INT8
 * form), as an alternative to the nested 8-bit view: per output row n,
 * scale[n] = amax / 127 in FP32 (amax: the largest |w| of the row's finite
 * weights) and q[n][k] = rint(w / scale[n]) (FP32, round half to even)
 * clamped to [-127, 127]; Inf becomes +-127, NaN 0, and a row whose scale is
 * 0 keeps q = 0.  1 byte per weight plus 4 per row, in one device allocation
 * (the copy is extra memory: the W12 handle stays the lossless one).
 */
typedef struct w12_i8 w12_i8;

/* INT8 copy of BF16 weights w_bf16[N][K] already in device memory; synchronises
 * with `stream`.  Errors: INVALID_ARG, UNSUPPORTED (N or K above 2^31), OOM, CUDA. */
w12_status w12_i8_encode_device(const void *w_bf16, int64_t N, int64_t K, w12_stream_t stream, w12_i8 **out);

/* INT8 copy of the weights a W12 handle holds (decoded into a temporary
 * N x K BF16 buffer, stream-ordered, then quantised). */
w12_status w12_i8_from_dev(const w12_dev *w, w12_stream_t stream, w12_i8 **out);

void w12_i8_free(w12_i8 *q);

/* Copy q (N*K bytes) and/or the scales (N floats) to host buffers (either may
 * be NULL); synchronises with `stream`. */
w12_status w12_i8_download(const w12_i8 *q, int8_t *q_host, float *scale_host, w12_stream_t stream);

/* Device status of an INT8 copy's GEMMs (as w12_dev_status), reset to OK. */
w12_status w12_i8_status(const w12_i8 *q, w12_stream_t stream);

/*
 * The Q pass over an INT8 copy: y[m][n] = scale[n] * sum_k x[m][k] q[n][k],
 * FP32 accumulation on the tensor cores (every q is exact in BF16).  Arguments,
 * limits, flags (W12_GEMM_INPUT_READY, W12_GEMM_OUT_BF16, W12_GEMM_SILU_MUL;
 * any other bit gives INVALID_ARG) and errors as w12_gemm_ex.  Every M runs on
 * the tensor-core kernel (M padded to 16, 32, 64, 128 or 256).
 */
w12_status w12_gemm_i8(const void *x_bf16, const w12_i8 *q, void *y, int M, int N, int K, unsigned flags,
                       w12_stream_t stream);

/*
 * Several W12 matrices that read the same activations, in one launch:
 * y_i[M][N_i] = x[M][K] . W_i^T for i < n, 1 <= n <= W12_MAX_GROUP (4), e.g.
 * the q, k and v projections of a layer, or its gate and up projections.
 * The row blocks of all n matrices are laid end to end and split over one
 * persistent grid, so the small matrices share the launch's start-up and
 * tail instead of paying one each; every weight is read once.  Each y_i
 * meets the same bound as a w12_gemm_ex call on W_i alone (the split of row
 * blocks over CTAs, hence the order in which partial sums are added, may
 * differ).  ws[i]: device handles, all with the same K and on
 * the current device; ys[i]: device outputs [M][N_i], FP32 or (flag
 * W12_GEMM_OUT_BF16) BF16, 16-byte aligned, caller-owned.  Flags:
 * W12_GEMM_Q8VIEW, W12_GEMM_INPUT_READY, W12_GEMM_OUT_BF16 (W12_GEMM_SILU_MUL
 * and other bits give INVALID_ARG).  Workspace, limits and errors as
 * w12_gemm_ex; a timeout is recorded in every handle's status word.
 */
#define W12_MAX_GROUP 4
w12_status w12_gemm_grouped(const void *x_bf16, const w12_dev *const *ws, void *const *ys, int n, int M, int K,
                            unsigned flags, w12_stream_t stream);

/*
 * End-to-end form of w12_gemm_grouped for host-resident activations: copies
 * x_host [M][K] (BF16 bits) -> x_dev, runs w12_gemm_grouped into ys_dev, and
 * copies each ys_dev[i] -> ys_host[i] ([M][N_i], FP32 or, with
 * W12_GEMM_OUT_BF16, BF16), all on `stream` (pinned host memory makes the
 * copies asynchronous: synchronise the stream before reading ys_host).
 * Outputs that follow one another in memory both on the device and on the
 * host go back in one transfer.  Every buffer is caller-owned; arguments,
 * flags and errors as w12_gemm_grouped, plus W12_ERR_INVALID_ARG for a
 * missing host buffer.
 */
w12_status w12_gemm_grouped_host(const uint16_t *x_host, void *x_dev, const w12_dev *const *ws,
                                 void *const *ys_dev, void *const *ys_host, int n, int M, int K, unsigned flags,
                                 w12_stream_t stream);

/*
 * End-to-end form of w12_gemm for host-resident activations: copies
 * x_host -> x_dev, runs w12_gemm into y_dev, copies y_dev -> y_host, all on
 * `stream` (use pinned host memory for asynchronous copies).  Every buffer is
 * caller-owned; nothing is allocated beyond w12_gemm's workspace.
 */
w12_status w12_gemm_host(const uint16_t *x_host, void *x_dev, const w12_dev *w, float *y_dev,
                         float *y_host, int M, int N, int K, w12_stream_t stream);

/*
 * w12_gemm without any device allocation, for callers that may not allocate:
 * code whose host process hands all device memory to its own pool, plug-ins
 * whose framework must own every allocation, loops that may not take the
 * allocator's locks.  (The pages have no counterpart; this is a library
 * convenience.)  Same arguments, result and errors as w12_gemm, but the
 * split-K scratch comes from one fixed 16 MiB array in device memory that
 * every GPU loading this library holds until exit; a call needing more
 * (over 8192 row blocks, or more than 2 * CTAs * M * 128 FP32 partial sums
 * -- on a 152-SM GB300, M above about 107 on most shapes) fails with
 * W12_ERR_UNSUPPORTED.  All calls on a device share the
 * array, so calls whose kernels overlap on the GPU (other streams, other
 * threads) race: serialise them.  The first call on each device looks up the
 * array, clears its counters and synchronises the device; make it before any
 * stream capture.
 */
w12_status w12_gemm_noalloc(const void *x_bf16, const w12_dev *w, float *y, int M, int N, int K,
                            w12_stream_t stream);

/*
 * Lossless decode on the device: out[N][K] BF16 bit patterns (device, caller
 * owned, 16-byte aligned), bit-identical to the matrix that was encoded [MF].
 */
w12_status w12_decode(const w12_dev *w, uint16_t *w_bf16_out, w12_stream_t stream);

/*
 * Synchronise `stream`, then read and clear the handle's device status word:
 * W12_OK, W12_ERR_TIMEOUT (a kernel's bounded wait ran out; its output is
 * invalid) or W12_ERR_CORRUPT (a kernel met metadata it could not use).
 */
w12_status w12_dev_status(const w12_dev *w, w12_stream_t stream);

/* Release every cached GEMM workspace of the current device, including those
 * a growing workspace replaced (synchronises).  CUDA graphs captured with
 * them must not be replayed afterwards. */
w12_status w12_release_workspaces(void);

/*
 * Test hooks for the failure path.  w12_set_spin_limit: the wall-time limit in
 * nanoseconds of every bounded device-side wait of later GEMM launches (0 =
 * the default, 200 ms); a kernel whose wait runs out records W12_ERR_TIMEOUT
 * in the handle's status word, stops waiting, lets its in-flight copies land
 * and returns.  w12_debug_inject_stall(1): later GEMM launches also wait on a
 * barrier that nothing ever signals, so they take that path on purpose.
 */
void w12_set_spin_limit(uint32_t limit_ns);

/* Name of the last CUDA error behind a W12_ERR_CUDA from a GEMM launch on this
 * host thread (static string; "no error" if none). */
const char *w12_last_cuda_error(void);
void w12_debug_inject_stall(int on);

#ifdef __cplusplus
}
#endif

#endif /* W12_H */
