/*
 * syn.h — C ABI of libsyn: GGUF block-quantized mul_mat on one GB300 (sm_103a).
 *
 * The operation ("The GGML ecosystem, and where synapse fits", section 5, "Products:
 * weights against quantized activations"; yakaai ggml documentation, examples/simple):
 *
 *   W  n_out x n_in weights in a block format, rows contiguous, each row n_in/B blocks
 *      (GGUF "ne = [cols, rows]", section 2 of the same page);
 *   X  n_tok x n_in fp32 activations, token-major;
 *   Y  n_tok x n_out fp32, Y[t*n_out + o] = sum_i W[o,i] * Xq[t,i]
 *      i.e. ggml_mul_mat(W, X) = (X W^T): each token's outputs are contiguous.
 *
 * Xq is X converted, row by row, to the weight format's vec_dot_type before the product
 * (Q8_0 for Q8_0, Q4_0 and Q5_0 weights, Q8_K for Q4_K and Q6_K weights, fp16 for F16
 * weights): the product is that of the converted activations, as on the pages, not the
 * exact fp32 product.
 *
 * Conventions for every entry point:
 *   - pointers are DEVICE pointers on the current CUDA device unless stated otherwise,
 *     owned by the caller; the library keeps no reference after the call returns;
 *   - work is enqueued on `stream` (a cudaStream_t; NULL = legacy default stream) and is
 *     asynchronous unless stated otherwise;
 *   - the return value is SYN_OK (0) or a negative SYN_ERR_* code; on an error nothing
 *     has been enqueued, except for SYN_ERR_CUDA (a launch failed) and SYN_ERR_TIMEOUT;
 *   - nothing throws, nothing prints;
 *   - the decode launches of syn_mul_mat / syn_mul_mat_batch release programmatic dependents
 *     (CUDA programmatic dependent launch) before they finish: a kernel of the caller's that
 *     is launched right after them with programmatic stream serialization allowed must call
 *     cudaGridDependencySynchronize() (griddepcontrol.wait) before it reads their outputs.
 *     Kernels launched without that attribute, and copies, are ordered as usual.
 */
#ifndef SYN_H
#define SYN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define SYN_API __attribute__((visibility("default")))
#else
#define SYN_API
#endif

typedef struct CUstream_st* syn_stream_t; /* identical to cudaStream_t */

/* Block formats (the library's own numbering, not ggml_type values).
 * Format table, "The GGML ecosystem, and where synapse fits", section 5:
 *   Q8_0  32 weights,  34 B: fp16 d, 32 int8 q;                       w = d*q
 *   Q4_K 256 weights, 144 B: fp16 d, fp16 dmin, 12 B of 6-bit scales and mins,
 *                            128 B of 4-bit q in 8 sub-blocks of 32;  w = d*sc*q - dmin*m
 *   Q6_K 256 weights, 210 B: 128 B low 4 bits, 64 B high 2 bits, 16 int8 scales, fp16 d;
 *                            16 sub-blocks of 16;                     w = d*sc*(q - 32)
 *   Q8_K 256 values,  292 B: fp32 d, 256 int8 q, 16 int16 sums of 16 q (activations only)
 *   Q4_0  32 weights,  18 B: fp16 d, 32 4-bit q;                      w = d*(q - 8)
 *   Q5_0  32 weights,  22 B: fp16 d, 32-bit qh (each q's fifth bit), 32 4-bit low parts;
 *                                                                     w = d*(q - 16)
 *   F16   1 weight,     2 B: IEEE binary16 (round to nearest even from fp32)
 * In-block byte order: the public GGUF layout (fields in the order listed above; Q4_0/Q5_0
 * store q[l] in the low and q[l+16] in the high nibble of byte l).
 * vec_dot_type (the activation format of the product): Q8_0 for Q8_0, Q4_0 and Q5_0; Q8_K
 * for Q4_K and Q6_K; F16 for F16 (the activations rounded to fp16; products exact, fp32 sums;
 * mul_mat needs n_in % 8 == 0 for F16 weights). */
enum {
    SYN_TYPE_Q8_0 = 1,
    SYN_TYPE_Q4_K = 2,
    SYN_TYPE_Q6_K = 3,
    SYN_TYPE_Q8_K = 4,
    SYN_TYPE_Q4_0 = 5,
    SYN_TYPE_Q5_0 = 6,
    SYN_TYPE_F16 = 7,
};

enum {
    SYN_OK = 0,
    SYN_ERR_TYPE = -1,    /* unknown format, or a format not allowed for this call     */
    SYN_ERR_SHAPE = -2,   /* a size <= 0 (or < 0 where 0 is allowed), or n_in % B != 0 */
    SYN_ERR_NULL = -3,    /* a required pointer is NULL                                 */
    SYN_ERR_ALIGN = -4,   /* a pointer is not 16-byte aligned                           */
    SYN_ERR_RANGE = -5,   /* quantize input non-finite, or a scale overflows fp16       */
    SYN_ERR_CUDA = -6,    /* a CUDA call or kernel launch failed                        */
    SYN_ERR_TIMEOUT = -7, /* a device-side wait gave up (bounded spin); results invalid */
    SYN_ERR_NOMEM = -8,   /* the workspace could not be allocated                       */
    SYN_ERR_DEVICE = -9,  /* the current device is not sm_103 / not usable              */
    SYN_ERR_TOO_LARGE = -10, /* the problem needs more than the fixed scratch array holds */
    SYN_ERR_FORMAT = -11, /* a GGUF file is malformed or not a GGUF file               */
    SYN_ERR_IO = -12,     /* a file could not be opened, mapped or written             */
    SYN_ERR_NOTFOUND = -13, /* no GGUF key / tensor with that name or index              */
    SYN_ERR_BOUNDS = -14, /* SYN_DEBUG build only: a kernel found an index or copy window
                             outside its buffers and skipped that access; results invalid */
};

/* Elements per block: 32 (Q8_0, Q4_0, Q5_0), 256 (Q4_K, Q6_K, Q8_K) or 1 (F16); -1 for an
 * unknown type. */
SYN_API int64_t syn_block_elems(int type);

/* Bytes per block: 34 (Q8_0), 144 (Q4_K), 210 (Q6_K), 292 (Q8_K), 18 (Q4_0), 22 (Q5_0),
 * 2 (F16); -1 for an unknown type. */
SYN_API int64_t syn_block_bytes(int type);

/* Bytes of one row of n elements: (n / elems) * bytes; -1 if the type is unknown or
 * n is not a positive multiple of the block size.  Pure host function. */
SYN_API int64_t syn_row_bytes(int type, int64_t n);

/* Quantize n_rows rows of n_per_row fp32 values (src, row-major, contiguous) into blocks
 * (dst, n_rows * syn_row_bytes bytes).  type: Q8_0, Q4_K, Q6_K, Q8_K, Q4_0, Q5_0 or F16.
 * Encoders (plain readings of the format table; bit-exact with the CPU oracle):
 *   Q8_0  d = fp16(amax/127); q = clamp(round(x / d_stored), -127, 127)
 *   Q8_K  d = amax/127 (fp32); q = clamp(round(x / d), -127, 127); bsums = sums of 16 q
 *   Q4_K  per 32-sub-block: lo = min(0, min x), s = (max x - lo)/15, m = -lo;
 *         d = fp16(max s / 63), dmin = fp16(max m / 63), sc = min(63, round(s/d)),
 *         mn = min(63, round(m/dmin)), q = clamp(round((x + dmin*mn)/(d*sc)), 0, 15)
 *   Q6_K  per 16-sub-block: s = amax/31; d = fp16(max s / 127), sc = min(127, round(s/d)),
 *         q = clamp(round(x/(d*sc)), -32, 31) + 32
 *   Q4_0  m = the block's value of largest magnitude (first one), d = fp16(m / -8),
 *         q = clamp(round(x / d) + 8, 0, 15)
 *   Q5_0  d = fp16(m / -16), q = clamp(round(x / d) + 16, 0, 31)
 *   F16   the IEEE half of x (an overflow to infinity is a range error)
 * round = ties away from zero; a zero scale gives zero codes (Q4_0/Q5_0: q = 8 / 16).
 * Returns SYN_ERR_RANGE if any input is NaN/Inf or a scale overflows fp16; to report
 * that, this call SYNCHRONIZES `stream` before returning (it is an offline operation).
 * Calls that overlap on the GPU share one status word and must not run concurrently.
 * Alignment: src and dst must be 16-byte aligned.  n_rows == 0 is a no-op. */
SYN_API int syn_quantize(int type, const float* src, void* dst, int64_t n_rows, int64_t n_per_row,
                 syn_stream_t stream);

/* Expand blocks back to fp32 ("dequantize_row_*", same page, section 5): dst gets
 * n_rows * n_per_row floats.  Q8_0: d*q; Q4_K: (d*sc)*q - (dmin*mn); Q6_K: (d*sc)*(q-32);
 * Q8_K: d*q; Q4_0: d*(q-8); Q5_0: d*(q-16); F16: the value.  Each product and difference is
 * one fp32 rounding (no FMA), so the result is bit-exact with the CPU oracle.
 * Asynchronous.  Alignment: 16 B. */
SYN_API int syn_dequantize(int type, const void* src, float* dst, int64_t n_rows, int64_t n_per_row,
                   syn_stream_t stream);

/* The same expansion to fp16 (Q4_K and Q6_K only; SYN_ERR_TYPE for the other formats): dst
 * gets n_rows * n_per_row IEEE halves, each the value syn_dequantize returns rounded once to
 * fp16 (to nearest, ties to even).  This is the weight operand the prefill product uses when
 * it expands weights first (syn_set_prefill_expand_tok).  Asynchronous.  Alignment: 16 B. */
SYN_API int syn_dequantize_f16(int type, const void* src, void* dst, int64_t n_rows, int64_t n_per_row,
                               syn_stream_t stream);

/* The activation step of the product on its own (from_float to the vec_dot_type):
 * X (n_tok x n_in fp32) -> codes qs (n_tok x n_in int8), scales d (n_tok x n_in/Bx fp32,
 * Bx = 32 for Q8_0/Q4_0/Q5_0 weights, 256 for K-quant weights; for the 32-blocks the value
 * of the stored fp16 scale) and, for K-quant weights only, bsums (n_tok x n_in/16 int16; may
 * be NULL otherwise).  wtype is the WEIGHT format (Q8_0, Q4_K, Q6_K, Q4_0 or Q5_0).  This
 * is the same device code the product kernels run on their inputs.  Asynchronous.
 * Alignment: 16 B. */
SYN_API int syn_quantize_activations(int wtype, const float* X, int64_t n_tok, int64_t n_in,
                             int8_t* qs, float* d, int16_t* bsums, syn_stream_t stream);

/* Y = ggml_mul_mat(W, X) as described at the top of this file.
 * type: Q8_0, Q4_K, Q6_K, Q4_0, Q5_0 or F16 (Q8_K is activation-only: SYN_ERR_TYPE).
 * n_tok <= the decode threshold (per format by default: 8 for Q4_K and Q6_K, 4 for Q8_0,
 * Q4_0 and Q5_0, 2 for F16; see syn_set_gemv_max_tok) runs the decode kernels: X is
 * converted (by a conversion launch into the library workspace, or, for narrow inputs,
 * inside the decode CTAs) and W is streamed once per group of up to 8 tokens.  Larger
 * n_tok runs the prefill path: one kernel converts X and writes the dequantized fp16
 * activations into the library workspace, a second runs the tensor-core GEMM on W tiles
 * dequantized to fp16 in shared memory (fp32 accumulation); from 1536 tokens (see
 * syn_set_prefill_expand_tok) Q6_K weights, and from 3072 Q4_K weights of rows up to 8192
 * values, are instead expanded to fp16 into the workspace by a launch of their own and the
 * GEMM reads them from there.
 * Accuracy: |y - y_ref| <= 1e-4 * ||dequant(w_row)||_2 * ||x||_2 per element, where
 * y_ref is the same product evaluated in fp64.  W, X, Y: 16-byte aligned, not aliased.
 * n_tok == 0 is a no-op.  Asynchronous.  The prefill path may grow the workspace (see
 * syn_reserve); growth allocates device memory and synchronizes the device, so reserve
 * before capturing a CUDA graph.  The workspace belongs to (device, stream): calls on one
 * stream are ordered; calls on different streams use different workspaces. */
SYN_API int syn_mul_mat(int type, const void* W, int64_t n_out, int64_t n_in,
                const float* X, int64_t n_tok, float* Y, syn_stream_t stream);

/* One product of a group (see syn_mul_mat_batch). */
typedef struct {
    int type;          /* a weight format: Q8_0, Q4_K, Q6_K, Q4_0, Q5_0 or F16 */
    const void* W;     /* n_out x n_in weights, 16-byte aligned */
    int64_t n_out;
    int64_t n_in;
    const float* X;    /* n_tok x n_in activations, 16-byte aligned */
    float* Y;          /* n_tok x n_out outputs, 16-byte aligned, not aliased */
} syn_mat_desc;

/* n independent products Y_i = ggml_mul_mat(W_i, X_i), all with n_tok tokens: the same
 * result as n calls of syn_mul_mat.  The quantized products with n_tok <= their format's
 * decode threshold (see syn_mul_mat) run in as few launches as the decode kernel's limits
 * allow (at most 16 matrices and 83,456 bytes of converted activations per token group and
 * launch), so the products of a layer (q, k, v, o, gate, up, down) share one launch and all
 * SMs stream their weights together.  The products with more tokens than their format
 * decodes (or rows too wide for the decode kernel) take the prefill path; those of them that
 * share one activation input (the same X pointer, n_in and vec_dot_type, e.g. q/k/v or
 * gate/up of a layer) convert it once and run one tensor-core launch each.  F16 products in
 * decode run as in syn_mul_mat.  Arguments are checked as for syn_mul_mat (including the
 * deterministic mode's row-width limit) before anything is enqueued.  Asynchronous. */
SYN_API int syn_mul_mat_batch(int n, const syn_mat_desc* descs, int64_t n_tok, syn_stream_t stream);

/* The grouped call with its inputs and outputs staged through host memory: copies x_bytes
 * from x_host to x_dev, runs syn_mul_mat_batch(n, descs, n_tok, stream), then copies
 * y_bytes from y_dev to y_host, all enqueued on `stream` in that order (one cudaMemcpyAsync
 * each way; x_dev / y_dev are typically one buffer holding every product's X / Y).  x_host
 * and y_host are HOST pointers (page-locked memory keeps the copies asynchronous); x_dev and
 * y_dev device pointers.  A byte count of 0 skips that copy (its pointers may then be NULL).
 * Returns as syn_mul_mat_batch, SYN_ERR_NULL for a missing pointer of a non-empty copy,
 * SYN_ERR_CUDA if a copy cannot be enqueued (nothing after it is enqueued).  Argument,
 * shape, alignment and device errors are returned before anything is enqueued; only
 * SYN_ERR_NOMEM (workspace growth failed) or SYN_ERR_CUDA can come after the input copy,
 * and possibly some products, were enqueued.  The result is in y_host once the stream has
 * reached the end of the call. */
SYN_API int syn_mul_mat_batch_staged(int n, const syn_mat_desc* descs, int64_t n_tok, const void* x_host,
                                     void* x_dev, size_t x_bytes, const void* y_dev, void* y_host,
                                     size_t y_bytes, syn_stream_t stream);

/* Pre-size the prefill workspace of (current device, stream) for products with up to
 * max_n_in inputs and max_n_tok tokens, so that later syn_mul_mat calls allocate nothing.
 * Prefill calls that expand their weights to fp16 (syn_set_prefill_expand_tok) need
 * n_out * n_in * 2 bytes more, which their first call allocates.  Synchronizes the device
 * when it (re)allocates. */
SYN_API int syn_reserve(int64_t max_n_in, int64_t max_n_tok, syn_stream_t stream);

/* Free every workspace the library holds on the current device (synchronizes it). */
SYN_API int syn_release(void);

/* Integer block sums for bit-exact checks (not on the hot path).  Xq holds n_tok rows of
 * packed vec_dot_type blocks (Q8_0 blocks for Q8_0/Q4_0/Q5_0 weights, Q8_K otherwise).
 * S[((t*n_out + o)*n_blocks + b)*2 + {0,1}]:  Q8_0 {I, 0}: I = sum qw*qx;
 * Q4_K {A, Bm}: A = sum_j sc_j * sum_{i in j} q_i*qx_i, Bm = sum_j mn_j * (bsum_2j + bsum_2j+1);
 * Q6_K {C, 0}: C = sum_j sc_j * sum_{i in j} (q_i - 32)*qx_i;
 * Q4_0 / Q5_0 {I, 0}: I = sum (qw - 8 / 16)*qx.  Asynchronous. */
SYN_API int syn_block_sums(int type, const void* W, int64_t n_out, int64_t n_in,
                   const void* Xq, int64_t n_tok, int32_t* S, syn_stream_t stream);

/* The tile schedule the prefill product picks for a shape on sms SMs (host only, no device
 * needed; for checks of the planner): out[0] = the K split S of split tiles (1: none),
 * out[1] = the row tiles (of 128 outputs) that run whole tiles, out[2] = 1 when the other row
 * tiles' tiles are shared stream-K (equal super-step ranges per CTA) instead of split S ways,
 * out[3] = the number of 128 x BN tiles (BN = n_tok rounded up to 16, at most 256).
 * SYN_ERR_SHAPE for non-positive sizes or sms, SYN_ERR_NULL for out. */
SYN_API int syn_debug_prefill_plan(int64_t n_out, int64_t n_in, int64_t n_tok, int sms, int* out);

/* Decode/prefill threshold.  By default (n < 0) it depends on the format: products with
 * n_tok <= 8 (Q4_K, Q6_K), <= 4 (Q8_0, Q4_0, Q5_0) or <= 2 (F16) use the decode kernels,
 * larger ones the tensor-core prefill (the measured crossovers on GB300).  n >= 0 sets the
 * same threshold for every format (0 forces the prefill path for every n_tok >= 1).
 * Returns the previous value (-1: per format).  Process-wide; the environment variable
 * SYN_GEMV_MAX_TOK, when set at load time, gives the initial value. */
SYN_API int syn_set_gemv_max_tok(int n);

/* Deterministic mode (on != 0; process-wide, default off; returns the previous setting).
 * The invariants follow synapse's ("The GGML ecosystem, and where synapse fits", section 7,
 * the table of what differs by design: each gemm row is bit-identical to gemv (G1); results
 * are bit-identical for any thread count (D1)).  In this mode every syn_mul_mat /
 * syn_mul_mat_batch product, whatever n_tok, runs on the decode kernels (token groups of up
 * to 8, weights re-read per group) and no output row is split between warps, so that each
 * Y element is computed by one fixed sequence of operations that depends only on the
 * format, n_in and the inputs.  Hence, bit for bit:
 *   - a token's row of Y is the same whatever the other tokens of the call (prefill rows
 *     equal decode rows: G1);
 *   - Y is the same for any SM limit (syn_set_sm_limit), grouping of products into
 *     syn_mul_mat_batch calls, or split of the tokens into calls (the counterpart of D1).
 * Accuracy is that of the decode path (the tolerance of syn_mul_mat).  Prefill is far
 * slower in this mode (no tensor cores).  Products whose converted activation row does not
 * fit the decode kernel's shared memory (n_in above 72,960 for Q4_K / Q6_K, 74,112 for
 * Q8_0, 70,208 for Q4_0 / Q5_0) return SYN_ERR_SHAPE in this mode.
 * syn_mul_mat_prefill_static is not affected (it always runs the tensor-core prefill). */
SYN_API int syn_set_deterministic(int on);

/* Prefill calls (the tensor-core path) first expand Q6_K weights from n tokens on, and Q4_K
 * weights of rows up to 8192 values from 2n tokens on, to fp16, once per product, into the
 * library's workspace (n_out * n_in * 2 more bytes, grown on first need like the activation
 * workspace), then run the tensor-core product on the fp16 weights; otherwise the product
 * expands each weight tile inside the product kernel, once per tile of up to 256 tokens.  Each expanded value is the fp32 dequantization
 * (syn_dequantize's, bit for bit) rounded once to fp16; the result stays within the
 * tolerance of syn_mul_mat either way.  n < 0 restores the default (1536); 0 expands at
 * every prefill call.  Process-wide; returns the previous value; the environment variable
 * SYN_PREFILL_EXPAND_TOK, when set at load time, gives the initial value.
 * syn_mul_mat_prefill_static never expands (it allocates nothing). */
SYN_API int syn_set_prefill_expand_tok(int n);

/* At most n SMs for the library's launches (n >= 1; 0 = all of them, the default).
 * Process-wide; returns the previous value, or -1 (and changes nothing) for n < 0.  Lets a
 * caller leave SMs to concurrent work; the grid of every kernel is sized to the limit. */
SYN_API int syn_set_sm_limit(int n);

/* Read (and with clear != 0, reset) the device-side error words of the current device:
 * SYN_OK, or SYN_ERR_TIMEOUT if a kernel of any entry point (syn_mul_mat_prefill_static
 * included) gave up a bounded wait since the last clear.  A kernel that gives up records
 * the timeout, stops its other threads, waits for the copies and tensor-core operations it
 * had already issued and returns: the device stays usable, the outputs of that call are
 * invalid.  In the SYN_DEBUG build (index checks in every kernel) it returns
 * SYN_ERR_BOUNDS if a check failed.  Synchronizes the device.  It allocates nothing: a
 * device on which no product has run reads SYN_OK. */
SYN_API int syn_device_status(int clear);

/* Index checks (not part of the product path).  The SYN_DEBUG build of the library
 * (`python -m gguf_block_quantized_gb300.build --variant debug`, libsyn_debug.so: same
 * entry points) checks, before each access, the indices and copy windows its kernels
 * derive from the launch geometry: weight-stage windows and slot sizes, TMA coordinates
 * and their 16-byte alignment, shared-memory activation areas, unit and tile coordinates,
 * output indices.  A failed check records the failure, skips the access, and
 * syn_device_status returns SYN_ERR_BOUNDS.  This entry point lets a caller see that the
 * checks are compiled in: it launches one kernel whose check is given an out-of-range
 * index on purpose (the guarded store, into a shared array, is skipped).  Returns SYN_OK
 * once launched in the SYN_DEBUG build (syn_device_status then returns SYN_ERR_BOUNDS),
 * 1 in other builds (nothing launched), SYN_ERR_CUDA if the launch failed. */
SYN_API int syn_debug_bounds_selftest(syn_stream_t stream);

/* Number of kernels this library has launched in this process (all devices). */
SYN_API int64_t syn_launch_count(void);

/* Bytes of the fixed device array behind syn_mul_mat_prefill_static: 32 MiB, enough for
 * n_tok * n_in <= 16,777,216 (e.g. 4096 tokens of 4096 inputs, 1170 tokens of 14336). */
#define SYN_STATIC_SCRATCH_BYTES (32u << 20)

/* The prefill product of syn_mul_mat (activation step, then the tensor-core GEMM) for any
 * n_tok >= 1, for callers that cannot allocate device memory: code running inside a fixed
 * memory arena or under an allocator or budget that forbids cudaMalloc, or that must not
 * let a library call cudaMalloc/cudaFree (which can synchronize the device) on its path.
 * The pages have no counterpart to this entry point; it exists for such callers.
 * It allocates nothing: the fp16 activation scratch is a static device array of
 * SYN_STATIC_SCRATCH_BYTES that the library holds on every device it is used on until
 * the process exits.  Products with n_tok * n_in * 2 > SYN_STATIC_SCRATCH_BYTES are
 * rejected with SYN_ERR_TOO_LARGE.  Arguments, layout, accuracy and the other error codes
 * are those of syn_mul_mat (F16 weights need n_in % 8 == 0, as there).  A bounded-wait
 * timeout of its kernels is reported by syn_device_status, like those of syn_mul_mat; the
 * status word sits at the head of the fixed array.  The first call on a device sets up that device (looks up the
 * array's device address, clears its status word, synchronizes the device): make it
 * before any stream capture.  Every call on a device shares the one array and overwrites
 * it, so calls that can overlap on the GPU (different streams without ordering between
 * them) race and give wrong results; order them.  Asynchronous.  Its kernel launches are
 * counted by syn_launch_count. */
SYN_API int syn_mul_mat_prefill_static(int type, const void* W, int64_t n_out, int64_t n_in,
                               const float* X, int64_t n_tok, float* Y, syn_stream_t stream);

/* ======================================================================================
 * GGUF container (host code; only syn_gguf_upload touches the GPU)
 *
 * Layout ("The GGML ecosystem, and where synapse fits", section 2, the GGUF diagram; "ggml
 * Documentation", GGUF specification, "File Structure" and the general.alignment key;
 * "llama.cpp and GGUF", "Tensor info, alignment, and mmap"), little-endian:
 *   header       "GGUF", version u32 (3), n_tensors u64, n_kv u64
 *   metadata     n_kv x { key string, value type u32, value }
 *   tensor info  n_tensors x { name string, n_dims u32, ne u64[n_dims], type u32, offset u64 }
 *   padding      zeros to a multiple of general.alignment (u32; 32 when absent; a multiple of 8)
 *   data         tensor i at data_start + offset_i (offset_i a multiple of the alignment)
 * A string is a u64 byte count followed by the bytes (no terminator); an array value is an
 * element type u32, a count u64 and the packed elements.  ne lists the innermost dimension
 * first: a weight matrix with n_in inputs and n_out outputs has ne = [n_in, n_out], rows
 * contiguous, exactly the W layout of syn_mul_mat.  Tensor offsets are relative to the
 * start of the data section.  The numeric codes below (value types, ggml tensor types)
 * follow the public GGUF specification; the pages name the types without their codes.
 * ====================================================================================== */

/* metadata value types */
enum {
    SYN_GGUF_UINT8 = 0, SYN_GGUF_INT8 = 1, SYN_GGUF_UINT16 = 2, SYN_GGUF_INT16 = 3,
    SYN_GGUF_UINT32 = 4, SYN_GGUF_INT32 = 5, SYN_GGUF_FLOAT32 = 6, SYN_GGUF_BOOL = 7,
    SYN_GGUF_STRING = 8, SYN_GGUF_ARRAY = 9, SYN_GGUF_UINT64 = 10, SYN_GGUF_INT64 = 11,
    SYN_GGUF_FLOAT64 = 12,
};

/* ggml tensor element types the reader can size (others are listed with nbytes = -1) */
enum {
    SYN_GGML_F32 = 0, SYN_GGML_F16 = 1, SYN_GGML_Q4_0 = 2, SYN_GGML_Q5_0 = 6,
    SYN_GGML_Q8_0 = 8, SYN_GGML_Q4_K = 12, SYN_GGML_Q6_K = 14, SYN_GGML_Q8_K = 15,
    SYN_GGML_BF16 = 30,
};

typedef struct syn_gguf syn_gguf;               /* an open, memory-mapped GGUF file */
typedef struct syn_gguf_writer syn_gguf_writer; /* a GGUF file being assembled       */

/* Opens and memory-maps a GGUF (version 2 or 3) file read-only and checks its structure:
 * magic and version, every string, array and tensor-info record inside the file, unique
 * keys and tensor names, general.alignment (u32, a non-zero multiple of 8), 1..4
 * dimensions each >= 1, rows of whole blocks, every offset a multiple of the alignment and
 * every sized tensor inside the file.  Returns NULL on failure with *status (if non-NULL)
 * set to SYN_ERR_NULL (path NULL), SYN_ERR_IO (open/stat/mmap failed) or SYN_ERR_FORMAT;
 * else *status = SYN_OK.  Pointers returned by the accessors below point into the mapping
 * and stay valid until syn_gguf_close.  Tensor data are at least alignment-aligned within
 * the (page-aligned) mapping.  A handle may be read from several threads at once. */
SYN_API syn_gguf* syn_gguf_open(const char* path, int* status);
SYN_API void syn_gguf_close(syn_gguf* g); /* unmaps; NULL is a no-op */

/* Header facts; -1 for a NULL handle.  data_start is the file offset of the data section. */
SYN_API int64_t syn_gguf_version(const syn_gguf* g);
SYN_API int64_t syn_gguf_n_tensors(const syn_gguf* g);
SYN_API int64_t syn_gguf_n_kv(const syn_gguf* g);
SYN_API int64_t syn_gguf_alignment(const syn_gguf* g);
SYN_API int64_t syn_gguf_data_start(const syn_gguf* g);

/* Index of the tensor called name (exact bytes), or -1. */
SYN_API int64_t syn_gguf_find_tensor(const syn_gguf* g, const char* name);

/* Tensor i's info; every output pointer may be NULL.  ne receives 4 values (unused
 * dimensions = 1).  *data is a HOST pointer into the mapping and *nbytes its size, or NULL
 * and -1 for an element type the reader cannot size.  SYN_ERR_NULL (g NULL) or
 * SYN_ERR_NOTFOUND (i out of range). */
SYN_API int syn_gguf_tensor_info(const syn_gguf* g, int64_t i, const char** name, uint32_t* ggml_type,
                                 int* n_dims, int64_t* ne, uint64_t* offset, const void** data,
                                 int64_t* nbytes);

/* The tensor called name as syn_mul_mat's weight operand: *type the library's format code
 * (SYN_TYPE_*), n_in = ne[0], n_out = ne[1]*ne[2]*ne[3], *data the HOST pointer into the
 * mapping and *nbytes = n_out * syn_row_bytes(type, n_in).  Output pointers may be NULL.
 * SYN_ERR_NULL, SYN_ERR_NOTFOUND, or SYN_ERR_TYPE when the element type is not one of
 * Q8_0, Q4_K, Q6_K, Q4_0, Q5_0, F16. */
SYN_API int syn_gguf_matrix(const syn_gguf* g, const char* name, int* type, int64_t* n_out, int64_t* n_in,
                            const void** data, int64_t* nbytes);

/* Copies tensor i's bytes from the mapping into the DEVICE buffer dst (dst_bytes long) with
 * one cudaMemcpyAsync on stream (pageable source: the copy has finished reading the
 * mapping when the call returns).  SYN_ERR_NULL, SYN_ERR_NOTFOUND, SYN_ERR_TYPE (tensor not
 * sized), SYN_ERR_SHAPE (dst_bytes too small) or SYN_ERR_CUDA. */
SYN_API int syn_gguf_upload(const syn_gguf* g, int64_t i, void* dst, int64_t dst_bytes, syn_stream_t stream);

/* Metadata entry i: key, value type, and for arrays the element type and count (0 for
 * other values).  Output pointers may be NULL.  SYN_ERR_NULL or SYN_ERR_NOTFOUND. */
SYN_API int syn_gguf_kv_info(const syn_gguf* g, int64_t i, const char** key, uint32_t* value_type,
                             uint32_t* elem_type, uint64_t* n_elems);

/* Typed getters by key.  SYN_ERR_NULL (any pointer NULL), SYN_ERR_NOTFOUND (no such key),
 * SYN_ERR_TYPE (the value has another type).  get_int takes every integer type and bool
 * (SYN_ERR_RANGE for a UINT64 above INT64_MAX); get_float takes FLOAT32 and FLOAT64;
 * get_string gives the bytes (not terminated) and their count; get_array gives the element
 * type, count and a pointer to the packed little-endian elements (for string arrays use
 * get_array_string, which returns element j or SYN_ERR_NOTFOUND past the end). */
SYN_API int syn_gguf_get_int(const syn_gguf* g, const char* key, int64_t* out);
SYN_API int syn_gguf_get_float(const syn_gguf* g, const char* key, double* out);
SYN_API int syn_gguf_get_string(const syn_gguf* g, const char* key, const char** bytes, int64_t* len);
SYN_API int syn_gguf_get_array(const syn_gguf* g, const char* key, uint32_t* elem_type, uint64_t* n,
                               const void** data);
SYN_API int syn_gguf_get_array_string(const syn_gguf* g, const char* key, uint64_t j, const char** bytes,
                                      int64_t* len);

/* Writer.  begin records the path and the alignment (a non-zero multiple of 8; when it is
 * not 32 the first metadata entry is general.alignment = alignment, u32) and returns NULL
 * for a NULL path or a bad alignment.  The kv_* calls append metadata entries in call order
 * (SYN_ERR_SHAPE for a repeated key or for general.alignment; SYN_ERR_TYPE for a value
 * type the call does not write: kv_int writes the integer types and BOOL, keeping the low
 * bytes of value; kv_float FLOAT32 (rounded from value) or FLOAT64; kv_array any scalar
 * element type, n elements of its size packed at data).  add_tensor appends a tensor (ne
 * innermost first, 1..4 dims; nbytes must equal the size its type and shape give; names
 * unique: SYN_ERR_SHAPE otherwise; SYN_ERR_TYPE for a type the reader cannot size); the
 * bytes are copied, each tensor placed at the next multiple of the alignment.  finish
 * writes the version-3 file (header, metadata, tensor info, zero padding, data) and frees
 * the writer whatever it returns (SYN_OK or SYN_ERR_IO); abort frees it without writing.
 * Everything is held in host memory until finish. */
SYN_API syn_gguf_writer* syn_gguf_writer_begin(const char* path, uint32_t alignment);
SYN_API int syn_gguf_writer_kv_int(syn_gguf_writer* w, const char* key, uint32_t value_type, int64_t value);
SYN_API int syn_gguf_writer_kv_float(syn_gguf_writer* w, const char* key, uint32_t value_type, double value);
SYN_API int syn_gguf_writer_kv_string(syn_gguf_writer* w, const char* key, const char* bytes, int64_t len);
SYN_API int syn_gguf_writer_kv_array(syn_gguf_writer* w, const char* key, uint32_t elem_type, uint64_t n,
                                     const void* data);
SYN_API int syn_gguf_writer_kv_string_array(syn_gguf_writer* w, const char* key, uint64_t n,
                                            const char* const* strs, const int64_t* lens);
SYN_API int syn_gguf_writer_add_tensor(syn_gguf_writer* w, const char* name, uint32_t ggml_type, int n_dims,
                                       const int64_t* ne, const void* data, int64_t nbytes);
SYN_API int syn_gguf_writer_finish(syn_gguf_writer* w);
SYN_API void syn_gguf_writer_abort(syn_gguf_writer* w);

/* Static text for a status code. */
SYN_API const char* syn_strerror(int status);

#ifdef __cplusplus
}
#endif

#endif /* SYN_H */
