/*
 * q8proj.h -- C ABI of the GB300 (sm_103a) int8 quantized projection library
 * (libq8proj.so).
 *
 * The path: an f32 activation is encoded once into a q8_0 "plane", either by a
 * standalone quantizer or by the producer kernel that computes it (RMSNorm or
 * SwiGLU), and that plane is contracted with Q8_0 weights by a batch-1 GEMV
 * (decode) or a GEMM (prefill).  For a decode token the encoding can also
 * happen inside the GEMV launch that consumes it (q8_0_gemv_fused), and the
 * gate/up GEMV can write the SwiGLU output's plane itself (q8_0_gemv_gate_up).
 *
 * Formats
 *   Q8_0 weight block: 34 bytes -- little-endian f16 scale d at +0, then 32
 *     int8 values at +2.  A weight matrix of n rows and k columns is n rows of
 *     k/32 consecutive blocks (row pitch 34*k/32 bytes), with no padding.
 *     ("Part 4 - Lecture 05 - Fusion and the Activation-Quantization
 *     Discipline", sec. 2.1.)
 *   q8_0 activation plane: per token row t and 32-element block b,
 *       qs[t*k + 32*b + j]  int8, j = 0..31
 *       ds[t*(k/32) + b]    uint32: f16 bits of d in bits 0..15, the int16
 *                           block sum ssum = sum_j q_j in bits 16..31
 *     with d = amax/127 (computed in f32), q = rint(x * (1/d)) clamped to
 *     [-127, 127], d stored rounded to f16.  The plane has rows_pad >= rows
 *     rows; rows rows..rows_pad-1 are written as zeros.
 *     ("54 - r51 - producer-fused A-quantize mode 1", sec. 2.1 and 3.1.)
 *
 * Conventions for every entry point
 *   - All data pointers are DEVICE pointers owned by the caller; the library
 *     never allocates, frees or caches device memory between calls.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Work is enqueued asynchronously; the call returns before the
 *     GPU finishes.  Errors that only the GPU can detect (a bounded wait that
 *     ran out) are reported by q8_check().
 *   - Outputs are overwritten, never accumulated into, and must not alias
 *     any input.
 *   - Sizes are int64_t element counts; k must be a positive multiple of 32.
 *   - Pointers must be 16-byte aligned (Q8_ERR_ALIGN otherwise).
 *   - The return value is a status code (Q8_OK = 0).  On a non-zero return
 *     nothing was enqueued.  There is no fallback path: a rejected shape is
 *     an error, not a slow path.
 */
#ifndef Q8PROJ_H
#define Q8PROJ_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define Q8_API __attribute__((visibility("default")))
#else
#define Q8_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

#define Q8_OK                 0
#define Q8_ERR_ARG            1  /* NULL pointer, non-positive or inconsistent size, k % 32 != 0 */
#define Q8_ERR_ALIGN          2  /* a pointer is not 16-byte aligned */
#define Q8_ERR_DEVICE         3  /* current device is not sm_103 (GB300) or cannot be queried */
#define Q8_ERR_LAUNCH         4  /* the kernel launch failed (cudaGetLastError) */
#define Q8_ERR_DEVICE_TIMEOUT 5  /* a bounded on-device wait ran out (reported by q8_check) */
#define Q8_ERR_CUDA           6  /* another CUDA runtime error (stream sync, symbol copy) */
#define Q8_ERR_TOO_BIG        7  /* the request needs more than the fixed scratch of q8_0_gemm_noalloc */

/* Recommended number of plane rows for `rows` tokens: rows rounded up to a
 * multiple of 128 (the GEMM's token tile).  Any rows_pad >= rows is accepted
 * by every entry point; this is a convenience only. */
Q8_API int64_t q8_plane_rows(int64_t rows);

/* Human-readable name of a status code (static storage; never NULL). */
Q8_API const char *q8_strerror(int status);

/*
 * quantize_q8_0 -- standalone q8_0 quantizer (the "prepass").
 *   x   : f32 [rows][k] row-major (input)
 *   qs  : int8 [rows_pad][k] (output plane values)
 *   ds  : uint32 [rows_pad][k/32] (output packed d | ssum)
 * rows >= 0 (rows = 0 only zero-fills), rows_pad >= max(rows, 1), k % 32 == 0.
 * Defined by the quantize body of "54 - r51 - producer-fused A-quantize
 * mode 1", sec. 3.2, and the zero tail of sec. 3.1.
 */
Q8_API int quantize_q8_0(const float *x, int64_t rows, int64_t k,
                  int8_t *qs, uint32_t *ds, int64_t rows_pad, void *stream);

/*
 * rmsnorm_quant -- RMSNorm fused with q8_0 quantization of its output.
 *   x   : f32 [rows][d] (input)       w : f32 [d] (input weight)
 *   y   : f32 [rows][d] (output, y = (x * rsqrt(mean(x^2) + eps)) * w), or
 *         NULL when y is dead -- every consumer reads the plane -- and only
 *         the plane is written ("mode 2", the sequel that "54 - r51 -
 *         producer-fused A-quantize mode 1" sec. 5 points to: the f32 write
 *         and its re-read are what is left to remove).
 *   qs, ds : plane of y with rows_pad rows (output); the plane is exactly the
 *            q8_0 encoding of the f32 values y holds (or would hold), the
 *            same bytes whether y is written or not.
 * d % 32 == 0, d <= 32768 (the row is held in registers), rows >= 0,
 * rows_pad >= max(rows, 1).
 * "54 - r51 - producer-fused A-quantize mode 1", sec. 2.3 and 3.2
 * (rms_norm_quant_f32_t: one pass writes y and the plane).
 */
Q8_API int rmsnorm_quant(const float *x, const float *w, float eps, float *y,
                  int64_t rows, int64_t d,
                  int8_t *qs, uint32_t *ds, int64_t rows_pad, void *stream);

/*
 * swiglu_quant -- SwiGLU fused with q8_0 quantization of its output.
 *   gate, up : f32 [rows][nf] (inputs)
 *   y        : f32 [rows][nf] (output, y = gate / (1 + exp(-gate)) * up), or
 *              NULL when y is dead (mode 2, as for rmsnorm_quant): 4 of the
 *              13.125 bytes per element this call moves are that write.
 *   qs, ds   : plane of y (output), exactly the q8_0 encoding of y, the same
 *              bytes whether y is written or not.
 * nf % 32 == 0, rows >= 0, rows_pad >= max(rows, 1).
 * "54 - r51 - producer-fused A-quantize mode 1", sec. 3.2
 * (swiglu_quant_f32_t).
 */
Q8_API int swiglu_quant(const float *gate, const float *up, float *y,
                 int64_t rows, int64_t nf,
                 int8_t *qs, uint32_t *ds, int64_t rows_pad, void *stream);

/*
 * q8_0_gemv -- batch-1 projection y[i] = sum_b d_w(i,b) * d_a(b) * sum_j qw*qa.
 *   w      : n rows of k/32 Q8_0 blocks (input, 16-byte aligned base)
 *   qs, ds : plane row 0 (input; only row 0 is read)
 *   y      : f32 [n] (output)
 * n >= 1, k % 32 == 0.  Row grouping and the split of k across warps are
 * chosen from (n, k) alone, deterministically; results are run-to-run
 * identical.  "Part 4 - Lecture 05", sec. 2.1-2.4.
 * The kernel is launched with programmatic dependent launch: it may start
 * streaming `w` while the kernel enqueued just before it on `stream` is
 * still running, and reads the plane only after that kernel has finished.
 * `w` (the model weights) must therefore not be written by the kernel
 * immediately preceding the call on the same stream.
 */
Q8_API int q8_0_gemv(const void *w, int64_t n, int64_t k,
              const int8_t *qs, const uint32_t *ds, float *y, void *stream);

/*
 * q8_0_gemv_grouped -- several batch-1 projections of ONE activation in one
 * launch: for each i < count, projs[i].y[r] = sum_b d_w * d_a * isum over the
 * rows of projs[i].w, all against plane row 0 of (qs, ds) with the same k.
 *   projs : host array of `count` descriptors (read during the call only);
 *           each w and y is a device pointer as for q8_0_gemv, n >= 1.
 *   count : 1..Q8_MAX_GROUP.
 * Rows of all projections are spread over the whole GPU together, so small
 * projections ride along with large ones instead of each paying a launch and
 * a partly idle grid.  Same numerics as q8_0_gemv (one row is always computed
 * the same way), and the same programmatic-dependent-launch precondition on w.
 * "Part 4 - Lecture 05", sec. 2.5 (one launch for the consumers of one
 * activation) and sec. 6 (generalised to projections of different widths).
 * When (k/32) % 8 != 0 the projections are launched one by one.
 */
#define Q8_MAX_GROUP 8
typedef struct q8_gemv_proj {
    const void *w;   /* n rows of k/32 Q8_0 blocks */
    int64_t n;       /* rows (outputs) */
    float *y;        /* f32 [n] output */
} q8_gemv_proj;

Q8_API int q8_0_gemv_grouped(const q8_gemv_proj *projs, int count, int64_t k,
                             const int8_t *qs, const uint32_t *ds, void *stream);

/*
 * q8_0_gemv_fused -- q8_0_gemv_grouped with its one-row producer in the same
 * launch: every CTA computes the producer's f32 row and its q8_0 encoding
 * straight into the shared memory it would otherwise fill from a plane, so
 * the producer's launch, the plane's write and re-read, and the hand-off
 * between two launches disappear.
 *   producer : Q8_PRODUCER_QUANT    a = x f32 [k]            (as quantize_q8_0)
 *              Q8_PRODUCER_RMSNORM  a = x f32 [k], norm_w = w f32 [k], eps
 *                                   (as rmsnorm_quant)
 *              Q8_PRODUCER_SWIGLU   a = gate f32 [k], b = up f32 [k]
 *                                   (as swiglu_quant)
 *              unused pointers may be NULL; all inputs are read only.
 *   projs, count, k : as for q8_0_gemv_grouped; each projs[i].y is written.
 * Result: bit for bit what the standalone producer (one row, rows_pad at most
 * the SM count -- e.g. q8_plane_rows(1)) followed by q8_0_gemv_grouped on its
 * plane returns: the producer arithmetic is one implementation shared by both
 * paths, and for RMSNorm the row's sum of squares is formed in the standalone
 * kernel's order.  No f32 row or plane is written.
 * Requires (k/32) % 8 == 0 and k <= 65536 (the staged path), k <= 32768 for
 * RMSNorm; otherwise Q8_ERR_ARG (run the producer and the GEMV as two calls).
 * Pointers 16-byte aligned (Q8_ERR_ALIGN).  The producer's inputs are read
 * only after the kernel enqueued before the call on `stream` has finished
 * (the same programmatic-dependent-launch rule as q8_0_gemv: the weights may
 * be streamed earlier); the outputs must not overlap the inputs.
 * "Part 4 - Lecture 05", sec. 3 (a one-row quantize costs a launch, not
 * bandwidth) and sec. 4 (its rule: make producer and consumer one launch, and
 * keep one implementation for the fused and the unfused path).
 */
#define Q8_PRODUCER_QUANT   1
#define Q8_PRODUCER_RMSNORM 2
#define Q8_PRODUCER_SWIGLU  3
Q8_API int q8_0_gemv_fused(const q8_gemv_proj *projs, int count, int64_t k, int producer,
                           const float *a, const float *b, const float *norm_w, float eps,
                           void *stream);

/*
 * q8_0_gemv_gate_up -- the gate and up projections of one token with SwiGLU
 * and its q8_0 encoding in the same launch: gate = Wg.x, up = Wu.x (x from
 * plane row 0 of (qs, ds), or produced in the launch as for q8_0_gemv_fused),
 * and the plane row of silu(gate) * up written straight to (qs_out, ds_out)
 * -- the input of the down projection -- with no f32 SwiGLU output and no
 * separate SwiGLU launch.  Row r of gate and row r of up are computed by the
 * same CTA; the warp that completes the 32 rows of a block encodes it.
 *   w_gate, w_up : nf rows of k/32 Q8_0 blocks each (inputs)
 *   qs, ds       : activation plane row 0 when producer == 0, else unused
 *   producer     : 0, Q8_PRODUCER_QUANT (a = x) or Q8_PRODUCER_RMSNORM
 *                  (a = x, norm_w, eps), as for q8_0_gemv_fused
 *   y_gate, y_up : f32 [nf] outputs, or NULL when not wanted
 *   qs_out       : int8 [nf], ds_out : uint32 [nf/32] -- one plane row (row 0
 *                  of a plane; other rows are not touched)
 * Result: y_gate / y_up bit for bit as q8_0_gemv_grouped (or _fused) writes
 * them, and the plane bit for bit as swiglu_quant writes it for those values
 * (the same SwiGLU and encoding arithmetic).
 * Requires nf % 32 == 0, (k/32) % 8 == 0, 2048 < k <= 65536 (whole rows per
 * warp on the staged path), k <= 32768 for RMSNorm; otherwise Q8_ERR_ARG.
 * Pointers 16-byte aligned (Q8_ERR_ALIGN).  The same programmatic-dependent-
 * launch rule as q8_0_gemv; outputs must not overlap inputs.
 * "54 - r51 - producer-fused A-quantize mode 1", sec. 3.2 (swiglu_quant_f32_t:
 * SwiGLU and the quantize of its output in one pass) and sec. 6 (consume the
 * data where it is hottest: here the registers of the gate/up GEMV); "Part 4 -
 * Lecture 05", sec. 4 (one launch instead of a buffer passed between two).
 */
Q8_API int q8_0_gemv_gate_up(const void *w_gate, const void *w_up, int64_t nf, int64_t k,
                             const int8_t *qs, const uint32_t *ds,
                             int producer, const float *a, const float *norm_w, float eps,
                             float *y_gate, float *y_up, int8_t *qs_out, uint32_t *ds_out,
                             void *stream);

/*
 * q8_0_gemv_batched -- the projection for a few tokens at once (decode over
 * a small batch of sequences): Y[t][i] = sum_b d_w(i,b) * d_a(t,b) * isum for
 * plane rows t < tokens, reading the weights from memory once for all of
 * them.  The formula is the GEMM's ("12 - r5-r6 re-ranking + structural
 * rewrite spec", sec. 2); the pages build only its two ends, the batch-1 GEMV
 * and the prefill GEMM, and this entry point fills the range between them.
 *   w      : n rows of k/32 Q8_0 blocks (input, 16-byte aligned)
 *   qs, ds : plane with at least `tokens` rows (input; rows >= tokens are
 *            not read)
 *   y      : f32 [tokens][n] row-major (output, overwritten)
 * 1 <= tokens <= Q8_GEMV_MAX_TOKENS, n >= 1, k % 32 == 0.  When
 * (k/32) % 8 == 0 the block dot products run on the tensor cores (int8 codes
 * widened exactly to f16, f32 accumulation of an exact integer) and each
 * block adds (d_w * d_a) * isum to one of four partial sums over k, which are
 * added in a fixed order: results are run-to-run identical.  Other k use the
 * generic kernel (weights read once per token).  Programmatic dependent
 * launch, with the same precondition on w as q8_0_gemv.
 * q8_0_gemm hands calls with t <= Q8_GEMV_MAX_TOKENS to this path (t == 1 to
 * q8_0_gemv), and calls with Q8_GEMV_MAX_TOKENS < t <= 64 to this path over
 * consecutive 16-token slices of the plane (each slice streams the weights
 * again; up to four passes cost less than the GEMM's pre-pass).
 */
#define Q8_GEMV_MAX_TOKENS 16
Q8_API int q8_0_gemv_batched(const void *w, int64_t n, int64_t k,
                             const int8_t *qs, const uint32_t *ds, int64_t tokens,
                             float *y, void *stream);

/*
 * q8_0_gemv_batched_grouped -- q8_0_gemv_batched for several projections of
 * the same activation rows in one launch: for each i < count,
 *     projs[i].y[t][r] = sum_b d_w(r,b) * d_a(t,b) * isum   (t < tokens)
 * over the rows of projs[i].w, all with the same k and plane.
 *   projs : host array of `count` descriptors (read during the call only);
 *           w and y are device pointers (16-byte aligned); y is f32
 *           [tokens][projs[i].n] row-major.
 *   count : 1..Q8_MAX_GROUP.
 *   qs, ds, tokens : as for q8_0_gemv_batched.
 * The projections' 128-row tiles form one grid, so a narrow projection (a
 * K or V of grouped-query attention) rides along with a wide one instead of
 * paying its own launch and a partly idle GPU.  The per-block arithmetic is
 * q8_0_gemv_batched's; the number of CTAs that split k for one tile (1..8) is
 * chosen from the launch's total tile count, so the partial sums over k may
 * be grouped differently than in a single call of one projection (equal bit
 * for bit where that number is the same).  Results are run-to-run identical.
 * When (k/32) % 8 != 0 the projections run one by one on the generic kernel.
 * Errors: Q8_ERR_ARG (count, shape, tokens, a NULL pointer), Q8_ERR_ALIGN,
 * Q8_ERR_DEVICE, Q8_ERR_LAUNCH.  Programmatic dependent launch as for
 * q8_0_gemv.  "Part 4 - Lecture 05", sec. 2.5 (one launch for the consumers
 * of one activation), applied to the small-batch formula above.
 */
Q8_API int q8_0_gemv_batched_grouped(const q8_gemv_proj *projs, int count, int64_t k,
                                     const int8_t *qs, const uint32_t *ds, int64_t tokens,
                                     void *stream);

/*
 * q4a_gemv -- batch-1 projection with asymmetric 4-bit weight blocks, the
 * consumer of the plane's int16 block sums:
 *     y[i] = sum_b ( d*d_a * sum_e nib_e*q_e  -  m*d_a * ssum_b ).
 * The weight value d*nib - m is the q4_K form d*s*nib - dmin*m of "12 - r5-r6
 * re-ranking + structural rewrite spec" (sec. 3) with one f16 scale and one
 * f16 min per 32 elements, and its min term takes the plane's ssum instead
 * of a second dot product, the use "54 - r51 - producer-fused A-quantize
 * mode 1" (sec. 2.1) gives the int16 field.
 *   w      : n rows of k/32 20-byte blocks (input, 16-byte aligned): f16 d at
 *            +0, f16 m at +2, then byte j (j < 16) holds element j in its low
 *            nibble and element j + 16 in its high nibble (unsigned 0..15).
 *   qs, ds : plane row 0 (input; only row 0 is read)
 *   y      : f32 [n] (output)
 * n >= 1, k % 128 == 0 (16-byte aligned rows of whole 4-block chunks),
 * k <= 206592 (the activation is staged in shared memory).  Per block two
 * fmas, d*d_a*isum then -m*d_a*ssum (both scale products exact in f32); the
 * split of a row over lanes depends on k only: results are run-to-run
 * identical.  Programmatic dependent launch: the plane is read only after the
 * kernel enqueued before it on `stream` has finished.
 */
Q8_API int q4a_gemv(const void *w, int64_t n, int64_t k,
                    const int8_t *qs, const uint32_t *ds, float *y, void *stream);

/*
 * q4a_gemv_batched -- the asymmetric 4-bit projection for a few tokens at
 * once, the weights streamed from HBM once for all of them:
 *     Y[t][i] = sum_b ( d*d_a(t,b) * sum_e nib_e*q_e(t)  -  m*d_a(t,b) * ssum(t,b) )
 * for tokens t < `tokens`.  Same weight blocks as q4a_gemv.
 *   qs, ds : plane rows 0..tokens-1 (input; rows at and past `tokens` are not
 *            read)
 *   y      : f32 [tokens][n] (output)
 * 1 <= tokens <= Q8_GEMV_MAX_TOKENS; k % 256 == 0 (8-block row pieces);
 * tokens == 1 runs q4a_gemv.  Per block: the exact integer dot of the nibbles
 * with the codes, then fma(d*d_a, isum) and fma(-(m*d_a), ssum) (scale
 * products exact in f32).  Partial sums over k are added in a fixed order:
 * results are run-to-run identical.  Errors: Q8_ERR_ARG (shape, tokens),
 * Q8_ERR_ALIGN (a pointer not 16-byte aligned), Q8_ERR_DEVICE (not sm_103),
 * Q8_ERR_LAUNCH.  Programmatic dependent launch as for q4a_gemv.
 */
Q8_API int q4a_gemv_batched(const void *w, int64_t n, int64_t k,
                            const int8_t *qs, const uint32_t *ds, int64_t tokens,
                            float *y, void *stream);

/*
 * q4a_gemv_batched_grouped -- q4a_gemv_batched for up to Q8_MAX_GROUP
 * projections of the same plane rows, as q8_0_gemv_batched_grouped is for
 * Q8_0 weights: projs[i].w holds projs[i].n rows of the 20-byte asymmetric
 * blocks, projs[i].y is f32 [tokens][projs[i].n]; k % 256 == 0, 1 <= tokens
 * <= Q8_GEMV_MAX_TOKENS.  For tokens >= 2 the projections' row tiles form one
 * launch of the small-batch kernel (per block the arithmetic of
 * q4a_gemv_batched; the number of CTAs splitting k follows the launch's total
 * tile count, so partial sums may be grouped differently than in a single
 * call, bit for bit equal where that number is the same); tokens == 1 runs
 * q4a_gemv projection by projection.  Errors as q4a_gemv_batched, plus
 * Q8_ERR_ARG for count outside 1..Q8_MAX_GROUP or a NULL descriptor.
 */
Q8_API int q4a_gemv_batched_grouped(const q8_gemv_proj *projs, int count, int64_t k,
                                    const int8_t *qs, const uint32_t *ds, int64_t tokens,
                                    void *stream);

/*
 * q8_0_gemm_workspace_bytes -- device workspace q8_0_gemm needs for n weight
 * rows, t tokens and width k: the weight codes as f16 (n*k*2 bytes), the
 * activation codes as f16 (t*k*2), and both sides' block scales as f32
 * (k/32 * 4 bytes per weight row and per token, rows and tokens rounded up to
 * the GEMM's 128 x 192 tiles), each part starting on a 1 KiB boundary; when
 * the tiles would leave most SMs idle (few weight rows or tokens) k is split
 * over up to 12 CTAs per tile and the workspace also holds their f32 partial
 * outputs (splits * t * n * 4 bytes, added in a fixed order by a reduction
 * kernel; splits * tiles <= 152, so at most about 15 MB).  The size depends
 * on (n, t, k) only.  0 when (k/32) % 8 != 0 or t <= 64 (those calls run
 * the generic or small-batch kernels and need none).
 */
Q8_API size_t q8_0_gemm_workspace_bytes(int64_t n, int64_t t, int64_t k);

/*
 * q8_0_gemm -- prefill projection Y[t][i] = sum_b d_w(i,b) * d_a(t,b) * isum.
 *   w      : n rows of k/32 Q8_0 blocks (input)
 *   qs, ds : plane with rows_pad >= t rows (input; rows >= t are not read)
 *   y      : f32 [t][n] row-major (output)
 *   workspace, workspace_bytes : caller-owned device scratch of at least
 *            q8_0_gemm_workspace_bytes(n, t, k) bytes, 16-byte aligned; its
 *            contents on entry are ignored and on return are unspecified.
 *            Two calls may share a workspace only if they are ordered on one
 *            stream.  May be NULL when that size is 0.
 * n >= 1, t >= 1, k % 32 == 0.  Every 32-wide k block is one q8_0 block on
 * both sides, so its integer dot product is scaled by d_w * d_a once.
 * Dispatch by shape: t == 1 -> q8_0_gemv; (k/32) % 8 != 0 -> the generic
 * kernel; t <= 64 -> q8_0_gemv_batched's kernel (over 16-token slices above
 * 16 tokens); otherwise the call enqueues two pre-passes that write the
 * weight codes and the plane's codes as f16 (exact) and both sides' block
 * scales as f32 into the workspace, then the tcgen05 GEMM (split over k when
 * its tiles alone would leave most SMs idle, with a reduction kernel after
 * it), all with programmatic dependent launch and the same precondition on w
 * as q8_0_gemv.
 * "12 - r5-r6 re-ranking + structural rewrite spec", sec. 2 and 3.1;
 * "54 - r51 - producer-fused A-quantize mode 1", sec. 2.1.
 */
Q8_API int q8_0_gemm(const void *w, int64_t n, int64_t k,
                     const int8_t *qs, const uint32_t *ds, int64_t t, int64_t rows_pad,
                     float *y, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Prepared weights for the prefill GEMM.  A model's weights do not change
 * between calls, so the weight pre-pass that q8_0_gemm enqueues on every
 * call (the codes widened to f16 exactly, d_w as f32 in the epilogue's
 * order) can run once per matrix instead:
 *
 * q8_0_gemm_prepared_weights_bytes -- size of the prepared form of an n x k
 * Q8_0 matrix: n*k*2 bytes of f16 codes and k/32*4 bytes of d_w per weight
 * row (rows rounded up to the GEMM's 128-row tiles), each part starting on a
 * 1 KiB boundary.  0 when (k/32) % 8 != 0 or the shape is past the GEMM's
 * grid limits (n > 65535*128, k > 2^30).
 *
 * q8_0_gemm_prepare_weights -- write that form of w into wprep (caller-owned
 * device memory of at least q8_0_gemm_prepared_weights_bytes(n, k) bytes,
 * 16-byte aligned; its layout is private to this library and valid for this
 * (n, k) only).  One kernel, enqueued on `stream` with programmatic dependent
 * launch.  Q8_ERR_ARG for a NULL pointer, a short buffer or a shape the GEMM
 * does not take, Q8_ERR_ALIGN for misaligned pointers.
 *
 * q8_0_gemm_prepared_workspace_bytes -- device workspace q8_0_gemm_prepared
 * needs: q8_0_gemm_workspace_bytes without the two weight parts.  0 when the
 * call takes a path that needs none (t <= 64 or (k/32) % 8 != 0).
 *
 * q8_0_gemm_prepared -- q8_0_gemm whose tcgen05 path reads prepared weights:
 * the same result, bit for bit, as q8_0_gemm(w, ...) (the same kernels on
 * the same operands), without the per-call weight pre-pass.
 *   w      : the Q8_0 matrix, read by the paths for t <= 64 and for
 *            (k/32) % 8 != 0; may be NULL when the call takes the tcgen05
 *            path (t > 64 and (k/32) % 8 == 0)
 *   wprep  : q8_0_gemm_prepare_weights(w, n, k, ...)'s output, read by the
 *            tcgen05 path (may be NULL otherwise).  Written earlier on this
 *            stream, or ordered before this call by the caller.
 *   qs, ds, t, rows_pad, y : as for q8_0_gemm
 *   workspace, workspace_bytes : at least
 *            q8_0_gemm_prepared_workspace_bytes(n, t, k) bytes, as for
 *            q8_0_gemm
 * "12 - r5-r6 re-ranking + structural rewrite spec", sec. 2 and 3.1 (the
 * per-block scale correction); "54 - r51 - producer-fused A-quantize mode 1",
 * sec. 2.1 (the plane).
 */
Q8_API size_t q8_0_gemm_prepared_weights_bytes(int64_t n, int64_t k);
Q8_API int q8_0_gemm_prepare_weights(const void *w, int64_t n, int64_t k,
                                     void *wprep, size_t wprep_bytes, void *stream);
Q8_API size_t q8_0_gemm_prepared_workspace_bytes(int64_t n, int64_t t, int64_t k);
Q8_API int q8_0_gemm_prepared(const void *w, const void *wprep, int64_t n, int64_t k,
                              const int8_t *qs, const uint32_t *ds, int64_t t, int64_t rows_pad,
                              float *y, void *workspace, size_t workspace_bytes, void *stream);

/*
 * q8_0_gemm_noalloc -- q8_0_gemm without a workspace argument, for callers
 * that cannot allocate device memory at this point: a serving engine that
 * handed all of the GPU's memory to its own pool at start-up, a plugin whose
 * host application forbids allocation after initialisation, or a
 * latency-critical path that cannot pay for cudaMalloc's implicit device
 * synchronisation.  The pages have no counterpart of this entry point; it
 * exists for those callers only.
 *   Arguments, results and numerics are those of q8_0_gemm (same kernels).
 *   The scratch q8_0_gemm takes from `workspace` comes instead from a 32 MiB
 *   array that is part of this library's device code
 *   (q8_0_gemm_noalloc_max_bytes()).  Every GPU that loads the library's GEMM
 *   code holds those 32 MiB until the process exits.  A request whose
 *   q8_0_gemm_workspace_bytes(n, t, k) exceeds it returns Q8_ERR_TOO_BIG
 *   (the f16 copies of both operands must fit: small projections, or t <= 64
 *   which needs no scratch at all).
 *   The entry point itself calls no cudaMalloc/cudaFree or allocating
 *   routine.  Its first call on a device looks up that device's address of
 *   the array (cudaGetSymbolAddress, with the device current), and so does
 *   the first call after the device's context has been replaced (for
 *   instance by cudaDeviceReset); make those calls before any stream capture.
 *   All calls share the one array and it keeps the last call's contents;
 *   nothing in it needs to start at zero (each call rewrites every byte it
 *   reads), but calls that overlap on the GPU -- different streams, or
 *   different host threads -- race on it and give undefined results.
 */
Q8_API int q8_0_gemm_noalloc(const void *w, int64_t n, int64_t k,
                             const int8_t *qs, const uint32_t *ds, int64_t t, int64_t rows_pad,
                             float *y, void *stream);

/* Size in bytes of the fixed scratch behind q8_0_gemm_noalloc. */
Q8_API size_t q8_0_gemm_noalloc_max_bytes(void);

/*
 * q8_0_gemm_mma -- the same contraction as q8_0_gemm on the warp-level int8
 * tensor instruction (mma.sync.m16n8k32.s8) instead of tcgen05: the legacy
 * tensor path, kept as an exact A/B baseline for q8_0_gemm.  Requires
 * (k/32) % 8 == 0 (Q8_ERR_ARG otherwise); arguments as q8_0_gemm.
 */
Q8_API int q8_0_gemm_mma(const void *w, int64_t n, int64_t k,
                         const int8_t *qs, const uint32_t *ds, int64_t t, int64_t rows_pad,
                         float *y, void *stream);

/*
 * q8_check -- synchronise `stream`, then read and clear the library's device
 * error word.  Returns Q8_OK, Q8_ERR_DEVICE_TIMEOUT if a bounded on-device
 * wait ran out since the last check (the affected outputs are undefined), or
 * Q8_ERR_CUDA if the synchronisation itself failed.
 */
Q8_API int q8_check(void *stream);

/* Number of SMs of the current device (0 on error); used by the host-side
 * dispatch and exported for tests. */
Q8_API int q8_num_sms(void);

#ifdef __cplusplus
}
#endif
#endif /* Q8PROJ_H */
