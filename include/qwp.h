/*
 * qwp -- batched-prefill GEMM over 4-bit quantized weights on GB300 (sm_103a).
 *
 * C ABI.  Every pointer argument named *_dev is a device pointer; every call
 * is asynchronous and ordered on `stream` (a cudaStream_t passed as void*,
 * NULL = the legacy default stream) and never synchronizes the host, except
 * qwp_device_status.  The caller owns and allocates every input and output
 * buffer.  Device memory of the library's own comes from a library-owned,
 * stream-ordered pool, released in stream order after the call: the fp16 copy
 * of x taken by q4k_gemm, q6k_gemm and w4a16_gemm_bf16, and, for decode-shaped
 * calls of any GEMM entry point (see below), the decode kernel's partial sums.
 * Every kernel of the library is launched with programmatic stream
 * serialization and waits for the grids before it (griddepcontrol.wait) before
 * touching memory they may write or read.
 *
 * Decode-shaped calls.  A GEMM with 1 <= M <= 8 tokens, K % 256 == 0 and at
 * least 600 (128-row tile, 256-wide super-block) items (ceil(N/128) * K/256)
 * can run a second kernel made for that regime ("How ZINC's RDNA4 batched
 * prefill went from 42 to 208 tok/s", section "The fix: K-parallel batched
 * DMMV"): same weights, same operand rounding and the same error bound, bf16
 * activations converted inside the kernel, and G * 8 KiB + ceil(N/128) * 4
 * bytes of pool scratch (G: the decode grid, at most 2 CTAs per SM) for the
 * tiles its CTAs share.
 * Results are deterministic (shared tiles are summed in a fixed order).  By
 * default (QWP_DECODE_AUTO) it takes such products only where it measured
 * faster than the prefill kernel on GB300: M <= 2 and N >= 24576 for Q4_K, N >=
 * 65536 for Q6_K, N >= 24576 at one token and N >= 65536 at two for W4A16; see
 * qwp_set_decode_policy.
 * Skinny-N calls.  A Q4_K product with at most 64 weight rows (N <= 64) and at
 * least 256 tokens runs a third kernel ("Skinny bf16 GEMM prefill_gemm_skinny.cu",
 * sparkinfer PR #511, Summary table): tokens are the tensor core's M side and
 * the activations are its operand as they are (bf16 or fp16, never converted),
 * K is split over a thread-block cluster and summed through distributed shared
 * memory in a fixed order.  With fp16 x the weights are the same single-rounded
 * fp16 operand as above; with bf16 x each weight is the pair hi = bf16(w32),
 * lo = bf16(w32 - hi) of its fp32 value w32, both multiplied with x (x.hi and
 * x.lo accumulated apart in fp32 and added at the end; relative weight error at
 * most 2^-18 + 2^-24, so no range limit on x and no QWP_ERR_RANGE).  Token
 * tiles of up to 128 tokens are cut so that the clusters fill the GPU in whole
 * waves.  It allocates nothing.
 * Every entry point returns QWP_OK (0) or a negative qwp_status; none throws.
 * Calls are thread-safe, with one exception: q4k_gemm_noalloc keeps its scratch
 * in fixed arrays that all its calls on a device share, so its calls must not
 * overlap on the GPU (see there).
 *
 * The method (web pages, by title and section):
 *  - "The dequant scratch round-trip is ZINC's last RDNA4 prefill tax",
 *    sections "The two passes hiding inside one matmul" and "What the
 *    roofline says": y = x . W^T where each 4-bit weight block is read from
 *    memory once (0.5625 byte per Q4_K weight), unpacked on chip and consumed
 *    by the matmul tile; no 16-bit copy of the weights is ever written.
 *  - "How ZINC's RDNA4 batched prefill went from 42 to 208 tok/s", sections
 *    "The two prefill paths" and "The fix: K-parallel batched DMMV": each
 *    weight row is read once per chunk of prompt tokens and applied to all of
 *    them; a stripe decodes as factor * q - bias.
 *  - "[ROCm][Perf] W4A16: packed fp16 prefill dequant", section "1. Packed
 *    fp16 dequant": the interleaved int4 word and the exact 0x6400|n unpack.
 *
 * Shapes.  x is [M, K] row-major, W is [N, K] (K contiguous within a row),
 * y is [M, N] row-major fp32 and is overwritten (y = x . W^T).
 */
#ifndef QWP_H
#define QWP_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define QWP_API __attribute__((visibility("default")))
#else
#define QWP_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    QWP_OK = 0,
    QWP_ERR_INVALID_ARG = -1,      /* null pointer, negative size, bad group size      */
    QWP_ERR_UNSUPPORTED_SHAPE = -2,/* K not a multiple of 256 (Q4_K) or of 64/group     */
    QWP_ERR_MISALIGNED = -3,       /* a device pointer is not 16-byte aligned            */
    QWP_ERR_CUDA = -4,             /* a CUDA runtime/driver call or a launch failed      */
    QWP_ERR_DEVICE = -5,           /* the current device is not an sm_103 GPU            */
    QWP_ERR_TIMEOUT = -6,          /* a kernel's bounded wait expired (qwp_device_status) */
    QWP_ERR_RANGE = -7,            /* an activation overflowed fp16 (qwp_device_status)   */
    QWP_ERR_SCRATCH_LIMIT = -8     /* q4k_gemm_noalloc: M*K beyond QWP_NOALLOC_MAX_X_ELEMS */
} qwp_status;

/* Human-readable name of a status code (static string). */
QWP_API const char *qwp_status_string(int status);

/*
 * Q4_K (GGML super-blocks of 256 weights along K, 144 bytes each: fp16 d,
 * fp16 dmin, 12 bytes of packed 6-bit scales[8]/mins[8], 128 bytes of
 * nibbles; w = d*sc_j*q - dmin*m_j).  Source: the GGML block format and the
 * "factor * q - bias" stripe of "How ZINC's RDNA4 batched prefill went from
 * 42 to 208 tok/s", section "The fix: K-parallel batched DMMV".
 */

/* Bytes of a repacked Q4_K matrix: N*K/256*144 (the repack is a byte permutation). */
QWP_API int q4k_repacked_bytes(int64_t N, int64_t K, size_t *out_bytes);

/*
 * Load-time repack of GGML Q4_K rows (w_ggml_dev: N rows of K/256 blocks,
 * row-major, N*K/256*144 bytes) into the tile-major order the GEMM streams
 * (w_tiled_dev, same size, caller-allocated, must not alias w_ggml_dev):
 * rows in tiles of 128; per tile and super-block a 16-byte header plane and
 * four 32-byte nibble planes.  K % 256 == 0.  Both pointers 16-byte aligned.
 */
QWP_API int q4k_repack(const void *w_ggml_dev, void *w_tiled_dev, int64_t N, int64_t K, void *stream);

/*
 * Test entry point: dequantize a repacked Q4_K matrix to fp32 w_out_dev[N][K].
 * Each value is the correctly rounded fp32 of d*sc*q - dmin*m (exact for all
 * finite fp16 d, dmin whose products fit fp32's range), computed by the same
 * unpack the GEMM uses.
 */
QWP_API int q4k_dequant(const void *w_tiled_dev, float *w_out_dev, int64_t N, int64_t K, void *stream);

/*
 * y_dev[M][N] (fp32) = x_dev[M][K] (fp16) . W^T, W the repacked Q4_K matrix.
 * Each weight is unpacked on chip to an fp16 tensor-core operand that is the
 * fp16 rounding of the exact weight d*sc*q - dmin*m: q*sc exactly (from the
 * 0x6400|n form of the nibble), d*(q*sc) - dmin*m in fp32 with an exact product
 * and an exact dmin*m, then one rounding to fp16 (relative error at most
 * 2^-11 * (1 + 2^-13); weights in fp16's subnormal range are exact, since every
 * weight is a multiple of 2^-24; requires |w| <= 65504, true of any practical
 * block); fp32 accumulation in tensor memory.  K % 256 == 0; M, N >= 0 (M == 0 or
 * N == 0 is a no-op); x_dev, w_tiled_dev and y_dev 16-byte aligned; x rows
 * contiguous (row stride K).  Allocates nothing, except the decode kernel's
 * scratch for decode-shaped calls.  Skinny-N calls (above) take the skinny-N
 * kernel.
 */
QWP_API int q4k_gemm_f16(const void *w_tiled_dev, const void *x_dev, float *y_dev,
                         int64_t M, int64_t N, int64_t K, void *stream);

/*
 * The same product for bf16 activations: x is first converted to fp16 (exact
 * for |x| in [2^-14, 65504]; smaller values lose at most 2^-25 absolutely;
 * larger ones overflow, which qwp_device_status reports as QWP_ERR_RANGE) into
 * M*K*2 bytes of scratch taken from a library-owned, stream-ordered memory pool
 * on the current device and released in stream order after the GEMM; then
 * q4k_gemm_f16 runs, launched so that its set-up overlaps the conversion.  The
 * prefill kernel converts x itself, in shared memory (same rounding and range
 * report; no conversion kernel, no scratch), when each of its CTAs runs one
 * work unit and converts at most 32 KB of x, or 64 KB of at most 16 token rows
 * (for example M <= 32 at N = 2048, K = 2048; qwp_gemm_plan tells the plan), and
 * for one token (M == 1).
 * Skinny-N calls (above) take x as bf16 in the skinny-N kernel: no
 * conversion, no scratch, no range limit.  Same shape and alignment rules as
 * q4k_gemm_f16.
 */
QWP_API int q4k_gemm(const void *w_tiled_dev, const void *x_dev, float *y_dev,
                     int64_t M, int64_t N, int64_t K, void *stream);

/*
 * A batch of independent Q4_K products of one shape in one launch (strided
 * batch): for p = 0 .. batch-1, y_p[M][N] = x_p[M][K] . W_p^T with W_p the
 * repacked matrix at w_tiled_dev + p * q4k_repacked_bytes(N, K), x_p at
 * x_dev + p*M*K elements and y_p at y_dev + p*M*N floats.  The units (128-row
 * tile x token tile) of all problems share one persistent grid, so a batch of
 * small products pays the launch, the pipeline fill and the tail once (the way
 * to approach the HBM roofline with GEMMs too small to fill the GPU alone, e.g.
 * the experts of a mixture-of-experts layer).  Same operand rounding, error
 * bound and rules as q4k_gemm (bf16 x, converted to fp16 into pool scratch
 * first, batch*M*K*2 bytes, or by the kernel itself under the conditions
 * described for q4k_gemm) and q4k_gemm_f16 (fp16 x); always the prefill kernel.
 * The three base pointers are 16-byte aligned (QWP_ERR_MISALIGNED otherwise);
 * problem p's y, p*M*N floats on, need not be.  batch <= 65535, batch*M*K and
 * batch*M*N <= 2^40 (QWP_ERR_UNSUPPORTED_SHAPE otherwise); batch == 0 is a no-op.
 */
QWP_API int q4k_gemm_batched(const void *w_tiled_dev, const void *x_dev, float *y_dev, int64_t batch,
                             int64_t M, int64_t N, int64_t K, void *stream);
QWP_API int q4k_gemm_batched_f16(const void *w_tiled_dev, const void *x_dev, float *y_dev, int64_t batch,
                                 int64_t M, int64_t N, int64_t K, void *stream);

/*
 * The largest activation q4k_gemm_noalloc accepts: M*K <= 8,388,608 values
 * (for example M <= 2048 at K = 4096, M <= 682 at K = 12288).
 */
#define QWP_NOALLOC_MAX_X_ELEMS 8388608

/*
 * q4k_gemm without any device allocation, for callers that must not allocate:
 * engines that reserve all device memory up front and forbid allocation once
 * they serve, callers whose allocator owns the memory the CUDA pools would
 * draw from, and latency-bound loops in which an allocation's cost or its
 * possible failure is not acceptable.  Same arguments, rules and result as
 * q4k_gemm (the same kernels run); the fp16 copy of x goes into a fixed array
 * of QWP_NOALLOC_MAX_X_ELEMS fp16 values (16 MiB) that is part of the library
 * and that every GPU loading the library's device code holds until the process
 * exits (calls whose prefill kernel converts x itself, as described for
 * q4k_gemm, do not use it).  M*K beyond that size returns QWP_ERR_SCRATCH_LIMIT before
 * any work.
 * Decode-shaped calls keep their partial sums in a second fixed array (4 MiB)
 * instead and read x directly (no fp16 copy); a decode-shaped call whose
 * partial sums would not fit there (G * 8 KiB + ceil(N/128) * 4 bytes above
 * 4 MiB, i.e. N beyond about 16 million rows) runs the prefill kernel through
 * the first array instead, so QWP_ERR_SCRATCH_LIMIT means M*K above the limit
 * and nothing else.
 * The first call on each device looks up the array's address on that device
 * (and loads the library's device code there if it is not loaded yet); make
 * that first call before any stream capture begins.  Every call on a device
 * shares the one array and leaves its x in it; each call writes all it reads
 * first, so nothing needs clearing, but calls whose work overlaps on the GPU
 * (different streams with no event or other ordering between them) race on
 * the array and give wrong results.  The method's pages have no counterpart to
 * this entry point: it exists only for callers that cannot allocate.
 */
QWP_API int q4k_gemm_noalloc(const void *w_tiled_dev, const void *x_dev, float *y_dev,
                             int64_t M, int64_t N, int64_t K, void *stream);

/*
 * Quantized activations: the activation side of the DP4a path ("The dequant
 * scratch round-trip is ZINC's last RDNA4 prefill tax", section "What removing
 * it was worth": Q8_1 activations, quantized first, then multiplied still packed
 * with the 4-bit weights).  Each token row of x is cut into blocks of 32 along K;
 * block j gets d = amax/127 (amax its largest |x|), and every value the code
 * q = round-half-away-from-zero(x * (1/d)) (0 when d == 0), each operation
 * correctly rounded in fp32 (GGML's Q8_1 rule; d is kept in fp32, not fp16, and
 * the block sum s of the codes exactly).  The pages give the idea, not the
 * rounding rule: this is the reading taken.
 *
 * Buffer layout (device, 16-byte aligned, opaque to callers except for its
 * size): tokens in groups of 8, the last group padded with zero tokens; group g
 * and super-block b (256 values along K) form one 2560-byte record at
 * (g*K/256 + b)*2560, token t of the group at t*320 inside it: 256 int8 codes
 * (each run of 8 elements e0..e7 stored as e0 e4 e1 e5 e2 e6 e3 e7, the byte order
 * of the repacked Q4_K nibbles), then the 8 fp32 scales d and the 8 code sums s
 * (fp32, exact) of its 32-value blocks.
 */

/* Bytes of the quantized activations of M tokens: ceil(M/8) * (K/256) * 2560.  K % 256 == 0. */
QWP_API int q8_activation_bytes(int64_t M, int64_t K, size_t *out_bytes);

/*
 * Quantize x_bf16_dev[M][K] (bf16, rows contiguous) into xq_dev (at least
 * q8_activation_bytes).  K % 256 == 0; both pointers 16-byte aligned.  One
 * kernel, no allocation.  A non-finite activation sets the range flag that
 * qwp_device_status reports as QWP_ERR_RANGE (its codes are then undefined).
 */
QWP_API int q8_quantize(const void *x_bf16_dev, void *xq_dev, int64_t M, int64_t K, void *stream);

/*
 * y_dev[M][N] (fp32) = sum over k of W[n][k] * d[m][k/32] * q[m][k]: the Q4_K
 * product with the quantized activations xq_dev (from q8_quantize with the same
 * M and K), for decode-shaped calls, 1 <= M <= 8.  Per row, 32-value block and
 * token, the 32 products of 4-bit weight codes and 8-bit activation codes are
 * summed exactly in integers (dp4a), then combined in fp32 as
 * d_x * (d*sc * dot - dmin*m * s): the result is the product of the weights with
 * the dequantized activations d*q up to fp32 rounding, at most
 * (K/32 + 4) * 2^-24 * sum_k (|d*sc*q_w| + |dmin*m|) * |d_x*q_x| per element.
 * The quantization itself changes x by at most d/2 per value (half a code),
 * which this entry point does not undo: it trades that for reading one byte per
 * activation and one integer instruction per 4 weights.  Runs on the decode
 * kernel (stream-K over 128-row tiles and 256-wide super-blocks); takes its
 * scratch (partials of shared tiles) from the library's stream-ordered pool.
 * K % 256 == 0; pointers 16-byte aligned; M > 8 returns QWP_ERR_UNSUPPORTED_SHAPE.
 */
QWP_API int q4k_q8_gemm(const void *w_tiled_dev, const void *xq_dev, float *y_dev,
                        int64_t M, int64_t N, int64_t K, void *stream);

/*
 * Q6_K (GGML blocks of 256 weights along K, 210 bytes each: ql[128] low four
 * bits of the 6-bit codes, qh[64] high two bits, int8 scales[16] (one per 16
 * weights), fp16 d last; w = d * scale * (q - 32)).  Source: "How ZINC's RDNA4
 * batched prefill went from 42 to 208 tok/s", sections "Bug 2: Q6_K had a gate
 * but no dispatcher" and "What changed" (Q4_K_M checkpoints keep ffn_down and
 * attn_v in Q6_K and the batched path needs a Q6_K kernel); the pages name the
 * format only, the layout is GGML's.
 */

/*
 * Bytes of a repacked Q6_K matrix: (K/256)*210 per stored row, the stored rows
 * being N rounded up so that the last 128-row tile holds a multiple of 8 rows
 * (at most 7 zero rows of padding; equal to the GGML size when N % 8 == 0).
 */
QWP_API int q6k_repacked_bytes(int64_t N, int64_t K, size_t *out_bytes);

/*
 * Load-time repack of GGML Q6_K rows (w_ggml_dev: N rows of K/256 blocks,
 * row-major, N*K/256*210 bytes) into the tile-major order the GEMM streams
 * (w_tiled_dev, q6k_repacked_bytes bytes, caller-allocated, must not alias):
 * per 128-row tile and super-block a d plane, a scale plane, four planes of
 * interleaved low nibbles and four planes of high bits.  K % 256 == 0.  Both
 * pointers 16-byte aligned.
 */
QWP_API int q6k_repack(const void *w_ggml_dev, void *w_tiled_dev, int64_t N, int64_t K, void *stream);

/*
 * Test entry point: the correctly rounded fp32 of d*scale*(q - 32) of a
 * repacked Q6_K matrix into w_out_dev[N][K] (d*scale is exact in fp32; one
 * rounding of the product).
 */
QWP_API int q6k_dequant(const void *w_tiled_dev, float *w_out_dev, int64_t N, int64_t K, void *stream);

/*
 * y_dev[M][N] (fp32) = x_dev[M][K] (fp16) . W^T, W the repacked Q6_K matrix.
 * Each weight is unpacked on chip to an fp16 tensor-core operand that is the
 * fp16 rounding of the exact weight d*scale*(q - 32): d*(q - 32) exactly in
 * fp32, times the scale exactly (at most 24 significant bits), then one
 * rounding to fp16 (relative error at most 2^-11; subnormal weights exact);
 * fp32 accumulation in tensor memory.  Same shape, alignment and no-allocation rules as q4k_gemm_f16.
 */
QWP_API int q6k_gemm_f16(const void *w_tiled_dev, const void *x_dev, float *y_dev,
                         int64_t M, int64_t N, int64_t K, void *stream);

/*
 * The same product for bf16 activations, converted to fp16 exactly as q4k_gemm
 * does (pool scratch, or in the GEMM kernel under the same conditions; same
 * rules, same QWP_ERR_RANGE report).
 */
QWP_API int q6k_gemm(const void *w_tiled_dev, const void *x_dev, float *y_dev,
                     int64_t M, int64_t N, int64_t K, void *stream);

/*
 * W4A16 (group-wise int4): wq[N][K/8] int32 words, each holding 8 codes along
 * K with val[2p] at bits 4p..4p+3 and val[2p+1] at bits 16+4p..19+4p;
 * scales[N][K/group] fp16; zeros[N][K/group] uint8 in 0..15 (asymmetric,
 * w = s * (q - zp)), or zeros_dev = NULL for the symmetric form w = s * (q - 8).
 * Source: "[ROCm][Perf] W4A16: packed fp16 prefill dequant", sections "1.
 * Packed fp16 dequant" and "2. dtype-aware gfx1151 tile selection" (a K-block
 * never straddles a group); its results table and "Duplicate-work check" name
 * the symmetric variant and the bf16-activation arm.  Requirements:
 * group % 64 == 0, K % group == 0.
 */

/* Bytes of a repacked W4A16 code matrix: N*K/2. */
QWP_API int w4a16_repacked_bytes(int64_t N, int64_t K, size_t *out_bytes);

/* Load-time repack of wq_dev [N][K/8] words into 128-row tiles of 64-wide K-blocks (same size). */
QWP_API int w4a16_repack(const void *wq_dev, void *wq_tiled_dev, int64_t N, int64_t K, void *stream);

/* Test entry point: exact fp32 s*(q - zp) of the repacked matrix into w_out_dev[N][K] (zeros_dev may be NULL). */
QWP_API int w4a16_dequant(const void *wq_tiled_dev, const void *scales_dev, const uint8_t *zeros_dev,
                  float *w_out_dev, int64_t N, int64_t K, int64_t group, void *stream);

/*
 * y_dev[M][N] (fp32) = x_dev[M][K] (fp16) . W^T.  Each weight is unpacked
 * with the exact 0x6400|n trick, (1024+q) - (1024+zp) exactly, then one fp16
 * multiply by the scale, and fed to the tensor cores (fp16 operands, fp32
 * accumulation).  Same alignment rules as q4k_gemm.
 */
QWP_API int w4a16_gemm(const void *wq_tiled_dev, const void *scales_dev, const uint8_t *zeros_dev,
               const void *x_dev, float *y_dev, int64_t M, int64_t N, int64_t K, int64_t group,
               void *stream);

/*
 * The same product for bf16 activations (the pages' bf16 arm): x is first
 * converted to fp16 into M*K*2 bytes of scratch from the library-owned,
 * stream-ordered pool (exact for |x| in [2^-14, 65504]; an overflow is reported
 * by qwp_device_status as QWP_ERR_RANGE), then w4a16_gemm runs, launched so that
 * its set-up overlaps the conversion; the GEMM kernel converts x itself under
 * the conditions described for q4k_gemm.  Same rules as w4a16_gemm.
 */
QWP_API int w4a16_gemm_bf16(const void *wq_tiled_dev, const void *scales_dev, const uint8_t *zeros_dev,
                    const void *x_dev, float *y_dev, int64_t M, int64_t N, int64_t K, int64_t group,
                    void *stream);

/*
 * Synchronize `stream`, then read and clear the library's device status word
 * on the current device.  Returns QWP_OK; QWP_ERR_TIMEOUT if a kernel's
 * bounded wait on an mbarrier expired (the kernel then released its tensor
 * memory and exited; its output is invalid; while a timeout is recorded, every
 * GEMM launch on that device exits at once without writing y); QWP_ERR_RANGE
 * if an entry point converting bf16 activations to fp16 met one beyond the
 * fp16 range (y then holds inf/nan), or q8_quantize met a non-finite one;
 * or QWP_ERR_CUDA.  Reading the word here clears it.
 */
QWP_API int qwp_device_status(void *stream);

/*
 * Which decode-shaped products (see the top of this file) the GEMM entry points
 * run on the decode kernel, process-wide: QWP_DECODE_AUTO (the default: M <= 2
 * and N >= 24576 for Q4_K, N >= 65536 for Q6_K, N >= 24576 at one token and N >=
 * 65536 at two for W4A16, where it measured faster), QWP_DECODE_NEVER (always the
 * prefill kernel) or QWP_DECODE_ALWAYS (every decode-shaped product).  Results
 * meet the same error bound either way.  Returns the previous policy (>= 0) or
 * QWP_ERR_INVALID_ARG.  Calls already issued keep the kernel they were given;
 * the setting is read at each call, so a graph captured under one policy keeps
 * the kernels it captured.
 */
enum qwp_decode_policy { QWP_DECODE_AUTO = 0, QWP_DECODE_NEVER = 1, QWP_DECODE_ALWAYS = 2 };
QWP_API int qwp_set_decode_policy(int policy);

/* 1 if a GEMM call of this weight format (0 W4A16, 1 Q4_K, 2 Q6_K) and shape
 * would run the decode kernel under the current policy, 0 if the prefill kernel
 * (host-only; no device call); QWP_ERR_INVALID_ARG for an unknown format. */
QWP_API int qwp_decode_selected(int format, int64_t M, int64_t N, int64_t K);

/*
 * The launch a GEMM call of this shape gets on the current device (host only:
 * it reads the device's properties but launches nothing).  `format`: 0 W4A16,
 * 1 Q4_K, 2 Q6_K.  plan_out[6] receives: [0] the kernel (1 the prefill kernel,
 * 2 the decode kernel, which leaves [1..5] at 0, 3 the skinny-N kernel, which
 * reports its split, clusters and token tile (at most 128 tokens) the same
 * way and 1 unit per cluster); [1] the split-K factor S (the
 * cluster size); [2] the clusters launched; [3] the token tile (tokens per
 * unit); [4] the units (128-row tiles x token tiles); [5] the units per cluster
 * at most.  Returns QWP_OK, QWP_ERR_INVALID_ARG (NULL plan_out, a size below 1,
 * an unknown format), QWP_ERR_UNSUPPORTED_SHAPE (K not a multiple of 256 for
 * Q4_K / Q6_K or of 64 for W4A16, a size above 2^30), QWP_ERR_DEVICE or
 * QWP_ERR_CUDA.
 */
QWP_API int qwp_gemm_plan(int format, int64_t M, int64_t N, int64_t K, int32_t *plan_out);

/*
 * The bound on each wait of the prefill kernel's main loop (ns, process-wide,
 * for calls launched afterwards; default 2 s; kept in SM clock cycles at 2.1
 * per ns, so it lasts longer at SM clocks below 2.1 GHz): a wait that runs out
 * records QWP_ERR_TIMEOUT for qwp_device_status, the kernel's CTAs wait (with
 * the default bound) for their own copies and MMAs in flight, meet their
 * cluster peers at a cluster barrier, release their tensor memory and exit;
 * later launches skip their work until the status is read.  A short bound makes
 * that path run on purpose (a test hook).  0 or more than 60 s:
 * QWP_ERR_INVALID_ARG.
 */
QWP_API int qwp_set_wait_timeout_ns(uint64_t ns);

#ifdef __cplusplus
}
#endif

#endif /* QWP_H */
