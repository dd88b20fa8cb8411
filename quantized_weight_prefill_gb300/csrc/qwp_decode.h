// Host entry of the decode-shaped (M <= 8 tokens) product kernel.
#pragma once

#include "qwp_internal.h"

namespace qwp {

// Weight formats of launch_decode (same numbering as the prefill kernel's), and
// DFMT_Q4K_Q8: Q4_K weights with 8-bit quantized activations (record order of
// qwp_format.cuh), multiplied with integer dot products.
enum : int { DFMT_W4A16 = 0, DFMT_Q4K = 1, DFMT_Q6K = 2, DFMT_Q4K_Q8 = 3 };

// The largest token count the decode kernel takes (one MMA's N).
constexpr int64_t DECODE_MAX_TOKENS = 8;

// The decode kernel is used for matrices of at least this many (128-row tile,
// 256-wide super-block) items; below it (under ~20M weights) the fixed start-up
// and hand-off costs of the decode kernel exceed what it saves over the prefill
// kernel (measured on GB300 at 1 to 8 tokens).
constexpr int64_t DECODE_MIN_ITEMS = 600;

// Whether an M x N x K product takes the decode kernel: 1 <= M <= 8, K % 256 == 0,
// at least DECODE_MIN_ITEMS items and few enough for its 32-bit work split.
inline bool decode_fits(int64_t M, int64_t N, int64_t K) {
    if (M < 1 || M > DECODE_MAX_TOKENS || K % 256 != 0) return false;
    const int64_t items = (N + 127) / 128 * (K / 256);
    return items >= DECODE_MIN_ITEMS && items <= (int64_t(1) << 22);
}

// Which products of decode shape the GEMM entry points give the decode kernel
// (qwp_set_decode_policy): AUTO follows decode_auto, NEVER keeps every product on
// the prefill kernel, ALWAYS takes every product that decode_fits.
enum : int { DECODE_POLICY_AUTO = 0, DECODE_POLICY_NEVER = 1, DECODE_POLICY_ALWAYS = 2 };

// The automatic choice, from both kernels timed on GB300 (Q4_K, Q6_K and W4A16,
// N from 2048 to 152064, K from 4096 to 12288, 1 to 8 tokens; last with the
// decode kernel at two CTAs per SM): the decode kernel is faster at one and two
// tokens from N = 24576 for Q4_K (M1 N24576 32.8 against 34.1 us, M2 33.2
// against 35.3, M1 N65536 65.7 against 71.9) and for W4A16 at one token (31.6
// against 33.4), at two tokens for W4A16 from N = 65536 (65.6 against 71.0), and
// for Q6_K from N = 65536 (a tie at 24576); the prefill kernel wins for narrower
// or K-heavy matrices (N <= 12288, or K = 12288 at N = 4096) and from three
// tokens on (M3 N152064 a tie, M4 +2.5%).
inline int64_t decode_auto_min_rows(int fmt, int64_t M) {
    if (fmt == DFMT_Q6K) return 65536;
    if (fmt == DFMT_W4A16 && M > 1) return 65536;
    return 24576;
}
constexpr int64_t DECODE_AUTO_MAX_TOKENS = 2;
inline bool decode_auto(int fmt, int64_t M, int64_t N, int64_t K) {
    return decode_fits(M, N, K) && M <= DECODE_AUTO_MAX_TOKENS && N >= decode_auto_min_rows(fmt, M);
}

// The current policy, and the choice it makes for an M x N x K product of
// weight format fmt (DFMT_*).
int decode_policy();
bool decode_selected(int fmt, int64_t M, int64_t N, int64_t K);

// Device scratch launch_decode needs for an N x K matrix of format `fmt` on the
// current device (partial sums of tiles shared by two or more CTAs, and one
// counter per 128-row tile); 0 if the device could not be queried.
size_t decode_scratch_bytes(int fmt, int64_t N, int64_t K);

// y[M][N] = x[M][K] . W^T for 1 <= M <= 8 and K % 256 == 0, W repacked in format
// `fmt`; x fp16, or bf16 when x_bf16 (converted in shared memory; an fp16
// overflow sets the range bit of the status word); for DFMT_Q4K_Q8, x is the
// quantized-activation records of the first token group (x_bf16 ignored).  `scratch` (16-byte aligned,
// at least decode_scratch_bytes) is used in stream order; its counters are
// cleared on `stream` before the kernel.  Allocates nothing.
int launch_decode(int fmt, const void *w, const void *scales, const uint8_t *zeros, const void *x, bool x_bf16,
                  float *y, int64_t M, int64_t N, int64_t K, int64_t group, void *scratch, size_t scratch_bytes,
                  cudaStream_t stream);

}  // namespace qwp
