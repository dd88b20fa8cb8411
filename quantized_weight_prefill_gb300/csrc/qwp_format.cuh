// Tile-major layouts of the repacked weights and the on-chip unpack of one
// 32-bit word of 4-bit codes.  Shared by the repack, dequant and GEMM kernels.
//
// Q4_K, repacked ("tiled") order.  Rows are grouped into tiles of TILE_ROWS
// (128) rows; the last tile holds R = N - 128*t rows.  Tile t starts at byte
// 128*t * (K/256) * 144.  Inside a tile, super-block b (256 weights along K)
// of all R rows is one contiguous group of R*144 bytes at offset b*R*144:
//   header plane   16*R bytes: row i's 16 header bytes (fp16 d, fp16 dmin,
//                  12 packed scale bytes, exactly as in the GGML block) at 16*i;
//   chunk plane c  (c = 0..3, 64 weights each) 32*R bytes at 16*R + 32*R*c,
//                  laid out [h = 0..1][row i][16 bytes]: the 8 words v = 0..7 of
//                  (row i, chunk c) sit at ((v/4)*R + i)*16 + 4*(v%4);
//   word v         elements 64c + 8v + t (t = 0..7) of the super-block in the
//                  interleaved nibble order of the W4A16 format: element t = 2p
//                  in bits 4p..4p+3, element t = 2p+1 in bits 16+4p..19+4p, so
//                  one AND-OR per pair p yields two K-adjacent fp16 lanes.
// The repack is a byte permutation: 144 bytes per 256 weights, as in GGML.  A
// warp of 32 consecutive rows reading one 16-byte quarter of its chunk reads
// 512 contiguous bytes of shared memory (no bank conflicts), and the whole
// group is one contiguous bulk copy.
//
// Q6_K, repacked order.  Same 128-row tiles, but the last tile's R rows are
// padded to Rp = R rounded up to a multiple of 8 (zero bytes), so that every
// group is a multiple of 16 bytes; full tiles have Rp = 128.  Tile t starts at
// byte 128*t * (K/256) * 210.  Inside a tile, super-block b of all Rp rows is
// one group of Rp*210 bytes at offset b*Rp*210:
//   d plane        2*Rp bytes: row i's fp16 d at 2*i;
//   scale plane    16*Rp bytes at 2*Rp: row i's 16 int8 scales at 16*i;
//   low plane c    (c = 0..3) 32*Rp bytes at 18*Rp + 32*Rp*c, [h][row i][16 B]
//                  like the Q4_K chunk planes: word v holds the low four bits of
//                  elements 64c + 8v + t in the interleaved nibble order;
//   high plane c   16*Rp bytes at 146*Rp + 16*Rp*c, [row i][16 B]: word u (0..3)
//                  holds the high two bits of elements 64c + 16u + t, t = 0..15:
//                  t = 2p + o (p = 0..3, o = 0..1) at bits 4+2p+16o, and
//                  t = 8 + 2p + o at bits (12+2p+16o) mod 32.  Rotating word u
//                  right by 2p (elements of low word 2u) or 8+2p (low word 2u+1)
//                  puts pair p's two fields at bits 4-5 and 20-21, just above the
//                  pair's low nibbles once the low word is shifted right by 4p.
// 210 bytes per 256 weights as in GGML (plus the row padding of the last tile).
//
// Quantized activations (the 8-bit codes of the DP4a-style product), record
// order.  Tokens are taken in groups of 8 (the last group padded with zero
// tokens); token group g and super-block b (256 values along K) form one record
// of 8 * Q8_TOKEN_BYTES bytes at (g * K/256 + b) * Q8_RECORD_BYTES, token t of
// the group at t * Q8_TOKEN_BYTES inside it:
//   bytes 0..255   the 256 int8 codes; each run of 8 elements e0..e7 is stored
//                  as e0 e4 e1 e5 e2 e6 e3 e7, so that its two 32-bit words line
//                  up byte for byte with the low and the high nibbles of the
//                  repacked Q4_K word of the same 8 elements;
//   bytes 256..287 the 8 fp32 scales d of the record's 32-value blocks;
//   bytes 288..319 the 8 code sums of those blocks, as fp32 (exact: |s| <= 4064).
// A record is one contiguous bulk copy.
//
// W4A16, repacked order.  Same 128-row tiles; tile t starts at 128*t * K/2.
// Inside, K-block j (64 weights along K) of all R rows is a plane of 32*R bytes
// at j*32*R, laid out [h][row i][16 bytes] as above, word v being the original
// interleaved word 8*j + v of row i, bits unchanged.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace qwp {

constexpr int TILE_ROWS = 128;
constexpr int Q4K_BLOCK = 256;
constexpr int Q4K_BLOCK_BYTES = 144;
constexpr int Q4K_HEADER_BYTES = 16;
constexpr int CHUNK_K = 64;          // weights per chunk (one 128-byte row of bf16 / fp16)
constexpr int CHUNK_ROW_BYTES = 32;  // packed bytes of one row's chunk
constexpr int Q6K_BLOCK_BYTES = 210;
constexpr int Q6K_SCALE_PLANE = 2;   // x Rp: byte offset of the scale plane
constexpr int Q6K_LOW_PLANE = 18;    // x Rp: first low plane
constexpr int Q6K_HIGH_PLANE = 146;  // x Rp: first high plane
constexpr int Q8_GROUP_TOKENS = 8;   // tokens per quantized-activation record
constexpr int Q8_TOKEN_BYTES = 320;  // one token's 256 codes, 8 scales, 8 sums
constexpr int Q8_RECORD_BYTES = Q8_GROUP_TOKENS * Q8_TOKEN_BYTES;

__host__ __device__ __forceinline__ int tile_rows(int64_t N, int64_t tile) {
    int64_t r = N - tile * TILE_ROWS;
    return static_cast<int>(r < TILE_ROWS ? r : TILE_ROWS);
}

// Byte offset of super-block b's group inside the tiled Q4_K matrix.
__host__ __device__ __forceinline__ int64_t q4k_group_offset(int64_t K, int64_t tile, int R,
                                                             int64_t b) {
    return tile * TILE_ROWS * (K / Q4K_BLOCK) * Q4K_BLOCK_BYTES + b * R * Q4K_BLOCK_BYTES;
}

// Rows of tile `tile` as stored in the Q6_K layout (a multiple of 8).
__host__ __device__ __forceinline__ int q6k_padded_rows(int R) { return (R + 7) & ~7; }

// Byte offset of super-block b's group inside the tiled Q6_K matrix (Rp padded rows).
__host__ __device__ __forceinline__ int64_t q6k_group_offset(int64_t K, int64_t tile, int Rp,
                                                             int64_t b) {
    return tile * TILE_ROWS * (K / Q4K_BLOCK) * Q6K_BLOCK_BYTES + b * Rp * Q6K_BLOCK_BYTES;
}

// Offsets inside a Q6_K group: low word v and high word u of (row i, chunk c).
__host__ __device__ __forceinline__ int q6k_low_word_offset(int Rp, int i, int c, int v) {
    return Q6K_LOW_PLANE * Rp + CHUNK_ROW_BYTES * Rp * c + ((v >> 2) * Rp + i) * 16 + 4 * (v & 3);
}
__host__ __device__ __forceinline__ int q6k_high_word_offset(int Rp, int i, int c, int u) {
    return Q6K_HIGH_PLANE * Rp + 16 * Rp * c + i * 16 + 4 * u;
}
// Bit position of the high two bits of element t (0..15) inside its high word.
__host__ __device__ __forceinline__ int q6k_high_bit(int t) {
    const int p = (t & 7) >> 1, o = t & 1;
    return (t < 8) ? 4 + 2 * p + 16 * o : (12 + 2 * p + 16 * o) & 31;
}

// Offset of word v of (row i, chunk c) inside a Q4_K super-block group.
__host__ __device__ __forceinline__ int q4k_word_offset(int R, int i, int c, int v) {
    return Q4K_HEADER_BYTES * R + CHUNK_ROW_BYTES * R * c + ((v >> 2) * R + i) * 16 + 4 * (v & 3);
}

// Byte offset of K-block j's plane inside the tiled W4A16 matrix.
__host__ __device__ __forceinline__ int64_t w4_plane_offset(int64_t K, int64_t tile, int R,
                                                            int64_t j) {
    return tile * TILE_ROWS * (K / 2) + j * R * CHUNK_ROW_BYTES;
}

__host__ __device__ __forceinline__ int w4_word_offset(int R, int i, int v) {
    return ((v >> 2) * R + i) * 16 + 4 * (v & 3);
}

// ---------------------------------------------------------------- nibble pairs

// Pair p (p = 0..3) of an interleaved word as raw fp16x2 bits (1024+q_{2p},
// 1024+q_{2p+1}): fp16 0x6400|n is exactly 1024 + n.
__device__ __forceinline__ uint32_t nib_pair_magic(uint32_t word, int p) {
    return ((word >> (4 * p)) & 0x000F000Fu) | 0x64006400u;
}

__device__ __forceinline__ __half2 as_half2(uint32_t bits) {
    return *reinterpret_cast<const __half2 *>(&bits);
}

__device__ __forceinline__ uint32_t as_u32(__half2 h) {
    return *reinterpret_cast<const uint32_t *>(&h);
}

// ---------------------------------------------------------------- Q4_K scales

// (1024 + sc_j, 1024 + m_j) of sub-block j (0..7) as raw fp16x2 bits, from the
// GGML packing: values 0..3 are the low 6 bits of packed bytes 0..3 (scales) and
// 4..7 (mins); values 4..7 take the low (scale) / high (min) nibble of bytes
// 8..11 and, as bits 4-5, the top two bits of bytes 0..3 (scale) / 4..7 (min).
__device__ __forceinline__ uint32_t q4k_scmin_magic(uint4 h, int j) {
    const int sh = 8 * (j & 3);
    const uint32_t b_lo = h.y >> sh;   // packed byte j%4 in bits 0-7
    const uint32_t b_mid = h.z >> sh;  // packed byte 4 + j%4
    uint32_t sc, m;
    if (j < 4) {
        sc = b_lo & 63u;
        m = b_mid & 63u;
    } else {
        const uint32_t b_hi = h.w >> sh;  // packed byte 8 + j%4
        sc = (b_hi & 15u) | ((b_lo >> 2) & 0x30u);
        m = ((b_hi >> 4) & 15u) | ((b_mid >> 2) & 0x30u);
    }
    return 0x64006400u | sc | (m << 16);
}

// Exact (sc_j, m_j) as fp16x2.
__device__ __forceinline__ __half2 q4k_scmin(uint4 h, int j) {
    return __hsub2(as_half2(q4k_scmin_magic(h, j)), as_half2(0x64006400u));
}

// dl = d*sc_j and ml = dmin*m_j of one sub-block, both exact in fp32.
__device__ __forceinline__ void q4k_subblock_scale(uint4 h, int j, float &dl, float &ml) {
    const float2 scm = __half22float2(q4k_scmin(h, j));
    dl = __half2float(__ushort_as_half(static_cast<unsigned short>(h.x & 0xFFFFu))) * scm.x;
    ml = __half2float(__ushort_as_half(static_cast<unsigned short>(h.x >> 16))) * scm.y;
}

// ---------------------------------------------------------------- Q4_K unpack

// The 8 weights of one interleaved word as exact fp32 (the dequant entry point):
// q exactly from the magic pair, then fmaf(dl, q, -ml) rounds the exact
// d*sc*q - dmin*m once.  w[i] holds the K-adjacent elements 2i, 2i+1.
__device__ __forceinline__ void q4k_word_f32(uint32_t word, float dl, float ml, float2 (&w)[4]) {
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const float2 q = __half22float2(__hsub2(as_half2(nib_pair_magic(word, p)), as_half2(0x64006400u)));
        w[p] = make_float2(fmaf(dl, q.x, -ml), fmaf(dl, q.y, -ml));
    }
}

// Per-sub-block constants of the GEMM's unpack.
struct Q4kSubH {
    __half2 sc2;      // (sc, sc)
    __half2 csc2;     // (-1024*sc, -1024*sc), exact
    __half2 sc16_2;   // (sc/16, sc/16), exact
    __half2 csc16_2;  // (-64*sc, -64*sc), exact
    unsigned short d; // fp16 bits of d
    float nml;        // -(dmin*m), exact in fp32 (at most 17 significant bits)
};

// The constants of one sub-block from the block's first header word (fp16 d in
// bits 0-15, fp16 dmin in bits 16-31) and its exact (sc, m) pair.
__device__ __forceinline__ Q4kSubH q4k_sub_consts(uint32_t hx, __half2 scm) {
    Q4kSubH k;
    k.sc2 = __low2half2(scm);
    k.csc2 = __hmul2(k.sc2, as_half2(0xE400E400u));     // x (-1024)
    k.sc16_2 = __hmul2(k.sc2, as_half2(0x2C002C00u));   // x (1/16)
    k.csc16_2 = __hmul2(k.sc2, as_half2(0xD400D400u));  // x (-64)
    k.d = static_cast<unsigned short>(hx & 0xFFFFu);
    k.nml = -(__half2float(__ushort_as_half(static_cast<unsigned short>(hx >> 16))) * __high2float(scm));
    return k;
}

__device__ __forceinline__ Q4kSubH q4k_sub_f16(uint4 h, int j) { return q4k_sub_consts(h.x, q4k_scmin(h, j)); }

// Both halves of an exact fp16 pair (a0, a1) through a*b + c, each with the
// product formed exactly and the sum rounded once to fp32 (the mixed-precision
// fma of sm_100 and later), then packed into fp16x2 with one more rounding.
__device__ __forceinline__ uint32_t fma_pair_f16_f32_f16(uint32_t a, unsigned short b, float c) {
    uint32_t r;
    asm("{\n\t.reg .b16 a0, a1;\n\t.reg .f32 lo, hi;\n\t"
        "mov.b32 {a0, a1}, %1;\n\t"
        "fma.rn.f32.f16 lo, a0, %2, %3;\n\t"
        "fma.rn.f32.f16 hi, a1, %2, %3;\n\t"
        "cvt.rn.f16x2.f32 %0, hi, lo;\n\t}"
        : "=r"(r)
        : "r"(a), "h"(b), "f"(c));
    return r;
}

// The 8 weights of one word as fp16x2 MMA operands, each the fp16 rounding of the
// exact d*sc*q - dmin*m.  (1024+q)*sc - 1024*sc is q*sc exactly (at most 945,
// inside fp16's 11-bit integer range; the fp16 fma does not round its product).
// Then d*(q*sc) - dmin*m is formed in fp32: the product (at most 21 significant
// bits) is exact inside the fma and dmin*m is exact, so one fp32 rounding at most
// (none unless the two terms are more than 24 bits apart), then one rounding to
// fp16: the operand's relative error is at most 2^-11 * (1 + 2^-13), and since the
// exact weight is a multiple of 2^-24, weights in fp16's subnormal range are exact.
// Pairs 1 and 3 are read in place from bits 4..7 of each half, as 1024 + 16q,
// which saves their shifts: (1024+16q)*(sc/16) - 64*sc is the same exact q*sc.
// The exact q*sc of the 8 weights of one word as 4 fp16 pairs (K order).
__device__ __forceinline__ void q4k_word_qsc(uint32_t word, const Q4kSubH &k, uint32_t (&q)[4]) {
    const uint32_t w8 = word >> 8;
    q[0] = as_u32(__hfma2(as_half2((word & 0x000F000Fu) | 0x64006400u), k.sc2, k.csc2));
    q[1] = as_u32(__hfma2(as_half2((word & 0x00F000F0u) | 0x64006400u), k.sc16_2, k.csc16_2));
    q[2] = as_u32(__hfma2(as_half2((w8 & 0x000F000Fu) | 0x64006400u), k.sc2, k.csc2));
    q[3] = as_u32(__hfma2(as_half2((w8 & 0x00F000F0u) | 0x64006400u), k.sc16_2, k.csc16_2));
}

__device__ __forceinline__ void q4k_word_f16x2(uint32_t word, const Q4kSubH &k, uint32_t (&p)[4]) {
    uint32_t q[4];
    q4k_word_qsc(word, k, q);
#pragma unroll
    for (int i = 0; i < 4; ++i) p[i] = fma_pair_f16_f32_f16(q[i], k.d, k.nml);
}

// The 8 weights of one word as pairs of bf16 operands whose sum carries about 16
// significant bits: w32 = RN32(d*(q*sc) - dmin*m) as above (no rounding to
// fp16), hi = RN_bf16(w32), lo = RN_bf16(w32 - hi) (the difference is exact in
// fp32); |w - (hi + lo)| <= (2^-18 + 2^-24)|w|.  For a bf16 x tile, whose
// values the tensor core then multiplies exactly.
__device__ __forceinline__ void q4k_word_bf16_hilo(uint32_t word, const Q4kSubH &k, uint32_t (&hi)[4],
                                                   uint32_t (&lo)[4]) {
    uint32_t q[4];
    q4k_word_qsc(word, k, q);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t h, l;
        asm("{\n\t.reg .b16 a0, a1;\n\t.reg .f32 w0, w1, h0, h1;\n\t.reg .b32 hb;\n\t"
            "mov.b32 {a0, a1}, %2;\n\t"
            "fma.rn.f32.f16 w0, a0, %3, %4;\n\t"
            "fma.rn.f32.f16 w1, a1, %3, %4;\n\t"
            "cvt.rn.bf16x2.f32 hb, w1, w0;\n\t"
            "shl.b32 %0, hb, 16;\n\t"
            "mov.b32 h0, %0;\n\t"
            "and.b32 %0, hb, 0xFFFF0000;\n\t"
            "mov.b32 h1, %0;\n\t"
            "sub.rn.f32 w0, w0, h0;\n\t"
            "sub.rn.f32 w1, w1, h1;\n\t"
            "cvt.rn.bf16x2.f32 %1, w1, w0;\n\t"
            "mov.b32 %0, hb;\n\t}"
            : "=&r"(h), "=r"(l)
            : "r"(q[i]), "h"(k.d), "f"(k.nml));
        hi[i] = h;
        lo[i] = l;
    }
}

// ---------------------------------------------------------------- Q6_K unpack

// Pair p of low word `lo` with its high bits from high word `hi` (set 0: the word's
// first 8 elements, set 1: the second 8) as raw fp16x2 bits (1024+q, 1024+q').
template <int kSet>
__device__ __forceinline__ uint32_t q6k_pair_magic(uint32_t lo, uint32_t hi, int p) {
    const uint32_t a = lo >> (4 * p);
    const uint32_t b = __funnelshift_r(hi, hi, (kSet ? 8 : 0) + 2 * p);
    return (a & 0x000F000Fu) | (b & 0x00300030u) | 0x64006400u;
}

// (q - 32) of a magic pair, exact: (1024 + q) - 1056.
__device__ __forceinline__ __half2 q6k_centered(uint32_t magic) {
    return __hsub2(as_half2(magic), as_half2(0x64206420u));
}

// Per-16-weight constants of the Q6_K unpack: fp16 d, -1056*d (exact in fp32) and
// the int8 scale as fp32.
struct Q6kSub {
    unsigned short d;
    float nd1056;
    float sc;
};

__device__ __forceinline__ Q6kSub q6k_sub(uint32_t dbits, int sc) {
    Q6kSub k;
    k.d = static_cast<unsigned short>(dbits & 0xFFFFu);
    k.nd1056 = -1056.f * __half2float(__ushort_as_half(k.d));
    k.sc = static_cast<float>(sc);
    return k;
}

// The 8 weights of low word `lo` as fp16x2 MMA operands, each the fp16 rounding of
// the exact d*sc*(q - 32): (1024+q)*d - 1056*d is d*(q - 32) exactly in fp32 (the
// mixed-precision fma forms the product exactly; the result has at most 17
// significant bits), times sc exactly (at most 24 bits), then one rounding to fp16.
template <int kSet>
__device__ __forceinline__ void q6k_word_f16x2(uint32_t lo, uint32_t hi, const Q6kSub &k, uint32_t (&p)[4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t m = q6k_pair_magic<kSet>(lo, hi, i);
        uint32_t r;
        asm("{\n\t.reg .b16 a0, a1;\n\t.reg .f32 lo, hi;\n\t"
            "mov.b32 {a0, a1}, %1;\n\t"
            "fma.rn.f32.f16 lo, a0, %2, %3;\n\t"
            "fma.rn.f32.f16 hi, a1, %2, %3;\n\t"
            "mul.rn.f32 lo, lo, %4;\n\t"
            "mul.rn.f32 hi, hi, %4;\n\t"
            "cvt.rn.f16x2.f32 %0, hi, lo;\n\t}"
            : "=r"(r)
            : "r"(m), "h"(k.d), "f"(k.nd1056), "f"(k.sc));
        p[i] = r;
    }
}

// The constants of the four 16-weight scale groups u of one 64-wide chunk (d is the
// block's fp16 bits, sc4 its four int8 scales).
__device__ __forceinline__ void q6k_chunk_scales(uint32_t dbits, uint32_t sc4, Q6kSub (&ks)[4]) {
#pragma unroll
    for (int u = 0; u < 4; ++u) ks[u] = q6k_sub(dbits, static_cast<int8_t>(static_cast<uint8_t>(sc4 >> (8 * u))));
}

// ---------------------------------------------------------------- W4A16 unpack

// Pair p (p = 0..3) of an interleaved word as fp16x2 (q_{2p} - zp, q_{2p+1} - zp),
// exact: (1024 + n) - (1024 + zp) has no rounding.
__device__ __forceinline__ __half2 w4_pair_minus_zero(uint32_t word, int p, __half2 magic_zp) {
    return __hsub2(as_half2(nib_pair_magic(word, p)), magic_zp);
}

// 1024 + zp in both halves.
__device__ __forceinline__ __half2 w4_magic_zero(uint32_t zp) {
    const uint32_t h = 0x6400u | (zp & 15u);
    const uint32_t bits = h | (h << 16);
    return *reinterpret_cast<const __half2 *>(&bits);
}

// The 8 weights of one word as fp16x2 pairs: one fp16 multiply by the scale.
__device__ __forceinline__ void w4_word_f16x2(uint32_t word, __half2 magic_zp, __half2 s2,
                                              uint32_t (&p)[4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __half2 v = __hmul2(w4_pair_minus_zero(word, i, magic_zp), s2);
        p[i] = *reinterpret_cast<uint32_t *>(&v);
    }
}

}  // namespace qwp
