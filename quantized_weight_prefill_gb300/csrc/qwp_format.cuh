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
//   word v         element 64c + 8v + u of the super-block (u = 0..7) in bits
//                  4u..4u+3.
// The repack is a byte permutation: 144 bytes per 256 weights, as in GGML.  A
// warp of 32 consecutive rows reading one 16-byte quarter of its chunk reads
// 512 contiguous bytes of shared memory (no bank conflicts), and the whole
// group is one contiguous bulk copy.
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

__host__ __device__ __forceinline__ int tile_rows(int64_t N, int64_t tile) {
    int64_t r = N - tile * TILE_ROWS;
    return static_cast<int>(r < TILE_ROWS ? r : TILE_ROWS);
}

// Byte offset of super-block b's group inside the tiled Q4_K matrix.
__host__ __device__ __forceinline__ int64_t q4k_group_offset(int64_t K, int64_t tile, int R,
                                                             int64_t b) {
    return tile * TILE_ROWS * (K / Q4K_BLOCK) * Q4K_BLOCK_BYTES + b * R * Q4K_BLOCK_BYTES;
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

// ---------------------------------------------------------------- Q4_K unpack

// The 6-bit scales and mins of the 8 sub-blocks from the 12 packed bytes
// (GGML packing: values 0..3 are the low 6 bits of bytes 0..3 / 4..7; values
// 4..7 take the low (scale) or high (min) nibble of bytes 8..11 and, as bits
// 4-5, the top two bits of bytes 0..3 (scale) / 4..7 (min)).
struct Q4kScales {
    float dl[8];  // d * sc_j, exact in fp32 (11 x 6 significant bits)
    float ml[8];  // dmin * m_j, exact in fp32
};

__device__ __forceinline__ void q4k_decode_header(uint4 h, Q4kScales &s) {
    const float d = __half2float(__ushort_as_half(static_cast<unsigned short>(h.x & 0xFFFFu)));
    const float dmin = __half2float(__ushort_as_half(static_cast<unsigned short>(h.x >> 16)));
    const uint32_t s03 = h.y;  // packed bytes 0..3
    const uint32_t s47 = h.z;  // packed bytes 4..7
    const uint32_t s8b = h.w;  // packed bytes 8..11
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t b_lo = (s03 >> (8 * j)) & 0xFFu;
        const uint32_t b_mid = (s47 >> (8 * j)) & 0xFFu;
        const uint32_t b_hi = (s8b >> (8 * j)) & 0xFFu;
        const uint32_t sc_lo = b_lo & 63u, m_lo = b_mid & 63u;
        const uint32_t sc_hi = (b_hi & 15u) | ((b_lo >> 6) << 4);
        const uint32_t m_hi = (b_hi >> 4) | ((b_mid >> 6) << 4);
        s.dl[j] = d * static_cast<float>(sc_lo);
        s.ml[j] = dmin * static_cast<float>(m_lo);
        s.dl[j + 4] = d * static_cast<float>(sc_hi);
        s.ml[j + 4] = dmin * static_cast<float>(m_hi);
    }
}

// dl = d*sc_j and ml = dmin*m_j of one sub-block j (0..7), both exact in fp32.
__device__ __forceinline__ void q4k_subblock_scale(uint4 h, int j, float &dl, float &ml) {
    const float d = __half2float(__ushort_as_half(static_cast<unsigned short>(h.x & 0xFFFFu)));
    const float dmin = __half2float(__ushort_as_half(static_cast<unsigned short>(h.x >> 16)));
    const int sh = 8 * (j & 3);
    const uint32_t b_lo = (h.y >> sh) & 0xFFu;   // packed byte j%4
    const uint32_t b_mid = (h.z >> sh) & 0xFFu;  // packed byte 4 + j%4
    uint32_t sc, m;
    if (j < 4) {
        sc = b_lo & 63u;
        m = b_mid & 63u;
    } else {
        const uint32_t b_hi = (h.w >> sh) & 0xFFu;  // packed byte 8 + j%4
        sc = (b_hi & 15u) | ((b_lo >> 6) << 4);
        m = (b_hi >> 4) | ((b_mid >> 6) << 4);
    }
    dl = d * static_cast<float>(sc);
    ml = dmin * static_cast<float>(m);
}

// Exact integer value of nibble u of `word` as fp32: 0x4B000000 | q is 2^23 + q.
__device__ __forceinline__ float nibble_f32(uint32_t word, int u) {
    return __uint_as_float(0x4B000000u | ((word >> (4 * u)) & 15u)) - 8388608.0f;
}

// The 8 weights of one word: fmaf(dl, q, -ml) rounds the exact d*sc*q - dmin*m once.
__device__ __forceinline__ void q4k_word_f32(uint32_t word, float dl, float ml, float (&w)[8]) {
#pragma unroll
    for (int u = 0; u < 8; ++u) w[u] = fmaf(dl, nibble_f32(word, u), -ml);
}

// The same 8 weights rounded once more to bf16, packed K-adjacent in pairs
// (lower K in the low half).
__device__ __forceinline__ void q4k_word_bf16x2(uint32_t word, float dl, float ml, uint32_t (&p)[4]) {
    float w[8];
    q4k_word_f32(word, dl, ml, w);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 v = __floats2bfloat162_rn(w[2 * i], w[2 * i + 1]);
        p[i] = *reinterpret_cast<uint32_t *>(&v);
    }
}

// ---------------------------------------------------------------- W4A16 unpack

// Pair p (p = 0..3) of an interleaved word as fp16x2 (q_{2p} - zp, q_{2p+1} - zp),
// exact: 0x6400|n is 1024 + n, and (1024 + n) - (1024 + zp) has no rounding.
__device__ __forceinline__ __half2 w4_pair_minus_zero(uint32_t word, int p, __half2 magic_zp) {
    const uint32_t bits = ((word >> (4 * p)) & 0x000F000Fu) | 0x64006400u;
    return __hsub2(*reinterpret_cast<const __half2 *>(&bits), magic_zp);
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
