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

// Packed fp32x2 arithmetic (two independent lanes per instruction, sm_100+).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// Per-sub-block constants of the word unpack below.  A nibble q at bits
// 4u..4u+3 of a word, OR-ed into the fp32 pattern 0x4B000000, reads as
// v = 2^23 + q*16^u exactly.  With s = dl*16^-u (exact: a power-of-two scale)
// fma(v, s, -2^23*s) = q*dl exactly (q*dl has at most 21 significant bits),
// and adding -ml rounds once: the result is the correctly rounded fp32 of
// d*sc*q - dmin*m.
struct Q4kSub {
    float2 s01, s23;  // multipliers of nibbles (0,1) and (2,3) of a half-word
    float2 c01, c23;  // -2^23 * s
    float2 nml;       // (-ml, -ml)
};

__device__ __forceinline__ Q4kSub q4k_sub_consts(float dl, float ml) {
    Q4kSub k;
    k.s01 = make_float2(dl, dl * 0.0625f);
    k.s23 = make_float2(dl * 0.00390625f, dl * 0.000244140625f);
    k.c01 = make_float2(-8388608.0f * k.s01.x, -8388608.0f * k.s01.y);
    k.c23 = make_float2(-8388608.0f * k.s23.x, -8388608.0f * k.s23.y);
    k.nml = make_float2(-ml, -ml);
    return k;
}

// The 8 weights of one word (element u in bits 4u..4u+3) as fp32, each the
// correctly rounded d*sc*q - dmin*m; returned as K-adjacent pairs.
__device__ __forceinline__ void q4k_word_f32(uint32_t word, const Q4kSub &k, float2 (&w)[4]) {
    const uint32_t hi = word >> 16;
    const float2 v01 = make_float2(__uint_as_float((word & 0x000Fu) | 0x4B000000u),
                                   __uint_as_float((word & 0x00F0u) | 0x4B000000u));
    const float2 v23 = make_float2(__uint_as_float((word & 0x0F00u) | 0x4B000000u),
                                   __uint_as_float((word & 0xF000u) | 0x4B000000u));
    const float2 v45 = make_float2(__uint_as_float((hi & 0x000Fu) | 0x4B000000u),
                                   __uint_as_float((hi & 0x00F0u) | 0x4B000000u));
    const float2 v67 = make_float2(__uint_as_float((hi & 0x0F00u) | 0x4B000000u),
                                   __uint_as_float((hi & 0xF000u) | 0x4B000000u));
    w[0] = fadd2(ffma2(v01, k.s01, k.c01), k.nml);
    w[1] = fadd2(ffma2(v23, k.s23, k.c23), k.nml);
    w[2] = fadd2(ffma2(v45, k.s01, k.c01), k.nml);
    w[3] = fadd2(ffma2(v67, k.s23, k.c23), k.nml);
}

// The same 8 weights rounded once more to bf16, packed K-adjacent in pairs
// (lower K in the low half).
__device__ __forceinline__ void q4k_word_bf16x2(uint32_t word, const Q4kSub &k, uint32_t (&p)[4]) {
    float2 w[4];
    q4k_word_f32(word, k, w);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 v = __floats2bfloat162_rn(w[i].x, w[i].y);
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
