// Load-time repack kernels, the dequant test entry points, the device status
// word and the device check.
#include <algorithm>
#include <atomic>

#include "qwp_format.cuh"
#include "qwp_internal.h"
#include "qwp_ptx.cuh"

namespace qwp {

// Status word written by kernels whose bounded waits expire (0 = no error).
__device__ uint32_t g_qwp_status;

int check_device() {
    static std::atomic<int> cache[64];  // 0 unknown, 1 sm_103, 2 other
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return QWP_ERR_CUDA;
    if (dev >= 0 && dev < 64) {
        const int c = cache[dev].load(std::memory_order_relaxed);
        if (c) return c == 1 ? QWP_OK : QWP_ERR_DEVICE;
    }
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return QWP_ERR_CUDA;
    const bool ok = (major == 10 && minor == 3);
    if (dev >= 0 && dev < 64) cache[dev].store(ok ? 1 : 2, std::memory_order_relaxed);
    return ok ? QWP_OK : QWP_ERR_DEVICE;
}

uint32_t *status_word() {
    static std::atomic<uint32_t *> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    if (dev >= 0 && dev < 64) {
        uint32_t *p = cache[dev].load(std::memory_order_acquire);
        if (p) return p;
    }
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_qwp_status) != cudaSuccess) return nullptr;
    if (dev >= 0 && dev < 64) cache[dev].store(static_cast<uint32_t *>(p), std::memory_order_release);
    return static_cast<uint32_t *>(p);
}

// ---------------------------------------------------------------- Q4_K repack

// One warp per (row n, super-block b): lanes 0..3 copy the 16 header bytes,
// lane l builds word v = l%8 of chunk c = l/8 from the GGML nibble bytes
// (element e < 32 of chunk c is the low nibble of byte 32c+e, element e >= 32
// the high nibble of byte 32c+e-32) in the interleaved order: element 8v+2p at
// bits 4p..4p+3, element 8v+2p+1 at bits 16+4p..19+4p.
__global__ void q4k_repack_kernel(const uint8_t *__restrict__ src, uint8_t *__restrict__ dst,
                                  int64_t N, int64_t K) {
    const int64_t nb = K / Q4K_BLOCK;
    const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (gw >= N * nb) return;
    const int lane = threadIdx.x & 31;
    const int64_t n = gw / nb, b = gw % nb;
    const int64_t tile = n / TILE_ROWS;
    const int i = static_cast<int>(n % TILE_ROWS);
    const int R = tile_rows(N, tile);
    const uint8_t *blk = src + (n * nb + b) * Q4K_BLOCK_BYTES;
    uint8_t *grp = dst + q4k_group_offset(K, tile, R, b);
    if (lane < 4)
        *reinterpret_cast<uint32_t *>(grp + Q4K_HEADER_BYTES * i + 4 * lane) =
            *reinterpret_cast<const uint32_t *>(blk + 4 * lane);
    const int c = lane >> 3, v = lane & 7;
    const uint8_t *qs = blk + Q4K_HEADER_BYTES + 32 * c;
    uint32_t word = 0;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const int e = 8 * v + u;
        const uint32_t byte = qs[e & 31];
        const uint32_t nib = (e < 32) ? (byte & 15u) : (byte >> 4);
        word |= nib << ((u & 1) ? 16 + 4 * (u >> 1) : 4 * (u >> 1));
    }
    *reinterpret_cast<uint32_t *>(grp + q4k_word_offset(R, i, c, v)) = word;
}

// One warp per (row, super-block); lane l dequantizes elements 8l..8l+7 and
// writes them with two 16-byte stores, so a warp writes 1 KiB contiguously.
__global__ void q4k_dequant_kernel(const uint8_t *__restrict__ w, float *__restrict__ out,
                                   int64_t N, int64_t K) {
    const int64_t nb = K / Q4K_BLOCK;
    const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (gw >= N * nb) return;
    const int lane = threadIdx.x & 31;
    const int64_t n = gw / nb, b = gw % nb;
    const int64_t tile = n / TILE_ROWS;
    const int i = static_cast<int>(n % TILE_ROWS);
    const int R = tile_rows(N, tile);
    const uint8_t *grp = w + q4k_group_offset(K, tile, R, b);
    const uint4 hdr = *reinterpret_cast<const uint4 *>(grp + Q4K_HEADER_BYTES * i);
    const int c = lane >> 3, v = lane & 7;
    float dl, ml;
    q4k_subblock_scale(hdr, 2 * c + (v >> 2), dl, ml);
    const uint32_t word = *reinterpret_cast<const uint32_t *>(grp + q4k_word_offset(R, i, c, v));
    float2 vals[4];
    q4k_word_f32(word, dl, ml, vals);
    float4 *o = reinterpret_cast<float4 *>(out + n * K + b * Q4K_BLOCK + 8 * lane);
    o[0] = make_float4(vals[0].x, vals[0].y, vals[1].x, vals[1].y);
    o[1] = make_float4(vals[2].x, vals[2].y, vals[3].x, vals[3].y);
}

// ---------------------------------------------------------------- Q6_K repack

// Low four bits and high two bits of element e (0..255) of a GGML Q6_K block:
// in half h, element 32j + l takes its low bits from ql[64h + l + 32(j%2)] (low
// nibble for j < 2, high nibble for j >= 2) and its high bits from bits 2j..2j+1
// of qh[32h + l].
__device__ __forceinline__ uint32_t q6k_src_low(const uint8_t *blk, int e) {
    const int h = e >> 7, j = (e >> 5) & 3, l = e & 31;
    const uint32_t byte = blk[64 * h + l + 32 * (j & 1)];
    return (j < 2) ? (byte & 15u) : (byte >> 4);
}
__device__ __forceinline__ uint32_t q6k_src_high(const uint8_t *blk, int e) {
    const int h = e >> 7, j = (e >> 5) & 3, l = e & 31;
    return (blk[128 + 32 * h + l] >> (2 * j)) & 3u;
}

// One warp per (stored row n, super-block b), stored rows running over the
// padded last tile too (its padding rows are written as zeros).  Lane l builds
// low word v = l%8 of chunk c = l/8; lanes 0..15 also build high word u = l%4 of
// chunk l/4; lane 0 copies d, lanes 0..3 four scale bytes each.
__global__ void q6k_repack_kernel(const uint8_t *__restrict__ src, uint8_t *__restrict__ dst,
                                  int64_t N, int64_t K, int64_t stored_rows) {
    const int64_t nb = K / Q4K_BLOCK;
    const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (gw >= stored_rows * nb) return;
    const int lane = threadIdx.x & 31;
    const int64_t n = gw / nb, b = gw % nb;
    const int64_t tile = n / TILE_ROWS;
    const int i = static_cast<int>(n % TILE_ROWS);
    const int Rp = q6k_padded_rows(tile_rows(N, tile));
    const bool real = n < N;
    const uint8_t *blk = src + (real ? (n * nb + b) * Q6K_BLOCK_BYTES : 0);
    uint8_t *grp = dst + q6k_group_offset(K, tile, Rp, b);
    if (lane == 0)
        *reinterpret_cast<uint16_t *>(grp + 2 * i) =
            real ? static_cast<uint16_t>(blk[208] | (blk[209] << 8)) : static_cast<uint16_t>(0);
    if (lane < 4) {
        uint32_t sc = 0;
        if (real)
            for (int t = 0; t < 4; ++t) sc |= static_cast<uint32_t>(blk[192 + 4 * lane + t]) << (8 * t);
        *reinterpret_cast<uint32_t *>(grp + Q6K_SCALE_PLANE * Rp + 16 * i + 4 * lane) = sc;
    }
    {
        const int c = lane >> 3, v = lane & 7;
        uint32_t word = 0;
        if (real)
#pragma unroll
            for (int t = 0; t < 8; ++t)
                word |= q6k_src_low(blk, 64 * c + 8 * v + t) << ((t & 1) ? 16 + 4 * (t >> 1) : 4 * (t >> 1));
        *reinterpret_cast<uint32_t *>(grp + q6k_low_word_offset(Rp, i, c, v)) = word;
    }
    if (lane < 16) {
        const int c = lane >> 2, u = lane & 3;
        uint32_t word = 0;
        if (real)
#pragma unroll
            for (int t = 0; t < 16; ++t) word |= q6k_src_high(blk, 64 * c + 16 * u + t) << q6k_high_bit(t);
        *reinterpret_cast<uint32_t *>(grp + q6k_high_word_offset(Rp, i, c, u)) = word;
    }
}

// One warp per (row, super-block); lane l dequantizes elements 8l..8l+7 (low
// word v = l%8 of chunk c = l/8): (q - 32) exactly from the GEMM's magic pair,
// then one fp32 rounding of d*sc (exact) times (q - 32).
__global__ void q6k_dequant_kernel(const uint8_t *__restrict__ w, float *__restrict__ out,
                                   int64_t N, int64_t K) {
    const int64_t nb = K / Q4K_BLOCK;
    const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (gw >= N * nb) return;
    const int lane = threadIdx.x & 31;
    const int64_t n = gw / nb, b = gw % nb;
    const int64_t tile = n / TILE_ROWS;
    const int i = static_cast<int>(n % TILE_ROWS);
    const int Rp = q6k_padded_rows(tile_rows(N, tile));
    const uint8_t *grp = w + q6k_group_offset(K, tile, Rp, b);
    const int c = lane >> 3, v = lane & 7;
    const float d = __half2float(__ushort_as_half(*reinterpret_cast<const uint16_t *>(grp + 2 * i)));
    const int sc = static_cast<int8_t>(grp[Q6K_SCALE_PLANE * Rp + 16 * i + 4 * c + (v >> 1)]);
    const float dl = d * static_cast<float>(sc);
    const uint32_t lo = *reinterpret_cast<const uint32_t *>(grp + q6k_low_word_offset(Rp, i, c, v));
    const uint32_t hi = *reinterpret_cast<const uint32_t *>(grp + q6k_high_word_offset(Rp, i, c, v >> 1));
    float vals[8];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const uint32_t m = (v & 1) ? q6k_pair_magic<1>(lo, hi, p) : q6k_pair_magic<0>(lo, hi, p);
        const float2 q = __half22float2(q6k_centered(m));
        vals[2 * p] = dl * q.x;
        vals[2 * p + 1] = dl * q.y;
    }
    float4 *o = reinterpret_cast<float4 *>(out + n * K + b * Q4K_BLOCK + 8 * lane);
    o[0] = make_float4(vals[0], vals[1], vals[2], vals[3]);
    o[1] = make_float4(vals[4], vals[5], vals[6], vals[7]);
}

// ---------------------------------------------------------------- W4A16 repack

// One thread per word; consecutive threads read consecutive source words.
__global__ void w4_repack_kernel(const uint32_t *__restrict__ src, uint8_t *__restrict__ dst,
                                 int64_t N, int64_t K) {
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t wpr = K / 8;
    if (idx >= N * wpr) return;
    const int64_t n = idx / wpr, rem = idx % wpr;
    const int64_t j = rem / 8;
    const int v = static_cast<int>(rem % 8);
    const int64_t tile = n / TILE_ROWS;
    const int i = static_cast<int>(n % TILE_ROWS);
    const int R = tile_rows(N, tile);
    *reinterpret_cast<uint32_t *>(dst + w4_plane_offset(K, tile, R, j) + w4_word_offset(R, i, v)) =
        src[idx];
}

// One thread per word: the exact (1024+q) - (1024+zp) of the GEMM's unpack,
// then an exact fp32 product with the scale (at most 11 + 5 significant bits).
// zeros == NULL: symmetric, zero point 8.
__global__ void w4_dequant_kernel(const uint8_t *__restrict__ w, const __half *__restrict__ scales,
                                  const uint8_t *__restrict__ zeros, float *__restrict__ out,
                                  int64_t N, int64_t K, int64_t group) {
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t wpr = K / 8;
    if (idx >= N * wpr) return;
    const int64_t n = idx / wpr, rem = idx % wpr;
    const int64_t j = rem / 8;
    const int v = static_cast<int>(rem % 8);
    const int64_t tile = n / TILE_ROWS;
    const int i = static_cast<int>(n % TILE_ROWS);
    const int R = tile_rows(N, tile);
    const uint32_t word = *reinterpret_cast<const uint32_t *>(
        w + w4_plane_offset(K, tile, R, j) + w4_word_offset(R, i, v));
    const int64_t k0 = CHUNK_K * j + 8 * v;
    const int64_t g = k0 / group;
    const float s = __half2float(scales[n * (K / group) + g]);
    const __half2 mz = w4_magic_zero(zeros ? zeros[n * (K / group) + g] : 8u);
    float vals[8];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const float2 qz = __half22float2(w4_pair_minus_zero(word, p, mz));
        vals[2 * p] = qz.x * s;
        vals[2 * p + 1] = qz.y * s;
    }
    float4 *o = reinterpret_cast<float4 *>(out + n * K + k0);
    o[0] = make_float4(vals[0], vals[1], vals[2], vals[3]);
    o[1] = make_float4(vals[4], vals[5], vals[6], vals[7]);
}

// Activations bf16 -> fp16 for the fp16 MMA path.  Every bf16 value of
// magnitude in [2^-14, 65504] converts exactly (8 significant bits fit fp16's
// 11); smaller values become fp16 subnormals (absolute error <= 2^-25); values
// that would round to infinity set the range flag in the status word.  Lets the
// dependent GEMM launch start (programmatic dependent launch) right away, and
// waits for the grids before it (which may write x or still read `out`).
__global__ void bf16_to_f16_kernel(const uint4 *__restrict__ in, uint4 *__restrict__ out, int64_t n8,
                                   uint32_t *status, uint32_t *zero, int nzero) {
    pdl_launch_dependents();
    pdl_wait();
    if (blockIdx.x == 0)
        for (int i = threadIdx.x; i < nzero; i += blockDim.x) zero[i] = 0u;
    bool overflow = false;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const uint4 v = in[i];
        const uint32_t src[4] = {v.x, v.y, v.z, v.w};
        uint32_t dst[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float lo = __uint_as_float(src[e] << 16);
            const float hi = __uint_as_float(src[e] & 0xFFFF0000u);
            overflow |= !(fabsf(lo) < 65520.f) || !(fabsf(hi) < 65520.f);
            dst[e] = as_u32(__floats2half2_rn(lo, hi));
        }
        out[i] = make_uint4(dst[0], dst[1], dst[2], dst[3]);
    }
    if (overflow) atomicOr(status, kStatusRangeBit);
}

int launch_bf16_to_f16(const void *x, void *out, int64_t n, cudaStream_t stream, uint32_t *zero, int nzero) {
    uint32_t *status = status_word();
    if (!status) return QWP_ERR_CUDA;
    const int64_t n8 = n / 8;
    const int64_t blocks = std::min<int64_t>((n8 + 255) / 256, 152 * 8);
    return launch_pdl(bf16_to_f16_kernel, static_cast<unsigned>(std::max<int64_t>(blocks, 1)), 256, stream,
                      static_cast<const uint4 *>(x), static_cast<uint4 *>(out), n8, status, zero, zero ? nzero : 0);
}

// Activation quantization to the record order of qwp_format.cuh: one warp per
// (token, super-block), lane l taking elements 8l..8l+7 (block l/4 of 32).  Per
// block: d = amax/127, q = round-half-away-from-zero(x * (1/d)) (0 when d == 0),
// each step correctly rounded in fp32 (GGML's Q8_1 rule with the scale kept in
// fp32), s = sum of the codes.  Tokens past M (padding of the last group) are
// written as zeros.  A non-finite x sets the range bit of the status word.
__global__ void q8_quantize_kernel(const uint4 *__restrict__ x, uint8_t *__restrict__ out, int M, int K,
                                   int64_t warps, uint32_t *status) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t wi = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (wi >= warps) return;  // surplus warps of the last block leave whole (wi is warp-uniform)
    const int lane = static_cast<int>(threadIdx.x & 31);
    const int nsb = K / Q4K_BLOCK;
    const int64_t m = wi / nsb;  // token (padded count)
    const int b = static_cast<int>(wi - m * nsb);
    float v[8];
    bool bad = false;
    if (m < M) {
        const uint4 raw = x[(m * K + static_cast<int64_t>(b) * Q4K_BLOCK) / 8 + lane];
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = 0.f;
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        bad |= !isfinite(v[i]);
        amax = fmaxf(amax, fabsf(v[i]));
    }
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const float d = __fdiv_rn(amax, 127.f);
    const float id = d != 0.f ? __fdiv_rn(1.f, d) : 0.f;
    int q[8], sum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        q[i] = static_cast<int>(roundf(__fmul_rn(v[i], id)));
        sum += q[i];
    }
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
    // e0 e4 e1 e5 | e2 e6 e3 e7
    const uint32_t lo = (q[0] & 0xFF) | ((q[4] & 0xFF) << 8) | ((q[1] & 0xFF) << 16) | (static_cast<uint32_t>(q[5]) << 24);
    const uint32_t hi = (q[2] & 0xFF) | ((q[6] & 0xFF) << 8) | ((q[3] & 0xFF) << 16) | (static_cast<uint32_t>(q[7]) << 24);
    const int64_t g = m / Q8_GROUP_TOKENS;
    uint8_t *rec = out + (g * nsb + b) * Q8_RECORD_BYTES + (m % Q8_GROUP_TOKENS) * Q8_TOKEN_BYTES;
    *reinterpret_cast<uint2 *>(rec + 8 * lane) = make_uint2(lo, hi);
    if ((lane & 3) == 0) {
        reinterpret_cast<float *>(rec + 256)[lane >> 2] = d;
        reinterpret_cast<float *>(rec + 288)[lane >> 2] = static_cast<float>(sum);
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(status, kStatusRangeBit);
}

static std::atomic<uint64_t> g_wait_timeout_ns{kDefaultTimeoutNs};

uint64_t wait_timeout_ns() { return g_wait_timeout_ns.load(std::memory_order_relaxed); }

static unsigned grid_for(int64_t threads, int block) {
    return static_cast<unsigned>((threads + block - 1) / block);
}

}  // namespace qwp

using namespace qwp;

extern "C" const char *qwp_status_string(int status) {
    switch (status) {
        case QWP_OK: return "QWP_OK";
        case QWP_ERR_INVALID_ARG: return "QWP_ERR_INVALID_ARG";
        case QWP_ERR_UNSUPPORTED_SHAPE: return "QWP_ERR_UNSUPPORTED_SHAPE";
        case QWP_ERR_MISALIGNED: return "QWP_ERR_MISALIGNED";
        case QWP_ERR_CUDA: return "QWP_ERR_CUDA";
        case QWP_ERR_DEVICE: return "QWP_ERR_DEVICE";
        case QWP_ERR_TIMEOUT: return "QWP_ERR_TIMEOUT";
        case QWP_ERR_RANGE: return "QWP_ERR_RANGE";
        case QWP_ERR_SCRATCH_LIMIT: return "QWP_ERR_SCRATCH_LIMIT";
        default: return "QWP_ERR_UNKNOWN";
    }
}

extern "C" int q4k_repacked_bytes(int64_t N, int64_t K, size_t *out_bytes) {
    if (!out_bytes || N < 0 || K < 0) return QWP_ERR_INVALID_ARG;
    if (K % Q4K_BLOCK) return QWP_ERR_UNSUPPORTED_SHAPE;
    *out_bytes = static_cast<size_t>(N) * static_cast<size_t>(K / Q4K_BLOCK) * Q4K_BLOCK_BYTES;
    return QWP_OK;
}

// Stored rows of the Q6_K layout: full tiles plus the last tile padded to a multiple of 8.
static int64_t q6k_stored_rows(int64_t N) {
    const int64_t full = N / TILE_ROWS * TILE_ROWS;
    return full + q6k_padded_rows(static_cast<int>(N - full));
}

extern "C" int q6k_repacked_bytes(int64_t N, int64_t K, size_t *out_bytes) {
    if (!out_bytes || N < 0 || K < 0) return QWP_ERR_INVALID_ARG;
    if (K % Q4K_BLOCK) return QWP_ERR_UNSUPPORTED_SHAPE;
    *out_bytes = static_cast<size_t>(q6k_stored_rows(N)) * static_cast<size_t>(K / Q4K_BLOCK) * Q6K_BLOCK_BYTES;
    return QWP_OK;
}

extern "C" int w4a16_repacked_bytes(int64_t N, int64_t K, size_t *out_bytes) {
    if (!out_bytes || N < 0 || K < 0) return QWP_ERR_INVALID_ARG;
    if (K % CHUNK_K) return QWP_ERR_UNSUPPORTED_SHAPE;
    *out_bytes = static_cast<size_t>(N) * static_cast<size_t>(K) / 2;
    return QWP_OK;
}

static int q4k_common_checks(const void *a, const void *b, int64_t N, int64_t K) {
    if (N < 0 || K < 0) return QWP_ERR_INVALID_ARG;
    if (K % Q4K_BLOCK) return QWP_ERR_UNSUPPORTED_SHAPE;
    if (N == 0 || K == 0) return QWP_OK;
    if (!a || !b) return QWP_ERR_INVALID_ARG;
    if (!aligned16(a) || !aligned16(b)) return QWP_ERR_MISALIGNED;
    if (a == b) return QWP_ERR_INVALID_ARG;  // outputs never alias inputs
    return check_device();
}

extern "C" int q4k_repack(const void *w_ggml, void *w_tiled, int64_t N, int64_t K, void *stream) {
    int rc = q4k_common_checks(w_ggml, w_tiled, N, K);
    if (rc || N == 0 || K == 0) return rc;
    const int64_t threads = N * (K / Q4K_BLOCK) * 32;
    q4k_repack_kernel<<<grid_for(threads, 256), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint8_t *>(w_ggml), static_cast<uint8_t *>(w_tiled), N, K);
    return launch_status();
}

extern "C" int q4k_dequant(const void *w_tiled, float *w_out, int64_t N, int64_t K, void *stream) {
    int rc = q4k_common_checks(w_tiled, w_out, N, K);
    if (rc || N == 0 || K == 0) return rc;
    const int64_t threads = N * (K / Q4K_BLOCK) * 32;
    q4k_dequant_kernel<<<grid_for(threads, 256), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint8_t *>(w_tiled), w_out, N, K);
    return launch_status();
}

extern "C" int q6k_repack(const void *w_ggml, void *w_tiled, int64_t N, int64_t K, void *stream) {
    int rc = q4k_common_checks(w_ggml, w_tiled, N, K);
    if (rc || N == 0 || K == 0) return rc;
    const int64_t rows = q6k_stored_rows(N);
    const int64_t threads = rows * (K / Q4K_BLOCK) * 32;
    q6k_repack_kernel<<<grid_for(threads, 256), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint8_t *>(w_ggml), static_cast<uint8_t *>(w_tiled), N, K, rows);
    return launch_status();
}

extern "C" int q6k_dequant(const void *w_tiled, float *w_out, int64_t N, int64_t K, void *stream) {
    int rc = q4k_common_checks(w_tiled, w_out, N, K);
    if (rc || N == 0 || K == 0) return rc;
    const int64_t threads = N * (K / Q4K_BLOCK) * 32;
    q6k_dequant_kernel<<<grid_for(threads, 256), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint8_t *>(w_tiled), w_out, N, K);
    return launch_status();
}

static int w4_common_checks(const void *a, const void *b, int64_t N, int64_t K) {
    if (N < 0 || K < 0) return QWP_ERR_INVALID_ARG;
    if (K % CHUNK_K) return QWP_ERR_UNSUPPORTED_SHAPE;
    if (N == 0 || K == 0) return QWP_OK;
    if (!a || !b) return QWP_ERR_INVALID_ARG;
    if (!aligned16(a) || !aligned16(b)) return QWP_ERR_MISALIGNED;
    if (a == b) return QWP_ERR_INVALID_ARG;  // outputs never alias inputs
    return check_device();
}

extern "C" int w4a16_repack(const void *wq, void *wq_tiled, int64_t N, int64_t K, void *stream) {
    int rc = w4_common_checks(wq, wq_tiled, N, K);
    if (rc || N == 0 || K == 0) return rc;
    const int64_t threads = N * (K / 8);
    w4_repack_kernel<<<grid_for(threads, 256), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint32_t *>(wq), static_cast<uint8_t *>(wq_tiled), N, K);
    return launch_status();
}

extern "C" int w4a16_dequant(const void *wq_tiled, const void *scales, const uint8_t *zeros,
                             float *w_out, int64_t N, int64_t K, int64_t group, void *stream) {
    if (group <= 0 || group % CHUNK_K) return QWP_ERR_INVALID_ARG;
    if (K % group) return QWP_ERR_UNSUPPORTED_SHAPE;
    if (N > 0 && K > 0 && !scales) return QWP_ERR_INVALID_ARG;
    int rc = w4_common_checks(wq_tiled, w_out, N, K);
    if (rc || N == 0 || K == 0) return rc;
    const int64_t threads = N * (K / 8);
    w4_dequant_kernel<<<grid_for(threads, 256), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint8_t *>(wq_tiled), static_cast<const __half *>(scales), zeros, w_out, N,
        K, group);
    return launch_status();
}

extern "C" int q8_activation_bytes(int64_t M, int64_t K, size_t *out_bytes) {
    if (M < 0 || K < 0 || !out_bytes) return QWP_ERR_INVALID_ARG;
    if (K % Q4K_BLOCK) return QWP_ERR_UNSUPPORTED_SHAPE;
    *out_bytes = static_cast<size_t>((M + Q8_GROUP_TOKENS - 1) / Q8_GROUP_TOKENS) * (K / Q4K_BLOCK) * Q8_RECORD_BYTES;
    return QWP_OK;
}

extern "C" int q8_quantize(const void *x_bf16, void *xq, int64_t M, int64_t K, void *stream) {
    if (M < 0 || K < 0) return QWP_ERR_INVALID_ARG;
    if (K % Q4K_BLOCK) return QWP_ERR_UNSUPPORTED_SHAPE;
    if (M == 0 || K == 0) return QWP_OK;
    if (!x_bf16 || !xq) return QWP_ERR_INVALID_ARG;
    if (!aligned16(x_bf16) || !aligned16(xq)) return QWP_ERR_MISALIGNED;
    if (M > (int64_t(1) << 31) - 8 || K > (int64_t(1) << 30)) return QWP_ERR_UNSUPPORTED_SHAPE;
    int rc = check_device();
    if (rc) return rc;
    uint32_t *status = status_word();
    if (!status) return QWP_ERR_CUDA;
    const int64_t mpad = (M + Q8_GROUP_TOKENS - 1) / Q8_GROUP_TOKENS * Q8_GROUP_TOKENS;
    const int64_t warps = mpad * (K / Q4K_BLOCK);
    return launch_pdl(q8_quantize_kernel, grid_for(warps * 32, 256), 256, static_cast<cudaStream_t>(stream),
                      static_cast<const uint4 *>(x_bf16), static_cast<uint8_t *>(xq), static_cast<int>(M),
                      static_cast<int>(K), warps, status);
}

extern "C" int qwp_set_wait_timeout_ns(uint64_t ns) {
    if (ns == 0 || ns > 60000000000ull) return QWP_ERR_INVALID_ARG;
    g_wait_timeout_ns.store(ns, std::memory_order_relaxed);
    return QWP_OK;
}

extern "C" int qwp_device_status(void *stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return QWP_ERR_CUDA;
    uint32_t *p = status_word();
    if (!p) return QWP_ERR_CUDA;
    uint32_t v = 0;
    if (cudaMemcpy(&v, p, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return QWP_ERR_CUDA;
    if (v && cudaMemset(p, 0, sizeof(v)) != cudaSuccess) return QWP_ERR_CUDA;
    if (v & kStatusTimeoutMask) return QWP_ERR_TIMEOUT;
    return v ? QWP_ERR_RANGE : QWP_OK;
}
