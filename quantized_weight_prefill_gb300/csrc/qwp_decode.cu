// Decode-shaped products (M <= 8 tokens) over the repacked weights.
//
// Method: the batched DMMV of "How ZINC's RDNA4 batched prefill went from 42 to
// 208 tok/s", section "The fix: K-parallel batched DMMV" (every weight row is
// read once and applied to all the chunk's tokens), and the small-token regime of
// "The dequant scratch round-trip is ZINC's last RDNA4 prefill tax", section
// "What the roofline says": with at most 8 tokens every weight is used at most 8
// times, so the product is bound by the packed-weight stream from HBM.  The
// tensor-memory pipeline of the prefill kernel would spend its fixed per-stage
// cost on a few tokens; here each warp unpacks straight into the A fragments of
// mma.sync m16n8k16 (16 weight rows x 8 tokens x 16 K, fp16 in, fp32 out) and no
// operand makes a round trip through shared or tensor memory.
//
// Work is split stream-K style: the items (128-row tile, 256-wide super-block),
// numbered tile-major, are cut into one contiguous range per CTA of a persistent
// grid, so that every SM streams the same number of weight bytes and each CTA
// pays its start-up latency once.  Roles per CTA:
//   warps 0..7  consumers: warp c computes rows 16c..16c+15 of the current tile
//               for all 8 token columns, accumulating over the tile's items;
//   warp 8      producer: one thread streams each item's weight group (one bulk
//               copy of the tile-major group) and the 8 x 256 activation slice
//               (four 2-D TMA boxes of 64 K, 128-byte swizzle, rows past M
//               zero-filled) through a ring; with bf16 activations the warp then
//               converts the slice's M token rows to fp16 in place.
// A tile that a CTA covers entirely is written to y directly.  A tile shared by
// several CTAs (at most the first and the last tile of each range) is finished by
// whichever of them arrives last: each leaves its partial sums in scratch and
// counts itself in on the tile's counter; the last one adds the partials in CTA
// order (deterministic) and writes y.  No CTA ever waits for another.
//
// K order inside an MMA is free as long as A and B agree: for the 8 MMAs of a
// 128-wide K window, lane (g, t) (g = lane/4, t = lane%4) supplies the K slots
// {2t, 2t+1, 2t+8, 2t+9}, mapped to the 32 weights of sub-block t of the window,
// so that each lane unpacks whole 32-weight sub-blocks (one scale set per 32
// weights, as in the prefill transform) and reads 64 contiguous bytes of its
// token's activations.
#include <algorithm>
#include <cstring>
#include <atomic>
#include <mutex>

#include "qwp_decode.h"
#include "qwp_format.cuh"
#include "qwp_ptx.cuh"

namespace qwp {

constexpr int DEC_TOKENS = 8;                     // MMA N: token columns
constexpr int DEC_CWARPS = 8;                     // consumer warps, 16 rows each
constexpr int DEC_THREADS = 32 * (DEC_CWARPS + 1);
constexpr int DEC_X_BYTES = DEC_TOKENS * Q4K_BLOCK * 2;  // one super-block of x: 4 boxes of 8 x 128 B
constexpr int DEC_PART_FLOATS = DEC_CWARPS * 32 * 4;     // one float4 per consumer lane

// Ring depth per format, two CTAs per SM each: Q4_K 4 slots of 23 KiB, Q6_K 3 of
// 27 KiB, W4A16 4 of 20 KiB, the 8-bit-activation product 4 of 23 KiB.  (Q4_K ran
// three CTAs per SM with 3 slots until its single-rounding operand: with that
// unpack two CTAs of 96 registers measured 4.5% faster, M1 N152064 143 -> 136 us.)
template <int kFmt>
__host__ __device__ constexpr int dec_stages() { return kFmt == DFMT_Q6K ? 3 : 4; }

// The weight format a kernel instance streams (the quantized-activation product
// reads Q4_K weights).
template <int kFmt>
__host__ __device__ constexpr int dec_wfmt() { return kFmt == DFMT_Q4K_Q8 ? DFMT_Q4K : kFmt; }

// Items the producer issues before the first one has landed.
constexpr int DEC_PRE = 4;

// Fewest items per CTA when the problem is small (fewer, longer CTAs: less
// start-up and fewer shared tiles to finish).
constexpr int DEC_MIN_ITEMS = 4;

struct DecodeArgs {
    const uint8_t *w;
    const __half *scales;   // W4A16
    const uint8_t *zeros;   // W4A16, or null (symmetric)
    const uint8_t *xq;      // DFMT_Q4K_Q8: the quantized-activation records of the token group
    float *y;
    uint32_t *status;
    float *part;            // [grid][2][DEC_PART_FLOATS]: partials of shared tiles
    uint32_t *count;        // [row tiles]: CTAs done with a shared tile (zero at launch)
    int64_t items;          // row tiles x super-blocks
    int M, N, K, group, groups_per_row, nsb;
    int stage_stride;       // bytes per ring slot: x (1 KiB aligned) then weights
    int bar_off;            // offset of the mbarriers
    int x_bf16;             // 1: x is bf16 and converted in shared memory
    uint64_t timeout_ns;
};

// Bounded wait (see the prefill kernel): false on timeout or once the CTA aborts.
__device__ __forceinline__ bool dec_wait(uint32_t bar, uint32_t parity, uint32_t *abort,
                                         uint32_t *status, uint64_t timeout_ns, uint32_t where,
                                         bool honour_abort = true) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 7u) == 0) {
            if (honour_abort && *reinterpret_cast<volatile uint32_t *>(abort)) return false;
            if (global_timer_ns() - t0 > timeout_ns) {
                *reinterpret_cast<volatile uint32_t *>(abort) = 1u;
                atomicCAS(status, 0u, 0x100u | where);
                return false;
            }
        }
    }
}

enum : uint32_t { DWAIT_FULL = 0x21, DWAIT_READY, DWAIT_EMPTY, DWAIT_DRAIN };

__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Barrier 1 among the consumer warps only (the producer warp never joins it).
__device__ __forceinline__ void consumers_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(DEC_CWARPS * 32) : "memory");
}

// Byte offsets inside a weight stage of the two rows a lane computes (clamped
// into the tile: rows past its end read a valid row, and their results are never
// stored) for the lane's 32-wide sub-block t of the first 128-wide window; the
// second window is wstride (two 64-wide chunks) further, its Q6_K scales 8 bytes
// and its Q6_K high words hstride further.  They depend on the tile's rows only.
template <int kFmt>
struct DecRows {
    int a_hdr, b_hdr;  // Q4_K: 16-byte headers; Q6_K: fp16 d
    int a_w, b_w;      // the sub-block's 4 low words
    int a_sc, b_sc;    // Q6_K: its two int8 scales
    int a_hi, b_hi;    // Q6_K: its two high words
    int wstride, hstride;
    int64_t na, nb;    // W4A16: global rows (scale and zero-point index)

    __device__ __forceinline__ void set(int R, int ra, int rb, int t, int64_t tile) {
        ra = min(ra, R - 1);
        rb = min(rb, R - 1);
        const int c = t >> 1, h = t & 1;
        if (kFmt == DFMT_Q4K) {
            a_hdr = Q4K_HEADER_BYTES * ra;
            b_hdr = Q4K_HEADER_BYTES * rb;
            a_w = Q4K_HEADER_BYTES * R + CHUNK_ROW_BYTES * R * c + (h * R + ra) * 16;
            b_w = a_w + (rb - ra) * 16;
            wstride = 2 * CHUNK_ROW_BYTES * R;
        } else if (kFmt == DFMT_Q6K) {
            const int Rp = q6k_padded_rows(R);
            a_hdr = 2 * ra;
            b_hdr = 2 * rb;
            a_sc = Q6K_SCALE_PLANE * Rp + 16 * ra + 2 * t;
            b_sc = a_sc + 16 * (rb - ra);
            a_w = Q6K_LOW_PLANE * Rp + CHUNK_ROW_BYTES * Rp * c + (h * Rp + ra) * 16;
            b_w = a_w + (rb - ra) * 16;
            a_hi = Q6K_HIGH_PLANE * Rp + 16 * Rp * c + 16 * ra + 8 * h;
            b_hi = a_hi + 16 * (rb - ra);
            wstride = 2 * CHUNK_ROW_BYTES * Rp;
            hstride = 32 * Rp;
        } else {
            a_w = CHUNK_ROW_BYTES * R * c + (h * R + ra) * 16;
            b_w = a_w + (rb - ra) * 16;
            wstride = 2 * CHUNK_ROW_BYTES * R;
            na = tile * TILE_ROWS + ra;
            nb = tile * TILE_ROWS + rb;
        }
    }
};

// (1024 + sc, 1024 + m) of Q4_K sub-block 4*kWin + t as raw fp16x2 bits, the byte
// shift sh = 8t precomputed (the GGML 6-bit packing, as q4k_scmin_magic).
template <int kWin>
__device__ __forceinline__ uint32_t q4k_scmin_lane(uint4 h, uint32_t sh) {
    const uint32_t b_lo = h.y >> sh, b_mid = h.z >> sh;
    uint32_t sc, m;
    if (kWin == 0) {
        sc = b_lo & 63u;
        m = b_mid & 63u;
    } else {
        const uint32_t b_hi = h.w >> sh;
        sc = (b_hi & 15u) | ((b_lo >> 2) & 0x30u);
        m = ((b_hi >> 4) & 15u) | ((b_mid >> 2) & 0x30u);
    }
    return 0x64006400u | sc | (m << 16);
}

// The unpack constants of one row's sub-block and its 4 words.
template <int kFmt>
struct DecSub {
    uint4 wv;
    Q4kSubH ks;        // Q4_K
    uint2 hv;          // Q6_K high words of the two 16-wide halves
    Q6kSub ds0, ds1;   // Q6_K constants of the halves
    __half2 s2, mz;    // W4A16 scale, 1024 + zero point

    template <int kWin>
    __device__ __forceinline__ void load(const uint8_t *wst, int hdr, int w, int sc, int hi, int wstride, int hstride,
                                         uint32_t sh, int64_t n, int gidx, const DecodeArgs &args) {
        wv = *reinterpret_cast<const uint4 *>(wst + w + kWin * wstride);
        if (kFmt == DFMT_Q4K) {
            const uint4 h = *reinterpret_cast<const uint4 *>(wst + hdr);
            ks = q4k_sub_consts(h.x, __hsub2(as_half2(q4k_scmin_lane<kWin>(h, sh)), as_half2(0x64006400u)));
        } else if (kFmt == DFMT_Q6K) {
            const uint32_t dbits = *reinterpret_cast<const uint16_t *>(wst + hdr);
            const uint32_t sc2 = *reinterpret_cast<const uint16_t *>(wst + sc + 8 * kWin);
            hv = *reinterpret_cast<const uint2 *>(wst + hi + kWin * hstride);
            ds0 = q6k_sub(dbits, static_cast<int8_t>(sc2 & 0xFFu));
            ds1 = q6k_sub(dbits, static_cast<int8_t>(sc2 >> 8));
        } else {
            const int64_t gi = n * args.groups_per_row + gidx;
            s2 = __half2half2(args.scales[gi]);
            mz = w4_magic_zero(args.zeros ? args.zeros[gi] : 8u);
        }
    }

    // Word u (0..3, elements 8u..8u+7 of the sub-block) as 4 fp16 pairs.
    template <int u>
    __device__ __forceinline__ void word(uint32_t (&p)[4]) const {
        const uint32_t w = u == 0 ? wv.x : u == 1 ? wv.y : u == 2 ? wv.z : wv.w;
        if (kFmt == DFMT_Q4K)
            q4k_word_f16x2(w, ks, p);
        else if (kFmt == DFMT_Q6K)
            q6k_word_f16x2<u & 1>(w, (u >> 1) ? hv.y : hv.x, (u >> 1) ? ds1 : ds0, p);
        else
            w4_word_f16x2(w, mz, s2, p);
    }
};

// The 4 MMAs of half u (0 or 1) of a lane's window: A pairs from words u and u + 2
// of rows a (a0, a2) and b (a1, a3); B pairs from x chunks u and u + 2.
template <int u, int kFmt>
__device__ __forceinline__ void dec_half(const DecSub<kFmt> &qa, const DecSub<kFmt> &qb, const uint8_t *xw,
                                         const int (&xo)[4], float (&acc)[4]) {
    uint32_t lo0[4], hi0[4], lo1[4], hi1[4];
    qa.template word<u>(lo0);
    qa.template word<u + 2>(hi0);
    qb.template word<u>(lo1);
    qb.template word<u + 2>(hi1);
    const uint4 xa = *reinterpret_cast<const uint4 *>(xw + xo[u]);
    const uint4 xc = *reinterpret_cast<const uint4 *>(xw + xo[u + 2]);
    const uint32_t b0[4] = {xa.x, xa.y, xa.z, xa.w}, b1[4] = {xc.x, xc.y, xc.z, xc.w};
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const uint32_t a[4] = {lo0[p], lo1[p], hi0[p], hi1[p]};
        mma_16816(acc, a, b0[p], b1[p]);
    }
}

// One 128-wide window (kWin) of an item: the lane's sub-block 4*kWin + t of rows a, b.
template <int kWin, int kFmt>
__device__ __forceinline__ void dec_window(const uint8_t *wst, const uint8_t *xst, const DecRows<kFmt> &o,
                                           const int (&xo)[4], uint32_t sh, int gidx, const DecodeArgs &args,
                                           float (&acc)[4]) {
    DecSub<kFmt> qa, qb;
    qa.template load<kWin>(wst, o.a_hdr, o.a_w, o.a_sc, o.a_hi, o.wstride, o.hstride, sh, o.na, gidx, args);
    qb.template load<kWin>(wst, o.b_hdr, o.b_w, o.b_sc, o.b_hi, o.wstride, o.hstride, sh, o.nb, gidx, args);
    const uint8_t *xw = xst + 2048 * kWin;  // the window's two 64-wide boxes
    dec_half<0>(qa, qb, xw, xo, acc);
    dec_half<1>(qa, qb, xw, xo, acc);
}

// Quantized activations: one item's share of a lane -- row rr of the tile (R rows,
// rr clamped into it) and sub-blocks 4*half .. 4*half+3 of the super-block -- for
// NT tokens.  Per sub-block j and token t the 32 products of the 4-bit weight codes
// with token t's 8-bit codes are summed exactly with 8 dp4a, as S = 16 * dot: the
// high nibbles are used in place (w & 0xF0F0F0F0, i.e. 16 * code) and the low ones
// moved up by a multiply (the shift runs on the FMA pipe, the masks on the ALU
// pipe), each against the matching word of codes of the record; then
//     acc[t] += d_t,j * ((d*sc_j / 16) * S - dmin*m_j * s_t,j),
// which is sum_k w_k * d_t,j * q_t,k over the sub-block (w = d*sc*q - dmin*m).
// d*sc_j / 16 and dmin*m_j are exact in fp32; |S| < 2^20 converts exactly.
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

template <int NT, int T0>
__device__ __forceinline__ void q8_item(const uint8_t *wst, const uint8_t *xst, int R, int rr, int half,
                                        float (&acc)[8]) {
    const uint4 h = *reinterpret_cast<const uint4 *>(wst + Q4K_HEADER_BYTES * rr);
    const float d16 = __half2float(__ushort_as_half(static_cast<unsigned short>(h.x & 0xFFFFu))) * 0.0625f;
    const float dmin = __half2float(__ushort_as_half(static_cast<unsigned short>(h.x >> 16)));
    // The row's words of sub-block 4*half (chunk 2*half, first half-plane); sub-block
    // 4*half + jj sits jj/2 chunk planes (32*R bytes) and jj%2 half-planes (16*R) further.
    const uint8_t *w0 = wst + Q4K_HEADER_BYTES * R + CHUNK_ROW_BYTES * R * (2 * half) + rr * 16;
    const uint8_t *x0 = xst + T0 * Q8_TOKEN_BYTES + 128 * half;  // token T0's codes of sub-block 4*half
    const float *dx0 = reinterpret_cast<const float *>(xst + T0 * Q8_TOKEN_BYTES + 256 + 16 * half);  // scale; sum +32 B
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
        const uint4 wv = *reinterpret_cast<const uint4 *>(w0 + (jj >> 1) * (CHUNK_ROW_BYTES * R) + (jj & 1) * (16 * R));
        const uint32_t w[4] = {wv.x, wv.y, wv.z, wv.w};
        uint32_t lo[4], hi[4];
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            lo[v] = (w[v] * 16u) & 0xF0F0F0F0u;  // 16 x elements 8v + (0, 4, 1, 5)
            hi[v] = w[v] & 0xF0F0F0F0u;          // 16 x elements 8v + (2, 6, 3, 7)
        }
        // The 6-bit scale and min of sub-block jj (half 0) or jj + 4 (half 1).
        const uint32_t sh = 8u * jj;
        const uint32_t b_lo = h.y >> sh, b_mid = h.z >> sh, b_hi = h.w >> sh;
        const uint32_t sc = half ? ((b_hi & 15u) | ((b_lo >> 2) & 0x30u)) : (b_lo & 63u);
        const uint32_t mn = half ? (((b_hi >> 4) & 15u) | ((b_mid >> 2) & 0x30u)) : (b_mid & 63u);
        const float dsc16 = d16 * static_cast<float>(sc), dm = dmin * static_cast<float>(mn);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const uint8_t *xt = x0 + t * Q8_TOKEN_BYTES + 32 * jj;
            const uint4 xa = *reinterpret_cast<const uint4 *>(xt);
            const uint4 xb = *reinterpret_cast<const uint4 *>(xt + 16);
            int s16 = dp4a_us(lo[0], xa.x, 0);
            s16 = dp4a_us(hi[0], xa.y, s16);
            s16 = dp4a_us(lo[1], xa.z, s16);
            s16 = dp4a_us(hi[1], xa.w, s16);
            s16 = dp4a_us(lo[2], xb.x, s16);
            s16 = dp4a_us(hi[2], xb.y, s16);
            s16 = dp4a_us(lo[3], xb.z, s16);
            s16 = dp4a_us(hi[3], xb.w, s16);
            const float dx = dx0[t * (Q8_TOKEN_BYTES / 4) + jj];
            const float sx = dx0[t * (Q8_TOKEN_BYTES / 4) + 8 + jj];
            acc[T0 + t] = fmaf(dx, fmaf(dsc16, static_cast<float>(s16), -(dm * sx)), acc[T0 + t]);
        }
    }
}

// The token count as a compile-time 1, 2 or 4 per pass, 8 tokens in two passes
// (the record's tokens past M are zero codes with zero scale and sum, so rounding
// M up adds exact zeros to accumulators that are never stored; the weight words are
// unpacked once per pass).  At two CTAs per SM (96 registers) no pass spills.
__device__ __forceinline__ void q8_item_m(const uint8_t *wst, const uint8_t *xst, int R, int rr, int half, int M,
                                          float (&acc)[8]) {
    if (M == 1) {
        q8_item<1, 0>(wst, xst, R, rr, half, acc);
    } else if (M == 2) {
        q8_item<2, 0>(wst, xst, R, rr, half, acc);
    } else {
        q8_item<4, 0>(wst, xst, R, rr, half, acc);
        if (M > 4) q8_item<4, 4>(wst, xst, R, rr, half, acc);
    }
}

// First item of CTA c's range, and the CTA whose range holds item i.
// (items * G < 2^32: 32-bit arithmetic.)
__device__ __forceinline__ uint32_t range_begin(uint32_t c, uint32_t items, uint32_t G) { return c * items / G; }
__device__ __forceinline__ uint32_t item_owner(uint32_t i, uint32_t items, uint32_t G) {
    return ((i + 1) * G - 1) / items;
}

template <int kFmt>
__global__ void __launch_bounds__(DEC_THREADS, 2)
    qwp_decode_kernel(const __grid_constant__ CUtensorMap tmap_x, const DecodeArgs args) {
    constexpr int NS = dec_stages<kFmt>();
    constexpr bool kQ8 = kFmt == DFMT_Q4K_Q8;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const uint32_t warp = warp_id();
    const uint32_t lane = lane_id();
    // Items and grid are small enough for 32-bit range arithmetic (the host checks
    // items * grid < 2^32).
    const uint32_t G = gridDim.x, cta = blockIdx.x, items = static_cast<uint32_t>(args.items);
    const uint32_t beg = cta * items / G, end = (cta + 1) * items / G;
    const int n_items = static_cast<int>(end - beg);
    const uint32_t nsb = static_cast<uint32_t>(args.nsb);

    const uint32_t bar0 = smem_u32(smem + args.bar_off);
    const uint32_t full = bar0, ready = bar0 + 8 * NS, empty = bar0 + 16 * NS;
    uint32_t *abort = reinterpret_cast<uint32_t *>(smem + args.bar_off + 24 * NS);
    uint32_t *last_flag = abort + 1;
    auto slot_x = [&](int s) { return smem + s * args.stage_stride; };
    auto slot_w = [&](int s) { return smem + s * args.stage_stride + DEC_X_BYTES; };

    // The producer's next item to issue, kept incrementally (no divisions per item):
    // its tile, super-block, weight-group address and bytes.
    uint32_t p_tile = 0, p_sb = 0, p_bytes = 0;
    const uint8_t *p_src = nullptr;
    auto p_setup_tile = [&]() {
        const int R = tile_rows(args.N, p_tile);
        if (dec_wfmt<kFmt>() == DFMT_Q4K) {
            p_bytes = static_cast<uint32_t>(R) * Q4K_BLOCK_BYTES;
            p_src = args.w + q4k_group_offset(args.K, p_tile, R, p_sb);
        } else if (kFmt == DFMT_Q6K) {
            const int Rp = q6k_padded_rows(R);
            p_bytes = static_cast<uint32_t>(Rp) * Q6K_BLOCK_BYTES;
            p_src = args.w + q6k_group_offset(args.K, p_tile, Rp, p_sb);
        } else {
            p_bytes = static_cast<uint32_t>(R) * CHUNK_ROW_BYTES * 4;
            p_src = args.w + w4_plane_offset(args.K, p_tile, R, 4 * static_cast<int64_t>(p_sb));
        }
    };
    // Lane 0 of the producer warp: item beg + st (= the next one) into slot st % NS.
    auto issue_next = [&](int st) {
        const int s = st % NS;
        if (kQ8) {
            // The super-block's quantized-activation record: one contiguous copy.
            mbar_arrive_expect_tx(full + 8 * s, p_bytes + Q8_RECORD_BYTES);
            bulk_copy_g2s(smem_u32(slot_w(s)), p_src, p_bytes, full + 8 * s);
            bulk_copy_g2s(smem_u32(slot_x(s)), args.xq + static_cast<int64_t>(p_sb) * Q8_RECORD_BYTES, Q8_RECORD_BYTES,
                          full + 8 * s);
        } else {
            mbar_arrive_expect_tx(full + 8 * s, p_bytes + DEC_X_BYTES);
            bulk_copy_g2s(smem_u32(slot_w(s)), p_src, p_bytes, full + 8 * s);
            const int k0 = static_cast<int>(p_sb) * Q4K_BLOCK;
            for (int b = 0; b < 4; ++b)
                tma_load_2d(smem_u32(slot_x(s) + 1024 * b), &tmap_x, k0 + 64 * b, 0, full + 8 * s);
        }
        if (++p_sb == nsb) {
            p_sb = 0;
            ++p_tile;
            if (st + 1 < n_items) p_setup_tile();
        } else {
            p_src += p_bytes;  // consecutive super-blocks of a tile are consecutive groups
        }
    };

    // The producer thread sets up the barriers and starts its first copies at once;
    // thread 0 meanwhile reads the status word (a failure recorded by an earlier
    // launch makes this one skip its work; the copies started are still waited for).
    constexpr int PTHREAD = 32 * DEC_CWARPS;
    int issued = 0;
    pdl_launch_dependents();
    if (threadIdx.x == PTHREAD) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(full + 8 * s, 1);
            mbar_init(ready + 8 * s, 1);
            mbar_init(empty + 8 * s, DEC_CWARPS);
        }
        fence_mbar_init();
        p_tile = beg / nsb;
        p_sb = beg - p_tile * nsb;
        if (n_items > 0) p_setup_tile();
        // x, the weights and the status word may come from the grids launched just
        // before (every other thread is ordered after this wait by the barrier below).
        pdl_wait();
        // A failure recorded earlier makes this launch skip its work; the status load
        // is issued before the first copies and its value used after them, so that
        // its latency overlaps theirs.
        const uint32_t status_now = *reinterpret_cast<volatile uint32_t *>(args.status);
        const int pre = min(min(NS, DEC_PRE), n_items);
        for (int st = 0; st < pre; ++st) issue_next(st);
        issued = pre;
        *abort = (status_now & kStatusTimeoutMask) ? 1u : 0u;
    }
    __syncthreads();
    bool ok = *reinterpret_cast<volatile uint32_t *>(abort) == 0;

    if (warp == DEC_CWARPS) {
        // ------------------------------------------------------------ producer
        issued = __shfl_sync(0xffffffffu, issued, 0);
        bool range = false;
        const int nconv = 32 * args.M;  // 16-byte chunks of the M token rows in a slice
        for (int st = 0; ok && st < n_items; ++st) {
            const int s = st % NS;
            if (!(ok = __all_sync(0xffffffffu, dec_wait(full + 8 * s, (st / NS) & 1, abort, args.status,
                                                        args.timeout_ns, DWAIT_FULL))))
                break;
            if (args.x_bf16) {
                // Convert the slice's M token rows in place, then release it.
                uint4 *xs = reinterpret_cast<uint4 *>(slot_x(s));
                for (int idx = static_cast<int>(lane); idx < nconv; idx += 32) {
                    const int b = idx / (8 * args.M), rem = idx % (8 * args.M);
                    uint4 *p = xs + 64 * b + rem;  // box b, token rem / 8, chunk rem % 8
                    const uint4 v = *p;
                    const uint32_t src[4] = {v.x, v.y, v.z, v.w};
                    uint32_t dst[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float lo = __uint_as_float(src[e] << 16);
                        const float hi = __uint_as_float(src[e] & 0xFFFF0000u);
                        range |= !(fabsf(lo) < 65520.f) || !(fabsf(hi) < 65520.f);
                        dst[e] = as_u32(__floats2half2_rn(lo, hi));
                    }
                    *p = make_uint4(dst[0], dst[1], dst[2], dst[3]);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(ready + 8 * s);
            }
            // Keep NS items ahead: items up to st + NS - 1 may go out; one that reuses a
            // slot waits until the consumers have released the slot's previous item
            // (at most item st - 1, which they were able to start).
            const int target = min(n_items - 1, st + NS - 1);
            while (ok && issued <= target) {
                const int k = issued;
                if (lane == 0) {
                    if (k >= NS)
                        ok = dec_wait(empty + 8 * ((k - NS) % NS), ((k - NS) / NS) & 1, abort, args.status,
                                      args.timeout_ns, DWAIT_EMPTY);
                    if (ok) issue_next(k);
                }
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                if (ok) ++issued;
            }
        }
        if (args.x_bf16 && __any_sync(0xffffffffu, range) && lane == 0) atomicOr(args.status, kStatusRangeBit);
        // Every copy issued lands before the CTA may exit.
        if (lane == 0)
            for (int st = max(0, issued - NS); st < issued; ++st)
                dec_wait(full + 8 * (st % NS), (st / NS) & 1, abort, args.status, args.timeout_ns, DWAIT_DRAIN, false);
        __syncwarp();
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int g = static_cast<int>(lane >> 2), t = static_cast<int>(lane & 3);
    const int r0 = 16 * static_cast<int>(warp) + g, r1 = r0 + 8;
    // Quantized activations: lane l takes row 16*warp + l%16 of the tile and half
    // l/16 of each super-block's sub-blocks; at the end of a tile the two halves
    // are added and lane l keeps tokens 4*(l/16) .. +3 of the row.
    const int qrow = 16 * static_cast<int>(warp) + static_cast<int>(lane & 15), qhalf = static_cast<int>(lane >> 4);
    const uint32_t wait_bar = args.x_bf16 ? ready : full;
    const uint32_t first_tile = beg / nsb;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float acc8[DEC_TOKENS] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    bool fine = ok;  // every item so far was consumed

    // Writes (sum of) this CTA's values of tile `tile` to y: rows r0/r1, tokens 2t,
    // 2t+1 (the MMA fragment), or row qrow, tokens 4*qhalf .. +3.
    auto store = [&](uint32_t tile, const float (&v)[4]) {
        const int R = tile_rows(args.N, tile);
        const int64_t nb = tile * TILE_ROWS;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int row = kQ8 ? qrow : r0 + 8 * (e >> 1);
            const int tok = kQ8 ? 4 * qhalf + e : 2 * t + (e & 1);
            if (row < R && tok < args.M) args.y[static_cast<int64_t>(tok) * args.N + nb + row] = v[e];
        }
    };
    // The tile ends (its last item, or this CTA's last item): write it or hand it on.
    auto flush = [&](uint32_t tile) {
        const bool whole = tile * nsb >= beg && (tile + 1) * nsb <= end;
        if (whole) {
            if (fine) store(tile, acc);
            return;
        }
        const int slot = tile == first_tile ? 0 : 1;
        float4 *mine = reinterpret_cast<float4 *>(args.part + (cta * 2 + slot) * DEC_PART_FLOATS) + warp * 32 + lane;
        *mine = make_float4(acc[0], acc[1], acc[2], acc[3]);
        __threadfence();
        consumers_sync();
        if (threadIdx.x == 0) {
            const uint32_t c_lo = item_owner(tile * nsb, items, G);
            const uint32_t c_hi = item_owner((tile + 1) * nsb - 1, items, G);
            const uint32_t prior = atomicAdd(args.count + tile, 1u);
            *last_flag = prior == static_cast<uint32_t>(c_hi - c_lo) ? 1u : 0u;
        }
        consumers_sync();
        if (*reinterpret_cast<volatile uint32_t *>(last_flag)) {
            __threadfence();
            const uint32_t c_lo = item_owner(tile * nsb, items, G);
            const uint32_t c_hi = item_owner((tile + 1) * nsb - 1, items, G);
            float v[4] = {0.f, 0.f, 0.f, 0.f};
            for (uint32_t c0 = c_lo; c0 <= c_hi; c0 += 4) {
                // Up to four partials in flight, added in CTA order.
                float4 pv[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint32_t c = c0 + q;
                    pv[q] = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (c <= c_hi) {
                        const int sl = tile == range_begin(c, items, G) / nsb ? 0 : 1;
                        pv[q] = __ldcg(reinterpret_cast<const float4 *>(args.part + (c * 2 + sl) * DEC_PART_FLOATS) +
                                       warp * 32 + lane);
                    }
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    v[0] += pv[q].x; v[1] += pv[q].y; v[2] += pv[q].z; v[3] += pv[q].w;
                }
            }
            const bool failed = *reinterpret_cast<volatile uint32_t *>(args.status) & kStatusTimeoutMask;
            if (!failed) store(tile, v);
            if (threadIdx.x == 0) args.count[tile] = 0u;  // leaves the counters as found
        }
    };

    // Lane constants: x chunk c (0..3) of window 0 sits in box t/2, line g, at
    // 16-byte position (4*(t%2) + c) ^ g (128-byte swizzle); the Q4_K scale shift.
    int xo[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) xo[c] = 1024 * (t >> 1) + 128 * g + 16 * ((4 * (t & 1) + c) ^ g);
    const uint32_t sh = 8u * static_cast<uint32_t>(t);
    DecRows<kFmt> rows;
    uint32_t rows_tile = 0xFFFFFFFFu;
    uint32_t tile = first_tile;
    uint32_t sb = beg - first_tile * nsb;  // (tile, super-block) of item beg + st
    int s = 0;                                          // ring slot of item st, and its phase
    uint32_t ph = 0;
    for (int st = 0; st < n_items; ++st) {
        if (fine) {
            fine = __all_sync(0xffffffffu, dec_wait(wait_bar + 8 * s, ph, abort, args.status, args.timeout_ns,
                                                    args.x_bf16 ? DWAIT_READY : DWAIT_FULL));
        }
        if (fine) {
            const uint8_t *wst = slot_w(s);
            const uint8_t *xst = slot_x(s);
            if constexpr (kQ8) {
                const int R = tile_rows(args.N, tile);
                q8_item_m(wst, xst, R, min(qrow, R - 1), qhalf, args.M, acc8);
            } else {
                if (tile != rows_tile) {
                    rows.set(tile_rows(args.N, tile), r0, r1, t, tile);
                    rows_tile = tile;
                }
                // W4A16: the quantisation group of the lane's sub-block in each window.
                int g0 = 0, g1 = 0;
                if (kFmt == DFMT_W4A16) {
                    const int kb = static_cast<int>(sb) * (Q4K_BLOCK / CHUNK_K) + (t >> 1);  // 64-wide block of window 0
                    g0 = (kb * CHUNK_K) / args.group;
                    g1 = ((kb + 2) * CHUNK_K) / args.group;
                }
                dec_window<0>(wst, xst, rows, xo, sh, g0, args, acc);
                dec_window<1>(wst, xst, rows, xo, sh, g1, args, acc);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty + 8 * s);
        }
        if (sb == nsb - 1 || st == n_items - 1) {
            if constexpr (kQ8) {
                // Lanes l and l ^ 16 hold the two halves of the same row.
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float mine = qhalf ? acc8[4 + e] : acc8[e], theirs_keep = qhalf ? acc8[e] : acc8[4 + e];
                    // Each lane sends the partner the tokens the partner keeps.
                    acc[e] = mine + __shfl_xor_sync(0xffffffffu, theirs_keep, 16);
                }
#pragma unroll
                for (int e = 0; e < DEC_TOKENS; ++e) acc8[e] = 0.f;
            }
            flush(tile);
            acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
        }
        if (++sb == nsb) {
            sb = 0;
            ++tile;
        }
        if (++s == NS) {
            s = 0;
            ph ^= 1u;
        }
    }
}

// ---------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn dec_encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

static int weight_stage_bytes(int fmt) {
    return fmt == DFMT_Q4K || fmt == DFMT_Q4K_Q8 ? TILE_ROWS * Q4K_BLOCK_BYTES
         : fmt == DFMT_Q6K ? TILE_ROWS * Q6K_BLOCK_BYTES
                           : TILE_ROWS * CHUNK_ROW_BYTES * 4;
}

struct DecLayout {
    int stage_stride, bar_off, smem;
};

template <int kFmt>
static DecLayout dec_layout() {
    DecLayout L;
    L.stage_stride = (DEC_X_BYTES + weight_stage_bytes(kFmt) + 1023) / 1024 * 1024;
    L.bar_off = dec_stages<kFmt>() * L.stage_stride;
    L.smem = L.bar_off + 24 * dec_stages<kFmt>() + 16 + 1024;  // + slack to align the base to 1 KiB
    return L;
}

// CTAs of the decode kernel resident at once on the current device.
template <int kFmt>
static int dec_slots(int *out) {
    static int cache[64];
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return QWP_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[dev]) {
        const DecLayout L = dec_layout<kFmt>();
        if (cudaFuncSetAttribute(qwp_decode_kernel<kFmt>, cudaFuncAttributeMaxDynamicSharedMemorySize, L.smem) !=
            cudaSuccess)
            return QWP_ERR_CUDA;
        int per_sm = 0, sms = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, qwp_decode_kernel<kFmt>, DEC_THREADS, L.smem) !=
                cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || per_sm < 1)
            return QWP_ERR_CUDA;
        cache[dev] = per_sm * sms;
    }
    *out = cache[dev];
    return QWP_OK;
}

template <int kFmt>
static int dec_grid(int64_t N, int64_t K, int64_t *grid) {
    int slots = 0;
    int rc = dec_slots<kFmt>(&slots);
    if (rc) return rc;
    const int64_t items = (N + TILE_ROWS - 1) / TILE_ROWS * (K / Q4K_BLOCK);
    *grid = std::max<int64_t>(1, std::min<int64_t>(items / DEC_MIN_ITEMS, slots));
    return QWP_OK;
}

template <int kFmt>
static int launch_decode_fmt(const void *w, const void *scales, const uint8_t *zeros, const void *x, bool x_bf16,
                             float *y, int64_t M, int64_t N, int64_t K, int64_t group, void *scratch,
                             size_t scratch_bytes, cudaStream_t stream) {
    int64_t G = 0;
    int rc = dec_grid<kFmt>(N, K, &G);
    if (rc) return rc;
    if ((N + TILE_ROWS - 1) / TILE_ROWS * (K / Q4K_BLOCK) * G >= (int64_t(1) << 32)) return QWP_ERR_UNSUPPORTED_SHAPE;
    uint32_t *status = status_word();
    if (!status) return QWP_ERR_CUDA;
    const int64_t row_tiles = (N + TILE_ROWS - 1) / TILE_ROWS;
    const size_t part_bytes = static_cast<size_t>(G) * 2 * DEC_PART_FLOATS * sizeof(float);
    if (scratch_bytes < part_bytes + static_cast<size_t>(row_tiles) * 4) return QWP_ERR_SCRATCH_LIMIT;
    uint32_t *count = reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(scratch) + part_bytes);
    if (cudaMemsetAsync(count, 0, static_cast<size_t>(row_tiles) * 4, stream) != cudaSuccess) {
        cudaGetLastError();
        return QWP_ERR_CUDA;
    }

    CUtensorMap map;
    memset(&map, 0, sizeof(map));  // unused by the quantized-activation product (x comes by bulk copy)
    if (kFmt != DFMT_Q4K_Q8) {
        EncodeTiledFn fn = dec_encode_fn();
        if (!fn) return QWP_ERR_CUDA;
        cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
        cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
        cuuint32_t box[2] = {64, DEC_TOKENS};
        cuuint32_t estr[2] = {1, 1};
        if (fn(&map, x_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
               const_cast<void *>(x), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return QWP_ERR_CUDA;
    }

    const DecLayout L = dec_layout<kFmt>();
    DecodeArgs a;
    a.w = static_cast<const uint8_t *>(w);
    a.scales = static_cast<const __half *>(scales);
    a.zeros = zeros;
    a.xq = kFmt == DFMT_Q4K_Q8 ? static_cast<const uint8_t *>(x) : nullptr;
    a.y = y;
    a.status = status;
    a.part = static_cast<float *>(scratch);
    a.count = count;
    a.items = row_tiles * (K / Q4K_BLOCK);
    a.M = static_cast<int>(M);
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    a.group = static_cast<int>(group > 0 ? group : 1);
    a.groups_per_row = group > 0 ? static_cast<int>(K / group) : 0;
    a.nsb = static_cast<int>(K / Q4K_BLOCK);
    a.stage_stride = L.stage_stride;
    a.bar_off = L.bar_off;
    a.x_bf16 = x_bf16 && kFmt != DFMT_Q4K_Q8 ? 1 : 0;
    a.timeout_ns = kDefaultTimeoutNs;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(G), 1, 1);
    cfg.blockDim = dim3(DEC_THREADS, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(L.smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, qwp_decode_kernel<kFmt>, map, a) != cudaSuccess) {
        cudaGetLastError();
        return QWP_ERR_CUDA;
    }
    return QWP_OK;
}

template <int kFmt>
static size_t scratch_need(int64_t N, int64_t K) {
    int64_t G = 0;
    if (dec_grid<kFmt>(N, K, &G)) return 0;
    const int64_t row_tiles = (N + TILE_ROWS - 1) / TILE_ROWS;
    return static_cast<size_t>(G) * 2 * DEC_PART_FLOATS * sizeof(float) + static_cast<size_t>(row_tiles) * 4;
}

size_t decode_scratch_bytes(int fmt, int64_t N, int64_t K) {
    switch (fmt) {
        case DFMT_Q4K: return scratch_need<DFMT_Q4K>(N, K);
        case DFMT_Q6K: return scratch_need<DFMT_Q6K>(N, K);
        case DFMT_W4A16: return scratch_need<DFMT_W4A16>(N, K);
        case DFMT_Q4K_Q8: return scratch_need<DFMT_Q4K_Q8>(N, K);
        default: return 0;
    }
}

int launch_decode(int fmt, const void *w, const void *scales, const uint8_t *zeros, const void *x, bool x_bf16,
                  float *y, int64_t M, int64_t N, int64_t K, int64_t group, void *scratch, size_t scratch_bytes,
                  cudaStream_t stream) {
    if (M < 1 || M > DEC_TOKENS || K % Q4K_BLOCK) return QWP_ERR_UNSUPPORTED_SHAPE;
    if (!scratch) return QWP_ERR_INVALID_ARG;
    switch (fmt) {
        case DFMT_Q4K:
            return launch_decode_fmt<DFMT_Q4K>(w, scales, zeros, x, x_bf16, y, M, N, K, group, scratch, scratch_bytes,
                                               stream);
        case DFMT_Q6K:
            return launch_decode_fmt<DFMT_Q6K>(w, scales, zeros, x, x_bf16, y, M, N, K, group, scratch, scratch_bytes,
                                               stream);
        case DFMT_W4A16:
            return launch_decode_fmt<DFMT_W4A16>(w, scales, zeros, x, x_bf16, y, M, N, K, group, scratch,
                                                 scratch_bytes, stream);
        case DFMT_Q4K_Q8:
            return launch_decode_fmt<DFMT_Q4K_Q8>(w, scales, zeros, x, false, y, M, N, K, group, scratch,
                                                  scratch_bytes, stream);
        default: return QWP_ERR_INVALID_ARG;
    }
}

static std::atomic<int> g_decode_policy{DECODE_POLICY_AUTO};

int decode_policy() { return g_decode_policy.load(std::memory_order_relaxed); }

bool decode_selected(int fmt, int64_t M, int64_t N, int64_t K) {
    switch (decode_policy()) {
        case DECODE_POLICY_NEVER: return false;
        case DECODE_POLICY_ALWAYS: return decode_fits(M, N, K);
        default: return decode_auto(fmt, M, N, K);
    }
}

}  // namespace qwp

extern "C" int qwp_set_decode_policy(int policy) {
    if (policy != qwp::DECODE_POLICY_AUTO && policy != qwp::DECODE_POLICY_NEVER && policy != qwp::DECODE_POLICY_ALWAYS)
        return QWP_ERR_INVALID_ARG;
    return qwp::g_decode_policy.exchange(policy, std::memory_order_relaxed);
}

extern "C" int qwp_decode_selected(int format, int64_t M, int64_t N, int64_t K) {
    if (format != qwp::DFMT_W4A16 && format != qwp::DFMT_Q4K && format != qwp::DFMT_Q6K) return QWP_ERR_INVALID_ARG;
    return qwp::decode_selected(format, M, N, K) ? 1 : 0;
}
