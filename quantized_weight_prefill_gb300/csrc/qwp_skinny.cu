// The skinny-N GEMM: y[M,N] = x[M,K] . W[N,K]^T for Q4_K weights with few rows
// (N <= 64) and many tokens.  sparkinfer PR #511, Summary table, row "Skinny
// bf16 GEMM prefill_gemm_skinny.cu": a product with a 32-wide output run on a
// 128 x 128 tile wastes three quarters of it and leaves most SMs idle.  Here the
// activations are the stream that matters (M*K*2 bytes against N*K*0.5625 of
// weights), so the roles of the general kernel are turned around:
//   * tokens are the MMA's M side: an x tile of up to 128 tokens (one 64-wide K
//     block) is the A operand, loaded by TMA into shared memory (128-byte
//     swizzle) and given to the tensor core as it is, bf16 or fp16: every
//     activation is read once, by the one CTA that uses it, and never converted.
//     The tile height is chosen per launch so that the grid fills the GPU in
//     whole waves (the MMA still covers 128 rows; rows past the tile are not
//     loaded and their results are never stored);
//   * the weights are the B operand (N padded to 16..64 rows): the packed Q4_K
//     stages are bulk-copied into shared memory and unpacked by the transform
//     warps into a ring of swizzled K-major tiles.  For fp16 x that is one fp16
//     tile per 64-wide K block, the single-rounding operand of the general
//     kernel.  For bf16 x (kind::f16 wants A and B of one type) it is two bf16
//     tiles, hi and lo, whose sum carries the weight to about 16 significant
//     bits, stacked as one operand of 2N rows: one MMA per K step (its time is
//     set by the 128 token rows, not by N at these widths) accumulates x.hi and
//     x.lo side by side, and the epilogue adds the two;
//   * the fp32 accumulator D[128 tokens x N (2N)] lives in tensor memory;
//   * K is split S ways across a thread-block cluster (grid S x token tiles, S a
//     power of two dividing the 256-wide stages); each CTA writes its partial
//     tile into its own (idle) x ring, and after a cluster barrier each rank sums
//     a 1/S slice of the tile's rows over the ranks, in rank order (deterministic), reading
//     its peers' shared memory, and writes y; a second cluster barrier keeps
//     every CTA alive until its peers have read it.
// One launch, no device memory of its own.  Roles:
//   warp 0        x producer (one thread, TMA)
//   warp 1        tensor-memory allocation; MMA issue (one elected lane)
//   warp 2        weight producer (one thread, bulk copies)
//   warps 3..10   weight transform (half a K block of 32 rows each); then warps
//                 3..6 drain the accumulator (one per tensor-memory lane
//                 quarter); with S > 1 every warp helps sum the slices
// Every mbarrier wait is bounded (qwp_sync.cuh); on expiry the CTA records the
// timeout, waits for its own copies and MMAs in flight, passes the cluster
// barriers, releases its tensor memory and exits.
#include <algorithm>
#include <mutex>

#include "qwp_decode.h"
#include "qwp_format.cuh"
#include "qwp_internal.h"
#include "qwp_ptx.cuh"
#include "qwp_sync.cuh"

namespace qwp {
namespace {

constexpr int SK_TOKENS = 128;                 // MMA M: the most tokens per CTA
constexpr int SK_MAX_N = 64;                   // weight rows (MMA N, padded to 16)
constexpr int SK_MAX_XS = 8;                   // x ring: one 64-wide K block per slot
constexpr int SK_X_PRE = 2;                    // x tiles requested before the block-wide barrier
constexpr int SK_MIN_XS = 3;
// An x slot: tm rows of 64 16-bit values (128 bytes), in whole 1 KiB swizzle atoms.
__host__ __device__ constexpr int sk_x_slot(int tm) { return (tm * 128 + 1023) & ~1023; }
constexpr int SK_W_SLOT = SK_MAX_N * Q4K_BLOCK_BYTES;
constexpr int SK_SHORT_STAGES = 4;             // K range of a "short" CTA, in 256-wide stages
// B ring (one 256-wide stage per slot) and packed-weight ring depths: two each,
// or, for a CTA whose K range is at most SK_SHORT_STAGES stages, all of them.
__host__ __device__ constexpr int sk_rings(bool short_k) { return short_k ? SK_SHORT_STAGES : 2; }
constexpr int SK_MAX_RING = SK_SHORT_STAGES;
constexpr int SK_NUM_BARS = 2 * SK_MAX_XS + 4 * SK_MAX_RING + 2;
constexpr int SK_SMEM = 227 * 1024;            // requested; the layout below fits inside
constexpr int SK_XFORM0 = 3, SK_NXFORM = 8;    // transform warps; the first four also drain the accumulator
constexpr int SK_THREADS = 32 * (SK_XFORM0 + SK_NXFORM);
constexpr uint32_t SK_TMEM_COLS = 2 * SK_MAX_N;  // bf16 x: the hi and the lo sums

// The shared-memory layout (offsets from the 1 KiB-aligned base): the x ring of
// `xs` slots of x_slot bytes (as many as fit, up to SK_MAX_XS), the B ring (a
// slot is one 256-wide stage: 4 blocks of n_pad rows x 128 bytes, for bf16 x of
// 2 n_pad rows: the hi rows, then the lo rows), the
// packed weight ring, the barriers and two words (tensor-memory base, abort flag).
struct SkLayout {
    int xs, b_slot, w_slot, off_b, off_w, off_bar, off_misc;
};
__host__ __device__ constexpr SkLayout sk_layout(int n_pad, bool bf16, int rows, bool short_k, int x_slot) {
    SkLayout l{};
    l.b_slot = (bf16 ? 2 : 1) * 4 * n_pad * 128;
    l.w_slot = short_k ? (rows * Q4K_BLOCK_BYTES + 15) & ~15 : SK_W_SLOT;
    const int R = sk_rings(short_k);
    const int rest = R * l.b_slot + R * l.w_slot + 8 * SK_NUM_BARS + 16 + 1024;  // + base alignment slack
    l.xs = (SK_SMEM - rest) / x_slot;
    if (l.xs > SK_MAX_XS) l.xs = SK_MAX_XS;
    l.off_b = l.xs * x_slot;
    l.off_w = l.off_b + R * l.b_slot;
    l.off_bar = l.off_w + R * l.w_slot;
    l.off_misc = l.off_bar + 8 * SK_NUM_BARS;
    return l;
}
static_assert(sk_layout(SK_MAX_N, true, SK_MAX_N, false, sk_x_slot(SK_TOKENS)).xs >= SK_MIN_XS,
              "the x ring keeps at least three slots");
static_assert(sk_layout(SK_MAX_N, true, SK_MAX_N, false, sk_x_slot(SK_TOKENS)).off_misc + 16 + 1024 <= SK_SMEM,
              "shared memory budget");
static_assert(sk_layout(SK_MAX_N, true, SK_MAX_N, false, sk_x_slot(1)).off_misc + 16 + 1024 <= SK_SMEM,
              "shared memory budget (smallest slots, SK_MAX_XS of them)");
// Whether a launch takes the short-K rings: its CTAs' K range is at most
// SK_SHORT_STAGES stages and the layout still leaves four x slots.
__host__ __device__ constexpr bool sk_short(int n_pad, bool bf16, int rows, int stages, int x_slot) {
    return stages <= SK_SHORT_STAGES && sk_layout(n_pad, bf16, rows, true, x_slot).xs >= 4;
}
static_assert(SK_SMEM <= 232448, "opt-in shared memory per CTA");
// The partial tile of one CTA overlays its x ring: [tm tokens][n_pad + 4] fp32
// (the 4 extra floats per row spread the rows over the banks), within the
// first SK_MIN_XS slots of at least tm * 128 bytes each.
static_assert((SK_MAX_N + 4) * 4 <= SK_MIN_XS * 128, "partial tile fits the x ring");

struct SkinnyArgs {
    const uint8_t *w;     // repacked Q4_K (one tile of R = N rows)
    float *y;             // [M][N]
    uint32_t *status;
    int M, N, K;
    int n_pad;            // N rounded up to 16
    int tm;               // tokens per CTA (token tile height, 1..SK_TOKENS)
    int splits;           // S (cluster size along x)
    int stages;           // 256-wide stages per CTA (K / 256 / S)
    int x_bf16;           // 1: x and the weight operands are bf16 (hi + lo), else fp16
    uint64_t timeout_cycles, drain_cycles;
};

enum : uint32_t { SW_X_EMPTY = 1, SW_X_FULL, SW_W_EMPTY, SW_W_FULL, SW_B_EMPTY, SW_B_FULL, SW_ACC, SW_DRAIN };

// Byte offset of 16-byte chunk c (0..7) of row r in a K-major, 128-byte swizzled
// operand tile (8-row atoms of 1 KiB; chunk c of row r sits at c ^ (r % 8)).
__device__ __forceinline__ uint32_t sw128_offset(int r, int c) {
    return static_cast<uint32_t>((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

// kShort: the rings of sk_rings(true) (see sk_short); compiled apart, so that the
// ring indexing stays constant in both (with run-time depths the longer shapes
// measured 2-5% slower).
template <bool kShort>
__global__ void __launch_bounds__(SK_THREADS, 1)
    qwp_skinny_kernel(const __grid_constant__ CUtensorMap tmap_x, const SkinnyArgs args) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const uint32_t warp = warp_id(), lane = lane_id();
    const bool bf16 = args.x_bf16 != 0;
    const int tm = args.tm;
    const int x_slot = sk_x_slot(tm);
    const SkLayout L = sk_layout(args.n_pad, bf16, args.N, kShort, x_slot);
    constexpr int BS = sk_rings(kShort), WS = sk_rings(kShort);
    const int XS = L.xs;
    const int S = args.splits;
    const int rank = static_cast<int>(blockIdx.x);  // cluster rank along K
    const int m0 = static_cast<int>(blockIdx.y) * tm;
    const int st0 = rank * args.stages;              // first 256-wide stage of this CTA
    const int nblk = 4 * args.stages;                // 64-wide K blocks of this CTA
    const int R = args.N;                            // weight rows (one tile)
    const uint32_t b_tile = static_cast<uint32_t>(args.n_pad) * 128u;  // n_pad rows of B (hi, lo, or fp16)
    const uint32_t b_blk = (bf16 ? 2u : 1u) * b_tile;                     // one 64-wide K block of B

    const uint32_t bar0 = smem_u32(smem + L.off_bar);
    const uint32_t x_full = bar0, x_empty = x_full + 8 * SK_MAX_XS;
    const uint32_t w_full = x_empty + 8 * SK_MAX_XS, w_empty = w_full + 8 * SK_MAX_RING;
    const uint32_t b_full = w_empty + 8 * SK_MAX_RING, b_empty = b_full + 8 * SK_MAX_RING;
    const uint32_t acc_full = b_empty + 8 * SK_MAX_RING, drain = acc_full + 8;
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + L.off_misc);  // [0] tensor memory, [1] abort
    const Ctl ctl{misc + 1, args.status, args.timeout_cycles, args.drain_cycles};
    const int x_pre = min(min(XS, SK_X_PRE), nblk), w_pre = min(WS, args.stages);  // copies started at set-up
    const uint32_t w_bytes = static_cast<uint32_t>(R) * Q4K_BLOCK_BYTES;
    const uint32_t x_bytes = static_cast<uint32_t>(tm) * 128u;  // one TMA box: tm rows of 64 values

    pdl_launch_dependents();
    if (threadIdx.x == 0) {
        for (int s = 0; s < XS; ++s) {
            mbar_init(x_full + 8 * s, 1);
            mbar_init(x_empty + 8 * s, 1);
        }
        for (int s = 0; s < WS; ++s) {
            mbar_init(w_full + 8 * s, 1);
            mbar_init(w_empty + 8 * s, SK_NXFORM);
        }
        for (int s = 0; s < BS; ++s) {
            mbar_init(b_full + 8 * s, SK_NXFORM);
            mbar_init(b_empty + 8 * s, 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(drain, 1);
        fence_mbar_init();
        prefetch_tensormap(&tmap_x);
        // x, the weights and the status word may come from the grids launched just
        // before; every other thread is ordered after this wait by the barrier below.
        pdl_wait();
        // A failure recorded earlier (and not yet read) makes this launch skip its
        // work; the copies below are still waited for.  The status load is issued
        // first and its value used only after the copies are issued, so that its
        // latency (about 1 us once every CTA's copies are queued) overlaps theirs.
        const uint32_t status_now = *reinterpret_cast<volatile uint32_t *>(args.status);
        // The first weight stages and x tiles start before the block-wide barrier
        // (their slots are empty); this thread is also the x producer.  Weights
        // first: their transform stands between the first x tile and its MMAs.
        // At most SK_X_PRE x tiles here (more, issued one by one before the
        // barrier, delayed every role: 1 us at M=4096, N=32, K=4096).
        for (int i = 0; i < w_pre; ++i) {
            mbar_arrive_expect_tx(w_full + 8 * i, w_bytes);
            bulk_copy_g2s(smem_u32(smem + L.off_w + i * L.w_slot), args.w + q4k_group_offset(args.K, 0, R, st0 + i),
                          w_bytes, w_full + 8 * i);
        }
        for (int j = 0; j < x_pre; ++j) {
            mbar_arrive_expect_tx(x_full + 8 * j, x_bytes);
            tma_load_2d(smem_u32(smem + j * x_slot), &tmap_x, (4 * st0 + j) * CHUNK_K, m0, x_full + 8 * j);
        }
        misc[1] = (status_now & kStatusTimeoutMask) ? 1u : 0u;
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(misc), SK_TMEM_COLS);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    const bool skip = misc[1] != 0;
    bool acc_ok = false;  // epilogue warps: the accumulator is complete

    if (warp == 0) {
        // ------------------------------------------------------------ x producer
        if (lane == 0 && skip)
            for (int j = 0; j < x_pre; ++j) wait_bar(x_full + 8 * j, 0, ctl, SW_DRAIN, false);
        if (lane == 0 && !skip) {
            int j = x_pre, xs = x_pre % XS;
            uint32_t ph = x_pre == XS ? 1u : 0u;  // the pass over the ring that block j starts
            for (; j < nblk; ++j) {
                if (j >= XS && !wait_bar(x_empty + 8 * xs, ph ^ 1, ctl, SW_X_EMPTY)) break;
                mbar_arrive_expect_tx(x_full + 8 * xs, x_bytes);
                tma_load_2d(smem_u32(smem + xs * x_slot), &tmap_x, (4 * st0 + j) * CHUNK_K, m0, x_full + 8 * xs);
                if (++xs == XS) {
                    xs = 0;
                    ph ^= 1;
                }
            }
            for (int g = max(0, j - XS); g < j; ++g)  // every copy issued lands before the CTA exits
                wait_bar(x_full + 8 * (g % XS), (g / XS) & 1, ctl, SW_DRAIN, false);
        }
    } else if (warp == 2) {
        // ------------------------------------------------------------ weight producer
        if (lane == 0 && skip)
            for (int i = 0; i < w_pre; ++i) wait_bar(w_full + 8 * i, 0, ctl, SW_DRAIN, false);
        if (lane == 0 && !skip) {
            int i = w_pre;
            for (; i < args.stages; ++i) {
                const int ws = i % WS;
                if (i >= WS && !wait_bar(w_empty + 8 * ws, ((i / WS) & 1) ^ 1, ctl, SW_W_EMPTY)) break;
                mbar_arrive_expect_tx(w_full + 8 * ws, w_bytes);
                bulk_copy_g2s(smem_u32(smem + L.off_w + ws * L.w_slot), args.w + q4k_group_offset(args.K, 0, R, st0 + i),
                              w_bytes, w_full + 8 * ws);
            }
            for (int g = max(0, i - WS); g < i; ++g)
                wait_bar(w_full + 8 * (g % WS), (g / WS) & 1, ctl, SW_DRAIN, false);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // Per 64-wide K block: 4 K steps of 16; both operands advance 32 bytes (2
        // descriptor units) per step.  bf16 x: the B operand is the hi and the lo
        // rows together (MMA N = 2 n_pad).
        if (!skip) {
            const uint32_t idesc =
                make_idesc_f16(bf16, SK_TOKENS, static_cast<uint32_t>((bf16 ? 2 : 1) * args.n_pad));
            bool ok = true;
            int xs = 0;
            uint32_t xph = 0;
            for (int i = 0; ok && i < args.stages; ++i) {
                const int bs = i % BS;
                if (!(ok = __all_sync(0xffffffffu, wait_bar(b_full + 8 * bs, (i / BS) & 1, ctl, SW_B_FULL)))) break;
                for (int blk = 0; blk < 4; ++blk) {
                    if (!(ok = __all_sync(0xffffffffu, wait_bar(x_full + 8 * xs, xph, ctl, SW_X_FULL)))) break;
                    tc_fence_after();
                    const uint64_t a_desc = smem_desc_sw128(smem_u32(smem + xs * x_slot));
                    const uint64_t b_desc =
                        smem_desc_sw128(smem_u32(smem + L.off_b + bs * L.b_slot) + blk * b_blk);
                    if (elect_one()) {
                        if (i == 0 && blk == 0)
                            mma_ss<false>(tmem, a_desc, b_desc, idesc);
                        else
                            mma_ss<true>(tmem, a_desc, b_desc, idesc);
#pragma unroll
                        for (int kk = 1; kk < 4; ++kk) mma_ss<true>(tmem, a_desc + 2u * kk, b_desc + 2u * kk, idesc);
                        mma_commit(x_empty + 8 * xs);
                    }
                    __syncwarp();
                    if (++xs == XS) {
                        xs = 0;
                        xph ^= 1;
                    }
                }
                if (ok && elect_one()) mma_commit(b_empty + 8 * bs);
                __syncwarp();
            }
            if (ok && elect_one()) mma_commit(acc_full);
            __syncwarp();
            if (!ok && lane == 0) {
                mma_commit(drain);
                wait_bar(drain, 0, ctl, SW_DRAIN, false);
            }
            __syncwarp();
        }
    } else {
        // ------------------------------------------------------------ weight transform
        // Per stage: the row groups g (32 rows each, ceil(n_pad/32) of them) x the 4
        // K blocks x their two 32-wide sub-blocks are shared out over the 8 warps;
        // lane = row within its group.  Rows R..n_pad-1 are written as zeros.
        // (Eight warps on half blocks rather than four on whole ones: 1-4% faster
        // where the weight side is widest, N = 64 or K = 12288.)
        const int xw = static_cast<int>(warp) - SK_XFORM0;
        const int groups = (args.n_pad + 31) / 32;
        bool ok = !skip;
        for (int i = 0; ok && i < args.stages; ++i) {
            const int ws = i % WS, bs = i % BS;
            if (!(ok = __all_sync(0xffffffffu, wait_bar(w_full + 8 * ws, (i / WS) & 1, ctl, SW_W_FULL)))) break;
            if (i >= BS &&
                !(ok = __all_sync(0xffffffffu, wait_bar(b_empty + 8 * bs, ((i / BS) & 1) ^ 1, ctl, SW_B_EMPTY))))
                break;
            const uint8_t *wst = smem + L.off_w + ws * L.w_slot;
            uint8_t *bst = smem + L.off_b + bs * L.b_slot;
            for (int pr = xw; pr < 8 * groups; pr += SK_NXFORM) {
                const int g = pr >> 3, blk = (pr >> 1) & 3, half = pr & 1;
                const int row = 32 * g + static_cast<int>(lane);
                if (row >= args.n_pad) continue;
                uint4 hdr = make_uint4(0, 0, 0, 0), wv = hdr;
                if (row < R) {
                    hdr = *reinterpret_cast<const uint4 *>(wst + Q4K_HEADER_BYTES * row);
                    const uint8_t *cp = wst + Q4K_HEADER_BYTES * R + CHUNK_ROW_BYTES * R * blk + row * 16;
                    wv = *reinterpret_cast<const uint4 *>(cp + 16 * R * half);
                }
                const Q4kSubH k = q4k_sub_f16(hdr, 2 * blk + half);
                const uint32_t w[4] = {wv.x, wv.y, wv.z, wv.w};
                uint8_t *bt = bst + blk * b_blk;
                if (bf16) {
                    uint8_t *lt = bt + b_tile;  // row n_pad + r: the swizzle of row r (n_pad % 8 == 0)
#pragma unroll
                    for (int u = 0; u < 4; ++u) {  // word v holds elements 8v..8v+7: 16-byte chunk v of the row
                        const int v = 4 * half + u;
                        uint32_t h[4], l[4];
                        q4k_word_bf16_hilo(w[u], k, h, l);
                        const uint32_t off = sw128_offset(row, v);
                        *reinterpret_cast<uint4 *>(bt + off) = make_uint4(h[0], h[1], h[2], h[3]);
                        *reinterpret_cast<uint4 *>(lt + off) = make_uint4(l[0], l[1], l[2], l[3]);
                    }
                } else {
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int v = 4 * half + u;
                        uint32_t p[4];
                        q4k_word_f16x2(w[u], k, p);
                        *reinterpret_cast<uint4 *>(bt + sw128_offset(row, v)) = make_uint4(p[0], p[1], p[2], p[3]);
                    }
                }
            }
            fence_proxy_async_smem();  // the B tiles are read by the tensor core
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(w_empty + 8 * ws);
                mbar_arrive(b_full + 8 * bs);
            }
        }
        // ------------------------------------------------------------ epilogue (accumulator)
        acc_ok = ok && __all_sync(0xffffffffu, wait_bar(acc_full, 0, ctl, SW_ACC));
        if (acc_ok) tc_fence_after();
    }

    // The accumulator: warps 3..6 (lane quarters 3, 0, 1, 2) hold rows 32q ..
    // 32q+31 of the MMA's 128, n_pad columns each (bf16 x: the hi sums, then
    // n_pad columns of lo sums, added here); rows from tm on are not the tile's
    // and are dropped.  S == 1: straight to y.  S > 1: into this CTA's x ring,
    // [row][n_pad + 4], for the cluster's reduction (every x tile has been
    // consumed once the accumulator is complete).
    const int pstride = args.n_pad + 4;
    float *pbuf = reinterpret_cast<float *>(smem);
    if (warp >= SK_XFORM0 && warp < SK_XFORM0 + 4) {
        const uint32_t q = warp & 3;
        const int row = static_cast<int>(q * 32 + lane), m = m0 + row;
        if (acc_ok) {
            for (int c0 = 0; c0 < args.n_pad; c0 += 16) {
                uint32_t v[16];
                tmem_ld_x16(tmem + ((q * 32u) << 16) + static_cast<uint32_t>(c0), v);
                if (bf16) {
                    uint32_t u[16];
                    tmem_ld_x16(tmem + ((q * 32u) << 16) + static_cast<uint32_t>(args.n_pad + c0), u);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) + __uint_as_float(u[e]));
                } else {
                    tmem_wait_ld();
                }
                if (S == 1) {
                    if (row < tm && m < args.M) {
                        float *yr = args.y + static_cast<int64_t>(m) * args.N + c0;
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            if (c0 + e < args.N) yr[e] = __uint_as_float(v[e]);
                    }
                } else if (row < tm) {
#pragma unroll
                    for (int e = 0; e < 16; e += 4)
                        *reinterpret_cast<float4 *>(pbuf + row * pstride + c0 + e) =
                            make_float4(__uint_as_float(v[e]), __uint_as_float(v[e + 1]), __uint_as_float(v[e + 2]),
                                        __uint_as_float(v[e + 3]));
                }
            }
        }
        tc_fence_before();
    }
    if (S > 1) {
        // Every rank's partial tile is in its shared memory (or the rank failed and
        // the status word says so); rank r sums rows [r*rows, (r+1)*rows) of the
        // tile (rows = ceil(tm/S) <= 128/S) over the ranks in rank order and writes them.  The second barrier keeps each CTA's
        // shared memory alive until its peers have read it: a thread arrives after
        // its sums (which consumed every value it loaded from a peer) are stored, so
        // it needs no release, and not waiting for the y stores to complete keeps
        // them off the barrier's path.
        __syncwarp();
        cluster_sync();
        if (!skip && !aborted(ctl)) {
            const int rows = (tm + S - 1) / S, groups = args.n_pad / 4;
            const uint32_t local = smem_u32(pbuf);
            for (int it = static_cast<int>(threadIdx.x); it < rows * groups; it += SK_THREADS) {
                const int row = rank * rows + it / groups, c = 4 * (it % groups);
                if (row >= tm) break;  // rows grow with it
                const uint32_t off = static_cast<uint32_t>((row * pstride + c) * 4);
                float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int r2 = 0; r2 < S; ++r2) {
                    const float4 v = ld_shared_cluster_f4(map_shared_rank(local + off, static_cast<uint32_t>(r2)));
                    a.x += v.x;
                    a.y += v.y;
                    a.z += v.z;
                    a.w += v.w;
                }
                const int m = m0 + row;
                if (m < args.M) {
                    float *yr = args.y + static_cast<int64_t>(m) * args.N + c;
                    const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (c + e < args.N) yr[e] = av[e];
                }
            }
        }
        __syncwarp();
        cluster_arrive_relaxed();
        cluster_wait();
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, SK_TMEM_COLS);
    }
}

// ---------------------------------------------------------------- host side

typedef CUresult (*SkEncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                    const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                    CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static SkEncodeTiledFn sk_encode_fn() {
    static SkEncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<SkEncodeTiledFn>(p);
    });
    return fn;
}

// The SM count and the clusters of S = 1, 2, 4, 8 CTAs that can be resident at
// once (cached per device), and the kernel's shared-memory attribute.  (Clusters
// of 8 fill only 15 x 8 of GB300's 152 SMs at this footprint, clusters of 4 36 x
// 4: a grid of more clusters than that runs in two waves.)
static int sk_cluster_cache[64][9];
static int sk_device_sms(int &sms) {
    static int cache[64];
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return QWP_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return QWP_ERR_CUDA;
        if (cudaFuncSetAttribute(qwp_skinny_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, SK_SMEM) !=
                cudaSuccess ||
            cudaFuncSetAttribute(qwp_skinny_kernel<false>, cudaFuncAttributeNonPortableClusterSizeAllowed, 0) !=
                cudaSuccess ||
            cudaFuncSetAttribute(qwp_skinny_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, SK_SMEM) !=
                cudaSuccess ||
            cudaFuncSetAttribute(qwp_skinny_kernel<true>, cudaFuncAttributeNonPortableClusterSizeAllowed, 0) !=
                cudaSuccess)
            return QWP_ERR_CUDA;
        for (int S = 1; S <= 8; S *= 2) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(static_cast<unsigned>(S), 64, 1);
            cfg.blockDim = dim3(SK_THREADS, 1, 1);
            cfg.dynamicSmemBytes = SK_SMEM;
            cudaLaunchAttribute attr;
            attr.id = cudaLaunchAttributeClusterDimension;
            attr.val.clusterDim.x = static_cast<unsigned>(S);
            attr.val.clusterDim.y = 1;
            attr.val.clusterDim.z = 1;
            cfg.attrs = &attr;
            cfg.numAttrs = 1;
            int clusters = 0;
            if (cudaOccupancyMaxActiveClusters(&clusters, qwp_skinny_kernel<false>, &cfg) != cudaSuccess) {
                cudaGetLastError();
                clusters = n / S;  // the plain SM-count rule
            }
            sk_cluster_cache[dev][S] = clusters;
        }
        cache[dev] = n;
    }
    sms = cache[dev];
    return QWP_OK;
}

// Resident clusters of S CTAs on the current device (after sk_device_sms).
static int sk_cluster_slots(int S, int sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 || S < 1 || S > 8) return sms / (S < 1 ? 1 : S);
    const int c = sk_cluster_cache[dev][S];
    return c > 0 ? c : sms / S;
}

}  // namespace

bool skinny_selected(int fmt, int64_t M, int64_t N, int64_t K) {
    return fmt == DFMT_Q4K && N >= 1 && N <= SK_MAX_N && M >= SKINNY_MIN_TOKENS && K > 0 && K % Q4K_BLOCK == 0 &&
           M <= (int64_t(1) << 30);
}

// Launch plan: S CTAs per cluster along K (a power of two up to 8 dividing the
// 256-wide stages) and token tiles of tm <= 128 rows, cut so that the clusters run
// in whole waves of resident clusters.  Per CTA and 64-wide K block the time is
// the larger of its x stream (tm rows of 128 bytes) and a floor set by its MMAs
// (128 rows whatever tm is), plus a fixed cost per wave and one for the cluster
// reduction; the cheapest plan wins.  In units of the stream time of one
// 128-byte row at the full-GPU rate (~3 ns on GB300): the floor is 77 rows, a
// wave or a reduction ~2 us.  (Timed on GB300 at M = 1024 ... 32768, N = 32,
// K = 4096, this picks the fastest of the forced plans at every size.)
int skinny_plan(int64_t M, int64_t K, int sms, int &splits, int64_t &tiles, int &tm) {
    const int64_t nst = K / Q4K_BLOCK;
    int dummy = 0;
    if (sk_device_sms(dummy)) return QWP_ERR_CUDA;
    const int64_t mma_rows = 77, fixed = 625;
    double best = 1e300;
    splits = 0;
    for (int S = 1; S <= 8 && nst % S == 0; S *= 2) {
        const int64_t slots = sk_cluster_slots(S, sms);
        if (slots < 1) continue;
        const int64_t waves = (M + SK_TOKENS * slots - 1) / (SK_TOKENS * slots);
        const int64_t h = (M + waves * slots - 1) / (waves * slots);  // <= SK_TOKENS
        const int64_t blocks = 4 * (nst / S);
        const double cost = static_cast<double>(waves) * (blocks * std::max(h, mma_rows) + fixed) + (S > 1 ? fixed : 0);
        if (cost < best) {
            best = cost;
            splits = S;
            tm = static_cast<int>(h);
        }
    }
    if (splits == 0) return QWP_ERR_CUDA;
    tiles = (M + tm - 1) / tm;
    return tiles <= 65535 ? QWP_OK : QWP_ERR_UNSUPPORTED_SHAPE;
}

int launch_skinny(const void *w, const void *x, bool x_bf16, float *y, int64_t M, int64_t N, int64_t K,
                  cudaStream_t stream) {
    int rc = check_device();
    if (rc) return rc;
    uint32_t *status = status_word();
    if (!status) return QWP_ERR_CUDA;
    int sms = 0;
    if ((rc = sk_device_sms(sms))) return rc;
    int S = 1, tm = SK_TOKENS;
    int64_t tiles = 0;
    if ((rc = skinny_plan(M, K, sms, S, tiles, tm))) return rc;
    SkEncodeTiledFn fn = sk_encode_fn();
    if (!fn) return QWP_ERR_CUDA;
    CUtensorMap map;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(CHUNK_K), static_cast<cuuint32_t>(tm)};
    cuuint32_t estr[2] = {1, 1};
    if (fn(&map, x_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(x),
           dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return QWP_ERR_CUDA;
    SkinnyArgs a;
    a.w = static_cast<const uint8_t *>(w);
    a.y = y;
    a.status = status;
    a.M = static_cast<int>(M);
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    a.n_pad = static_cast<int>((N + 15) / 16 * 16);
    a.tm = tm;
    a.splits = S;
    a.stages = static_cast<int>(K / Q4K_BLOCK / S);
    a.x_bf16 = x_bf16 ? 1 : 0;
    a.timeout_cycles = ns_to_cycles(wait_timeout_ns());
    a.drain_cycles = ns_to_cycles(kDefaultTimeoutNs);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(S), static_cast<unsigned>(tiles), 1);
    cfg.blockDim = dim3(SK_THREADS, 1, 1);
    cfg.dynamicSmemBytes = SK_SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(S);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    const bool short_k = sk_short(a.n_pad, x_bf16, a.N, a.stages, sk_x_slot(tm));
    if (cudaLaunchKernelEx(&cfg, short_k ? qwp_skinny_kernel<true> : qwp_skinny_kernel<false>, map, a) !=
        cudaSuccess) {
        cudaGetLastError();
        return QWP_ERR_CUDA;
    }
    return QWP_OK;
}

}  // namespace qwp
