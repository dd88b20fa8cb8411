// Fused dequant-in-tile GEMM on the 5th-generation tensor cores (tcgen05).
//
// y[M,N] = x[M,K] . W[N,K]^T with W in 4-bit form.  Method: "The dequant
// scratch round-trip is ZINC's last RDNA4 prefill tax", sections "The two
// passes hiding inside one matmul" and "What the roofline says" -- every
// packed weight block is read from global memory once, unpacked on chip and
// consumed by the matmul tile; no 16-bit weight copy ever reaches DRAM.  Token
// batching follows "How ZINC's RDNA4 batched prefill went from 42 to 208
// tok/s", section "The two prefill paths": each weight row is applied to a
// whole chunk of prompt tokens per read.
//
// One CTA computes a 128-row (weights) x BN-token (BN <= 256) tile of y^T over
// a range of K:
//   warp 0        x producer: one thread issues a 2-D TMA load (128-byte
//                 swizzle) per 64-wide K block of x into the x ring;
//   warp 1        allocates tensor memory; one thread issues tcgen05.mma;
//   warp 2        weight producer: one bulk copy per 256-wide K stage of packed
//                 weights into the weight ring;
//   warps 3..18   transform: four groups of 4 warps; group g owns K block g of
//                 every weight stage (4 blocks of 64); warp (group g, quarter q)
//                 unpacks rows 32q..32q+31 (its tensor-memory lane quarter) of
//                 that block, 64 weights per thread, to fp16 and stores them with
//                 one tcgen05.st into the A ring in tensor memory; the same warps
//                 later drain the fp32 accumulator (tcgen05.ld) into y.
// Tensor memory (512 columns): accumulator [128 lanes x BN] at column 0, an
// 8-deep ring of A operand blocks (128 lanes x 64 K = 32 columns) at 256.
// The MMA is D[128 x BN] += A[128 x 16] (tensor memory) . B[BN x 16]^T (shared
// memory), so weights are the M side and tokens the N side: a tile reuses each
// unpacked weight for BN tokens.  When the grid would leave SMs idle, K is split
// across a thread-block cluster and the partial tiles are summed in rank order
// through distributed shared memory.
//
// Every mbarrier wait is bounded: on expiry the thread records a timeout in
// the library's status word and sets a CTA-wide abort flag; all roles then
// wait (bounded) for their own copies and MMAs in flight, the tensor memory is
// released and the CTA exits.
#include <algorithm>
#include <atomic>
#include <mutex>

#include "qwp_format.cuh"
#include "qwp_internal.h"
#include "qwp_ptx.cuh"

namespace qwp {

constexpr int XFORM_GROUPS = 4;                    // groups take K blocks in turn, one per weight stage
constexpr int NUM_XFORM_WARPS = 4 * XFORM_GROUPS;  // 4 warps (one per lane quarter) cover one K block
constexpr int FIRST_XFORM_WARP = 3;
constexpr int NUM_THREADS = 32 * (FIRST_XFORM_WARP + NUM_XFORM_WARPS);
constexpr int X_MAX_STAGES = 8;  // <= A_STAGES: the x ring reuses the mma_done ring (see below)
constexpr int W_MAX_STAGES = 8;
constexpr int A_STAGES = 8;
constexpr int BN_MAX = 256;
constexpr int KB_PER_STAGE = 4;  // 64-wide K blocks per weight stage
constexpr int MAX_SPLITS = 8;    // portable cluster size
constexpr uint32_t ACC_COL = 0;
constexpr uint32_t A_COL = 256;
constexpr uint32_t TMEM_COLS = 512;

// Shared memory: a ring region (x stages, then weight stages; reused for the
// split-K partial sums after the main loop), then the mbarriers and misc words.
constexpr int RING_BYTES = 224 * 1024;
constexpr int OFF_BAR = RING_BYTES;
constexpr int NUM_BARS = 2 * X_MAX_STAGES + 2 * W_MAX_STAGES + 2 * A_STAGES + 2;
constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + slack to align the base to 1 KiB
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(X_MAX_STAGES <= A_STAGES, "the x ring is released through the mma_done ring");
static_assert(A_STAGES % 4 == 0, "commit groups of up to 4 blocks tile the A ring");
static_assert(XFORM_GROUPS == KB_PER_STAGE, "each transform warp owns one K block of every weight stage");
static_assert(512 * (BN_MAX + MAX_SPLITS) <= RING_BYTES, "split-K partials must fit the ring region");

struct GemmArgs {
    const uint8_t *w;       // repacked weights
    const __half *scales;   // W4A16: [N][K/group]
    const uint8_t *zeros;   // W4A16: [N][K/group]
    float *y;               // [M][N]
    uint32_t *status;       // library status word
    int M, N, K, group;
    int bn;                 // token tile = MMA N (multiple of 16, <= 256)
    int kb_per_split;       // 64-wide K blocks per CTA along K (multiple of 4)
    int splits;             // CTAs along K = cluster size (1 = no reduction)
    int x_stages, w_stages; // x ring slots (one commit group of K blocks each), weight ring stages
    int groups_per_row;     // W4A16: K / group
    int kb_per_group;       // W4A16: group / 64
    int kbg_shift;          // log2(kb_per_group) when it is a power of two, else -1
    int x_stage_bytes, w_stage_bytes;
    int cb_shift;           // log2(CB), CB = K blocks per commit group (1, 2 or 4; divides every split's blocks)
    uint64_t timeout_ns;
};

// Status codes recorded on a timeout: which wait gave up.
enum : uint32_t {
    WAIT_W_EMPTY = 1, WAIT_X_EMPTY, WAIT_X_FULL, WAIT_A_FULL, WAIT_W_FULL, WAIT_A_EMPTY,
    WAIT_ACC_FULL, WAIT_DRAIN
};

struct Ctl {
    uint32_t *abort;  // shared-memory flag
    uint32_t *status;
    uint64_t timeout_ns;
};

// Bounded wait on phase `parity` of `bar`.  False if it timed out or the CTA is
// aborting (this CTA or, through the status word, any other); a timeout
// records `where` in the status word.  The loop mostly sits in try_wait (which
// suspends the thread in hardware); the clock and the global status word are
// looked at only every 64 polls.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Ctl &ctl,
                                         uint32_t where, bool honour_abort = true) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if (honour_abort && *reinterpret_cast<volatile uint32_t *>(ctl.abort)) return false;
        if ((it & 63u) == 0) {
            if (honour_abort && (*reinterpret_cast<volatile uint32_t *>(ctl.status) & kStatusTimeoutMask)) {
                *reinterpret_cast<volatile uint32_t *>(ctl.abort) = 1u;  // another CTA failed
                return false;
            }
            if (global_timer_ns() - t0 > ctl.timeout_ns) {
                *reinterpret_cast<volatile uint32_t *>(ctl.abort) = 1u;
                atomicCAS(ctl.status, 0u, 0x100u | where);
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool aborted(const Ctl &ctl) {
    return *reinterpret_cast<volatile uint32_t *>(ctl.abort) != 0;
}

// Unpack one row's half of a 64-wide K block (4 words = 32 weights) into 16
// packed fp16 pairs regs[off .. off+15] of the A operand.
template <bool kQ4K>
__device__ __forceinline__ void unpack_quarter(uint4 wv, const Q4kSubH &ks, __half2 mz, __half2 s2,
                                               uint32_t (&regs)[32], int off) {
    const uint32_t w[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t p[4];
        if (kQ4K)
            q4k_word_f16x2(w[i], ks, p);
        else
            w4_word_f16x2(w[i], mz, s2, p);
#pragma unroll
        for (int e = 0; e < 4; ++e) regs[off + 4 * i + e] = p[e];
    }
}

template <bool kQ4K>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    qwp_gemm_kernel(const __grid_constant__ CUtensorMap tmap_x, const GemmArgs args) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const uint32_t warp = warp_id();
    const uint32_t lane = lane_id();

    const int tile = blockIdx.x;
    const int R = tile_rows(args.N, tile);
    const int m0 = blockIdx.y * args.bn;
    const int nkb_total = args.K / CHUNK_K;
    const int kb_begin = blockIdx.z * args.kb_per_split;
    const int kb_end = min(nkb_total, kb_begin + args.kb_per_split);
    const int nkb = kb_end - kb_begin;
    const int nstage = (nkb + KB_PER_STAGE - 1) / KB_PER_STAGE;
    const int XS = args.x_stages, WS = args.w_stages;
    uint8_t *const x_ring = smem;
    uint8_t *const w_ring = smem + XS * args.x_stage_bytes;

    const uint32_t bar0 = smem_u32(smem + OFF_BAR);
    // The MMA issuer works in commit groups of CB = 2^cb_shift consecutive K blocks:
    // one x_full wait (the group's CB x tiles share one ring slot and barrier), one
    // a_full wait (every transform warp arrives once per group), 4*CB MMAs and one
    // tcgen05.commit.  A single thread issues every MMA of the CTA, and its fixed
    // cost per loop iteration (waits, fence, bookkeeping) is several hundred cycles
    // on a busy SM, so it is paid per group rather than per 64-wide block.
    // mma_done[(j % A_STAGES) >> cb_shift] completes when the MMAs of the group
    // holding block j (and all before it) are done; that releases the group's A
    // slots and its x slot (the x ring has at most A_STAGES / CB slots, so no phase
    // of mma_done is skipped).
    const int cbs = args.cb_shift;
    const int dslots = A_STAGES >> cbs;  // commit-group slots of the A ring
    const int ngroups = nkb >> cbs;      // nkb is a multiple of CB
    const uint32_t x_full = bar0, mma_done = x_full + 8 * X_MAX_STAGES;
    const uint32_t w_full = mma_done + 8 * X_MAX_STAGES, w_empty = w_full + 8 * W_MAX_STAGES;
    const uint32_t a_full = w_empty + 8 * W_MAX_STAGES, unused = a_full + 8 * A_STAGES;
    const uint32_t acc_full = unused + 8 * A_STAGES, drain = acc_full + 8;
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + OFF_MISC);  // [0] tmem base, [1] abort
    const Ctl ctl{misc + 1, args.status, args.timeout_ns};

    // Copy of weight stage s (K blocks 4s.. of this CTA's range) into ring slot ws.
    auto load_weight_stage = [&](int s, int ws) {
        const int kb0 = kb_begin + KB_PER_STAGE * s;
        const int nblk = min(KB_PER_STAGE, kb_end - kb0);
        const uint8_t *src;
        uint32_t bytes;
        if (kQ4K) {
            src = args.w + q4k_group_offset(args.K, tile, R, kb0 / KB_PER_STAGE);
            bytes = static_cast<uint32_t>(R) * Q4K_BLOCK_BYTES;
        } else {
            src = args.w + w4_plane_offset(args.K, tile, R, kb0);
            bytes = static_cast<uint32_t>(R) * CHUNK_ROW_BYTES * nblk;
        }
        mbar_arrive_expect_tx(w_full + 8 * ws, bytes);
        bulk_copy_g2s(smem_u32(w_ring + ws * args.w_stage_bytes), src, bytes, w_full + 8 * ws);
    };
    // The weight producer's thread sets up the barriers and starts the first weight
    // copies before the block-wide barrier (their slots are empty).
    const int w_pre = min(WS, nstage);
    if (threadIdx.x == 64) {
        for (int s = 0; s < X_MAX_STAGES; ++s) mbar_init(x_full + 8 * s, 1);
        for (int s = 0; s < A_STAGES; ++s) mbar_init(mma_done + 8 * s, 1);
        for (int s = 0; s < W_MAX_STAGES; ++s) {
            mbar_init(w_full + 8 * s, 1);
            mbar_init(w_empty + 8 * s, NUM_XFORM_WARPS);
        }
        // A commit group of CB <= XFORM_GROUPS blocks is stored by CB transform groups.
        for (int s = 0; s < A_STAGES; ++s)
            mbar_init(a_full + 8 * s, (NUM_XFORM_WARPS / XFORM_GROUPS) << cbs);
        mbar_init(acc_full, 1);
        mbar_init(drain, 1);
        // A failure recorded earlier (and not yet read by qwp_device_status) makes
        // every later launch skip its work instead of waiting out its own timeouts.
        const bool failed = (*reinterpret_cast<volatile uint32_t *>(args.status) & kStatusTimeoutMask) != 0;
        misc[1] = failed ? 1u : 0u;
        fence_mbar_init();
        prefetch_tensormap(&tmap_x);
        if (!failed)
            for (int s = 0; s < w_pre; ++s) load_weight_stage(s, s);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(misc), TMEM_COLS);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    const bool skip = misc[1] != 0;
    bool acc_ok = false;  // transform warps: the accumulator is complete

    if (warp == 0) {
        // ------------------------------------------------------------ x producer
        if (lane == 0 && !skip) {
            // x may be written by the grid launched just before this one (the
            // activation conversion); nothing else here depends on it.
            asm volatile("griddepcontrol.wait;" ::: "memory");
            int issued = 0;
            int xs = 0;         // ring slot (running counters: no division in the loop)
            int dk = 0;         // mma_done slot of group g - XS, and its phase
            uint32_t dph = 0;
            const uint32_t tile_bytes = static_cast<uint32_t>(args.bn) * 128u;
            for (int g = 0; g < ngroups; ++g) {
                if (g >= XS) {  // slot xs last held group g - XS
                    if (!wait_bar(mma_done + 8 * dk, dph, ctl, WAIT_X_EMPTY)) break;
                    if (++dk == dslots) { dk = 0; dph ^= 1; }
                }
                mbar_arrive_expect_tx(x_full + 8 * xs, tile_bytes << cbs);
                for (int c = 0; c < (1 << cbs); ++c)
                    tma_load_2d(smem_u32(x_ring + xs * args.x_stage_bytes + c * tile_bytes), &tmap_x,
                                (kb_begin + (g << cbs) + c) * CHUNK_K, m0, x_full + 8 * xs);
                issued = g + 1;
                if (++xs == XS) xs = 0;
            }
            // Every copy issued above lands before the CTA may exit.
            for (int g = max(0, issued - XS); g < issued; ++g)
                wait_bar(x_full + 8 * (g % XS), (g / XS) & 1, ctl, WAIT_DRAIN, false);
        }
    } else if (warp == 2) {
        // ------------------------------------------------------------ weight producer
        if (lane == 0 && !skip) {
            int issued = w_pre;  // stages 0 .. w_pre-1 went out before the block-wide barrier
            int ws = 0;
            uint32_t wph = 1;    // stage w_pre reuses slot 0 (second use: wait for its first release)
            for (int s = w_pre; s < nstage; ++s) {
                if (!wait_bar(w_empty + 8 * ws, wph ^ 1, ctl, WAIT_W_EMPTY)) break;
                load_weight_stage(s, ws);
                issued = s + 1;
                if (++ws == WS) { ws = 0; wph ^= 1; }
            }
            for (int s = max(0, issued - WS); s < issued; ++s)
                wait_bar(w_full + 8 * (s % WS), (s / WS) & 1, ctl, WAIT_DRAIN, false);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && !skip) {
            const uint32_t idesc = make_idesc_f16(false, TILE_ROWS, static_cast<uint32_t>(args.bn));  // fp16 A and B
            bool ok = true;
            int xs = 0, gs = 0;       // x ring slot; commit-group slot of the A ring
            uint32_t xph = 0, gph = 0;
            const uint32_t tile_desc = static_cast<uint32_t>(args.bn) * 128u >> 4;  // one x tile, in descriptor units
            for (int g = 0; g < ngroups; ++g) {
                ok = wait_bar(x_full + 8 * xs, xph, ctl, WAIT_X_FULL) &&
                     wait_bar(a_full + 8 * gs, gph, ctl, WAIT_A_FULL);
                if (!ok) break;
                tc_fence_after();
                uint64_t bdesc = smem_desc_sw128(smem_u32(x_ring + xs * args.x_stage_bytes));
                uint32_t acol = tmem + A_COL + (32u << cbs) * gs;
                for (int c = 0; c < (1 << cbs); ++c, bdesc += tile_desc, acol += 32u) {
#pragma unroll
                    for (int kk = 0; kk < CHUNK_K / 16; ++kk)
                        mma_ts(tmem + ACC_COL, acol + 8u * kk, bdesc + 2u * kk, idesc, (g | c | kk) != 0);
                }
                mma_commit(mma_done + 8 * gs);
                if (++xs == XS) { xs = 0; xph ^= 1; }
                if (++gs == dslots) { gs = 0; gph ^= 1; }
            }
            if (ok) {
                mma_commit(acc_full);
            } else {
                mma_commit(drain);
                wait_bar(drain, 0, ctl, WAIT_DRAIN, false);
            }
        }
    } else {
        // ------------------------------------------------------------ transform + epilogue
        const uint32_t xw = warp - FIRST_XFORM_WARP;
        const int grp = static_cast<int>(xw >> 2);   // this warp's K blocks: j % XFORM_GROUPS == grp
        const uint32_t quarter = warp & 3;            // tensor-memory lanes 32*quarter .. +31
        const int r = static_cast<int>(quarter * 32 + lane);
        const bool valid = r < R;
        const int64_t n = static_cast<int64_t>(tile) * TILE_ROWS + r;
        const uint32_t lane_base = (quarter * 32u) << 16;
        bool ok = !skip;
        int ws = -1;       // weight ring slot of this warp's current stage, and its phase
        uint32_t wph = 0;

        // Unpack K block j (the block of weight stage j / 4 that this warp owns) of
        // this thread's row into `regs`: 64 weights as 32 fp16 pairs.  Waits for the
        // stage and releases it after reading (the warp reads nothing else of it).
        auto prepare = [&](int j, uint32_t (&regs)[32]) -> bool {
            const int c = j & (KB_PER_STAGE - 1);
            if (++ws == WS) { ws = 0; wph ^= 1; }
            const uint8_t *wst = w_ring + ws * args.w_stage_bytes;
            // Every lane waits; the warp moves on together (tcgen05.st/ld are warp-collective).
            if (!__all_sync(0xffffffffu, wait_bar(w_full + 8 * ws, wph, ctl, WAIT_W_FULL))) return false;
            uint4 wv0 = make_uint4(0, 0, 0, 0), wv1 = make_uint4(0, 0, 0, 0);
            Q4kSubH k0, k1;
            __half2 s2 = __float2half2_rn(0.f), mz = w4_magic_zero(0);
            if (kQ4K) {
                uint4 hdr = make_uint4(0, 0, 0, 0);
                if (valid) {
                    hdr = *reinterpret_cast<const uint4 *>(wst + Q4K_HEADER_BYTES * r);
                    const uint8_t *cp = wst + Q4K_HEADER_BYTES * R + CHUNK_ROW_BYTES * R * c + r * 16;
                    wv0 = *reinterpret_cast<const uint4 *>(cp);
                    wv1 = *reinterpret_cast<const uint4 *>(cp + 16 * R);
                }
                k0 = q4k_sub_f16(hdr, 2 * c);
                k1 = q4k_sub_f16(hdr, 2 * c + 1);
            } else if (valid) {
                const uint8_t *cp = wst + CHUNK_ROW_BYTES * R * c + r * 16;
                wv0 = *reinterpret_cast<const uint4 *>(cp);
                wv1 = *reinterpret_cast<const uint4 *>(cp + 16 * R);
                const int64_t ng = args.groups_per_row;
                const int kbi = kb_begin + j;
                const int64_t g = args.kbg_shift >= 0 ? (kbi >> args.kbg_shift) : (kbi / args.kb_per_group);
                s2 = __half2half2(args.scales[n * ng + g]);
                mz = w4_magic_zero(args.zeros[n * ng + g]);
            }
            // This warp's reads of the stage are done.
            __syncwarp();
            if (lane == 0) mbar_arrive(w_empty + 8 * ws);
            unpack_quarter<kQ4K>(wv0, k0, mz, s2, regs, 0);
            unpack_quarter<kQ4K>(wv1, k1, mz, s2, regs, 16);
            return true;
        };
        // Store block j into its A ring slot once the MMAs of the block that last
        // used the slot (j - A_STAGES) are done.
        auto issue = [&](int j, const uint32_t (&regs)[32]) -> bool {
            const int as = j % A_STAGES;
            if (!__all_sync(0xffffffffu,
                            wait_bar(mma_done + 8 * (as >> cbs), ((j / A_STAGES) & 1) ^ 1, ctl, WAIT_A_EMPTY)))
                return false;
            tc_fence_after();
            tmem_st_x32(tmem + lane_base + A_COL + 32u * as, regs);
            return true;
        };
        // Block j's tensor-memory store lands; publish it to the MMA issuer.
        auto finish = [&](int j) {
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(a_full + 8 * ((j % A_STAGES) >> cbs));
        };

        // This warp's blocks are j = grp, grp + 4, ...: one per weight stage.  The
        // unpack of the next block overlaps the tensor-memory store of the current one.
        // (The first block is published before the next one is unpacked, so that the
        // MMAs can start as early as possible.)
        uint32_t regs[32];
        if (ok && grp < nkb) ok = prepare(grp, regs);
        for (int j = grp; ok && j < nkb; j += XFORM_GROUPS) {
            if (!(ok = issue(j, regs))) break;
            if (j == grp) finish(j);
            if (j + XFORM_GROUPS < nkb && !(ok = prepare(j + XFORM_GROUPS, regs))) break;
            if (j != grp) finish(j);
        }
        tmem_wait_st();  // no tensor-memory store may be in flight past this point
        __syncwarp();
        acc_ok = ok && __all_sync(0xffffffffu, wait_bar(acc_full, 0, ctl, WAIT_ACC_FULL));
        if (acc_ok && args.splits == 1) {
            tc_fence_after();
            for (int ci = grp; ci < args.bn / 16; ci += NUM_XFORM_WARPS / 4) {
                uint32_t v[16];
                tmem_ld_x16(tmem + lane_base + ACC_COL + 16u * ci, v);
                tmem_wait_ld();
                if (valid) {
                    const int mb = m0 + 16 * ci;
#pragma unroll
                    for (int t = 0; t < 16; ++t)
                        if (mb + t < args.M)
                            __stcs(args.y + static_cast<int64_t>(mb + t) * args.N + n, __uint_as_float(v[t]));
                }
            }
        }
        tc_fence_before();
    }

    __syncthreads();
    if (args.splits > 1) {
        // Deterministic split-K reduction through distributed shared memory.  CTA
        // `rank` of the cluster owns tokens [rank*per, rank*per + per) of the tile.
        // Once every CTA is past its main loop (its ring region is free), each CTA
        // pushes its partial accumulator for every token straight from tensor memory
        // into the owner's ring region, laid out [source rank][token][row]; after the
        // second cluster barrier each owner sums its tokens over the source ranks in
        // rank order and writes y.  Every CTA reaches both barriers whatever happened
        // above (all waits before them are bounded).
        const int S = args.splits;
        const uint32_t rank = cluster_ctarank();
        const int per = (args.bn + S - 1) / S;
        const uint32_t buf = smem_u32(smem);
        cluster_sync();
        if (acc_ok && !aborted(ctl)) {
            tc_fence_after();
            const uint32_t xw = warp - FIRST_XFORM_WARP;
            const uint32_t quarter = warp & 3;
            const int row = static_cast<int>(quarter * 32 + lane);
            const uint32_t lane_base = (quarter * 32u) << 16;
            for (int ci = static_cast<int>(xw >> 2); ci < args.bn / 16; ci += NUM_XFORM_WARPS / 4) {
                uint32_t v[16];
                tmem_ld_x16(tmem + lane_base + ACC_COL + 16u * ci, v);
                tmem_wait_ld();
                int owner = (16 * ci) / per, tt = 16 * ci - owner * per;
                uint32_t dst = map_shared_rank(buf, owner);
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                    st_shared_cluster_f32(dst + static_cast<uint32_t>(((static_cast<int>(rank) * per + tt) * TILE_ROWS + row) * 4),
                                          __uint_as_float(v[t]));
                    if (++tt == per && t < 15) {
                        tt = 0;
                        dst = map_shared_rank(buf, ++owner);
                    }
                }
            }
            tc_fence_before();
        }
        cluster_sync();
        const int t0 = min(args.bn, static_cast<int>(rank) * per);
        const int t1 = min(args.bn, t0 + per);
        if (!aborted(ctl)) {
            const float *part = reinterpret_cast<const float *>(smem);
            const int items = (t1 - t0) * (TILE_ROWS / 4);
            for (int it = threadIdx.x; it < items; it += NUM_THREADS) {
                const int tt = it / (TILE_ROWS / 4);
                const int r4 = 4 * (it % (TILE_ROWS / 4));
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int q = 0; q < S; ++q) {
                    const float4 v = *reinterpret_cast<const float4 *>(part + (q * per + tt) * TILE_ROWS + r4);
                    acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
                }
                const int m = m0 + t0 + tt;
                if (m < args.M) {
                    float *yr = args.y + static_cast<int64_t>(m) * args.N + static_cast<int64_t>(tile) * TILE_ROWS;
                    const float a4[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (r4 + e < R) __stcs(yr + r4 + e, a4[e]);
                }
            }
        }
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ---------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// x [M][K] 16-bit, box = 64 (K) x bn (rows), 128-byte swizzle, zero fill out of bounds.
static int encode_x_map(CUtensorMap *map, const void *x, int64_t M, int64_t K, int bn) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return QWP_ERR_CUDA;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(CHUNK_K), static_cast<cuuint32_t>(bn)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                    const_cast<void *>(x), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? QWP_OK : QWP_ERR_CUDA;
}

// Token tile: the fewest tiles of at most 256 tokens, each a multiple of 16.
static int choose_bn(int64_t M) {
    const int64_t tiles = (M + BN_MAX - 1) / BN_MAX;
    const int64_t per = (M + tiles - 1) / tiles;
    return static_cast<int>((per + 15) / 16 * 16);
}

struct DeviceInfo {
    int sms = 0;
    int slots[2][MAX_SPLITS + 1] = {};  // [kQ4K][S]: CTAs resident at once with clusters of S
    bool ready[2] = {false, false};
};

template <bool kQ4K>
static int device_info(DeviceInfo *&out) {
    static DeviceInfo info[64];
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return QWP_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    DeviceInfo &d = info[dev];
    if (!d.ready[kQ4K]) {
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return QWP_ERR_CUDA;
        if (cudaFuncSetAttribute(qwp_gemm_kernel<kQ4K>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SMEM_BYTES) != cudaSuccess)
            return QWP_ERR_CUDA;
        d.slots[kQ4K][1] = d.sms;
        for (int S = 2; S <= MAX_SPLITS; ++S) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(1, 1, S * 64);
            cfg.blockDim = dim3(NUM_THREADS, 1, 1);
            cfg.dynamicSmemBytes = SMEM_BYTES;
            cudaLaunchAttribute attr;
            attr.id = cudaLaunchAttributeClusterDimension;
            attr.val.clusterDim.x = 1;
            attr.val.clusterDim.y = 1;
            attr.val.clusterDim.z = S;
            cfg.attrs = &attr;
            cfg.numAttrs = 1;
            int clusters = 0;
            if (cudaOccupancyMaxActiveClusters(&clusters, qwp_gemm_kernel<kQ4K>, &cfg) != cudaSuccess) {
                cudaGetLastError();
                clusters = 0;
            }
            d.slots[kQ4K][S] = clusters * S;
        }
        d.ready[kQ4K] = true;
    }
    out = &d;
    return QWP_OK;
}

// Split-K factor: model the time as (waves of resident CTAs) x (fixed cost of
// two weight stages + the K stages per split) and take the cheapest.
static int choose_splits(const int *slots, int64_t base_ctas, int nstages) {
    int best = 1;
    double best_cost = 1e30;
    for (int S = 1; S <= MAX_SPLITS && S <= nstages; ++S) {
        const int per = (nstages + S - 1) / S;
        if ((nstages + per - 1) / per != S || slots[S] <= 0) continue;  // no empty or duplicate splits
        const int64_t waves = (base_ctas * S + slots[S] - 1) / slots[S];
        const double cost = static_cast<double>(waves) * (2.0 + per);
        if (cost < best_cost - 1e-9) {
            best_cost = cost;
            best = S;
        }
    }
    return best;
}

// x is fp16 [M, K].  `after_prior` launches with programmatic stream
// serialization so the kernel's set-up and weight prefetch overlap the grid just
// before it (the x producer waits for that grid with griddepcontrol.wait).
template <bool kQ4K>
static int launch_gemm(const void *w, const void *scales, const uint8_t *zeros, const void *x,
                       float *y, int64_t M, int64_t N, int64_t K, int64_t group, cudaStream_t stream,
                       uint64_t timeout_ns, bool after_prior) {
    int rc = check_device();
    if (rc) return rc;
    DeviceInfo *info = nullptr;
    if ((rc = device_info<kQ4K>(info))) return rc;
    uint32_t *status = status_word();
    if (!status) return QWP_ERR_CUDA;
    const int bn = choose_bn(M);
    CUtensorMap map;
    if ((rc = encode_x_map(&map, x, M, K, bn))) return rc;

    GemmArgs a;
    a.w = static_cast<const uint8_t *>(w);
    a.scales = static_cast<const __half *>(scales);
    a.zeros = zeros;
    a.y = y;
    a.status = status;
    a.M = static_cast<int>(M);
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    a.group = static_cast<int>(group);
    a.groups_per_row = group > 0 ? static_cast<int>(K / group) : 0;
    a.kb_per_group = group > 0 ? static_cast<int>(group / CHUNK_K) : 1;
    a.kbg_shift = -1;
    for (int sh = 0; sh < 31; ++sh)
        if ((1 << sh) == a.kb_per_group) a.kbg_shift = sh;
    a.bn = bn;
    a.timeout_ns = timeout_ns;
    // Commit groups: 4 blocks for short MMAs (N <= 128), else 2; never more than
    // divides the K blocks (every split's block count is then a multiple too).
    const int64_t nkb_total = K / CHUNK_K;
    int cbs = bn <= 128 ? 2 : 1;
    while (cbs > 0 && nkb_total % (1 << cbs)) --cbs;
    a.cb_shift = cbs;
    a.x_stage_bytes = (bn * 128) << cbs;
    a.w_stage_bytes = kQ4K ? TILE_ROWS * Q4K_BLOCK_BYTES : TILE_ROWS * CHUNK_ROW_BYTES * KB_PER_STAGE;
    a.w_stages = 4;
    a.x_stages = std::min(A_STAGES >> cbs, (RING_BYTES - a.w_stages * a.w_stage_bytes) / a.x_stage_bytes);
    a.w_stages = std::min(W_MAX_STAGES, (RING_BYTES - a.x_stages * a.x_stage_bytes) / a.w_stage_bytes);

    const int64_t row_tiles = (N + TILE_ROWS - 1) / TILE_ROWS;
    const int64_t tok_tiles = (M + bn - 1) / bn;
    const int nkb = static_cast<int>(K / CHUNK_K);
    const int nstages = (nkb + KB_PER_STAGE - 1) / KB_PER_STAGE;
    const int S = choose_splits(info->slots[kQ4K], row_tiles * tok_tiles, nstages);
    a.splits = S;
    a.kb_per_split = ((nstages + S - 1) / S) * KB_PER_STAGE;
    if (row_tiles > 0x7fffffff || tok_tiles > 65535) return QWP_ERR_UNSUPPORTED_SHAPE;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(row_tiles), static_cast<unsigned>(tok_tiles), S);
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attrs[2];
    unsigned nattr = 0;
    if (S > 1) {
        attrs[nattr].id = cudaLaunchAttributeClusterDimension;
        attrs[nattr].val.clusterDim.x = 1;
        attrs[nattr].val.clusterDim.y = 1;
        attrs[nattr].val.clusterDim.z = S;
        ++nattr;
    }
    if (after_prior) {
        attrs[nattr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attrs[nattr].val.programmaticStreamSerializationAllowed = 1;
        ++nattr;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = nattr;
    if (cudaLaunchKernelEx(&cfg, qwp_gemm_kernel<kQ4K>, map, a) != cudaSuccess) {
        cudaGetLastError();
        return QWP_ERR_CUDA;
    }
    return QWP_OK;
}

}  // namespace qwp

using namespace qwp;

static int gemm_shape_checks(const void *w, const void *x, const float *y, int64_t M, int64_t N,
                             int64_t K) {
    if (M < 0 || N < 0 || K < 0) return QWP_ERR_INVALID_ARG;
    if (M > (1ll << 30) || N > (1ll << 30) || K > (1ll << 30)) return QWP_ERR_UNSUPPORTED_SHAPE;
    if (M == 0 || N == 0) return QWP_OK;
    if (!w || !x || !y) return QWP_ERR_INVALID_ARG;
    if (!aligned16(w) || !aligned16(x) || !aligned16(y)) return QWP_ERR_MISALIGNED;
    return QWP_OK;
}

// Scratch for fp16 activations: a library-owned stream-ordered memory pool per
// device (allocations are freed, in stream order, right after the GEMM).
static int scratch_pool(cudaMemPool_t *out) {
    static cudaMemPool_t pools[64];
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return QWP_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    if (!pools[dev]) {
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t p;
        if (cudaMemPoolCreate(&p, &props) != cudaSuccess) return QWP_ERR_CUDA;
        uint64_t keep = UINT64_MAX;  // keep freed blocks for reuse
        cudaMemPoolSetAttribute(p, cudaMemPoolAttrReleaseThreshold, &keep);
        pools[dev] = p;
    }
    *out = pools[dev];
    return QWP_OK;
}

extern "C" int q4k_gemm_f16(const void *w_tiled, const void *x, float *y, int64_t M, int64_t N,
                            int64_t K, void *stream) {
    if (K % Q4K_BLOCK || K == 0) return K < 0 ? QWP_ERR_INVALID_ARG : QWP_ERR_UNSUPPORTED_SHAPE;
    int rc = gemm_shape_checks(w_tiled, x, y, M, N, K);
    if (rc || M == 0 || N == 0) return rc;
    return launch_gemm<true>(w_tiled, nullptr, nullptr, x, y, M, N, K, 0,
                             static_cast<cudaStream_t>(stream), kDefaultTimeoutNs, false);
}

extern "C" int q4k_gemm(const void *w_tiled, const void *x, float *y, int64_t M, int64_t N,
                        int64_t K, void *stream) {
    if (K % Q4K_BLOCK || K == 0) return K < 0 ? QWP_ERR_INVALID_ARG : QWP_ERR_UNSUPPORTED_SHAPE;
    int rc = gemm_shape_checks(w_tiled, x, y, M, N, K);
    if (rc || M == 0 || N == 0) return rc;
    if ((rc = check_device())) return rc;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaMemPool_t pool;
    if ((rc = scratch_pool(&pool))) return rc;
    void *x16 = nullptr;
    if (cudaMallocFromPoolAsync(&x16, static_cast<size_t>(M) * K * 2, pool, s) != cudaSuccess) {
        cudaGetLastError();
        return QWP_ERR_CUDA;
    }
    rc = launch_bf16_to_f16(x, x16, M * K, s);
    if (!rc) rc = launch_gemm<true>(w_tiled, nullptr, nullptr, x16, y, M, N, K, 0, s, kDefaultTimeoutNs, true);
    if (cudaFreeAsync(x16, s) != cudaSuccess && !rc) rc = QWP_ERR_CUDA;
    return rc;
}

extern "C" int w4a16_gemm(const void *wq_tiled, const void *scales, const uint8_t *zeros,
                          const void *x, float *y, int64_t M, int64_t N, int64_t K, int64_t group,
                          void *stream) {
    if (group <= 0 || group % CHUNK_K) return QWP_ERR_INVALID_ARG;
    if (K % group || K == 0) return K < 0 ? QWP_ERR_INVALID_ARG : QWP_ERR_UNSUPPORTED_SHAPE;
    int rc = gemm_shape_checks(wq_tiled, x, y, M, N, K);
    if (rc || M == 0 || N == 0) return rc;
    if (!scales || !zeros) return QWP_ERR_INVALID_ARG;
    return launch_gemm<false>(wq_tiled, scales, zeros, x, y, M, N, K, group,
                              static_cast<cudaStream_t>(stream), kDefaultTimeoutNs, false);
}
