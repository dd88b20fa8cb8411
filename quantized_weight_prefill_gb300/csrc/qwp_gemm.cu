// Fused dequant-in-tile GEMM on the 5th-generation tensor cores (tcgen05).
//
// y[M,N] = x[M,K] . W[N,K]^T with W in 4-bit (Q4_K, W4A16) or 6-bit (Q6_K) form.  Method: "The dequant
// scratch round-trip is ZINC's last RDNA4 prefill tax", sections "The two
// passes hiding inside one matmul" and "What the roofline says" -- every
// packed weight block is read from global memory once, unpacked on chip and
// consumed by the matmul tile; no 16-bit weight copy ever reaches DRAM.  Token
// batching follows "How ZINC's RDNA4 batched prefill went from 42 to 208
// tok/s", section "The two prefill paths": each weight row is applied to a
// whole chunk of prompt tokens per read.
//
// The grid is persistent: one CTA per SM (a cluster of S CTAs when K is split S
// ways) loops over units, a unit being a 128-row (weights) x BN-token (BN <= 256)
// tile of y^T; CTA rank s of a cluster computes K range s of every unit.  The
// rings run on across units, so the copies and unpacking of the next unit
// overlap the end of the current one.  Roles:
//   warp 0        x producer: one thread issues 2-D TMA loads (128-byte swizzle),
//                 one per 64-wide K block, into the x ring;
//   warp 1        allocates tensor memory; runs the MMA loop, one elected lane
//                 issuing every tcgen05.mma;
//   warp 2        weight producer: one bulk copy per 256-wide K stage of packed
//                 weights into the weight ring;
//   warps 3..18   transform: four groups of 4 warps; group g owns K block g of
//                 every weight stage (4 blocks of 64); warp (group g, quarter q)
//                 unpacks rows 32q..32q+31 (its tensor-memory lane quarter) of
//                 that block, 64 weights per thread, to fp16 and stores them with
//                 one tcgen05.st into the A ring in tensor memory;
//   warps 19..22  epilogue (two-accumulator kernel only): drain the fp32
//                 accumulator (tcgen05.ld) into y, or, with split-K, into the
//                 owning CTA of the cluster, which sums the partials in rank
//                 order (deterministic) and writes y.
// Tensor memory (512 columns): the A ring (8 blocks of 128 lanes x 64 K = 32
// columns) at column 256; below it one accumulator [128 lanes x BN], drained by
// the transform warps between units (the one-accumulator kernel: BN > 128, 19
// warps), or two of 128 columns when BN <= 128, so that the epilogue of a unit
// overlaps the MMAs of the next (the two-accumulator kernel: 23 warps, split-K
// allowed).  The MMA is D[128 x BN] += A[128 x 16] (tensor memory) .
// B[BN x 16]^T (shared memory): weights are the M side and tokens the N side, so
// a tile reuses each unpacked weight for BN tokens.
//
// Every mbarrier wait is bounded: on expiry the thread records a timeout in
// the library's status word and sets a CTA-wide abort flag; all roles then
// wait (bounded) for their own copies and MMAs in flight, the tensor memory is
// released and the CTA exits.
#include <algorithm>
#include <atomic>
#include <mutex>

#include "qwp_decode.h"
#include "qwp_format.cuh"
#include "qwp_internal.h"
#include "qwp_ptx.cuh"
#include "qwp_sync.cuh"

namespace qwp {

// Weight formats (the kernel's template parameter).
enum : int { FMT_W4A16 = DFMT_W4A16, FMT_Q4K = DFMT_Q4K, FMT_Q6K = DFMT_Q6K, NUM_FMTS = 3 };

constexpr int XFORM_GROUPS = 4;                    // groups take K blocks in turn, one per weight stage
constexpr int NUM_XFORM_WARPS = 4 * XFORM_GROUPS;  // 4 warps (one per lane quarter) cover one K block
constexpr int FIRST_XFORM_WARP = 3;
constexpr int FIRST_EPI_WARP = FIRST_XFORM_WARP + NUM_XFORM_WARPS;
constexpr int NUM_EPI_WARPS = 4;                   // one per tensor-memory lane quarter
constexpr int NUM_THREADS = 32 * (FIRST_EPI_WARP + NUM_EPI_WARPS);
// With one accumulator the transform warps drain it and there are no epilogue
// warps: 19 warps (at most 5 per scheduler) leave 96 registers per thread
// instead of 80.
constexpr int NUM_THREADS_1ACC = 32 * FIRST_EPI_WARP;
__host__ __device__ constexpr int block_threads(bool two_acc) { return two_acc ? NUM_THREADS : NUM_THREADS_1ACC; }
constexpr int X_MAX_STAGES = 8;  // <= A_STAGES: the x ring reuses the mma_done ring (see below)
constexpr int W_MAX_STAGES = 8;
constexpr int A_STAGES = 8;
constexpr int BN_MAX = 256;
constexpr int KB_PER_STAGE = 4;  // 64-wide K blocks per weight stage
constexpr int MAX_SPLITS = 8;    // portable cluster size
// bf16 x is converted in the kernel (no conversion kernel) for up to this many
// tokens: the MMA warp converts the token row of each x slot right before its
// MMAs, one 16-byte chunk per lane and group (at one token 6-16% faster than a
// conversion kernel; at two tokens mixed; at eight, with eight chunks per lane on
// the MMA warp's critical path, up to 44% slower).
constexpr int CONVERT_MAX_M = 1;
constexpr uint32_t ACC_COL = 0;
constexpr uint32_t ACC_STRIDE = 128;  // second accumulator buffer (token tiles of <= 128)
constexpr uint32_t A_COL = 256;
constexpr uint32_t TMEM_COLS = 512;

// Split-K: tokens of a unit owned by each of S cluster ranks, a multiple of 4.
// Partial sums travel between ranks as quads (4 consecutive tokens of one row,
// 16 bytes): a partial buffer holds, per source rank q, the owner's `per` tokens
// quad-major, float index ((q*per + t) / 4) * 4*TILE_ROWS + 4*row + t % 4, so a
// warp's 32 rows write and read 512 contiguous bytes per quad.
__host__ __device__ constexpr int split_per(int bn, int S) { return ((bn + S - 1) / S + 3) & ~3; }

// Shared memory: a ring region (x slots, then weight stages, then, with split-K,
// the buffer that receives the cluster's partial sums), then mbarriers and misc words.
constexpr int RING_BYTES = 224 * 1024;
constexpr int OFF_BAR = RING_BYTES;
constexpr int NUM_BARS = 2 * X_MAX_STAGES + 2 * W_MAX_STAGES + 2 * A_STAGES + 4 + 5;
constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + slack to align the base to 1 KiB
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(X_MAX_STAGES <= A_STAGES, "the x ring is released through the mma_done ring");
static_assert(A_STAGES % 4 == 0, "commit groups of up to 4 blocks tile the A ring");
static_assert(XFORM_GROUPS == KB_PER_STAGE, "each transform warp owns one K block of every weight stage");
static_assert(2 * ACC_STRIDE <= A_COL, "two accumulator buffers of 128 columns fit below the A ring");

struct GemmArgs {
    const uint8_t *w;       // repacked weights
    const __half *scales;   // W4A16: [N][K/group]
    const uint8_t *zeros;   // W4A16: [N][K/group], or null: symmetric (zero point 8)
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
    int n_units;            // row tiles x token tiles; cluster c runs units c, c + gridDim.x, ...
    int row_tiles;
    int acc_bufs;           // 2 when two accumulators fit (bn <= 128), else 1
    int part_off;           // shared-memory offset of the split-K partial buffer
    int part_overlay;       // 1: one unit per CTA, the partial buffer overlays the idle rings
    int x_convert;          // x is bf16, converted to fp16 in shared memory: 1 by the MMA warp (one
                            // token), 2 by the epilogue warps (one unit per CTA); 0: x is fp16
    int batch;              // independent problems of one shape (1: a single GEMM)
    int units_per_problem;  // row tiles x token tiles of one problem
    int64_t w_batch_bytes;  // bytes from one problem's weights to the next's
    uint64_t timeout_cycles;  // bound on a main-loop wait, in SM clock cycles
    uint64_t drain_cycles;    // bound on a wait for the CTA's own work in flight
};

// Status codes recorded on a timeout: which wait gave up.
enum : uint32_t {
    WAIT_W_EMPTY = 1, WAIT_X_EMPTY, WAIT_X_FULL, WAIT_A_FULL, WAIT_W_FULL, WAIT_A_EMPTY,
    WAIT_ACC_FULL, WAIT_DRAIN, WAIT_ACC_EMPTY, WAIT_PART
};


// One commit group: CB 64-wide K blocks of 4 MMAs (K = 16 each).  A block c sits at
// tensor-memory column acol + 32c, its x tile at B-descriptor low word
// b_lo + tile_desc*c; K step kk advances A by 8 columns and B by 32 bytes.  The
// group accumulates onto D unless it is the first of its unit (acc_in false).
template <int CB>
__device__ __forceinline__ void mma_group(uint32_t dcol, uint32_t acol, uint32_t b_lo, uint32_t b_hi,
                                          uint32_t tile_desc, uint32_t idesc, bool acc_in) {
    static_assert(CHUNK_K == 64, "4 MMAs of K = 16 per block");
    if (acc_in)
        mma_ts_w<true>(dcol, acol, b_lo, b_hi, idesc);
    else
        mma_ts_w<false>(dcol, acol, b_lo, b_hi, idesc);
#pragma unroll
    for (int kk = 1; kk < 4; ++kk) mma_ts_w<true>(dcol, acol + 8u * kk, b_lo + 2u * kk, b_hi, idesc);
#pragma unroll
    for (int c = 1; c < CB; ++c)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            mma_ts_w<true>(dcol, acol + 32u * c + 8u * kk, b_lo + tile_desc * c + 2u * kk, b_hi, idesc);
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

// Q6_K: low words 4q..4q+3 of a chunk (wv) with their high words h0 (sub-block
// 2q) and h1 (sub-block 2q+1) into regs[off .. off+15].
__device__ __forceinline__ void unpack_q6k_quarter(uint4 wv, uint32_t h0, uint32_t h1, const Q6kSub &k0,
                                                   const Q6kSub &k1, uint32_t (&regs)[32], int off) {
    uint32_t p[4];
    q6k_word_f16x2<0>(wv.x, h0, k0, p);
#pragma unroll
    for (int e = 0; e < 4; ++e) regs[off + e] = p[e];
    q6k_word_f16x2<1>(wv.y, h0, k0, p);
#pragma unroll
    for (int e = 0; e < 4; ++e) regs[off + 4 + e] = p[e];
    q6k_word_f16x2<0>(wv.z, h1, k1, p);
#pragma unroll
    for (int e = 0; e < 4; ++e) regs[off + 8 + e] = p[e];
    q6k_word_f16x2<1>(wv.w, h1, k1, p);
#pragma unroll
    for (int e = 0; e < 4; ++e) regs[off + 12 + e] = p[e];
}

// Split-K: y for the quad (tokens m .. m+3, row `row` of row tile `tile`), tokens
// at or beyond M and rows at or beyond R left out.  A warp's 32 consecutive rows
// write 128 contiguous bytes per token.
__device__ __forceinline__ void store_quad(float *y, float4 acc, int m, int tile, int row, int R, int M,
                                           int64_t N) {
    if (row >= R) return;
    float *yc = y + static_cast<int64_t>(m) * N + static_cast<int64_t>(tile) * TILE_ROWS + row;
    const float a4[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
    for (int e = 0; e < 4; ++e)
        if (m + e < M) __stcs(yc + e * N, a4[e]);
}

// Split-K: an owner's sum of its tokens [t0, t1) of the tile over the S source
// regions of its partial buffer (quad-major, see split_per), in rank order, to y.
// Threads first, first + stride, .. take (quad, row) items, rows fastest.
__device__ __forceinline__ void reduce_quads(const float4 *pbuf, int S, int per, int t0, int t1, int first,
                                             int stride, float *y, int m0, int tile, int R, int M, int64_t N) {
    const int items = (t1 - t0) / 4 * TILE_ROWS;
    for (int itm = first; itm < items; itm += stride) {
        const int qd = itm / TILE_ROWS, rr = itm % TILE_ROWS;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int q = 0; q < S; ++q) {
            const float4 pv = pbuf[(q * (per / 4) + qd) * TILE_ROWS + rr];
            acc.x += pv.x; acc.y += pv.y; acc.z += pv.z; acc.w += pv.w;
        }
        store_quad(y, acc, m0 + t0 + 4 * qd, tile, rr, R, M, N);
    }
}

// kTwoAcc: token tiles of at most 128, two accumulators, split-K allowed, 23
// warps; else one accumulator, no split-K and no epilogue warps (the two are
// compiled apart, so that neither carries the other's code and registers).
// kBatch: a strided batch of problems (x through a rank-3 tensor map); compiled
// apart too, since the per-unit problem offsets cost single GEMMs ~1 us.
// kMulti: a CTA may run several units (else at most one: no epilogue-warp loop
// and no split-K buffer of its own are compiled in; the launches of one unit per
// CTA measured up to 0.5 us slower with that code present).
template <int kFmt, bool kTwoAcc, bool kBatch = false, bool kMulti = true>
__global__ void __launch_bounds__(block_threads(kTwoAcc), 1)
    qwp_gemm_kernel(const __grid_constant__ CUtensorMap tmap_x, const GemmArgs args) {
    constexpr bool kQ4K = kFmt == FMT_Q4K;
    constexpr bool kQ6K = kFmt == FMT_Q6K;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const uint32_t warp = warp_id();
    const uint32_t lane = lane_id();

    // This CTA's K range (its cluster rank along K) is the same for every unit.
    const int S = kTwoAcc ? args.splits : 1;
    const int nkb_total = args.K / CHUNK_K;
    const int kb_begin = blockIdx.z * args.kb_per_split;
    const int kb_end = min(nkb_total, kb_begin + args.kb_per_split);
    const int nkb = kb_end - kb_begin;
    const int nstage = (nkb + KB_PER_STAGE - 1) / KB_PER_STAGE;
    const int XS = args.x_stages, WS = args.w_stages;
    uint8_t *const x_ring = smem;
    uint8_t *const w_ring = smem + XS * args.x_stage_bytes;
    const int nbufs = kTwoAcc ? 2 : 1;
    const int units0 = static_cast<int>(blockIdx.x);  // units units0, units0 + gridDim.x, ...
    const int ustep = static_cast<int>(gridDim.x);
    const int nunits = args.n_units;
    const int n_mine = units0 < nunits ? (nunits - 1 - units0) / ustep + 1 : 0;  // units of this CTA
    // Row tile and token tile of unit u: consecutive units share a token tile, so
    // concurrently running CTAs read the same activation tile (one read, L2 hits);
    // the packed weights are the smaller stream per unit.
    // Batched calls number the units problem-major; problem p's weights, x and y
    // sit p strides further (x through the third coordinate of its tensor map).
    auto unit_prob = [&](int u) { return kBatch ? u / args.units_per_problem : 0; };
    auto unit_tile = [&](int u) { return (u - unit_prob(u) * args.units_per_problem) % args.row_tiles; };
    auto unit_m0 = [&](int u) { return ((u - unit_prob(u) * args.units_per_problem) / args.row_tiles) * args.bn; };
    auto unit_y = [&](int u) { return args.y + static_cast<int64_t>(unit_prob(u)) * args.M * args.N; };

    const uint32_t bar0 = smem_u32(smem + OFF_BAR);
    // The MMA issuer works in commit groups of CB = 2^cb_shift consecutive K blocks:
    // one a_full wait (every transform warp of the group's blocks arrives), one
    // x_full wait (the group's CB x tiles share one ring slot and barrier), 4*CB
    // MMAs and one tcgen05.commit.  A single thread issues every MMA of the CTA,
    // and its fixed cost per loop iteration (waits, fence, bookkeeping) is several
    // hundred cycles on a busy SM, so it is paid per group rather than per block.
    // mma_done[(J % A_STAGES) >> cb_shift] completes when the MMAs of the group
    // holding the CTA's J-th block (counted over all its units) are done; that
    // releases the group's A slots and its x slot (the x ring has at most
    // A_STAGES / CB slots, so no phase of mma_done is skipped).
    const int cbs = args.cb_shift;
    const int dslots = A_STAGES >> cbs;  // commit-group slots of the A ring
    const int ngroups = nkb >> cbs;      // nkb is a multiple of CB
    const uint32_t x_full = bar0, mma_done = x_full + 8 * X_MAX_STAGES;
    const uint32_t w_full = mma_done + 8 * A_STAGES, w_empty = w_full + 8 * W_MAX_STAGES;
    const uint32_t a_full = w_empty + 8 * W_MAX_STAGES, acc_full = a_full + 8 * A_STAGES;
    const uint32_t acc_empty = acc_full + 16, part_full = acc_empty + 16, part_free = part_full + 8;
    const uint32_t part_last = part_free + 8, drain = part_last + 8, rings_idle = drain + 8;
    const uint32_t x_conv = rings_idle + 8;  // x slot converted to fp16 (x_convert == 2)
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + OFF_MISC);  // [0] tmem base, [1] abort
    const Ctl ctl{misc + 1, args.status, args.timeout_cycles, args.drain_cycles};

    // Copy of weight stage s (K blocks kb_begin + 4s ..) of unit u's row tile into ring slot ws.
    auto load_weight_stage = [&](int u, int s, int ws) {
        const int tile = unit_tile(u);
        const uint8_t *wp = args.w + static_cast<int64_t>(unit_prob(u)) * args.w_batch_bytes;
        const int R = tile_rows(args.N, tile);
        const int kb0 = kb_begin + KB_PER_STAGE * s;
        const int nblk = min(KB_PER_STAGE, kb_end - kb0);
        const uint8_t *src;
        uint32_t bytes;
        if (kQ4K) {
            src = wp + q4k_group_offset(args.K, tile, R, kb0 / KB_PER_STAGE);
            bytes = static_cast<uint32_t>(R) * Q4K_BLOCK_BYTES;
        } else if (kQ6K) {
            const int Rp = q6k_padded_rows(R);
            src = wp + q6k_group_offset(args.K, tile, Rp, kb0 / KB_PER_STAGE);
            bytes = static_cast<uint32_t>(Rp) * Q6K_BLOCK_BYTES;
        } else {
            src = wp + w4_plane_offset(args.K, tile, R, kb0);
            bytes = static_cast<uint32_t>(R) * CHUNK_ROW_BYTES * nblk;
        }
        mbar_arrive_expect_tx(w_full + 8 * ws, bytes);
        bulk_copy_g2s(smem_u32(w_ring + ws * args.w_stage_bytes), src, bytes, w_full + 8 * ws);
    };
    // The weight producer's thread sets up the barriers and starts the first weight
    // copies of its first unit before the block-wide barrier (their slots are empty).
    const int w_pre = units0 < nunits ? min(WS, nstage) : 0;
    pdl_launch_dependents();
    if (threadIdx.x == 64) {
        for (int s = 0; s < X_MAX_STAGES; ++s) {
            mbar_init(x_full + 8 * s, 1);
            mbar_init(x_conv + 8 * s, NUM_EPI_WARPS);
        }
        for (int s = 0; s < A_STAGES; ++s) mbar_init(mma_done + 8 * s, 1);
        for (int s = 0; s < W_MAX_STAGES; ++s) {
            mbar_init(w_full + 8 * s, 1);
            mbar_init(w_empty + 8 * s, NUM_XFORM_WARPS);
        }
        // A commit group of CB <= XFORM_GROUPS blocks is stored by CB transform groups.
        for (int s = 0; s < A_STAGES; ++s)
            mbar_init(a_full + 8 * s, (NUM_XFORM_WARPS / XFORM_GROUPS) << cbs);
        // The accumulator is drained by the transform warps when there is one, by
        // the epilogue warps when there are two.
        for (int b = 0; b < 2; ++b) {
            mbar_init(acc_full + 8 * b, 1);
            mbar_init(acc_empty + 8 * b, nbufs == 2 ? NUM_EPI_WARPS : NUM_XFORM_WARPS);
        }
        // Split-K: every epilogue warp of every CTA of the cluster arrives once per unit.
        mbar_init(part_full, NUM_EPI_WARPS * S);
        mbar_init(part_free, NUM_EPI_WARPS * S);
        mbar_init(part_last, NUM_XFORM_WARPS * S);  // the last unit: every transform warp of every rank
        mbar_init(rings_idle, S);                   // the last unit: one arrival per rank
        mbar_init(drain, 1);
        fence_mbar_init();
        prefetch_tensormap(&tmap_x);
        // The weights may come from a repack launched just before, the status word
        // from any earlier kernel; every other thread is ordered after this wait by
        // the block-wide barrier below.
        pdl_wait();
        // A failure recorded earlier (and not yet read by qwp_device_status) makes
        // every later launch skip its work instead of waiting out its own timeouts
        // (the weight copies started below are still waited for).  The status load
        // is issued before the copies and its value used after them, so that its
        // latency overlaps theirs instead of adding to the set-up.
        const uint32_t status_now = *reinterpret_cast<volatile uint32_t *>(args.status);
        for (int s = 0; s < w_pre; ++s) load_weight_stage(units0, s, s);
        misc[1] = (status_now & kStatusTimeoutMask) ? 1u : 0u;
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(misc), TMEM_COLS);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    // Split-K with a partial buffer of its own: peers arrive on this CTA's
    // barriers and write into the buffer, so the barriers must be initialised
    // cluster-wide before any thread touches another CTA.  Every thread arrives
    // here and waits once, just before its first remote access (epilogue warps) or
    // at the last unit (the others).  (With the buffer overlaying the rings, the
    // last unit is reduced between two cluster barriers instead.)
    const bool split_mbar = kMulti && S > 1 && !args.part_overlay;
    if (split_mbar) cluster_arrive_relaxed();
    // This thread has arrived on the cluster barrier above and not yet waited on it
    // (the epilogue warps wait at their start, the others at the last unit).
    bool cluster_wait_due = split_mbar && warp < FIRST_EPI_WARP;
    tc_fence_after();
    const uint32_t tmem = misc[0];
    const bool skip = misc[1] != 0;
    bool xform_ok = false;  // transform warps: every unit's blocks were stored

    if (warp == 0) {
        // ------------------------------------------------------------ x producer
        if (lane == 0 && !skip) {
            pdl_wait();  // x may come from the grid launched just before (ordered already; explicit here)
            int issued = 0;     // groups issued over all units
            int xs = 0;         // ring slot (running counters: no division in the loop)
            int dk = 0;         // mma_done slot of group `issued - XS`, and its phase
            uint32_t dph = 0;
            bool ok = true;
            const uint32_t tile_bytes = static_cast<uint32_t>(args.bn) * 128u;
            for (int u = units0; ok && u < nunits; u += ustep) {
                const int m0 = unit_m0(u), xp = unit_prob(u);
                for (int g = 0; g < ngroups; ++g) {
                    if (issued >= XS) {  // slot xs last held group issued - XS
                        if (!(ok = wait_bar(mma_done + 8 * dk, dph, ctl, WAIT_X_EMPTY))) break;
                        if (++dk == dslots) { dk = 0; dph ^= 1; }
                    }
                    mbar_arrive_expect_tx(x_full + 8 * xs, tile_bytes << cbs);
                    for (int c = 0; c < (1 << cbs); ++c) {
                        const uint32_t dst = smem_u32(x_ring + xs * args.x_stage_bytes + c * tile_bytes);
                        const int kc = (kb_begin + (g << cbs) + c) * CHUNK_K;
                        if (kBatch)
                            tma_load_3d(dst, &tmap_x, kc, m0, xp, x_full + 8 * xs);
                        else
                            tma_load_2d(dst, &tmap_x, kc, m0, x_full + 8 * xs);
                    }
                    ++issued;
                    if (++xs == XS) xs = 0;
                }
            }
            // Every copy issued above lands before the CTA may exit.
            for (int g = max(0, issued - XS); g < issued; ++g)
                wait_bar(x_full + 8 * (g % XS), (g / XS) & 1, ctl, WAIT_DRAIN, false);
        }
    } else if (warp == 2) {
        // ------------------------------------------------------------ weight producer
        if (lane == 0 && skip)
            for (int s = 0; s < w_pre; ++s) wait_bar(w_full + 8 * s, 0, ctl, WAIT_DRAIN, false);
        if (lane == 0 && !skip) {
            int issued = 0;  // stages over all units; the first w_pre went out above
            int ws = 0;
            uint32_t wph = 0;
            bool ok = true;
            for (int u = units0; ok && u < nunits; u += ustep) {
                const int tile = unit_tile(u);
                for (int s = 0; s < nstage; ++s) {
                    if (issued >= w_pre) {
                        if (issued >= WS && !(ok = wait_bar(w_empty + 8 * ws, wph ^ 1, ctl, WAIT_W_EMPTY))) break;
                        load_weight_stage(u, s, ws);
                    }
                    ++issued;
                    if (++ws == WS) { ws = 0; wph ^= 1; }
                }
            }
            for (int s = max(0, issued - WS); s < issued; ++s)
                wait_bar(w_full + 8 * (s % WS), (s / WS) & 1, ctl, WAIT_DRAIN, false);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs the loop (its values stay warp-uniform) and one elected
        // lane issues the MMAs and commits: the issuer shares its scheduler with
        // transform warps, so every instruction it saves per MMA shortens the
        // MMA stream.
        if (!skip) {
            const uint32_t idesc = make_idesc_f16(false, TILE_ROWS, static_cast<uint32_t>(args.bn));  // fp16 A and B
            bool ok = true;
            int xs = 0, gs = 0;       // x ring slot; commit-group slot of the A ring
            uint32_t xph = 0, gph = 0;
            const uint64_t xdesc0 = smem_desc_sw128(smem_u32(x_ring));
            const uint32_t x_lo0 = static_cast<uint32_t>(xdesc0), x_hi = static_cast<uint32_t>(xdesc0 >> 32);
            const uint32_t x_step = static_cast<uint32_t>(args.x_stage_bytes) >> 4;  // one x slot, descriptor units
            const uint32_t tile_desc = static_cast<uint32_t>(args.bn) * 128u >> 4;   // one x tile, descriptor units
            const int conv_rows = min(args.bn, args.M);  // bf16 x: token rows of a tile (one token tile)
            const int x_tile_bytes = args.bn * 128;
            bool big = false;  // bf16 x: an activation beyond fp16's range
            int it = 0;
            for (int u = units0; ok && u < nunits; u += ustep, ++it) {
                // The unit accumulates into buffer b once the epilogue has drained b.
                const int b = nbufs == 2 ? (it & 1) : 0;
                const int use = nbufs == 2 ? (it >> 1) : it;  // earlier uses of buffer b
                if (!(ok = __all_sync(0xffffffffu, wait_bar(acc_empty + 8 * b, (use & 1) ^ 1, ctl, WAIT_ACC_EMPTY))))
                    break;
                tc_fence_after();
                const uint32_t dcol = tmem + ACC_COL + ACC_STRIDE * static_cast<uint32_t>(b);
                for (int g = 0; g < ngroups; ++g) {
                    ok = __all_sync(0xffffffffu, wait_bar((!kMulti && args.x_convert == 2 ? x_conv : x_full) + 8 * xs, xph, ctl,
                                                              WAIT_X_FULL) &&
                                                     wait_bar(a_full + 8 * gs, gph, ctl, WAIT_A_FULL));
                    if (!ok) break;
                    if (args.x_convert == 1) {
                        // bf16 x of a few tokens: the token rows of the group's tiles (8
                        // chunks of 8 consecutive K each; the swizzle moves whole chunks
                        // within a row) to fp16 in place; the other rows are the copies'
                        // zero fill, zero in fp16 too.
                        uint8_t *slot = x_ring + xs * args.x_stage_bytes;
                        for (int j = static_cast<int>(lane); j < (conv_rows * 8) << cbs; j += 32) {
                            uint4 *chunk = reinterpret_cast<uint4 *>(slot + (j / (conv_rows * 8)) * x_tile_bytes) +
                                           j % (conv_rows * 8);
                            const uint4 v = *chunk;
                            const uint32_t src[4] = {v.x, v.y, v.z, v.w};
                            uint32_t dst[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float lo = __uint_as_float(src[e] << 16);
                                const float hi = __uint_as_float(src[e] & 0xFFFF0000u);
                                big |= !(fabsf(lo) < 65520.f) || !(fabsf(hi) < 65520.f);
                                dst[e] = as_u32(__floats2half2_rn(lo, hi));
                            }
                            *chunk = make_uint4(dst[0], dst[1], dst[2], dst[3]);
                        }
                        fence_proxy_async_smem();  // read by the tensor core next
                        __syncwarp();
                    }
                    tc_fence_after();
                    const uint32_t b_lo = x_lo0 + x_step * static_cast<uint32_t>(xs);
                    const uint32_t acol = tmem + A_COL + (32u << cbs) * static_cast<uint32_t>(gs);
                    if (elect_one()) {
                        if (cbs == 2)
                            mma_group<4>(dcol, acol, b_lo, x_hi, tile_desc, idesc, g != 0);
                        else if (cbs == 1)
                            mma_group<2>(dcol, acol, b_lo, x_hi, tile_desc, idesc, g != 0);
                        else
                            mma_group<1>(dcol, acol, b_lo, x_hi, tile_desc, idesc, g != 0);
                        mma_commit(mma_done + 8 * gs);
                    }
                    __syncwarp();
                    if (++xs == XS) { xs = 0; xph ^= 1; }
                    if (++gs == dslots) { gs = 0; gph ^= 1; }
                }
                if (ok && elect_one()) mma_commit(acc_full + 8 * b);
                __syncwarp();
            }
            if (__any_sync(0xffffffffu, big) && lane == 0) atomicOr(args.status, kStatusRangeBit);
            if (!ok && lane == 0) {
                mma_commit(drain);
                wait_bar(drain, 0, ctl, WAIT_DRAIN, false);
            }
            __syncwarp();
        }
    } else if (warp < FIRST_EPI_WARP) {
        // ------------------------------------------------------------ transform
        const uint32_t xw = warp - FIRST_XFORM_WARP;
        const int grp = static_cast<int>(xw >> 2);   // this warp's block of every weight stage
        const uint32_t quarter = warp & 3;            // tensor-memory lanes 32*quarter .. +31
        const int r = static_cast<int>(quarter * 32 + lane);
        const uint32_t lane_base = (quarter * 32u) << 16;
        bool ok = !skip;
        int ws = -1;       // weight ring slot of this warp's current stage, and its phase
        uint32_t wph = 0;

        // Weight stage s of row tile `tile`: wait for it; if it holds this warp's block
        // (block 4s + grp of the CTA's range; a short last stage may not), unpack the
        // thread's row of it into `regs` (64 weights as 32 fp16 pairs); release the
        // stage.  Returns false on timeout or abort.
        auto prepare = [&](int tile, int s, uint32_t (&regs)[32], bool &has_block) -> bool {
            if (++ws == WS) { ws = 0; wph ^= 1; }
            const uint8_t *wst = w_ring + ws * args.w_stage_bytes;
            // Every lane waits; the warp moves on together (tcgen05.st/ld are warp-collective).
            if (!__all_sync(0xffffffffu, wait_bar(w_full + 8 * ws, wph, ctl, WAIT_W_FULL))) return false;
            const int R = tile_rows(args.N, tile);
            const bool valid = r < R;
            const int jj = KB_PER_STAGE * s + grp;  // block index within the CTA's range
            has_block = jj < nkb;
            uint4 wv0 = make_uint4(0, 0, 0, 0), wv1 = make_uint4(0, 0, 0, 0);
            Q4kSubH k0, k1;
            __half2 s2 = __float2half2_rn(0.f), mz = w4_magic_zero(0);
            uint4 hv = make_uint4(0, 0, 0, 0);  // Q6_K: high-bit words of this block
            Q6kSub ds[4];                       // Q6_K: constants of its four 16-weight scale groups
            if (kQ6K)
                for (int u = 0; u < 4; ++u) ds[u] = q6k_sub(0u, 0);
            if (has_block) {
                if (kQ6K) {
                    if (valid) {
                        const int Rp = q6k_padded_rows(R);
                        const uint32_t dbits = *reinterpret_cast<const uint16_t *>(wst + 2 * r);
                        const uint32_t sc4 =
                            *reinterpret_cast<const uint32_t *>(wst + Q6K_SCALE_PLANE * Rp + 16 * r + 4 * grp);
                        const uint8_t *lp = wst + Q6K_LOW_PLANE * Rp + CHUNK_ROW_BYTES * Rp * grp + r * 16;
                        wv0 = *reinterpret_cast<const uint4 *>(lp);
                        wv1 = *reinterpret_cast<const uint4 *>(lp + 16 * Rp);
                        hv = *reinterpret_cast<const uint4 *>(wst + Q6K_HIGH_PLANE * Rp + 16 * Rp * grp + r * 16);
                        q6k_chunk_scales(dbits, sc4, ds);
                    }
                } else if (kQ4K) {
                    uint4 hdr = make_uint4(0, 0, 0, 0);
                    if (valid) {
                        hdr = *reinterpret_cast<const uint4 *>(wst + Q4K_HEADER_BYTES * r);
                        const uint8_t *cp = wst + Q4K_HEADER_BYTES * R + CHUNK_ROW_BYTES * R * grp + r * 16;
                        wv0 = *reinterpret_cast<const uint4 *>(cp);
                        wv1 = *reinterpret_cast<const uint4 *>(cp + 16 * R);
                    }
                    k0 = q4k_sub_f16(hdr, 2 * grp);
                    k1 = q4k_sub_f16(hdr, 2 * grp + 1);
                } else if (valid) {
                    const uint8_t *cp = wst + CHUNK_ROW_BYTES * R * grp + r * 16;
                    wv0 = *reinterpret_cast<const uint4 *>(cp);
                    wv1 = *reinterpret_cast<const uint4 *>(cp + 16 * R);
                    const int64_t n = static_cast<int64_t>(tile) * TILE_ROWS + r;
                    const int64_t ng = args.groups_per_row;
                    const int kbi = kb_begin + jj;
                    const int64_t g = args.kbg_shift >= 0 ? (kbi >> args.kbg_shift) : (kbi / args.kb_per_group);
                    s2 = __half2half2(args.scales[n * ng + g]);
                    mz = w4_magic_zero(args.zeros ? args.zeros[n * ng + g] : 8u);  // no zeros: symmetric
                }
            }
            // This warp's reads of the stage are done.
            __syncwarp();
            if (lane == 0) mbar_arrive(w_empty + 8 * ws);
            if (has_block) {
                if (kQ6K) {
                    unpack_q6k_quarter(wv0, hv.x, hv.y, ds[0], ds[1], regs, 0);
                    unpack_q6k_quarter(wv1, hv.z, hv.w, ds[2], ds[3], regs, 16);
                } else {
                    unpack_quarter<kQ4K>(wv0, k0, mz, s2, regs, 0);
                    unpack_quarter<kQ4K>(wv1, k1, mz, s2, regs, 16);
                }
            }
            return true;
        };
        // Store the CTA's J-th block into its A ring slot once the MMAs of block
        // J - A_STAGES (the slot's previous content) are done.
        auto issue = [&](int J, const uint32_t (&regs)[32]) -> bool {
            const int as = J & (A_STAGES - 1);
            if (!__all_sync(0xffffffffu, wait_bar(mma_done + 8 * (as >> cbs), ((J / A_STAGES) & 1) ^ 1, ctl,
                                                  WAIT_A_EMPTY)))
                return false;
            tc_fence_after();
            tmem_st_x32(tmem + lane_base + A_COL + 32u * as, regs);
            return true;
        };
        // Block J's tensor-memory store lands; publish it to the MMA issuer.
        auto finish = [&](int J) {
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(a_full + 8 * ((J & (A_STAGES - 1)) >> cbs));
        };

        // With one accumulator the transform warps drain it into y between units
        // (the MMAs of the next unit wait for that anyway): unit `uu`, the CTA's
        // `itx`-th, split-K never applies (it needs two accumulators).
        auto drain_unit = [&](int uu, int itx) -> bool {
            if (!__all_sync(0xffffffffu, wait_bar(acc_full, itx & 1, ctl, WAIT_ACC_FULL))) return false;
            tc_fence_after();
            const int tile = unit_tile(uu), m0 = unit_m0(uu);
            const int R = tile_rows(args.N, tile);
            const int64_t N = args.N;
            // Chunk ci (8 token columns) holds tokens m0 + 8ci ..; this warp takes every
            // fourth chunk from its group's, so its y pointer and the count of tokens
            // left step by 32 tokens.  (Stepping a pointer rather than forming each
            // address from the token index keeps this loop cheap: it runs while the
            // MMAs wait for the accumulator, 8 stores per load.)
            float *yc = unit_y(uu) + (static_cast<int64_t>(m0) + 8 * grp) * N + static_cast<int64_t>(tile) * TILE_ROWS + r;
            const int64_t chunk_step = 8 * (NUM_XFORM_WARPS / 4) * N;
            int left = args.M - m0 - 8 * grp;
            const bool row_ok = r < R;
            // 8 columns at a time: this warp's 32 unpacked weights stay live meanwhile.
            for (int ci = grp; ci < args.bn / 8;
                 ci += NUM_XFORM_WARPS / 4, yc += chunk_step, left -= 8 * (NUM_XFORM_WARPS / 4)) {
                uint32_t v[8];
                tmem_ld_x8(tmem + lane_base + ACC_COL + 8u * ci, v);
                tmem_wait_ld();
                if (row_ok) {
                    float *p = yc;
#pragma unroll
                    for (int t = 0; t < 8; ++t, p += N)
                        if (t < left) __stcs(p, __uint_as_float(v[t]));
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty);
            return true;
        };

        // The warp walks the weight stages of all its units in order; per stage it
        // owns at most one block.  A block unpacked into `regs` is stored (issue) and
        // published (finish) before the next stage is unpacked into the same
        // registers: publishing at once, rather than after the next unpack, hands the
        // MMAs their operand a whole unpack earlier, which the shallow A ring needs.
        uint32_t regs[32];
        bool have = false;  // regs hold block have_J
        int have_J = 0;
        int it = 0;
        for (int u = units0; ok && u < nunits; u += ustep, ++it) {
            const int tile = unit_tile(u);
            for (int s = 0; s < nstage; ++s) {
                if (have) {
                    if (!(ok = issue(have_J, regs))) break;
                    finish(have_J);
                    have = false;
                }
                bool nb = false;
                if (!(ok = prepare(tile, s, regs, nb))) break;
                // One accumulator: the previous unit is complete once its last block
                // (published above) has gone through the MMAs; drain it while this
                // unit's first block waits in registers.
                if (nbufs == 1 && s == 0 && it > 0 && !(ok = drain_unit(u - ustep, it - 1))) break;
                if (nb) {
                    have = true;
                    have_J = it * nkb + KB_PER_STAGE * s + grp;
                }
            }
        }
        if (ok && have && (ok = issue(have_J, regs))) finish(have_J);
        if (ok && nbufs == 1 && it > 0) ok = drain_unit(units0 + (it - 1) * ustep, it - 1);
        xform_ok = ok;
        tmem_wait_st();  // no tensor-memory store may be in flight past this point
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const uint32_t quarter = warp & 3;
        const int row = static_cast<int>(quarter * 32 + lane);
        const uint32_t lane_base = (quarter * 32u) << 16;
        const uint32_t rank = S > 1 ? cluster_ctarank() : 0u;
        const int per = split_per(args.bn, S);  // tokens owned by each cluster rank
        const uint32_t part = smem_u32(smem + args.part_off);
        // One unit per CTA and bf16 x: until the accumulator is complete these warps
        // have nothing else to do, so they convert every x slot to fp16 in place
        // as it lands (round to nearest, the range bit of the status word set on an
        // overflow, as the conversion kernel does), then hand it to the MMA warp.
        // Only the token rows of a tile are converted; the other rows are the
        // copies' zero fill, zero in fp16 too.
        if constexpr (!kMulti) {
            if (args.x_convert == 2 && !skip) {
                const int et = static_cast<int>((warp - FIRST_EPI_WARP) * 32 + lane);
                const int x_tile_bytes = args.bn * 128;
                bool big = false, cok = true;
                int xs = 0;
                uint32_t xph = 0;
                for (int u = units0; cok && u < nunits; u += ustep) {
                    const int rows = min(args.bn, args.M - unit_m0(u));  // token rows of this unit's tiles
                    const int chunks = (rows * 8) << cbs;                // 16-byte chunks of a slot's token rows
                    for (int g = 0; g < ngroups; ++g) {
                        if (!(cok = __all_sync(0xffffffffu, wait_bar(x_full + 8 * xs, xph, ctl, WAIT_X_FULL)))) break;
                        uint8_t *slot = x_ring + xs * args.x_stage_bytes;
                        for (int j = et; j < chunks; j += NUM_EPI_WARPS * 32) {
                            uint4 *chunk = reinterpret_cast<uint4 *>(slot + (j / (rows * 8)) * x_tile_bytes) + j % (rows * 8);
                            const uint4 v = *chunk;
                            const uint32_t src[4] = {v.x, v.y, v.z, v.w};
                            uint32_t dst[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float lo = __uint_as_float(src[e] << 16);
                                const float hi = __uint_as_float(src[e] & 0xFFFF0000u);
                                big |= !(fabsf(lo) < 65520.f) || !(fabsf(hi) < 65520.f);
                                dst[e] = as_u32(__floats2half2_rn(lo, hi));
                            }
                            *chunk = make_uint4(dst[0], dst[1], dst[2], dst[3]);
                        }
                        fence_proxy_async_smem();  // read by the tensor core next
                        __syncwarp();
                        if (lane == 0) mbar_arrive(x_conv + 8 * xs);
                        if (++xs == args.x_stages) { xs = 0; xph ^= 1; }
                    }
                }
                if (__any_sync(0xffffffffu, big) && lane == 0) atomicOr(args.status, kStatusRangeBit);
            }
        }
        // Two accumulators: these warps finish every unit but the CTA's last one
        // (which all transform warps finish together after the main loop).
        if (split_mbar) cluster_wait();
        bool ok = !skip && nbufs == 2;
        int it = 0;
        for (int u = units0; kMulti && ok && u + ustep < nunits; u += ustep, ++it) {
            const int tile = unit_tile(u), m0 = unit_m0(u);
            const int R = tile_rows(args.N, tile);
            const int b = nbufs == 2 ? (it & 1) : 0;
            const int use = nbufs == 2 ? (it >> 1) : it;
            if (!(ok = __all_sync(0xffffffffu, wait_bar<false, true>(acc_full + 8 * b, use & 1, ctl, WAIT_ACC_FULL))))
                break;
            tc_fence_after();
            const uint32_t dcol = tmem + lane_base + ACC_COL + ACC_STRIDE * static_cast<uint32_t>(b);
            if (S == 1) {
                const int64_t n = static_cast<int64_t>(tile) * TILE_ROWS + row;
                for (int c0 = 0; c0 < args.bn; c0 += 32) {
                    uint32_t v[32];
                    tmem_ld_x16(dcol + c0, *reinterpret_cast<uint32_t(*)[16]>(v));
                    const bool two = c0 + 16 < args.bn;
                    if (two) tmem_ld_x16(dcol + c0 + 16, *reinterpret_cast<uint32_t(*)[16]>(v + 16));
                    tmem_wait_ld();
                    if (row < R) {
                        float *yc = unit_y(u) + static_cast<int64_t>(m0 + c0) * args.N + n;
                        const int nt = min(two ? 32 : 16, args.M - (m0 + c0));
#pragma unroll
                        for (int t = 0; t < 32; ++t)
                            if (t < nt) __stcs(yc + static_cast<int64_t>(t) * args.N, __uint_as_float(v[t]));
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acc_empty + 8 * b);
            } else {
                // Split-K through distributed shared memory.  Rank q owns tokens
                // [q*per, q*per + per) of the tile.  Each CTA pushes its partial for
                // every token, quad by quad, into the owner's buffer (source rank
                // `rank`'s region, see split_per) once the owners have consumed the
                // previous unit (part_free), then tells the owners (part_full); each
                // owner sums its tokens over the source ranks in rank order
                // (deterministic) and writes y.
                if (it > 0 && !(ok = __all_sync(0xffffffffu, wait_bar_cluster(part_free, (it - 1) & 1, ctl, WAIT_PART))))
                    break;
                int owner = 0, tt = 0;  // owner rank of the next quad, and its first token there
                uint32_t dst = map_shared_rank(part, 0) +
                               static_cast<uint32_t>(((static_cast<int>(rank) * per) / 4 * TILE_ROWS + row) * 16);
                for (int c0 = 0; c0 < args.bn; c0 += 16) {
                    uint32_t v[16];
                    tmem_ld_x16(dcol + c0, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        st_shared_cluster_f32x4(dst, v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                        dst += TILE_ROWS * 16;
                        if ((tt += 4) == per) {  // the next quad belongs to the next rank (if any)
                            tt = 0;
                            if (++owner < S)
                                dst = map_shared_rank(part, owner) +
                                      static_cast<uint32_t>(((static_cast<int>(rank) * per) / 4 * TILE_ROWS + row) * 16);
                        }
                    }
                }
                tc_fence_before();
                fence_acq_rel_cluster();  // every lane's remote stores before lane 0's release
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(acc_empty + 8 * b);
                    for (int q = 0; q < S; ++q) mbar_arrive_remote(map_shared_rank(part_full, q));
                }
                if (!(ok = __all_sync(0xffffffffu, wait_bar_cluster(part_full, it & 1, ctl, WAIT_PART)))) break;
                const int t0 = min(args.bn, static_cast<int>(rank) * per);
                const int t1 = min(args.bn, t0 + per);
                reduce_quads(reinterpret_cast<const float4 *>(smem + args.part_off), S, per, t0, t1,
                             static_cast<int>((warp - FIRST_EPI_WARP) * 32 + lane), NUM_EPI_WARPS * 32,
                             unit_y(u), m0, tile, R, args.M, args.N);
                // The buffer may be refilled once every epilogue warp here has read it.
                fence_acq_rel_cluster();
                __syncwarp();
                if (lane == 0)
                    for (int q = 0; q < S; ++q) mbar_arrive_remote(map_shared_rank(part_free, q));
            }
        }
        // The owners arrive on this CTA's part_free once they have read the partials
        // of the last unit pushed from here: wait for that before the CTA may exit.
        if (ok && S > 1 && it > 0) __all_sync(0xffffffffu, wait_bar_cluster(part_free, (it - 1) & 1, ctl, WAIT_PART));
        tc_fence_before();
    }

    // Two accumulators: the CTA's last unit, finished by the transform warps.  With
    // split-K each transform warp pushes its partials into the owners' buffers,
    // arrives on the owners' part_last barrier, and the non-epilogue warps of every
    // CTA then sum its tokens over the ranks in rank order and write y.  With a
    // partial buffer of its own (several units per CTA) the epilogue warps may still
    // be reducing the previous unit through it, so the last unit's partials go to a
    // second buffer at the start of the owners' rings instead: a CTA's rings are
    // idle once its last unit's MMAs are done, which it tells every rank through
    // rings_idle, and the push waits until all ranks have.  With the buffer
    // overlaying the rings (one unit per CTA), a first cluster barrier makes sure
    // every CTA's rings are idle before the push and a second one that the pushes
    // have landed.
    if (!split_mbar) __syncthreads();
    if (nbufs == 2 && n_mine > 0) {
        const int lit = n_mine - 1;
        const int lu = units0 + lit * ustep;
        const int tile = unit_tile(lu), m0 = unit_m0(lu);
        const int R = tile_rows(args.N, tile);
        const int b = lit & 1;
        const bool xf = warp >= FIRST_XFORM_WARP && warp < FIRST_EPI_WARP;
        const uint32_t xw = warp - FIRST_XFORM_WARP;
        const int grp = static_cast<int>(xw >> 2);
        const uint32_t quarter = warp & 3;
        const int row = static_cast<int>(quarter * 32 + lane);
        const uint32_t dcol = tmem + ((quarter * 32u) << 16) + ACC_COL + ACC_STRIDE * static_cast<uint32_t>(b);
        bool acc_ok = false;
        if (xf && xform_ok)
            acc_ok = __all_sync(0xffffffffu, wait_bar(acc_full + 8 * b, (lit >> 1) & 1, ctl, WAIT_ACC_FULL));
        if (S == 1) {
            if (acc_ok) {
                tc_fence_after();
                const int64_t n = static_cast<int64_t>(tile) * TILE_ROWS + row;
                for (int ci = grp; ci < args.bn / 16; ci += NUM_XFORM_WARPS / 4) {
                    uint32_t v[16];
                    tmem_ld_x16(dcol + 16u * ci, v);
                    tmem_wait_ld();
                    if (row < R) {
                        const int mb = m0 + 16 * ci;
#pragma unroll
                        for (int t = 0; t < 16; ++t)
                            if (mb + t < args.M)
                                __stcs(unit_y(lu) + static_cast<int64_t>(mb + t) * args.N + n, __uint_as_float(v[t]));
                    }
                }
                tc_fence_before();
            }
        } else if (!split_mbar) {
            // One unit per CTA: every CTA's rings are idle now (its MMAs are done and
            // all its warps passed the barrier above), so each writes its partial
            // tile into its own rings, [token][row]; after a cluster barrier (release
            // / acquire) rank q sums its tokens over the ranks' shared memory in rank
            // order and writes y; a last barrier keeps every CTA's shared memory alive
            // until its peers have read it (a thread arrives after storing the sums
            // of everything it read, so that arrival needs no release).
            const uint32_t rank = cluster_ctarank();
            const int per = (args.bn + S - 1) / S;
            float *own = reinterpret_cast<float *>(smem);
            if (xf && acc_ok && !aborted(ctl)) {
                tc_fence_after();
                for (int ci = grp; ci < args.bn / 16; ci += NUM_XFORM_WARPS / 4) {
                    uint32_t v[16];
                    tmem_ld_x16(dcol + 16u * ci, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int t = 0; t < 16; ++t) own[(16 * ci + t) * TILE_ROWS + row] = __uint_as_float(v[t]);
                }
                tc_fence_before();
            }
            __syncwarp();
            cluster_sync();
            const int t0 = min(args.bn, static_cast<int>(rank) * per);
            const int t1 = min(args.bn, t0 + per);
            if (!aborted(ctl)) {
                const uint32_t own_addr = smem_u32(own);
                const int items = (t1 - t0) * (TILE_ROWS / 4);
                for (int itm = threadIdx.x; itm < items; itm += NUM_THREADS) {
                    const int tt = t0 + itm / (TILE_ROWS / 4);
                    const int r4 = 4 * (itm % (TILE_ROWS / 4));
                    const uint32_t off = static_cast<uint32_t>((tt * TILE_ROWS + r4) * 4);
                    // All S remote loads are issued before the first sum needs one
                    // (a dependent load-add chain costs S round trips over the cluster).
                    float4 pv[MAX_SPLITS];
#pragma unroll
                    for (int q = 0; q < MAX_SPLITS; ++q)
                        if (q < S) pv[q] = ld_shared_cluster_f4(map_shared_rank(own_addr + off, static_cast<uint32_t>(q)));
                    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int q = 0; q < MAX_SPLITS; ++q)
                        if (q < S) { acc.x += pv[q].x; acc.y += pv[q].y; acc.z += pv[q].z; acc.w += pv[q].w; }
                    const int m = m0 + tt;
                    if (m < args.M) {
                        float *yr = unit_y(lu) + static_cast<int64_t>(m) * args.N + static_cast<int64_t>(tile) * TILE_ROWS;
                        const float a4[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            if (r4 + e < R) __stcs(yr + r4 + e, a4[e]);
                    }
                }
            }
            __syncwarp();
            cluster_arrive_relaxed();
            cluster_wait();
        } else {
            // Several units per CTA, the last one through the partial buffers at the
            // start of the owners' rings (see above).
            const uint32_t rank = cluster_ctarank();
            const int per = split_per(args.bn, S);
            const uint32_t part = smem_u32(smem);
            if (cluster_wait_due) cluster_wait();  // (the epilogue warps waited already)
            cluster_wait_due = false;
            if (xf) {
                // This CTA's MMAs are done (or failed): its rings are idle.
                if (warp == FIRST_XFORM_WARP && lane == 0)
                    for (int q = 0; q < S; ++q) mbar_arrive_remote(map_shared_rank(rings_idle, q));
                const bool push_ok = __all_sync(0xffffffffu, wait_bar<true, false>(rings_idle, 0, ctl, WAIT_PART)) && acc_ok;
                if (push_ok && !aborted(ctl)) {
                    tc_fence_after();
                    // Quad Q (tokens 4Q .. 4Q+3) goes to the rank owning it; this
                    // warp's quads are grp, grp + 4, .. (16 tokens apart).
                    int owner = (4 * grp) / per, tt = 4 * grp - owner * per;
                    for (int Q = grp; Q < args.bn / 4; Q += NUM_XFORM_WARPS / 4) {
                        uint32_t v[4];
                        tmem_ld_x4(dcol + 4u * Q, v);
                        tmem_wait_ld();
                        st_shared_cluster_f32x4(
                            map_shared_rank(part, owner) +
                                static_cast<uint32_t>((((static_cast<int>(rank) * per + tt) / 4) * TILE_ROWS + row) * 16),
                            v[0], v[1], v[2], v[3]);
                        for (tt += 16; tt >= per && owner + 1 < S; tt -= per) ++owner;
                    }
                    tc_fence_before();
                }
                // Arrive even after a failure (the status word already says so), so
                // that the owners need not wait out their own timeouts.
                fence_acq_rel_cluster();
                __syncwarp();
                if (lane == 0)
                    for (int q = 0; q < S; ++q) mbar_arrive_remote(map_shared_rank(part_last, q));
            }
            // The epilogue warps take no part: they may still be busy.
            const bool summer = warp < FIRST_EPI_WARP;
            const bool all_in = summer && __all_sync(0xffffffffu, wait_bar<true, false>(part_last, 0, ctl, WAIT_PART));
            const int t0 = min(args.bn, static_cast<int>(rank) * per);
            const int t1 = min(args.bn, t0 + per);
            if (summer && all_in && !aborted(ctl))
                reduce_quads(reinterpret_cast<const float4 *>(smem), S, per, t0, t1, static_cast<int>(threadIdx.x),
                             FIRST_EPI_WARP * 32, unit_y(lu), m0, tile, R, args.M, args.N);
        }
    }
    // With split-K, no CTA of the cluster leaves before every peer is done with
    // its shared memory.  With one unit per CTA every thread passes two full
    // cluster barriers on every path and the remote stores happen between them.
    // With a partial buffer of its own, on the normal path every remote write or
    // arrival aimed at a CTA is one that a thread there waited for, but after a
    // timeout those waits are skipped, so a full cluster barrier (release /
    // acquire) closes every path.  Every thread of every CTA reaches it: all
    // waits before it are bounded.
    if (split_mbar) {
        __syncwarp();
        if (cluster_wait_due) cluster_wait();
        cluster_sync();
    }
    // Every read of tensor memory (epilogue and transform warps) is done before it
    // is released.
    __syncthreads();
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
// x as [batch][M][K] (rank 2 when batch == 1), box 64 K x bn tokens.
static int encode_x_map(CUtensorMap *map, const void *x, int64_t M, int64_t K, int bn, bool bf16, int64_t batch) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return QWP_ERR_CUDA;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M), static_cast<cuuint64_t>(batch)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(K) * 2, static_cast<cuuint64_t>(M) * K * 2};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(CHUNK_K), static_cast<cuuint32_t>(bn), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                    batch > 1 ? 3 : 2,
                    const_cast<void *>(x), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? QWP_OK : QWP_ERR_CUDA;
}

// Token tile: the fewest tiles of at most `cap` tokens, each a multiple of 16.
static int choose_bn(int64_t M, int cap) {
    const int64_t tiles = (M + cap - 1) / cap;
    const int64_t per = (M + tiles - 1) / tiles;
    return static_cast<int>((per + 15) / 16 * 16);
}

struct DeviceInfo {
    int sms = 0;
    int slots[NUM_FMTS][MAX_SPLITS + 1] = {};  // [format][S]: CTAs resident at once with clusters of S
    bool ready[NUM_FMTS] = {};
};

// The kernel instances of one format and batch mode: lift their dynamic
// shared-memory limit to SMEM_BYTES (non-zero on failure).
template <int kFmt, bool kBatch>
static int allow_smem() {
    const auto lift = [](const void *k) {
        return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) != cudaSuccess;
    };
    return lift(reinterpret_cast<const void *>(qwp_gemm_kernel<kFmt, true, kBatch, true>)) ||
           lift(reinterpret_cast<const void *>(qwp_gemm_kernel<kFmt, true, kBatch, false>)) ||
           lift(reinterpret_cast<const void *>(qwp_gemm_kernel<kFmt, false, kBatch, true>));
}

// Launch of the instance for a plan: two accumulators or one, several units per
// CTA or at most one.
template <int kFmt, bool kBatch>
static cudaError_t launch_instance(const cudaLaunchConfig_t &cfg, const CUtensorMap &map, const GemmArgs &a,
                                   bool multi) {
    if (a.acc_bufs != 2) return cudaLaunchKernelEx(&cfg, qwp_gemm_kernel<kFmt, false, kBatch, true>, map, a);
    return multi ? cudaLaunchKernelEx(&cfg, qwp_gemm_kernel<kFmt, true, kBatch, true>, map, a)
                 : cudaLaunchKernelEx(&cfg, qwp_gemm_kernel<kFmt, true, kBatch, false>, map, a);
}

template <int kFmt>
static int device_info(DeviceInfo *&out) {
    static DeviceInfo info[64];
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return QWP_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    DeviceInfo &d = info[dev];
    if (!d.ready[kFmt]) {
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return QWP_ERR_CUDA;
        if (allow_smem<kFmt, false>()) return QWP_ERR_CUDA;
        if constexpr (kFmt == FMT_Q4K)  // the strided-batch kernels (same resources, same slots)
            if (allow_smem<kFmt, true>()) return QWP_ERR_CUDA;
        d.slots[kFmt][1] = d.sms;
        for (int S = 2; S <= MAX_SPLITS; ++S) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(1, 1, S * 64);
            cfg.blockDim = dim3(block_threads(true), 1, 1);
            cfg.dynamicSmemBytes = SMEM_BYTES;
            cudaLaunchAttribute attr;
            attr.id = cudaLaunchAttributeClusterDimension;
            attr.val.clusterDim.x = 1;
            attr.val.clusterDim.y = 1;
            attr.val.clusterDim.z = S;
            cfg.attrs = &attr;
            cfg.numAttrs = 1;
            int clusters = 0;
            if (cudaOccupancyMaxActiveClusters(&clusters, qwp_gemm_kernel<kFmt, true>, &cfg) != cudaSuccess) {
                cudaGetLastError();
                clusters = 0;
            }
            d.slots[kFmt][S] = clusters * S;
        }
        d.ready[kFmt] = true;
    }
    out = &d;
    return QWP_OK;
}

// Launch plan of one GEMM: split-K factor S (cluster size), number of resident
// clusters, commit-group size and the shared-memory layout.
struct Plan {
    int S = 1, clusters = 0, cbs = 0, x_stages = 0, w_stages = 0, part_off = 0;
    bool overlay = false;
    double cost = 1e30;
};

// Shared-memory layout for a given split and commit-group size; false if the
// rings would be too shallow.  With split-K and several units per CTA (`reserve`)
// the partial buffer gets space of its own (peers push into it while this CTA's
// rings are busy); with one unit per CTA it overlays the rings, idle by then.
static bool layout(int bn, int S, int cbs, int w_stage_bytes, bool reserve, Plan &p) {
    const int x_stage = (bn * 128) << cbs;
    int avail = RING_BYTES;
    if (S > 1 && reserve) {
        const int part_bytes = S * split_per(bn, S) * TILE_ROWS * 4;
        avail = (RING_BYTES - part_bytes) & ~1023;
    }
    // Keep room for 4 weight stages if the x ring still gets 2 slots, else for 2.
    int xs = std::min(A_STAGES >> cbs, (avail - 4 * w_stage_bytes) / x_stage);
    if (xs < 2) xs = std::min(A_STAGES >> cbs, (avail - 2 * w_stage_bytes) / x_stage);
    if (xs < 2 && !(xs == 1 && cbs == 0)) return false;
    if (xs < 1) return false;
    const int ws = std::min(W_MAX_STAGES, (avail - xs * x_stage) / w_stage_bytes);
    if (ws < 2) return false;
    p.cbs = cbs;
    p.x_stages = xs;
    p.w_stages = ws;
    p.part_off = (S > 1 && reserve) ? avail : 0;
    return true;
}

// Units are (row tile, token tile) pairs; a cluster of S CTAs splits each unit's
// K range S ways and the clusters loop over the units.  Time is modelled as
// (rounds of units per cluster) x (weight stages per CTA and unit + a small
// per-unit cost), plus a fixed cost for the reduction when S > 1; the cheapest
// plan wins.  Commit groups are 4 blocks for short MMAs (N <= 128), else 2,
// never more than divides the K blocks (every split's block count is then a
// multiple too) and smaller if the x ring would not fit.
static Plan choose_plan(const int *slots, int64_t units, int nstages, int64_t nkb_total, int bn,
                        int w_stage_bytes) {
    Plan best;
    for (int S = 1; S <= MAX_SPLITS && S <= nstages; ++S) {
        const int per = (nstages + S - 1) / S;
        if ((nstages + per - 1) / per != S || slots[S] < S) continue;  // no empty or duplicate splits
        if (S > 1 && bn > static_cast<int>(ACC_STRIDE)) continue;      // partial buffer too large
        Plan p;
        p.S = S;
        p.clusters = static_cast<int>(std::min<int64_t>(units, slots[S] / S));
        const int64_t rounds = (units + p.clusters - 1) / p.clusters;
        int cbs = bn <= 128 ? 2 : 1;
        while (cbs > 0 && nkb_total % (1 << cbs)) --cbs;
        while (!layout(bn, S, cbs, w_stage_bytes, rounds > 1, p) && cbs > 0) --cbs;
        p.overlay = S > 1 && rounds == 1;
        if (p.w_stages == 0) continue;
        p.cost = static_cast<double>(rounds) * (per + 0.25) + (S > 1 ? 1.0 : 0.0);
        if (p.cost < best.cost - 1e-9) best = p;
    }
    return best;
}

// Bytes of one weight stage (128 rows x 256 K) in format kFmt.
template <int kFmt>
constexpr int weight_stage_bytes() {
    return kFmt == FMT_Q4K   ? TILE_ROWS * Q4K_BLOCK_BYTES
           : kFmt == FMT_Q6K ? TILE_ROWS * Q6K_BLOCK_BYTES
                             : TILE_ROWS * CHUNK_ROW_BYTES * KB_PER_STAGE;
}

// Token tile, launch plan and unit count of an M x N x K product in format kFmt
// on the current device (host only).
template <int kFmt>
static int plan_gemm(int64_t M, int64_t N, int64_t K, Plan &plan, int &bn, int64_t &units, int64_t batch = 1) {
    DeviceInfo *info = nullptr;
    const int rc = device_info<kFmt>(info);
    if (rc) return rc;
    const int64_t row_tiles = (N + TILE_ROWS - 1) / TILE_ROWS;
    const int64_t nkb_total = K / CHUNK_K;
    const int nstages = static_cast<int>((nkb_total + KB_PER_STAGE - 1) / KB_PER_STAGE);
    const int w_stage_bytes = weight_stage_bytes<kFmt>();
    // Token tile: the widest (fewest tiles of <= 256 tokens) unless tiles of <= 128,
    // which allow split-K and two accumulators, give a cheaper plan (few units).
    bn = choose_bn(M, BN_MAX);
    int64_t tok_tiles = (M + bn - 1) / bn;
    if (batch * row_tiles * tok_tiles > 0x7fffffff) return QWP_ERR_UNSUPPORTED_SHAPE;
    plan = choose_plan(info->slots[kFmt], batch * row_tiles * tok_tiles, nstages, nkb_total, bn, w_stage_bytes);
    if (bn > static_cast<int>(ACC_STRIDE)) {
        const int bn2 = choose_bn(M, static_cast<int>(ACC_STRIDE));
        const int64_t tt2 = (M + bn2 - 1) / bn2;
        if (batch * row_tiles * tt2 <= 0x7fffffff) {
            const Plan p2 = choose_plan(info->slots[kFmt], batch * row_tiles * tt2, nstages, nkb_total, bn2, w_stage_bytes);
            if (p2.cost < plan.cost - 1e-9) {
                plan = p2;
                bn = bn2;
                tok_tiles = tt2;
            }
        }
    }
    if (plan.clusters <= 0) return QWP_ERR_UNSUPPORTED_SHAPE;
    units = row_tiles * tok_tiles;  // of one problem
    return QWP_OK;
}

// How the prefill kernel converts bf16 x itself for a plan: 2 when every CTA
// runs at most one unit with two accumulators (the epilogue warps are free until
// the end) and its x is small, 1 for one token (the MMA warp), else 0 (the
// caller converts x first).  Each CTA converts the x of its own unit and K range,
// so CTAs that share a token tile convert it again; measured on GB300, up to
// 32 KB per CTA (64 KB with at most 16 token rows) the launch saved over the
// conversion kernel (Q4_K M=8 N4096 K4096 11.4 -> 10.0 us, M=32 N2048 K2048 8.4
// -> 8.0 us, M=8 N4096 K12288 20.3 -> 19.3 us, M=16 N6144 K4096 15.4 -> 15.0
// us), while 64 KB of 32 rows (M=32 N4096 K4096) took 11.4 -> 11.8 us, 229 KB
// (M=105, N4096, K4096, split-K 4) 13.8 -> 21.5 us and 131 KB (a batch of eight
// M=32 N2048 K2048 products) 17.5 -> 20.7 us.
static int x_convert_mode(const Plan &plan, int bn, int64_t units_all, int64_t M, int64_t K) {
    const int64_t k_cta = (K / CHUNK_K + plan.S - 1) / plan.S * CHUNK_K;  // K of one split, at most
    const int64_t rows = std::min<int64_t>(bn, M);
    const int64_t bytes = rows * k_cta * 2;
    const bool small = bytes <= 32 * 1024 || (rows <= 16 && bytes <= 64 * 1024);
    if (units_all <= plan.clusters && bn <= static_cast<int>(ACC_STRIDE) && small) return 2;
    return M <= CONVERT_MAX_M ? 1 : 0;
}

// Whether a bf16-x product of this shape (one problem, or a strided batch) is
// converted inside the prefill kernel (no conversion kernel, no scratch).
template <int kFmt>
static bool converts_in_kernel(int64_t M, int64_t N, int64_t K, int64_t batch = 1) {
    Plan plan;
    int bn = 0;
    int64_t units = 0;
    if (plan_gemm<kFmt>(M, N, K, plan, bn, units, batch)) return false;
    return x_convert_mode(plan, bn, batch * units, M, K) != 0;
}

// x is fp16 [M, K], or bf16 when x_bf16 (converted in shared memory by the
// kernel, see x_convert_mode; QWP_ERR_UNSUPPORTED_SHAPE if the plan allows
// neither way).  Launched with programmatic stream serialization: the kernel's
// set-up overlaps the end of the grid before it.
template <int kFmt>
static int launch_gemm(const void *w, const void *scales, const uint8_t *zeros, const void *x,
                       float *y, int64_t M, int64_t N, int64_t K, int64_t group, cudaStream_t stream,
                       bool x_bf16 = false, int64_t batch = 1, int64_t w_batch_bytes = 0) {
    int rc = check_device();
    if (rc) return rc;
    uint32_t *status = status_word();
    if (!status) return QWP_ERR_CUDA;
    Plan plan;
    int bn = 0;
    int64_t units = 0;
    if ((rc = plan_gemm<kFmt>(M, N, K, plan, bn, units, batch))) return rc;
    const int64_t row_tiles = (N + TILE_ROWS - 1) / TILE_ROWS;
    const int nstages = static_cast<int>((K / CHUNK_K + KB_PER_STAGE - 1) / KB_PER_STAGE);
    const int conv = x_bf16 ? x_convert_mode(plan, bn, batch * units, M, K) : 0;
    if (x_bf16 && !conv) return QWP_ERR_UNSUPPORTED_SHAPE;
    CUtensorMap map;
    if ((rc = encode_x_map(&map, x, M, K, bn, x_bf16, batch))) return rc;

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
    a.timeout_cycles = ns_to_cycles(wait_timeout_ns());
    a.drain_cycles = ns_to_cycles(kDefaultTimeoutNs);
    a.cb_shift = plan.cbs;
    a.x_stage_bytes = (bn * 128) << plan.cbs;
    a.w_stage_bytes = weight_stage_bytes<kFmt>();
    a.x_stages = plan.x_stages;
    a.w_stages = plan.w_stages;
    a.part_off = plan.part_off;
    a.part_overlay = plan.overlay ? 1 : 0;
    a.x_convert = conv;
    a.splits = plan.S;
    a.kb_per_split = ((nstages + plan.S - 1) / plan.S) * KB_PER_STAGE;
    a.n_units = static_cast<int>(batch * units);
    a.batch = static_cast<int>(batch);
    a.units_per_problem = static_cast<int>(units);
    a.w_batch_bytes = w_batch_bytes;
    a.row_tiles = static_cast<int>(row_tiles);
    a.acc_bufs = bn <= static_cast<int>(ACC_STRIDE) ? 2 : 1;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(plan.clusters), 1, plan.S);
    cfg.blockDim = dim3(block_threads(a.acc_bufs == 2), 1, 1);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attrs[2];
    unsigned nattr = 0;
    if (plan.S > 1) {
        attrs[nattr].id = cudaLaunchAttributeClusterDimension;
        attrs[nattr].val.clusterDim.x = 1;
        attrs[nattr].val.clusterDim.y = 1;
        attrs[nattr].val.clusterDim.z = plan.S;
        ++nattr;
    }
    attrs[nattr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[nattr].val.programmaticStreamSerializationAllowed = 1;
    ++nattr;
    cfg.attrs = attrs;
    cfg.numAttrs = nattr;
    // Several units per CTA when the units outnumber the clusters.
    const bool multi = static_cast<int64_t>(a.n_units) > static_cast<int64_t>(plan.clusters);
    cudaError_t le;
    if constexpr (kFmt == FMT_Q4K) {
        le = batch > 1 ? launch_instance<kFmt, true>(cfg, map, a, multi) : launch_instance<kFmt, false>(cfg, map, a, multi);
    } else {
        if (batch > 1) return QWP_ERR_UNSUPPORTED_SHAPE;  // strided batches are Q4_K only
        le = launch_instance<kFmt, false>(cfg, map, a, multi);
    }
    if (le != cudaSuccess) {
        cudaGetLastError();
        return QWP_ERR_CUDA;
    }
    return QWP_OK;
}

int launch_q4k_prefill_fixed(const void *w, const void *x, void *x16, float *y, int64_t M, int64_t N, int64_t K,
                             cudaStream_t stream) {
    int rc = check_device();
    if (rc) return rc;
    if (converts_in_kernel<FMT_Q4K>(M, N, K))
        return launch_gemm<FMT_Q4K>(w, nullptr, nullptr, x, y, M, N, K, 0, stream, true);
    if ((rc = launch_bf16_to_f16(x, x16, M * K, stream))) return rc;
    return launch_gemm<FMT_Q4K>(w, nullptr, nullptr, x16, y, M, N, K, 0, stream);
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

// Decode-shaped calls (at most 8 tokens, K a multiple of 256) go to the decode
// kernel, which streams the same repacked weights without the tensor-memory
// pipeline (and converts bf16 activations itself); its scratch comes from the pool.
static bool decode_shaped(int fmt, int64_t M, int64_t N, int64_t K) { return decode_selected(fmt, M, N, K); }

static int run_decode(int fmt, const void *w, const void *scales, const uint8_t *zeros, const void *x, bool x_bf16,
                      float *y, int64_t M, int64_t N, int64_t K, int64_t group, cudaStream_t s) {
    int rc = check_device();
    if (rc) return rc;
    const size_t bytes = decode_scratch_bytes(fmt, N, K);
    if (!bytes) return QWP_ERR_CUDA;
    cudaMemPool_t pool;
    if ((rc = scratch_pool(&pool))) return rc;
    void *scratch = nullptr;
    if (cudaMallocFromPoolAsync(&scratch, bytes, pool, s) != cudaSuccess) {
        cudaGetLastError();
        return QWP_ERR_CUDA;
    }
    rc = launch_decode(fmt, w, scales, zeros, x, x_bf16, y, M, N, K, group, scratch, bytes, s);
    if (cudaFreeAsync(scratch, s) != cudaSuccess && !rc) rc = QWP_ERR_CUDA;
    return rc;
}

extern "C" int q4k_gemm_f16(const void *w_tiled, const void *x, float *y, int64_t M, int64_t N,
                            int64_t K, void *stream) {
    if (K % Q4K_BLOCK || K == 0) return K < 0 ? QWP_ERR_INVALID_ARG : QWP_ERR_UNSUPPORTED_SHAPE;
    int rc = gemm_shape_checks(w_tiled, x, y, M, N, K);
    if (rc || M == 0 || N == 0) return rc;
    if (decode_shaped(DFMT_Q4K, M, N, K))
        return run_decode(DFMT_Q4K, w_tiled, nullptr, nullptr, x, false, y, M, N, K, 0,
                          static_cast<cudaStream_t>(stream));
    if (skinny_selected(DFMT_Q4K, M, N, K))
        return launch_skinny(w_tiled, x, false, y, M, N, K, static_cast<cudaStream_t>(stream));
    return launch_gemm<FMT_Q4K>(w_tiled, nullptr, nullptr, x, y, M, N, K, 0,
                             static_cast<cudaStream_t>(stream));
}

extern "C" int q4k_gemm(const void *w_tiled, const void *x, float *y, int64_t M, int64_t N,
                        int64_t K, void *stream) {
    if (K % Q4K_BLOCK || K == 0) return K < 0 ? QWP_ERR_INVALID_ARG : QWP_ERR_UNSUPPORTED_SHAPE;
    int rc = gemm_shape_checks(w_tiled, x, y, M, N, K);
    if (rc || M == 0 || N == 0) return rc;
    if ((rc = check_device())) return rc;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (decode_shaped(DFMT_Q4K, M, N, K)) return run_decode(DFMT_Q4K, w_tiled, nullptr, nullptr, x, true, y, M, N, K, 0, s);
    if (skinny_selected(DFMT_Q4K, M, N, K)) return launch_skinny(w_tiled, x, true, y, M, N, K, s);
    // One unit per CTA, or one token: the kernel converts x itself (no conversion
    // kernel, no scratch).
    if (converts_in_kernel<FMT_Q4K>(M, N, K))
        return launch_gemm<FMT_Q4K>(w_tiled, nullptr, nullptr, x, y, M, N, K, 0, s, true);
    cudaMemPool_t pool;
    if ((rc = scratch_pool(&pool))) return rc;
    void *x16 = nullptr;
    if (cudaMallocFromPoolAsync(&x16, static_cast<size_t>(M) * K * 2, pool, s) != cudaSuccess) {
        cudaGetLastError();
        return QWP_ERR_CUDA;
    }
    rc = launch_bf16_to_f16(x, x16, M * K, s);
    if (!rc) rc = launch_gemm<FMT_Q4K>(w_tiled, nullptr, nullptr, x16, y, M, N, K, 0, s);
    if (cudaFreeAsync(x16, s) != cudaSuccess && !rc) rc = QWP_ERR_CUDA;
    return rc;
}

// A batch of independent Q4_K products of one shape in one launch: problem p's
// repacked weights at w_tiled + p*q4k_repacked_bytes(N, K), its x at x + p*M*K and
// its y at y + p*M*N; the units of all problems share the persistent grid.
static int q4k_batched(const void *w_tiled, const void *x, bool x_bf16, float *y, int64_t batch, int64_t M,
                       int64_t N, int64_t K, void *stream) {
    if (batch < 0 || M < 0 || N < 0 || K < 0) return QWP_ERR_INVALID_ARG;
    if (K % Q4K_BLOCK || K == 0) return QWP_ERR_UNSUPPORTED_SHAPE;
    if (batch == 0) return QWP_OK;
    int rc = gemm_shape_checks(w_tiled, x, y, M, N, K);
    if (rc || M == 0 || N == 0) return rc;
    if (batch > 65535 || batch * M * K > (int64_t(1) << 40) || batch * M * N > (int64_t(1) << 40))
        return QWP_ERR_UNSUPPORTED_SHAPE;
    if ((rc = check_device())) return rc;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t wbytes = N * (K / Q4K_BLOCK) * Q4K_BLOCK_BYTES;
    if (!x_bf16 || converts_in_kernel<FMT_Q4K>(M, N, K, batch))
        return launch_gemm<FMT_Q4K>(w_tiled, nullptr, nullptr, x, y, M, N, K, 0, s, x_bf16, batch, wbytes);
    cudaMemPool_t pool;
    if ((rc = scratch_pool(&pool))) return rc;
    void *x16 = nullptr;
    if (cudaMallocFromPoolAsync(&x16, static_cast<size_t>(batch * M * K) * 2, pool, s) != cudaSuccess) {
        cudaGetLastError();
        return QWP_ERR_CUDA;
    }
    rc = launch_bf16_to_f16(x, x16, batch * M * K, s);
    if (!rc) rc = launch_gemm<FMT_Q4K>(w_tiled, nullptr, nullptr, x16, y, M, N, K, 0, s, false, batch, wbytes);
    if (cudaFreeAsync(x16, s) != cudaSuccess && !rc) rc = QWP_ERR_CUDA;
    return rc;
}

extern "C" int q4k_gemm_batched(const void *w_tiled, const void *x, float *y, int64_t batch, int64_t M, int64_t N,
                                int64_t K, void *stream) {
    return q4k_batched(w_tiled, x, true, y, batch, M, N, K, stream);
}

extern "C" int q4k_gemm_batched_f16(const void *w_tiled, const void *x, float *y, int64_t batch, int64_t M,
                                    int64_t N, int64_t K, void *stream) {
    return q4k_batched(w_tiled, x, false, y, batch, M, N, K, stream);
}

extern "C" int q4k_q8_gemm(const void *w_tiled, const void *xq, float *y, int64_t M, int64_t N, int64_t K,
                           void *stream) {
    if (K % Q4K_BLOCK || K == 0) return K < 0 ? QWP_ERR_INVALID_ARG : QWP_ERR_UNSUPPORTED_SHAPE;
    int rc = gemm_shape_checks(w_tiled, xq, y, M, N, K);
    if (rc || M == 0 || N == 0) return rc;
    if (M > DECODE_MAX_TOKENS) return QWP_ERR_UNSUPPORTED_SHAPE;
    return run_decode(DFMT_Q4K_Q8, w_tiled, nullptr, nullptr, xq, false, y, M, N, K, 0,
                      static_cast<cudaStream_t>(stream));
}

extern "C" int q6k_gemm_f16(const void *w_tiled, const void *x, float *y, int64_t M, int64_t N,
                            int64_t K, void *stream) {
    if (K % Q4K_BLOCK || K == 0) return K < 0 ? QWP_ERR_INVALID_ARG : QWP_ERR_UNSUPPORTED_SHAPE;
    int rc = gemm_shape_checks(w_tiled, x, y, M, N, K);
    if (rc || M == 0 || N == 0) return rc;
    if (decode_shaped(DFMT_Q6K, M, N, K))
        return run_decode(DFMT_Q6K, w_tiled, nullptr, nullptr, x, false, y, M, N, K, 0,
                          static_cast<cudaStream_t>(stream));
    return launch_gemm<FMT_Q6K>(w_tiled, nullptr, nullptr, x, y, M, N, K, 0,
                                static_cast<cudaStream_t>(stream));
}

extern "C" int q6k_gemm(const void *w_tiled, const void *x, float *y, int64_t M, int64_t N,
                        int64_t K, void *stream) {
    if (K % Q4K_BLOCK || K == 0) return K < 0 ? QWP_ERR_INVALID_ARG : QWP_ERR_UNSUPPORTED_SHAPE;
    int rc = gemm_shape_checks(w_tiled, x, y, M, N, K);
    if (rc || M == 0 || N == 0) return rc;
    if ((rc = check_device())) return rc;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (decode_shaped(DFMT_Q6K, M, N, K)) return run_decode(DFMT_Q6K, w_tiled, nullptr, nullptr, x, true, y, M, N, K, 0, s);
    // One unit per CTA, or one token: the kernel converts x itself (no conversion
    // kernel, no scratch).
    if (converts_in_kernel<FMT_Q6K>(M, N, K))
        return launch_gemm<FMT_Q6K>(w_tiled, nullptr, nullptr, x, y, M, N, K, 0, s, true);
    cudaMemPool_t pool;
    if ((rc = scratch_pool(&pool))) return rc;
    void *x16 = nullptr;
    if (cudaMallocFromPoolAsync(&x16, static_cast<size_t>(M) * K * 2, pool, s) != cudaSuccess) {
        cudaGetLastError();
        return QWP_ERR_CUDA;
    }
    rc = launch_bf16_to_f16(x, x16, M * K, s);
    if (!rc) rc = launch_gemm<FMT_Q6K>(w_tiled, nullptr, nullptr, x16, y, M, N, K, 0, s);
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
    if (!scales) return QWP_ERR_INVALID_ARG;
    if (decode_shaped(DFMT_W4A16, M, N, K))
        return run_decode(DFMT_W4A16, wq_tiled, scales, zeros, x, false, y, M, N, K, group,
                          static_cast<cudaStream_t>(stream));
    return launch_gemm<FMT_W4A16>(wq_tiled, scales, zeros, x, y, M, N, K, group,
                              static_cast<cudaStream_t>(stream));
}

extern "C" int w4a16_gemm_bf16(const void *wq_tiled, const void *scales, const uint8_t *zeros,
                               const void *x, float *y, int64_t M, int64_t N, int64_t K, int64_t group,
                               void *stream) {
    if (group <= 0 || group % CHUNK_K) return QWP_ERR_INVALID_ARG;
    if (K % group || K == 0) return K < 0 ? QWP_ERR_INVALID_ARG : QWP_ERR_UNSUPPORTED_SHAPE;
    int rc = gemm_shape_checks(wq_tiled, x, y, M, N, K);
    if (rc || M == 0 || N == 0) return rc;
    if (!scales) return QWP_ERR_INVALID_ARG;
    if ((rc = check_device())) return rc;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (decode_shaped(DFMT_W4A16, M, N, K)) return run_decode(DFMT_W4A16, wq_tiled, scales, zeros, x, true, y, M, N, K, group, s);
    // One unit per CTA, or one token: the kernel converts x itself (no conversion
    // kernel, no scratch).
    if (converts_in_kernel<FMT_W4A16>(M, N, K))
        return launch_gemm<FMT_W4A16>(wq_tiled, scales, zeros, x, y, M, N, K, group, s, true);
    cudaMemPool_t pool;
    if ((rc = scratch_pool(&pool))) return rc;
    void *x16 = nullptr;
    if (cudaMallocFromPoolAsync(&x16, static_cast<size_t>(M) * K * 2, pool, s) != cudaSuccess) {
        cudaGetLastError();
        return QWP_ERR_CUDA;
    }
    rc = launch_bf16_to_f16(x, x16, M * K, s);
    if (!rc) rc = launch_gemm<FMT_W4A16>(wq_tiled, scales, zeros, x16, y, M, N, K, group, s);
    if (cudaFreeAsync(x16, s) != cudaSuccess && !rc) rc = QWP_ERR_CUDA;
    return rc;
}

extern "C" int qwp_gemm_plan(int format, int64_t M, int64_t N, int64_t K, int32_t *plan_out) {
    if (!plan_out || M < 1 || N < 1 || K < 1) return QWP_ERR_INVALID_ARG;
    if (format != FMT_W4A16 && format != FMT_Q4K && format != FMT_Q6K) return QWP_ERR_INVALID_ARG;
    if (M > (1ll << 30) || N > (1ll << 30) || K > (1ll << 30)) return QWP_ERR_UNSUPPORTED_SHAPE;
    if (K % (format == FMT_W4A16 ? CHUNK_K : Q4K_BLOCK)) return QWP_ERR_UNSUPPORTED_SHAPE;
    for (int i = 0; i < 6; ++i) plan_out[i] = 0;
    if (decode_shaped(format, M, N, K)) {
        plan_out[0] = 2;
        return QWP_OK;
    }
    int rc = check_device();
    if (rc) return rc;
    if (skinny_selected(format, M, N, K)) {
        int dev = 0, sms = 0, S = 1, tm = 0;
        int64_t tiles = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return QWP_ERR_CUDA;
        if ((rc = skinny_plan(M, K, sms, S, tiles, tm))) return rc;
        plan_out[0] = 3;
        plan_out[1] = S;
        plan_out[2] = static_cast<int32_t>(tiles);
        plan_out[3] = tm;
        plan_out[4] = static_cast<int32_t>(tiles);
        plan_out[5] = 1;
        return QWP_OK;
    }
    Plan plan;
    int bn = 0;
    int64_t units = 0;
    rc = format == FMT_Q4K   ? plan_gemm<FMT_Q4K>(M, N, K, plan, bn, units)
         : format == FMT_Q6K ? plan_gemm<FMT_Q6K>(M, N, K, plan, bn, units)
                             : plan_gemm<FMT_W4A16>(M, N, K, plan, bn, units);
    if (rc) return rc;
    plan_out[0] = 1;
    plan_out[1] = plan.S;
    plan_out[2] = plan.clusters;
    plan_out[3] = bn;
    plan_out[4] = static_cast<int32_t>(units);
    plan_out[5] = static_cast<int32_t>((units + plan.clusters - 1) / plan.clusters);
    return QWP_OK;
}
