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
// One CTA computes a 128-row (weights) x BN-token (BN <= 256) tile of y^T:
//   warp 0        producer: one thread issues a bulk copy per 256-wide K
//                 stage of packed weights and a 2-D TMA load (128-byte swizzle)
//                 per 64-wide K block of x;
//   warp 1        allocates tensor memory and one thread issues tcgen05.mma;
//   warps 2..9    transform: thread (quarter q, half h) owns weight row 32q+lane
//                 and half of each 64-wide K block; it unpacks its 32 weights to
//                 bf16 (Q4_K) or fp16 (W4A16) and stores them with tcgen05.st
//                 into the A operand ring in tensor memory;
//                 afterwards the same warps drain the fp32 accumulator
//                 (tcgen05.ld) into y.
// Tensor memory (512 columns): accumulator [128 lanes x BN] at column 0, an
// 8-deep ring of A operand blocks (128 lanes x 64 K = 32 columns) at 256.
// The MMA is D[128 x BN] += A[128 x 16] (tensor memory) . B[BN x 16]^T (shared
// memory), so weights are the M side and tokens the N side: a tile reuses each
// unpacked weight for BN tokens.
//
// Every mbarrier wait is bounded: on expiry the thread records a timeout in
// the library's status word and sets a CTA-wide abort flag; all roles then
// wait (bounded) for their own copies and MMAs in flight, the tensor memory is
// released and the CTA exits.
#include <atomic>
#include <mutex>

#include "qwp_format.cuh"
#include "qwp_internal.h"
#include "qwp_ptx.cuh"

namespace qwp {

constexpr int NUM_XFORM_WARPS = 8;
constexpr int NUM_THREADS = 64 + 32 * NUM_XFORM_WARPS;
constexpr int X_STAGES = 4;
constexpr int W_STAGES = 3;
constexpr int A_STAGES = 8;
constexpr int BN_MAX = 256;
constexpr int X_STAGE_BYTES = BN_MAX * 128;
constexpr int W_STAGE_BYTES = TILE_ROWS * Q4K_BLOCK_BYTES;  // 18432 (W4A16 stages use 16384)
constexpr int KB_PER_STAGE = 4;                             // 64-wide K blocks per weight stage
constexpr uint32_t ACC_COL = 0;
constexpr uint32_t A_COL = 256;
constexpr uint32_t TMEM_COLS = 512;

constexpr int OFF_X = 0;
constexpr int OFF_W = OFF_X + X_STAGES * X_STAGE_BYTES;
constexpr int OFF_BAR = OFF_W + W_STAGES * W_STAGE_BYTES;
constexpr int NUM_BARS = 2 * X_STAGES + 2 * W_STAGES + 2 * A_STAGES + 2;
constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
constexpr int SMEM_USED = OFF_MISC + 16;
constexpr int SMEM_BYTES = SMEM_USED + 1024;  // slack to align the base to 1024 bytes
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(OFF_W % 1024 == 0 && X_STAGE_BYTES % 1024 == 0, "swizzle atoms need 1 KiB alignment");

struct GemmArgs {
    const uint8_t *w;       // repacked weights
    const __half *scales;   // W4A16: [N][K/group]
    const uint8_t *zeros;   // W4A16: [N][K/group]
    float *y;               // [M][N]
    uint32_t *status;       // library status word
    int M, N, K, group;
    int bn;                 // token tile = MMA N (multiple of 16, <= 256)
    int kb_per_split;       // 64-wide K blocks per CTA along K
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

// Bounded wait on phase `parity` of `bar`.  False if it timed out or another
// thread of the CTA aborted; a timeout records `where` in the status word.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Ctl &ctl,
                                         uint32_t where, bool honour_abort = true) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (honour_abort && (*reinterpret_cast<volatile uint32_t *>(ctl.abort) ||
                             *reinterpret_cast<volatile uint32_t *>(ctl.status))) {
            *reinterpret_cast<volatile uint32_t *>(ctl.abort) = 1u;  // another CTA already failed
            return false;
        }
        if (global_timer_ns() - t0 > ctl.timeout_ns) {
            *reinterpret_cast<volatile uint32_t *>(ctl.abort) = 1u;
            atomicCAS(ctl.status, 0u, 0x100u | where);
            return false;
        }
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

    const uint32_t bar0 = smem_u32(smem + OFF_BAR);
    const uint32_t x_full = bar0, x_empty = x_full + 8 * X_STAGES;
    const uint32_t w_full = x_empty + 8 * X_STAGES, w_empty = w_full + 8 * W_STAGES;
    const uint32_t a_full = w_empty + 8 * W_STAGES, a_empty = a_full + 8 * A_STAGES;
    const uint32_t acc_full = a_empty + 8 * A_STAGES, drain = acc_full + 8;
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + OFF_MISC);  // [0] tmem base, [1] abort
    const Ctl ctl{misc + 1, args.status, args.timeout_ns};

    if (threadIdx.x == 0) {
        for (int s = 0; s < X_STAGES; ++s) {
            mbar_init(x_full + 8 * s, 1);
            mbar_init(x_empty + 8 * s, 1);
        }
        for (int s = 0; s < W_STAGES; ++s) {
            mbar_init(w_full + 8 * s, 1);
            mbar_init(w_empty + 8 * s, NUM_XFORM_WARPS);
        }
        for (int s = 0; s < A_STAGES; ++s) {
            mbar_init(a_full + 8 * s, NUM_XFORM_WARPS);
            mbar_init(a_empty + 8 * s, 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(drain, 1);
        // A failure recorded earlier (and not yet read by qwp_device_status) makes
        // every later launch exit at once instead of waiting out its own timeouts.
        misc[1] = *reinterpret_cast<volatile uint32_t *>(args.status) ? 1u : 0u;
        fence_mbar_init();
        prefetch_tensormap(&tmap_x);
    }
    __syncthreads();
    if (misc[1]) return;
    if (warp == 1) {
        tmem_alloc(smem_u32(misc), TMEM_COLS);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int issued_x = 0, issued_w = 0;
            for (int s = 0; s < nstage; ++s) {
                const int ws = s % W_STAGES;
                if (!wait_bar(w_empty + 8 * ws, ((s / W_STAGES) & 1) ^ 1, ctl, WAIT_W_EMPTY)) break;
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
                bulk_copy_g2s(smem_u32(smem + OFF_W + ws * W_STAGE_BYTES), src, bytes, w_full + 8 * ws);
                issued_w = s + 1;
                bool ok = true;
                for (int c = 0; c < nblk; ++c) {
                    const int j = KB_PER_STAGE * s + c;
                    const int xs = j % X_STAGES;
                    if (!wait_bar(x_empty + 8 * xs, ((j / X_STAGES) & 1) ^ 1, ctl, WAIT_X_EMPTY)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(x_full + 8 * xs, static_cast<uint32_t>(args.bn) * 128u);
                    tma_load_2d(smem_u32(smem + OFF_X + xs * X_STAGE_BYTES), &tmap_x,
                                (kb0 + c) * CHUNK_K, m0, x_full + 8 * xs);
                    issued_x = j + 1;
                }
                if (!ok) break;
            }
            // Every copy issued above has landed before the CTA may exit.
            for (int j = max(0, issued_x - X_STAGES); j < issued_x; ++j)
                wait_bar(x_full + 8 * (j % X_STAGES), (j / X_STAGES) & 1, ctl, WAIT_DRAIN, false);
            for (int s = max(0, issued_w - W_STAGES); s < issued_w; ++s)
                wait_bar(w_full + 8 * (s % W_STAGES), (s / W_STAGES) & 1, ctl, WAIT_DRAIN, false);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = make_idesc_f16(kQ4K, TILE_ROWS, static_cast<uint32_t>(args.bn));
            bool ok = true;
            for (int j = 0; j < nkb && ok; ++j) {
                const int xs = j % X_STAGES, as = j % A_STAGES;
                ok = wait_bar(x_full + 8 * xs, (j / X_STAGES) & 1, ctl, WAIT_X_FULL) &&
                     wait_bar(a_full + 8 * as, (j / A_STAGES) & 1, ctl, WAIT_A_FULL);
                if (!ok) break;
                tc_fence_after();
                const uint64_t bdesc = smem_desc_sw128(smem_u32(smem + OFF_X + xs * X_STAGE_BYTES));
#pragma unroll
                for (int kk = 0; kk < CHUNK_K / 16; ++kk)
                    mma_ts(tmem + ACC_COL, tmem + A_COL + 32u * as + 8u * kk, bdesc + 2u * kk, idesc,
                           (j | kk) != 0);
                mma_commit(x_empty + 8 * xs);
                mma_commit(a_empty + 8 * as);
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
        const uint32_t xw = warp - 2;
        const uint32_t quarter = warp & 3;  // tensor-memory lanes 32*quarter .. +31
        const int half = static_cast<int>(xw >> 2);
        const int r = static_cast<int>(quarter * 32 + lane);
        const bool valid = r < R;
        const int64_t n = static_cast<int64_t>(tile) * TILE_ROWS + r;
        const uint32_t lane_base = (quarter * 32u) << 16;
        bool ok = true;
        for (int s = 0; s < nstage && ok; ++s) {
            const int ws = s % W_STAGES;
            // Every lane waits; the warp moves on together (tcgen05.st/ld are warp-collective).
            if (!__all_sync(0xffffffffu, wait_bar(w_full + 8 * ws, (s / W_STAGES) & 1, ctl, WAIT_W_FULL))) {
                ok = false;
                break;
            }
            const uint8_t *wst = smem + OFF_W + ws * W_STAGE_BYTES;
            const int kb0 = kb_begin + KB_PER_STAGE * s;
            const int nblk = min(KB_PER_STAGE, kb_end - kb0);
            uint4 hdr = make_uint4(0, 0, 0, 0);
            if (kQ4K && valid) hdr = *reinterpret_cast<const uint4 *>(wst + Q4K_HEADER_BYTES * r);
#pragma unroll
            for (int c = 0; c < KB_PER_STAGE; ++c) {
                if (c >= nblk) break;
                const int j = KB_PER_STAGE * s + c;
                const int as = j % A_STAGES;
                uint32_t regs[16];
                if (kQ4K) {
                    uint4 wv = make_uint4(0, 0, 0, 0);
                    if (valid)
                        wv = *reinterpret_cast<const uint4 *>(wst + Q4K_HEADER_BYTES * R +
                                                              CHUNK_ROW_BYTES * R * c +
                                                              (half * R + r) * 16);
                    float dl, ml;
                    q4k_subblock_scale(hdr, 2 * c + half, dl, ml);
                    uint32_t p[4];
                    q4k_word_bf16x2(wv.x, dl, ml, p);
                    regs[0] = p[0]; regs[1] = p[1]; regs[2] = p[2]; regs[3] = p[3];
                    q4k_word_bf16x2(wv.y, dl, ml, p);
                    regs[4] = p[0]; regs[5] = p[1]; regs[6] = p[2]; regs[7] = p[3];
                    q4k_word_bf16x2(wv.z, dl, ml, p);
                    regs[8] = p[0]; regs[9] = p[1]; regs[10] = p[2]; regs[11] = p[3];
                    q4k_word_bf16x2(wv.w, dl, ml, p);
                    regs[12] = p[0]; regs[13] = p[1]; regs[14] = p[2]; regs[15] = p[3];
                } else {
                    uint4 wv = make_uint4(0, 0, 0, 0);
                    __half2 s2 = __float2half2_rn(0.f);
                    __half2 mz = w4_magic_zero(0);
                    if (valid) {
                        wv = *reinterpret_cast<const uint4 *>(wst + CHUNK_ROW_BYTES * R * c +
                                                              (half * R + r) * 16);
                        const int64_t ng = args.K / args.group;
                        const int64_t g = (static_cast<int64_t>(kb0 + c) * CHUNK_K) / args.group;
                        s2 = __half2half2(args.scales[n * ng + g]);
                        mz = w4_magic_zero(args.zeros[n * ng + g]);
                    }
                    uint32_t p[4];
                    w4_word_f16x2(wv.x, mz, s2, p);
                    regs[0] = p[0]; regs[1] = p[1]; regs[2] = p[2]; regs[3] = p[3];
                    w4_word_f16x2(wv.y, mz, s2, p);
                    regs[4] = p[0]; regs[5] = p[1]; regs[6] = p[2]; regs[7] = p[3];
                    w4_word_f16x2(wv.z, mz, s2, p);
                    regs[8] = p[0]; regs[9] = p[1]; regs[10] = p[2]; regs[11] = p[3];
                    w4_word_f16x2(wv.w, mz, s2, p);
                    regs[12] = p[0]; regs[13] = p[1]; regs[14] = p[2]; regs[15] = p[3];
                }
                if (!__all_sync(0xffffffffu,
                                wait_bar(a_empty + 8 * as, ((j / A_STAGES) & 1) ^ 1, ctl, WAIT_A_EMPTY))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                tmem_st_x16(tmem + lane_base + A_COL + 32u * as + 16u * half, regs);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(a_full + 8 * as);
            }
            __syncwarp();
            if (ok && lane == 0) mbar_arrive(w_empty + 8 * ws);
        }
        __syncwarp();
        if (ok && __all_sync(0xffffffffu, wait_bar(acc_full, 0, ctl, WAIT_ACC_FULL))) {
            tc_fence_after();
            for (int ci = half; ci < args.bn / 16; ci += 2) {
                uint32_t v[16];
                tmem_ld_x16(tmem + lane_base + ACC_COL + 16u * ci, v);
                tmem_wait_ld();
                if (valid) {
                    const int mb = m0 + 16 * ci;
#pragma unroll
                    for (int t = 0; t < 16; ++t)
                        if (mb + t < args.M)
                            args.y[static_cast<int64_t>(mb + t) * args.N + n] = __uint_as_float(v[t]);
                }
            }
        }
        tc_fence_before();
    }

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
static int encode_x_map(CUtensorMap *map, const void *x, bool bf16, int64_t M, int64_t K, int bn) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return QWP_ERR_CUDA;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(CHUNK_K), static_cast<cuuint32_t>(bn)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
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

template <bool kQ4K>
static int set_smem_attr() {
    static std::atomic<uint64_t> done_mask{0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return QWP_ERR_CUDA;
    const uint64_t bit = 1ull << (dev & 63);
    if (done_mask.load() & bit) return QWP_OK;
    if (cudaFuncSetAttribute(qwp_gemm_kernel<kQ4K>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SMEM_BYTES) != cudaSuccess)
        return QWP_ERR_CUDA;
    done_mask.fetch_or(bit);
    return QWP_OK;
}

template <bool kQ4K>
static int launch_gemm(const void *w, const void *scales, const uint8_t *zeros, const void *x,
                       float *y, int64_t M, int64_t N, int64_t K, int64_t group, cudaStream_t stream,
                       uint64_t timeout_ns) {
    int rc = check_device();
    if (rc) return rc;
    if ((rc = set_smem_attr<kQ4K>())) return rc;
    uint32_t *status = status_word();
    if (!status) return QWP_ERR_CUDA;
    const int bn = choose_bn(M);
    CUtensorMap map;
    if ((rc = encode_x_map(&map, x, kQ4K, M, K, bn))) return rc;
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
    a.bn = bn;
    a.kb_per_split = static_cast<int>(K / CHUNK_K);
    a.timeout_ns = timeout_ns;
    dim3 grid(static_cast<unsigned>((N + TILE_ROWS - 1) / TILE_ROWS),
              static_cast<unsigned>((M + bn - 1) / bn), 1);
    qwp_gemm_kernel<kQ4K><<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(map, a);
    return launch_status();
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

extern "C" int q4k_gemm(const void *w_tiled, const void *x, float *y, int64_t M, int64_t N,
                        int64_t K, void *stream) {
    if (K % Q4K_BLOCK || K == 0) return K < 0 ? QWP_ERR_INVALID_ARG : QWP_ERR_UNSUPPORTED_SHAPE;
    int rc = gemm_shape_checks(w_tiled, x, y, M, N, K);
    if (rc || M == 0 || N == 0) return rc;
    return launch_gemm<true>(w_tiled, nullptr, nullptr, x, y, M, N, K, 0,
                             static_cast<cudaStream_t>(stream), kDefaultTimeoutNs);
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
                              static_cast<cudaStream_t>(stream), kDefaultTimeoutNs);
}
