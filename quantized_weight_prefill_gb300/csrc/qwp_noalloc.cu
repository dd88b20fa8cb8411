// q4k_gemm_noalloc: the bf16-activation Q4_K GEMM for callers that may not
// allocate device memory.  q4k_gemm converts x to fp16 into scratch taken from
// a stream-ordered pool; here that scratch is a fixed array compiled into the
// library instead, so a call allocates nothing.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/qwp.h"
#include "qwp_decode.h"
#include "qwp_internal.h"

// The fp16 copy of x.  Every GPU on which this library's device code is loaded
// holds these QWP_NOALLOC_MAX_X_ELEMS * 2 bytes until the process exits.  In
// host code the name is only a handle for cudaGetSymbolAddress, never an address.
static __device__ __align__(256) uint16_t g_x16_scratch[QWP_NOALLOC_MAX_X_ELEMS];

// Scratch of decode-shaped calls (M <= 8): partial sums of the 128-row tiles that
// two or more CTAs share and one counter per tile (4 MiB, held the same way).
constexpr size_t kDecodeScratchBytes = 4u << 20;
static __device__ __align__(256) uint8_t g_decode_scratch[kDecodeScratchBytes];

namespace {

constexpr int kMaxDevices = 64;

// Device addresses of g_x16_scratch and g_decode_scratch on the current device,
// looked up once per device (the lookup also loads this code onto the device if
// needed).
int scratch_address(void **out, void **decode_out) {
    static void *addr[kMaxDevices], *dec_addr[kMaxDevices];
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return QWP_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr, *q = nullptr;
        if (cudaGetSymbolAddress(&p, g_x16_scratch) != cudaSuccess || !p ||
            cudaGetSymbolAddress(&q, g_decode_scratch) != cudaSuccess || !q) {
            cudaGetLastError();
            return QWP_ERR_CUDA;
        }
        addr[dev] = p;
        dec_addr[dev] = q;
    }
    *out = addr[dev];
    *decode_out = dec_addr[dev];
    return QWP_OK;
}

}  // namespace

extern "C" int q4k_gemm_noalloc(const void *w_tiled, const void *x, float *y, int64_t M, int64_t N,
                                int64_t K, void *stream) {
    using namespace qwp;
    if (K % 256 || K == 0) return K < 0 ? QWP_ERR_INVALID_ARG : QWP_ERR_UNSUPPORTED_SHAPE;
    if (M < 0 || N < 0) return QWP_ERR_INVALID_ARG;
    if (M > (1ll << 30) || N > (1ll << 30) || K > (1ll << 30)) return QWP_ERR_UNSUPPORTED_SHAPE;
    if (M == 0 || N == 0) return QWP_OK;
    if (!w_tiled || !x || !y) return QWP_ERR_INVALID_ARG;
    if (!aligned16(w_tiled) || !aligned16(x) || !aligned16(y)) return QWP_ERR_MISALIGNED;
    if (M > static_cast<int64_t>(QWP_NOALLOC_MAX_X_ELEMS) / K) return QWP_ERR_SCRATCH_LIMIT;
    int rc = check_device();
    if (rc) return rc;
    void *x16 = nullptr, *dec = nullptr;
    if ((rc = scratch_address(&x16, &dec))) return rc;
    // Decode-shaped calls: the decode kernel converts x itself and keeps its
    // partial sums in the fixed decode array, when they fit there (for very wide
    // matrices they may not: those run the prefill kernel below instead, whose
    // fp16 copy of x always fits once M*K has passed the check above).
    const size_t dec_need = decode_selected(DFMT_Q4K, M, N, K) ? decode_scratch_bytes(DFMT_Q4K, N, K) : 0;
    if (dec_need && dec_need <= kDecodeScratchBytes)
        return launch_decode(DFMT_Q4K, w_tiled, nullptr, nullptr, x, true, y, M, N, K, 0, dec, kDecodeScratchBytes,
                             static_cast<cudaStream_t>(stream));
    // The skinny-N kernel reads bf16 x as it is and allocates nothing.
    if (skinny_selected(DFMT_Q4K, M, N, K))
        return launch_skinny(w_tiled, x, true, y, M, N, K, static_cast<cudaStream_t>(stream));
    // The conversion writes all M*K elements the GEMM reads, so nothing left
    // in the array by an earlier call is ever read; units are never split
    // between CTAs here, so the GEMM needs no workspace.
    return launch_q4k_prefill_fixed(w_tiled, x, x16, y, M, N, K, static_cast<cudaStream_t>(stream));
}
