// Host-side helpers shared by the translation units of the library.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/qwp.h"

namespace qwp {

// QWP_OK if the current device is an sm_103 GPU (cached per device), else QWP_ERR_DEVICE / QWP_ERR_CUDA.
int check_device();

// Device address of the library's status word on the current device (nullptr on failure).
uint32_t *status_word();

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Launch errors of the last launch on this thread, as a qwp_status.
inline int launch_status() {
    return cudaGetLastError() == cudaSuccess ? QWP_OK : QWP_ERR_CUDA;
}

// Launches `kernel` with programmatic stream serialization (the kernel calls
// pdl_wait before touching memory that earlier grids write or read).
template <typename... KArgs, typename... Args>
int launch_pdl(void (*kernel)(KArgs...), unsigned grid, unsigned block, cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(block, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...) != cudaSuccess) {
        cudaGetLastError();
        return QWP_ERR_CUDA;
    }
    return QWP_OK;
}

// Status word bits: a timeout records 0x100 | (which wait) in the low 16 bits;
// an activation outside the fp16 range sets kStatusRangeBit.
constexpr uint32_t kStatusTimeoutMask = 0xFFFFu;
constexpr uint32_t kStatusRangeBit = 0x10000u;

// Converts n bf16 values (n % 8 == 0, both pointers 16-byte aligned) to fp16 on
// `stream`, and zeroes `nzero` 32-bit words at `zero` (may be null); the launch
// allows a programmatic dependent launch to follow.
int launch_bf16_to_f16(const void *x, void *out, int64_t n, cudaStream_t stream, uint32_t *zero = nullptr,
                       int nzero = 0);

// The prefill (tcgen05) kernel for a Q4_K product with bf16 x, whatever the decode
// policy says, converting x into the caller's array x16 (M*K fp16 values; one
// token: inside the GEMM kernel) and
// never splitting units between CTAs, so that it allocates nothing (x, w, y
// checked by the caller).
int launch_q4k_prefill_fixed(const void *w, const void *x, void *x16, float *y, int64_t M, int64_t N, int64_t K,
                             cudaStream_t stream);

// The skinny-N kernel (qwp_skinny.cu): Q4_K products with at most 64 weight rows
// and at least SKINNY_MIN_TOKENS tokens.  x is bf16 or fp16, read as it is by the
// tensor core; allocates nothing.
constexpr int64_t SKINNY_MIN_TOKENS = 256;
bool skinny_selected(int fmt, int64_t M, int64_t N, int64_t K);
// Its launch: `splits` CTAs per cluster along K, `tiles` token tiles of `tm`
// (<= 128) tokens.
int skinny_plan(int64_t M, int64_t K, int sms, int &splits, int64_t &tiles, int &tm);
int launch_skinny(const void *w, const void *x, bool x_bf16, float *y, int64_t M, int64_t N, int64_t K,
                  cudaStream_t stream);

// Default bound on any single mbarrier wait inside a kernel; the waits for a
// CTA's own copies and MMAs in flight before it exits always use it.
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;  // 2 s

// The bound on the prefill kernel's main-loop waits (qwp_set_wait_timeout_ns;
// kDefaultTimeoutNs unless changed).
uint64_t wait_timeout_ns();

}  // namespace qwp
