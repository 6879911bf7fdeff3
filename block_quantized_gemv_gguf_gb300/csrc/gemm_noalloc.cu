// gemm_noalloc.cu -- qmm_gemm_noalloc: the tensor-core GEMM for callers that
// are not allowed to allocate device memory and cannot hand the library a
// workspace.
//
// The GEMM needs scratch only when X is f32: X is rounded to bf16 into a
// buffer of N*K*2 bytes before the tensor cores read it.  Here that buffer is
// a fixed, file-scope device array instead of caller-provided memory.  Every
// device that loads this library holds the array (QMM_NOALLOC_SCRATCH_BYTES)
// until the process exits.
//
// Host code must not use the array's name as a device pointer: in host code
// it names a host-side stand-in.  Its device address is looked up with
// cudaGetSymbolAddress, once per device, with that device current, on the
// first call made on that device, and cached.  cudaDeviceReset destroys the
// array with the context, so the cached address is not valid after it: a
// process that resets a device must not call this entry point again.
#include <mutex>

#include "../../include/qmm.h"

namespace {

__device__ __align__(256) uint8_t g_noalloc_scratch[QMM_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kMaxDevices];

// Device address of the scratch array on the current device (set-up on the
// first call per device).  Returns nullptr on failure.
void *scratch_on_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return nullptr;
        g_noalloc_ptr[dev] = p;
    }
    return g_noalloc_ptr[dev];
}

}  // namespace

extern "C" qmm_status qmm_gemm_noalloc(qmm_wtype wt, const void *W, size_t w_bytes, int64_t M, int64_t K,
                                       const void *X, qmm_xtype xt, int64_t N, float *Y, void *stream) {
    // the argument checks of qmm_gemm come first, so that a bad argument is
    // reported as such whatever the size of X
    int E = 0, B = 0;
    if (qmm_block_info(wt, &E, &B) != QMM_OK) return QMM_ERR_INVALID_ARG;
    if (xt != QMM_X_F32 && xt != QMM_X_BF16) return QMM_ERR_INVALID_ARG;
    if (!W || !X || !Y) return QMM_ERR_INVALID_ARG;
    if (N < 1 || K < 1 || M < 1 || N > QMM_GEMM_MAX_N || K % E) return QMM_ERR_INVALID_ARG;
    if (w_bytes < (size_t)M * (size_t)(K / E) * (size_t)B) return QMM_ERR_INVALID_ARG;
    const size_t need = qmm_gemm_workspace_bytes(N, K, xt);
    if (need > (size_t)QMM_NOALLOC_SCRATCH_BYTES) return QMM_ERR_UNSUPPORTED;   // N*K*2 too large
    if (need == 0) return qmm_gemm(wt, W, w_bytes, M, K, X, xt, N, Y, nullptr, 0, stream);
    void *scratch = scratch_on_current_device();
    if (!scratch) return QMM_ERR_CUDA;
    // The whole N*K*2-byte prefix is rewritten by the conversion kernel before
    // the GEMM reads it, so nothing has to be cleared between calls.
    return qmm_gemm(wt, W, w_bytes, M, K, X, xt, N, Y, scratch, (size_t)QMM_NOALLOC_SCRATCH_BYTES, stream);
}
