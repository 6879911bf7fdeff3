// kernels.h -- host-side launchers of the device kernels (library internal).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace qmm {

// out[M,K] = dequantized W (f32, one rounding of the exact value).
cudaError_t launch_dequant(int fmt, const uint8_t *W, int64_t M, int64_t K, float *out, cudaStream_t st);

// Byte-addressed GEMV for any alignment, 1 <= N <= 16.
cudaError_t launch_gemv_generic(int fmt, const uint8_t *W, int64_t M, int64_t K, const void *X, int xbf16,
                                int N, float *Y, cudaStream_t st);

// Tensor-core GEMV, 1 <= N <= 16 (K % 256 == 0, 16-byte aligned W rows and
// X).  wmap: raw weight bytes as u16 [M][row_bytes/2], box {window/2, 64};
// xmap: X [N][K] (f32 or bf16), box {256, N}.
cudaError_t launch_gemv_mma(int fmt, const CUtensorMap &wmap, const CUtensorMap &xmap, int xbf16, int64_t M,
                            int64_t K, int N, float *Y, int num_sms, unsigned *status, uint64_t limit,
                            cudaStream_t st);

// Raw bytes of one 256-weight chunk of a row in the GEMV's staging.
int gemv_window_bytes(int fmt);

// Rows per GEMV tile (the weight tensor map's box height) for M rows.
int gemv_tile_rows(int64_t M, int num_sms);

// bf16 out[i] = round-to-nearest-even(X[i]).
cudaError_t launch_x_to_bf16(const float *X, int64_t count, uint16_t *out, cudaStream_t st);

// Tensor-core GEMM.  wmap: raw weight bytes viewed as u16 [M][row_bytes/2],
// box {window/2, 128}; xmap: bf16 X [N][K], box {64, BN}, 128-byte swizzle.
struct GemmArgs {
    int fmt;
    int64_t M, K;
    int N;
    int bn;          // token tile (64, 128 or 256)
    float *Y;
    unsigned *status;
    uint64_t wait_limit;
};
cudaError_t launch_gemm_tc(const GemmArgs &a, const CUtensorMap &wmap, const CUtensorMap &xmap, cudaStream_t st);

// Window of raw weight bytes one 256-weight chunk of a row occupies in the
// GEMM's shared-memory staging (bytes; a multiple of 16).
int gemm_raw_window_bytes(int fmt);

}  // namespace qmm
