// kernels.h -- host-side launchers of the device kernels (library internal).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace qmm {

// Counts e == cudaSuccess as one kernel launch and returns e (every launch
// site of the library returns through it).
cudaError_t launched(cudaError_t e);

// out[M,K] = dequantized W (f32, one rounding of the exact value).
cudaError_t launch_dequant(int fmt, const uint8_t *W, int64_t M, int64_t K, float *out, cudaStream_t st);

// Byte-addressed GEMV for any alignment, 1 <= N <= 16.
cudaError_t launch_gemv_generic(int fmt, const uint8_t *W, int64_t M, int64_t K, const void *X, int xbf16,
                                int N, float *Y, cudaStream_t st);

// Requested launch shape of the tensor-core GEMV (0 = automatic).
struct GemvTuning {
    int rows;       // rows per tile: 64, 128 or 256
    int rg;         // 16-row groups per compute warp of the resident-X kernel (1 or 2)
    int ks;         // K split (cluster size, 1..8)
    int resident;   // 0 disables the resident-X kernel
};

// What will run: the resident-X kernel (P * N <= 2 MMA columns; resident ==
// 1), the ring kernel (0) or the integer kernel (2), its tile height (= the
// weight tensor map's box height), row groups per warp and K split.
struct GemvPlan {
    int resident;
    int rows;
    int rg;
    int ks;
};
GemvPlan plan_gemv(int64_t M, int64_t K, int N, int xbf16, int num_sms, const GemvTuning &tun);

// Weight matrices of one GEMV launch (several share X: fused projections).
// The host fills wmap (box {window/2, plan.rows}), Y and M per matrix; the
// launcher fills tile0.
constexpr int QMM_MAX_SEGS = 4;
struct GemvSegs {
    CUtensorMap wmap[QMM_MAX_SEGS];
    float *Y[QMM_MAX_SEGS];
    int M[QMM_MAX_SEGS];
    int tile0[QMM_MAX_SEGS + 1];   // first tile of each matrix; [nseg] = all tiles
    int nseg;
};

// Tensor-core GEMV, 1 <= N <= 16 (K % 256 == 0, 16-byte aligned W rows and
// X), executing `plan` over every matrix of `segs`.  xmap: X [N][K] (f32 or
// bf16), box {256, N}; X: the same tensor by address.  pdl: launched as a
// programmatic dependent of the preceding kernel (weights are read before it
// ends).  amax_ws != nullptr (one matrix only): argmax mode.  Y is not
// written; amax_ws holds N keys and a finished-CTA counter (zeroed by the
// caller, 8 * (N + 1) bytes), and the last CTA writes idx[n] (row of token
// n's largest output, the lowest row on ties) and val[n] (that output).
cudaError_t launch_gemv_mma(int fmt, const GemvPlan &plan, const GemvSegs &segs, const CUtensorMap &xmap,
                            const void *X, int xbf16, int64_t K, int N, bool pdl, unsigned *status, uint64_t limit,
                            cudaStream_t st, unsigned long long *amax_ws = nullptr, int32_t *idx = nullptr,
                            float *val = nullptr);

// Streaming decode GEMV for N = 1 (K % 256 == 0, K <= 32768, 16-byte
// aligned W, rows and X): CTAs of `warps` warps own whole rows; each warp
// streams stages of 32 tasks (R rows x one 256-weight column each) through
// S shared-memory slots.
struct StreamPlan {
    int grid;
    int warps;
    int S;
    int R;      // rows per task: 1, 2 or 4
    int smem;   // dynamic shared memory bytes
    int direct; // 1: the direct-load variant (registers, no shared-memory ring; S = 0)
    int stagger;// S >= 2: one stage issued up front, the next once the current has landed
    int nseg;   // weight matrices sharing X; segment i runs on CTAs cta0[i] .. cta0[i + 1] - 1
    int cta0[QMM_MAX_SEGS + 1];
};
// Requested plan parameters; 0 = chosen by the planner.  cps: CTAs per SM;
// direct: 1 the direct-load variant, 2 the staged kernel.
struct StreamForce {
    int r, warps, slots, cps, direct;
    int stagger;   // 2: no staggered stage issue with slots >= 2 (on otherwise)
};
// false: the shape does not fit the kernel (another GEMV kernel runs), or
// a forced parameter cannot be met.
bool plan_gemv_stream(int fmt, int64_t M, int64_t K, int num_sms, const StreamForce &force, StreamPlan &p);
// The same for nseg (<= QMM_MAX_SEGS) matrices of Ms[i] rows sharing X and K:
// one launch, the CTAs split over the matrices in proportion to their rows.
bool plan_gemv_stream(int fmt, const int64_t *Ms, int nseg, int64_t K, int num_sms, const StreamForce &force,
                      StreamPlan &p);
// y[M] = W x.  pdl: programmatic dependent of the preceding kernel (the
// weight copies start before it ends; X and Y wait for it).
// amax_ws != nullptr: argmax mode as in launch_gemv_mma (Y is not written).
cudaError_t launch_gemv_stream(int fmt, const StreamPlan &p, const uint8_t *W, int64_t M, int64_t K, const void *X,
                               int xbf16, float *Y, bool pdl, unsigned *status, uint64_t limit, cudaStream_t st,
                               unsigned long long *amax_ws = nullptr, int32_t *idx = nullptr, float *val = nullptr);
// p.nseg matrices (Ws[i], Ms[i] rows, output Ys[i]) planned by the
// multi-matrix plan_gemv_stream; argmax mode needs a single matrix.
cudaError_t launch_gemv_stream(int fmt, const StreamPlan &p, const uint8_t *const *Ws, float *const *Ys,
                               const int64_t *Ms, int64_t K, const void *X, int xbf16, bool pdl, unsigned *status,
                               uint64_t limit, cudaStream_t st, unsigned long long *amax_ws = nullptr,
                               int32_t *idx = nullptr, float *val = nullptr);

// Tensor-core GEMV for 1 <= N <= 8 (mma.sync f16 on the exact codes) of
// Q8_0 / Q4_0 / Q4_K / Q5_K rows (K % 256 == 0, K <= 32768, 16-byte aligned
// W, rows and X).  wmap: W as u16 [M][row_bytes / 2], box
// {gemv_tc_unit_bytes / 2, 16}.  One CTA per SM owns whole 16-row groups.
struct TcPlan {
    int grid;
    int warps;
    int S;
    int smem;
};
int gemv_tc_unit_bytes(int fmt);   // 0: format not handled
bool plan_gemv_tc(int fmt, int64_t M, int64_t K, int N, int num_sms, int force_warps, TcPlan &p);
// amax_ws != nullptr: argmax mode as in launch_gemv_mma (Y is not written).
cudaError_t launch_gemv_tc(int fmt, const TcPlan &p, const CUtensorMap &wmap, const uint8_t *W, int64_t M, int64_t K,
                           const void *X, int xbf16, int N, float *Y, bool pdl, unsigned *status, uint64_t limit,
                           cudaStream_t st, unsigned long long *amax_ws = nullptr, int32_t *idx = nullptr,
                           float *val = nullptr);

// Integer tensor-core GEMV (mma.sync m16n8k32 on the weights' integer codes),
// same weight maps, segments, plans and argmax mode as launch_gemv_mma.
//  * exact: X f32 or bf16 [N][K] as exact int8 digits; N <= 2 (Q6_K: N == 1).
//  * q8:    X given as Q8_0 activations: quants int8 [N][K], scales f32
//           [N][K/32] (16-byte aligned); N <= 16.
// *_maxc: the largest K slice (256-weight chunks) one CTA can hold for that
// variant and tile height (0: unsupported), the bound for the K split.
int gemv_i8_exact_maxc(int fmt, int N, int xbf16, int rows, int rg);
int gemv_i8_q8_maxc(int fmt, int N, int rows);
cudaError_t launch_gemv_i8_exact(int fmt, const GemvPlan &plan, const GemvSegs &segs, const void *X, int xbf16,
                                 int64_t K, int N, bool pdl, unsigned *status, uint64_t limit, cudaStream_t st,
                                 unsigned long long *amax_ws = nullptr, int32_t *idx = nullptr, float *val = nullptr);
cudaError_t launch_gemv_i8_q8(int fmt, const GemvPlan &plan, const GemvSegs &segs, const int8_t *quants,
                              const float *scales, int64_t K, int N, bool pdl, unsigned *status, uint64_t limit,
                              cudaStream_t st, unsigned long long *amax_ws = nullptr, int32_t *idx = nullptr,
                              float *val = nullptr);

// Q8_0 activations of X (f32 or bf16, count % 32 == 0): scales[count/32],
// quants[count].  pdl: programmatic dependent of the preceding kernel.
// launch_quantize_q8_0_bf16: the same quantizer, writing instead
// out[i] = bf16(scale * code) (the dequantized activation, rounded to bf16).
cudaError_t launch_quantize_q8_0(const void *X, int xbf16, int64_t count, float *scales, int8_t *quants, bool pdl,
                                 cudaStream_t st);
cudaError_t launch_quantize_q8_0_bf16(const void *X, int xbf16, int64_t count, uint16_t *out, bool pdl,
                                      cudaStream_t st);

// K split of a GEMV over `tiles` row tiles: the smallest power of two (<= 8)
// giving at least 1.5 CTAs per SM, and (max_cps > 0) slices of at most
// max_cps chunks; force > 0 requests a split.  0: no split fits max_cps.
int plan_ks_host(int64_t tiles, int nchunks, int num_sms, int max_cps, int force);

// out[i] = silu(g[i]) * u[i] for i < count.  pdl: programmatic dependent
// of the preceding kernel (which writes g and u).
cudaError_t launch_swiglu(const float *g, const float *u, int64_t count, float *out, bool pdl, cudaStream_t st);

// Raw bytes of one 256-weight chunk of a row in the GEMV's staging.
int gemv_window_bytes(int fmt);

// Rows per GEMV tile (the weight tensor map's box height) for M rows.
int gemv_tile_rows(int64_t M, int num_sms);

// bf16 out[i] = round-to-nearest-even(X[i]).  pdl: launched as a
// programmatic dependent of the preceding kernel.
cudaError_t launch_x_to_bf16(const float *X, int64_t count, uint16_t *out, bool pdl, cudaStream_t st);

// Tensor-core GEMM.  wmap: raw weight bytes viewed as u16 [M][row_bytes/2],
// box {window/2, 128}; xmap: bf16 X as a 3-D tensor {64 k, N tokens, K/64
// k-blocks} (strides K*2 and 128 bytes), box {64, BN, XG}, 128-byte swizzle,
// XG = gemm_x_stages_per_copy(BN).
struct GemmArgs {
    int fmt;
    int64_t M, K;
    int N;
    int bn;          // token tile (64, 128 or 256)
    float *Y;
    float *Y2;       // second matrix's output (wmap2; same M and K), or null
    int ks;          // K split over a (1, 1, ks) cluster: 1, 2 or 4 (ks <= K / 256)
    int mt0, mtn;    // this launch's 128-row tiles: mt0 .. mt0 + mtn - 1 (with Y2, the
                     // second matrix's tiles follow the first's)
    unsigned *status;
    uint64_t wait_limit;
    int pdl;         // programmatic dependent launch (weights read before the preceding kernel ends)
};
// With a.Y2 set, one launch computes two matrices of the same shape that
// share X (wmap -> Y, wmap2 -> Y2); otherwise wmap2 is not read.
cudaError_t launch_gemm_tc(const GemmArgs &a, const CUtensorMap &wmap, const CUtensorMap &wmap2,
                           const CUtensorMap &xmap, cudaStream_t st);

int gemm_x_stages_per_copy(int bn);
// Clusters of ks CTAs (1, 2, 4) of the GEMM kernel for (fmt, bn) that can be
// resident at once on the current device (0 if the query fails).
int gemm_max_clusters(int fmt, int bn, int ks);

// Window of raw weight bytes one 256-weight chunk of a row occupies in the
// GEMM's shared-memory staging (bytes; a multiple of 16).
int gemm_raw_window_bytes(int fmt);

}  // namespace qmm
