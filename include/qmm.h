/*
 * qmm.h -- C ABI of the GB300 (sm_103a) block-quantized projection matmul.
 *
 *     Y[n, m] = sum_k  X[n, k] * w(m, k)        0 <= n < N, 0 <= m < M
 *
 * W[M, K] is stored in GGUF/ggml block-quantized layouts and dequantized on
 * the fly inside the kernels.  This is the projection matmul of the dense
 * transformer in "cera 0.5.0 src/model/llama.rs" (per-token decode GEMV,
 * project_logits / project_logits_batched for the LM head,
 * forward_prefill_batched for the batched prefill GEMM) whose scalar
 * definition is matmul_q4_0_f32 / matmul_q8_0_f32 / matmul_q4km_f32 and the
 * gemv_* row loops of "cera 0.5.2 src/backend/cpu.rs".
 *
 * Layouts (all little endian, blocks stored back to back):
 *   W      row m is K / E_blk consecutive blocks; rows are consecutive, so
 *          row m starts at byte m * (K / E_blk) * B_blk ("cera 0.5.2
 *          src/backend/cpu.rs" matmul_*_f32).
 *   Q8_0   34 B / 32 weights: f16 d @0, int8 q[32] @2; w = d * q.
 *   Q4_0   18 B / 32 weights: f16 d @0, qs[16] @2; weight e < 16 is the low
 *          nibble of qs[e], weight e >= 16 the high nibble of qs[e-16];
 *          w = (nibble - 8) * d ("cera 0.5.2 src/backend/cpu.rs",
 *          repack_q4_0_8x8).
 *   Q4_K   144 B / 256 weights: f16 d @0, f16 dmin @2, 12 packed scale bytes
 *          @4, qs[128] @16.  Sub-block s = e / 32 uses the low (s even) or
 *          high (s odd) nibble of qs[(s/2)*32 + e%32]; six-bit (sc_s, m_s)
 *          are packed in GGUF order; w = d*sc_s*q - dmin*m_s ("cera 0.5.2
 *          src/backend/cpu.rs", repack_q4_k_8x8).
 *   Q6_K   210 B / 256 weights: ql[128] @0, qh[64] @128, int8 scales[16]
 *          @192, f16 d @208; weight e = 128h + 32j + l takes its low four
 *          bits from ql[64h + 32(j%2) + l] (low nibble for j < 2, high for
 *          j >= 2) and bits 2j..2j+1 of qh[32h + l] as bits 4..5;
 *          w = d * scales[e/16] * (q - 32) (GGUF layout; the 210-byte size is
 *          "cera 0.3.1 src/model/gpu_lfm2.rs", weight upload).
 *   Q5_K   176 B / 256 weights: f16 d @0, f16 dmin @2, 12 scale bytes @4
 *          (packed as Q4_K), qh[32] @16, qs[128] @48; weight e = 32s + l
 *          takes Q4_K's nibble of qs[(s/2)*32 + l] and bit s of qh[l] as
 *          bit 4; w = d*sc_s*q - dmin*m_s (GGUF layout; the 176-byte size is
 *          "cera 0.3.1 src/model/gpu_lfm2.rs", weight upload).
 *   X      [N, K] row-major, f32 or bf16, device memory.
 *   Y      [N, M] row-major f32, device memory, OVERWRITTEN (not accumulated,
 *          as the scalar row loops assign their sum).
 *
 * Conventions common to every call:
 *   - All pointers are device pointers unless the name says host.  The
 *     caller owns every buffer; the library allocates nothing per call.  The
 *     only allocation is one small device status word per device, made on the
 *     first call on that device.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Every call is asynchronous and stream ordered; there is no
 *     hidden global state, so calls on different streams may run
 *     concurrently on disjoint outputs.
 *   - Arguments are validated on the host before anything is launched; on a
 *     validation error nothing is written and no kernel runs.  The checks
 *     mirror the release asserts of "cera 0.5.2 src/backend/cpu.rs"
 *     gemm_preq_dispatch (K a multiple of the block size, enough weight
 *     bytes for M rows) turned into status codes, plus: pointers non-null,
 *     M, K >= 1, N within the call's range, Y not overlapping W or X.
 *   - An unknown format is QMM_ERR_INVALID_ARG (the pages' GEMV dispatcher
 *     panics on it); a supported format on a path that cannot take the given
 *     shape or alignment is QMM_ERR_UNSUPPORTED, never a silent fallback
 *     (the pages warn that a silent per-token fallback cost ~4x prefill;
 *     "cera 0.5.0 src/model/llama.rs", forward_prefill_batched).
 *   - Device-side waits are bounded.  A kernel that gives up records
 *     QMM_ERR_TIMEOUT in the device status word; qmm_last_device_error
 *     reports and clears it.
 */
#ifndef QMM_H
#define QMM_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define QMM_API __attribute__((visibility("default")))
#else
#define QMM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { QMM_Q8_0 = 0, QMM_Q4_0 = 1, QMM_Q4_K = 2, QMM_Q6_K = 3, QMM_Q5_K = 4 } qmm_wtype;
typedef enum { QMM_X_F32 = 0, QMM_X_BF16 = 1 } qmm_xtype;
typedef enum {
    QMM_OK = 0,
    QMM_ERR_INVALID_ARG = 1,
    QMM_ERR_UNSUPPORTED = 2,
    QMM_ERR_CUDA = 3,
    QMM_ERR_TIMEOUT = 4
} qmm_status;

/* Largest N per call of each path.  512 is the batched-prefill chunk
 * ("cera 0.3.1 src/model/gpu_lfm2.rs", MAX_PREFILL_TOKENS). */
#define QMM_GEMV_MAX_N 16
#define QMM_GEMM_MAX_N 512
/* Largest N qmm_matmul sends to the GEMV by default (the environment
 * variable QMM_GEMV_MAX_N can change it): measured on GB300 over the seven
 * projections of one decoder layer (Q4_K/Q6_K, CUDA graphs), the GEMV takes
 * 95-131 us for N = 2..8 and 216-281 us for N = 9..16, the K-split GEMM
 * 135-141 us for every N from 2 to 32. */
#define QMM_MATMUL_GEMV_MAX_N 8

/*
 * Multi-token GEMV, 1 <= N <= QMM_GEMV_MAX_N: decode (N = 1) and small-N
 * batches such as speculative verification through the LM head
 * ("cera 0.5.0 src/model/llama.rs", project_logits and
 * project_logits_batched).  Every weight block is read from HBM once and
 * reused for all N tokens; arithmetic is f32 on the exact dequantized
 * weights (|error| <= 1e-5 * sum|w x| + 1e-6 against exact arithmetic).
 *   W        raw blocks, w_bytes >= M * (K / E_blk) * B_blk.  Any alignment;
 *            the fast path needs W 16-byte aligned and a row size that is a
 *            multiple of 16 bytes, otherwise a byte-addressed path runs.
 *   X        [N, K] f32 or bf16 (xt), 4-byte (f32) / 2-byte (bf16) aligned.
 *   Y        [N, M] f32, 4-byte aligned, overwritten.
 */
QMM_API qmm_status qmm_gemv(qmm_wtype wt, const void *W, size_t w_bytes, int64_t M, int64_t K,
                    const void *X, qmm_xtype xt, int64_t N, float *Y, void *stream);

/*
 * Fused projections: up to QMM_MAX_MATRICES weight matrices of one format
 * that share X (Q/K/V of an attention layer, gate and up of a feed-forward
 * layer), in one launch: Y_i[N, M_i] = X[N, K] . dequant(W_i)[M_i, K]^T
 * ("cera 0.5.2 src/backend/cpu.rs", gemv_q4_0_fused2_with_q8 and
 * gemv_q4_0_concat3_with_q8: several matrices, one pass over a shared x).
 * Every output meets the qmm_gemv bound against exact arithmetic (the K
 * split, and so the f32 summation order, follows the total row count).
 *   mats[i]   W (raw blocks), w_bytes, M (rows) and Y ([N, M] f32,
 *             overwritten) of matrix i; no Y may overlap any W, X or other Y.
 *   K, X, xt, N   as for qmm_gemv, shared.
 * The fast path needs every W 16-byte aligned (and the conditions of
 * qmm_gemv); otherwise each matrix runs the byte-addressed path.
 */
#define QMM_MAX_MATRICES 4
typedef struct {
    const void *W;
    size_t w_bytes;
    int64_t M;
    float *Y;
} qmm_matrix;
QMM_API qmm_status qmm_gemv_multi(qmm_wtype wt, const qmm_matrix *mats, int nmat, int64_t K, const void *X,
                          qmm_xtype xt, int64_t N, void *stream);

/*
 * Greedy decode through the LM head: for each token n, the row of the
 * largest output of the GEMV above and that output, without writing the M
 * outputs anywhere ("cera 0.5.2 src/backend/cpu.rs", gemv_with_preq_argmax;
 * "cera 0.3.1 src/model/gpu_lfm2.rs", forward_greedy_inner and
 * encode_argmax_pass, which read back the argmax instead of the logits).
 * The outputs are computed exactly as qmm_gemv computes them, so idx/val
 * equal the argmax of qmm_gemv's Y, bit for bit.  Ties go to the lowest row
 * (the pages' sampler is not on them: reading).
 *   W, X, N   as for qmm_gemv; the fast path only (16-byte aligned W and X,
 *             K % 256 == 0, row size a multiple of 16 bytes), else
 *             QMM_ERR_UNSUPPORTED.
 *   idx, val  device arrays of N int32 / N float, overwritten.
 *   workspace device buffer of at least 8 * (N + 1) bytes, 8-byte aligned
 *             (per-token partial results and a counter; contents on return
 *             unspecified).
 * Stream-ordered: a memset of the workspace, then the GEMV, whose last CTA
 * writes idx and val.
 */
QMM_API qmm_status qmm_gemv_argmax(qmm_wtype wt, const void *W, size_t w_bytes, int64_t M, int64_t K,
                           const void *X, qmm_xtype xt, int64_t N, int32_t *idx, float *val,
                           void *workspace, size_t ws_bytes, void *stream);

/*
 * Prefill GEMM on the tensor cores, 1 <= N <= QMM_GEMM_MAX_N
 * ("cera 0.5.0 src/model/llama.rs", forward_prefill_batched and its
 * per-layer projection GEMMs; "cera 0.3.1 src/model/gpu_lfm2.rs",
 * build_mul_mat_pipeline: weights are dequantized once per K tile in shared
 * memory and reused across all token columns).  Weight tiles are staged by
 * TMA, dequantized to bf16 in shared memory and multiplied by tcgen05 MMA
 * with f32 accumulation in tensor memory (|error| <= 2e-3 * sum|w x| + 1e-5).
 * Requirements (else QMM_ERR_UNSUPPORTED): K % 256 == 0 (K % 2048 == 0 for
 * Q6_K), W and X 16-byte aligned.
 *   workspace  device scratch of at least qmm_gemm_workspace_bytes(N, K, xt)
 *              bytes, 16-byte aligned (may be NULL when that size is 0):
 *              f32 X is converted to bf16 there before the GEMM.
 */
QMM_API qmm_status qmm_gemm(qmm_wtype wt, const void *W, size_t w_bytes, int64_t M, int64_t K,
                    const void *X, qmm_xtype xt, int64_t N, float *Y,
                    void *workspace, size_t ws_bytes, void *stream);

/*
 * qmm_gemm without a workspace, for callers that may not allocate device
 * memory: a plugin or custom operator whose host framework owns every byte of
 * device memory and offers no scratch argument, a deployment with a fixed,
 * pre-planned memory budget, or a latency-critical path that must avoid the
 * device-wide synchronization cudaMalloc / cudaFree can cause.
 * (The cera pages have no counterpart: their kernels run on CPU threads and
 * reuse host Vec scratch, and the wgpu path allocates its buffers at load.)
 *
 * Same arguments and results as qmm_gemm.  When X is f32 the bf16 copy of X
 * goes to a library-owned, statically sized device array of
 * QMM_NOALLOC_SCRATCH_BYTES instead of a workspace; every GPU that loads the
 * library holds that array until the process exits.  Nothing is allocated by
 * this call.
 *   - N*K*2 > QMM_NOALLOC_SCRATCH_BYTES (f32 X) returns QMM_ERR_UNSUPPORTED
 *     and launches nothing; bf16 X needs no scratch and has no extra limit.
 *   - The first call on a device looks up the array's device address for
 *     that device (cudaGetSymbolAddress) and caches it; make that first call
 *     before any stream capture.  cudaDeviceReset invalidates the cached
 *     address: calling this entry point after a reset of its device is not
 *     supported.
 *   - Arguments are checked as qmm_gemm checks them, before the size limit:
 *     a bad argument returns QMM_ERR_INVALID_ARG whatever N*K.
 *   - All calls share the one array.  Each call rewrites the part it uses
 *     before reading it, so no clearing is needed, but calls whose kernels
 *     overlap on the GPU (different streams, no ordering between them) race
 *     on the array and give wrong results: order them on one stream or with
 *     events.
 */
#define QMM_NOALLOC_SCRATCH_BYTES (16u << 20)
QMM_API qmm_status qmm_gemm_noalloc(qmm_wtype wt, const void *W, size_t w_bytes, int64_t M, int64_t K,
                                    const void *X, qmm_xtype xt, int64_t N, float *Y, void *stream);

/* Bytes of workspace qmm_gemm / qmm_matmul need: N*K*2 for f32 X, else 0. */
QMM_API size_t qmm_gemm_workspace_bytes(int64_t N, int64_t K, qmm_xtype xt);

/*
 * N-based dispatcher, 1 <= N <= QMM_GEMM_MAX_N: N <= QMM_MATMUL_GEMV_MAX_N
 * runs qmm_gemv (its tolerance), larger N runs qmm_gemm (its tolerance).  Same arguments as qmm_gemm (the
 * workspace is only touched on the GEMM path).
 */
QMM_API qmm_status qmm_matmul(qmm_wtype wt, const void *W, size_t w_bytes, int64_t M, int64_t K,
                      const void *X, qmm_xtype xt, int64_t N, float *Y,
                      void *workspace, size_t ws_bytes, void *stream);

/*
 * qmm_matmul with the per-step inputs and outputs in HOST memory:
 * copies X_host -> x_dev, runs qmm_matmul, copies y_dev -> Y_host, all
 * asynchronously on `stream` (pin the host buffers for overlap).  W stays
 * resident in device memory.  x_dev (>= N*K*sizeof(x element) bytes) and
 * y_dev (>= N*M*4 bytes) are caller-provided device staging buffers.  The
 * host output is valid after the stream is synchronized.  Every argument
 * check of qmm_matmul (run on x_dev and y_dev), plus x_dev not overlapping
 * W, is made before the first copy: on an error status nothing has been
 * copied or launched.  The sizes of x_dev and y_dev cannot be checked
 * (plain pointers); they are the caller's promise.
 */
QMM_API qmm_status qmm_matmul_host(qmm_wtype wt, const void *W, size_t w_bytes, int64_t M, int64_t K,
                           const void *X_host, qmm_xtype xt, int64_t N, float *Y_host,
                           void *x_dev, float *y_dev,
                           void *workspace, size_t ws_bytes, void *stream);

/*
 * Dequantize W[M, K] to f32 out[M, K] (row-major, device).  Every value is
 * the exact dequantized weight rounded once to nearest-even f32 (exact for
 * Q8_0, Q4_0 and Q6_K).  Used to check the block decoders bit for bit.
 */
QMM_API qmm_status qmm_dequant(qmm_wtype wt, const void *W, size_t w_bytes, int64_t M, int64_t K,
                       float *out, void *stream);

/* Weights and bytes per block of a format (Q8_0 32/34, Q4_0 32/18,
 * Q4_K 256/144, Q6_K 256/210). */
QMM_API qmm_status qmm_block_info(qmm_wtype wt, int *elems, int *bytes);

/*
 * Synchronizes `stream`, then returns and clears the current device's status
 * word: QMM_OK, or QMM_ERR_TIMEOUT if a kernel gave up on a bounded wait
 * since the last call, or QMM_ERR_CUDA if the stream reports an error.
 */
QMM_API qmm_status qmm_last_device_error(void *stream);

/* Static, human-readable name of a status code. */
QMM_API const char *qmm_status_str(qmm_status s);

/*
 * Number of kernels this library has launched in this process so far, across
 * all devices and streams: each successful launch counts once, including a
 * launch recorded into a CUDA graph under stream capture (a graph replay
 * launches nothing through the library and is not counted).  Callers take
 * the difference over a region, e.g. the capture of one pass of their work,
 * to learn how many kernels that work runs.  Never fails.
 */
QMM_API uint64_t qmm_kernel_launches(void);

/*
 * Static-weights mode, process wide, for launches issued after the call
 * (default off; the environment variable QMM_STATIC_WEIGHTS=1 turns it on
 * until this function is first called).  On: the tensor-core GEMV and GEMM
 * and the GEMM's bf16 conversion are launched as programmatic dependents of
 * the preceding kernel on the stream, and each starts streaming its weight
 * blocks W before that kernel has finished; X is read and Y written only
 * after it has.  This hides most of the launch and first-byte latency of a
 * chain of projections (a decode step).  The caller promises that no kernel
 * on the stream writes W between the calls that read it (weights loaded once
 * and then only read, as in inference); otherwise leave it off.  The pages
 * have no counterpart: it is a property of how calls are queued on a GPU.
 */
QMM_API void qmm_set_static_weights(int on);

/*
 * Test hook: upper bound, in SM clock cycles, on every device-side wait of
 * the tensor-core GEMM (default about two seconds).  A tiny limit makes the
 * waits give up, which tests use to exercise the QMM_ERR_TIMEOUT path
 * without a hang.  Affects launches issued after the call, process wide.
 */
QMM_API void qmm_set_wait_limit(uint64_t cycles);

/*
 * Gate/up projections with the SwiGLU product ("cera 0.5.2
 * src/backend/cpu.rs", gemv_q4_0_gate_up_swiglu_with_q8 and
 * silu_mul_inplace):  Y[n, m] = silu(g) * u,  g = sum_k x(n,k) wg(m,k),
 * u = sum_k x(n,k) wu(m,k),  silu(v) = v / (1 + exp(-v)).  Wg and Wu are two
 * M x K matrices of format wt sharing X; 1 <= N <= 16.  Both projections run
 * in one launch of the fused GEMV (qmm_gemv_multi), writing g and u to
 * `workspace` (device, 16-byte aligned, >= 2 * N * M * 4 bytes: g [N][M]
 * then u [N][M], left there), and a second kernel, a programmatic dependent
 * of the first, writes Y [N][M].  g and u meet the qmm_gemv tolerance; Y
 * carries it through the activation (plus f32 rounding of exp and the
 * quotient).  No buffer may overlap another.
 */
QMM_API qmm_status qmm_gemv_swiglu(qmm_wtype wt, const void *Wg, size_t wg_bytes, const void *Wu,
                                   size_t wu_bytes, int64_t M, int64_t K, const void *X, qmm_xtype xt,
                                   int64_t N, float *Y, void *workspace, size_t ws_bytes, void *stream);

/*
 * GEMV kernel choice for 1 <= N <= 2 (Q6_K: N == 1): on (1, or QMM_GEMV_I8=1
 * in the environment) runs the integer tensor-core kernel, which feeds X to
 * mma.sync as exact int8 digits (per
 * 32-element block: T = rint(x 2^(29-E)), E the exponent of the block's
 * largest |x|, in four base-256 digits; |x - T 2^(E-29)| <= 2^-30 * 2^E),
 * and the weights' integer codes as 8-bit operands; off (0, the default)
 * runs the bf16 tensor-core kernel for every N.  Both meet the GEMV
 * tolerance of qmm_gemv.
 * -1 returns to the environment's choice.  Process-wide; takes effect at
 * the next call.  X blocks whose largest |x| is below 2^-98 count as zero
 * on the integer kernel, and a block holding a NaN or an infinity gives NaN
 * outputs.
 */
QMM_API void qmm_set_gemv_i8(int on);

/*
 * GEMV kernel choice for 2 <= N <= 4 (QMM_TC_MAX_N, at most 8) on Q8_0,
 * Q4_0, Q4_K and Q5_K rows: on (1, or QMM_GEMV_TC=1 in the environment)
 * runs the 16-row-tile tensor-core kernel, which feeds X to mma.sync as two
 * binary16 pieces of x * 2^-e with one power-of-two scale e per token
 * (|x - (hi + lo) 2^e| <= 2^-22 |x| + 2^-40 max_k |x|); off (0, the default)
 * runs the ring kernel, whose bf16 pieces keep the f32 exponent range.
 * The tensor-core kernel meets the GEMV tolerance unless a token's
 * activations span more than about 2^39 between entries that meet
 * non-zero weights (an entry 2^40 below the token's largest is lost); the
 * default kernels have no such limit.  -1 returns to the environment's
 * choice.  Process-wide; takes effect at the next call.  The cera pages
 * have no counterpart: this is a GB300 kernel choice.
 */
QMM_API void qmm_set_gemv_tc(int on);

/*
 * Plan of the one-token (N = 1) streaming GEMV, for tuning and tests.
 * rows_per_task: 1, 2 or 4 rows whose units at one 256-weight column one
 * lane computes against the same x values; warps: warps per CTA (1..16);
 * slots: stage slots per warp (1..3); ctas_per_sm: 1 or 2; direct: 1 runs
 * the direct-load variant where it applies (Q4_0 and Q4_K rows: each lane
 * reads its unit with 16-byte global loads into registers, no shared-memory
 * ring; one row per task, no slots), 2 the staged kernel.  0 lets the
 * planner choose that parameter; -1 returns it to the environment
 * (QMM_STREAM_R, QMM_STREAM_WARPS, QMM_STREAM_SLOTS, QMM_STREAM_CPS,
 * QMM_STREAM_DIRECT, each 0 or unset for the planner's choice).  A shape
 * whose forced plan does not fit (shared memory, or rows per task above 1
 * for Q6_K rows whose unit count does not divide 32) runs another GEMV
 * kernel.  Every plan computes the same per-unit sums; only the order in
 * which a row's unit sums are added (and, for Q6_K, its sub-block sums)
 * can differ between plans.  Process-wide; takes effect at the next call.
 * The cera pages have no counterpart: this is a GB300 kernel choice.
 */
QMM_API void qmm_set_gemv_stream(int rows_per_task, int warps, int slots, int ctas_per_sm, int direct);

/*
 * The streaming GEMV's plan for an M x K matrix of type wt on the current
 * device under the present settings: plan[0..5] = grid (CTAs), warps per
 * CTA, slots per warp, rows per task, dynamic shared memory bytes, 1 for
 * the direct-load variant.  plan: 6 host int32, caller-owned.
 * QMM_ERR_UNSUPPORTED: the shape does not fit the kernel (qmm_gemv then
 * runs another kernel); QMM_ERR_CUDA: no device.
 */
QMM_API qmm_status qmm_gemv_stream_plan(qmm_wtype wt, int64_t M, int64_t K, int32_t *plan);

/*
 * Q8_0 activations ("cera 0.5.2 src/backend/cpu.rs",
 * quantize_f32_to_q8_0_into / quantize_f32_to_q8_0_scalar).  For each
 * 32-element block of X[N][K] (f32, or bf16 widened exactly): amax = max |x|
 * (NaN elements ignored), d = amax / 127, id = 1/d if d != 0 and 1/d is
 * finite else 0; scales[b] = d rounded to binary16 and back to f32;
 * quants[e] = rint(x * id) (ties to even) clamped to [-128, 127], NaN -> 0.
 * Every step is correctly rounded f32, so the codes and scales equal any
 * IEEE implementation's bit for bit.  scales: f32 [N][K/32], quants: int8
 * [N][K], device, caller-owned, not overlapping X or each other.  K % 32 ==
 * 0.  Asynchronous on `stream`.
 */
QMM_API qmm_status qmm_quantize_q8_0(const void *X, qmm_xtype xt, int64_t N, int64_t K, float *scales,
                                     int8_t *quants, void *stream);

/*
 * Y[n, m] = sum_b d_w(m, b) scales[n][b] sum_{e in b} q_w(m, e) quants[n][e]
 * (Q4_0 and Q6_K codes with their offsets, Q4_K with its min term), i.e.
 * the projection of dequant(W) on the dequantized Q8_0 activations: the
 * int8 decode arithmetic of "cera 0.5.2 src/backend/cpu.rs"
 * (gemm_preq_dispatch: weights against pre-quantized activation scales and
 * quants).  1 <= N <= 16.  The integer sums are exact; only the f32
 * combination of block scales rounds (|Y - exact| <= 1e-5 * sum|w x_q| +
 * 1e-6).  Needs the tensor-core geometry: K % 256 == 0, W, scales and
 * quants 16-byte aligned, 16-byte row pitch; otherwise
 * QMM_ERR_UNSUPPORTED (there is no byte-addressed variant).  Y: f32 [N][M],
 * overwritten, not overlapping any input.
 */
QMM_API qmm_status qmm_gemv_preq(qmm_wtype wt, const void *W, size_t w_bytes, int64_t M, int64_t K,
                                 const float *scales, const int8_t *quants, int64_t N, float *Y, void *stream);

/* Workspace of qmm_gemv_q8act: the quants (N*K bytes, padded to 16) then the
 * scales (N*K/32 floats). */
QMM_API size_t qmm_q8act_workspace_bytes(int64_t N, int64_t K);

/*
 * qmm_quantize_q8_0 of X into `workspace` followed by qmm_gemv_preq on it
 * (two kernels, stream-ordered): the Q8_0-activation GEMV of f32 or bf16 X,
 * 1 <= N <= 16.  workspace: device, 16-byte aligned, at least
 * qmm_q8act_workspace_bytes(N, K), not overlapping W, X or Y.
 */
QMM_API qmm_status qmm_gemv_q8act(qmm_wtype wt, const void *W, size_t w_bytes, int64_t M, int64_t K,
                                  const void *X, qmm_xtype xt, int64_t N, float *Y, void *workspace,
                                  size_t ws_bytes, void *stream);

/*
 * Prefill on Q8_0 activations, 1 <= N <= QMM_GEMM_MAX_N: the arithmetic of
 * the pages' batched path ("cera 0.5.2 src/backend/cpu.rs",
 * gemm_preq_dispatch after quantize_f32_to_q8_0_into: every 32-element block
 * of each token quantized to Q8_0, then the weights against the quantized
 * activations).  X[N][K] (f32 or bf16) is quantized exactly as
 * qmm_quantize_q8_0 does, each activation is replaced by bf16(scale * code)
 * (scale * code is exact in f32, then rounded once to bf16) in `workspace`
 * (>= qmm_gemm_q8act_workspace_bytes(N, K) = N*K*2 bytes, 16-byte aligned,
 * not overlapping W, X or Y), and the tensor-core GEMM of qmm_gemm runs on
 * it.  Y[N][M] f32, overwritten.  Reference: the exact projection of
 * dequant(W) on the dequantized activations; tolerance that of qmm_gemm
 * (2e-3 * sum|w x_q| + 1e-5).  Needs qmm_gemm's geometry (K % 256 == 0,
 * 16-byte aligned rows and W), else QMM_ERR_UNSUPPORTED.  Two kernels,
 * asynchronous on `stream`; nothing is written on an error status.
 */
QMM_API size_t qmm_gemm_q8act_workspace_bytes(int64_t N, int64_t K);
QMM_API qmm_status qmm_gemm_q8act(qmm_wtype wt, const void *W, size_t w_bytes, int64_t M, int64_t K,
                                  const void *X, qmm_xtype xt, int64_t N, float *Y, void *workspace,
                                  size_t ws_bytes, void *stream);

/*
 * Gate/up projections with the SwiGLU product on the tensor-core GEMM,
 * 1 <= N <= QMM_GEMM_MAX_N ("cera 0.5.2 src/backend/cpu.rs",
 * gemv_q4_0_gate_up_swiglu_with_q8 and silu_mul_inplace, for prefill):
 * Y[n, m] = silu(g) * u with g = X Wg^T, u = X Wu^T, two M x K matrices of
 * format wt sharing X.  One GEMM launch computes both projections (its grid
 * covers the row tiles of Wg and then those of Wu; X is converted to bf16
 * once when it is f32), then a programmatically dependent kernel writes Y.
 * workspace (device, 16-byte aligned, >= qmm_gemm_swiglu_workspace_bytes):
 * the bf16 X (f32 X only, padded to 16 bytes), then g [N][M] and u [N][M]
 * (left there).  g and u meet the qmm_gemm tolerance; Y carries it through
 * the activation.  Same geometry requirements as qmm_gemm; no buffer may
 * overlap another.
 */
QMM_API size_t qmm_gemm_swiglu_workspace_bytes(int64_t N, int64_t M, int64_t K, qmm_xtype xt);
QMM_API qmm_status qmm_gemm_swiglu(qmm_wtype wt, const void *Wg, size_t wg_bytes, const void *Wu,
                                   size_t wu_bytes, int64_t M, int64_t K, const void *X, qmm_xtype xt,
                                   int64_t N, float *Y, void *workspace, size_t ws_bytes, void *stream);

#ifdef __cplusplus
}
#endif
#endif
