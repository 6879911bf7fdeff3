/*
 * qmm_oracle.h -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously-correct host implementation of the block-quantized
 * projection matmul  Y[n,m] = sum_k w(m,k) * x(n,k)  over GGUF/ggml weight
 * blocks (Q8_0, Q4_0, Q4_K, Q6_K), in IEEE double precision.
 *
 * Only the test-suite, the smoke check and the benchmark's CPU-baseline leg
 * may load or call this code.  The CUDA library never includes, links or
 * calls it, and it shares no header, table or helper with the CUDA library.
 *
 * Sources (cera, docs.rs source pages):
 *   - "cera 0.5.2 src/backend/cpu.rs": matmul_q4_0_f32, matmul_q8_0_f32,
 *     matmul_q4km_f32 (the scalar definition: per row, sum over blocks of a
 *     block dot product, output overwritten), repack_q4_0_8x8 (Q4_0 byte
 *     layout and nibble order, value = nibble - 8), repack_q4_k_8x8 (Q4_K
 *     field order d, dmin, scales, qs; sub-block nibble order; the products
 *     d*sc and dmin*m), gemm_preq_dispatch (k must be a multiple of the block
 *     size; weight bytes >= m * blocks * block_bytes).
 *   - "cera 0.5.2 src/backend/cpu.rs": quantize_f32_to_q8_0_scalar (the
 *     Q8_0 activation quantizer of the int8 decode and prefill paths: scale
 *     amax/127 through binary16, codes rounded half to even and clamped).
 *   - "cera 0.3.1 src/model/gpu_lfm2.rs": GpuLfm2Model::new weight upload
 *     (block byte sizes: Q4_K 144 B, Q6_K 210 B per 256 weights).
 * Readings where the pages are silent (Q8_0 field order, Q4_K 6-bit scale
 * packing, Q6_K and Q5_K byte order and bit maps) follow the published
 * GGUF/ggml block definitions and are marked READING at the function that
 * uses them.
 *
 * Pins: every function here is checked by the CPU test-suite against worked
 * blocks, closed forms, invariants, a library f16 decoder and an independent
 * brute-force path.  The Q4_K scale packing and the Q6_K bit map are pinned
 * only to their READING (no GGUF file is available to compare with), and so
 * is the Q5_K layout: parity unpinned against real GGUF files for those
 * three layouts.
 */
#ifndef QMM_ORACLE_H
#define QMM_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Weight formats, numbered as the library's public enum. */
enum { ORC_Q8_0 = 0, ORC_Q4_0 = 1, ORC_Q4_K = 2, ORC_Q6_K = 3, ORC_Q5_K = 4 };
/* Activation element types. */
enum { ORC_X_F32 = 0, ORC_X_BF16 = 1 };

/* Elements / bytes per block; returns 0 on success, -1 for an unknown format. */
int orc_block_info(int wtype, int *elems, int *bytes);

/* IEEE binary16 bit pattern -> exact double (normals, subnormals, +-0, inf, nan). */
double orc_f16_to_f64(uint16_t h);

/* Dequantize one block to exact doubles (out has 32 or 256 entries). */
int orc_dequant_block(int wtype, const uint8_t *blk, double *out);

/* Dequantize W[M,K] (raw blocks, row-major) to exact doubles [M,K]. */
int orc_dequant(int wtype, const uint8_t *w, int64_t M, int64_t K, double *out);

/* Same values rounded once (round-to-nearest-even) to float. */
int orc_dequant_f32(int wtype, const uint8_t *w, int64_t M, int64_t K, float *out);

/*
 * Y[n, j] = sum_k w(rows[j], k) * x(n, k),  S[n, j] = sum_k |w(rows[j],k) * x(n,k)|
 * for j in [0, nrows), both in double.  x is [N,K] row-major, f32 or bf16
 * (bf16 given as uint16 bit patterns).  rows == NULL means rows 0..nrows-1.
 * Y and S are [N, nrows] row-major.  nthreads <= 0 uses every online core.
 * Returns 0, or -1 on a bad argument.
 */
int orc_matmul_rows(int wtype, const uint8_t *w, int64_t M, int64_t K,
                    const void *x, int xtype, int64_t N,
                    const int64_t *rows, int64_t nrows,
                    double *Y, double *S, int nthreads);

/*
 * IEEE binary32 -> binary16 bit pattern, round to nearest even: subnormal
 * results, overflow to infinity (|f| >= 65520), NaN stays a (quiet) NaN.
 */
uint16_t orc_f32_to_f16(float f);

/*
 * Q8_0 quantization of activations ("cera 0.5.2 src/backend/cpu.rs",
 * quantize_f32_to_q8_0_scalar), per 32-element block of x[0..n):
 *   amax = max |x| (NaN elements ignored, as the float max fold does);
 *   d = amax / 127 (float);  id = 1/d if d != 0 and 1/d is finite, else 0;
 *   scales[b] = d rounded to binary16 and back;
 *   quants[e] = rint(x[e] * id) (ties to even), clamped to [-128, 127],
 *   NaN -> 0 (the saturating float-to-int8 conversion).
 * All arithmetic in float.  n % 32 != 0 -> -1, else 0.
 */
int orc_quantize_q8_0(const float *x, int64_t n, float *scales, int8_t *quants);

#ifdef __cplusplus
}
#endif
#endif
