// generic.cu -- byte-addressed kernels that accept any alignment:
//   * dequant      : W -> f32 [M,K] (the bit-exact decoder check)
//   * gemv_generic : Y[N,M] = X[N,K] W^T for 1 <= N <= 16, one warp per row
//   * x_to_bf16    : f32 -> bf16 (round to nearest even) for the GEMM input
#include "decode_bytes.cuh"
#include "kernels.h"

namespace qmm {

template <int F>
__global__ void __launch_bounds__(256) dequant_kernel(const uint8_t *__restrict__ W, int64_t M, int64_t K,
                                                      float *__restrict__ out) {
    const int64_t units_per_row = K / 32;
    const int64_t total = M * units_per_row;
    const int64_t row_bytes = K / Blk<F>::E * Blk<F>::B;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t m = i / units_per_row, u = i % units_per_row;
        float w[32];
        decode_unit<F>(W + m * row_bytes, u, w);
        float4 *o = reinterpret_cast<float4 *>(out + m * K + u * 32);
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = make_float4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
    }
}

template <int F, bool XBF16>
__global__ void __launch_bounds__(256) gemv_generic_kernel(const uint8_t *__restrict__ W, int64_t M, int64_t K,
                                                           const void *__restrict__ Xv, int N,
                                                           float *__restrict__ Y) {
    const int lane = threadIdx.x & 31;
    const int64_t m = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (m >= M) return;
    const int64_t row_bytes = K / Blk<F>::E * Blk<F>::B;
    const uint8_t *row = W + m * row_bytes;
    float acc[16];
#pragma unroll
    for (int n = 0; n < 16; ++n) acc[n] = 0.f;
    for (int64_t u = lane; u < K / 32; u += 32) {
        float w[32];
        decode_unit<F>(row, u, w);
#pragma unroll
        for (int n = 0; n < 16; ++n) {
            if (n < N) {
                float s = 0.f;
                if constexpr (XBF16) {
                    const __nv_bfloat16 *x = reinterpret_cast<const __nv_bfloat16 *>(Xv) + n * K + u * 32;
#pragma unroll
                    for (int e = 0; e < 32; ++e) s = fmaf(w[e], __bfloat162float(x[e]), s);
                } else {
                    const float *x = reinterpret_cast<const float *>(Xv) + n * K + u * 32;
#pragma unroll
                    for (int e = 0; e < 32; ++e) s = fmaf(w[e], __ldg(x + e), s);
                }
                acc[n] += s;
            }
        }
    }
#pragma unroll
    for (int n = 0; n < 16; ++n) {
        if (n < N) {
            float v = acc[n];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            if (lane == 0) Y[(int64_t)n * M + m] = v;
        }
    }
}

// 8 elements per thread per step (two 16-byte loads, one 16-byte store) when
// X and out are 16-byte aligned; grid-stride, so any count is covered.
__global__ void x_to_bf16_kernel(const float *__restrict__ X, int64_t count, __nv_bfloat16 *__restrict__ out) {
    pdl_launch_dependents();
    pdl_wait();   // X may come from the preceding kernel
    const int64_t stride = (int64_t)gridDim.x * blockDim.x * 8;
    const bool vec = ((reinterpret_cast<uintptr_t>(X) | reinterpret_cast<uintptr_t>(out)) & 15) == 0;
    for (int64_t i8 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 8; i8 < count; i8 += stride) {
        if (vec && i8 + 7 < count) {
            const float4 a = *reinterpret_cast<const float4 *>(X + i8);
            const float4 b = *reinterpret_cast<const float4 *>(X + i8 + 4);
            uint4 o;
            o.x = pack_bf16x2(a.x, a.y);
            o.y = pack_bf16x2(a.z, a.w);
            o.z = pack_bf16x2(b.x, b.y);
            o.w = pack_bf16x2(b.z, b.w);
            *reinterpret_cast<uint4 *>(out + i8) = o;
        } else {
            for (int64_t i = i8; i < count && i < i8 + 8; ++i) out[i] = __float2bfloat16_rn(X[i]);
        }
    }
}

// out[i] = silu(g[i]) * u[i], silu(v) = v / (1 + exp(-v)) ("cera 0.5.2
// src/backend/cpu.rs", silu_mul_inplace: the SwiGLU product of the gate and
// up projections).  exp overflows to infinity for v < -88, where the
// quotient is -0: the exact value is below 1e-36 * |v|.
__device__ __forceinline__ float silu_mul(float v, float w) { return v / (1.0f + expf(-v)) * w; }

// Grid-stride over 4-element groups (16-byte loads and stores when all three
// arrays are 16-byte aligned), a few thousand CTAs at most: one element per
// thread in a CTA per 256 elements made block scheduling the limit.
__global__ void swiglu_kernel(const float *__restrict__ g, const float *__restrict__ u, int64_t count,
                              float *__restrict__ out) {
    pdl_launch_dependents();
    pdl_wait();   // g and u come from the preceding kernel
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t t0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const bool vec = (((uintptr_t)g | (uintptr_t)u | (uintptr_t)out) & 15u) == 0;
    const int64_t n4 = vec ? count / 4 : 0;
    for (int64_t i = t0; i < n4; i += stride) {
        const float4 a = reinterpret_cast<const float4 *>(g)[i], b = reinterpret_cast<const float4 *>(u)[i];
        reinterpret_cast<float4 *>(out)[i] =
            make_float4(silu_mul(a.x, b.x), silu_mul(a.y, b.y), silu_mul(a.z, b.z), silu_mul(a.w, b.w));
    }
    for (int64_t i = 4 * n4 + t0; i < count; i += stride) out[i] = silu_mul(g[i], u[i]);
}

static int grid_for(int64_t work, int per_block) {
    int64_t g = (work + per_block - 1) / per_block;
    if (g > (1 << 20)) g = 1 << 20;
    return (int)(g < 1 ? 1 : g);
}

cudaError_t launch_dequant(int fmt, const uint8_t *W, int64_t M, int64_t K, float *out, cudaStream_t st) {
    const int g = grid_for(M * (K / 32), 256);
    switch (fmt) {
    case Q8_0: dequant_kernel<Q8_0><<<g, 256, 0, st>>>(W, M, K, out); break;
    case Q4_0: dequant_kernel<Q4_0><<<g, 256, 0, st>>>(W, M, K, out); break;
    case Q4_K: dequant_kernel<Q4_K><<<g, 256, 0, st>>>(W, M, K, out); break;
    case Q6_K: dequant_kernel<Q6_K><<<g, 256, 0, st>>>(W, M, K, out); break;
    case Q5_K: dequant_kernel<Q5_K><<<g, 256, 0, st>>>(W, M, K, out); break;
    default: return cudaErrorInvalidValue;
    }
    return launched(cudaGetLastError());
}

template <int F>
static void gemv_generic_dispatch(const uint8_t *W, int64_t M, int64_t K, const void *X, int xbf16, int N,
                                  float *Y, cudaStream_t st) {
    const int g = (int)((M + 7) / 8);
    if (xbf16)
        gemv_generic_kernel<F, true><<<g, 256, 0, st>>>(W, M, K, X, N, Y);
    else
        gemv_generic_kernel<F, false><<<g, 256, 0, st>>>(W, M, K, X, N, Y);
}

cudaError_t launch_gemv_generic(int fmt, const uint8_t *W, int64_t M, int64_t K, const void *X, int xbf16,
                                int N, float *Y, cudaStream_t st) {
    switch (fmt) {
    case Q8_0: gemv_generic_dispatch<Q8_0>(W, M, K, X, xbf16, N, Y, st); break;
    case Q4_0: gemv_generic_dispatch<Q4_0>(W, M, K, X, xbf16, N, Y, st); break;
    case Q4_K: gemv_generic_dispatch<Q4_K>(W, M, K, X, xbf16, N, Y, st); break;
    case Q6_K: gemv_generic_dispatch<Q6_K>(W, M, K, X, xbf16, N, Y, st); break;
    case Q5_K: gemv_generic_dispatch<Q5_K>(W, M, K, X, xbf16, N, Y, st); break;
    default: return cudaErrorInvalidValue;
    }
    return launched(cudaGetLastError());
}

cudaError_t launch_x_to_bf16(const float *X, int64_t count, uint16_t *out, bool pdl, cudaStream_t st) {
    if (count <= 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid_for((count + 7) / 8, 256), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, x_to_bf16_kernel, X, count, reinterpret_cast<__nv_bfloat16 *>(out));
    if (e != cudaSuccess) return e;
    return launched(cudaGetLastError());
}

}  // namespace qmm

namespace qmm {

cudaError_t launch_swiglu(const float *g, const float *u, int64_t count, float *out, bool pdl, cudaStream_t st) {
    if (count <= 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    const int64_t groups = (count + 3) / 4;
    int64_t blocks = (groups + 255) / 256;
    if (blocks > 2432) blocks = 2432;   // 16 per SM on 152 SMs
    cfg.gridDim = dim3((unsigned)blocks, 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, swiglu_kernel, g, u, count, out);
    if (e != cudaSuccess) return e;
    return launched(cudaGetLastError());
}

}  // namespace qmm
