// gemv_i8_q8.cu -- Q8_0 activations ("cera 0.5.2 src/backend/cpu.rs",
// quantize_f32_to_q8_0_scalar) and the integer tensor-core GEMV on them,
// 1 <= N <= 16.  See gemv_i8.cuh.
#include "gemv_i8.cuh"

namespace qmm {
namespace {

// One warp per 32-element block, lane e = element e.  The float steps follow
// the quantizer: amax = max |x| (a NaN element never wins a max), d =
// amax / 127, id = 1/d when d != 0 and 1/d is finite (else 0), code =
// rint(x * id) clamped to [-128, 127] with NaN -> 0, scale = d through
// binary16.  Division, reciprocal and product are correctly rounded, so the
// codes and scales are those of any IEEE float implementation.
// BF16OUT: instead of codes and scales, write the dequantized activation
// bf16(scale * code) (scale * code is exact in f32: 11 x 8 bits), the X
// operand of the tensor-core GEMM on Q8_0 activations.
template <bool XBF16, bool BF16OUT>
__global__ void __launch_bounds__(256) quantize_q8_0_kernel(const void *__restrict__ Xv, int64_t nblocks,
                                                             float *__restrict__ scales, int8_t *__restrict__ quants,
                                                             __nv_bfloat16 *__restrict__ xq) {
    const int lane = threadIdx.x & 31;
    pdl_launch_dependents();
    pdl_wait();   // X may come from the preceding kernel
    for (int64_t b = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5); b < nblocks; b += (int64_t)gridDim.x * 8) {
        float v;
        if constexpr (XBF16)
            v = __uint_as_float((uint32_t)reinterpret_cast<const uint16_t *>(Xv)[b * 32 + lane] << 16);
        else
            v = reinterpret_cast<const float *>(Xv)[b * 32 + lane];
        float amax = fabsf(v);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        amax = fmaxf(0.f, amax);
        const float d = __fdiv_rn(amax, 127.0f);
        const float r = __frcp_rn(d);
        const float id = (d != 0.0f && isfinite(r)) ? r : 0.0f;
        float q = rintf(__fmul_rn(v, id));
        q = isnan(q) ? 0.0f : fminf(fmaxf(q, -128.0f), 127.0f);
        const float dh = __half2float(__float2half_rn(d));
        if constexpr (BF16OUT) {
            xq[b * 32 + lane] = __float2bfloat16_rn(dh * q);
        } else {
            quants[b * 32 + lane] = (int8_t)(int)q;
            if (lane == 0) scales[b] = dh;
        }
    }
}

template <int F, int NTOK>
cudaError_t q8_rows(const GemvPlan &p, const GemvSegs &segs, const XIn &xin, int64_t K, int N, bool pdl,
                    unsigned *status, uint64_t limit, cudaStream_t st, const AmaxOut &amax) {
    if (p.rows == 64) return launch_i8<F, XM_Q8, NTOK, false, 4, 1>(p, segs, xin, K, N, pdl, status, limit, st, amax);
    if (p.rows == 128) return launch_i8<F, XM_Q8, NTOK, false, 8, 1>(p, segs, xin, K, N, pdl, status, limit, st, amax);
    return cudaErrorInvalidValue;
}

template <int F>
cudaError_t q8_n(const GemvPlan &p, const GemvSegs &segs, const XIn &xin, int64_t K, int N, bool pdl,
                 unsigned *status, uint64_t limit, cudaStream_t st, const AmaxOut &amax) {
    if (N == 1) return q8_rows<F, 1>(p, segs, xin, K, N, pdl, status, limit, st, amax);
    if (N <= 4) return q8_rows<F, 4>(p, segs, xin, K, N, pdl, status, limit, st, amax);
    if (N <= 8) return q8_rows<F, 8>(p, segs, xin, K, N, pdl, status, limit, st, amax);
    if (N <= 16) return q8_rows<F, 16>(p, segs, xin, K, N, pdl, status, limit, st, amax);
    return cudaErrorInvalidValue;
}

template <int F>
int maxc_f(int N, int rows) {
    auto pick = [&](auto c64, auto c128) { return rows == 64 ? c64 : c128; };
    if (N == 1) return pick(i8_maxc<F, XM_Q8, 1, false, 4, 1>(), i8_maxc<F, XM_Q8, 1, false, 8, 1>());
    if (N <= 4) return pick(i8_maxc<F, XM_Q8, 4, false, 4, 1>(), i8_maxc<F, XM_Q8, 4, false, 8, 1>());
    if (N <= 8) return pick(i8_maxc<F, XM_Q8, 8, false, 4, 1>(), i8_maxc<F, XM_Q8, 8, false, 8, 1>());
    if (N <= 16) return pick(i8_maxc<F, XM_Q8, 16, false, 4, 1>(), i8_maxc<F, XM_Q8, 16, false, 8, 1>());
    return 0;
}

}  // namespace

namespace {
cudaError_t launch_quant(const void *X, int xbf16, int64_t count, float *scales, int8_t *quants, uint16_t *xq,
                         bool pdl, cudaStream_t st) {
    const int64_t nblocks = count / 32;
    if (nblocks <= 0) return cudaSuccess;
    // grid-stride: at most 16 CTAs per SM of 152 (one 32-element block per
    // warp and CTA pass; more, smaller CTAs made block scheduling the limit)
    int64_t grid = (nblocks + 7) / 8;
    if (grid > 2432) grid = 2432;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    __nv_bfloat16 *o = reinterpret_cast<__nv_bfloat16 *>(xq);
    cudaError_t e;
    if (xq)
        e = xbf16 ? cudaLaunchKernelEx(&cfg, quantize_q8_0_kernel<true, true>, X, nblocks, scales, quants, o)
                  : cudaLaunchKernelEx(&cfg, quantize_q8_0_kernel<false, true>, X, nblocks, scales, quants, o);
    else
        e = xbf16 ? cudaLaunchKernelEx(&cfg, quantize_q8_0_kernel<true, false>, X, nblocks, scales, quants, o)
                  : cudaLaunchKernelEx(&cfg, quantize_q8_0_kernel<false, false>, X, nblocks, scales, quants, o);
    if (e != cudaSuccess) return e;
    return launched(cudaGetLastError());
}
}  // namespace

cudaError_t launch_quantize_q8_0(const void *X, int xbf16, int64_t count, float *scales, int8_t *quants, bool pdl,
                                 cudaStream_t st) {
    return launch_quant(X, xbf16, count, scales, quants, nullptr, pdl, st);
}

cudaError_t launch_quantize_q8_0_bf16(const void *X, int xbf16, int64_t count, uint16_t *out, bool pdl,
                                      cudaStream_t st) {
    return launch_quant(X, xbf16, count, nullptr, nullptr, out, pdl, st);
}

int gemv_i8_q8_maxc(int fmt, int N, int rows) {
    if (rows != 64 && rows != 128) return 0;
    switch (fmt) {
    case Q8_0: return maxc_f<Q8_0>(N, rows);
    case Q4_0: return maxc_f<Q4_0>(N, rows);
    case Q4_K: return maxc_f<Q4_K>(N, rows);
    case Q6_K: return maxc_f<Q6_K>(N, rows);
    case Q5_K: return maxc_f<Q5_K>(N, rows);
    default: return 0;
    }
}

cudaError_t launch_gemv_i8_q8(int fmt, const GemvPlan &plan, const GemvSegs &segs, const int8_t *quants,
                              const float *scales, int64_t K, int N, bool pdl, unsigned *status, uint64_t limit,
                              cudaStream_t st, unsigned long long *amax_ws, int32_t *idx, float *val) {
    if (plan.ks < 1 || plan.ks > 8) return cudaErrorInvalidValue;
    if (segs.nseg < 1 || segs.nseg > QMM_MAX_SEGS || (amax_ws && segs.nseg != 1)) return cudaErrorInvalidValue;
    const AmaxOut amax{amax_ws, amax_ws ? reinterpret_cast<unsigned *>(amax_ws + N) : nullptr, idx, val};
    const XIn xin{quants, scales};
    switch (fmt) {
    case Q8_0: return q8_n<Q8_0>(plan, segs, xin, K, N, pdl, status, limit, st, amax);
    case Q4_0: return q8_n<Q4_0>(plan, segs, xin, K, N, pdl, status, limit, st, amax);
    case Q4_K: return q8_n<Q4_K>(plan, segs, xin, K, N, pdl, status, limit, st, amax);
    case Q6_K: return q8_n<Q6_K>(plan, segs, xin, K, N, pdl, status, limit, st, amax);
    case Q5_K: return q8_n<Q5_K>(plan, segs, xin, K, N, pdl, status, limit, st, amax);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace qmm
