// gemv_i8_exact.cu -- the integer tensor-core GEMV on exact int8 digits of
// f32 or bf16 X (1 <= N <= 2; Q6_K: N == 1).  See gemv_i8.cuh.
#include "gemv_i8.cuh"

namespace qmm {
namespace {

template <int F, int NTOK, bool XBF16>
cudaError_t exact_rows(const GemvPlan &p, const GemvSegs &segs, const XIn &xin, int64_t K, int N, bool pdl,
                       unsigned *status, uint64_t limit, cudaStream_t st, const AmaxOut &amax) {
    if (p.rows == 64) return launch_i8<F, XM_EXACT, NTOK, XBF16, 4, 1>(p, segs, xin, K, N, pdl, status, limit, st, amax);
    if (p.rows == 128 && p.rg == 2)
        return launch_i8<F, XM_EXACT, NTOK, XBF16, 4, 2>(p, segs, xin, K, N, pdl, status, limit, st, amax);
    if (p.rows == 128) return launch_i8<F, XM_EXACT, NTOK, XBF16, 8, 1>(p, segs, xin, K, N, pdl, status, limit, st, amax);
    return cudaErrorInvalidValue;
}

template <int F, bool XBF16>
cudaError_t exact_n(const GemvPlan &p, const GemvSegs &segs, const XIn &xin, int64_t K, int N, bool pdl,
                    unsigned *status, uint64_t limit, cudaStream_t st, const AmaxOut &amax) {
    if (N == 1) return exact_rows<F, 1, XBF16>(p, segs, xin, K, N, pdl, status, limit, st, amax);
    if constexpr (F != Q6_K) {
        if (N == 2) return exact_rows<F, 2, XBF16>(p, segs, xin, K, N, pdl, status, limit, st, amax);
    }
    return cudaErrorInvalidValue;
}

template <int F, int NTOK, bool XBF16>
int maxc_rows(int rows, int rg) {
    if (rows == 64) return i8_maxc<F, XM_EXACT, NTOK, XBF16, 4, 1>();
    return rg == 2 ? i8_maxc<F, XM_EXACT, NTOK, XBF16, 4, 2>() : i8_maxc<F, XM_EXACT, NTOK, XBF16, 8, 1>();
}

template <int F>
int maxc_f(int N, int xbf16, int rows, int rg) {
    if (N == 1) return xbf16 ? maxc_rows<F, 1, true>(rows, rg) : maxc_rows<F, 1, false>(rows, rg);
    if (F != Q6_K && N == 2) return xbf16 ? maxc_rows<F, 2, true>(rows, rg) : maxc_rows<F, 2, false>(rows, rg);
    return 0;
}

}  // namespace

int gemv_i8_exact_maxc(int fmt, int N, int xbf16, int rows, int rg) {
    if (rows != 64 && rows != 128) return 0;
    switch (fmt) {
    case Q8_0: return maxc_f<Q8_0>(N, xbf16, rows, rg);
    case Q4_0: return maxc_f<Q4_0>(N, xbf16, rows, rg);
    case Q4_K: return maxc_f<Q4_K>(N, xbf16, rows, rg);
    case Q6_K: return maxc_f<Q6_K>(N, xbf16, rows, rg);
    case Q5_K: return maxc_f<Q5_K>(N, xbf16, rows, rg);
    default: return 0;
    }
}

cudaError_t launch_gemv_i8_exact(int fmt, const GemvPlan &plan, const GemvSegs &segs, const void *X, int xbf16,
                                 int64_t K, int N, bool pdl, unsigned *status, uint64_t limit, cudaStream_t st,
                                 unsigned long long *amax_ws, int32_t *idx, float *val) {
    if (plan.ks < 1 || plan.ks > 8) return cudaErrorInvalidValue;
    if (segs.nseg < 1 || segs.nseg > QMM_MAX_SEGS || (amax_ws && segs.nseg != 1)) return cudaErrorInvalidValue;
    const AmaxOut amax{amax_ws, amax_ws ? reinterpret_cast<unsigned *>(amax_ws + N) : nullptr, idx, val};
    const XIn xin{X, nullptr};
    switch (fmt) {
    case Q8_0: return xbf16 ? exact_n<Q8_0, true>(plan, segs, xin, K, N, pdl, status, limit, st, amax)
                            : exact_n<Q8_0, false>(plan, segs, xin, K, N, pdl, status, limit, st, amax);
    case Q4_0: return xbf16 ? exact_n<Q4_0, true>(plan, segs, xin, K, N, pdl, status, limit, st, amax)
                            : exact_n<Q4_0, false>(plan, segs, xin, K, N, pdl, status, limit, st, amax);
    case Q4_K: return xbf16 ? exact_n<Q4_K, true>(plan, segs, xin, K, N, pdl, status, limit, st, amax)
                            : exact_n<Q4_K, false>(plan, segs, xin, K, N, pdl, status, limit, st, amax);
    case Q6_K: return xbf16 ? exact_n<Q6_K, true>(plan, segs, xin, K, N, pdl, status, limit, st, amax)
                            : exact_n<Q6_K, false>(plan, segs, xin, K, N, pdl, status, limit, st, amax);
    case Q5_K: return xbf16 ? exact_n<Q5_K, true>(plan, segs, xin, K, N, pdl, status, limit, st, amax)
                            : exact_n<Q5_K, false>(plan, segs, xin, K, N, pdl, status, limit, st, amax);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace qmm
