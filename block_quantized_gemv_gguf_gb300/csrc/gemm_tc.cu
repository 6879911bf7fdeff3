// gemm_tc.cu -- prefill GEMM Y[N,M] = X[N,K] * dequant(W)[M,K]^T on the
// 5th-generation tensor cores (tcgen05), for 16 < N <= 512 tokens.
//
// One CTA computes a 128-row (weights) x BN-column (tokens) tile of Y^T over
// the whole K.  Warp roles (224 threads):
//   warp 0      TMA producer of raw weight bytes: one 2-D tensor copy per
//               256-weight chunk of the tile's 128 rows (u16 view of W);
//   warp 1      TMA producer of bf16 X tiles (64 k x BN tokens, 128-byte
//               swizzle = the canonical K-major UMMA layout);
//   warp 2      TMEM allocation and the single MMA-issuing thread:
//               tcgen05.mma kind::f16, M=128, N=BN, K=16, f32 accumulator;
//   warps 3..6  dequantizers: thread i owns weight row i of the tile, decodes
//               64 weights per stage straight from the raw bytes to bf16 and
//               writes them swizzled as the K-major A operand; afterwards the
//               same warps read the accumulator out of TMEM and store Y.
// Each weight block is dequantized once per CTA and reused by all BN token
// columns of the MMA, which is what makes the tile compute-bound at N >= 256
// ("cera 0.3.1 src/model/gpu_lfm2.rs", build_mul_mat_pipeline: decode a
// k-tile of W into shared memory once, reuse it across every token column).
//
// All waits are bounded (wait_limit cycles).  A CTA that gives up sets a
// shared abort flag that every other wait observes, drains its own in-flight
// TMA copies and MMAs, frees its TMEM, writes QMM_ERR_TIMEOUT to the status
// word and returns.
#include <atomic>

#include "common.cuh"
#include "kernels.h"

namespace qmm {

namespace {

constexpr int BM = 128;          // weight rows per tile (TMEM lanes)
constexpr int KC = 256;          // weights per raw chunk
constexpr int BK = 64;           // weights per MMA stage (one 128-byte row)
constexpr int SR = 2;            // raw chunk stages
constexpr int NUM_THREADS = 224;
constexpr int WARP_WPROD = 0, WARP_XPROD = 1, WARP_MMA = 2, WARP_DQ0 = 3;

template <int F> struct Raw;
template <> struct Raw<Q8_0> { static constexpr int bytes = 272; };   // 8 blocks of 34
template <> struct Raw<Q4_0> { static constexpr int bytes = 144; };   // 8 blocks of 18
template <> struct Raw<Q4_K> { static constexpr int bytes = 144; };   // 1 super-block
template <> struct Raw<Q6_K> { static constexpr int bytes = 240; };   // 210 B + alignment slack

template <int F, int BN> struct Layout {
    static constexpr int SA = BN == 256 ? 3 : 4;
    static constexpr int A_BYTES = BM * 128;
    static constexpr int X_BYTES = BN * 128;
    static constexpr int RAW_BYTES = BM * Raw<F>::bytes;
    static constexpr int OFF_A = 0;
    static constexpr int OFF_X = OFF_A + SA * A_BYTES;
    static constexpr int OFF_RAW = OFF_X + SA * X_BYTES;
    static constexpr int OFF_BAR = OFF_RAW + SR * RAW_BYTES;
    static constexpr int NUM_BARS = 2 * SR + 3 * SA + 1;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
    static constexpr int TOTAL = OFF_MISC + 64;
    static constexpr int SMEM = TOTAL + 1024;     // 1024-byte alignment slack
    static constexpr int TMEM_COLS = BN < 32 ? 32 : BN;
    static_assert(SMEM <= 232448, "shared memory budget");
};

struct Ctl {
    volatile unsigned *abort;
    uint64_t limit;
};

// Bounded wait that also gives up as soon as another thread has aborted.
__device__ __forceinline__ bool wait_ok(const Ctl &c, uint64_t *bar, uint32_t parity, uint64_t limit) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*c.abort) return false;
        if ((uint64_t)(clock64() - t0) > limit) {
            *c.abort = 1u;
            return false;
        }
    }
}

// Drain wait: used after an abort for copies this thread issued itself;
// those complete on their own, so only the time limit applies.
__device__ __forceinline__ void drain(uint64_t *bar, uint32_t parity, uint64_t limit) {
    (void)mbar_wait(bar, parity, limit);
}

// ---------------------------------------------------------------------------
// Dequantization of 64 weights (one MMA stage) of one row, straight from the
// raw bytes in shared memory into 32 bf16x2 words (k order).
// The integer codes are turned into floats 128 + v (or 32768 + v) by byte
// permutes into the mantissa of a constant, and the offset is folded into a
// per-block constant: w = scale * (128 + v) - scale * (128 + offset).
// ---------------------------------------------------------------------------
template <int F>
__device__ __forceinline__ void dequant64(const uint8_t *rb, int sub, uint32_t (&o)[32]);

template <>
__device__ __forceinline__ void dequant64<Q4_0>(const uint8_t *rb, int sub, uint32_t (&o)[32]) {
#pragma unroll
    for (int bb = 0; bb < 2; ++bb) {
        const uint8_t *b = rb + 18 * (2 * sub + bb);
        const float d = f16_bits(*reinterpret_cast<const uint16_t *>(b));
        const float c = -136.f * d;   // exact: d * (128 + q) - 136 d = d (q - 8)
        float w[32];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const uint32_t word = lds_u32_a2(b + 2 + 4 * t);
            const uint32_t lo = word & 0x0F0F0F0Fu, hi = (word >> 4) & 0x0F0F0F0Fu;
            w[4 * t + 0] = fmaf(d, byte_as_128_plus<0>(lo), c);
            w[4 * t + 1] = fmaf(d, byte_as_128_plus<1>(lo), c);
            w[4 * t + 2] = fmaf(d, byte_as_128_plus<2>(lo), c);
            w[4 * t + 3] = fmaf(d, byte_as_128_plus<3>(lo), c);
            w[16 + 4 * t + 0] = fmaf(d, byte_as_128_plus<0>(hi), c);
            w[16 + 4 * t + 1] = fmaf(d, byte_as_128_plus<1>(hi), c);
            w[16 + 4 * t + 2] = fmaf(d, byte_as_128_plus<2>(hi), c);
            w[16 + 4 * t + 3] = fmaf(d, byte_as_128_plus<3>(hi), c);
        }
#pragma unroll
        for (int e = 0; e < 16; ++e) o[16 * bb + e] = pack_bf16x2(w[2 * e], w[2 * e + 1]);
    }
}

template <>
__device__ __forceinline__ void dequant64<Q8_0>(const uint8_t *rb, int sub, uint32_t (&o)[32]) {
#pragma unroll
    for (int bb = 0; bb < 2; ++bb) {
        const uint8_t *b = rb + 34 * (2 * sub + bb);
        const float d = f16_bits(*reinterpret_cast<const uint16_t *>(b));
        const float c = -32896.f * d;  // exact: d * (32768 + q + 128) - 32896 d = d q
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const uint32_t u = lds_u32_a2(b + 2 + 4 * t) ^ 0x80808080u;
            // 32768 + byte: byte in mantissa bits 8..15 of 32768.0f (0x47000000)
            const float f0 = __uint_as_float(__byte_perm(u, 0x47000000u, 0x7504u));
            const float f1 = __uint_as_float(__byte_perm(u, 0x47000000u, 0x7514u));
            const float f2 = __uint_as_float(__byte_perm(u, 0x47000000u, 0x7524u));
            const float f3 = __uint_as_float(__byte_perm(u, 0x47000000u, 0x7534u));
            o[16 * bb + 2 * t] = pack_bf16x2(fmaf(d, f0, c), fmaf(d, f1, c));
            o[16 * bb + 2 * t + 1] = pack_bf16x2(fmaf(d, f2, c), fmaf(d, f3, c));
        }
    }
}

__device__ __forceinline__ void q4k_sm(const uint8_t *S, int s, float &sc, float &mn) {
    if (s < 4) {
        sc = (float)(S[s] & 63);
        mn = (float)(S[s + 4] & 63);
    } else {
        sc = (float)((S[s + 4] & 15) | ((S[s - 4] >> 6) << 4));
        mn = (float)((S[s + 4] >> 4) | ((S[s] >> 6) << 4));
    }
}

template <>
__device__ __forceinline__ void dequant64<Q4_K>(const uint8_t *rb, int sub, uint32_t (&o)[32]) {
    const float d = f16_bits(*reinterpret_cast<const uint16_t *>(rb));
    const float dmin = f16_bits(*reinterpret_cast<const uint16_t *>(rb + 2));
    float sc0, mn0, sc1, mn1;
    q4k_sm(rb + 4, 2 * sub, sc0, mn0);
    q4k_sm(rb + 4, 2 * sub + 1, sc1, mn1);
    const float a0 = d * sc0, a1 = d * sc1;
    const float c0 = -(128.f * a0 + dmin * mn0), c1 = -(128.f * a1 + dmin * mn1);
    const uint4 *qs = reinterpret_cast<const uint4 *>(rb + 16 + 32 * sub);
    const uint4 q0 = qs[0], q1 = qs[1];
    const uint32_t words[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        const uint32_t lo = words[t] & 0x0F0F0F0Fu, hi = (words[t] >> 4) & 0x0F0F0F0Fu;
        o[2 * t] = pack_bf16x2(fmaf(a0, byte_as_128_plus<0>(lo), c0), fmaf(a0, byte_as_128_plus<1>(lo), c0));
        o[2 * t + 1] = pack_bf16x2(fmaf(a0, byte_as_128_plus<2>(lo), c0), fmaf(a0, byte_as_128_plus<3>(lo), c0));
        o[16 + 2 * t] = pack_bf16x2(fmaf(a1, byte_as_128_plus<0>(hi), c1), fmaf(a1, byte_as_128_plus<1>(hi), c1));
        o[16 + 2 * t + 1] =
            pack_bf16x2(fmaf(a1, byte_as_128_plus<2>(hi), c1), fmaf(a1, byte_as_128_plus<3>(hi), c1));
    }
}

// Q6_K: rb already points at the super-block (window offset applied).
template <>
__device__ __forceinline__ void dequant64<Q6_K>(const uint8_t *rb, int sub, uint32_t (&o)[32]) {
    const int h = sub >> 1, jp = sub & 1;
    const float d = f16_bits(*reinterpret_cast<const uint16_t *>(rb + 208));
    const int8_t *sc = reinterpret_cast<const int8_t *>(rb + 192);
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
        const int J = 2 * jp + jj;                  // e = 128 h + 32 J + l
        const uint8_t *ql = rb + 64 * h + 32 * jj;   // J % 2 == jj
        const uint8_t *qh = rb + 128 + 32 * h;
        const float ds0 = d * (float)sc[8 * h + 2 * J], ds1 = d * (float)sc[8 * h + 2 * J + 1];
        const float c0 = -160.f * ds0, c1 = -160.f * ds1;  // exact: ds (128 + q) - 160 ds = ds (q - 32)
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const uint32_t lw = lds_u32_a2(ql + 4 * t), hw = lds_u32_a2(qh + 4 * t);
            const uint32_t q = ((lw >> (4 * jp)) & 0x0F0F0F0Fu) | (((hw >> (2 * J)) & 0x03030303u) << 4);
            const float a = t < 4 ? ds0 : ds1, c = t < 4 ? c0 : c1;
            o[16 * jj + 2 * t] = pack_bf16x2(fmaf(a, byte_as_128_plus<0>(q), c), fmaf(a, byte_as_128_plus<1>(q), c));
            o[16 * jj + 2 * t + 1] =
                pack_bf16x2(fmaf(a, byte_as_128_plus<2>(q), c), fmaf(a, byte_as_128_plus<3>(q), c));
        }
    }
}

template <int F, int BN>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap xmap, int M, int K,
                   int N, float *__restrict__ Y, unsigned *status, uint64_t wait_limit) {
    using L = Layout<F, BN>;
    constexpr int SA = L::SA;
    constexpr int RAWB = Raw<F>::bytes;
    extern __shared__ uint8_t smem_dyn[];
    // 1024-byte aligned base derived from the shared array (keeps the
    // accesses below in the shared window)
    uint8_t *smem = smem_dyn + ((1024u - (smem_u32(smem_dyn) & 1023u)) & 1023u);
    uint8_t *sA = smem + L::OFF_A;
    uint8_t *sX = smem + L::OFF_X;
    uint8_t *sRaw = smem + L::OFF_RAW;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::OFF_BAR);
    uint64_t *raw_full = bars, *raw_empty = bars + SR;
    uint64_t *x_full = bars + 2 * SR, *a_full = x_full + SA, *ab_empty = a_full + SA;
    uint64_t *acc_full = ab_empty + SA;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::OFF_MISC);
    unsigned *abort_flag = reinterpret_cast<unsigned *>(smem + L::OFF_MISC + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * BM, n0 = blockIdx.y * BN;
    const int nkc = K / KC;
    const int nsteps = nkc * (KC / BK);
    const Ctl ctl{abort_flag, wait_limit};
    const uint64_t drain_limit = wait_limit < (1ull << 31) ? (1ull << 31) : wait_limit;

    if (threadIdx.x == 0) {
        for (int r = 0; r < SR; ++r) {
            mbar_init(&raw_full[r], 1);
            mbar_init(&raw_empty[r], 4);
        }
        for (int s = 0; s < SA; ++s) {
            mbar_init(&x_full[s], 1);
            mbar_init(&a_full[s], 4);
            mbar_init(&ab_empty[s], 1);
        }
        mbar_init(acc_full, 1);
        *abort_flag = 0u;
        fence_barrier_init();
    }
    if (warp == WARP_WPROD && lane == 0) prefetch_tensormap(&wmap);
    if (warp == WARP_XPROD && lane == 0) prefetch_tensormap(&xmap);
    if (warp == WARP_MMA) {
        tmem_alloc(tmem_slot, L::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_d = *tmem_slot;
    pdl_launch_dependents();

    if (warp == WARP_WPROD) {
        if (lane == 0) {
            int issued = 0;   // raw chunks are issued in order 0, 1, ..., issued-1
            for (int c = 0; c < nkc; ++c) {
                const int r = c % SR;
                if (c >= SR && !wait_ok(ctl, &raw_empty[r], ((c / SR) - 1) & 1, wait_limit)) break;
                if (*abort_flag) break;
                int xb;   // first byte of the chunk's window within the row
                if constexpr (F == Q6_K)
                    xb = (210 * c) & ~15;
                else
                    xb = c * RAWB;
                mbar_arrive_expect_tx(&raw_full[r], (uint32_t)L::RAW_BYTES);
                tma_load_2d(sRaw + r * L::RAW_BYTES, &wmap, &raw_full[r], xb >> 1, m0);
                issued = c + 1;
            }
            if (*abort_flag)   // drain: the last load issued into each stage
                for (int c = issued - SR < 0 ? 0 : issued - SR; c < issued; ++c)
                    drain(&raw_full[c % SR], (c / SR) & 1, drain_limit);
        }
    } else if (warp == WARP_XPROD) {
        if (lane == 0) {
            // Weights stream from the start; X (which may be written by the
            // preceding kernel, e.g. the bf16 conversion) only after it ends.
            pdl_wait();
            int issued = 0;
            for (int t = 0; t < nsteps; ++t) {
                const int s = t % SA;
                if (t >= SA && !wait_ok(ctl, &ab_empty[s], ((t / SA) - 1) & 1, wait_limit)) break;
                if (*abort_flag) break;
                mbar_arrive_expect_tx(&x_full[s], (uint32_t)L::X_BYTES);
                tma_load_2d(sX + s * L::X_BYTES, &xmap, &x_full[s], t * BK, n0);
                issued = t + 1;
            }
            if (*abort_flag)
                for (int t = issued - SA < 0 ? 0 : issued - SA; t < issued; ++t)
                    drain(&x_full[t % SA], (t / SA) & 1, drain_limit);
        }
    } else if (warp == WARP_MMA) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(BM, BN);
            for (int t = 0; t < nsteps; ++t) {
                const int s = t % SA;
                const uint32_t par = (t / SA) & 1;
                if (!wait_ok(ctl, &x_full[s], par, wait_limit)) break;
                if (!wait_ok(ctl, &a_full[s], par, wait_limit)) break;
                tc_fence_after();
                const uint32_t a0 = smem_u32(sA + s * L::A_BYTES), b0 = smem_u32(sX + s * L::X_BYTES);
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk)
                    umma_bf16(tmem_d, sdesc_k_sw128(a0 + 32 * kk), sdesc_k_sw128(b0 + 32 * kk), idesc,
                              (t | kk) != 0);
                umma_commit(&ab_empty[s]);
            }
            umma_commit(acc_full);   // also on abort: lets the epilogue drain the MMAs
        }
    } else {
        // ---------------- dequantizers, then epilogue ----------------
        const int i = threadIdx.x - WARP_DQ0 * 32;   // row of the tile, 0..127
        bool ok = true;
        for (int c = 0; c < nkc && ok; ++c) {
            const int r = c % SR;
            // Every lane waits; the vote keeps the decision warp-uniform.
            if (!__all_sync(0xffffffffu, wait_ok(ctl, &raw_full[r], (c / SR) & 1, wait_limit))) {
                ok = false;
                break;
            }
            const uint8_t *rb = sRaw + r * L::RAW_BYTES + i * RAWB;
            if constexpr (F == Q6_K) rb += (210 * c) & 15;
#pragma unroll 1
            for (int sub = 0; sub < KC / BK; ++sub) {
                const int t = c * (KC / BK) + sub;
                const int s = t % SA;
                if (t >= SA &&
                    !__all_sync(0xffffffffu, wait_ok(ctl, &ab_empty[s], ((t / SA) - 1) & 1, wait_limit))) {
                    ok = false;
                    break;
                }
                uint32_t o[32];
                dequant64<F>(rb, sub, o);
                uint8_t *arow = sA + s * L::A_BYTES + i * 128;
#pragma unroll
                for (int cc = 0; cc < 8; ++cc)
                    *reinterpret_cast<uint4 *>(arow + ((cc ^ (i & 7)) << 4)) =
                        make_uint4(o[4 * cc], o[4 * cc + 1], o[4 * cc + 2], o[4 * cc + 3]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&a_full[s]);
            }
            if (!ok) break;
            __syncwarp();
            if (lane == 0) mbar_arrive(&raw_empty[r]);
        }
        // Epilogue: TMEM lane = tile row.  Warp w may only touch lanes 32*(w%4)..+31.
        const bool acc_ok = mbar_wait(acc_full, 0, 2 * drain_limit);
        pdl_wait();   // Y: order after the preceding kernel
        tc_fence_after();
        if (__all_sync(0xffffffffu, acc_ok && !*abort_flag)) {
            const int q = warp & 3;
            const int row = m0 + 32 * q + lane;
#pragma unroll 1
            for (int j = 0; j < BN / 16; ++j) {
                uint32_t v[16];
                tmem_ld_32x32b_x16(tmem_d + ((uint32_t)(32 * q) << 16) + 16 * j, v);
                tmem_ld_wait();
                if (row < M) {
#pragma unroll
                    for (int cidx = 0; cidx < 16; ++cidx) {
                        const int n = n0 + 16 * j + cidx;
                        if (n < N) Y[(int64_t)n * M + row] = __uint_as_float(v[cidx]);
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == WARP_MMA) {
        tc_fence_after();
        tmem_dealloc(tmem_d, L::TMEM_COLS);
    }
    if (threadIdx.x == 0 && *abort_flag) report_status(status, kStatusTimeout);
}

template <int F, int BN>
cudaError_t launch_one(const GemmArgs &a, const CUtensorMap &wmap, const CUtensorMap &xmap, cudaStream_t st) {
    using L = Layout<F, BN>;
    auto kern = gemm_tc_kernel<F, BN>;
    static std::atomic<uint64_t> configured{0};   // one bit per device ordinal
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(configured.load() & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((a.M + BM - 1) / BM), (unsigned)((a.N + BN - 1) / BN), 1);
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = L::SMEM;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = a.pdl ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, kern, wmap, xmap, (int)a.M, (int)a.K, a.N, a.Y, a.status, a.wait_limit);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int F>
cudaError_t launch_fmt(const GemmArgs &a, const CUtensorMap &wmap, const CUtensorMap &xmap, cudaStream_t st) {
    switch (a.bn) {
    case 64: return launch_one<F, 64>(a, wmap, xmap, st);
    case 128: return launch_one<F, 128>(a, wmap, xmap, st);
    case 256: return launch_one<F, 256>(a, wmap, xmap, st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

int gemm_raw_window_bytes(int fmt) {
    switch (fmt) {
    case Q8_0: return Raw<Q8_0>::bytes;
    case Q4_0: return Raw<Q4_0>::bytes;
    case Q4_K: return Raw<Q4_K>::bytes;
    case Q6_K: return Raw<Q6_K>::bytes;
    default: return 0;
    }
}

cudaError_t launch_gemm_tc(const GemmArgs &a, const CUtensorMap &wmap, const CUtensorMap &xmap, cudaStream_t st) {
    switch (a.fmt) {
    case Q8_0: return launch_fmt<Q8_0>(a, wmap, xmap, st);
    case Q4_0: return launch_fmt<Q4_0>(a, wmap, xmap, st);
    case Q4_K: return launch_fmt<Q4_K>(a, wmap, xmap, st);
    case Q6_K: return launch_fmt<Q6_K>(a, wmap, xmap, st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace qmm
