// gemv_fast.cu -- multi-token GEMV, 1 <= N <= 16, for 16-byte aligned weights:
//
//     Y[n, m] = sum_k X[n, k] * w(m, k)
//
// Each weight block is read from HBM once and reused for every token (the
// point of batching the LM head in "cera 0.5.0 src/model/llama.rs",
// project_logits_batched).  The reduction over k runs on the tensor cores
// with exact operands, which keeps the kernel bound by HBM bytes instead of
// f32 FMA issue at N > 1:
//   * A = the integer codes of the weights (Q4_0: q-8, Q8_0: q as 16*hi+lo,
//     Q4_K: q, Q6_K: q-32), all exact in bf16, built with byte permutes into
//     the mantissa of 128.0 and one exact bf16x2 subtraction;
//   * B = X as bf16 pieces: one piece for bf16 X, hi + lo for f32 X
//     (|x - hi - lo| <= 2^-18 |x|), each piece its own MMA column;
//   * mma.sync m16n8k16 bf16 -> f32; the per-block scale (d, d*sc or
//     d*scale) and the Q4_K min term (dmin*m * sum of x over the sub-block)
//     are applied to the f32 fragments, so every product is exact and only
//     f32 accumulation rounds (well inside 1e-5 * sum|w x|).
// The k order inside each 16-wide MMA step is permuted so that thread t of a
// quad owns elements 4t..4t+3: one 32-bit word of packed codes per row.
//
// CTA = 4 compute warps (16 rows each, 64 rows) + 1 TMA producer warp.  Raw
// weight bytes arrive by 2-D TMA (64 rows x one 256-weight chunk) into a
// ring of stages; per chunk the compute warps build the B fragments of X and
// a table of per-row scales in shared memory, then run the MMAs.  For small
// M the K range is split over a thread-block cluster and the partial sums
// are reduced through distributed shared memory by cluster rank 0, in a fixed
// order (deterministic, no atomics, Y is written exactly once).
#include <atomic>

#include "common.cuh"
#include "kernels.h"

namespace qmm {
namespace {

constexpr int ROWS = 64;
constexpr int CW = 4;                  // compute warps
constexpr int THREADS = (CW + 1) * 32; // + producer warp
constexpr int KC = 256;                // weights per chunk
constexpr int SCW = 20;                // scale-table row stride (floats): conflict-free LDS.128

template <int F> struct GWin;
template <> struct GWin<Q8_0> { static constexpr int bytes = 272; static constexpr int stages = 4; };
template <> struct GWin<Q4_0> { static constexpr int bytes = 144; static constexpr int stages = 6; };
template <> struct GWin<Q4_K> { static constexpr int bytes = 144; static constexpr int stages = 6; };
template <> struct GWin<Q6_K> { static constexpr int bytes = 240; static constexpr int stages = 4; };

template <int F, int NT> struct GL {
    static constexpr int S = GWin<F>::stages;
    static constexpr int WIN = GWin<F>::bytes;
    static constexpr int RAW = ROWS * WIN;                    // multiple of 1024
    static constexpr int XS = 16 * NT * 32 * 8;                // B fragments of one chunk
    static constexpr int SCT = ROWS * SCW * 4;                 // scale table of one chunk
    static constexpr int SXB = 8 * 16 * 4;                     // Q4_K sub-block sums of x
    static constexpr int OFF_RAW = 0;
    static constexpr int OFF_XS = OFF_RAW + S * RAW;
    static constexpr int OFF_SC = OFF_XS + 2 * XS;
    static constexpr int OFF_SX = OFF_SC + 2 * SCT;
    static constexpr int OFF_RED = OFF_SX + 2 * SXB;
    static constexpr int OFF_BAR = OFF_RED + ROWS * 16 * 4;
    static constexpr int OFF_MISC = OFF_BAR + 2 * S * 8;
    static constexpr int TOTAL = OFF_MISC + 16;
    static constexpr int SMEM = TOTAL + 1024;
};

// ---------------------------------------------------------------------------
// small device helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t bsub2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
// bf16x2 (M + b0, M + b1) from bytes 0,1 (SEL01) or 2,3 (SEL23) of `v`,
// where M is the bf16 whose high byte is `hi` (0x43: 128, 0x45: 2048).
template <uint32_t HI>
__device__ __forceinline__ uint32_t pair01(uint32_t v) { return __byte_perm(v, HI, 0x4140u); }
template <uint32_t HI>
__device__ __forceinline__ uint32_t pair23(uint32_t v) { return __byte_perm(v, HI, 0x4342u); }

constexpr uint32_t BF2(uint32_t h) { return h | (h << 16); }   // bf16 pair from one bf16 bit pattern
constexpr uint32_t C128 = BF2(0x4300u), C136 = BF2(0x4308u), C160 = BF2(0x4320u), C2176 = BF2(0x4508u);

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint2 b) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b.x), "r"(b.y));
}

// A fragment from two words of byte codes (row g, row g+8): elements 4t..4t+3.
template <uint32_t HI, uint32_t OFFS>
__device__ __forceinline__ void afrag(uint32_t (&a)[4], uint32_t vg, uint32_t vg8) {
    a[0] = bsub2(pair01<HI>(vg), OFFS);
    a[1] = bsub2(pair01<HI>(vg8), OFFS);
    a[2] = bsub2(pair23<HI>(vg), OFFS);
    a[3] = bsub2(pair23<HI>(vg8), OFFS);
}

__device__ __forceinline__ uint16_t lds_u16(const uint8_t *p) { return *reinterpret_cast<const uint16_t *>(p); }

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ float ld_dsmem_f32(const float *local, uint32_t rank) {
    uint32_t la = smem_u32(local), ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(la), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra) : "memory");
    return v;
}
__device__ __forceinline__ void named_sync_compute() {
    asm volatile("bar.sync 1, %0;" ::"n"(CW * 32) : "memory");
}

// Bounded wait that gives up early once the CTA has aborted.
__device__ __forceinline__ bool gwait(volatile unsigned *abort_flag, uint64_t *bar, uint32_t parity, uint64_t limit) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if ((uint64_t)(clock64() - t0) > limit) {
            *abort_flag = 1u;
            return false;
        }
    }
}

// ---------------------------------------------------------------------------
// Per-chunk preparation (all 128 compute threads):
//  * B fragments of X for the chunk: xs[ks][j][lane] = {b0, b1}; column
//    8j+g of the MMA is (token (8j+g)/P, piece (8j+g)%P); element 4t+i of
//    k-step ks is x[n][k0 + 16 ks + 4t + i];
//  * the per-row scale table sc[row][0..15] of the chunk (format specific);
//  * Q4_K only: sx[s][n] = sum of x[n] over sub-block s.
// ---------------------------------------------------------------------------
template <int NT, int P, bool XBF16>
__device__ __forceinline__ void build_xs(uint2 *xs, const void *Xv, int K, int N, int64_t k0, int ct) {
    // one item = (ks, token n, t): 4 consecutive x values -> P fragment halves
    const int items = 16 * N * 4;
    for (int it = ct; it < items; it += CW * 32) {
        const int t = it & 3, n = (it >> 2) % N, ks = (it >> 2) / N;
        const int64_t k = k0 + 16 * ks + 4 * t;
        uint32_t hi01, hi23, lo01 = 0, lo23 = 0;
        if constexpr (XBF16) {
            const uint2 v = *reinterpret_cast<const uint2 *>(reinterpret_cast<const uint16_t *>(Xv) + (int64_t)n * K + k);
            hi01 = v.x;
            hi23 = v.y;
        } else {
            const float4 v = *reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(Xv) + (int64_t)n * K + k);
            hi01 = pack_bf16x2(v.x, v.y);
            hi23 = pack_bf16x2(v.z, v.w);
            if constexpr (P == 2) {
                const float r0 = v.x - __uint_as_float(hi01 << 16), r1 = v.y - __uint_as_float(hi01 & 0xFFFF0000u);
                const float r2 = v.z - __uint_as_float(hi23 << 16), r3 = v.w - __uint_as_float(hi23 & 0xFFFF0000u);
                lo01 = pack_bf16x2(r0, r1);
                lo23 = pack_bf16x2(r2, r3);
            }
        }
#pragma unroll
        for (int p = 0; p < P; ++p) {
            const int col = P * n + p;            // MMA column
            const int j = col >> 3, g = col & 7;
            const int lane = 4 * g + t;
            xs[(ks * NT + j) * 32 + lane] = p == 0 ? make_uint2(hi01, hi23) : make_uint2(lo01, lo23);
        }
    }
}

template <int F, int NT, int P, bool XBF16>
__device__ __forceinline__ void prep_chunk(uint2 *xs, float *sct, float *sx, const uint8_t *raw, int woff,
                                           const void *Xv, int K, int N, int64_t k0, int ct) {
    build_xs<NT, P, XBF16>(xs, Xv, K, N, k0, ct);
    constexpr int WIN = GWin<F>::bytes;
    // scale table: 64 rows x 16 entries, 8 per thread
    {
        const int row = ct >> 1, half = ct & 1;
        const uint8_t *rb = raw + row * WIN + woff;
        float *o = sct + row * SCW;
        if constexpr (F == Q4_0 || F == Q8_0) {
            constexpr int BB = F == Q4_0 ? 18 : 34;
            if (half == 0) {
#pragma unroll
                for (int b = 0; b < 8; ++b) o[b] = f16_bits(lds_u16(rb + BB * b));
            }
        } else if constexpr (F == Q4_K) {
            const float d = f16_bits(lds_u16(rb)), dmin = f16_bits(lds_u16(rb + 2));
            const uint32_t w0 = *reinterpret_cast<const uint32_t *>(rb + 4);
            const uint32_t w1 = *reinterpret_cast<const uint32_t *>(rb + 8);
            const uint32_t w2 = *reinterpret_cast<const uint32_t *>(rb + 12);
            // bytes: sc[0..3], mn[0..3], sc[4..7], mn[4..7]
            const uint32_t sc03 = w0 & 0x3F3F3F3Fu, mn03 = w1 & 0x3F3F3F3Fu;
            const uint32_t sc47 = (w2 & 0x0F0F0F0Fu) | (((w0 >> 6) & 0x03030303u) << 4);
            const uint32_t mn47 = ((w2 >> 4) & 0x0F0F0F0Fu) | (((w1 >> 6) & 0x03030303u) << 4);
            const uint32_t sc = half ? sc47 : sc03, mn = half ? mn47 : mn03;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                o[4 * half + i] = d * (float)((sc >> (8 * i)) & 0xFFu);          // d * sc_s
                o[8 + 4 * half + i] = dmin * (float)((mn >> (8 * i)) & 0xFFu);   // dmin * m_s
            }
        } else {  // Q6_K: d * scales[G], G = 0..15
            const float d = f16_bits(lds_u16(rb + 208));
            const int8_t *s = reinterpret_cast<const int8_t *>(rb + 192);
#pragma unroll
            for (int i = 0; i < 8; ++i) o[8 * half + i] = d * (float)s[8 * half + i];
        }
    }
    if constexpr (F == Q4_K) {
        // sx[s][n] = sum_{e<32} x[n][k0 + 32 s + e]
        for (int it = ct; it < 8 * N; it += CW * 32) {
            const int s = it & 7, n = it >> 3;
            float acc = 0.f;
            if constexpr (XBF16) {
                const uint16_t *x = reinterpret_cast<const uint16_t *>(Xv) + (int64_t)n * K + k0 + 32 * s;
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    const uint32_t v = *reinterpret_cast<const uint32_t *>(x + e);
                    acc += __uint_as_float(v << 16) + __uint_as_float(v & 0xFFFF0000u);
                }
            } else {
                const float4 *x = reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(Xv) +
                                                                   (int64_t)n * K + k0 + 32 * s);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float4 v = x[e];
                    acc += (v.x + v.y) + (v.z + v.w);
                }
            }
            sx[s * 16 + n] = acc;
        }
    }
}

// Accumulate one scaled MMA result.  P == 2: columns 2t, 2t+1 are the two
// pieces of token 4j+t (summed); P == 1: two tokens 8j+2t, 8j+2t+1.
template <int P>
__device__ __forceinline__ void acc_scaled(float *acc, const float (&d)[4], float sg, float sg8) {
    if constexpr (P == 2) {
        acc[0] = fmaf(sg, d[0] + d[1], acc[0]);
        acc[1] = fmaf(sg8, d[2] + d[3], acc[1]);
    } else {
        acc[0] = fmaf(sg, d[0], acc[0]);
        acc[1] = fmaf(sg, d[1], acc[1]);
        acc[2] = fmaf(sg8, d[2], acc[2]);
        acc[3] = fmaf(sg8, d[3], acc[3]);
    }
}

// ---------------------------------------------------------------------------
// Chunk compute for one warp: 16 rows (g, g+8 per thread) x 256 weights.
// ---------------------------------------------------------------------------
template <int F, int NT, int P>
__device__ __forceinline__ void compute_chunk(float (&acc)[NT][4], const uint8_t *rg, const uint8_t *rg8,
                                              const uint2 *xs, const float *scg, const float *scg8, const float *sx,
                                              int lane, int t) {
    if constexpr (F == Q4_0) {
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            const uint32_t wg = lds_u32_a2(rg + 18 * b + 2 + 4 * t), wg8 = lds_u32_a2(rg8 + 18 * b + 2 + 4 * t);
            uint32_t a0[4], a1[4];
            afrag<0x43u, C136>(a0, wg & 0x0F0F0F0Fu, wg8 & 0x0F0F0F0Fu);
            afrag<0x43u, C136>(a1, (wg >> 4) & 0x0F0F0F0Fu, (wg8 >> 4) & 0x0F0F0F0Fu);
            const float sg = scg[b], sg8 = scg8[b];
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                float d[4] = {0.f, 0.f, 0.f, 0.f};
                mma16816(d, a0, xs[((2 * b) * NT + j) * 32 + lane]);
                mma16816(d, a1, xs[((2 * b + 1) * NT + j) * 32 + lane]);
                acc_scaled<P>(acc[j], d, sg, sg8);
            }
        }
    } else if constexpr (F == Q8_0) {
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            const float sg = scg[b], sg8 = scg8[b];
            uint32_t al[2][4], ah[2][4];
#pragma unroll
            for (int grp = 0; grp < 2; ++grp) {
                const uint32_t ug = lds_u32_a2(rg + 34 * b + 2 + 16 * grp + 4 * t) ^ 0x80808080u;
                const uint32_t ug8 = lds_u32_a2(rg8 + 34 * b + 2 + 16 * grp + 4 * t) ^ 0x80808080u;
                // q = 16 * (hi - 8) + lo with hi, lo the nibbles of q + 128
                afrag<0x43u, C128>(al[grp], ug & 0x0F0F0F0Fu, ug8 & 0x0F0F0F0Fu);
                afrag<0x45u, C2176>(ah[grp], (ug >> 4) & 0x0F0F0F0Fu, (ug8 >> 4) & 0x0F0F0F0Fu);
            }
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                float d[4] = {0.f, 0.f, 0.f, 0.f};
                const uint2 b0 = xs[((2 * b) * NT + j) * 32 + lane], b1 = xs[((2 * b + 1) * NT + j) * 32 + lane];
                mma16816(d, al[0], b0);
                mma16816(d, ah[0], b0);
                mma16816(d, al[1], b1);
                mma16816(d, ah[1], b1);
                acc_scaled<P>(acc[j], d, sg, sg8);
            }
        }
    } else if constexpr (F == Q4_K) {
        const uint8_t *qg = rg + 16, *qg8 = rg8 + 16;
#pragma unroll
        for (int pr = 0; pr < 4; ++pr) {            // sub-blocks 2pr (low nibbles), 2pr+1 (high)
            const uint32_t w0g = *reinterpret_cast<const uint32_t *>(qg + 32 * pr + 4 * t);
            const uint32_t w1g = *reinterpret_cast<const uint32_t *>(qg + 32 * pr + 16 + 4 * t);
            const uint32_t w0g8 = *reinterpret_cast<const uint32_t *>(qg8 + 32 * pr + 4 * t);
            const uint32_t w1g8 = *reinterpret_cast<const uint32_t *>(qg8 + 32 * pr + 16 + 4 * t);
#pragma unroll
            for (int hn = 0; hn < 2; ++hn) {
                const int s = 2 * pr + hn, sh = 4 * hn;
                uint32_t a0[4], a1[4];
                afrag<0x43u, C128>(a0, (w0g >> sh) & 0x0F0F0F0Fu, (w0g8 >> sh) & 0x0F0F0F0Fu);
                afrag<0x43u, C128>(a1, (w1g >> sh) & 0x0F0F0F0Fu, (w1g8 >> sh) & 0x0F0F0F0Fu);
                const float dsg = scg[s], dsg8 = scg8[s], dmg = scg[8 + s], dmg8 = scg8[8 + s];
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    float d[4] = {0.f, 0.f, 0.f, 0.f};
                    mma16816(d, a0, xs[((2 * s) * NT + j) * 32 + lane]);
                    mma16816(d, a1, xs[((2 * s + 1) * NT + j) * 32 + lane]);
                    // w = d*sc*q - dmin*m  =>  sum w x = (d sc) sum q x - (dmin m) sum x
                    if constexpr (P == 2) {
                        const float sxn = sx[s * 16 + 4 * j + t];
                        acc[j][0] = fmaf(dsg, d[0] + d[1], fmaf(-dmg, sxn, acc[j][0]));
                        acc[j][1] = fmaf(dsg8, d[2] + d[3], fmaf(-dmg8, sxn, acc[j][1]));
                    } else {
                        const float sx0 = sx[s * 16 + 8 * j + 2 * t], sx1 = sx[s * 16 + 8 * j + 2 * t + 1];
                        acc[j][0] = fmaf(dsg, d[0], fmaf(-dmg, sx0, acc[j][0]));
                        acc[j][1] = fmaf(dsg, d[1], fmaf(-dmg, sx1, acc[j][1]));
                        acc[j][2] = fmaf(dsg8, d[2], fmaf(-dmg8, sx0, acc[j][2]));
                        acc[j][3] = fmaf(dsg8, d[3], fmaf(-dmg8, sx1, acc[j][3]));
                    }
                }
            }
        }
    } else {  // Q6_K: element e = 128h + 32J + l, l = 16 lh + 4t + i, k-step G = 8h + 2J + lh
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int lh = 0; lh < 2; ++lh) {
                const int lo = 16 * lh + 4 * t;
                const uint32_t hg = lds_u32_a2(rg + 128 + 32 * h + lo), hg8 = lds_u32_a2(rg8 + 128 + 32 * h + lo);
                const uint32_t l0g = lds_u32_a2(rg + 64 * h + lo), l0g8 = lds_u32_a2(rg8 + 64 * h + lo);
                const uint32_t l1g = lds_u32_a2(rg + 64 * h + 32 + lo), l1g8 = lds_u32_a2(rg8 + 64 * h + 32 + lo);
#pragma unroll
                for (int J = 0; J < 4; ++J) {
                    const int G = 8 * h + 2 * J + lh;
                    const uint32_t lwg = (J & 1) ? l1g : l0g, lwg8 = (J & 1) ? l1g8 : l0g8;
                    const int ns = 4 * (J >> 1);
                    const uint32_t qg = ((lwg >> ns) & 0x0F0F0F0Fu) | (((hg >> (2 * J)) & 0x03030303u) << 4);
                    const uint32_t qg8 = ((lwg8 >> ns) & 0x0F0F0F0Fu) | (((hg8 >> (2 * J)) & 0x03030303u) << 4);
                    uint32_t a[4];
                    afrag<0x43u, C160>(a, qg, qg8);
                    const float sg = scg[G], sg8 = scg8[G];
#pragma unroll
                    for (int j = 0; j < NT; ++j) {
                        float d[4] = {0.f, 0.f, 0.f, 0.f};
                        mma16816(d, a, xs[(G * NT + j) * 32 + lane]);
                        acc_scaled<P>(acc[j], d, sg, sg8);
                    }
                }
            }
        }
    }
}

template <int F, int NT, int P, bool XBF16>
__global__ void __launch_bounds__(THREADS) gemv_mma_kernel(const __grid_constant__ CUtensorMap wmap,
                                                           const void *__restrict__ X, int M, int K, int N,
                                                           float *__restrict__ Y, int cps, unsigned *status,
                                                           uint64_t wait_limit) {
    using L = GL<F, NT>;
    constexpr int S = L::S;
    extern __shared__ uint8_t smem_dyn[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~(uintptr_t)1023);
    uint8_t *sraw = smem + L::OFF_RAW;
    uint2 *sxs = reinterpret_cast<uint2 *>(smem + L::OFF_XS);
    float *ssc = reinterpret_cast<float *>(smem + L::OFF_SC);
    float *ssx = reinterpret_cast<float *>(smem + L::OFF_SX);
    float *sred = reinterpret_cast<float *>(smem + L::OFF_RED);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::OFF_BAR);
    uint64_t *empty = full + S;
    volatile unsigned *abort_flag = reinterpret_cast<volatile unsigned *>(smem + L::OFF_MISC);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * ROWS;
    const int nchunks = K / KC;
    const int c_begin = blockIdx.y * cps;
    const int c_end = min(nchunks, c_begin + cps);
    const int nloc = c_end > c_begin ? c_end - c_begin : 0;
    const int KS = gridDim.y;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], CW);
        }
        *abort_flag = 0u;
        fence_barrier_init();
    }
    __syncthreads();

    float acc[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;

    if (warp == CW) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            prefetch_tensormap(&wmap);
            int last[S];
            for (int s = 0; s < S; ++s) last[s] = -1;
            for (int c = 0; c < nloc; ++c) {
                const int s = c % S;
                if (c >= S && !gwait(abort_flag, &empty[s], ((c / S) - 1) & 1, wait_limit)) break;
                if (*abort_flag) break;
                const int cg = c_begin + c;
                const int xb = F == Q6_K ? ((210 * cg) & ~15) : cg * L::WIN;
                mbar_arrive_expect_tx(&full[s], (uint32_t)L::RAW);
                tma_load_2d(sraw + s * L::RAW, &wmap, &full[s], xb >> 1, m0);
                last[s] = c;
            }
            if (*abort_flag)
                for (int s = 0; s < S; ++s)
                    if (last[s] >= 0) (void)mbar_wait(&full[s], (last[s] / S) & 1, wait_limit < (1ull << 31) ? (1ull << 31) : wait_limit);
        }
    } else {
        // ---------------- compute warps ----------------
        const int ct = threadIdx.x;           // 0..127
        const int g = lane >> 2, t = lane & 3;
        const int rg = 16 * warp + g;         // tile rows of this thread: rg, rg + 8
        for (int c = 0; c < nloc; ++c) {
            const int s = c % S, buf = c & 1;
            const int cg = c_begin + c;
            const int woff = F == Q6_K ? ((210 * cg) & 15) : 0;
            // warp-uniform decision: mma.sync below must run on all 32 lanes
            const bool ok = __all_sync(0xffffffffu, gwait(abort_flag, &full[s], (c / S) & 1, wait_limit) &&
                                                        !*abort_flag);
            uint2 *xs = sxs + buf * (L::XS / 8);
            float *sct = ssc + buf * (L::SCT / 4);
            float *sx = ssx + buf * (L::SXB / 4);
            const uint8_t *raw = sraw + s * L::RAW;
            if (ok)
                prep_chunk<F, NT, P, XBF16>(xs, sct, sx, raw, woff, X, K, N, (int64_t)cg * KC, ct);
            named_sync_compute();
            if (ok) {
                const uint8_t *pg = raw + rg * L::WIN + woff;
                compute_chunk<F, NT, P>(acc, pg, pg + 8 * L::WIN, xs, sct + rg * SCW, sct + (rg + 8) * SCW, sx, lane,
                                        t);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
    }

    // ---------------- reduction over the K split and store ----------------
    const bool aborted = *abort_flag != 0u;
    if (KS == 1) {
        if (warp < CW && !aborted) {
            const int g = lane >> 2, t = lane & 3;
            const int r0 = m0 + 16 * warp + g, r1 = r0 + 8;
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                if constexpr (P == 2) {
                    const int n = 4 * j + t;
                    if (n < N) {
                        if (r0 < M) Y[(int64_t)n * M + r0] = acc[j][0];
                        if (r1 < M) Y[(int64_t)n * M + r1] = acc[j][1];
                    }
                } else {
                    const int n0 = 8 * j + 2 * t;
                    if (n0 < N) {
                        if (r0 < M) Y[(int64_t)n0 * M + r0] = acc[j][0];
                        if (r1 < M) Y[(int64_t)n0 * M + r1] = acc[j][2];
                    }
                    if (n0 + 1 < N) {
                        if (r0 < M) Y[(int64_t)(n0 + 1) * M + r0] = acc[j][1];
                        if (r1 < M) Y[(int64_t)(n0 + 1) * M + r1] = acc[j][3];
                    }
                }
            }
        }
    } else {
        // partials -> shared memory [row][token]; rank 0 of the cluster sums
        if (warp < CW) {
            const int g = lane >> 2, t = lane & 3;
            const int r0 = 16 * warp + g, r1 = r0 + 8;
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                if constexpr (P == 2) {
                    const int n = 4 * j + t;
                    if (n < 16) {
                        sred[r0 * 16 + n] = acc[j][0];
                        sred[r1 * 16 + n] = acc[j][1];
                    }
                } else {
                    const int n0 = 8 * j + 2 * t;
                    if (n0 + 1 < 16) {
                        sred[r0 * 16 + n0] = acc[j][0];
                        sred[r0 * 16 + n0 + 1] = acc[j][1];
                        sred[r1 * 16 + n0] = acc[j][2];
                        sred[r1 * 16 + n0 + 1] = acc[j][3];
                    }
                }
            }
        }
        cluster_sync_all();
        if (cluster_ctarank() == 0 && warp < CW) {
            // rank r's CTA holds K-slice r; every CTA of the cluster ran the
            // same number of barriers, so an abort anywhere shows here only
            // through the status word.
            for (int idx = threadIdx.x; idx < ROWS * N; idx += CW * 32) {
                const int row = idx / N, n = idx % N;
                float v = 0.f;
                for (int r = 0; r < KS; ++r) v += ld_dsmem_f32(sred + row * 16 + n, (uint32_t)r);
                if (m0 + row < M && !aborted) Y[(int64_t)n * M + m0 + row] = v;
            }
        }
        cluster_sync_all();
    }
    if (threadIdx.x == 0 && aborted) report_status(status, kStatusTimeout);
}

template <int F, int NT, int P, bool XBF16>
cudaError_t launch_t(const CUtensorMap &wmap, const void *X, int64_t M, int64_t K, int N, float *Y, int num_sms,
                     unsigned *status, uint64_t limit, cudaStream_t st) {
    using L = GL<F, NT>;
    auto kern = gemv_mma_kernel<F, NT, P, XBF16>;
    static std::atomic<uint64_t> configured{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (!(configured.load() & (1ull << (dev & 63)))) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
        if (e != cudaSuccess) return e;
        configured.fetch_or(1ull << (dev & 63));
    }
    const int tiles = (int)((M + ROWS - 1) / ROWS);
    const int nchunks = (int)(K / KC);
    int ks = 1;
    while (ks < 8 && (int64_t)tiles * ks * 2 < (int64_t)num_sms * 3 && ks * 2 <= nchunks) ks *= 2;
    const int cps = (nchunks + ks - 1) / ks;
    ks = (nchunks + cps - 1) / cps;   // no empty slices
    // cluster dims must divide the grid: round ks up to a power of two
    int ksp = 1;
    while (ksp < ks) ksp *= 2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)tiles, (unsigned)ksp, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = L::SMEM;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = (unsigned)ksp;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = ksp > 1 ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, kern, wmap, X, (int)M, (int)K, N, Y, cps, status, limit);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int F, bool XBF16>
cudaError_t launch_f(const CUtensorMap &wmap, const void *X, int64_t M, int64_t K, int N, float *Y, int num_sms,
                     unsigned *status, uint64_t limit, cudaStream_t st) {
    constexpr int P = XBF16 ? 1 : 2;
    const int cols = P * N;
    const int nt = (cols + 7) / 8;
    if constexpr (XBF16) {
        if (nt <= 1) return launch_t<F, 1, 1, true>(wmap, X, M, K, N, Y, num_sms, status, limit, st);
        return launch_t<F, 2, 1, true>(wmap, X, M, K, N, Y, num_sms, status, limit, st);
    } else {
        switch (nt) {
        case 1: return launch_t<F, 1, 2, false>(wmap, X, M, K, N, Y, num_sms, status, limit, st);
        case 2: return launch_t<F, 2, 2, false>(wmap, X, M, K, N, Y, num_sms, status, limit, st);
        case 3: return launch_t<F, 3, 2, false>(wmap, X, M, K, N, Y, num_sms, status, limit, st);
        default: return launch_t<F, 4, 2, false>(wmap, X, M, K, N, Y, num_sms, status, limit, st);
        }
    }
}

}  // namespace

int gemv_window_bytes(int fmt) {
    switch (fmt) {
    case Q8_0: return GWin<Q8_0>::bytes;
    case Q4_0: return GWin<Q4_0>::bytes;
    case Q4_K: return GWin<Q4_K>::bytes;
    case Q6_K: return GWin<Q6_K>::bytes;
    default: return 0;
    }
}

cudaError_t launch_gemv_mma(int fmt, const CUtensorMap &wmap, const void *X, int xbf16, int64_t M, int64_t K, int N,
                            float *Y, int num_sms, unsigned *status, uint64_t limit, cudaStream_t st) {
    if (N < 1 || N > 16) return cudaErrorInvalidValue;
    switch (fmt) {
    case Q8_0: return xbf16 ? launch_f<Q8_0, true>(wmap, X, M, K, N, Y, num_sms, status, limit, st)
                            : launch_f<Q8_0, false>(wmap, X, M, K, N, Y, num_sms, status, limit, st);
    case Q4_0: return xbf16 ? launch_f<Q4_0, true>(wmap, X, M, K, N, Y, num_sms, status, limit, st)
                            : launch_f<Q4_0, false>(wmap, X, M, K, N, Y, num_sms, status, limit, st);
    case Q4_K: return xbf16 ? launch_f<Q4_K, true>(wmap, X, M, K, N, Y, num_sms, status, limit, st)
                            : launch_f<Q4_K, false>(wmap, X, M, K, N, Y, num_sms, status, limit, st);
    case Q6_K: return xbf16 ? launch_f<Q6_K, true>(wmap, X, M, K, N, Y, num_sms, status, limit, st)
                            : launch_f<Q6_K, false>(wmap, X, M, K, N, Y, num_sms, status, limit, st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace qmm
