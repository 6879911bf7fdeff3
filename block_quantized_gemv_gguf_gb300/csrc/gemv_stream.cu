// gemv_stream.cu -- decode GEMV for one token (N = 1), 16-byte aligned rows:
//
//     y[m] = sum_k w(m, k) * x[k]
//
// the per-token projection of "cera 0.5.0 src/model/llama.rs" (decode) and
// the row loops of "cera 0.5.2 src/backend/cpu.rs" (matmul_*_f32 /
// gemv_dispatch), restated for one GB300 SM per CTA:
//
//   * Work unit = 256 consecutive weights of one row (8 Q4_0 / Q8_0 blocks,
//     or one Q4_K / Q5_K / Q6_K super-block): 144, 272, 176 or 210 bytes.
//     A CTA owns whole rows; its rows are one contiguous byte range of W.
//   * Each warp streams its own "stages" of 32 consecutive units of that
//     range (one 1-D bulk copy per stage, completion on a warp-private
//     mbarrier, a ring of S slots).  Lane l of the warp owns unit l of the
//     stage.  No data passes between warps until the very end.
//   * The weight copies are issued before the kernel waits on the preceding
//     grid (the weights are static; X and Y are ordered behind it).
//   * X (f32; bf16 widened) sits in shared memory once per CTA, in 16-byte
//     chunks XOR-swizzled by unit index so that the 32 lanes of a warp, each
//     on its own unit, read it without bank conflicts.
//   * Arithmetic: every integer code becomes an exact f32 by a byte permute
//     into the mantissa of 2^23 and one packed subtraction (which also
//     removes the format's offset), then a packed f32 FMA with x.  Each
//     block's (or sub-block's) scale multiplies the f32 block sum; the
//     Q4_K / Q5_K min term uses the sub-block sums of x.
//   * Row results: a segmented warp-shuffle reduction by row over each
//     stage (a row held entirely in one stage is stored directly); rows that
//     cross stages are summed from per-stage partials in stage order at the
//     end.  Every sum has a fixed order: the result is deterministic.
//
// All waits are bounded; a warp that gives up raises the CTA's abort flag,
// waits (bounded) for its own copies in flight, and the CTA reports
// QMM_ERR_TIMEOUT in the status word.
#include <atomic>

#include "amax.cuh"
#include "common.cuh"
#include "kernels.h"

namespace qmm {
namespace {

template <int F> struct UnitBytes;
template <> struct UnitBytes<Q8_0> { static constexpr int B = 272; };   // 8 blocks of 34
template <> struct UnitBytes<Q4_0> { static constexpr int B = 144; };   // 8 blocks of 18
template <> struct UnitBytes<Q4_K> { static constexpr int B = 144; };
template <> struct UnitBytes<Q5_K> { static constexpr int B = 176; };
template <> struct UnitBytes<Q6_K> { static constexpr int B = 210; };

constexpr int kLanes = 32;
// A stage slot: 32 units, padded (the Q6_K reader fetches up to 4 bytes past
// its unit) and rounded to 128 bytes.
__host__ __device__ constexpr int slot_bytes(int ub) { return (kLanes * ub + 16 + 127) / 128 * 128; }

// ---------------------------------------------------------------------------
// Exact integer codes as f32: a byte permute puts a code byte into the
// mantissa of 2^23 (the f32 reads 2^23 + byte), one packed subtraction
// removes 2^23 and the format's offset exactly.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float mag(uint32_t w, uint32_t k) {
    return __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7540u | k));
}
__device__ __forceinline__ float2 f2(float a, float b) { return make_float2(a, b); }
__device__ __forceinline__ float2 mag01(uint32_t w) { return f2(mag(w, 0), mag(w, 1)); }
__device__ __forceinline__ float2 mag23(uint32_t w) { return f2(mag(w, 2), mag(w, 3)); }

// acc += (codes of bytes 0..3 of v + off) * x[0..3]
__device__ __forceinline__ float2 dot4(float2 acc, uint32_t v, float2 off, float4 x) {
    acc = __ffma2_rn(__fadd2_rn(mag01(v), off), f2(x.x, x.y), acc);
    return __ffma2_rn(__fadd2_rn(mag23(v), off), f2(x.z, x.w), acc);
}

// Offset-free codes (Q4_K, Q5_K: q in 0..31) as exact f32 subnormals: a byte
// permute puts the code alone into the low byte, so the f32 reads
// q * 2^-149 with no constant to remove.  X is stored scaled per 32-element
// block by 2^k (k from the block's largest |x|, below), so the products
// q * x * 2^(k - 149) are normal numbers; the block sum is scaled back by
// 2^64 * 2^(85 - k) (two exact power-of-two multiplies).
__device__ __forceinline__ float sub_code(uint32_t w, uint32_t k) {
    return __uint_as_float(__byte_perm(w, 0u, 0x4440u | k));
}
// acc += codes of bytes 0..3 of v (as subnormals) * x[0..3]
__device__ __forceinline__ float2 dot4s(float2 acc, uint32_t v, float4 x) {
    acc = __ffma2_rn(f2(sub_code(v, 0), sub_code(v, 1)), f2(x.x, x.y), acc);
    return __ffma2_rn(f2(sub_code(v, 2), sub_code(v, 3)), f2(x.z, x.w), acc);
}
__device__ __forceinline__ float unscale(float v, float fb) { return (v * 0x1p64f) * fb; }

// The unit's 64 chunks of x, XOR-swizzled: logical chunk 8k + t sits at
// p[t][8k] (the XOR only touches t, so k is an immediate offset).
struct XRow {
    const float4 *p[8];
    __device__ __forceinline__ XRow(const float4 *x0, int sw) {
#pragma unroll
        for (int t = 0; t < 8; ++t) p[t] = x0 + (t ^ sw);
    }
    __device__ __forceinline__ float4 operator()(int q) const { return p[q & 7][q & ~7]; }
};

// 32-bit word at byte offset `o` (even, compile-time after unrolling) of a
// register copy of 16-byte aligned bytes.
template <int NW>
__device__ __forceinline__ uint32_t word_at(const uint32_t (&r)[NW], int o) {
    return (o & 2) ? __byte_perm(r[o >> 2], r[(o >> 2) + 1], 0x5432u) : r[o >> 2];
}
template <int NW>
__device__ __forceinline__ uint32_t half_at(const uint32_t (&r)[NW], int o) {
    return (o & 2) ? (r[o >> 2] >> 16) : (r[o >> 2] & 0xFFFFu);
}

template <int NW>
__device__ __forceinline__ void lds_words(uint32_t (&r)[NW], const uint8_t *p) {
    const uint4 *q = reinterpret_cast<const uint4 *>(p);
#pragma unroll
    for (int i = 0; i < NW / 4; ++i) {
        const uint4 v = q[i];
        r[4 * i] = v.x;
        r[4 * i + 1] = v.y;
        r[4 * i + 2] = v.z;
        r[4 * i + 3] = v.w;
    }
}

// ---------------------------------------------------------------------------
// One unit: sum over its 256 weights of w * x.  ub: the unit's bytes in
// shared memory; x: the unit's 64 x chunks; xs8: the 8 sub-block sums of x
// of the unit (Q4_K / Q5_K).
// ---------------------------------------------------------------------------
template <int F>
__device__ __forceinline__ float unit_dot(const uint8_t *ub, const XRow &x, const float *xs8, const float *fb8);

// Q4_0: 8 blocks; block b at byte 18b: f16 d, 16 bytes qs; element e < 16
// is the low nibble of qs[e], e >= 16 the high nibble of qs[e - 16];
// w = (nibble - 8) * d.
template <>
__device__ __forceinline__ float unit_dot<Q4_0>(const uint8_t *ub, const XRow &x, const float *, const float *) {
    uint32_t r[36];
    lds_words(r, ub);
    const float2 off = f2(-8388616.f, -8388616.f);   // -(2^23 + 8)
    float y = 0.f;
#pragma unroll
    for (int b = 0; b < 8; ++b) {
        const float d = f16_bits(half_at(r, 18 * b));
        float2 acc = f2(0.f, 0.f);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const uint32_t w = word_at(r, 18 * b + 2 + 4 * t);
            acc = dot4(acc, w & 0x0F0F0F0Fu, off, x(8 * b + t));
            acc = dot4(acc, (w >> 4) & 0x0F0F0F0Fu, off, x(8 * b + 4 + t));
        }
        y = fmaf(d, acc.x + acc.y, y);
    }
    return y;
}

// Q8_0: 8 blocks; block b at byte 34b: f16 d, 32 int8 q; w = q * d.  The
// code byte with its sign bit flipped is q + 128.  Each half (4 blocks) is
// read separately to bound the registers.
template <>
__device__ __forceinline__ float unit_dot<Q8_0>(const uint8_t *ub, const XRow &x, const float *, const float *) {
    const float2 off = f2(-8388736.f, -8388736.f);   // -(2^23 + 128)
    float y = 0.f;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t r[36];
        lds_words(r, ub + 128 * h);   // bytes 128h .. 128h + 143 cover blocks 4h .. 4h + 3
#pragma unroll
        for (int bb = 0; bb < 4; ++bb) {
            const int b = 4 * h + bb;
            const int o = 34 * b - 128 * h;
            const float d = f16_bits(half_at(r, o));
            float2 acc = f2(0.f, 0.f);
#pragma unroll
            for (int t = 0; t < 8; ++t)
                acc = dot4(acc, word_at(r, o + 2 + 4 * t) ^ 0x80808080u, off, x(8 * b + t));
            y = fmaf(d, acc.x + acc.y, y);
        }
    }
    return y;
}

// Q4_K / Q5_K header: d, dmin, and the eight 6-bit (scale, min) pairs of the
// 12 bytes at offset 4 (GGUF K-quant packing), as dsc[s] = d * sc_s and
// dmn[s] = dmin * m_s (both exact in f32).
__device__ __forceinline__ void kq_header(uint32_t r0, uint32_t w0, uint32_t w1, uint32_t w2, float (&dsc)[8],
                                          float (&dmn)[8]) {
    const float d = f16_bits(r0 & 0xFFFFu), dmin = f16_bits(r0 >> 16);
    const uint32_t scA = w0 & 0x3F3F3F3Fu, mnA = w1 & 0x3F3F3F3Fu;
    const uint32_t scB = (w2 & 0x0F0F0F0Fu) | ((w0 >> 2) & 0x30303030u);
    const uint32_t mnB = ((w2 >> 4) & 0x0F0F0F0Fu) | ((w1 >> 2) & 0x30303030u);
    const float2 m23 = f2(-8388608.f, -8388608.f);   // -(2^23)
    float2 v;
    v = __fadd2_rn(mag01(scA), m23); dsc[0] = d * v.x; dsc[1] = d * v.y;
    v = __fadd2_rn(mag23(scA), m23); dsc[2] = d * v.x; dsc[3] = d * v.y;
    v = __fadd2_rn(mag01(scB), m23); dsc[4] = d * v.x; dsc[5] = d * v.y;
    v = __fadd2_rn(mag23(scB), m23); dsc[6] = d * v.x; dsc[7] = d * v.y;
    v = __fadd2_rn(mag01(mnA), m23); dmn[0] = dmin * v.x; dmn[1] = dmin * v.y;
    v = __fadd2_rn(mag23(mnA), m23); dmn[2] = dmin * v.x; dmn[3] = dmin * v.y;
    v = __fadd2_rn(mag01(mnB), m23); dmn[4] = dmin * v.x; dmn[5] = dmin * v.y;
    v = __fadd2_rn(mag23(mnB), m23); dmn[6] = dmin * v.x; dmn[7] = dmin * v.y;
}

// Q4_K: d @0, dmin @2, scales @4..15, qs @16..143; element e = 32 s + l is
// the low (s even) or high (s odd) nibble of qs[32 (s / 2) + l];
// w = d sc_s q - dmin m_s, summed as dsc_s * sum(q x) - dmn_s * sum(x).
// sum(q x) from subnormal codes and the block-scaled x (fb8: the unit's 8
// scale-back factors), sum(x) from the f32 sums of the unscaled x (xs8).
template <>
__device__ __forceinline__ float unit_dot<Q4_K>(const uint8_t *ub, const XRow &x, const float *xs8,
                                                const float *fb8) {
    uint32_t r[36];
    lds_words(r, ub);
    float dsc[8], dmn[8];
    kq_header(r[0], r[1], r[2], r[3], dsc, dmn);
    const float4 xa = *reinterpret_cast<const float4 *>(xs8), xb = *reinterpret_cast<const float4 *>(xs8 + 4);
    const float xsum[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
    const float4 fa = *reinterpret_cast<const float4 *>(fb8), fc = *reinterpret_cast<const float4 *>(fb8 + 4);
    const float fb[8] = {fa.x, fa.y, fa.z, fa.w, fc.x, fc.y, fc.z, fc.w};
    float y = 0.f;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        float2 alo = f2(0.f, 0.f), ahi = f2(0.f, 0.f);
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const uint32_t w = r[4 + 8 * p + t];
            alo = dot4s(alo, w & 0x0F0F0F0Fu, x(16 * p + t));
            ahi = dot4s(ahi, (w >> 4) & 0x0F0F0F0Fu, x(16 * p + 8 + t));
        }
        y = fmaf(dsc[2 * p], unscale(alo.x + alo.y, fb[2 * p]), y);
        y = fmaf(-dmn[2 * p], xsum[2 * p], y);
        y = fmaf(dsc[2 * p + 1], unscale(ahi.x + ahi.y, fb[2 * p + 1]), y);
        y = fmaf(-dmn[2 * p + 1], xsum[2 * p + 1], y);
    }
    return y;
}

// Q5_K: as Q4_K with qh[32] @16 and qs @48; bit s of qh[l] is bit 4 of
// element 32 s + l.
template <>
__device__ __forceinline__ float unit_dot<Q5_K>(const uint8_t *ub, const XRow &x, const float *xs8,
                                                const float *fb8) {
    uint32_t r[44];
    lds_words(r, ub);
    float dsc[8], dmn[8];
    kq_header(r[0], r[1], r[2], r[3], dsc, dmn);
    const float4 xa = *reinterpret_cast<const float4 *>(xs8), xb = *reinterpret_cast<const float4 *>(xs8 + 4);
    const float xsum[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
    const float4 fa = *reinterpret_cast<const float4 *>(fb8), fc = *reinterpret_cast<const float4 *>(fb8 + 4);
    const float fb[8] = {fa.x, fa.y, fa.z, fa.w, fc.x, fc.y, fc.z, fc.w};
    float y = 0.f;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        float2 alo = f2(0.f, 0.f), ahi = f2(0.f, 0.f);
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const uint32_t w = r[12 + 8 * p + t], qh = r[4 + t];
            const uint32_t qlo = (w & 0x0F0F0F0Fu) | (((qh >> (2 * p)) & 0x01010101u) << 4);
            const uint32_t qhi = ((w >> 4) & 0x0F0F0F0Fu) | (((qh >> (2 * p + 1)) & 0x01010101u) << 4);
            alo = dot4s(alo, qlo, x(16 * p + t));
            ahi = dot4s(ahi, qhi, x(16 * p + 8 + t));
        }
        y = fmaf(dsc[2 * p], unscale(alo.x + alo.y, fb[2 * p]), y);
        y = fmaf(-dmn[2 * p], xsum[2 * p], y);
        y = fmaf(dsc[2 * p + 1], unscale(ahi.x + ahi.y, fb[2 * p + 1]), y);
        y = fmaf(-dmn[2 * p + 1], xsum[2 * p + 1], y);
    }
    return y;
}

// Q6_K: ql[128] @0, qh[64] @128, int8 scales[16] @192, f16 d @208.
// Element e = 128 h + 32 j + l: low 4 bits from ql[64 h + 32 (j % 2) + l]
// (low nibble for j < 2, high for j >= 2), bits 4..5 = bits 2j, 2j+1 of
// qh[32 h + l]; w = d * scales[e / 16] * (q - 32).  The unit starts at an
// even byte; words are assembled from 4-byte aligned loads.
template <>
__device__ __forceinline__ float unit_dot<Q6_K>(const uint8_t *ub, const XRow &x, const float *, const float *) {
    const uint32_t sh = (uint32_t)(reinterpret_cast<uintptr_t>(ub) & 2u) * 8u;   // 0 or 16 bits
    const uint32_t *wp = reinterpret_cast<const uint32_t *>(ub - (sh >> 3));
    auto W = [&](int i) { return __funnelshift_r(wp[i], wp[i + 1], sh); };
    const float d = f16_bits(W(52));
    float ds[16];
    const float2 m128 = f2(-8388736.f, -8388736.f);   // -(2^23 + 128)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t s = W(48 + i) ^ 0x80808080u;
        const float2 a = __fadd2_rn(mag01(s), m128), b = __fadd2_rn(mag23(s), m128);
        ds[4 * i] = d * a.x;
        ds[4 * i + 1] = d * a.y;
        ds[4 * i + 2] = d * b.x;
        ds[4 * i + 3] = d * b.y;
    }
    const float2 off = f2(-8388640.f, -8388640.f);   // -(2^23 + 32)
    float y = 0.f;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        float2 acc[4][2];
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[j][0] = acc[j][1] = f2(0.f, 0.f);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const uint32_t qa = W(16 * h + u), qb = W(16 * h + 8 + u), qh = W(32 + 8 * h + u);
            const uint32_t q0 = (qa & 0x0F0F0F0Fu) | ((qh << 4) & 0x30303030u);
            const uint32_t q1 = (qb & 0x0F0F0F0Fu) | ((qh << 2) & 0x30303030u);
            const uint32_t q2 = ((qa >> 4) & 0x0F0F0F0Fu) | (qh & 0x30303030u);
            const uint32_t q3 = ((qb >> 4) & 0x0F0F0F0Fu) | ((qh >> 2) & 0x30303030u);
            const int hv = u >> 2;
            acc[0][hv] = dot4(acc[0][hv], q0, off, x(32 * h + u));
            acc[1][hv] = dot4(acc[1][hv], q1, off, x(32 * h + 8 + u));
            acc[2][hv] = dot4(acc[2][hv], q2, off, x(32 * h + 16 + u));
            acc[3][hv] = dot4(acc[3][hv], q3, off, x(32 * h + 24 + u));
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            y = fmaf(ds[8 * h + 2 * j], acc[j][0].x + acc[j][0].y, y);
            y = fmaf(ds[8 * h + 2 * j + 1], acc[j][1].x + acc[j][1].y, y);
        }
    }
    return y;
}

// ---------------------------------------------------------------------------
// The kernel.
// ---------------------------------------------------------------------------
struct StreamArgs {
    const uint8_t *W;
    const void *X;
    float *Y;
    int64_t M;
    int K;
    int S;             // ring slots per warp
    int off_x;         // shared-memory offsets (bytes)
    int off_xsum;
    int off_part;
    int off_bar;
    int off_flag;
    unsigned *status;
    uint64_t limit;
    AmaxOut amax;      // argmax mode when amax.keys is set: no output is stored
};

__device__ __forceinline__ bool warp_wait(volatile unsigned *abort_flag, uint64_t *bar, uint32_t parity,
                                          uint64_t limit) {
    bool ok = true;
    if (!mbar_try_wait(bar, parity)) {
        const long long t0 = clock64();
        for (;;) {
            if (mbar_try_wait_sleep(bar, parity, 1000u)) break;
            if (*abort_flag) {
                ok = false;
                break;
            }
            if ((uint64_t)(clock64() - t0) > limit) {
                *abort_flag = 1u;
                ok = false;
                break;
            }
        }
    }
    return __all_sync(0xffffffffu, ok);
}

template <int F, bool XBF16>
__global__ void __launch_bounds__(512, 1) gemv_stream_kernel(const __grid_constant__ StreamArgs a) {
    extern __shared__ __align__(1024) uint8_t sm[];
    constexpr int UB = UnitBytes<F>::B;
    constexpr int SLOT = slot_bytes(UB);
    const int nw = blockDim.x >> 5, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = a.S;
    const int U = a.K >> 8;                                     // units per row
    const int64_t r0 = (int64_t)blockIdx.x * a.M / gridDim.x;
    const int64_t r1 = (int64_t)(blockIdx.x + 1) * a.M / gridDim.x;
    const int nrows = (int)(r1 - r0);
    const int nunits = nrows * U;
    const int nst = (nunits + kLanes - 1) / kLanes;            // stages of the CTA
    const uint8_t *wcta = a.W + r0 * (int64_t)U * UB;
    const int64_t cta_bytes = (int64_t)nunits * UB;

    float *xs = reinterpret_cast<float *>(sm + a.off_x);
    float *xsum = reinterpret_cast<float *>(sm + a.off_xsum);
    float *part = reinterpret_cast<float *>(sm + a.off_part);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + a.off_bar);
    volatile unsigned *abort_flag = reinterpret_cast<volatile unsigned *>(sm + a.off_flag);

    if (threadIdx.x == 0) {
        for (int i = 0; i < nw * S; ++i) mbar_init(&bars[i], 1);
        *abort_flag = 0u;
        fence_barrier_init();
    }
    __syncthreads();
    pdl_launch_dependents();

    // this warp's stages: s = warp + nw * j, j = 0 .. my_nst - 1
    const int my_nst = warp < nst ? (nst - 1 - warp) / nw + 1 : 0;
    auto issue = [&](int j) {
        const int s = warp + nw * j;
        const int64_t off = (int64_t)s * kLanes * UB;
        const int64_t rem = cta_bytes - off;
        const uint32_t bytes = (uint32_t)(rem < kLanes * UB ? rem : kLanes * UB);
        const int slot = warp * S + j % S;
        mbar_arrive_expect_tx(&bars[slot], bytes);
        tma_load_1d(sm + (size_t)slot * SLOT, wcta + off, bytes, &bars[slot]);
    };
    // weights first: they do not depend on the preceding grid
    if (lane == 0)
        for (int j = 0; j < S && j < my_nst; ++j) issue(j);

    pdl_wait();   // X and Y are ordered behind the preceding grid

    // X -> shared memory, f32, chunk (p, q) of 4 floats at p * 64 + (q ^ (p & 7)).
    // Q4_K / Q5_K: each 32-element block (8 consecutive chunks, 8 consecutive
    // threads: K / 4 is a multiple of 64, so every warp runs every round)
    // is stored times 2^k, k = 126 - E clamped to [-1, 127] (E: the binary
    // exponent of the block's largest |x|), with its scale-back factor
    // 2^(85 - k) and the f32 sum of its unscaled elements.
    // The loads of a batch of XB chunks per thread are all issued before any
    // is used, so that staging costs about one L2 round trip per batch.
    {
        float4 *xs4 = reinterpret_cast<float4 *>(xs);
        const int nch = a.K >> 2;
        constexpr int XB = 8;
        for (int c0 = threadIdx.x; c0 < nch; c0 += XB * blockDim.x) {
            float4 vb[XB];
#pragma unroll
            for (int i = 0; i < XB; ++i) {
                const int c = c0 + i * (int)blockDim.x;
                if (c < nch) {
                    if constexpr (XBF16) {
                        const uint2 b = reinterpret_cast<const uint2 *>(a.X)[c];
                        vb[i] = make_float4(__uint_as_float(b.x << 16), __uint_as_float(b.x & 0xFFFF0000u),
                                            __uint_as_float(b.y << 16), __uint_as_float(b.y & 0xFFFF0000u));
                    } else {
                        vb[i] = reinterpret_cast<const float4 *>(a.X)[c];
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < XB; ++i) {
                const int c = c0 + i * (int)blockDim.x;
                if (c >= nch) break;   // warp-uniform: nch is a multiple of 64
                float4 v = vb[i];
                if constexpr (kmin_fmt(F)) {
                    float m = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
                    float sx = (v.x + v.y) + (v.z + v.w);
#pragma unroll
                    for (int o = 1; o < 8; o <<= 1) {
                        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                        sx += __shfl_xor_sync(0xffffffffu, sx, o);
                    }
                    int k = 126 - ((int)(__float_as_uint(m) >> 23) - 127);
                    k = k < -1 ? -1 : (k > 127 ? 127 : k);
                    const float sc = __uint_as_float((uint32_t)(127 + k) << 23);   // 2^k
                    v.x *= sc;
                    v.y *= sc;
                    v.z *= sc;
                    v.w *= sc;
                    if ((c & 7) == 0) {
                        xsum[c >> 3] = sx;
                        xsum[(a.K >> 5) + (c >> 3)] = __uint_as_float((uint32_t)(212 - k) << 23);   // 2^(85 - k)
                    }
                }
                const int p = c >> 6, q = c & 63;
                xs4[(p << 6) | (q ^ (p & 7))] = v;
            }
        }
    }
    __syncthreads();

    const float4 *xs4 = reinterpret_cast<const float4 *>(xs);
    float *__restrict__ Yc = a.Y + r0;
    const bool amax = a.amax.keys != nullptr;
    unsigned long long best = 0ull;   // argmax mode: this thread's best (value, row) key
    int done = 0;   // stages of this warp consumed
    for (int j = 0; j < my_nst; ++j) {
        const int slot = warp * S + j % S;
        if (!warp_wait(abort_flag, &bars[slot], (uint32_t)(j / S) & 1u, a.limit)) break;
        const int s = warp + nw * j;
        const int u = s * kLanes + lane;
        float v = 0.f;
        int key = 0x7FFFFFFF;
        if (u < nunits) {
            key = u / U;                   // row of the unit (within the CTA)
            const int p = u - key * U;     // unit within the row
            const XRow xr(xs4 + (p << 6), p & 7);
            v = unit_dot<F>(sm + (size_t)slot * SLOT + lane * UB, xr, xsum + 8 * p, xsum + (a.K >> 5) + 8 * p);
        }
        __syncwarp();
        if (lane == 0 && j + S < my_nst) issue(j + S);   // every lane has read the slot
        done = j + 1;
        // segmented reduction by row: each row's first lane of the stage
        // ends up with the stage's sum for that row
#pragma unroll
        for (int o = 1; o < kLanes; o <<= 1) {
            const float vo = __shfl_down_sync(0xffffffffu, v, o);
            const int ko = __shfl_down_sync(0xffffffffu, key, o);
            if (lane + o < kLanes && ko == key) v += vo;
        }
        const int kp = __shfl_up_sync(0xffffffffu, key, 1);
        if (u < nunits && (lane == 0 || kp != key)) {
            const bool starts = key * U >= s * kLanes;
            const bool ends = key * U + U <= (s + 1) * kLanes;
            if (starts && ends) {
                if (amax)
                    amax_fold(best, v, (int)(r0 + key));
                else
                    Yc[key] = v;
            } else
                part[2 * s + (starts ? 1 : 0)] = v;   // 0: row begun earlier, 1: row continues later
        }
    }
    // copies still in flight (only after an abort): wait for them before exit
    if (lane == 0) {
        const int issued = my_nst < done + S ? my_nst : done + S;
        for (int j = done; j < issued; ++j)
            (void)mbar_wait(&bars[warp * S + j % S], (uint32_t)(j / S) & 1u,
                            a.limit < (1ull << 31) ? (1ull << 31) : a.limit);
    }
    __syncthreads();
    if (*abort_flag) {
        if (threadIdx.x == 0) report_status(a.status, kStatusTimeout);
        return;
    }
    // rows that cross stages: stage partials in stage order
    for (int rl = threadIdx.x; rl < nrows; rl += blockDim.x) {
        const int sa = (rl * U) / kLanes, sb = (rl * U + U - 1) / kLanes;
        if (sa == sb) continue;
        float v = part[2 * sa + 1];
        for (int s = sa + 1; s <= sb; ++s) v += part[2 * s];
        if (amax)
            amax_fold(best, v, (int)(r0 + rl));
        else
            Yc[rl] = v;
    }
    if (amax) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const unsigned long long x = __shfl_xor_sync(0xffffffffu, best, o);
            best = x > best ? x : best;
        }
        if (lane == 0 && best != 0ull) {
            atomicMax(a.amax.keys, best);
            __threadfence();
        }
        amax_last_cta(a.amax, 1);
    }
}

int unit_bytes_of(int fmt) {
    switch (fmt) {
    case Q8_0: return UnitBytes<Q8_0>::B;
    case Q4_0: return UnitBytes<Q4_0>::B;
    case Q4_K: return UnitBytes<Q4_K>::B;
    case Q6_K: return UnitBytes<Q6_K>::B;
    case Q5_K: return UnitBytes<Q5_K>::B;
    default: return 0;
    }
}

constexpr int kSmemMax = 232448 - 1024;   // the opt-in maximum, less room for static shared words
constexpr int kSmemPerSM = 233472;        // shared memory of one SM (two CTAs: each also has 1 KB reserved)

// Shared-memory layout for nw warps, S slots, K and up to nst stages.
struct StreamLayout {
    int off_x, off_xsum, off_part, off_bar, off_flag, total;
};
StreamLayout stream_layout(int fmt, int nw, int S, int64_t K, int64_t nst) {
    StreamLayout L;
    const int slot = slot_bytes(unit_bytes_of(fmt));
    int64_t o = (int64_t)nw * S * slot;
    L.off_x = (int)o;
    o += K * 4;
    L.off_xsum = (int)o;
    o += kmin_fmt(fmt) ? K / 4 : 0;   // per 32-element block: the sum of x, then the scale-back factor
    o = (o + 15) / 16 * 16;
    L.off_part = (int)o;
    o += (nst * 8 + 15) / 16 * 16;
    L.off_bar = (int)o;
    o += (int64_t)nw * S * 8;
    L.off_flag = (int)o;
    o += 16;
    L.total = o > (1ll << 30) ? (1 << 30) : (int)o;
    return L;
}

template <int F, bool XBF16>
cudaError_t launch_typed(const StreamPlan &p, const StreamArgs &a, bool pdl, cudaStream_t st) {
    auto kern = gemv_stream_kernel<F, XBF16>;
    static std::atomic<int> configured[64];   // largest dynamic shared memory set, per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured[dev & 63].load() < p.smem) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax);
        if (e != cudaSuccess) return e;
        configured[dev & 63].store(kSmemMax);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.grid, 1, 1);
    cfg.blockDim = dim3((unsigned)(p.warps * 32), 1, 1);
    cfg.dynamicSmemBytes = (size_t)p.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, kern, a);
    if (e != cudaSuccess) return e;
    return launched(cudaGetLastError());
}

template <int F>
cudaError_t launch_fmt(const StreamPlan &p, const StreamArgs &a, int xbf16, bool pdl, cudaStream_t st) {
    return xbf16 ? launch_typed<F, true>(p, a, pdl, st) : launch_typed<F, false>(p, a, pdl, st);
}

}  // namespace

bool plan_gemv_stream(int fmt, int64_t M, int64_t K, int num_sms, int force_warps, StreamPlan &p) {
    const int ub = unit_bytes_of(fmt);
    if (!ub || K % 256 || M < 1 || num_sms < 1 || K > (1 << 15)) return false;
    if ((K / 256 * ub) % 16) return false;   // rows must start 16-byte aligned
    // Short launches (K <= 4096, at most 64 MB of weights) run two CTAs of
    // at most 8 warps per SM: when one launch follows another on the stream,
    // the next launch's CTAs then start (and stream their weights) on SMs
    // where the previous launch's CTAs are still finishing.  Measured on
    // Q4_0 / Q8_0 / Q4_K rows of 4096: 5-6% shorter launches; long rows
    // (every CTA stages all of X) and long launches do better with one.
    const int64_t wbytes = M * (K / 256) * ub;
    int cps = K <= 4096 && wbytes <= (64ll << 20) ? 2 : 1;
    if (force_warps > 16 / cps) cps = 1;
    const int lim = cps == 2 ? kSmemPerSM / 2 - 3072 : kSmemMax;
    int64_t grid = M < (int64_t)cps * num_sms ? M : (int64_t)cps * num_sms;
    for (int attempt = 0; attempt < 8; ++attempt) {
        const int64_t rows = (M + grid - 1) / grid;
        const int64_t nst = (rows * (K / 256) + kLanes - 1) / kLanes;
        for (int nw : {16, 12, 8, 4}) {
            if (force_warps ? nw != force_warps : nw > 16 / cps) continue;
            for (int S : {3, 2}) {
                const StreamLayout L = stream_layout(fmt, nw, S, K, nst);
                if (L.total <= lim) {
                    p.grid = (int)grid;
                    p.warps = nw;
                    p.S = S;
                    p.smem = L.total;
                    return true;
                }
            }
        }
        if (grid >= M) break;
        grid = grid * 2 < M ? grid * 2 : M;   // more, smaller CTAs: fewer partials each
    }
    return false;
}

cudaError_t launch_gemv_stream(int fmt, const StreamPlan &p, const uint8_t *W, int64_t M, int64_t K, const void *X,
                               int xbf16, float *Y, bool pdl, unsigned *status, uint64_t limit, cudaStream_t st,
                               unsigned long long *amax_ws, int32_t *idx, float *val) {
    const int64_t rows = (M + p.grid - 1) / p.grid;
    const int64_t nst = (rows * (K / 256) + kLanes - 1) / kLanes;
    const StreamLayout L = stream_layout(fmt, p.warps, p.S, K, nst);
    if (L.total > p.smem) return cudaErrorInvalidValue;
    StreamArgs a;
    a.W = W;
    a.X = X;
    a.Y = Y;
    a.M = M;
    a.K = (int)K;
    a.S = p.S;
    a.off_x = L.off_x;
    a.off_xsum = L.off_xsum;
    a.off_part = L.off_part;
    a.off_bar = L.off_bar;
    a.off_flag = L.off_flag;
    a.status = status;
    a.limit = limit;
    a.amax = AmaxOut{amax_ws, amax_ws ? reinterpret_cast<unsigned *>(amax_ws + 1) : nullptr, idx, val};
    switch (fmt) {
    case Q8_0: return launch_fmt<Q8_0>(p, a, xbf16, pdl, st);
    case Q4_0: return launch_fmt<Q4_0>(p, a, xbf16, pdl, st);
    case Q4_K: return launch_fmt<Q4_K>(p, a, xbf16, pdl, st);
    case Q6_K: return launch_fmt<Q6_K>(p, a, xbf16, pdl, st);
    case Q5_K: return launch_fmt<Q5_K>(p, a, xbf16, pdl, st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace qmm
