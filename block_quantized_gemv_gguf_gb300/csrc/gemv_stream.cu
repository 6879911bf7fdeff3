// gemv_stream.cu -- decode GEMV for one token (N = 1), 16-byte aligned rows:
//
//     y[m] = sum_k w(m, k) * x[k]
//
// the per-token projection of "cera 0.5.0 src/model/llama.rs" (decode) and
// the row loops of "cera 0.5.2 src/backend/cpu.rs" (matmul_*_f32 /
// gemv_dispatch), restated for GB300 SMs (one or two CTAs per SM):
//
//   * Unit = 256 consecutive weights of one row (8 Q4_0 / Q8_0 blocks, or
//     one Q4_K / Q5_K / Q6_K super-block): 144, 272, 176 or 210 bytes.
//     A CTA owns whole rows of one weight matrix; its rows are one
//     contiguous byte range of W.  Up to four matrices sharing X and K run
//     in one launch, the CTAs split over them by rows (a segment table).
//   * Task = the units of R consecutive rows (a "row group", R = 1, 2 or 4)
//     at one unit column p: the R units share the same 256 x values, which
//     a lane reads from shared memory once and applies to all R rows, so the
//     shared-memory traffic of X (4 bytes per weight at R = 1, against 0.56
//     bytes of Q4_0 weights) drops R-fold.
//   * Tasks are numbered group-major (t = g U + p, U units per row).  Each
//     warp streams its own "stages" of 32 consecutive tasks: one bulk copy
//     per (row, run of columns) piece of the stage -- a single copy when the
//     stage is contiguous in W -- completing on a warp-private mbarrier, in a
//     ring of S slots (S >= 2: each stage issued once the previous one has
//     landed).  Lane l owns task l of the stage.  No data passes between
//     warps until the very end.
//   * The weight copies are issued before the kernel waits on the preceding
//     grid (the weights are static; X and Y are ordered behind it).
//   * X (f32; bf16 widened) sits in shared memory once per CTA, in 16-byte
//     chunks XOR-swizzled by unit column so that the 32 lanes of a warp,
//     each on its own column, read it without bank conflicts.
//   * Arithmetic: every integer code becomes an exact f32 by a byte permute
//     into the mantissa of 2^23 and one packed subtraction (which also
//     removes the format's offset), then a packed f32 FMA with x; Q4_K and
//     Q5_K codes, which carry no offset, are exact f32 subnormals against X
//     scaled per block by a power of two.  Each block's (or sub-block's)
//     scale multiplies the f32 block sum; the Q4_K / Q5_K min term uses the
//     sub-block sums of x.
//   * Row results: a segmented warp-shuffle reduction by row group over each
//     stage (a group held entirely in one stage is stored directly); groups
//     that cross stages are summed from per-stage partials in stage order at
//     the end.  Every sum has a fixed order: the result is deterministic.
//   * plan_gemv_stream picks R, CTAs per SM, warps and slots from the shape
//     (rules measured on GB300, stated there); gemv_direct_kernel, a variant
//     that loads each lane's unit straight into registers, runs on request.
//
// All waits are bounded; a warp that gives up raises the CTA's abort flag,
// waits (bounded) for its own copies in flight, and the CTA reports
// QMM_ERR_TIMEOUT in the status word.
#include <algorithm>
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
// A stage slot: 32 tasks of R units, padded (the Q6_K reader fetches up to
// 4 bytes past its unit) and rounded to 128 bytes.
__host__ __device__ constexpr int slot_bytes(int ub, int R) { return (kLanes * R * ub + 16 + 127) / 128 * 128; }

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

// The unit column's 64 chunks of x, XOR-swizzled: logical chunk 8k + t sits
// at p[t][8k] (the XOR only touches t, so k is an immediate offset).
struct XRow {
    const float4 *p[8];
    __device__ __forceinline__ XRow(const float4 *x0, int sw) {
#pragma unroll
        for (int t = 0; t < 8; ++t) p[t] = x0 + (t ^ sw);
    }
    __device__ __forceinline__ float4 operator()(int q) const { return p[q & 7][q & ~7]; }
};

// 32-bit word at byte offset `o` (even, compile-time after unrolling) of a
// register copy of 4-byte aligned bytes.
template <int NW>
__device__ __forceinline__ uint32_t word_at(const uint32_t (&r)[NW], int o) {
    return (o & 2) ? __byte_perm(r[o >> 2], r[(o >> 2) + 1], 0x5432u) : r[o >> 2];
}
template <int NW>
__device__ __forceinline__ uint32_t half_at(const uint32_t (&r)[NW], int o) {
    return (o & 2) ? (r[o >> 2] >> 16) : (r[o >> 2] & 0xFFFFu);
}

// NW words from an 8-byte aligned shared-memory address.
template <int NW>
__device__ __forceinline__ void lds_w64(uint32_t (&r)[NW], const uint8_t *p) {
    const uint2 *q = reinterpret_cast<const uint2 *>(p);
#pragma unroll
    for (int i = 0; i < NW / 2; ++i) {
        const uint2 v = q[i];
        r[2 * i] = v.x;
        r[2 * i + 1] = v.y;
    }
}
// NW words from a 16-byte aligned shared-memory address.
template <int NW>
__device__ __forceinline__ void lds_w128(uint32_t (&r)[NW], const uint8_t *p) {
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
// One task: for each of R units (row i at ub + i * rs; same unit column),
// y[i] = sum over its 256 weights of w * x.  x: the column's 64 x chunks;
// xs8 / fb8: the column's 8 sub-block sums of x and scale-back factors
// (Q4_K / Q5_K).  Within a unit the order of every sum is fixed.
// ---------------------------------------------------------------------------
template <int F, int R>
__device__ __forceinline__ void task_dot(const uint8_t *ub, int rs, const XRow &x, const float *xs8, const float *fb8,
                                         float (&y)[R]);

// Q4_0: 8 blocks; block b at byte 18b: f16 d, 16 bytes qs; element e < 16
// is the low nibble of qs[e], e >= 16 the high nibble of qs[e - 16];
// w = (nibble - 8) * d.  Blocks are read in pairs through 40-byte windows
// at 8-byte aligned word offsets 0, 8, 18, 26.
template <int R>
__device__ __forceinline__ void q40_task(const uint8_t *ub, int rs, const XRow &x, float (&y)[R]) {
    const float2 off = f2(-8388616.f, -8388616.f);   // -(2^23 + 8)
#pragma unroll
    for (int i = 0; i < R; ++i) y[i] = 0.f;
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        constexpr int kW0[4] = {0, 8, 18, 26};
        const int w0 = kW0[h];
        uint32_t r[R][10];
#pragma unroll
        for (int i = 0; i < R; ++i) lds_w64(r[i], ub + i * rs + 4 * w0);
#pragma unroll
        for (int bb = 0; bb < 2; ++bb) {
            const int b = 2 * h + bb;
            const int o = 18 * b - 4 * w0;
            float2 acc[R];
#pragma unroll
            for (int i = 0; i < R; ++i) acc[i] = f2(0.f, 0.f);
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const float4 xl = x(8 * b + t), xh = x(8 * b + 4 + t);
#pragma unroll
                for (int i = 0; i < R; ++i) {
                    const uint32_t w = word_at(r[i], o + 2 + 4 * t);
                    acc[i] = dot4(acc[i], w & 0x0F0F0F0Fu, off, xl);
                    acc[i] = dot4(acc[i], (w >> 4) & 0x0F0F0F0Fu, off, xh);
                }
            }
#pragma unroll
            for (int i = 0; i < R; ++i) y[i] = fmaf(f16_bits(half_at(r[i], o)), acc[i].x + acc[i].y, y[i]);
        }
    }
}

// Q8_0: 8 blocks; block b at byte 34b: f16 d, 32 int8 q; w = q * d.  The
// code byte with its sign bit flipped is q + 128.  Each block is read
// through a 40-byte window at an 8-byte aligned word offset.
template <int R>
__device__ __forceinline__ void q80_task(const uint8_t *ub, int rs, const XRow &x, float (&y)[R]) {
    const float2 off = f2(-8388736.f, -8388736.f);   // -(2^23 + 128)
#pragma unroll
    for (int i = 0; i < R; ++i) y[i] = 0.f;
#pragma unroll
    for (int b = 0; b < 8; ++b) {
        constexpr int kW0[8] = {0, 8, 16, 24, 34, 42, 50, 58};
        const int w0 = kW0[b];
        const int o = 34 * b - 4 * w0;
        uint32_t r[R][10];
#pragma unroll
        for (int i = 0; i < R; ++i) lds_w64(r[i], ub + i * rs + 4 * w0);
        float2 acc[R];
#pragma unroll
        for (int i = 0; i < R; ++i) acc[i] = f2(0.f, 0.f);
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const float4 xv = x(8 * b + t);
#pragma unroll
            for (int i = 0; i < R; ++i) acc[i] = dot4(acc[i], word_at(r[i], o + 2 + 4 * t) ^ 0x80808080u, off, xv);
        }
#pragma unroll
        for (int i = 0; i < R; ++i) y[i] = fmaf(f16_bits(half_at(r[i], o)), acc[i].x + acc[i].y, y[i]);
    }
}

// Q4_K / Q5_K header: d, dmin, and the eight 6-bit (scale, min) pairs of the
// 12 bytes at offset 4 (GGUF K-quant packing).  Sub-blocks 0..3 take byte s
// of (scA, mnA), sub-blocks 4..7 byte s - 4 of (scB, mnB).
struct KHead {
    float d, dmin;
    uint32_t scA, mnA, scB, mnB;
    __device__ __forceinline__ void load(const uint8_t *ub) {
        const uint4 h = *reinterpret_cast<const uint4 *>(ub);
        d = f16_bits(h.x & 0xFFFFu);
        dmin = f16_bits(h.x >> 16);
        scA = h.y & 0x3F3F3F3Fu;
        mnA = h.z & 0x3F3F3F3Fu;
        scB = (h.w & 0x0F0F0F0Fu) | ((h.y >> 2) & 0x30303030u);
        mnB = ((h.w >> 4) & 0x0F0F0F0Fu) | ((h.z >> 2) & 0x30303030u);
    }
    // d * sc and dmin * m of sub-blocks 2p and 2p + 1 (exact in f32)
    __device__ __forceinline__ void pair(int p, float2 &dsc, float2 &dmn) const {
        const float2 m23 = f2(-8388608.f, -8388608.f);   // -(2^23)
        const uint32_t sc = p < 2 ? scA : scB, mn = p < 2 ? mnA : mnB;
        const float2 vs = __fadd2_rn((p & 1) ? mag23(sc) : mag01(sc), m23);
        const float2 vm = __fadd2_rn((p & 1) ? mag23(mn) : mag01(mn), m23);
        dsc = f2(d * vs.x, d * vs.y);
        dmn = f2(dmin * vm.x, dmin * vm.y);
    }
};

// Q4_K: d @0, dmin @2, scales @4..15, qs @16..143; element e = 32 s + l is
// the low (s even) or high (s odd) nibble of qs[32 (s / 2) + l];
// w = d sc_s q - dmin m_s, summed as dsc_s * sum(q x) - dmn_s * sum(x).
// sum(q x) from subnormal codes and the block-scaled x (fb8: the column's 8
// scale-back factors), sum(x) from the f32 sums of the unscaled x (xs8).
template <int R>
__device__ __forceinline__ void q4k_task(const uint8_t *ub, int rs, const XRow &x, const float *xs8, const float *fb8,
                                         float (&y)[R]) {
    KHead hd[R];
#pragma unroll
    for (int i = 0; i < R; ++i) {
        hd[i].load(ub + i * rs);
        y[i] = 0.f;
    }
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        uint32_t r[R][8];
#pragma unroll
        for (int i = 0; i < R; ++i) lds_w128(r[i], ub + i * rs + 16 + 32 * p);
        float2 alo[R], ahi[R];
#pragma unroll
        for (int i = 0; i < R; ++i) alo[i] = ahi[i] = f2(0.f, 0.f);
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const float4 xl = x(16 * p + t), xh = x(16 * p + 8 + t);
#pragma unroll
            for (int i = 0; i < R; ++i) {
                alo[i] = dot4s(alo[i], r[i][t] & 0x0F0F0F0Fu, xl);
                ahi[i] = dot4s(ahi[i], (r[i][t] >> 4) & 0x0F0F0F0Fu, xh);
            }
        }
        const float sl = xs8[2 * p], sh = xs8[2 * p + 1], fl = fb8[2 * p], fh = fb8[2 * p + 1];
#pragma unroll
        for (int i = 0; i < R; ++i) {
            float2 dsc, dmn;
            hd[i].pair(p, dsc, dmn);
            y[i] = fmaf(dsc.x, unscale(alo[i].x + alo[i].y, fl), y[i]);
            y[i] = fmaf(-dmn.x, sl, y[i]);
            y[i] = fmaf(dsc.y, unscale(ahi[i].x + ahi[i].y, fh), y[i]);
            y[i] = fmaf(-dmn.y, sh, y[i]);
        }
    }
}

// Q5_K: as Q4_K with qh[32] @16 and qs @48; bit s of qh[l] is bit 4 of
// element 32 s + l.
template <int R>
__device__ __forceinline__ void q5k_task(const uint8_t *ub, int rs, const XRow &x, const float *xs8, const float *fb8,
                                         float (&y)[R]) {
    KHead hd[R];
#pragma unroll
    for (int i = 0; i < R; ++i) {
        hd[i].load(ub + i * rs);
        y[i] = 0.f;
    }
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        float2 alo[R], ahi[R];
#pragma unroll
        for (int i = 0; i < R; ++i) alo[i] = ahi[i] = f2(0.f, 0.f);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {   // words 4 hf .. 4 hf + 3 of the 32-byte pieces
            uint32_t q[R][4], qh[R][4];
#pragma unroll
            for (int i = 0; i < R; ++i) {
                lds_w128(q[i], ub + i * rs + 48 + 32 * p + 16 * hf);
                lds_w128(qh[i], ub + i * rs + 16 + 16 * hf);
            }
#pragma unroll
            for (int tt = 0; tt < 4; ++tt) {
                const int t = 4 * hf + tt;
                const float4 xl = x(16 * p + t), xh = x(16 * p + 8 + t);
#pragma unroll
                for (int i = 0; i < R; ++i) {
                    const uint32_t w = q[i][tt], hb = qh[i][tt];
                    const uint32_t qlo = (w & 0x0F0F0F0Fu) | (((hb >> (2 * p)) & 0x01010101u) << 4);
                    const uint32_t qhi = ((w >> 4) & 0x0F0F0F0Fu) | (((hb >> (2 * p + 1)) & 0x01010101u) << 4);
                    alo[i] = dot4s(alo[i], qlo, xl);
                    ahi[i] = dot4s(ahi[i], qhi, xh);
                }
            }
        }
        const float sl = xs8[2 * p], sh = xs8[2 * p + 1], fl = fb8[2 * p], fh = fb8[2 * p + 1];
#pragma unroll
        for (int i = 0; i < R; ++i) {
            float2 dsc, dmn;
            hd[i].pair(p, dsc, dmn);
            y[i] = fmaf(dsc.x, unscale(alo[i].x + alo[i].y, fl), y[i]);
            y[i] = fmaf(-dmn.x, sl, y[i]);
            y[i] = fmaf(dsc.y, unscale(ahi[i].x + ahi[i].y, fh), y[i]);
            y[i] = fmaf(-dmn.y, sh, y[i]);
        }
    }
}

// Q6_K: ql[128] @0, qh[64] @128, int8 scales[16] @192, f16 d @208.
// Element e = 128 h + 32 j + l: low 4 bits from ql[64 h + 32 (j % 2) + l]
// (low nibble for j < 2, high for j >= 2), bits 4..5 = bits 2j, 2j+1 of
// qh[32 h + l]; w = d * scales[e / 16] * (q - 32).  A unit starts at an
// even byte; words are assembled from 4-byte aligned loads.
struct Q6Row {
    const uint32_t *wp;
    uint32_t sh;
    __device__ __forceinline__ explicit Q6Row(const uint8_t *ub) {
        sh = (uint32_t)(reinterpret_cast<uintptr_t>(ub) & 2u) * 8u;   // 0 or 16 bits
        wp = reinterpret_cast<const uint32_t *>(ub - (sh >> 3));
    }
    __device__ __forceinline__ uint32_t operator()(int i) const { return __funnelshift_r(wp[i], wp[i + 1], sh); }
};

template <int R>
__device__ __forceinline__ void q6k_task(const uint8_t *ub, int rs, const XRow &x, float (&y)[R]) {
    const float2 off = f2(-8388640.f, -8388640.f);   // -(2^23 + 32)
    const float2 m128 = f2(-8388736.f, -8388736.f);  // -(2^23 + 128)
    float d[R];
#pragma unroll
    for (int i = 0; i < R; ++i) {
        d[i] = f16_bits(Q6Row(ub + i * rs)(52));
        y[i] = 0.f;
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int hv = 0; hv < 2; ++hv) {
            float2 acc[R][4];
#pragma unroll
            for (int i = 0; i < R; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = f2(0.f, 0.f);
#pragma unroll
            for (int uu = 0; uu < 4; ++uu) {
                const int u = 4 * hv + uu;
                const float4 x0 = x(32 * h + u), x1 = x(32 * h + 8 + u), x2 = x(32 * h + 16 + u),
                             x3 = x(32 * h + 24 + u);
#pragma unroll
                for (int i = 0; i < R; ++i) {
                    const Q6Row W(ub + i * rs);
                    const uint32_t qa = W(16 * h + u), qb = W(16 * h + 8 + u), qh = W(32 + 8 * h + u);
                    const uint32_t q0 = (qa & 0x0F0F0F0Fu) | ((qh << 4) & 0x30303030u);
                    const uint32_t q1 = (qb & 0x0F0F0F0Fu) | ((qh << 2) & 0x30303030u);
                    const uint32_t q2 = ((qa >> 4) & 0x0F0F0F0Fu) | (qh & 0x30303030u);
                    const uint32_t q3 = ((qb >> 4) & 0x0F0F0F0Fu) | ((qh >> 2) & 0x30303030u);
                    acc[i][0] = dot4(acc[i][0], q0, off, x0);
                    acc[i][1] = dot4(acc[i][1], q1, off, x1);
                    acc[i][2] = dot4(acc[i][2], q2, off, x2);
                    acc[i][3] = dot4(acc[i][3], q3, off, x3);
                }
            }
            // scales 8h + 2j + hv, j = 0..3: bytes hv, 2 + hv of words 48 + 2h, 49 + 2h
#pragma unroll
            for (int i = 0; i < R; ++i) {
                const Q6Row W(ub + i * rs);
                const uint32_t sa = W(48 + 2 * h) ^ 0x80808080u, sb = W(49 + 2 * h) ^ 0x80808080u;
                const float2 s01 = __fadd2_rn(f2(mag(sa, hv), mag(sa, 2 + hv)), m128);
                const float2 s23 = __fadd2_rn(f2(mag(sb, hv), mag(sb, 2 + hv)), m128);
                y[i] = fmaf(d[i] * s01.x, acc[i][0].x + acc[i][0].y, y[i]);
                y[i] = fmaf(d[i] * s01.y, acc[i][1].x + acc[i][1].y, y[i]);
                y[i] = fmaf(d[i] * s23.x, acc[i][2].x + acc[i][2].y, y[i]);
                y[i] = fmaf(d[i] * s23.y, acc[i][3].x + acc[i][3].y, y[i]);
            }
        }
    }
}

template <int F, int R>
__device__ __forceinline__ void task_dot(const uint8_t *ub, int rs, const XRow &x, const float *xs8, const float *fb8,
                                         float (&y)[R]) {
    if constexpr (F == Q4_0) q40_task<R>(ub, rs, x, y);
    else if constexpr (F == Q8_0) q80_task<R>(ub, rs, x, y);
    else if constexpr (F == Q4_K) q4k_task<R>(ub, rs, x, xs8, fb8, y);
    else if constexpr (F == Q5_K) q5k_task<R>(ub, rs, x, xs8, fb8, y);
    else q6k_task<R>(ub, rs, x, y);
}

// ---------------------------------------------------------------------------
// The kernel.
// ---------------------------------------------------------------------------
struct StreamArgs {
    // up to QMM_MAX_SEGS weight matrices sharing X: segment i has rows Ms[i]
    // at Ws[i], output Ys[i], and CTAs cta0[i] .. cta0[i + 1] - 1
    const uint8_t *Ws[QMM_MAX_SEGS];
    float *Ys[QMM_MAX_SEGS];
    int64_t Ms[QMM_MAX_SEGS];
    int cta0[QMM_MAX_SEGS + 1];
    int nseg;
    const void *X;
    int K;
    int S;             // ring slots per warp
    int stagger;       // S >= 2: one stage issued up front, stage j + S - 1 once stage j has landed
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

// A stage is one contiguous byte range of W when its rows are consecutive
// (R = 1) or it holds whole row groups (U divides 32).
__host__ __device__ constexpr bool stage_contiguous(int R, int U) { return R == 1 || kLanes % U == 0; }

template <int F, bool XBF16, int R>
__global__ void __launch_bounds__(512, 1) gemv_stream_kernel(const __grid_constant__ StreamArgs a) {
    extern __shared__ __align__(1024) uint8_t sm[];
    constexpr int UB = UnitBytes<F>::B;
    constexpr int SLOT = slot_bytes(UB, R);
    const int nw = blockDim.x >> 5, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = a.S;
    const int U = a.K >> 8;                                     // units per row
    int sg = 0;   // this CTA's weight matrix
    while (sg + 1 < a.nseg && (int)blockIdx.x >= a.cta0[sg + 1]) ++sg;
    const int lb = (int)blockIdx.x - a.cta0[sg], nb = a.cta0[sg + 1] - a.cta0[sg];
    const int64_t r0 = (int64_t)lb * a.Ms[sg] / nb;
    const int64_t r1 = (int64_t)(lb + 1) * a.Ms[sg] / nb;
    const int nrows = (int)(r1 - r0);
    const int ngrp = (nrows + R - 1) / R;                       // row groups (the last may be short)
    const int ntasks = ngrp * U;
    const int nst = (ntasks + kLanes - 1) / kLanes;            // stages of the CTA
    const uint8_t *wcta = a.Ws[sg] + r0 * (int64_t)U * UB;
    const bool contiguous = stage_contiguous(R, U);

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
    // Stage layout in its slot: the stage's tasks split into segments by
    // row group; segment [L, E) of group g holds its R rows one after the
    // other, n = E - L units each: unit (lane l, row i) at R L + i n + (l - L).
    // Warp-collective.
    auto issue = [&](int j) {
        const int s = warp + nw * j;
        const int t0 = s * kLanes;
        const int te = min(t0 + kLanes, ntasks);
        const int slot = warp * S + j % S;
        uint8_t *dst = sm + (size_t)slot * SLOT;
        uint64_t *bar = &bars[slot];
        if (contiguous) {
            if (lane == 0) {
                int64_t u0, nu;   // first unit (in W's order) and unit count
                if (R == 1) {
                    u0 = t0;
                    nu = te - t0;
                } else {
                    const int ra = (t0 / U) * R, rb = min((te / U) * R, nrows);
                    u0 = (int64_t)ra * U;
                    nu = (int64_t)(rb - ra) * U;
                }
                const uint32_t bytes = (uint32_t)(nu * UB);
                mbar_arrive_expect_tx(bar, bytes);
                tma_load_1d(dst, wcta + u0 * UB, bytes, bar);
            }
        } else {
            const int g0 = t0 / U;
            if (lane == 0) {
                uint32_t bytes = 0;
                for (int g = g0; g * U < te; ++g) {
                    const int n = min(te, (g + 1) * U) - max(t0, g * U);
                    bytes += (uint32_t)(n * min(R, nrows - g * R) * UB);
                }
                mbar_arrive_expect_tx(bar, bytes);
            }
            __syncwarp();
            for (int k = lane;; k += kLanes) {   // piece k: row k % R of segment k / R
                const int g = g0 + k / R, i = k % R;
                if (g * U >= te) break;
                if (g * R + i >= nrows) continue;
                const int L = max(t0, g * U) - t0, n = min(te, (g + 1) * U) - t0 - L;
                const uint8_t *src = wcta + ((int64_t)(g * R + i) * U + (t0 + L - g * U)) * UB;
                tma_load_1d(dst + (size_t)(R * L + i * n) * UB, src, (uint32_t)(n * UB), bar);
            }
        }
    };
    // weights first: they do not depend on the preceding grid
    const bool stagger = a.stagger && S >= 2;
    int nissued = 0;   // stages of this warp issued so far (warp-uniform)
    for (; nissued < (stagger ? 1 : S) && nissued < my_nst; ++nissued) issue(nissued);

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
    float *__restrict__ Yc = a.Ys[sg] + r0;
    const bool amax = a.amax.keys != nullptr;
    unsigned long long best = 0ull;   // argmax mode: this thread's best (value, row) key
    int done = 0;   // stages of this warp consumed
    for (int j = 0; j < my_nst; ++j) {
        const int slot = warp * S + j % S;
        if (!warp_wait(abort_flag, &bars[slot], (uint32_t)(j / S) & 1u, a.limit)) break;
        // staggered: the next stage's copy goes out as soon as this one has
        // landed (its slot held stage j - 1, consumed last iteration)
        for (; stagger && nissued < my_nst && nissued <= j + S - 1; ++nissued) issue(nissued);
        const int s = warp + nw * j;
        const int t0 = s * kLanes;
        const int te = min(t0 + kLanes, ntasks);
        const int t = t0 + lane;
        float v[R];
        int key = 0x7FFFFFFF, g = 0;
        if (t < te) {
            g = t / U;                               // row group of the task
            const int p = t - g * U;                 // unit column
            const int L = max(t0, g * U) - t0, n = min(te, (g + 1) * U) - t0 - L;
            key = g;
            const XRow xr(xs4 + (p << 6), p & 7);
            task_dot<F, R>(sm + (size_t)slot * SLOT + (size_t)(R * L + (lane - L)) * UB, n * UB, xr, xsum + 8 * p,
                           xsum + (a.K >> 5) + 8 * p, v);
        } else {
#pragma unroll
            for (int i = 0; i < R; ++i) v[i] = 0.f;
        }
        __syncwarp();
        if (!stagger && j + S < my_nst) issue(nissued++);   // every lane has read the slot: stage j + S
        done = j + 1;
        // segmented reduction by row group: each group's first lane of the
        // stage ends up with the stage's sums for the group's rows
#pragma unroll
        for (int o = 1; o < kLanes; o <<= 1) {
            const int ko = __shfl_down_sync(0xffffffffu, key, o);
            const bool same = lane + o < kLanes && ko == key;
#pragma unroll
            for (int i = 0; i < R; ++i) {
                const float vo = __shfl_down_sync(0xffffffffu, v[i], o);
                if (same) v[i] += vo;
            }
        }
        const int kp = __shfl_up_sync(0xffffffffu, key, 1);
        if (t < te && (lane == 0 || kp != key)) {
            const bool starts = g * U >= t0;
            const bool ends = (g + 1) * U <= t0 + kLanes;
#pragma unroll
            for (int i = 0; i < R; ++i) {
                const int row = g * R + i;
                if (row >= nrows) break;
                if (starts && ends) {
                    if (amax)
                        amax_fold(best, v[i], (int)(r0 + row));
                    else
                        Yc[row] = v[i];
                } else {
                    part[(2 * s + (starts ? 1 : 0)) * R + i] = v[i];   // 0: begun earlier, 1: continues later
                }
            }
        }
    }
    // copies still in flight (only after an abort): wait for them before exit
    if (lane == 0) {
        for (int j = done; j < nissued; ++j)
            (void)mbar_wait(&bars[warp * S + j % S], (uint32_t)(j / S) & 1u,
                            a.limit < (1ull << 31) ? (1ull << 31) : a.limit);
    }
    __syncthreads();
    if (*abort_flag) {
        if (threadIdx.x == 0) report_status(a.status, kStatusTimeout);
        return;
    }
    // row groups that cross stages: stage partials in stage order
    for (int rl = threadIdx.x; rl < nrows; rl += blockDim.x) {
        const int g = rl / R, i = rl - g * R;
        const int sa = (g * U) / kLanes, sb = (g * U + U - 1) / kLanes;
        if (sa == sb) continue;
        float v = part[(2 * sa + 1) * R + i];
        for (int s = sa + 1; s <= sb; ++s) v += part[2 * s * R + i];
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

// ---------------------------------------------------------------------------
// Direct-load variant for the 144-byte units (Q4_0, Q4_K): no shared-memory
// ring and no mbarrier hand-off.  Each lane reads its own unit with nine
// 16-byte read-only global loads straight into registers, two units per lane
// in flight (ping-pong register buffers: the next unit's loads are issued
// before the current unit's arithmetic).  X, the row reduction and the
// partial sums are as in the staged kernel with one row per task.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ldg_unit(uint32_t (&r)[36], const uint8_t *g) {
    const uint4 *q = reinterpret_cast<const uint4 *>(g);
#pragma unroll
    for (int i = 0; i < 9; ++i) {
        const uint4 v = __ldg(q + i);
        r[4 * i] = v.x;
        r[4 * i + 1] = v.y;
        r[4 * i + 2] = v.z;
        r[4 * i + 3] = v.w;
    }
}

template <int F>
__device__ __forceinline__ float unit_dot_regs(const uint32_t (&r)[36], const XRow &x, const float *xs8,
                                               const float *fb8) {
    float y = 0.f;
    if constexpr (F == Q4_0) {
        const float2 off = f2(-8388616.f, -8388616.f);   // -(2^23 + 8)
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            float2 acc = f2(0.f, 0.f);
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const uint32_t w = word_at(r, 18 * b + 2 + 4 * t);
                acc = dot4(acc, w & 0x0F0F0F0Fu, off, x(8 * b + t));
                acc = dot4(acc, (w >> 4) & 0x0F0F0F0Fu, off, x(8 * b + 4 + t));
            }
            y = fmaf(f16_bits(half_at(r, 18 * b)), acc.x + acc.y, y);
        }
    } else {   // Q4_K
        KHead hd;
        hd.d = f16_bits(r[0] & 0xFFFFu);
        hd.dmin = f16_bits(r[0] >> 16);
        hd.scA = r[1] & 0x3F3F3F3Fu;
        hd.mnA = r[2] & 0x3F3F3F3Fu;
        hd.scB = (r[3] & 0x0F0F0F0Fu) | ((r[1] >> 2) & 0x30303030u);
        hd.mnB = ((r[3] >> 4) & 0x0F0F0F0Fu) | ((r[2] >> 2) & 0x30303030u);
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            float2 alo = f2(0.f, 0.f), ahi = f2(0.f, 0.f);
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                const uint32_t w = r[4 + 8 * p + t];
                alo = dot4s(alo, w & 0x0F0F0F0Fu, x(16 * p + t));
                ahi = dot4s(ahi, (w >> 4) & 0x0F0F0F0Fu, x(16 * p + 8 + t));
            }
            float2 dsc, dmn;
            hd.pair(p, dsc, dmn);
            y = fmaf(dsc.x, unscale(alo.x + alo.y, fb8[2 * p]), y);
            y = fmaf(-dmn.x, xs8[2 * p], y);
            y = fmaf(dsc.y, unscale(ahi.x + ahi.y, fb8[2 * p + 1]), y);
            y = fmaf(-dmn.y, xs8[2 * p + 1], y);
        }
    }
    return y;
}

template <int F, bool XBF16>
__global__ void __launch_bounds__(512, 1) gemv_direct_kernel(const __grid_constant__ StreamArgs a) {
    extern __shared__ __align__(1024) uint8_t sm[];
    constexpr int UB = UnitBytes<F>::B;
    static_assert(UB == 144, "direct loads: 144-byte units");
    const int nw = blockDim.x >> 5, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int U = a.K >> 8;
    int sg = 0;   // this CTA's weight matrix
    while (sg + 1 < a.nseg && (int)blockIdx.x >= a.cta0[sg + 1]) ++sg;
    const int lb = (int)blockIdx.x - a.cta0[sg], nb = a.cta0[sg + 1] - a.cta0[sg];
    const int64_t r0 = (int64_t)lb * a.Ms[sg] / nb;
    const int64_t r1 = (int64_t)(lb + 1) * a.Ms[sg] / nb;
    const int nrows = (int)(r1 - r0);
    const int nunits = nrows * U;
    const int nst = (nunits + kLanes - 1) / kLanes;
    const uint8_t *wcta = a.Ws[sg] + r0 * (int64_t)U * UB;
    float *xs = reinterpret_cast<float *>(sm + a.off_x);
    float *xsum = reinterpret_cast<float *>(sm + a.off_xsum);
    float *part = reinterpret_cast<float *>(sm + a.off_part);
    pdl_launch_dependents();

    const int my_nst = warp < nst ? (nst - 1 - warp) / nw + 1 : 0;
    auto unit_of = [&](int j) { return (warp + nw * j) * kLanes + lane; };
    uint32_t ra[36], rb[36];
    // the first two units: the weights do not depend on the preceding grid
    if (my_nst > 0 && unit_of(0) < nunits) ldg_unit(ra, wcta + (int64_t)unit_of(0) * UB);
    if (my_nst > 1 && unit_of(1) < nunits) ldg_unit(rb, wcta + (int64_t)unit_of(1) * UB);

    pdl_wait();   // X and Y are ordered behind the preceding grid
    {   // X -> shared memory, as in the staged kernel
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
                if (c >= nch) break;
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
                    const float sc = __uint_as_float((uint32_t)(127 + k) << 23);
                    v.x *= sc;
                    v.y *= sc;
                    v.z *= sc;
                    v.w *= sc;
                    if ((c & 7) == 0) {
                        xsum[c >> 3] = sx;
                        xsum[(a.K >> 5) + (c >> 3)] = __uint_as_float((uint32_t)(212 - k) << 23);
                    }
                }
                const int p = c >> 6, q = c & 63;
                xs4[(p << 6) | (q ^ (p & 7))] = v;
            }
        }
    }
    __syncthreads();

    const float4 *xs4 = reinterpret_cast<const float4 *>(xs);
    float *__restrict__ Yc = a.Ys[sg] + r0;
    const bool amax = a.amax.keys != nullptr;
    unsigned long long best = 0ull;
    auto process = [&](int j, const uint32_t(&r)[36]) {
        const int s = warp + nw * j;
        const int u = s * kLanes + lane;
        float v = 0.f;
        int key = 0x7FFFFFFF;
        if (u < nunits) {
            key = u / U;
            const int p = u - key * U;
            v = unit_dot_regs<F>(r, XRow(xs4 + (p << 6), p & 7), xsum + 8 * p, xsum + (a.K >> 5) + 8 * p);
        }
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
                part[2 * s + (starts ? 1 : 0)] = v;
        }
    };
    for (int j = 0; j < my_nst; j += 2) {
        process(j, ra);
        if (j + 2 < my_nst && unit_of(j + 2) < nunits) ldg_unit(ra, wcta + (int64_t)unit_of(j + 2) * UB);
        if (j + 1 < my_nst) {
            process(j + 1, rb);
            if (j + 3 < my_nst && unit_of(j + 3) < nunits) ldg_unit(rb, wcta + (int64_t)unit_of(j + 3) * UB);
        }
    }
    __syncthreads();
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

// Shared-memory layout for R rows per task, nw warps, S slots, K and up to
// nst stages.
struct StreamLayout {
    int off_x, off_xsum, off_part, off_bar, off_flag, total;
};
StreamLayout stream_layout(int fmt, int R, int nw, int S, int64_t K, int64_t nst) {
    StreamLayout L;
    const int slot = slot_bytes(unit_bytes_of(fmt), R);
    int64_t o = (int64_t)nw * S * slot;
    L.off_x = (int)o;
    o += K * 4;
    L.off_xsum = (int)o;
    o += kmin_fmt(fmt) ? K / 4 : 0;   // per 32-element block: the sum of x, then the scale-back factor
    o = (o + 15) / 16 * 16;
    L.off_part = (int)o;
    o += (nst * 8 * R + 15) / 16 * 16;
    L.off_bar = (int)o;
    o += (int64_t)nw * S * 8;
    L.off_flag = (int)o;
    o += 16;
    L.total = o > (1ll << 30) ? (1 << 30) : (int)o;
    return L;
}

// Kern: the kernel itself (a template argument, so that each kernel keeps
// its own record of the shared-memory attribute set on each device).
template <auto Kern>
cudaError_t launch_kernel(const StreamPlan &p, const StreamArgs &a, bool pdl, cudaStream_t st) {
    const auto kern = Kern;
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

template <int F, bool XBF16, int R>
cudaError_t launch_typed(const StreamPlan &p, const StreamArgs &a, bool pdl, cudaStream_t st) {
    return launch_kernel<gemv_stream_kernel<F, XBF16, R>>(p, a, pdl, st);
}

template <int F, bool XBF16>
cudaError_t launch_rows(const StreamPlan &p, const StreamArgs &a, bool pdl, cudaStream_t st) {
    if constexpr (UnitBytes<F>::B == 144) {
        if (p.direct) return launch_kernel<gemv_direct_kernel<F, XBF16>>(p, a, pdl, st);
    }
    switch (p.R) {
    case 1: return launch_typed<F, XBF16, 1>(p, a, pdl, st);
    case 2: return launch_typed<F, XBF16, 2>(p, a, pdl, st);
    case 4: return launch_typed<F, XBF16, 4>(p, a, pdl, st);
    default: return cudaErrorInvalidValue;
    }
}

template <int F>
cudaError_t launch_fmt(const StreamPlan &p, const StreamArgs &a, int xbf16, bool pdl, cudaStream_t st) {
    return xbf16 ? launch_rows<F, true>(p, a, pdl, st) : launch_rows<F, false>(p, a, pdl, st);
}

}  // namespace

// Split `grid` CTAs over the segments in proportion to their rows (at least
// one, at most M_i each); returns the most rows any CTA gets.
static int64_t split_ctas(const int64_t *Ms, int nseg, int64_t M, int64_t grid, int (&cta0)[QMM_MAX_SEGS + 1]) {
    int64_t rows_max = 0;
    cta0[0] = 0;
    for (int i = 0; i < nseg; ++i) {
        int64_t c = (grid * Ms[i] + M / 2) / M;
        c = c < 1 ? 1 : (c > Ms[i] ? Ms[i] : c);
        cta0[i + 1] = cta0[i] + (int)c;
        const int64_t r = (Ms[i] + c - 1) / c;
        rows_max = r > rows_max ? r : rows_max;
    }
    return rows_max;
}

bool plan_gemv_stream(int fmt, int64_t M, int64_t K, int num_sms, const StreamForce &force, StreamPlan &p) {
    return plan_gemv_stream(fmt, &M, 1, K, num_sms, force, p);
}

bool plan_gemv_stream(int fmt, const int64_t *Ms, int nseg, int64_t K, int num_sms, const StreamForce &force,
                      StreamPlan &p) {
    const int ub = unit_bytes_of(fmt);
    if (nseg < 1 || nseg > QMM_MAX_SEGS) return false;
    int64_t M = 0;   // all segments' rows
    for (int i = 0; i < nseg; ++i) {
        if (Ms[i] < 1) return false;
        M += Ms[i];
    }
    if (!ub || K % 256 || num_sms < 1 || K > (1 << 15) || M > (1ll << 31) - 1) return false;
    if ((K / 256 * ub) % 16) return false;   // rows must start 16-byte aligned
    const int U = (int)(K / 256);
    const int64_t wbytes = M * U * ub;
    const bool short_launch = wbytes <= (64ll << 20);
    // Rows per task (measured on the Llama-3-8B decode shapes, GB300): two
    // where every SM still gets at least 4 stages of 32 tasks and a stage is
    // one contiguous copy; of the piecewise stages only the offset-free
    // K-quants (Q4_K, Q5_K: the fewest ALU instructions per weight, so the
    // X reads weigh most) gain from two.  Four rows per task need slots so
    // large that too few warps fit: only on request.  Piecewise stages need
    // 16-byte aligned units (all formats but Q6_K).
    int R = 1;
    if ((double)M * U / (2.0 * kLanes * num_sms) >= 4.0 &&
        (stage_contiguous(2, U) || (kmin_fmt(fmt) && ub % 16 == 0)))
        R = 2;
    if (force.r) {
        if (force.r != 1 && force.r != 2 && force.r != 4) return false;
        if (!stage_contiguous(force.r, U) && ub % 16) return false;
        R = force.r;
    }
    // The direct-load variant (144-byte units, one row per task): on request.
    const bool direct = force.direct == 1 && ub == 144;
    if (direct) R = 1;
    // Two CTAs per SM for launches of short rows (K <= 4096: X is cheap to
    // stage twice) up to 64 MB with at least 8 rows per CTA; one otherwise
    // (a launch of very few rows per SM is mostly the staging of X).
    int cps = K <= 4096 && short_launch && M >= 16ll * num_sms ? 2 : 1;
    if (force.cps == 1 || force.cps == 2) cps = force.cps;
    if (force.warps > 16 / cps || force.slots > 3) return false;
    const int lim = cps == 2 ? kSmemPerSM / 2 - 3072 : kSmemMax;
    // Every CTA takes more than 1 / (cps + 1) of the SM's shared memory, so
    // that no SM ever holds more than cps CTAs of one launch.  Without that
    // floor, when launches follow one another (programmatic dependent
    // launch), the CTAs of the next launch pile up on the SMs that free up
    // first and leave others idle; measured on a 32-layer decoder sequence.
    const int floor_smem = kSmemPerSM / (cps + 1) + 1024;
    int64_t grid = M < (int64_t)cps * num_sms ? M : (int64_t)cps * num_sms;
    for (int attempt = 0; attempt < 8; ++attempt) {
        int cta0[QMM_MAX_SEGS + 1];
        const int64_t rows = split_ctas(Ms, nseg, M, grid, cta0);
        const int64_t nst = ((rows + R - 1) / R * U + kLanes - 1) / kLanes;
        // Slots: one per warp unless forced.  Two slots with staggered issue
        // (stage j + 1's copy goes out once stage j has landed) run the big
        // shapes alone 3-4% faster (14336 x 4096, 4096 x 14336), but their
        // larger footprint keeps the next launch's CTAs off the SM until
        // they exit: the following launch lost as much, and a 32-layer
        // decoder sequence ran 3% slower.
        const int S = direct ? 0 : force.slots ? force.slots : 1;
        // Warps: n_fit = the most that fit (at most 16 per SM); of the counts
        // from 0.6 n_fit to n_fit, the one whose warps get the most even share
        // of the CTA's stages -- a warp with one stage more than the others
        // keeps the SM half idle at the end -- and among those the most
        // warps; a warp per stage (at least 8) when one round covers the CTA.
        const double tasks = (double)((rows + R - 1) / R * U) / kLanes;   // stages, the last one fractional
        int n_fit = 0;
        for (int nw = force.warps ? force.warps : 16 / cps; nw >= 1 && !n_fit; --nw) {
            if (stream_layout(fmt, R, nw, S, K, nst).total <= lim) n_fit = nw;
            if (force.warps) break;
        }
        int best = 0;
        double best_bal = -1.0;
        const bool one_round = !force.warps && n_fit > 8 && nst <= n_fit;
        if (one_round) best = (int)std::max<int64_t>(8, nst);
        for (int nw = n_fit; !one_round && nw >= 1 && 5 * nw >= 3 * n_fit && (!force.warps || nw == n_fit); --nw) {
            const int64_t r = (nst + nw - 1) / nw;
            const double bal = r <= 1 ? 1.0 : tasks / ((double)nw * r);
            if (bal > best_bal + 0.02) {
                best = nw;
                best_bal = bal;
            }
        }
        if (best) {
            const StreamLayout L = stream_layout(fmt, R, best, S, K, nst);
            p.grid = cta0[nseg];
            p.nseg = nseg;
            for (int i = 0; i <= nseg; ++i) p.cta0[i] = cta0[i];
            p.warps = best;
            p.S = S;
            p.R = R;
            p.smem = std::max(L.total, std::min(floor_smem, lim));
            p.direct = direct ? 1 : 0;
            p.stagger = S >= 2 && force.stagger != 2 ? 1 : 0;
            return true;
        }
        if (grid >= M) break;
        grid = grid * 2 < M ? grid * 2 : M;   // more, smaller CTAs: fewer partials each
    }
    return false;
}

cudaError_t launch_gemv_stream(int fmt, const StreamPlan &p, const uint8_t *W, int64_t M, int64_t K, const void *X,
                               int xbf16, float *Y, bool pdl, unsigned *status, uint64_t limit, cudaStream_t st,
                               unsigned long long *amax_ws, int32_t *idx, float *val) {
    return launch_gemv_stream(fmt, p, &W, &Y, &M, K, X, xbf16, pdl, status, limit, st, amax_ws, idx, val);
}

cudaError_t launch_gemv_stream(int fmt, const StreamPlan &p, const uint8_t *const *Ws, float *const *Ys,
                               const int64_t *Ms, int64_t K, const void *X, int xbf16, bool pdl, unsigned *status,
                               uint64_t limit, cudaStream_t st, unsigned long long *amax_ws, int32_t *idx,
                               float *val) {
    if (p.nseg < 1 || p.nseg > QMM_MAX_SEGS || (amax_ws && p.nseg != 1)) return cudaErrorInvalidValue;
    StreamArgs a;
    int64_t rows = 0;
    for (int i = 0; i < p.nseg; ++i) {
        const int c = p.cta0[i + 1] - p.cta0[i];
        if (c < 1 || Ms[i] < 1) return cudaErrorInvalidValue;
        const int64_t r = (Ms[i] + c - 1) / c;
        rows = r > rows ? r : rows;
        a.Ws[i] = Ws[i];
        a.Ys[i] = Ys[i];
        a.Ms[i] = Ms[i];
    }
    for (int i = 0; i <= p.nseg; ++i) a.cta0[i] = p.cta0[i];
    a.nseg = p.nseg;
    if (a.cta0[p.nseg] != p.grid) return cudaErrorInvalidValue;
    const int64_t nst = ((rows + p.R - 1) / p.R * (K / 256) + kLanes - 1) / kLanes;
    const StreamLayout L = stream_layout(fmt, p.R, p.warps, p.S, K, nst);
    if (L.total > p.smem) return cudaErrorInvalidValue;
    a.X = X;
    a.K = (int)K;
    a.S = p.S;
    a.stagger = p.stagger;
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
