// gemv_tc.cu -- GEMV for 1 <= N <= 8 tokens on mma.sync (f16 in, f32
// accumulate), weights straight from their GGUF bytes:
//
//     Y[n, m] = sum_k X[n, k] * w(m, k)
//
// the decode projection of "cera 0.5.0 src/model/llama.rs" and the batched
// positions of its project_logits_batched (one weight read for every token),
// for Q8_0, Q4_0, Q4_K and Q5_K rows whose 256-weight units are 16-byte
// aligned.
//
// Layout and flow:
//   * A "tile" is 16 rows x one 256-weight unit of K (the rows' bytes of that
//     unit).  A CTA owns a contiguous range of 16-row groups; each warp
//     walks its own list of tiles through a private ring of S shared-memory
//     slots, one 2-D TMA copy per tile, completion on a warp-private
//     mbarrier.  At the start, one thread asks L2 to prefetch the CTA's
//     weight bytes, so HBM sees the whole range at once; the tile copies
//     then mostly hit L2.
//   * The weights are static: their copies (and the prefetch) start before
//     the kernel waits on the preceding grid; X and Y are ordered behind it.
//   * X is split per token into binary16 pieces hi + lo of x * 2^-e (e per
//     token, so that max |x| * 2^-e < 2^15; |x - (hi + lo) 2^e| <=
//     2^-22 |x| + 2^-40 max|x|) and stored in the MMA B-fragment order; token
//     n's pieces are MMA columns 2n, 2n + 1.
//   * A operand: the integer codes, exact in binary16: a code v in the
//     mantissa of 1024.0 (one bitwise op makes two of them, one per 16-bit
//     half), then one packed f16 add removes 1024 and the format's offset
//     (or, for Q4_K / Q5_K, one packed f16 FMA forms sc * q).  A nibble left
//     at bits 4..7 reads as 16 q; the matching X pieces are stored divided
//     by 16, so no shift is needed.
//   * Each MMA (16 rows x 16 k x 8 columns) is exact in its products and
//     accumulates in f32; the per-block (Q8_0, Q4_0) or per-super-block
//     (Q4_K, Q5_K: d, and dmin times a second MMA of the 6-bit mins with the
//     sub-block sums of x) scale multiplies the f32 result.
//   * Rows: a warp that owns whole 16-row groups writes Y directly; when a
//     CTA has fewer groups than warps, the warps split K and the partial
//     sums are added in warp order in shared memory (deterministic).
// All waits are bounded; a warp that gives up raises the CTA's abort flag,
// waits (bounded) for its own copies in flight, and the CTA reports
// QMM_ERR_TIMEOUT in the status word.
#include <atomic>

#include "amax.cuh"
#include "common.cuh"
#include "kernels.h"

namespace qmm {
namespace {

constexpr int kTR = 16;   // rows per tile (MMA M)

template <int F> struct TcUnit;   // bytes of one 256-weight unit of a row
template <> struct TcUnit<Q8_0> { static constexpr int B = 272; };
template <> struct TcUnit<Q4_0> { static constexpr int B = 144; };
template <> struct TcUnit<Q4_K> { static constexpr int B = 144; };
template <> struct TcUnit<Q5_K> { static constexpr int B = 176; };

// Whether natural element e (0..255) of a unit is held as 16 * code (its X
// pieces are stored divided by 16).
template <int F>
__host__ __device__ constexpr bool x16_elem(int e) {
    return F == Q4_0 ? (e & 31) >= 16 : (F == Q4_K || F == Q5_K) ? ((e >> 5) & 1) != 0 : false;
}

// ---------------------------------------------------------------------------
// small device helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t hadd2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t r;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
    return r;
}
constexpr uint32_t kMagic = 0x64006400u;   // (1024, 1024)
constexpr uint32_t kM1024 = 0xE400E400u;   // (-1024, -1024)
constexpr uint32_t kM1032 = 0xE408E408u;   // (-1032, -1032)
constexpr uint32_t kM1152 = 0xE480E480u;   // (-1152, -1152)

// two codes of a packed word as (1024 + code) binary16 halves
__device__ __forceinline__ uint32_t nib_lo(uint32_t w) { return (w & 0x000F000Fu) | kMagic; }   // bytes 0, 2 low nibbles
__device__ __forceinline__ uint32_t nib_hi(uint32_t w) { return (w & 0x00F000F0u) | kMagic; }   // bytes 0, 2 high nibbles (x16)
__device__ __forceinline__ uint32_t byte_pr(uint32_t w) { return (w & 0x00FF00FFu) ^ 0x64806480u; }   // bytes 0, 2 with the sign bit flipped

// 32-bit word of shared memory at an address known to be 2 mod 4
__device__ __forceinline__ uint32_t lds_mis2(const uint8_t *p) {
    const uint32_t *q = reinterpret_cast<const uint32_t *>(p - 2);
    return __byte_perm(q[0], q[1], 0x5432u);
}
template <bool MIS>
__device__ __forceinline__ uint32_t ldw(const uint8_t *p) {
    if constexpr (MIS) return lds_mis2(p);
    else return *reinterpret_cast<const uint32_t *>(p);
}
__device__ __forceinline__ float ldh(const uint8_t *p) { return f16_bits(*reinterpret_cast<const uint16_t *>(p)); }

// d += A * B, m16n8k16, f16 x f16 -> f32
__device__ __forceinline__ void mma(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint2 b) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b.x), "r"(b.y));
}

// B fragments of one tile: for n-tile j the lane's column is 8j + g (token
// (8j + g) / 2, piece (8j + g) % 2); kgroup q (16 elements of the unit) is 32
// bytes on from the tile's base.  Columns past 2N read a valid column again:
// their outputs are never used.
template <int NT>
struct BFrag {
    const uint8_t *p[NT];
    __device__ __forceinline__ uint2 operator()(int j, int q) const {
        return *reinterpret_cast<const uint2 *>(p[j] + 32 * q);
    }
    // one 32-bit word (the sub-block sums: b0 only)
    __device__ __forceinline__ uint32_t word(int j) const { return *reinterpret_cast<const uint32_t *>(p[j]); }
};

// d = A * B (+ the zero quad z, which stays in registers: nothing is
// re-zeroed per MMA)
struct ZQ {
    float z[4];
};
__device__ __forceinline__ ZQ zq() {
    ZQ q;
    asm("mov.b32 %0, 0;\n\tmov.b32 %1, 0;\n\tmov.b32 %2, 0;\n\tmov.b32 %3, 0;"
        : "=f"(q.z[0]), "=f"(q.z[1]), "=f"(q.z[2]), "=f"(q.z[3]));
    return q;
}
__device__ __forceinline__ void mma_z(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint2 b,
                                      const ZQ &z) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b.x), "r"(b.y), "f"(z.z[0]), "f"(z.z[1]), "f"(z.z[2]),
          "f"(z.z[3]));
}

template <int NT>
__device__ __forceinline__ void zero(float (&d)[NT][4]) {
#pragma unroll
    for (int j = 0; j < NT; ++j) d[j][0] = d[j][1] = d[j][2] = d[j][3] = 0.f;
}

// ---------------------------------------------------------------------------
// One tile (16 rows x 256 weights): accumulate into yg[j] (row g, token
// 4j + t) and yg8[j] (row g + 8).  rg / rg8: the rows' bytes of the unit.
// ---------------------------------------------------------------------------
template <int F, int NT>
__device__ __forceinline__ void tile_dot(const uint8_t *rg, const uint8_t *rg8, const BFrag<NT> &B,
                                         const BFrag<NT> &Bs, int t, float (&yg)[NT], float (&yg8)[NT], const ZQ &z);

// Q4_0: block b at 18b: f16 d, qs[16]; kgroup 2b = low nibbles (elements
// 0..15), 2b + 1 = high nibbles (16..31); w = (nibble - 8) d.
template <>
__device__ __forceinline__ void tile_dot<Q4_0, 1>(const uint8_t *rg, const uint8_t *rg8, const BFrag<1> &B,
                                                  const BFrag<1> &, int t, float (&yg)[1], float (&yg8)[1], const ZQ &z) {
#pragma unroll
    for (int b = 0; b < 8; ++b) {
        const int o = 18 * b + 2 + 4 * t;
        uint32_t w, w8;
        if (b & 1) {
            w = ldw<false>(rg + o);
            w8 = ldw<false>(rg8 + o);
        } else {
            w = ldw<true>(rg + o);
            w8 = ldw<true>(rg8 + o);
        }
        const float dg = ldh(rg + 18 * b), dg8 = ldh(rg8 + 18 * b);
        const uint32_t s = w >> 8, s8 = w8 >> 8;
        float D[4];
        mma_z(D, hadd2(nib_lo(w), kM1032), hadd2(nib_lo(w8), kM1032), hadd2(nib_lo(s), kM1032),
              hadd2(nib_lo(s8), kM1032), B(0, 2 * b), z);
        mma(D, hadd2(nib_hi(w), kM1152), hadd2(nib_hi(w8), kM1152), hadd2(nib_hi(s), kM1152),
            hadd2(nib_hi(s8), kM1152), B(0, 2 * b + 1));
        yg[0] = fmaf(dg, D[0] + D[1], yg[0]);
        yg8[0] = fmaf(dg8, D[2] + D[3], yg8[0]);
    }
}

template <>
__device__ __forceinline__ void tile_dot<Q4_0, 2>(const uint8_t *rg, const uint8_t *rg8, const BFrag<2> &B,
                                                  const BFrag<2> &, int t, float (&yg)[2], float (&yg8)[2], const ZQ &z) {
#pragma unroll
    for (int b = 0; b < 8; ++b) {
        const int o = 18 * b + 2 + 4 * t;
        uint32_t w, w8;
        if (b & 1) {
            w = ldw<false>(rg + o);
            w8 = ldw<false>(rg8 + o);
        } else {
            w = ldw<true>(rg + o);
            w8 = ldw<true>(rg8 + o);
        }
        const float dg = ldh(rg + 18 * b), dg8 = ldh(rg8 + 18 * b);
        const uint32_t s = w >> 8, s8 = w8 >> 8;
        const uint32_t l0 = hadd2(nib_lo(w), kM1032), l1 = hadd2(nib_lo(w8), kM1032), l2 = hadd2(nib_lo(s), kM1032),
                       l3 = hadd2(nib_lo(s8), kM1032);
        const uint32_t h0 = hadd2(nib_hi(w), kM1152), h1 = hadd2(nib_hi(w8), kM1152), h2 = hadd2(nib_hi(s), kM1152),
                       h3 = hadd2(nib_hi(s8), kM1152);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            float D[4];
            mma_z(D, l0, l1, l2, l3, B(j, 2 * b), z);
            mma(D, h0, h1, h2, h3, B(j, 2 * b + 1));
            yg[j] = fmaf(dg, D[0] + D[1], yg[j]);
            yg8[j] = fmaf(dg8, D[2] + D[3], yg8[j]);
        }
    }
}

// Q8_0: block b at 34b: f16 d, 32 int8 q; kgroup 2b = elements 0..15 (words
// 0..3 of qs), 2b + 1 = elements 16..31; w = q d.
template <int NT>
__device__ __forceinline__ void tile_q8_0(const uint8_t *rg, const uint8_t *rg8, const BFrag<NT> &B, int t,
                                          float (&yg)[NT], float (&yg8)[NT], const ZQ &z) {
#pragma unroll
    for (int b = 0; b < 8; ++b) {
        const float dg = ldh(rg + 34 * b), dg8 = ldh(rg8 + 34 * b);
        uint32_t a[2][4];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int o = 34 * b + 2 + 16 * h + 4 * t;
            uint32_t w, w8;
            if (b & 1) {
                w = ldw<false>(rg + o);
                w8 = ldw<false>(rg8 + o);
            } else {
                w = ldw<true>(rg + o);
                w8 = ldw<true>(rg8 + o);
            }
            a[h][0] = hadd2(byte_pr(w), kM1152);
            a[h][1] = hadd2(byte_pr(w8), kM1152);
            a[h][2] = hadd2(byte_pr(w >> 8), kM1152);
            a[h][3] = hadd2(byte_pr(w8 >> 8), kM1152);
        }
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            float D[4];
            mma_z(D, a[0][0], a[0][1], a[0][2], a[0][3], B(j, 2 * b), z);
            mma(D, a[1][0], a[1][1], a[1][2], a[1][3], B(j, 2 * b + 1));
            yg[j] = fmaf(dg, D[0] + D[1], yg[j]);
            yg8[j] = fmaf(dg8, D[2] + D[3], yg8[j]);
        }
    }
}
template <>
__device__ __forceinline__ void tile_dot<Q8_0, 1>(const uint8_t *rg, const uint8_t *rg8, const BFrag<1> &B,
                                                  const BFrag<1> &, int t, float (&yg)[1], float (&yg8)[1], const ZQ &z) {
    tile_q8_0<1>(rg, rg8, B, t, yg, yg8, z);
}
template <>
__device__ __forceinline__ void tile_dot<Q8_0, 2>(const uint8_t *rg, const uint8_t *rg8, const BFrag<2> &B,
                                                  const BFrag<2> &, int t, float (&yg)[2], float (&yg8)[2], const ZQ &z) {
    tile_q8_0<2>(rg, rg8, B, t, yg, yg8, z);
}

// Q4_K / Q5_K: d @0, dmin @2, 12 bytes of 6-bit scales / mins @4 (GGUF
// K-quant packing).  The scale of sub-block s is folded into the codes:
// A = sc_s * q via one f16 FMA (exact, < 2^14); one chained accumulator per
// tile then holds sum_s sc_s sum(q x), times d.  The min term
// dmin * sum_s m_s * (sum of x over s) is one more MMA: A = the mins of the
// lane's sub-blocks 2t, 2t + 1, B = the sub-block sums of x (pieces).
struct KqRow {
    uint32_t sc[8];   // (sc_s, sc_s) as f16x2
    uint32_t nc[8];   // (-1024 sc_s, -1024 sc_s)
    uint32_t mn;      // (m_{2t}, m_{2t+1}) as f16x2
    float d, dmin;
};
__device__ __forceinline__ void kq_row(const uint8_t *rb, int t, KqRow &r) {
    const uint4 h = *reinterpret_cast<const uint4 *>(rb);
    r.d = f16_bits(h.x & 0xFFFFu);
    r.dmin = f16_bits(h.x >> 16);
    const uint32_t w0 = h.y, w1 = h.z, w2 = h.w;
    const uint32_t scA = w0 & 0x3F3F3F3Fu, mnA = w1 & 0x3F3F3F3Fu;
    const uint32_t scB = (w2 & 0x0F0F0F0Fu) | ((w0 >> 2) & 0x30303030u);
    const uint32_t mnB = ((w2 >> 4) & 0x0F0F0F0Fu) | ((w1 >> 2) & 0x30303030u);
#pragma unroll
    for (int s = 0; s < 8; ++s) {
        const uint32_t src = s < 4 ? scA : scB;
        const uint32_t k = (uint32_t)(s & 3);
        // bytes (sc_s, 0x64, sc_s, 0x64): (1024 + sc_s) in both halves
        const uint32_t m = __byte_perm(src, 0x64u, 0x4040u | k | (k << 8));
        r.sc[s] = hadd2(m, kM1024);
        r.nc[s] = hmul2(r.sc[s], kM1024);
    }
    const uint32_t msrc = t < 2 ? mnA : mnB;
    const uint32_t k0 = (uint32_t)(2 * (t & 1));
    r.mn = hadd2(__byte_perm(msrc, 0x64u, 0x4040u | k0 | ((k0 + 1) << 8)), kM1024);
}

template <int F, int NT>
__device__ __forceinline__ void tile_kq(const uint8_t *rg, const uint8_t *rg8, const BFrag<NT> &B,
                                        const BFrag<NT> &Bs, int t, float (&yg)[NT], float (&yg8)[NT], const ZQ &z) {
    KqRow R, R8;
    kq_row(rg, t, R);
    kq_row(rg8, t, R8);
    constexpr int QS = F == Q4_K ? 16 : 48;   // offset of qs
    float D[NT][4];
    zero(D);
#pragma unroll
    for (int p = 0; p < 4; ++p) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {   // kgroup half: elements l = 16h .. 16h + 15 of the sub-blocks
            const int o = QS + 32 * p + 16 * h + 4 * t;
            const uint32_t w = *reinterpret_cast<const uint32_t *>(rg + o);
            const uint32_t w8 = *reinterpret_cast<const uint32_t *>(rg8 + o);
            const uint32_t s = w >> 8, s8 = w8 >> 8;
            uint32_t l0 = nib_lo(w), l1 = nib_lo(w8), l2 = nib_lo(s), l3 = nib_lo(s8);
            uint32_t h0 = nib_hi(w), h1 = nib_hi(w8), h2 = nib_hi(s), h3 = nib_hi(s8);
            if constexpr (F == Q5_K) {
                // bit s of qh[l] is bit 4 of element l of sub-block s (bit 8 of the 16 q form)
                const int qo = 16 + 16 * h + 4 * t;
                const uint32_t qh = *reinterpret_cast<const uint32_t *>(rg + qo);
                const uint32_t qh8 = *reinterpret_cast<const uint32_t *>(rg8 + qo);
                const uint32_t q2 = qh >> 8, q28 = qh8 >> 8;
                auto lb = [&](uint32_t v) { return ((v >> (2 * p)) << 4) & 0x00100010u; };
                auto hb = [&](uint32_t v) { return ((v >> (2 * p + 1)) << 8) & 0x01000100u; };
                l0 |= lb(qh);
                l1 |= lb(qh8);
                l2 |= lb(q2);
                l3 |= lb(q28);
                h0 |= hb(qh);
                h1 |= hb(qh8);
                h2 |= hb(q2);
                h3 |= hb(q28);
            }
            const int sl = 2 * p, sh = 2 * p + 1;
            const uint32_t al0 = hfma2(l0, R.sc[sl], R.nc[sl]), al1 = hfma2(l1, R8.sc[sl], R8.nc[sl]);
            const uint32_t al2 = hfma2(l2, R.sc[sl], R.nc[sl]), al3 = hfma2(l3, R8.sc[sl], R8.nc[sl]);
            const uint32_t ah0 = hfma2(h0, R.sc[sh], R.nc[sh]), ah1 = hfma2(h1, R8.sc[sh], R8.nc[sh]);
            const uint32_t ah2 = hfma2(h2, R.sc[sh], R.nc[sh]), ah3 = hfma2(h3, R8.sc[sh], R8.nc[sh]);
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                mma(D[j], al0, al1, al2, al3, B(j, 4 * p + h));        // sub-block 2p: kgroups 4p, 4p + 1
                mma(D[j], ah0, ah1, ah2, ah3, B(j, 4 * p + 2 + h));    // sub-block 2p + 1: kgroups 4p + 2, 4p + 3
            }
        }
    }
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        float Dm[4];
        mma_z(Dm, R.mn, R8.mn, 0u, 0u, make_uint2(Bs.word(j), 0u), z);
        yg[j] = fmaf(R.d, D[j][0] + D[j][1], fmaf(-32.f * R.dmin, Dm[0] + Dm[1], yg[j]));
        yg8[j] = fmaf(R8.d, D[j][2] + D[j][3], fmaf(-32.f * R8.dmin, Dm[2] + Dm[3], yg8[j]));
    }
}
template <>
__device__ __forceinline__ void tile_dot<Q4_K, 1>(const uint8_t *rg, const uint8_t *rg8, const BFrag<1> &B,
                                                  const BFrag<1> &Bs, int t, float (&yg)[1], float (&yg8)[1], const ZQ &z) {
    tile_kq<Q4_K, 1>(rg, rg8, B, Bs, t, yg, yg8, z);
}
template <>
__device__ __forceinline__ void tile_dot<Q4_K, 2>(const uint8_t *rg, const uint8_t *rg8, const BFrag<2> &B,
                                                  const BFrag<2> &Bs, int t, float (&yg)[2], float (&yg8)[2], const ZQ &z) {
    tile_kq<Q4_K, 2>(rg, rg8, B, Bs, t, yg, yg8, z);
}
template <>
__device__ __forceinline__ void tile_dot<Q5_K, 1>(const uint8_t *rg, const uint8_t *rg8, const BFrag<1> &B,
                                                  const BFrag<1> &Bs, int t, float (&yg)[1], float (&yg8)[1], const ZQ &z) {
    tile_kq<Q5_K, 1>(rg, rg8, B, Bs, t, yg, yg8, z);
}
template <>
__device__ __forceinline__ void tile_dot<Q5_K, 2>(const uint8_t *rg, const uint8_t *rg8, const BFrag<2> &B,
                                                  const BFrag<2> &Bs, int t, float (&yg)[2], float (&yg8)[2], const ZQ &z) {
    tile_kq<Q5_K, 2>(rg, rg8, B, Bs, t, yg, yg8, z);
}

// ---------------------------------------------------------------------------
// The kernel.
// ---------------------------------------------------------------------------
struct TcArgs {
    const void *X;
    float *Y;
    const uint8_t *W;      // for the L2 prefetch
    int64_t M;
    int K;
    int N;
    int S;                 // ring slots per warp
    int owner;             // 1: warps own whole 16-row groups; 0: warps split K
    int xpitch;            // bytes per X piece array (2K + 32)
    int spitch;            // bytes per sub-block-sum piece array
    int off_x, off_s, off_scale, off_part, off_bar, off_flag;   // shared-memory offsets
    uint32_t prefetch;     // L2 prefetch budget per CTA (bytes)
    unsigned *status;
    uint64_t limit;
    AmaxOut amax;          // argmax mode when amax.keys is set: no output is stored
};

__device__ __forceinline__ bool tc_wait(volatile unsigned *abort_flag, uint64_t *bar, uint32_t parity,
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

__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// binary16 bits of v, round to nearest even
__device__ __forceinline__ uint32_t h16(float v) { return (uint32_t)__half_as_ushort(__float2half_rn(v)); }

template <int F, int NT, bool XBF16>
__global__ void __launch_bounds__(512, 1) gemv_tc_kernel(const __grid_constant__ CUtensorMap wmap,
                                                          const __grid_constant__ TcArgs a) {
    extern __shared__ __align__(1024) uint8_t sm[];
    constexpr int UB = TcUnit<F>::B;
    constexpr int TILE = kTR * UB;
    constexpr bool KQ = F == Q4_K || F == Q5_K;
    const int nw = blockDim.x >> 5, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int S = a.S, N = a.N, K = a.K;
    const int U = K >> 8;
    const int64_t RG = (a.M + kTR - 1) / kTR;
    const int64_t rg0 = (int64_t)blockIdx.x * RG / gridDim.x, rg1 = (int64_t)(blockIdx.x + 1) * RG / gridDim.x;
    const int nrg = (int)(rg1 - rg0);
    const bool owner = a.owner != 0;   // warps own whole row groups; else they split K
    // this warp's tiles: owner: groups warp, warp + nw, ... (all units each);
    // split: flat index tau = warp + nw * j over (group, unit)
    const int ntiles = owner ? ((nrg - warp + nw - 1) / nw) * U : (nrg * U - warp + nw - 1) / nw;
    // (group, unit) of this warp's tile j, advanced one step at a time
    struct Pos {
        int rgl, u;
    };
    auto pos0 = [&]() -> Pos { return owner ? Pos{warp, 0} : Pos{warp / U, warp % U}; };
    auto step = [&](Pos &q) {
        if (owner) {
            if (++q.u == U) {
                q.u = 0;
                q.rgl += nw;
            }
        } else {
            q.u += nw;
            while (q.u >= U) {
                q.u -= U;
                ++q.rgl;
            }
        }
    };

    uint8_t *slots = sm;
    uint8_t *xp = sm + a.off_x;
    uint8_t *xsums = sm + a.off_s;
    float *xscale = reinterpret_cast<float *>(sm + a.off_scale);
    float *part = reinterpret_cast<float *>(sm + a.off_part);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + a.off_bar);
    volatile unsigned *abort_flag = reinterpret_cast<volatile unsigned *>(sm + a.off_flag);
    unsigned *smax = reinterpret_cast<unsigned *>(sm + a.off_flag + 16);   // per-token max |x| bits
    unsigned long long *skey = reinterpret_cast<unsigned long long *>(sm + a.off_flag + 48);   // argmax keys
    const bool amax = a.amax.keys != nullptr;

    if (threadIdx.x == 0) {
        for (int i = 0; i < nw * S; ++i) mbar_init(&bars[i], 1);
        *abort_flag = 0u;
        fence_barrier_init();
    }
    if (threadIdx.x < 8) {
        smax[threadIdx.x] = 0u;
        skey[threadIdx.x] = 0ull;
    }
    if (threadIdx.x == 32) {
        prefetch_tensormap(&wmap);
        // the CTA's rows are one contiguous byte range of W: let L2 fetch it now
        const int64_t rb = (int64_t)U * UB;
        const int64_t r0 = rg0 * kTR, r1 = rg1 * kTR < a.M ? rg1 * kTR : a.M;
        int64_t bytes = (r1 - r0) * rb;
        if (bytes > (int64_t)a.prefetch) bytes = a.prefetch;
        const uint8_t *p = a.W + r0 * rb;
        for (int64_t o = 0; o < bytes; o += 65536) {
            const int64_t n = bytes - o < 65536 ? bytes - o : 65536;
            prefetch_l2(p + o, (uint32_t)n);
        }
    }
    __syncthreads();
    pdl_launch_dependents();

    Pos ip = pos0();   // next tile to copy
    int islot = 0;
    auto issue = [&]() {
        const int slot = warp * S + islot;
        islot = islot + 1 == S ? 0 : islot + 1;
        mbar_arrive_expect_tx(&bars[slot], (uint32_t)TILE);
        tma_load_2d(slots + (size_t)slot * TILE, &wmap, &bars[slot], (ip.u * UB) >> 1, (int)((rg0 + ip.rgl) * kTR));
        step(ip);
    };
    if (lane == 0)
        for (int j = 0; j < S && j < ntiles; ++j) issue();

    pdl_wait();   // X and Y are ordered behind the preceding grid

    // ---- X pieces: per token n, scale 2^-e_n with max |x| 2^-e_n in [2^14, 2^15) ----
    const int K4 = K >> 2;
    auto ld4 = [&](int n, int c) -> float4 {
        if constexpr (XBF16) {
            const uint2 b = reinterpret_cast<const uint2 *>(a.X)[(int64_t)n * K4 + c];
            return make_float4(__uint_as_float(b.x << 16), __uint_as_float(b.x & 0xFFFF0000u),
                               __uint_as_float(b.y << 16), __uint_as_float(b.y & 0xFFFF0000u));
        } else {
            return reinterpret_cast<const float4 *>(a.X)[(int64_t)n * K4 + c];
        }
    };
    for (int n = 0; n < N; ++n) {
        float m = 0.f;
        for (int c = threadIdx.x; c < K4; c += blockDim.x) {
            const float4 v = ld4(n, c);
            m = fmaxf(m, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) atomicMax(&smax[n], __float_as_uint(m));
    }
    __syncthreads();
    if (threadIdx.x < N) {
        const uint32_t mb = smax[threadIdx.x];
        int e = 0;
        if (mb != 0u && mb < 0x7F800000u) e = (int)((mb >> 23) & 0xFFu) - 127 - 14;   // max 2^-e < 2^15
        if (e < -100) e = -100;
        if (e > 100) e = 100;
        xscale[2 * threadIdx.x] = __uint_as_float((uint32_t)(127 - e) << 23);       // 2^-e
        xscale[2 * threadIdx.x + 1] = __uint_as_float((uint32_t)(127 + e) << 23);   // 2^e
    }
    __syncthreads();
    // hi = f16(x 2^-e), lo = f16(x 2^-e - hi); each group of 4 elements is
    // stored in slot order 0, 2, 1, 3 (the lane's b0 = elements 0, 2 and
    // b1 = elements 1, 3 of its quad are then one 8-byte word)
    for (int i = threadIdx.x; i < N * K4; i += blockDim.x) {
        const int n = i / K4, c = i - n * K4;
        float4 v = ld4(n, c);
        float sc = xscale[2 * n];
        if (x16_elem<F>((4 * c) & 255)) sc *= 0.0625f;
        v.x *= sc;
        v.y *= sc;
        v.z *= sc;
        v.w *= sc;
        const __half2 h02 = __floats2half2_rn(v.x, v.z), h13 = __floats2half2_rn(v.y, v.w);
        const float2 f02 = __half22float2(h02), f13 = __half22float2(h13);
        const __half2 l02 = __floats2half2_rn(v.x - f02.x, v.z - f02.y);
        const __half2 l13 = __floats2half2_rn(v.y - f13.x, v.w - f13.y);
        *reinterpret_cast<uint2 *>(xp + (size_t)(2 * n) * a.xpitch + 8 * c) =
            make_uint2(*reinterpret_cast<const uint32_t *>(&h02), *reinterpret_cast<const uint32_t *>(&h13));
        *reinterpret_cast<uint2 *>(xp + (size_t)(2 * n + 1) * a.xpitch + 8 * c) =
            make_uint2(*reinterpret_cast<const uint32_t *>(&l02), *reinterpret_cast<const uint32_t *>(&l13));
    }
    if constexpr (KQ) {
        // sub-block sums of x 2^-e, times 2^-5 (so that they stay below 2^15)
        const int nsb = K >> 5;
        for (int i = threadIdx.x; i < N * nsb; i += blockDim.x) {
            const int n = i / nsb, sb = i - n * nsb;
            float acc = 0.f;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const float4 v = ld4(n, 8 * sb + c);
                acc += (v.x + v.y) + (v.z + v.w);
            }
            acc *= xscale[2 * n] * 0.03125f;
            const uint32_t hi = h16(acc);
            const uint32_t lo = h16(acc - __half2float(__ushort_as_half((unsigned short)hi)));
            *reinterpret_cast<uint16_t *>(xsums + (size_t)(2 * n) * a.spitch + 2 * sb) = (uint16_t)hi;
            *reinterpret_cast<uint16_t *>(xsums + (size_t)(2 * n + 1) * a.spitch + 2 * sb) = (uint16_t)lo;
        }
    }
    __syncthreads();

    // ---- tiles ----
    float yg[NT], yg8[NT];
#pragma unroll
    for (int j = 0; j < NT; ++j) yg[j] = yg8[j] = 0.f;
    int cur = -1;   // row group (local) of the accumulators
    auto flush = [&](int rgl) {
        if (rgl < 0) return;
        if (owner) {
            const int64_t r = (rg0 + rgl) * kTR + g;
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                const int n = 4 * j + t;
                if (n < N) {
                    const float sc = xscale[2 * n + 1];
                    if (amax) {
                        unsigned long long b = 0ull;
                        if (r < a.M) amax_fold(b, yg[j] * sc, (int)r);
                        if (r + 8 < a.M) amax_fold(b, yg8[j] * sc, (int)(r + 8));
                        if (b) atomicMax(&skey[n], b);
                    } else {
                        if (r < a.M) a.Y[(int64_t)n * a.M + r] = yg[j] * sc;
                        if (r + 8 < a.M) a.Y[(int64_t)n * a.M + r + 8] = yg8[j] * sc;
                    }
                }
            }
        } else {
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                const int n = 4 * j + t;
                if (n < N) {
                    float *pp = part + (((size_t)rgl * nw + warp) * kTR) * 8 + n;
                    pp[g * 8] = yg[j];
                    pp[(g + 8) * 8] = yg8[j];
                }
            }
        }
#pragma unroll
        for (int j = 0; j < NT; ++j) yg[j] = yg8[j] = 0.f;
    };
    const ZQ z = zq();
    // the lane's B columns (a column past 2N reads column col % 2N again)
    const uint8_t *xcol[NT];
    const uint8_t *scol[NT];
#pragma unroll
    for (int jj = 0; jj < NT; ++jj) {
        const int col = (8 * jj + g) % (2 * N);   // token col / 2, piece col % 2
        xcol[jj] = xp + (size_t)col * a.xpitch + 8 * t;
        scol[jj] = xsums + (size_t)col * a.spitch + 4 * t;   // sub-block sums 2t, 2t + 1
    }
    int done = 0;
    Pos cp = pos0();   // tile being computed
    int cslot = 0, cpar = 0;
    for (int j = 0; j < ntiles; ++j) {
        if (cp.rgl != cur) {
            flush(cur);
            cur = cp.rgl;
        }
        const int slot = warp * S + cslot;
        if (!tc_wait(abort_flag, &bars[slot], (uint32_t)cpar, a.limit)) break;
        const uint8_t *tb = slots + (size_t)slot * TILE;
        BFrag<NT> B, Bs;
#pragma unroll
        for (int jj = 0; jj < NT; ++jj) {
            B.p[jj] = xcol[jj] + cp.u * 512;
            Bs.p[jj] = scol[jj] + cp.u * 16;
        }
        tile_dot<F, NT>(tb + g * UB, tb + (g + 8) * UB, B, Bs, t, yg, yg8, z);
        __syncwarp();
        if (lane == 0 && j + S < ntiles) issue();   // every lane is done with the slot
        done = j + 1;
        step(cp);
        if (++cslot == S) {
            cslot = 0;
            cpar ^= 1;
        }
    }
    if (done == ntiles) flush(cur);
    // copies still in flight (only after an abort): wait for them before exit
    if (lane == 0) {
        const int issued = ntiles < done + S ? ntiles : done + S;
        for (int j = done; j < issued; ++j)
            (void)mbar_wait(&bars[warp * S + j % S], (uint32_t)(j / S) & 1u,
                            a.limit < (1ull << 31) ? (1ull << 31) : a.limit);
    }
    __syncthreads();
    if (*abort_flag) {
        if (threadIdx.x == 0) report_status(a.status, kStatusTimeout);
        return;
    }
    if (!owner) {
        // partial sums of every warp, in warp order
        for (int i = threadIdx.x; i < nrg * kTR * N; i += blockDim.x) {
            const int n = i % N, rr = (i / N) % kTR, rgl = i / (N * kTR);
            const int64_t r = (rg0 + rgl) * kTR + rr;
            if (r >= a.M) continue;
            float v = 0.f;
            for (int w = 0; w < nw; ++w) {
                // warps that got no tile of this group wrote nothing: skip them
                const int first = (rgl * U - w + nw - 1) / nw;   // first j of warp w in the group
                const int tau = w + nw * first;
                if (tau >= (rgl + 1) * U) continue;
                v += part[(((size_t)rgl * nw + w) * kTR + rr) * 8 + n];
            }
            if (amax)
                atomicMax(&skey[n], amax_key(v * xscale[2 * n + 1], (int)r));
            else
                a.Y[(int64_t)n * a.M + r] = v * xscale[2 * n + 1];
        }
    }
    if (amax) {
        __syncthreads();
        if ((int)threadIdx.x < N && skey[threadIdx.x]) {
            atomicMax(a.amax.keys + threadIdx.x, skey[threadIdx.x]);
            __threadfence();
        }
        amax_last_cta(a.amax, N);
    }
}

struct TcLayout {
    int off_x, off_s, off_scale, off_part, off_bar, off_flag, total, xpitch, spitch;
};
int tc_unit_bytes(int fmt) {
    switch (fmt) {
    case Q8_0: return TcUnit<Q8_0>::B;
    case Q4_0: return TcUnit<Q4_0>::B;
    case Q4_K: return TcUnit<Q4_K>::B;
    case Q5_K: return TcUnit<Q5_K>::B;
    default: return 0;
    }
}
TcLayout tc_layout(int fmt, int nw, int S, int64_t K, int N, int64_t nrg_min, int64_t nrg_max) {
    TcLayout L;
    const int tile = kTR * tc_unit_bytes(fmt);
    int64_t o = (int64_t)nw * S * tile;
    L.xpitch = (int)(2 * K + 32);
    L.off_x = (int)o;
    o += (int64_t)2 * N * L.xpitch;
    const bool kq = fmt == Q4_K || fmt == Q5_K;
    L.spitch = (int)((K / 32) * 2 + 32);
    L.off_s = (int)o;
    o += kq ? (int64_t)2 * N * L.spitch : 0;
    o = (o + 15) / 16 * 16;
    L.off_scale = (int)o;
    o += 64;
    L.off_part = (int)o;
    if (nrg_min < nw) o += nrg_max * nw * kTR * 8 * 4;   // K split: partial sums per (group, warp)
    o = (o + 15) / 16 * 16;
    L.off_bar = (int)o;
    o += (int64_t)nw * S * 8;
    L.off_flag = (int)o;
    o += 16 + 32 + 64;   // abort flag, per-token max |x|, argmax keys
    L.total = o > (1ll << 30) ? (1 << 30) : (int)o;
    return L;
}

constexpr int kTcSmemMax = 232448 - 1024;   // the opt-in maximum, less room for static shared words

template <int F, int NT, bool XBF16>
cudaError_t tc_launch_typed(const TcPlan &p, const CUtensorMap &wmap, const TcArgs &a, bool pdl, cudaStream_t st) {
    auto kern = gemv_tc_kernel<F, NT, XBF16>;
    static std::atomic<int> configured[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured[dev & 63].load() < p.smem) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmemMax);
        if (e != cudaSuccess) return e;
        configured[dev & 63].store(kTcSmemMax);
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
    e = cudaLaunchKernelEx(&cfg, kern, wmap, a);
    if (e != cudaSuccess) return e;
    return launched(cudaGetLastError());
}

template <int F>
cudaError_t tc_launch_fmt(const TcPlan &p, const CUtensorMap &wmap, const TcArgs &a, int xbf16, bool pdl,
                          cudaStream_t st) {
    if (a.N <= 4)
        return xbf16 ? tc_launch_typed<F, 1, true>(p, wmap, a, pdl, st) : tc_launch_typed<F, 1, false>(p, wmap, a, pdl, st);
    return xbf16 ? tc_launch_typed<F, 2, true>(p, wmap, a, pdl, st) : tc_launch_typed<F, 2, false>(p, wmap, a, pdl, st);
}

}  // namespace

int gemv_tc_unit_bytes(int fmt) { return tc_unit_bytes(fmt); }

bool plan_gemv_tc(int fmt, int64_t M, int64_t K, int N, int num_sms, int force_warps, TcPlan &p) {
    const int ub = tc_unit_bytes(fmt);
    if (!ub || N < 1 || N > 8 || K % 256 || M < 1 || num_sms < 1 || K > (1 << 15)) return false;
    const int64_t RG = (M + kTR - 1) / kTR;
    const int64_t grid = RG < num_sms ? RG : num_sms;
    const int64_t nrg_max = (RG + grid - 1) / grid, nrg_min = RG / grid;
    for (int nw : {16, 8, 4}) {
        if (force_warps && nw != force_warps) continue;
        for (int S : {6, 4, 3, 2}) {
            const TcLayout L = tc_layout(fmt, nw, S, K, N, nrg_min, nrg_max);
            if (L.total <= kTcSmemMax) {
                p.grid = (int)grid;
                p.warps = nw;
                p.S = S;
                p.smem = L.total;
                return true;
            }
        }
    }
    return false;
}

cudaError_t launch_gemv_tc(int fmt, const TcPlan &p, const CUtensorMap &wmap, const uint8_t *W, int64_t M, int64_t K,
                           const void *X, int xbf16, int N, float *Y, bool pdl, unsigned *status, uint64_t limit,
                           cudaStream_t st, unsigned long long *amax_ws, int32_t *idx, float *val) {
    const int64_t RG = (M + kTR - 1) / kTR;
    const int64_t nrg_max = (RG + p.grid - 1) / p.grid, nrg_min = RG / p.grid;
    const TcLayout L = tc_layout(fmt, p.warps, p.S, K, N, nrg_min, nrg_max);
    if (L.total > p.smem) return cudaErrorInvalidValue;
    TcArgs a;
    a.X = X;
    a.Y = Y;
    a.W = W;
    a.M = M;
    a.K = (int)K;
    a.N = N;
    a.S = p.S;
    a.xpitch = L.xpitch;
    a.spitch = L.spitch;
    a.off_x = L.off_x;
    a.off_s = L.off_s;
    a.off_scale = L.off_scale;
    a.off_part = L.off_part;
    a.off_bar = L.off_bar;
    a.off_flag = L.off_flag;
    a.prefetch = 512u << 10;
    a.owner = RG / p.grid >= p.warps ? 1 : 0;   // every CTA has at least `warps` groups
    a.status = status;
    a.limit = limit;
    a.amax = AmaxOut{amax_ws, amax_ws ? reinterpret_cast<unsigned *>(amax_ws + N) : nullptr, idx, val};
    switch (fmt) {
    case Q8_0: return tc_launch_fmt<Q8_0>(p, wmap, a, xbf16, pdl, st);
    case Q4_0: return tc_launch_fmt<Q4_0>(p, wmap, a, xbf16, pdl, st);
    case Q4_K: return tc_launch_fmt<Q4_K>(p, wmap, a, xbf16, pdl, st);
    case Q5_K: return tc_launch_fmt<Q5_K>(p, wmap, a, xbf16, pdl, st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace qmm
