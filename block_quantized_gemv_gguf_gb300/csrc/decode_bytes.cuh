// decode_bytes.cuh -- block decoders that read the raw block bytes one byte at
// a time (valid for any alignment).  One "unit" is 32 consecutive weights of
// a row: a whole Q8_0 / Q4_0 block, or one 32-weight sub-block of a Q4_K /
// Q6_K super-block.  Every weight is produced as the exact dequantized value
// rounded once to f32:
//   Q8_0  w = d * q                       (exact)
//   Q4_0  w = (nibble - 8) * d            (exact)
//   Q4_K  w = fma(d*sc, q, -(dmin*m))     (d*sc, q, dmin*m exact; one rounding)
//   Q6_K  w = (d*scale) * (q - 32)        (exact, < 24 significant bits)
//   Q5_K  w = fma(d*sc, q, -(dmin*m))     (as Q4_K, q = nibble | qh bit << 4)
#pragma once

#include "common.cuh"

namespace qmm {

__device__ __forceinline__ uint32_t ldb(const uint8_t *p) { return (uint32_t)__ldg(p); }
__device__ __forceinline__ uint32_t ld16(const uint8_t *p) { return ldb(p) | (ldb(p + 1) << 8); }

// Q4_K six-bit (scale, min) of sub-block s, GGUF packing of the 12 bytes S.
__device__ __forceinline__ void q4k_scale_min_bytes(const uint8_t *S, int s, int &sc, int &mn) {
    if (s < 4) {
        sc = (int)(ldb(S + s) & 63u);
        mn = (int)(ldb(S + s + 4) & 63u);
    } else {
        sc = (int)((ldb(S + s + 4) & 15u) | ((ldb(S + s - 4) >> 6) << 4));
        mn = (int)((ldb(S + s + 4) >> 4) | ((ldb(S + s) >> 6) << 4));
    }
}

// Decode unit u (32 weights) of the row starting at `row`.
template <int F>
__device__ __forceinline__ void decode_unit(const uint8_t *row, int64_t u, float (&w)[32]) {
    if constexpr (F == Q8_0) {
        const uint8_t *b = row + u * 34;
        const float d = f16_bits(ld16(b));
#pragma unroll
        for (int e = 0; e < 32; ++e) w[e] = d * (float)(int8_t)ldb(b + 2 + e);
    } else if constexpr (F == Q4_0) {
        const uint8_t *b = row + u * 18;
        const float d = f16_bits(ld16(b));
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const uint32_t v = ldb(b + 2 + e);
            w[e] = (float)((int)(v & 15u) - 8) * d;
            w[e + 16] = (float)((int)(v >> 4) - 8) * d;
        }
    } else if constexpr (F == Q4_K) {
        const uint8_t *b = row + (u >> 3) * 144;
        const int s = (int)(u & 7);
        const float d = f16_bits(ld16(b));
        const float dmin = f16_bits(ld16(b + 2));
        int sc, mn;
        q4k_scale_min_bytes(b + 4, s, sc, mn);
        const float dsc = d * (float)sc;
        const float dmn = dmin * (float)mn;
        const uint8_t *qs = b + 16 + (s >> 1) * 32;
        const int shift = (s & 1) * 4;
#pragma unroll
        for (int l = 0; l < 32; ++l) {
            const float q = (float)((ldb(qs + l) >> shift) & 15u);
            w[l] = __fmaf_rn(dsc, q, -dmn);
        }
    } else if constexpr (F == Q5_K) {
        const uint8_t *b = row + (u >> 3) * 176;
        const int s = (int)(u & 7);
        const float d = f16_bits(ld16(b));
        const float dmin = f16_bits(ld16(b + 2));
        int sc, mn;
        q4k_scale_min_bytes(b + 4, s, sc, mn);
        const float dsc = d * (float)sc;
        const float dmn = dmin * (float)mn;
        const uint8_t *qh = b + 16;
        const uint8_t *qs = b + 48 + (s >> 1) * 32;
        const int shift = (s & 1) * 4;
#pragma unroll
        for (int l = 0; l < 32; ++l) {
            const float q = (float)(((ldb(qs + l) >> shift) & 15u) | (((ldb(qh + l) >> s) & 1u) << 4));
            w[l] = __fmaf_rn(dsc, q, -dmn);
        }
    } else {  // Q6_K
        const uint8_t *b = row + (u >> 3) * 210;
        const int s = (int)(u & 7);          // e = 32 s + l = 128 h + 32 J + l
        const int h = s >> 2, J = s & 3;
        const float d = f16_bits(ld16(b + 208));
        const uint8_t *ql = b + 64 * h + 32 * (J & 1);
        const uint8_t *qh = b + 128 + 32 * h;
        const int lshift = (J >> 1) * 4, hshift = 2 * J;
        const float ds0 = d * (float)(int8_t)ldb(b + 192 + 2 * s);
        const float ds1 = d * (float)(int8_t)ldb(b + 192 + 2 * s + 1);
#pragma unroll
        for (int l = 0; l < 32; ++l) {
            const int q = (int)(((ldb(ql + l) >> lshift) & 15u) | (((ldb(qh + l) >> hshift) & 3u) << 4));
            w[l] = (l < 16 ? ds0 : ds1) * (float)(q - 32);
        }
    }
}

}  // namespace qmm
