// gemv_i8.cuh -- integer tensor-core GEMV, 1 <= N <= 16, for 16-byte aligned
// weights (instantiated by gemv_i8_exact.cu and gemv_i8_q8.cu):
//
//     Y[n, m] = sum_k x(n, k) * w(m, k)
//
// A = the weights' integer codes as 8-bit MMA operands, taken straight from
// the block bytes with masks (Q4_0 and Q4_K: nibbles, u8; Q6_K: low nibble
// | two high bits, u8; Q8_0: the code bytes themselves, s8).  One
// mma.sync m16n8k32 covers a 16-row x 32-weight tile, i.e. one 32-weight
// block of 16 rows, with exact int32 accumulation.  B = X as int8 digits:
//   * XM_EXACT: per 32-element block of a token, E = the binary exponent of
//     the block's largest |x| and T = rint(x * 2^(29-E)) (|T| < 2^30: x to
//     within 2^-30 of the block's max |x|), written as four balanced
//     base-256 digits, one MMA column each (digit j weighs 2^-8j), and the
//     block scale 2^(E-5).  The integer part of the sum is exact, so the
//     result is the f32 GEMV's up to f32 rounding of the per-block scaling.
//   * XM_Q8: X already quantized to Q8_0 activations (the quantizer of
//     "cera 0.5.2 src/backend/cpu.rs", quantize_f32_to_q8_0_scalar): one
//     digit, the code; the block scale is the quantizer's binary16 d.  This
//     is the pages' int8 decode arithmetic, sum_b d_w d_x sum(q_w q_x).
// The weight offset (Q4_0: 8, Q6_K: 32) and the int->float conversion ride
// in the MMA's accumulator input: C = 0x4B400000 - offset * (sum of the
// column's digits over the block), so D read as f32 is 1.5 * 2^23 +
// sum((q - offset) * digit) exactly (the sum stays below 2^22 in
// magnitude), and one f32x2 subtraction gives it as a float.
// Q6_K scales every 16 weights: its MMA columns come in pairs per digit, the
// first holding the digits of elements 0..15 (zeros for 16..31), the second
// those of 16..31.  Q4_K's min term is dmin * m_s times the sum of the
// represented x over the sub-block, added per token.
//
// CTA = CW compute warps (RG groups of 16 rows each) + 1 TMA warp.  The TMA
// warp streams the tile's weight bytes, 256 weights per chunk, through a
// ring of stages (2-D tensor map, 240/272/144-byte row windows) and, after
// the preceding kernel on the stream has finished, copies the CTA's K slice
// of X (raw values, or codes and scales) once.  The compute warps turn that
// slice into B fragments, accumulator inputs and block scales held in shared
// memory for the whole K slice, then run the chunks.  Small-M shapes split K
// over a thread-block cluster; partial sums meet in distributed shared
// memory (fixed order, no atomics).
#pragma once

#include "gemv_shared.cuh"

namespace qmm {
namespace {

constexpr int XM_EXACT = 0;
constexpr int XM_Q8 = 1;
constexpr int I8_MAGIC = 0x4B400000;          // f32 bits of 1.5 * 2^23
constexpr float I8_MAGIC_F = 12582912.0f;
constexpr uint32_t M4 = 0x0F0F0F0Fu;

// Weight offset folded into the accumulator input.
template <int F> struct I8Off { static constexpr int v = 0; };
template <> struct I8Off<Q4_0> { static constexpr int v = 8; };
template <> struct I8Off<Q6_K> { static constexpr int v = 32; };

template <int F, int MODE, int NTOK, bool XBF16, int CW, int RG> struct GI {
    static constexpr int H = F == Q6_K ? 2 : 1;                 // column halves (Q6_K: 16-weight scales)
    static constexpr int D = MODE == XM_EXACT ? 4 : 1;          // digits per value
    static constexpr int P = D * H;                             // MMA columns per token
    static constexpr int NCOL = NTOK * P;
    static constexpr int NT = (NCOL + 7) / 8;                   // n8 tiles
    static constexpr int NT1 = (NTOK + 7) / 8;                  // tiles of the one-column-per-token layout
    static constexpr bool FOLD = NTOK == 1;                     // X block scale folded into the row scales
    static constexpr bool CI = I8Off<F>::v != 0;                // per-column accumulator inputs
    static constexpr int ROWS = 16 * CW * RG;
    static constexpr int WARP_TMA = CW;
    static constexpr int THREADS = (CW + 1) * 32;
    static constexpr int WIN = GWin<F>::bytes;
    static constexpr int STAGE = ROWS * WIN;
    static constexpr int S = CW * RG >= 8 ? 2 : 3;
    static constexpr int XES = MODE == XM_Q8 ? 1 : (XBF16 ? 2 : 4);
    // shared bytes per 256-weight chunk of the K slice
    static constexpr int RAW_C = NTOK * 256 * XES + (MODE == XM_Q8 ? NTOK * 32 : 0);
    // stored B columns per tile: all 8, or (one tile, fewer used columns)
    // the used ones rounded up to a power of two; lanes of the other columns
    // read a stored column's fragment again and their results are dropped
    static constexpr int NCW = NT > 1 ? 8 : (NCOL > 4 ? 8 : (NCOL > 2 ? 4 : (NCOL > 1 ? 2 : 1)));
    static constexpr int FRAG_C = 8 * NT * NCW * 32;
    static constexpr int CI_C = CI ? 8 * NT * 64 : 0;
    static constexpr int XS_C = FOLD ? 8 * 4 : 8 * NT * 32;
    static constexpr int SX_C = kmin_fmt(F) ? 8 * 16 * 4 : 0;
    static constexpr int PER_C = RAW_C + FRAG_C + CI_C + XS_C + SX_C;
    static constexpr int rup(int v, int a) { return (v + a - 1) / a * a; }
    // fixed areas first; the X areas after them are sized at launch for the
    // K slice (c chunks), so short slices keep a small footprint
    static constexpr int OFF_STAGE = 0;
    static constexpr int OFF_SCT = S * STAGE;
    static constexpr int OFF_SCR = OFF_SCT + ROWS * SCW * 4;    // per-warp scratch of the final transform
    static constexpr int OFF_BAR = OFF_SCR + CW * 16 * 8 * 4;
    static constexpr int OFF_MISC = OFF_BAR + (2 * S + 1) * 8;
    static constexpr int OFF_X = rup(OFF_MISC + 16, 128);      // staged X; the reduction buffer afterwards
    static constexpr int SMEM_LIMIT = 232448 - 512;          // room for the kernel's static shared words
    __host__ __device__ static constexpr int rawb(int c) { return rup(c * RAW_C > ROWS * 64 ? c * RAW_C : ROWS * 64, 128); }
    __host__ __device__ static constexpr int off_frag(int c) { return OFF_X + rawb(c); }
    __host__ __device__ static constexpr int off_ci(int c) { return off_frag(c) + c * FRAG_C; }
    __host__ __device__ static constexpr int off_xs(int c) { return off_ci(c) + c * CI_C; }
    __host__ __device__ static constexpr int off_sx(int c) { return off_xs(c) + c * XS_C; }
    __host__ __device__ static constexpr int smem(int c) { return off_sx(c) + c * SX_C + 1024; }
    static constexpr int maxc_search() {
        int c = 1;
        while (smem(c + 1) <= SMEM_LIMIT) ++c;
        return c;
    }
    static constexpr int MAXC = maxc_search();
    // CTAs per SM at a typical slice of 8 chunks (at most 4): the register
    // budget the compiler may use without lowering that occupancy
    static constexpr int MINB = SMEM_LIMIT / smem(8) >= 4 ? 4 : (SMEM_LIMIT / smem(8) >= 1 ? SMEM_LIMIT / smem(8) : 1);
    static_assert(STAGE % 1024 == 0 && OFF_BAR % 8 == 0, "alignment");
    static_assert(smem(1) <= SMEM_LIMIT, "shared memory");
    static_assert(MODE == XM_Q8 || NCOL <= 16, "exact digits: at most two column tiles");
};

// X input of the kernel: raw X (XM_EXACT) or Q8_0 codes [N][K] and scales
// [N][K/32] (XM_Q8).
struct XIn {
    const void *x;
    const float *scales;
};

// d = A * B + C, m16n8k32, int8 operands, int32 accumulate; C = (c0, c1) for
// both row halves.
template <bool S8A>
__device__ __forceinline__ void imma(int (&d)[4], const uint32_t (&a)[4], uint2 b, int4 c) {
    if constexpr (S8A)
        asm volatile(
            "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%10,%11,%12,%13};"
            : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b.x), "r"(b.y), "r"(c.x), "r"(c.y), "r"(c.z),
              "r"(c.w));
    else
        asm volatile(
            "mma.sync.aligned.m16n8k32.row.col.s32.u8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%10,%11,%12,%13};"
            : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b.x), "r"(b.y), "r"(c.x), "r"(c.y), "r"(c.z),
              "r"(c.w));
}

// The integers the MMA summed for the thread's two columns of row g (D[0],
// D[1]) and row g + 8 (D[2], D[3]): (f32 bits of D) - 1.5 * 2^23, exactly.
__device__ __forceinline__ void unmagic(float2 &e, float2 &e8, const int (&d)[4]) {
    const float2 m = make_float2(-I8_MAGIC_F, -I8_MAGIC_F);
    e = __fadd2_rn(make_float2(__int_as_float(d[0]), __int_as_float(d[1])), m);
    e8 = __fadd2_rn(make_float2(__int_as_float(d[2]), __int_as_float(d[3])), m);
}

// 4x4 byte transpose: out[j] byte i = byte (3 - j) of u[i]  (digit j of
// element i when u[i] = T_i + 0x808080: digit 0 is the signed top byte,
// digits 1..3 are offset by 128).
__device__ __forceinline__ void digits4(uint32_t (&dw)[4], const uint32_t (&u)[4]) {
    const uint32_t t0 = __byte_perm(u[0], u[1], 0x5140u), t1 = __byte_perm(u[0], u[1], 0x7362u);
    const uint32_t t2 = __byte_perm(u[2], u[3], 0x5140u), t3 = __byte_perm(u[2], u[3], 0x7362u);
    dw[3] = __byte_perm(t0, t2, 0x5410u) ^ 0x80808080u;
    dw[2] = __byte_perm(t0, t2, 0x7632u) ^ 0x80808080u;
    dw[1] = __byte_perm(t1, t3, 0x5410u) ^ 0x80808080u;
    dw[0] = __byte_perm(t1, t3, 0x7632u);
}

__device__ __forceinline__ int sum_s8x4(uint32_t w) { return __dp4a((int)w, 0x01010101, 0); }

// ---------------------------------------------------------------------------
// X slice -> B fragments, accumulator inputs, block scales (and Q4_K's
// per-token block sums).  Work items (token n, block, group of 4 elements),
// 8 consecutive lanes per block; every lane runs every round (shuffles).
//   frag: uint32 [blk][tile][lane = 4 g + t][2]     (b0: k 4t.., b1: k 16+4t..)
//   ci:   int   [blk][tile][8]  C input of each column (offset formats)
//   xs:   FOLD: float [blk] block scale of token 0
//         else: float [blk][tile][8] block scale x digit weight of each column
//   sx:   Q4_K: float [blk][16] sum of the represented x of token n
// ---------------------------------------------------------------------------
template <int F, int MODE, int NTOK, bool XBF16, int CW, int RG>
__device__ __forceinline__ void prep_x_i8(const uint8_t *sraw, int kslice, int N, uint32_t *frag, int *ci, float *xs,
                                          float *sx, int tid) {
    using L = GI<F, MODE, NTOK, XBF16, CW, RG>;
    constexpr int NT = L::NT, H = L::H, D = L::D, NCW = L::NCW;
    const int nblk = kslice / 32;
    const int total = N * nblk * 8;
    for (int base = 0; base < total; base += CW * 32) {
        const int it = base + tid;
        const bool act = it < total;
        const int grp = it & 7, blk = (it >> 3) % nblk, n = (it >> 3) / nblk;
        uint32_t dw[D];
        float scale;
        if constexpr (MODE == XM_EXACT) {
            float v[4] = {0.f, 0.f, 0.f, 0.f};
            if (act) {
                const int e = n * kslice + blk * 32 + 4 * grp;
                if constexpr (XBF16) {
                    const uint2 r = *reinterpret_cast<const uint2 *>(sraw + 2 * e);
                    v[0] = __uint_as_float(r.x << 16);
                    v[1] = __uint_as_float(r.x & 0xFFFF0000u);
                    v[2] = __uint_as_float(r.y << 16);
                    v[3] = __uint_as_float(r.y & 0xFFFF0000u);
                } else {
                    const float4 r = *reinterpret_cast<const float4 *>(sraw + 4 * e);
                    v[0] = r.x;
                    v[1] = r.y;
                    v[2] = r.z;
                    v[3] = r.w;
                }
            }
            // largest |x| of the block as bits (NaN and inf sort above every finite value)
            uint32_t m = max(max(__float_as_uint(v[0]) & 0x7FFFFFFFu, __float_as_uint(v[1]) & 0x7FFFFFFFu),
                             max(__float_as_uint(v[2]) & 0x7FFFFFFFu, __float_as_uint(v[3]) & 0x7FFFFFFFu));
            m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
            m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
            m = max(m, __shfl_xor_sync(0xffffffffu, m, 4));
            const int E = (int)(m >> 23) - 127;
            const bool finite = m < 0x7F800000u;
            // blocks whose largest |x| is below 2^-98 (or zero) contribute 0;
            // a non-finite block contributes NaN
            const bool ok = finite && E >= -98;
            const float p = ok ? __uint_as_float((uint32_t)(29 - E + 127) << 23) : 0.f;
            uint32_t u[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) u[i] = (uint32_t)(__float2int_rn(v[i] * p) + 0x808080);
            uint32_t d4[4];
            digits4(d4, u);
#pragma unroll
            for (int j = 0; j < D; ++j) dw[j] = d4[j];
            scale = ok ? __uint_as_float((uint32_t)(E - 5 + 127) << 23) : (finite ? 0.f : __uint_as_float(0x7FC00000u));
        } else {
            const int nb_all = kslice / 32;
            dw[0] = act ? *reinterpret_cast<const uint32_t *>(sraw + n * kslice + blk * 32 + 4 * grp) : 0u;
            const float *ssc = reinterpret_cast<const float *>(sraw + N * kslice);
            scale = act ? ssc[n * nb_all + blk] : 0.f;
        }
        // digit sums over the block (H == 1) or over each half block (H == 2)
        int ds[D];
#pragma unroll
        for (int j = 0; j < D; ++j) {
            int s = sum_s8x4(dw[j]);
            s += __shfl_xor_sync(0xffffffffu, s, 1);
            s += __shfl_xor_sync(0xffffffffu, s, 2);
            if constexpr (H == 1) s += __shfl_xor_sync(0xffffffffu, s, 4);
            ds[j] = s;
        }
        float bsum = 0.f;   // Q4_K/Q5_K: sum of the represented x over the block
        if constexpr (kmin_fmt(F)) {
#pragma unroll
            for (int j = 0; j < D; ++j) bsum += __uint_as_float((uint32_t)(127 - 8 * j) << 23) * (float)ds[j];
            bsum *= scale;
        }
        if (act) {
            const int t = grp & 3, slot = grp >> 2, h = H == 2 ? (grp >> 2) : 0;
#pragma unroll
            for (int j = 0; j < D; ++j) {
                const int col = (n * D + j) * H + h;
                const int tile = col >> 3, gg = col & 7;
                frag[((blk * NT + tile) * 4 * NCW + 4 * gg + t) * 2 + slot] = dw[j];
                if constexpr (H == 2) {
                    const int col2 = (n * D + j) * 2 + (1 - h);
                    frag[((blk * NT + (col2 >> 3)) * 4 * NCW + 4 * (col2 & 7) + t) * 2 + slot] = 0u;
                }
                if (t == 0 && (H == 2 || slot == 0)) {      // one writer per column
                    if constexpr (L::CI) {
                        int *c4 = ci + ((blk * NT + tile) * 4 + (gg >> 1)) * 4 + (gg & 1);
                        c4[0] = c4[2] = I8_MAGIC - I8Off<F>::v * ds[j];
                    }
                    if constexpr (!L::FOLD)
                        xs[(blk * NT + tile) * 8 + gg] = scale * __uint_as_float((uint32_t)(127 - 8 * j) << 23);
                }
            }
            if (grp == 0) {
                if constexpr (L::FOLD) xs[blk] = scale;
                if constexpr (kmin_fmt(F)) sx[blk * 16 + n] = bsum;
            }
        }
    }
}

// Scale-table rows 16w..16w+15 of warp w (lane = (row, half)): the weights'
// per-block (Q4_0, Q8_0), per-sub-block (Q4_K: d*sc, then dmin*m) or
// per-16 (Q6_K: d*scales) factors; with FOLD, times the X block scale.
template <int F, bool FOLD>
__device__ __forceinline__ void prep_scales_i8(float *sct, const uint8_t *raw, int woff, int w, int lane,
                                               const float *xs8) {
    constexpr int WIN = GWin<F>::bytes;
    auto st4 = [&](int row, int e0, float a, float b, float c, float d) {
        *reinterpret_cast<float4 *>(sct + sct_index(row, e0)) = make_float4(a, b, c, d);
    };
    auto xf = [&](int b) { return FOLD ? xs8[b] : 1.f; };
    const int row = 16 * w + (lane >> 1), half = lane & 1;
    const uint8_t *rb = raw + row * WIN + woff;
    if constexpr (F == Q4_0 || F == Q8_0) {
        constexpr int BB = F == Q4_0 ? 18 : 34;
        const uint8_t *b = rb + BB * 4 * half;
        const int b0 = 4 * half;
        st4(row, b0, f16_bits(lds_u16(b)) * xf(b0), f16_bits(lds_u16(b + BB)) * xf(b0 + 1),
            f16_bits(lds_u16(b + 2 * BB)) * xf(b0 + 2), f16_bits(lds_u16(b + 3 * BB)) * xf(b0 + 3));
    } else if constexpr (kmin_fmt(F)) {   // Q4_K, Q5_K: same header fields
        const float d = f16_bits(lds_u16(rb)), dmin = f16_bits(lds_u16(rb + 2));
        const uint32_t w0 = ld32(rb + 4), w1 = ld32(rb + 8), w2 = ld32(rb + 12);
        // bytes: sc[0..3], mn[0..3], sc[4..7], mn[4..7] (GGUF 6-bit packing)
        const uint32_t sc = half ? ((w2 & 0x0F0F0F0Fu) | (((w0 >> 6) & 0x03030303u) << 4)) : (w0 & 0x3F3F3F3Fu);
        const uint32_t mn = half ? (((w2 >> 4) & 0x0F0F0F0Fu) | (((w1 >> 6) & 0x03030303u) << 4)) : (w1 & 0x3F3F3F3Fu);
        const int s0 = 4 * half;
        st4(row, s0, d * (float)(sc & 0xFFu) * xf(s0), d * (float)((sc >> 8) & 0xFFu) * xf(s0 + 1),
            d * (float)((sc >> 16) & 0xFFu) * xf(s0 + 2), d * (float)(sc >> 24) * xf(s0 + 3));
        st4(row, 8 + s0, dmin * (float)(mn & 0xFFu), dmin * (float)((mn >> 8) & 0xFFu),
            dmin * (float)((mn >> 16) & 0xFFu), dmin * (float)(mn >> 24));
    } else {  // Q6_K: d * scales[G], G = 0..15; the X block of G is G / 2
        const float d = f16_bits(lds_u16(rb + 208));
        const int8_t *sc = reinterpret_cast<const int8_t *>(rb + 192 + 8 * half);
        const int g0 = 8 * half;
        st4(row, g0, d * (float)sc[0] * xf(g0 / 2), d * (float)sc[1] * xf(g0 / 2), d * (float)sc[2] * xf(g0 / 2 + 1),
            d * (float)sc[3] * xf(g0 / 2 + 1));
        st4(row, g0 + 4, d * (float)sc[4] * xf(g0 / 2 + 2), d * (float)sc[5] * xf(g0 / 2 + 2),
            d * (float)sc[6] * xf(g0 / 2 + 3), d * (float)sc[7] * xf(g0 / 2 + 3));
    }
}

// Per-thread view of the X tables for one chunk: this lane's fragment, C
// inputs and column scales of block b, tile j.
template <int NT, int NCW = 8>
struct XView {
    const uint2 *frag;    // + (b * NT + j) * 4 * NCW
    const int4 *ci;       // + (b * NT + j) * 4: {c(2t), c(2t+1), c(2t), c(2t+1)}
    const float2 *xs;     // + (b * NT + j) * 4  (non-FOLD)
    __device__ __forceinline__ uint2 B(int b, int j) const { return frag[(b * NT + j) * 4 * NCW]; }
    __device__ __forceinline__ int4 C(int b, int j) const { return ci[(b * NT + j) * 4]; }
    __device__ __forceinline__ float2 X(int b, int j) const { return xs[(b * NT + j) * 4]; }
};

// One IMMA of block b (local to the chunk), tile j, and its epilogue into
// acc (slots: row g columns 2t, 2t+1; row g + 8 columns 2t, 2t+1).
//  * exact digits, H == 1: the thread's columns are digits j, j + 1 of one
//    token; they are combined (e_j + 2^-8 e_{j+1}) and scaled once per row,
//    into slot 0 / 2 (the digit weight of j is applied at the end);
//  * H == 2: the columns are the two halves of one (token, digit), each with
//    its own row scale (sh.x, sh.y), summed into slot 0 / 2;
//  * Q8_0 activations, H == 1: the columns are two tokens, each with its
//    own block scale, into all four slots.
// s, s8: row scales of rows g, g + 8 (H == 2: one per half).
template <int MODE, int H, bool S8A, bool CI, bool FOLD, int NT, int NCW>
__device__ __forceinline__ void imma_step(float (&acc)[4], const uint32_t (&a)[4], const XView<NT, NCW> &xv, int b,
                                          int j, float2 s, float2 s8) {
    int d[4];
    if constexpr (CI) {
        imma<S8A>(d, a, xv.B(b, j), xv.C(b, j));
    } else {
        imma<S8A>(d, a, xv.B(b, j), make_int4(I8_MAGIC, I8_MAGIC, I8_MAGIC, I8_MAGIC));
    }
    float2 e, e8;
    unmagic(e, e8, d);
    if constexpr (MODE == XM_EXACT && H == 1) {
        float sg = s.x, sg8 = s8.x;
        if constexpr (!FOLD) {
            const float x = xv.X(b, j).x;
            sg *= x;
            sg8 *= x;
        }
        acc[0] = fmaf(sg, fmaf(e.y, 0.00390625f, e.x), acc[0]);
        acc[2] = fmaf(sg8, fmaf(e8.y, 0.00390625f, e8.x), acc[2]);
    } else if constexpr (H == 2) {
        if constexpr (!FOLD) {
            const float x = xv.X(b, j).x;
            s.x *= x;
            s.y *= x;
            s8.x *= x;
            s8.y *= x;
        }
        acc[0] = fmaf(s.y, e.y, fmaf(s.x, e.x, acc[0]));
        acc[2] = fmaf(s8.y, e8.y, fmaf(s8.x, e8.x, acc[2]));
    } else {
        if constexpr (FOLD) {
            acc[0] = fmaf(s.x, e.x, acc[0]);
            acc[2] = fmaf(s8.x, e8.x, acc[2]);
        } else {
            const float2 x = xv.X(b, j);
            acc[0] = fmaf(s.x * x.x, e.x, acc[0]);
            acc[1] = fmaf(s.x * x.y, e.y, acc[1]);
            acc[2] = fmaf(s8.x * x.x, e8.x, acc[2]);
            acc[3] = fmaf(s8.x * x.y, e8.y, acc[3]);
        }
    }
}

// Chunk compute for one warp: rows g, g + 8 (row pointers rg, rg8 into the
// stage) x 256 weights.  sx: Q4_K block sums of this chunk, [b][16];
// mtok/mmsk: per slot, the token whose min term this thread adds and 1/0.
template <int F, int MODE, int NT, int NCW, bool FOLD, bool MIS>
__device__ __forceinline__ void compute_chunk_i8(float (&acc)[NT][4], const uint8_t *rg, const uint8_t *rg8,
                                                 const XView<NT, NCW> &xv, const float *sct, int r, const float *sx,
                                                 const int (&mtok)[NT][2], const float (&mmsk)[NT][2], int t) {
    constexpr bool CI = I8Off<F>::v != 0;
    if constexpr (F == Q4_0) {
        float sg[8], sg8[8];
        ld_scales<8>(sg, sct, r, 0);
        ld_scales<8>(sg8, sct, r + 8, 0);
#pragma unroll
        for (int bp = 0; bp < 4; ++bp) {            // blocks 2bp (codes at +2), 2bp+1 (codes at +20)
            const uint8_t *pg = rg + 36 * bp, *pg8 = rg8 + 36 * bp;
            const uint32_t qeg = __byte_perm(ld32(pg + 4 * t), ld32(pg + 4 * t + 4), 0x5432u);
            const uint32_t qeg8 = __byte_perm(ld32(pg8 + 4 * t), ld32(pg8 + 4 * t + 4), 0x5432u);
            const uint32_t qog = ld32(pg + 20 + 4 * t), qog8 = ld32(pg8 + 20 + 4 * t);
#pragma unroll
            for (int bb = 0; bb < 2; ++bb) {
                const int b = 2 * bp + bb;
                const uint32_t wg = bb ? qog : qeg, wg8 = bb ? qog8 : qeg8;
                // byte i of word t: element 4t+i (low nibble), 16+4t+i (high)
                const uint32_t a[4] = {wg & M4, wg8 & M4, (wg >> 4) & M4, (wg8 >> 4) & M4};
#pragma unroll
                for (int j = 0; j < NT; ++j) imma_step<MODE, 1, false, CI, FOLD, NT, NCW>(acc[j], a, xv, b, j, make_float2(sg[b], 0.f), make_float2(sg8[b], 0.f));
            }
        }
    } else if constexpr (F == Q8_0) {
        float sg[8], sg8[8];
        ld_scales<8>(sg, sct, r, 0);
        ld_scales<8>(sg8, sct, r + 8, 0);
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            // codes of block b at 34 b + 2: 4-aligned for odd b, 2 mod 4 for even b
            const uint8_t *pg = rg + 34 * b + 2, *pg8 = rg8 + 34 * b + 2;
            uint32_t a[4];
            if (b & 1) {
                a[0] = ld32(pg + 4 * t);
                a[1] = ld32(pg8 + 4 * t);
                a[2] = ld32(pg + 16 + 4 * t);
                a[3] = ld32(pg8 + 16 + 4 * t);
            } else {
                a[0] = ld32_off2(pg + 4 * t);
                a[1] = ld32_off2(pg8 + 4 * t);
                a[2] = ld32_off2(pg + 16 + 4 * t);
                a[3] = ld32_off2(pg8 + 16 + 4 * t);
            }
#pragma unroll
            for (int j = 0; j < NT; ++j) imma_step<MODE, 1, true, CI, FOLD, NT, NCW>(acc[j], a, xv, b, j, make_float2(sg[b], 0.f), make_float2(sg8[b], 0.f));
        }
    } else if constexpr (F == Q4_K) {
        float dsg[8], dsg8[8], dmg[8], dmg8[8];
        ld_scales<8>(dsg, sct, r, 0);
        ld_scales<8>(dsg8, sct, r + 8, 0);
        ld_scales<8>(dmg, sct, r, 8);
        ld_scales<8>(dmg8, sct, r + 8, 8);
        const uint8_t *qg = rg + 16, *qg8 = rg8 + 16;
#pragma unroll
        for (int pr = 0; pr < 4; ++pr) {            // sub-blocks 2pr (low nibbles), 2pr+1 (high)
            const uint32_t w0g = ld32(qg + 32 * pr + 4 * t), w1g = ld32(qg + 32 * pr + 16 + 4 * t);
            const uint32_t w0g8 = ld32(qg8 + 32 * pr + 4 * t), w1g8 = ld32(qg8 + 32 * pr + 16 + 4 * t);
#pragma unroll
            for (int hn = 0; hn < 2; ++hn) {
                const int s = 2 * pr + hn, sh = 4 * hn;
                const uint32_t a[4] = {(w0g >> sh) & M4, (w0g8 >> sh) & M4, (w1g >> sh) & M4, (w1g8 >> sh) & M4};
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    imma_step<MODE, 1, false, false, FOLD, NT, NCW>(acc[j], a, xv, s, j, make_float2(dsg[s], 0.f),
                                                                    make_float2(dsg8[s], 0.f));
                    // w = d sc q - dmin m  =>  - dmin m * (sum of x over the sub-block), once per
                    // token, on the slot of the token's first column
                    const float x0 = mmsk[j][0] != 0.f ? sx[s * 16 + mtok[j][0]] : 0.f;
                    acc[j][0] = fmaf(-dmg[s], x0, acc[j][0]);
                    acc[j][2] = fmaf(-dmg8[s], x0, acc[j][2]);
                    if constexpr (MODE == XM_Q8) {
                        const float x1 = mmsk[j][1] != 0.f ? sx[s * 16 + mtok[j][1]] : 0.f;
                        acc[j][1] = fmaf(-dmg[s], x1, acc[j][1]);
                        acc[j][3] = fmaf(-dmg8[s], x1, acc[j][3]);
                    }
                }
            }
        }
    } else if constexpr (F == Q5_K) {
        float dsg[8], dsg8[8], dmg[8], dmg8[8];
        ld_scales<8>(dsg, sct, r, 0);
        ld_scales<8>(dsg8, sct, r + 8, 0);
        ld_scales<8>(dmg, sct, r, 8);
        ld_scales<8>(dmg8, sct, r + 8, 8);
        const uint8_t *qg = rg + 48, *qg8 = rg8 + 48;
        // bit s of qh[l] is bit 4 of sub-block s's element l
        const uint32_t h0g = ld32(rg + 16 + 4 * t), h1g = ld32(rg + 32 + 4 * t);
        const uint32_t h0g8 = ld32(rg8 + 16 + 4 * t), h1g8 = ld32(rg8 + 32 + 4 * t);
#pragma unroll
        for (int pr = 0; pr < 4; ++pr) {            // sub-blocks 2pr (low nibbles), 2pr+1 (high)
            const uint32_t w0g = ld32(qg + 32 * pr + 4 * t), w1g = ld32(qg + 32 * pr + 16 + 4 * t);
            const uint32_t w0g8 = ld32(qg8 + 32 * pr + 4 * t), w1g8 = ld32(qg8 + 32 * pr + 16 + 4 * t);
#pragma unroll
            for (int hn = 0; hn < 2; ++hn) {
                const int s = 2 * pr + hn, sh = 4 * hn;
                const uint32_t a[4] = {((w0g >> sh) & M4) | (((h0g >> s) & 0x01010101u) << 4),
                                       ((w0g8 >> sh) & M4) | (((h0g8 >> s) & 0x01010101u) << 4),
                                       ((w1g >> sh) & M4) | (((h1g >> s) & 0x01010101u) << 4),
                                       ((w1g8 >> sh) & M4) | (((h1g8 >> s) & 0x01010101u) << 4)};
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    imma_step<MODE, 1, false, false, FOLD, NT, NCW>(acc[j], a, xv, s, j, make_float2(dsg[s], 0.f),
                                                                    make_float2(dsg8[s], 0.f));
                    const float x0 = mmsk[j][0] != 0.f ? sx[s * 16 + mtok[j][0]] : 0.f;
                    acc[j][0] = fmaf(-dmg[s], x0, acc[j][0]);
                    acc[j][2] = fmaf(-dmg8[s], x0, acc[j][2]);
                    if constexpr (MODE == XM_Q8) {
                        const float x1 = mmsk[j][1] != 0.f ? sx[s * 16 + mtok[j][1]] : 0.f;
                        acc[j][1] = fmaf(-dmg[s], x1, acc[j][1]);
                        acc[j][3] = fmaf(-dmg8[s], x1, acc[j][3]);
                    }
                }
            }
        }
    } else {  // Q6_K: element e = 128h + 32J + l; X block 4h + J; 16-weight groups G0 = 8h + 2J, G0 + 1
        float sg[16], sg8[16];
        ld_scales<16>(sg, sct, r, 0);
        ld_scales<16>(sg8, sct, r + 8, 0);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t hq[2], hq8[2], l0[2], l08[2], l1[2], l18[2];
#pragma unroll
            for (int lh = 0; lh < 2; ++lh) {
                const int lo = 16 * lh + 4 * t;
                hq[lh] = ldw<MIS>(rg + 128 + 32 * h + lo);
                hq8[lh] = ldw<MIS>(rg8 + 128 + 32 * h + lo);
                l0[lh] = ldw<MIS>(rg + 64 * h + lo);
                l08[lh] = ldw<MIS>(rg8 + 64 * h + lo);
                l1[lh] = ldw<MIS>(rg + 64 * h + 32 + lo);
                l18[lh] = ldw<MIS>(rg8 + 64 * h + 32 + lo);
            }
#pragma unroll
            for (int J = 0; J < 4; ++J) {
                const int ns = 4 * (J >> 1);
                uint32_t q[2], q8[2];
#pragma unroll
                for (int lh = 0; lh < 2; ++lh) {
                    const uint32_t lw = (J & 1) ? l1[lh] : l0[lh], lw8 = (J & 1) ? l18[lh] : l08[lh];
                    q[lh] = ((lw >> ns) & M4) | (((hq[lh] >> (2 * J)) & 0x03030303u) << 4);
                    q8[lh] = ((lw8 >> ns) & M4) | (((hq8[lh] >> (2 * J)) & 0x03030303u) << 4);
                }
                const uint32_t a[4] = {q[0], q8[0], q[1], q8[1]};
                const int b = 4 * h + J, G0 = 8 * h + 2 * J;
#pragma unroll
                for (int j = 0; j < NT; ++j)
                    imma_step<MODE, 2, false, true, FOLD, NT, NCW>(acc[j], a, xv, b, j, make_float2(sg[G0], sg[G0 + 1]),
                                                                   make_float2(sg8[G0], sg8[G0 + 1]));
            }
        }
    }
}

template <int F, int MODE, int NTOK, bool XBF16, int CW, int RG>
__global__ void __launch_bounds__(GI<F, MODE, NTOK, XBF16, CW, RG>::THREADS, GI<F, MODE, NTOK, XBF16, CW, RG>::MINB)
    gemv_i8_kernel(const __grid_constant__ GemvSegs segs, const XIn xin, int K, int N, int cps, unsigned *status,
                   uint64_t wait_limit, AmaxOut amax) {
    using L = GI<F, MODE, NTOK, XBF16, CW, RG>;
    constexpr int S = L::S, NT = L::NT, P = L::P, H = L::H;
    extern __shared__ uint8_t smem_dyn[];
    uint8_t *smem = smem_dyn + ((1024u - (smem_u32(smem_dyn) & 1023u)) & 1023u);
    uint8_t *sstage = smem + L::OFF_STAGE;
    // X areas sized for cps chunks (the launch sized the dynamic shared memory the same way)
    uint8_t *sraw = smem + L::OFF_X;
    uint32_t *sfrag = reinterpret_cast<uint32_t *>(smem + L::off_frag(cps));
    int *sci = reinterpret_cast<int *>(smem + L::off_ci(cps));
    float *sxs = reinterpret_cast<float *>(smem + L::off_xs(cps));
    float *ssx = reinterpret_cast<float *>(smem + L::off_sx(cps));
    float *sct = reinterpret_cast<float *>(smem + L::OFF_SCT);
    float *sred = reinterpret_cast<float *>(smem + L::OFF_X);
    float *sscr = reinterpret_cast<float *>(smem + L::OFF_SCR);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::OFF_BAR);
    uint64_t *empty = full + S;
    uint64_t *xfull = empty + S;
    volatile unsigned *abort_flag = reinterpret_cast<volatile unsigned *>(smem + L::OFF_MISC);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int sg = 0;
    while (sg + 1 < segs.nseg && (int)blockIdx.x >= segs.tile0[sg + 1]) ++sg;
    const CUtensorMap *wmap = &segs.wmap[sg];
    const int M = segs.M[sg];
    float *__restrict__ Y = segs.Y[sg];
    const int m0 = ((int)blockIdx.x - segs.tile0[sg]) * L::ROWS;
    const int nchunks = K / KC;
    const int c_begin = blockIdx.y * cps;
    const int c_end = min(nchunks, c_begin + cps);
    const int nloc = c_end > c_begin ? c_end - c_begin : 0;
    const int KS = gridDim.y;
    const int kslice = nloc * KC;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], CW);
        }
        mbar_init(xfull, 1);
        *abort_flag = 0u;
        fence_barrier_init();
    }
    __syncthreads();
    pdl_launch_dependents();

    float acc[RG][NT][4];
#pragma unroll
    for (int q = 0; q < RG; ++q)
#pragma unroll
        for (int j = 0; j < NT; ++j) acc[q][j][0] = acc[q][j][1] = acc[q][j][2] = acc[q][j][3] = 0.f;

    if (warp == L::WARP_TMA) {
        if (lane == 0) {
            const uint64_t drain_limit = wait_limit < (1ull << 31) ? (1ull << 31) : wait_limit;
            prefetch_tensormap(wmap);
            int issued = 0;
            bool x_issued = false;
            for (int c = 0; c < nloc; ++c) {
                const int s = c % S;
                if (c >= S && !gwait(abort_flag, &empty[s], ((c / S) - 1) & 1, wait_limit)) break;
                if (*abort_flag) break;
                const int cg = c_begin + c;
                const int xb = F == Q6_K ? ((210 * cg) & ~15) : cg * L::WIN;
                mbar_arrive_expect_tx(&full[s], (uint32_t)L::STAGE);
                tma_load_2d(sstage + s * L::STAGE, wmap, &full[s], xb >> 1, m0);
                issued = c + 1;
                if (c == (nloc < S ? nloc : S) - 1) {
                    // weights stream before the preceding kernel on the stream
                    // has finished; X only after it
                    pdl_wait();
                    if constexpr (MODE == XM_EXACT) {
                        const uint32_t rowb = (uint32_t)kslice * L::XES;
                        mbar_arrive_expect_tx(xfull, rowb * (uint32_t)N);
                        for (int n = 0; n < N; ++n)
                            tma_load_1d(sraw + n * rowb,
                                        static_cast<const uint8_t *>(xin.x) +
                                            ((int64_t)n * K + (int64_t)c_begin * KC) * L::XES,
                                        rowb, xfull);
                    } else {
                        // codes [n][kslice] then scales [n][kslice / 32]
                        const uint32_t rowb = (uint32_t)kslice, srow = (uint32_t)(kslice / 32) * 4;
                        mbar_arrive_expect_tx(xfull, (rowb + srow) * (uint32_t)N);
                        for (int n = 0; n < N; ++n) {
                            tma_load_1d(sraw + n * rowb,
                                        static_cast<const uint8_t *>(xin.x) + (int64_t)n * K + (int64_t)c_begin * KC,
                                        rowb, xfull);
                            tma_load_1d(sraw + N * rowb + n * srow,
                                        xin.scales + (int64_t)n * (K / 32) + (int64_t)c_begin * (KC / 32), srow,
                                        xfull);
                        }
                    }
                    x_issued = true;
                }
            }
            if (*abort_flag) {
                for (int c = issued - S < 0 ? 0 : issued - S; c < issued; ++c)
                    (void)mbar_wait(&full[c % S], (c / S) & 1, drain_limit);
                if (x_issued) (void)mbar_wait(xfull, 0, drain_limit);
            }
        }
    } else {
        pdl_wait();   // Y is written below: order after the preceding kernel
        const int tid = threadIdx.x;
        const bool x_ok = nloc == 0 || __all_sync(0xffffffffu, gwait(abort_flag, xfull, 0, wait_limit));
        if (x_ok) prep_x_i8<F, MODE, NTOK, XBF16, CW, RG>(sraw, kslice, N, sfrag, sci, sxs, ssx, tid);
        asm volatile("bar.sync 1, %0;" ::"r"(CW * 32) : "memory");   // compute warps only

        const int g = lane >> 2, t = lane & 3;
        constexpr int NCW = L::NCW;
        XView<NT, NCW> xv0;
        xv0.frag = reinterpret_cast<const uint2 *>(sfrag) + 4 * (g % NCW) + t;
        xv0.ci = reinterpret_cast<const int4 *>(sci) + t;
        xv0.xs = reinterpret_cast<const float2 *>(sxs) + t;
        // Q4_K min term: slot i of tile j (column 8j + 2t + i) adds it for its
        // token if it is that token's first column
        int mtok[NT][2];
        float mmsk[NT][2];
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int col = 8 * j + 2 * t + i;
                mtok[j][i] = col / P < 16 ? col / P : 15;
                mmsk[j][i] = (col % P == 0 && col / P < N) ? 1.f : 0.f;
            }
        for (int c = 0; c < nloc && x_ok; ++c) {
            const int s = c % S;
            const int cg = c_begin + c;
            const int woff = F == Q6_K ? ((210 * cg) & 15) : 0;
            if (!__all_sync(0xffffffffu, gwait(abort_flag, &full[s], (c / S) & 1, wait_limit) && !*abort_flag))
                break;
            const uint8_t *raw = sstage + s * L::STAGE;
#pragma unroll
            for (int q = 0; q < RG; ++q) prep_scales_i8<F, L::FOLD>(sct, raw, woff, RG * warp + q, lane, sxs + 8 * c);
            __syncwarp();
            XView<NT, NCW> xv = xv0;
            xv.frag += c * 8 * NT * 4 * NCW;
            xv.ci += c * 8 * NT * 4;
            xv.xs += c * 8 * NT * 4;
            const float *sxc = ssx + c * 8 * 16;
#pragma unroll
            for (int q = 0; q < RG; ++q) {
                const int rg = 16 * (RG * warp + q) + g;
                const uint8_t *pg = raw + rg * L::WIN + woff;
                if (F == Q6_K && (woff & 2))
                    compute_chunk_i8<F, MODE, NT, NCW, L::FOLD, true>(acc[q], pg, pg + 8 * L::WIN, xv, sct, rg, sxc, mtok,
                                                                 mmsk, t);
                else
                    compute_chunk_i8<F, MODE, NT, NCW, L::FOLD, false>(acc[q], pg, pg + 8 * L::WIN, xv, sct, rg, sxc, mtok,
                                                                  mmsk, t);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
    }

    // Columns -> one value per (row, token), laid out as one column per
    // token (finish_tile's P == 1 layout).  With FOLD the digit weights are
    // applied here (every block shares them).
    float acc1[RG][L::NT1][4];
#pragma unroll
    for (int q = 0; q < RG; ++q)
#pragma unroll
        for (int j = 0; j < L::NT1; ++j) acc1[q][j][0] = acc1[q][j][1] = acc1[q][j][2] = acc1[q][j][3] = 0.f;
    if (warp < CW) {
        const int g = lane >> 2, t = lane & 3;
        float *scr = sscr + warp * 16 * 8;
#pragma unroll
        for (int q = 0; q < RG; ++q) {
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                float w0 = 1.f, w1 = 1.f;
                if constexpr (L::FOLD && L::D > 1) {
                    w0 = __uint_as_float((uint32_t)(127 - 8 * (((8 * j + 2 * t) % P) / H)) << 23);
                    w1 = __uint_as_float((uint32_t)(127 - 8 * (((8 * j + 2 * t + 1) % P) / H)) << 23);
                }
                scr[g * 8 + 2 * t] = acc[q][j][0] * w0;
                scr[g * 8 + 2 * t + 1] = acc[q][j][1] * w1;
                scr[(g + 8) * 8 + 2 * t] = acc[q][j][2] * w0;
                scr[(g + 8) * 8 + 2 * t + 1] = acc[q][j][3] * w1;
                __syncwarp();
#pragma unroll
                for (int j1 = 0; j1 < L::NT1; ++j1)
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        const int n = 8 * j1 + 2 * t + i;
                        if (n < NTOK && (n * P) / 8 == j) {
                            float v = 0.f, v8 = 0.f;
#pragma unroll
                            for (int p = 0; p < P; ++p) {
                                v += scr[g * 8 + n * P + p - 8 * j];
                                v8 += scr[(g + 8) * 8 + n * P + p - 8 * j];
                            }
                            acc1[q][j1][i] += v;
                            acc1[q][j1][2 + i] += v8;
                        }
                    }
                __syncwarp();
            }
        }
    }
    const bool aborted = *abort_flag != 0u;
    finish_tile<L::NT1, 1, CW, RG>(acc1, sred, Y, M, N, m0, KS, aborted, warp, lane, amax.keys);
    amax_last_cta(amax, N);
    if (threadIdx.x == 0 && aborted) report_status(status, kStatusTimeout);
}

template <int F, int MODE, int NTOK, bool XBF16, int CW, int RG>
cudaError_t launch_i8(const GemvPlan &plan, const GemvSegs &segs0, const XIn &xin, int64_t K, int N, bool pdl,
                      unsigned *status, uint64_t limit, cudaStream_t st, const AmaxOut &amax) {
    using L = GI<F, MODE, NTOK, XBF16, CW, RG>;
    if (plan.rows != L::ROWS || N > NTOK) return cudaErrorInvalidValue;
    const int nchunks = (int)(K / KC);
    const int cps = (nchunks + plan.ks - 1) / plan.ks;   // as launch_cluster computes it
    if (cps > L::MAXC) return cudaErrorInvalidValue;
    auto kern = gemv_i8_kernel<F, MODE, NTOK, XBF16, CW, RG>;
    static std::atomic<uint64_t> configured{0};
    cudaError_t e = set_smem_once(kern, L::smem(L::MAXC), configured);
    if (e != cudaSuccess) return e;
    GemvSegs sg = segs0;
    const int64_t tiles = set_tiles(sg, L::ROWS);
    return launch_cluster(kern, L::smem(cps), L::THREADS, tiles, plan.ks, nchunks, st, pdl, sg, xin, K, N, status,
                          limit, amax);
}

// Largest K slice (in 256-weight chunks) one CTA can hold for this variant.
template <int F, int MODE, int NTOK, bool XBF16, int CW, int RG>
constexpr int i8_maxc() {
    return GI<F, MODE, NTOK, XBF16, CW, RG>::MAXC;
}

}  // namespace
}  // namespace qmm
