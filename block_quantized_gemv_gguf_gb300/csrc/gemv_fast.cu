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
// CTA = CW compute warps (16 rows each; CW = 4 or 8) + 1 TMA warp.  Per
// 256-weight chunk, 2-D TMA brings the raw weight bytes of the tile's rows and
// the raw X slice [N][256] into a ring of stages.  Each compute warp turns its
// share of the next chunk's X slice into MMA B fragments (a second ring, one
// chunk ahead, handed over with mbarriers) and decodes the scales of its own
// rows; nothing on the compute warps' path waits on global memory.  For small
// M the K range is split over a thread-block cluster and the partial sums
// are reduced through distributed shared memory by cluster rank 0, in a fixed
// order (deterministic, no atomics, Y is written exactly once).
#include "gemv_shared.cuh"

namespace qmm {
namespace {

// Tile geometry: CW compute warps x 16 rows, plus one TMA warp.
template <int F, int NT, int CW> struct GL {
    static constexpr int ROWS = 16 * CW;
    static constexpr int WARP_TMA = CW;
    static constexpr int THREADS = (CW + 1) * 32;
    static constexpr int S = (CW == 8 || NT >= 3) ? 2 : 3;     // TMA stages of weights
    static constexpr int XRS = 3;                              // TMA slots of raw X slices
    static constexpr int XR = 2;                               // X-fragment ring slots
    static constexpr int WIN = GWin<F>::bytes;
    static constexpr int RAWW = ROWS * WIN;                   // multiple of 1024
    static constexpr int XRAW = 4096 * NT;                     // raw X slice: up to 4NT f32 / 8NT bf16 rows
    static constexpr int STAGE = RAWW;
    static constexpr int XS = 16 * NT * 32 * 8;                // B fragments of one chunk
    static constexpr int SXB = kmin_fmt(F) ? 8 * 16 * 4 : 0;   // Q4_K/Q5_K sub-block sums of x
    static constexpr int XSLOT = XS + SXB;
    static constexpr int SCT = ROWS * SCW * 4;                 // scale table (each warp owns its 16 rows)
    static constexpr int OFF_STAGE = 0;
    static constexpr int OFF_XRAW = S * STAGE;
    static constexpr int OFF_XR = OFF_XRAW + XRS * XRAW;
    static constexpr int OFF_RED = OFF_XR;                     // reduction buffer aliases the X ring
    static constexpr int OFF_SCT = OFF_XR + XR * XSLOT;
    static constexpr int OFF_BAR = OFF_SCT + SCT;
    static constexpr int NBAR = 2 * S + 2 * XRS + 2 * XR;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int TOTAL = OFF_MISC + 16;
    static constexpr int SMEM = TOTAL + 1024;
    // CTAs per SM the shared memory allows (at most 4): the register budget
    // the compiler may use without lowering that occupancy
    static constexpr int MINB = 232448 / SMEM >= 4 ? 4 : (232448 / SMEM >= 1 ? 232448 / SMEM : 1);
    static_assert(XR * XSLOT >= ROWS * 16 * 4, "reduction buffer fits in the X ring");
    static_assert(XSLOT % 16 == 0 && STAGE % 1024 == 0 && XRAW % 1024 == 0, "alignment");
    static_assert(SMEM <= 232448, "shared memory");
};

// ---------------------------------------------------------------------------
// small device helpers
// ---------------------------------------------------------------------------
// a + nb (bf16x2); nb holds the negated offsets, so the subtraction of the
// magic-number offset is one plain add
__device__ __forceinline__ uint32_t badd2(uint32_t a, uint32_t nb) {
    uint32_t r;
    asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(nb));
    return r;
}
// bf16x2 (M + b0, M + b1) from bytes 0,1 (SEL01) or 2,3 (SEL23) of `v`,
// where M is the bf16 whose high byte is `hi` (0x43: 128, 0x45: 2048).
// The constant in a register the compiler may not rematerialize (one
// register for the whole loop instead of an immediate load per use).
template <uint32_t C>
__device__ __forceinline__ uint32_t in_reg() {
    uint32_t r;
    asm("mov.b32 %0, %1;" : "=r"(r) : "n"(C));
    return r;
}

// hi: a register holding HI in its low byte.
__device__ __forceinline__ uint32_t pair01(uint32_t v, uint32_t hi) { return __byte_perm(v, hi, 0x4140u); }
__device__ __forceinline__ uint32_t pair23(uint32_t v, uint32_t hi) { return __byte_perm(v, hi, 0x4342u); }

constexpr uint32_t BF2(uint32_t h) { return h | (h << 16); }   // bf16 pair from one bf16 bit pattern
// negated offsets -128, -136, -160, -2176 as bf16 pairs
constexpr uint32_t C128 = BF2(0xC300u), C136 = BF2(0xC308u), C160 = BF2(0xC320u), C2176 = BF2(0xC508u);

// A quad of zeros the compiler keeps in registers (the zero accumulator of
// every first MMA of a block reads it; nothing re-zeroes registers per MMA).
struct ZeroQuad {
    float z[4];
};
__device__ __forceinline__ ZeroQuad zero_quad() {
    ZeroQuad q;
    asm("mov.b32 %0, 0;\n\tmov.b32 %1, 0;\n\tmov.b32 %2, 0;\n\tmov.b32 %3, 0;"
        : "=f"(q.z[0]), "=f"(q.z[1]), "=f"(q.z[2]), "=f"(q.z[3]));
    return q;
}

// d = A * B + 0
__device__ __forceinline__ void mma16816_z(float (&d)[4], const uint32_t (&a)[4], uint2 b, const ZeroQuad &z) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b.x), "r"(b.y), "f"(z.z[0]), "f"(z.z[1]), "f"(z.z[2]),
          "f"(z.z[3]));
}

// d += A * B
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint2 b) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b.x), "r"(b.y));
}


// A fragment from two words of byte codes (row g, row g+8): elements 4t..4t+3;
// offs = the negated offset pair (so the code value is pair + offs).
template <uint32_t HI>
__device__ __forceinline__ void afrag(uint32_t (&a)[4], uint32_t vg, uint32_t vg8, uint32_t offs) {
    const uint32_t hi = in_reg<HI>();
    a[0] = badd2(pair01(vg, hi), offs);
    a[1] = badd2(pair01(vg8, hi), offs);
    a[2] = badd2(pair23(vg, hi), offs);
    a[3] = badd2(pair23(vg8, hi), offs);
}

// ---------------------------------------------------------------------------
// Per-chunk preparation from the TMA-staged raw bytes, shared by the compute
// warps (warp w of CW takes every CW-th piece of work):
//  * B fragments of X: xs[ks][j][lane] = {b0, b1}; MMA column 8j+g is
//    (token (8j+g)/P, piece (8j+g)%P); element 4t+i of k-step ks is
//    x[n][k0 + 16 ks + 4t + i];
//  * Q4_K: sx[s][n] = sum of x[n] over sub-block s;
//  * each warp's own 16 rows of the scale table sct[row][0..15].
// ---------------------------------------------------------------------------
template <int F, int NT, int P, bool XBF16, int CW>
__device__ __forceinline__ void prep_x(uint2 *xs, float *sx, const uint8_t *xraw, int N, int w, int lane) {
    // One pass of a warp fills one fragment block (ks, j): lane (g, t) holds
    // column 8j+g = (token n, piece p) at elements 4t..4t+3 of k-step ks.
    // Reads of a quarter-warp are 64 contiguous bytes of one token and the
    // stores are 256 contiguous bytes: no bank conflicts either way.
    const int t = lane & 3;
    const int ncols = P * N;
    // With a single 8-column tile (NT == 1) and fewer than 8 used columns, a
    // pass covers cpp columns x (8 / cpp) k-steps so that no lane idles.
    const int cpp = NT > 1 ? 8 : (ncols > 4 ? 8 : ncols > 2 ? 4 : ncols > 1 ? 2 : 1);
    const int kpp = 8 / cpp;
    const int g = (lane >> 2) % cpp, ksl = (lane >> 2) / cpp;
    for (int pass = w; pass < (16 * NT) / kpp; pass += CW) {
        const int blk = pass * kpp + ksl;        // = ks * NT + j
        const int ks = blk / NT, j = blk % NT;
        const int col = 8 * j + g;
        if (col >= ncols) continue;              // unused MMA column: never read back
        const int n = col / P, p = col % P;
        uint32_t b0, b1;
        if constexpr (XBF16) {
            const uint2 v = *reinterpret_cast<const uint2 *>(xraw + (n * 256 + 16 * ks + 4 * t) * 2);
            b0 = v.x;
            b1 = v.y;
        } else {
            const float4 v = *reinterpret_cast<const float4 *>(xraw + (n * 256 + 16 * ks + 4 * t) * 4);
            const uint32_t hi01 = pack_bf16x2(v.x, v.y), hi23 = pack_bf16x2(v.z, v.w);
            if (P == 1 || p == 0) {
                b0 = hi01;
                b1 = hi23;
            } else {
                const float r0 = v.x - __uint_as_float(hi01 << 16), r1 = v.y - __uint_as_float(hi01 & 0xFFFF0000u);
                const float r2 = v.z - __uint_as_float(hi23 << 16), r3 = v.w - __uint_as_float(hi23 & 0xFFFF0000u);
                b0 = pack_bf16x2(r0, r1);
                b1 = pack_bf16x2(r2, r3);
            }
        }
        xs[blk * 32 + 4 * g + t] = make_uint2(b0, b1);
    }
    if constexpr (kmin_fmt(F)) {
        for (int it = 32 * w + lane; it < 8 * N; it += 32 * CW) {
            const int s = it & 7, n = it >> 3;
            float acc = 0.f;
            if constexpr (XBF16) {
                const uint32_t *x = reinterpret_cast<const uint32_t *>(xraw + (n * 256 + 32 * s) * 2);
#pragma unroll
                for (int e = 0; e < 16; ++e) acc += __uint_as_float(x[e] << 16) + __uint_as_float(x[e] & 0xFFFF0000u);
            } else {
                const float4 *x = reinterpret_cast<const float4 *>(xraw + (n * 256 + 32 * s) * 4);
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

// Scale-table rows 16w..16w+15 of warp w: lane = (row, half).
template <int F>
__device__ __forceinline__ void prep_scales(float *sct, const uint8_t *raw, int woff, int w, int lane) {
    constexpr int WIN = GWin<F>::bytes;
    auto st4 = [&](int row, int e0, float a, float b, float c, float d) {
        *reinterpret_cast<float4 *>(sct + sct_index(row, e0)) = make_float4(a, b, c, d);
    };
    {
        const int row = 16 * w + (lane >> 1), half = lane & 1;
        const uint8_t *rb = raw + row * WIN + woff;
        if constexpr (F == Q4_0 || F == Q8_0) {
            constexpr int BB = F == Q4_0 ? 18 : 34;
            const uint8_t *b = rb + BB * 4 * half;
            st4(row, 4 * half, f16_bits(lds_u16(b)), f16_bits(lds_u16(b + BB)), f16_bits(lds_u16(b + 2 * BB)),
                f16_bits(lds_u16(b + 3 * BB)));
        } else if constexpr (kmin_fmt(F)) {   // Q4_K, Q5_K: same header fields
            const float d = f16_bits(lds_u16(rb)), dmin = f16_bits(lds_u16(rb + 2));
            const uint32_t w0 = ld32(rb + 4), w1 = ld32(rb + 8), w2 = ld32(rb + 12);
            // bytes: sc[0..3], mn[0..3], sc[4..7], mn[4..7] (GGUF 6-bit packing)
            const uint32_t sc = half ? ((w2 & 0x0F0F0F0Fu) | (((w0 >> 6) & 0x03030303u) << 4)) : (w0 & 0x3F3F3F3Fu);
            const uint32_t mn =
                half ? (((w2 >> 4) & 0x0F0F0F0Fu) | (((w1 >> 6) & 0x03030303u) << 4)) : (w1 & 0x3F3F3F3Fu);
            st4(row, 4 * half, d * (float)(sc & 0xFFu), d * (float)((sc >> 8) & 0xFFu),   // d * sc_s
                d * (float)((sc >> 16) & 0xFFu), d * (float)(sc >> 24));
            st4(row, 8 + 4 * half, dmin * (float)(mn & 0xFFu), dmin * (float)((mn >> 8) & 0xFFu),   // dmin * m_s
                dmin * (float)((mn >> 16) & 0xFFu), dmin * (float)(mn >> 24));
        } else {  // Q6_K: d * scales[G], G = 0..15
            const float d = f16_bits(lds_u16(rb + 208));
            const int8_t *sc = reinterpret_cast<const int8_t *>(rb + 192 + 8 * half);
            st4(row, 8 * half, d * (float)sc[0], d * (float)sc[1], d * (float)sc[2], d * (float)sc[3]);
            st4(row, 8 * half + 4, d * (float)sc[4], d * (float)sc[5], d * (float)sc[6], d * (float)sc[7]);
        }
    }
}

// Accumulate one scaled MMA result into the four fragment accumulators
// (columns 2t, 2t+1 of rows g and g+8; for P == 2 these are the two pieces
// of one token and are summed at the very end).
__device__ __forceinline__ void acc_scaled(float *acc, const float (&d)[4], float sg, float sg8) {
    ffma2(acc[0], acc[1], sg, sg, d[0], d[1]);
    ffma2(acc[2], acc[3], sg8, sg8, d[2], d[3]);
}

// ---------------------------------------------------------------------------
// Chunk compute for one warp: 16 rows (g, g+8 per thread) x 256 weights.
// Row windows start 16-byte aligned (Q6_K: + woff, even); every 32-bit code
// word is read with its alignment known at compile time (MIS: woff % 4 == 2).
// ---------------------------------------------------------------------------
template <int KSTR, int JSTR>
__device__ __forceinline__ uint2 bfrag(const uint8_t *xb, int ks, int j) {
    return *reinterpret_cast<const uint2 *>(xb + ks * KSTR + j * JSTR);
}

// xb: this lane's B fragment of k-step 0, tile 0 of the chunk; fragment
// (ks, j) is at xb + ks * KSTR + j * JSTR.
template <int F, int NT, int P, bool MIS, int KSTR, int JSTR>
__device__ __forceinline__ void compute_chunk(float (&acc)[NT][4], const uint8_t *rg, const uint8_t *rg8,
                                              const uint8_t *xb, const float *sct, int r, const float *sx, int t) {
    const uint32_t k128 = in_reg<C128>(), k136 = in_reg<C136>(), k160 = in_reg<C160>(), k2176 = in_reg<C2176>();
    const ZeroQuad zq = zero_quad();
    if constexpr (F == Q4_0) {
        float sg[8], sg8[8];
        ld_scales<8>(sg, sct, r, 0);
        ld_scales<8>(sg8, sct, r + 8, 0);
#pragma unroll
        for (int bp = 0; bp < 4; ++bp) {            // blocks 2bp, 2bp+1: 36 bytes from a 4-aligned start
            const uint8_t *pg = rg + 36 * bp, *pg8 = rg8 + 36 * bp;
            const uint32_t qeg = __byte_perm(ld32(pg + 4 * t), ld32(pg + 4 * t + 4), 0x5432u);
            const uint32_t qeg8 = __byte_perm(ld32(pg8 + 4 * t), ld32(pg8 + 4 * t + 4), 0x5432u);
            const uint32_t qog = ld32(pg + 20 + 4 * t), qog8 = ld32(pg8 + 20 + 4 * t);
#pragma unroll
            for (int bb = 0; bb < 2; ++bb) {
                const int b = 2 * bp + bb;
                const uint32_t wg = bb ? qog : qeg, wg8 = bb ? qog8 : qeg8;
                uint32_t a0[4], a1[4];
                afrag<0x43u>(a0, wg & 0x0F0F0F0Fu, wg8 & 0x0F0F0F0Fu, k136);
                afrag<0x43u>(a1, (wg >> 4) & 0x0F0F0F0Fu, (wg8 >> 4) & 0x0F0F0F0Fu, k136);
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    float d[4];
                    mma16816_z(d, a0, bfrag<KSTR, JSTR>(xb, 2 * b, j), zq);
                    mma16816(d, a1, bfrag<KSTR, JSTR>(xb, 2 * b + 1, j));
                    acc_scaled(acc[j], d, sg[b], sg8[b]);
                }
            }
        }
    } else if constexpr (F == Q8_0) {
        float sg[8], sg8[8];
        ld_scales<8>(sg, sct, r, 0);
        ld_scales<8>(sg8, sct, r + 8, 0);
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            // block b at 34 b: odd blocks have 4-aligned codes, even blocks 2 mod 4
            const uint8_t *pg = rg + 34 * b + 2, *pg8 = rg8 + 34 * b + 2;
            uint32_t al[2][4], ah[2][4];
#pragma unroll
            for (int grp = 0; grp < 2; ++grp) {
                const int o = 16 * grp + 4 * t;
                const uint32_t ug = ((b & 1) ? ld32(pg + o) : ld32_off2(pg + o)) ^ 0x80808080u;
                const uint32_t ug8 = ((b & 1) ? ld32(pg8 + o) : ld32_off2(pg8 + o)) ^ 0x80808080u;
                // q = 16 * (hi - 8) + lo with hi, lo the nibbles of q + 128
                afrag<0x43u>(al[grp], ug & 0x0F0F0F0Fu, ug8 & 0x0F0F0F0Fu, k128);
                afrag<0x45u>(ah[grp], (ug >> 4) & 0x0F0F0F0Fu, (ug8 >> 4) & 0x0F0F0F0Fu, k2176);
            }
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                float d[4];
                const uint2 b0 = bfrag<KSTR, JSTR>(xb, 2 * b, j), b1 = bfrag<KSTR, JSTR>(xb, 2 * b + 1, j);
                mma16816_z(d, al[0], b0, zq);
                mma16816(d, ah[0], b0);
                mma16816(d, al[1], b1);
                mma16816(d, ah[1], b1);
                acc_scaled(acc[j], d, sg[b], sg8[b]);
            }
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
                uint32_t a0[4], a1[4];
                afrag<0x43u>(a0, (w0g >> sh) & 0x0F0F0F0Fu, (w0g8 >> sh) & 0x0F0F0F0Fu, k128);
                afrag<0x43u>(a1, (w1g >> sh) & 0x0F0F0F0Fu, (w1g8 >> sh) & 0x0F0F0F0Fu, k128);
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    float d[4];
                    mma16816_z(d, a0, bfrag<KSTR, JSTR>(xb, 2 * s, j), zq);
                    mma16816(d, a1, bfrag<KSTR, JSTR>(xb, 2 * s + 1, j));
                    // w = d*sc*q - dmin*m  =>  sum w x = (d sc) sum q x - (dmin m) sum x
                    acc_scaled(acc[j], d, dsg[s], dsg8[s]);
                    if constexpr (P == 2) {       // min term once per token (on the hi piece)
                        const float sxn = sx[s * 16 + 4 * j + t];
                        acc[j][0] = fmaf(-dmg[s], sxn, acc[j][0]);
                        acc[j][2] = fmaf(-dmg8[s], sxn, acc[j][2]);
                    } else {
                        const float sx0 = sx[s * 16 + 8 * j + 2 * t], sx1 = sx[s * 16 + 8 * j + 2 * t + 1];
                        ffma2(acc[j][0], acc[j][1], -dmg[s], -dmg[s], sx0, sx1);
                        ffma2(acc[j][2], acc[j][3], -dmg8[s], -dmg8[s], sx0, sx1);
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
        // bit s of qh[l] is bit 4 of sub-block s's element l (l = 4t+i, 16+4t+i)
        const uint32_t h0g = ld32(rg + 16 + 4 * t), h1g = ld32(rg + 32 + 4 * t);
        const uint32_t h0g8 = ld32(rg8 + 16 + 4 * t), h1g8 = ld32(rg8 + 32 + 4 * t);
#pragma unroll
        for (int pr = 0; pr < 4; ++pr) {            // sub-blocks 2pr (low nibbles), 2pr+1 (high)
            const uint32_t w0g = ld32(qg + 32 * pr + 4 * t), w1g = ld32(qg + 32 * pr + 16 + 4 * t);
            const uint32_t w0g8 = ld32(qg8 + 32 * pr + 4 * t), w1g8 = ld32(qg8 + 32 * pr + 16 + 4 * t);
#pragma unroll
            for (int hn = 0; hn < 2; ++hn) {
                const int s = 2 * pr + hn, sh = 4 * hn;
                const uint32_t c0g = ((w0g >> sh) & 0x0F0F0F0Fu) | (((h0g >> s) & 0x01010101u) << 4);
                const uint32_t c0g8 = ((w0g8 >> sh) & 0x0F0F0F0Fu) | (((h0g8 >> s) & 0x01010101u) << 4);
                const uint32_t c1g = ((w1g >> sh) & 0x0F0F0F0Fu) | (((h1g >> s) & 0x01010101u) << 4);
                const uint32_t c1g8 = ((w1g8 >> sh) & 0x0F0F0F0Fu) | (((h1g8 >> s) & 0x01010101u) << 4);
                uint32_t a0[4], a1[4];
                afrag<0x43u>(a0, c0g, c0g8, k128);
                afrag<0x43u>(a1, c1g, c1g8, k128);
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    float d[4];
                    mma16816_z(d, a0, bfrag<KSTR, JSTR>(xb, 2 * s, j), zq);
                    mma16816(d, a1, bfrag<KSTR, JSTR>(xb, 2 * s + 1, j));
                    acc_scaled(acc[j], d, dsg[s], dsg8[s]);
                    if constexpr (P == 2) {       // min term once per token (on the hi piece)
                        const float sxn = sx[s * 16 + 4 * j + t];
                        acc[j][0] = fmaf(-dmg[s], sxn, acc[j][0]);
                        acc[j][2] = fmaf(-dmg8[s], sxn, acc[j][2]);
                    } else {
                        const float sx0 = sx[s * 16 + 8 * j + 2 * t], sx1 = sx[s * 16 + 8 * j + 2 * t + 1];
                        ffma2(acc[j][0], acc[j][1], -dmg[s], -dmg[s], sx0, sx1);
                        ffma2(acc[j][2], acc[j][3], -dmg8[s], -dmg8[s], sx0, sx1);
                    }
                }
            }
        }
    } else {  // Q6_K: element e = 128h + 32J + l, l = 16 lh + 4t + i, k-step G = 8h + 2J + lh
        float sg[16], sg8[16];
        ld_scales<16>(sg, sct, r, 0);
        ld_scales<16>(sg8, sct, r + 8, 0);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int lh = 0; lh < 2; ++lh) {
                const int lo = 16 * lh + 4 * t;
                const uint32_t hg = ldw<MIS>(rg + 128 + 32 * h + lo), hg8 = ldw<MIS>(rg8 + 128 + 32 * h + lo);
                const uint32_t l0g = ldw<MIS>(rg + 64 * h + lo), l0g8 = ldw<MIS>(rg8 + 64 * h + lo);
                const uint32_t l1g = ldw<MIS>(rg + 64 * h + 32 + lo), l1g8 = ldw<MIS>(rg8 + 64 * h + 32 + lo);
#pragma unroll
                for (int J = 0; J < 4; ++J) {
                    const int G = 8 * h + 2 * J + lh;
                    const uint32_t lwg = (J & 1) ? l1g : l0g, lwg8 = (J & 1) ? l1g8 : l0g8;
                    const int ns = 4 * (J >> 1);
                    const uint32_t qg = ((lwg >> ns) & 0x0F0F0F0Fu) | (((hg >> (2 * J)) & 0x03030303u) << 4);
                    const uint32_t qg8 = ((lwg8 >> ns) & 0x0F0F0F0Fu) | (((hg8 >> (2 * J)) & 0x03030303u) << 4);
                    uint32_t a[4];
                    afrag<0x43u>(a, qg, qg8, k160);
#pragma unroll
                    for (int j = 0; j < NT; ++j) {
                        float d[4];
                        mma16816_z(d, a, bfrag<KSTR, JSTR>(xb, G, j), zq);
                        acc_scaled(acc[j], d, sg[G], sg8[G]);
                    }
                }
            }
        }
    }
}

template <int F, int NT, int P, bool XBF16, int CW>
__global__ void __launch_bounds__(GL<F, NT, CW>::THREADS, GL<F, NT, CW>::MINB)
    gemv_mma_kernel(const __grid_constant__ GemvSegs segs, const __grid_constant__ CUtensorMap xmap, int K, int N,
                    int cps, unsigned *status, uint64_t wait_limit, AmaxOut amax) {
    using L = GL<F, NT, CW>;
    constexpr int S = L::S, XR = L::XR, ROWS = L::ROWS;
    extern __shared__ uint8_t smem_dyn[];
    // 1024-byte aligned base, derived from the shared array itself so that
    // every access below compiles to a shared-window load or store
    uint8_t *smem = smem_dyn + ((1024u - (smem_u32(smem_dyn) & 1023u)) & 1023u);
    uint8_t *sstage = smem + L::OFF_STAGE;
    uint8_t *sxraw = smem + L::OFF_XRAW;
    uint8_t *sxr = smem + L::OFF_XR;
    float *sct = reinterpret_cast<float *>(smem + L::OFF_SCT);
    float *sred = reinterpret_cast<float *>(smem + L::OFF_RED);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::OFF_BAR);
    uint64_t *empty = full + S;
    uint64_t *rxfull = empty + S;          // raw X slot landed
    uint64_t *rxempty = rxfull + L::XRS;   // raw X slot consumed by every warp's share
    uint64_t *xfull = rxempty + L::XRS;    // X fragments of a chunk complete
    uint64_t *xempty = xfull + XR;
    volatile unsigned *abort_flag = reinterpret_cast<volatile unsigned *>(smem + L::OFF_MISC);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // this CTA's weight matrix (segment) and tile within it
    int sg = 0;
    while (sg + 1 < segs.nseg && (int)blockIdx.x >= segs.tile0[sg + 1]) ++sg;
    const CUtensorMap *wmap = &segs.wmap[sg];
    const int M = segs.M[sg];
    float *__restrict__ Y = segs.Y[sg];
    const int m0 = ((int)blockIdx.x - segs.tile0[sg]) * ROWS;
    const int nchunks = K / KC;
    const int c_begin = blockIdx.y * cps;
    const int c_end = min(nchunks, c_begin + cps);
    const int nloc = c_end > c_begin ? c_end - c_begin : 0;
    const int KS = gridDim.y;
    const uint32_t xbytes = (uint32_t)N * 256u * (XBF16 ? 2u : 4u);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], CW);
        }
        for (int s = 0; s < L::XRS; ++s) {
            mbar_init(&rxfull[s], 1);
            mbar_init(&rxempty[s], CW);
        }
        for (int s = 0; s < XR; ++s) {
            mbar_init(&xfull[s], CW);
            mbar_init(&xempty[s], CW);
        }
        *abort_flag = 0u;
        fence_barrier_init();
    }
    __syncthreads();
    pdl_launch_dependents();

    float acc[1][NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) acc[0][j][0] = acc[0][j][1] = acc[0][j][2] = acc[0][j][3] = 0.f;

    if (warp == L::WARP_TMA) {
        // ---------------- TMA producers: lane 0 weights, lane 1 raw X ----------------
        const uint64_t drain_limit = wait_limit < (1ull << 31) ? (1ull << 31) : wait_limit;
        if (lane == 0) {
            prefetch_tensormap(wmap);
            int issued = 0;   // loads are issued in chunk order 0, 1, ..., issued-1
            for (int c = 0; c < nloc; ++c) {
                const int s = c % S;
                if (c >= S && !gwait(abort_flag, &empty[s], ((c / S) - 1) & 1, wait_limit)) break;
                if (*abort_flag) break;
                const int cg = c_begin + c;
                const int xb = F == Q6_K ? ((210 * cg) & ~15) : cg * L::WIN;
                mbar_arrive_expect_tx(&full[s], (uint32_t)L::RAWW);
                tma_load_2d(sstage + s * L::STAGE, wmap, &full[s], xb >> 1, m0);
                issued = c + 1;
            }
            if (*abort_flag)   // drain: the last load issued into each stage
                for (int c = issued - S < 0 ? 0 : issued - S; c < issued; ++c)
                    (void)mbar_wait(&full[c % S], (c / S) & 1, drain_limit);
        } else if (lane == 1) {
            prefetch_tensormap(&xmap);
            pdl_wait();   // X may come from the preceding kernel
            constexpr int XRS = L::XRS;
            int issued = 0;
            for (int c = 0; c < nloc; ++c) {
                const int s = c % XRS;
                if (c >= XRS && !gwait(abort_flag, &rxempty[s], ((c / XRS) - 1) & 1, wait_limit)) break;
                if (*abort_flag) break;
                mbar_arrive_expect_tx(&rxfull[s], xbytes);
                tma_load_2d(sxraw + s * L::XRAW, &xmap, &rxfull[s], (c_begin + c) * KC, 0);
                issued = c + 1;
            }
            if (*abort_flag)
                for (int c = issued - XRS < 0 ? 0 : issued - XRS; c < issued; ++c)
                    (void)mbar_wait(&rxfull[c % XRS], (c / XRS) & 1, drain_limit);
        }
    } else {
        // ---------------- compute warps ----------------
        pdl_wait();   // Y is written below: order after the preceding kernel
        const int g = lane >> 2, t = lane & 3;
        const int rg = 16 * warp + g;         // tile rows of this thread: rg, rg + 8
        // Build this warp's share of the X fragments of local chunk c.
        auto build_share = [&](int c) -> bool {
            const int rs = c % L::XRS, xs = c % XR;
            if (!__all_sync(0xffffffffu, gwait(abort_flag, &rxfull[rs], (c / L::XRS) & 1, wait_limit))) return false;
            if (c >= XR &&
                !__all_sync(0xffffffffu, gwait(abort_flag, &xempty[xs], ((c / XR) - 1) & 1, wait_limit)))
                return false;
            uint8_t *slot = sxr + xs * L::XSLOT;
            prep_x<F, NT, P, XBF16, CW>(reinterpret_cast<uint2 *>(slot), reinterpret_cast<float *>(slot + L::XS),
                                        sxraw + rs * L::XRAW, N, warp, lane);
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&xfull[xs]);
                mbar_arrive(&rxempty[rs]);
            }
            return true;
        };
        bool ok = nloc == 0 || build_share(0);
        for (int c = 0; c < nloc && ok; ++c) {
            if (c + 1 < nloc && !build_share(c + 1)) break;   // one chunk ahead
            const int s = c % S, xs = c % XR;
            const int cg = c_begin + c;
            const int woff = F == Q6_K ? ((210 * cg) & 15) : 0;
            // weights of chunk c; this warp's scale rows; everyone's X
            // fragments of chunk c
            if (!__all_sync(0xffffffffu, gwait(abort_flag, &full[s], (c / S) & 1, wait_limit))) break;
            const uint8_t *raw = sstage + s * L::STAGE;
            prep_scales<F>(sct, raw, woff, warp, lane);
            __syncwarp();
            // warp-uniform decisions: mma.sync below must run on all 32 lanes
            if (!__all_sync(0xffffffffu, gwait(abort_flag, &xfull[xs], (c / XR) & 1, wait_limit) && !*abort_flag))
                break;
            const uint8_t *pg = raw + rg * L::WIN + woff;
            const uint8_t *slot = sxr + xs * L::XSLOT;
            const uint8_t *xb = slot + 8 * lane;
            const float *sxl = reinterpret_cast<const float *>(slot + L::XS);
            if (F == Q6_K && (woff & 2))
                compute_chunk<F, NT, P, true, NT * 256, 256>(acc[0], pg, pg + 8 * L::WIN, xb, sct, rg, sxl, t);
            else
                compute_chunk<F, NT, P, false, NT * 256, 256>(acc[0], pg, pg + 8 * L::WIN, xb, sct, rg, sxl, t);
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&empty[s]);
                mbar_arrive(&xempty[xs]);
            }
        }
    }

    const bool aborted = *abort_flag != 0u;
    finish_tile<NT, P, CW, 1>(acc, sred, Y, M, N, m0, KS, aborted, warp, lane, amax.keys);
    amax_last_cta(amax, N);
    if (threadIdx.x == 0 && aborted) report_status(status, kStatusTimeout);
}

// ---------------------------------------------------------------------------
// Resident-X variant for a single MMA column tile (P * N <= 8 columns: the
// decode GEMV and a few tokens).  The B fragments of the CTA's whole K slice
// are built once, straight from global X, while the first weight stages are
// in flight; after that the compute warps only wait for weights.  Lanes of
// MMA columns past the used ones read a zero area with the same stride, so
// every fragment load is a plain shared load with a compile-time offset.
// ---------------------------------------------------------------------------
template <int F, int NC, int CW, int RG> struct GR {
    static constexpr int ROWS = 16 * CW * RG;                // RG groups of 16 rows per compute warp
    static constexpr int WARP_TMA = CW;
    static constexpr int THREADS = (CW + 1) * 32;
    static constexpr int WIN = GWin<F>::bytes;
    static constexpr int STAGE = ROWS * WIN;                 // multiple of 1024
    static constexpr int S = CW * RG >= 8 ? 2 : 3;           // weight stages
    static constexpr int XRES = 16384;                       // resident B fragments
    static constexpr int KSB = NC * 32;                      // fragment bytes per k-step
    static constexpr int MAXC = XRES / (16 * KSB);           // chunks a CTA may own
    static constexpr int ZB = NC < 8 ? 16 * KSB : 0;         // zero fragments (unused columns)
    static constexpr int SXB = kmin_fmt(F) ? MAXC * 8 * 16 * 4 : 0;   // Q4_K/Q5_K sub-block sums of x
    static constexpr int SCT = ROWS * SCW * 4;
    static constexpr int OFF_STAGE = 0;
    static constexpr int OFF_X = S * STAGE;
    static constexpr int OFF_Z = OFF_X + XRES;
    static constexpr int OFF_SX = OFF_Z + ZB;
    static constexpr int OFF_SCT = OFF_SX + SXB;
    // The raw X slice [N][K slice] lands in the fragment area itself: it has
    // the same size (P * N columns of 2-byte pieces = N rows of 4/P-byte
    // elements) and is converted in place (all reads, barrier, all writes).
    static constexpr int OFF_XRAW = OFF_X;
    static constexpr int OFF_RED = OFF_X;                    // reused after the last chunk
    static constexpr int OFF_BAR = OFF_SCT + SCT;
    static constexpr int OFF_MISC = OFF_BAR + (2 * S + 1) * 8;
    static constexpr int SMEM = OFF_MISC + 16 + 1024;
    static constexpr int MINB = 232448 / SMEM >= 4 ? 4 : (232448 / SMEM >= 1 ? 232448 / SMEM : 1);
    static_assert(ROWS * 16 * 4 <= XRES, "reduction buffer fits in the fragment area");
    static_assert(STAGE % 1024 == 0 && OFF_BAR % 8 == 0, "alignment");
    static_assert(SMEM <= 232448, "shared memory");
};

template <int F, int NC, int P, bool XBF16, int CW, int RG>
__global__ void __launch_bounds__(GR<F, NC, CW, RG>::THREADS, GR<F, NC, CW, RG>::MINB)
    gemv_res_kernel(const __grid_constant__ GemvSegs segs, const void *__restrict__ Xv, int K, int N, int cps,
                    unsigned *status, uint64_t wait_limit, AmaxOut amax) {
    using L = GR<F, NC, CW, RG>;
    constexpr int S = L::S;
    extern __shared__ uint8_t smem_dyn[];
    uint8_t *smem = smem_dyn + ((1024u - (smem_u32(smem_dyn) & 1023u)) & 1023u);
    uint8_t *sstage = smem + L::OFF_STAGE;
    uint8_t *sfrag = smem + L::OFF_X;
    uint8_t *szero = smem + L::OFF_Z;
    float *ssx = reinterpret_cast<float *>(smem + L::OFF_SX);
    float *sct = reinterpret_cast<float *>(smem + L::OFF_SCT);
    float *sred = reinterpret_cast<float *>(smem + L::OFF_RED);
    const uint8_t *sxraw = smem + L::OFF_XRAW;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::OFF_BAR);
    uint64_t *empty = full + S;
    uint64_t *xfull = empty + S;
    volatile unsigned *abort_flag = reinterpret_cast<volatile unsigned *>(smem + L::OFF_MISC);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // this CTA's weight matrix (segment) and tile within it
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
    constexpr int XES = XBF16 ? 2 : 4;
    const int kslice = nloc * KC;   // elements of the K slice

    float acc[RG][1][4];
#pragma unroll
    for (int q = 0; q < RG; ++q) acc[q][0][0] = acc[q][0][1] = acc[q][0][2] = acc[q][0][3] = 0.f;
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
                    // Weights are read before the preceding kernel on the
                    // stream has finished (they must not be written by it);
                    // X only after it.
                    pdl_wait();
                    // the X slice, one contiguous row piece per token (16-byte
                    // aligned: K and the slice start are multiples of 256)
                    const uint32_t rowb = (uint32_t)kslice * XES;
                    mbar_arrive_expect_tx(xfull, rowb * (uint32_t)N);
                    for (int n = 0; n < N; ++n)
                        tma_load_1d(smem + L::OFF_XRAW + n * rowb,
                                    static_cast<const uint8_t *>(Xv) + ((int64_t)n * K + (int64_t)c_begin * KC) * XES,
                                    rowb, xfull);
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
        // ---- B fragments of the slice, converted in place from the staged X:
        // item it = (ks * NC + col) * 4 + t; every thread first reads all of
        // its items into registers, then (after a barrier) writes them ----
        pdl_wait();   // Y is written below: order after the preceding kernel
        const int tid = threadIdx.x;
        const bool x_ok = nloc == 0 || __all_sync(0xffffffffu, gwait(abort_flag, xfull, 0, wait_limit));
        constexpr int IPT = (L::MAXC * 16 * NC * 4 + CW * 32 - 1) / (CW * 32);   // items per thread, at most
        const int nitems = nloc * 16 * NC * 4;
        uint2 fr[IPT];
#pragma unroll
        for (int i = 0; i < IPT; ++i) {
            const int it = tid + i * CW * 32;
            fr[i] = make_uint2(0u, 0u);
            if (x_ok && it < nitems) {
                const int t = it & 3, col = (it >> 2) % NC, ks = (it >> 2) / NC;
                const int n = col / P, p = col % P;
                if (n < N) {
                    const int e = n * kslice + 16 * ks + 4 * t;
                    if constexpr (XBF16) {
                        fr[i] = *reinterpret_cast<const uint2 *>(sxraw + 2 * e);
                    } else {
                        const float4 f = *reinterpret_cast<const float4 *>(sxraw + 4 * e);
                        const uint32_t hi01 = pack_bf16x2(f.x, f.y), hi23 = pack_bf16x2(f.z, f.w);
                        if (P == 1 || p == 0) {
                            fr[i] = make_uint2(hi01, hi23);
                        } else {
                            fr[i].x = pack_bf16x2(f.x - __uint_as_float(hi01 << 16),
                                                  f.y - __uint_as_float(hi01 & 0xFFFF0000u));
                            fr[i].y = pack_bf16x2(f.z - __uint_as_float(hi23 << 16),
                                                  f.w - __uint_as_float(hi23 & 0xFFFF0000u));
                        }
                    }
                }
            }
        }
        if constexpr (kmin_fmt(F)) {
            // ssx[c][s][n] = sum of x[n] over sub-block s of local chunk c (separate area)
            for (int it = tid; it < nloc * 128; it += CW * 32) {
                const int n = it & 15, sb = (it >> 4) & 7, c = it >> 7;
                float a = 0.f;
                if (x_ok && n < N) {
                    const int e = n * kslice + c * KC + 32 * sb;
                    if constexpr (XBF16) {
                        const uint4 *x = reinterpret_cast<const uint4 *>(sxraw + 2 * e);
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const uint4 u = x[q];
                            a += (__uint_as_float(u.x << 16) + __uint_as_float(u.x & 0xFFFF0000u)) +
                                 (__uint_as_float(u.y << 16) + __uint_as_float(u.y & 0xFFFF0000u));
                            a += (__uint_as_float(u.z << 16) + __uint_as_float(u.z & 0xFFFF0000u)) +
                                 (__uint_as_float(u.w << 16) + __uint_as_float(u.w & 0xFFFF0000u));
                        }
                    } else {
                        const float4 *x = reinterpret_cast<const float4 *>(sxraw + 4 * e);
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const float4 v = x[q];
                            a += (v.x + v.y) + (v.z + v.w);
                        }
                    }
                }
                ssx[it] = a;
            }
        }
        asm volatile("bar.sync 1, %0;" ::"r"(CW * 32) : "memory");   // every raw read is done
#pragma unroll
        for (int i = 0; i < IPT; ++i) {
            const int it = tid + i * CW * 32;
            if (it < nitems) *reinterpret_cast<uint2 *>(sfrag + 8 * it) = fr[i];
        }
        for (int it = tid; it < L::ZB / 8; it += CW * 32) *reinterpret_cast<uint2 *>(szero + 8 * it) = make_uint2(0u, 0u);
        asm volatile("bar.sync 1, %0;" ::"r"(CW * 32) : "memory");   // compute warps only

        const int g = lane >> 2, t = lane & 3;
        const uint8_t *xb0 = g < NC ? sfrag + 8 * (4 * g + t) : szero + 8 * t;
        const int cstride = g < NC ? 16 * L::KSB : 0;
        for (int c = 0; c < nloc && x_ok; ++c) {
            const int s = c % S;
            const int cg = c_begin + c;
            const int woff = F == Q6_K ? ((210 * cg) & 15) : 0;
            if (!__all_sync(0xffffffffu, gwait(abort_flag, &full[s], (c / S) & 1, wait_limit) && !*abort_flag))
                break;
            const uint8_t *raw = sstage + s * L::STAGE;
#pragma unroll
            for (int q = 0; q < RG; ++q) prep_scales<F>(sct, raw, woff, RG * warp + q, lane);
            __syncwarp();
            const uint8_t *xb = xb0 + c * cstride;
            const float *sxl = ssx + c * 128;
            // the RG row groups are independent MMA chains (and share the
            // B fragments), which the scheduler interleaves
#pragma unroll
            for (int q = 0; q < RG; ++q) {
                const int rg = 16 * (RG * warp + q) + g;
                const uint8_t *pg = raw + rg * L::WIN + woff;
                if (F == Q6_K && (woff & 2))
                    compute_chunk<F, 1, P, true, L::KSB, 0>(acc[q], pg, pg + 8 * L::WIN, xb, sct, rg, sxl, t);
                else
                    compute_chunk<F, 1, P, false, L::KSB, 0>(acc[q], pg, pg + 8 * L::WIN, xb, sct, rg, sxl, t);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
    }

    const bool aborted = *abort_flag != 0u;
    finish_tile<1, P, CW, RG>(acc, sred, Y, M, N, m0, KS, aborted, warp, lane, amax.keys);
    amax_last_cta(amax, N);
    if (threadIdx.x == 0 && aborted) report_status(status, kStatusTimeout);
}

// x_arg: the kernel's second parameter (X tensor map or X address).
struct GemvCall {
    const GemvSegs *segs;
    const CUtensorMap *xmap;
    const void *X;
    int64_t K;
    int N;
    GemvPlan plan;
    bool pdl;
    unsigned *status;
    uint64_t limit;
    cudaStream_t st;
    AmaxOut amax;               // argmax mode when amax.keys is not null
};

template <int F, int NT, int P, bool XBF16, int CW>
cudaError_t launch_ring(const GemvCall &c) {
    using L = GL<F, NT, CW>;
    if (c.plan.rows != L::ROWS) return cudaErrorInvalidValue;   // must match the weight map's box
    auto kern = gemv_mma_kernel<F, NT, P, XBF16, CW>;
    static std::atomic<uint64_t> configured{0};
    cudaError_t e = set_smem_once(kern, L::SMEM, configured);
    if (e != cudaSuccess) return e;
    GemvSegs sg = *c.segs;
    const int64_t tiles = set_tiles(sg, L::ROWS);
    return launch_cluster(kern, L::SMEM, L::THREADS, tiles, c.plan.ks, (int)(c.K / KC), c.st, c.pdl, sg, *c.xmap, c.K,
                          c.N, c.status, c.limit, c.amax);
}

template <int F, int NC, int P, bool XBF16, int CW, int RG>
cudaError_t launch_res(const GemvCall &c) {
    using L = GR<F, NC, CW, RG>;
    if (c.plan.rows != L::ROWS) return cudaErrorInvalidValue;   // must match the weight map's box
    const int nchunks = (int)(c.K / KC);
    if ((nchunks + c.plan.ks - 1) / c.plan.ks > L::MAXC) return cudaErrorInvalidValue;
    auto kern = gemv_res_kernel<F, NC, P, XBF16, CW, RG>;
    static std::atomic<uint64_t> configured{0};
    cudaError_t e = set_smem_once(kern, L::SMEM, configured);
    if (e != cudaSuccess) return e;
    GemvSegs sg = *c.segs;
    const int64_t tiles = set_tiles(sg, L::ROWS);
    return launch_cluster(kern, L::SMEM, L::THREADS, tiles, c.plan.ks, nchunks, c.st, c.pdl, sg, c.X, c.K, c.N,
                          c.status, c.limit, c.amax);
}

template <int F, int NC, int P, bool XBF16>
cudaError_t launch_res_tile(const GemvCall &c) {
    if (c.plan.rows == 64) return launch_res<F, NC, P, XBF16, 4, 1>(c);
    if (c.plan.rows == 128)
        return c.plan.rg == 2 ? launch_res<F, NC, P, XBF16, 4, 2>(c) : launch_res<F, NC, P, XBF16, 8, 1>(c);
    return launch_res<F, NC, P, XBF16, 8, 2>(c);
}

template <int F, int NT, int P, bool XBF16>
cudaError_t launch_cw(const GemvCall &c) {
    if (c.plan.resident) {
        if (NT != 1) return cudaErrorInvalidValue;
        return P * c.N == 1 ? launch_res_tile<F, 1, P, XBF16>(c) : launch_res_tile<F, 2, P, XBF16>(c);
    }
    if (c.plan.rows == 128) return launch_ring<F, NT, P, XBF16, 8>(c);
    return launch_ring<F, NT, P, XBF16, 4>(c);
}

template <int F, bool XBF16>
cudaError_t launch_f(const GemvCall &c) {
    constexpr int P = XBF16 ? 1 : 2;
    const int nt = (P * c.N + 7) / 8;
    if constexpr (XBF16) {
        if (nt <= 1) return launch_cw<F, 1, 1, true>(c);
        return launch_cw<F, 2, 1, true>(c);
    } else {
        switch (nt) {
        case 1: return launch_cw<F, 1, 2, false>(c);
        case 2: return launch_cw<F, 2, 2, false>(c);
        case 3: return launch_cw<F, 3, 2, false>(c);
        default: return launch_cw<F, 4, 2, false>(c);
        }
    }
}

}  // namespace

int plan_ks_host(int64_t tiles, int nchunks, int num_sms, int max_cps, int force) {
    return plan_ks(tiles, nchunks, num_sms, max_cps, force);
}

int gemv_tile_rows(int64_t M, int num_sms) {
    // 128-row tiles (8 compute warps) once there are enough rows to fill the
    // GPU twice over without a K split; 64-row tiles otherwise.
    return M >= (int64_t)128 * 2 * num_sms ? 128 : 64;
}

int gemv_window_bytes(int fmt) {
    switch (fmt) {
    case Q8_0: return GWin<Q8_0>::bytes;
    case Q4_0: return GWin<Q4_0>::bytes;
    case Q4_K: return GWin<Q4_K>::bytes;
    case Q6_K: return GWin<Q6_K>::bytes;
    case Q5_K: return GWin<Q5_K>::bytes;
    default: return 0;
    }
}

GemvPlan plan_gemv(int64_t M, int64_t K, int N, int xbf16, int num_sms, const GemvTuning &tun) {
    GemvPlan p{};
    const int cols = (xbf16 ? 1 : 2) * N;
    const int nchunks = (int)(K / KC);
    int rows = tun.rows ? tun.rows : gemv_tile_rows(M, num_sms);
    if (tun.resident && cols <= 2) {
        // MAXC of the resident layout: 16 KB of fragments, cols * 32 bytes per k-step
        const int maxc = 16384 / (16 * 32 * cols);
        const int rg = rows == 256 ? 2 : (rows == 128 ? (tun.rg == 2 ? 2 : 1) : 1);
        const int64_t tiles = (M + rows - 1) / rows;
        const int ks = plan_ks(tiles, nchunks, num_sms, maxc, tun.ks);
        if (ks > 0) {
            p.resident = 1;
            p.rows = rows;
            p.rg = rg;
            p.ks = ks;
            return p;
        }
    }
    p.resident = 0;
    p.rows = rows >= 128 ? 128 : 64;
    p.rg = 1;
    p.ks = plan_ks((M + p.rows - 1) / p.rows, nchunks, num_sms, 0, tun.ks);
    return p;
}

cudaError_t launch_gemv_mma(int fmt, const GemvPlan &plan, const GemvSegs &segs, const CUtensorMap &xmap,
                            const void *X, int xbf16, int64_t K, int N, bool pdl, unsigned *status, uint64_t limit,
                            cudaStream_t st, unsigned long long *amax_ws, int32_t *idx, float *val) {
    if (N < 1 || N > 16 || plan.ks < 1 || plan.ks > 8) return cudaErrorInvalidValue;
    if (segs.nseg < 1 || segs.nseg > QMM_MAX_SEGS || (amax_ws && segs.nseg != 1)) return cudaErrorInvalidValue;
    const AmaxOut amax{amax_ws, amax_ws ? reinterpret_cast<unsigned *>(amax_ws + N) : nullptr, idx, val};
    const GemvCall c{&segs, &xmap, X, K, N, plan, pdl, status, limit, st, amax};
    switch (fmt) {
    case Q8_0: return xbf16 ? launch_f<Q8_0, true>(c) : launch_f<Q8_0, false>(c);
    case Q4_0: return xbf16 ? launch_f<Q4_0, true>(c) : launch_f<Q4_0, false>(c);
    case Q4_K: return xbf16 ? launch_f<Q4_K, true>(c) : launch_f<Q4_K, false>(c);
    case Q6_K: return xbf16 ? launch_f<Q6_K, true>(c) : launch_f<Q6_K, false>(c);
    case Q5_K: return xbf16 ? launch_f<Q5_K, true>(c) : launch_f<Q5_K, false>(c);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace qmm
