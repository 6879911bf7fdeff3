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
#include <atomic>

#include "common.cuh"
#include "kernels.h"

namespace qmm {
namespace {

constexpr int KC = 256;                // weights per chunk
constexpr int SCW = 16;                // scale-table row: 16 floats, 16-byte chunks XOR-swizzled by row

// Index of scale entry e (0..15) of row r in the scale table; chunk (e/4) is
// swizzled with bits 1..2 of the row so that the 8 row groups of a warp hit
// distinct banks on 16-byte loads.
__host__ __device__ constexpr int sct_index(int r, int e) {
    return r * SCW + (((e >> 2) ^ ((r >> 1) & 3)) << 2) + (e & 3);
}

template <int F> struct GWin;
template <> struct GWin<Q8_0> { static constexpr int bytes = 272; };
template <> struct GWin<Q4_0> { static constexpr int bytes = 144; };
template <> struct GWin<Q4_K> { static constexpr int bytes = 144; };
template <> struct GWin<Q6_K> { static constexpr int bytes = 240; };

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
    static constexpr int SXB = F == Q4_K ? 8 * 16 * 4 : 0;     // Q4_K sub-block sums of x
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
    static_assert(XR * XSLOT >= ROWS * 16 * 4, "reduction buffer fits in the X ring");
    static_assert(XSLOT % 16 == 0 && STAGE % 1024 == 0 && XRAW % 1024 == 0, "alignment");
    static_assert(SMEM <= 232448, "shared memory");
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
__device__ __forceinline__ uint32_t ld32(const uint8_t *p) { return *reinterpret_cast<const uint32_t *>(p); }
// Four bytes at p with p % 4 == 2 (known at compile time by the caller).
__device__ __forceinline__ uint32_t ld32_off2(const uint8_t *p) {
    const uint32_t *q = reinterpret_cast<const uint32_t *>(p - 2);
    return __byte_perm(q[0], q[1], 0x5432u);
}
template <bool MIS>
__device__ __forceinline__ uint32_t ldw(const uint8_t *p) { return MIS ? ld32_off2(p) : ld32(p); }

// (a0, a1) += (s0, s1) * (d0, d1), one packed f32x2 FMA.
__device__ __forceinline__ void ffma2(float &a0, float &a1, float s0, float s1, float d0, float d1) {
    asm("{\n\t.reg .b64 ra, rb, rc;\n\t"
        "mov.b64 ra, {%2,%3};\n\tmov.b64 rb, {%4,%5};\n\tmov.b64 rc, {%0,%1};\n\t"
        "fma.rn.f32x2 rc, ra, rb, rc;\n\tmov.b64 {%0,%1}, rc;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "f"(s0), "f"(s1), "f"(d0), "f"(d1));
}

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
    if constexpr (F == Q4_K) {
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
        } else if constexpr (F == Q4_K) {
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

// Entries e0..e0+7 (e0 a multiple of 8) of row r of the scale table.
__device__ __forceinline__ void ld_scales8(float (&v)[8], const float *sct, int r, int e0) {
    const float4 a = *reinterpret_cast<const float4 *>(sct + sct_index(r, e0));
    const float4 b = *reinterpret_cast<const float4 *>(sct + sct_index(r, e0 + 4));
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// ---------------------------------------------------------------------------
// Chunk compute for one warp: 16 rows (g, g+8 per thread) x 256 weights.
// Row windows start 16-byte aligned (Q6_K: + woff, even); every 32-bit code
// word is read with its alignment known at compile time (MIS: woff % 4 == 2).
// ---------------------------------------------------------------------------
template <int F, int NT, int P, bool MIS>
__device__ __forceinline__ void compute_chunk(float (&acc)[NT][4], const uint8_t *rg, const uint8_t *rg8,
                                              const uint2 *xs, const float *sct, int r, const float *sx, int lane,
                                              int t) {
    if constexpr (F == Q4_0) {
        float sg[8], sg8[8];
        ld_scales8(sg, sct, r, 0);
        ld_scales8(sg8, sct, r + 8, 0);
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
                afrag<0x43u, C136>(a0, wg & 0x0F0F0F0Fu, wg8 & 0x0F0F0F0Fu);
                afrag<0x43u, C136>(a1, (wg >> 4) & 0x0F0F0F0Fu, (wg8 >> 4) & 0x0F0F0F0Fu);
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    float d[4] = {0.f, 0.f, 0.f, 0.f};
                    mma16816(d, a0, xs[((2 * b) * NT + j) * 32 + lane]);
                    mma16816(d, a1, xs[((2 * b + 1) * NT + j) * 32 + lane]);
                    acc_scaled(acc[j], d, sg[b], sg8[b]);
                }
            }
        }
    } else if constexpr (F == Q8_0) {
        float sg[8], sg8[8];
        ld_scales8(sg, sct, r, 0);
        ld_scales8(sg8, sct, r + 8, 0);
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
                acc_scaled(acc[j], d, sg[b], sg8[b]);
            }
        }
    } else if constexpr (F == Q4_K) {
        float dsg[8], dsg8[8], dmg[8], dmg8[8];
        ld_scales8(dsg, sct, r, 0);
        ld_scales8(dsg8, sct, r + 8, 0);
        ld_scales8(dmg, sct, r, 8);
        ld_scales8(dmg8, sct, r + 8, 8);
        const uint8_t *qg = rg + 16, *qg8 = rg8 + 16;
#pragma unroll
        for (int pr = 0; pr < 4; ++pr) {            // sub-blocks 2pr (low nibbles), 2pr+1 (high)
            const uint32_t w0g = ld32(qg + 32 * pr + 4 * t), w1g = ld32(qg + 32 * pr + 16 + 4 * t);
            const uint32_t w0g8 = ld32(qg8 + 32 * pr + 4 * t), w1g8 = ld32(qg8 + 32 * pr + 16 + 4 * t);
#pragma unroll
            for (int hn = 0; hn < 2; ++hn) {
                const int s = 2 * pr + hn, sh = 4 * hn;
                uint32_t a0[4], a1[4];
                afrag<0x43u, C128>(a0, (w0g >> sh) & 0x0F0F0F0Fu, (w0g8 >> sh) & 0x0F0F0F0Fu);
                afrag<0x43u, C128>(a1, (w1g >> sh) & 0x0F0F0F0Fu, (w1g8 >> sh) & 0x0F0F0F0Fu);
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    float d[4] = {0.f, 0.f, 0.f, 0.f};
                    mma16816(d, a0, xs[((2 * s) * NT + j) * 32 + lane]);
                    mma16816(d, a1, xs[((2 * s + 1) * NT + j) * 32 + lane]);
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
    } else {  // Q6_K: element e = 128h + 32J + l, l = 16 lh + 4t + i, k-step G = 8h + 2J + lh
        float sg[16], sg8[16];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float4 a = *reinterpret_cast<const float4 *>(sct + sct_index(r, 4 * q));
            const float4 b = *reinterpret_cast<const float4 *>(sct + sct_index(r + 8, 4 * q));
            sg[4 * q] = a.x; sg[4 * q + 1] = a.y; sg[4 * q + 2] = a.z; sg[4 * q + 3] = a.w;
            sg8[4 * q] = b.x; sg8[4 * q + 1] = b.y; sg8[4 * q + 2] = b.z; sg8[4 * q + 3] = b.w;
        }
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
                    afrag<0x43u, C160>(a, qg, qg8);
#pragma unroll
                    for (int j = 0; j < NT; ++j) {
                        float d[4] = {0.f, 0.f, 0.f, 0.f};
                        mma16816(d, a, xs[(G * NT + j) * 32 + lane]);
                        acc_scaled(acc[j], d, sg[G], sg8[G]);
                    }
                }
            }
        }
    }
}

template <int F, int NT, int P, bool XBF16, int CW>
__global__ void __launch_bounds__(GL<F, NT, CW>::THREADS)
    gemv_mma_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap xmap, int M, int K,
                    int N, float *__restrict__ Y, int cps, unsigned *status, uint64_t wait_limit) {
    using L = GL<F, NT, CW>;
    constexpr int S = L::S, XR = L::XR, ROWS = L::ROWS;
    extern __shared__ uint8_t smem_dyn[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~(uintptr_t)1023);
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
    const int m0 = blockIdx.x * ROWS;
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

    float acc[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;

    if (warp == L::WARP_TMA) {
        // ---------------- TMA producers: lane 0 weights, lane 1 raw X ----------------
        const uint64_t drain_limit = wait_limit < (1ull << 31) ? (1ull << 31) : wait_limit;
        if (lane == 0) {
            prefetch_tensormap(&wmap);
            int issued = 0;   // loads are issued in chunk order 0, 1, ..., issued-1
            for (int c = 0; c < nloc; ++c) {
                const int s = c % S;
                if (c >= S && !gwait(abort_flag, &empty[s], ((c / S) - 1) & 1, wait_limit)) break;
                if (*abort_flag) break;
                const int cg = c_begin + c;
                const int xb = F == Q6_K ? ((210 * cg) & ~15) : cg * L::WIN;
                mbar_arrive_expect_tx(&full[s], (uint32_t)L::RAWW);
                tma_load_2d(sstage + s * L::STAGE, &wmap, &full[s], xb >> 1, m0);
                issued = c + 1;
            }
            if (*abort_flag)   // drain: the last load issued into each stage
                for (int c = issued - S < 0 ? 0 : issued - S; c < issued; ++c)
                    (void)mbar_wait(&full[c % S], (c / S) & 1, drain_limit);
        } else if (lane == 1) {
            prefetch_tensormap(&xmap);
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
            const uint2 *xsl = reinterpret_cast<const uint2 *>(slot);
            const float *sxl = reinterpret_cast<const float *>(slot + L::XS);
            if (F == Q6_K && (woff & 2))
                compute_chunk<F, NT, P, true>(acc, pg, pg + 8 * L::WIN, xsl, sct, rg, sxl, lane, t);
            else
                compute_chunk<F, NT, P, false>(acc, pg, pg + 8 * L::WIN, xsl, sct, rg, sxl, lane, t);
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&empty[s]);
                mbar_arrive(&xempty[xs]);
            }
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
                        if (r0 < M) Y[(int64_t)n * M + r0] = acc[j][0] + acc[j][1];
                        if (r1 < M) Y[(int64_t)n * M + r1] = acc[j][2] + acc[j][3];
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
        // partials -> shared memory [row][token] (aliases the X ring: wait until
        // every warp of the CTA is done with it); rank 0 of the cluster sums
        __syncthreads();
        if (warp < CW) {
            const int g = lane >> 2, t = lane & 3;
            const int r0 = 16 * warp + g, r1 = r0 + 8;
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                if constexpr (P == 2) {
                    const int n = 4 * j + t;
                    if (n < 16) {
                        sred[r0 * 16 + n] = acc[j][0] + acc[j][1];
                        sred[r1 * 16 + n] = acc[j][2] + acc[j][3];
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

template <int F, int NT, int P, bool XBF16, int CW>
cudaError_t launch_t(const CUtensorMap &wmap, const CUtensorMap &xmap, int64_t M, int64_t K, int N, float *Y,
                     int num_sms, unsigned *status, uint64_t limit, cudaStream_t st) {
    using L = GL<F, NT, CW>;
    constexpr int ROWS = L::ROWS;
    auto kern = gemv_mma_kernel<F, NT, P, XBF16, CW>;
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
    cfg.blockDim = dim3(L::THREADS, 1, 1);
    cfg.dynamicSmemBytes = L::SMEM;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = (unsigned)ksp;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = ksp > 1 ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, kern, wmap, xmap, (int)M, (int)K, N, Y, cps, status, limit);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int F, int NT, int P, bool XBF16>
cudaError_t launch_cw(const CUtensorMap &wmap, const CUtensorMap &xmap, int64_t M, int64_t K, int N, float *Y,
                      int num_sms, unsigned *status, uint64_t limit, cudaStream_t st) {
    if (gemv_tile_rows(M, num_sms) == 128)
        return launch_t<F, NT, P, XBF16, 8>(wmap, xmap, M, K, N, Y, num_sms, status, limit, st);
    return launch_t<F, NT, P, XBF16, 4>(wmap, xmap, M, K, N, Y, num_sms, status, limit, st);
}

template <int F, bool XBF16>
cudaError_t launch_f(const CUtensorMap &wmap, const CUtensorMap &xmap, int64_t M, int64_t K, int N, float *Y,
                     int num_sms, unsigned *status, uint64_t limit, cudaStream_t st) {
    constexpr int P = XBF16 ? 1 : 2;
    const int cols = P * N;
    const int nt = (cols + 7) / 8;
    if constexpr (XBF16) {
        if (nt <= 1) return launch_cw<F, 1, 1, true>(wmap, xmap, M, K, N, Y, num_sms, status, limit, st);
        return launch_cw<F, 2, 1, true>(wmap, xmap, M, K, N, Y, num_sms, status, limit, st);
    } else {
        switch (nt) {
        case 1: return launch_cw<F, 1, 2, false>(wmap, xmap, M, K, N, Y, num_sms, status, limit, st);
        case 2: return launch_cw<F, 2, 2, false>(wmap, xmap, M, K, N, Y, num_sms, status, limit, st);
        case 3: return launch_cw<F, 3, 2, false>(wmap, xmap, M, K, N, Y, num_sms, status, limit, st);
        default: return launch_cw<F, 4, 2, false>(wmap, xmap, M, K, N, Y, num_sms, status, limit, st);
        }
    }
}

}  // namespace

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
    default: return 0;
    }
}

cudaError_t launch_gemv_mma(int fmt, const CUtensorMap &wmap, const CUtensorMap &xmap, int xbf16, int64_t M,
                            int64_t K, int N, float *Y, int num_sms, unsigned *status, uint64_t limit,
                            cudaStream_t st) {
    if (N < 1 || N > 16) return cudaErrorInvalidValue;
    switch (fmt) {
    case Q8_0: return xbf16 ? launch_f<Q8_0, true>(wmap, xmap, M, K, N, Y, num_sms, status, limit, st)
                            : launch_f<Q8_0, false>(wmap, xmap, M, K, N, Y, num_sms, status, limit, st);
    case Q4_0: return xbf16 ? launch_f<Q4_0, true>(wmap, xmap, M, K, N, Y, num_sms, status, limit, st)
                            : launch_f<Q4_0, false>(wmap, xmap, M, K, N, Y, num_sms, status, limit, st);
    case Q4_K: return xbf16 ? launch_f<Q4_K, true>(wmap, xmap, M, K, N, Y, num_sms, status, limit, st)
                            : launch_f<Q4_K, false>(wmap, xmap, M, K, N, Y, num_sms, status, limit, st);
    case Q6_K: return xbf16 ? launch_f<Q6_K, true>(wmap, xmap, M, K, N, Y, num_sms, status, limit, st)
                            : launch_f<Q6_K, false>(wmap, xmap, M, K, N, Y, num_sms, status, limit, st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace qmm
