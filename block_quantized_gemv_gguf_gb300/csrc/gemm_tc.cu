// gemm_tc.cu -- prefill GEMM Y[N,M] = X[N,K] * dequant(W)[M,K]^T on the
// 5th-generation tensor cores (tcgen05), for 16 < N <= 512 tokens.
//
// One CTA computes a 128-row (weights) x BN-column (tokens) tile of Y^T over
// the whole K.  Warp roles (352 threads):
//   warp 0      TMA producer of raw weight bytes: one 2-D tensor copy per
//               256-weight chunk of the tile's 128 rows (u16 view of W);
//   warp 1      TMA producer of bf16 X tiles (64 k x BN tokens, 128-byte
//               swizzle = the canonical K-major UMMA layout);
//   warp 2      TMEM allocation and the single MMA-issuing thread:
//               tcgen05.mma kind::f16, M=128, N=BN, K=16, f32 accumulator;
//   warps 3..10 dequantizers: thread i owns half (32 weights) of weight row
//               i % 128 of each 64-k stage, decodes it straight from the raw
//               bytes to bf16 and writes it swizzled as the K-major A
//               operand (eight warps, so that the per-stage decode latency
//               hides behind the other warps); afterwards the same warps
//               read the accumulator out of TMEM (two warps per lane
//               quarter, half of the columns each) and store Y.
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
constexpr int DQW = 8;                        // dequantizer (and epilogue) warps
constexpr int NUM_THREADS = (3 + DQW) * 32;   // 352
constexpr int WARP_WPROD = 0, WARP_XPROD = 1, WARP_MMA = 2, WARP_DQ0 = 3;

template <int F> struct Raw;
template <> struct Raw<Q8_0> { static constexpr int bytes = 272; };   // 8 blocks of 34
template <> struct Raw<Q4_0> { static constexpr int bytes = 144; };   // 8 blocks of 18
template <> struct Raw<Q4_K> { static constexpr int bytes = 144; };   // 1 super-block
template <> struct Raw<Q6_K> { static constexpr int bytes = 240; };   // 210 B + alignment slack
template <> struct Raw<Q5_K> { static constexpr int bytes = 176; };   // 1 super-block

template <int F, int BN> struct Layout {
    static constexpr int X_BYTES = BN * 128;
    static constexpr int RAW_BYTES = BM * Raw<F>::bytes;
    // The dequantized A operand lives in tensor memory: SA stages of 32
    // columns (64 bf16 per lane = row) after the BN accumulator columns.
    static constexpr int SA = 8;
    static constexpr int TMEM_COLS = 512;
    static constexpr int A_COL0 = BN;
    static_assert(BN + SA * 32 <= TMEM_COLS, "tensor memory");
    // Shared memory: X copies and raw weight chunks.  One weight copy brings
    // a 256-weight chunk of all 128 rows; one X copy brings XG stages (a 3-D
    // box: 64 k x BN tokens x XG k-blocks).
    static constexpr int XG = 1;                            // stages per X copy (measured best)
    static constexpr int XSLOT = XG * X_BYTES;
    static constexpr int BUDGET = 227 * 1024 - 2048;
    static constexpr int SR = BUDGET - 2 * XSLOT >= 4 * RAW_BYTES ? 4 : (BUDGET - 2 * XSLOT >= 3 * RAW_BYTES ? 3 : 2);
    static constexpr int SX_FIT = (BUDGET - SR * RAW_BYTES) / XSLOT;
    static constexpr int SX = SX_FIT >= 8 ? 8 : (SX_FIT >= 4 ? 4 : SX_FIT);   // X copies in flight
    static_assert(SX >= 2, "at least two X slots");
    static constexpr int OFF_X = 0;
    static constexpr int OFF_RAW = OFF_X + SX * XSLOT;
    static constexpr int OFF_BAR = OFF_RAW + SR * RAW_BYTES;
    // raw_full/empty[SR], x_full/empty[SX], a_full/empty[SA], acc_full
    static constexpr int NUM_BARS = 2 * SR + 2 * SX + 2 * SA + 1;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
    static constexpr int TOTAL = OFF_MISC + 64;
    static constexpr int SMEM = TOTAL + 1024;     // 1024-byte alignment slack
    static_assert(SMEM <= 232448, "shared memory budget");
    // K split: the slice partials (BM x BN f32) reuse the X and raw areas
    static_assert(BM * BN * 4 <= OFF_BAR, "split-K partials fit below the barriers");
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

// Cluster-wide barrier (every thread of every CTA of the cluster arrives).
__device__ __forceinline__ void cluster_sync_epi() { cluster_sync_all(); }

// 16 bytes of CTA `rank`'s shared memory at the offset of `local`.
__device__ __forceinline__ float4 ld_dsmem_f32x4(const float4 *local, uint32_t rank) {
    const uint32_t ra = cluster_addr(local, rank);
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(ra)
                 : "memory");
    return v;
}

// Drain wait: used after an abort for copies this thread issued itself;
// those complete on their own, so only the time limit applies.
__device__ __forceinline__ void drain(uint64_t *bar, uint32_t parity, uint64_t limit) {
    (void)mbar_wait(bar, parity, limit);
}

// ---------------------------------------------------------------------------
// Dequantization.  The integer codes are turned into floats 128 + v (or
// 32768 + v) by byte permutes into the mantissa of a constant, and the
// offset is folded into a per-block constant:
//     w = scale * (128 + v) - scale * (128 + offset).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void q4k_sm(const uint8_t *S, int s, float &sc, float &mn) {
    if (s < 4) {
        sc = (float)(S[s] & 63);
        mn = (float)(S[s + 4] & 63);
    } else {
        sc = (float)((S[s + 4] & 15) | ((S[s - 4] >> 6) << 4));
        mn = (float)((S[s + 4] >> 4) | ((S[s] >> 6) << 4));
    }
}

// ---------------------------------------------------------------------------
// Half of a stage: 32 weights (k = 32h .. 32h+31 of the 64-k stage `sub`) of
// one row, straight from the raw bytes to 16 bf16x2 words in k order.
// ---------------------------------------------------------------------------
template <int F>
__device__ __forceinline__ void dequant32(const uint8_t *rb, int sub, int h, uint32_t (&o)[16]);

template <>
__device__ __forceinline__ void dequant32<Q4_0>(const uint8_t *rb, int sub, int h, uint32_t (&o)[16]) {
    const uint8_t *b = rb + 18 * (2 * sub + h);
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
    for (int e = 0; e < 16; ++e) o[e] = pack_bf16x2(w[2 * e], w[2 * e + 1]);
}

template <>
__device__ __forceinline__ void dequant32<Q8_0>(const uint8_t *rb, int sub, int h, uint32_t (&o)[16]) {
    const uint8_t *b = rb + 34 * (2 * sub + h);
    const float d = f16_bits(*reinterpret_cast<const uint16_t *>(b));
    const float c = -32896.f * d;  // exact: d * (32768 + q + 128) - 32896 d = d q
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        const uint32_t u = lds_u32_a2(b + 2 + 4 * t) ^ 0x80808080u;
        const float f0 = __uint_as_float(__byte_perm(u, 0x47000000u, 0x7504u));
        const float f1 = __uint_as_float(__byte_perm(u, 0x47000000u, 0x7514u));
        const float f2 = __uint_as_float(__byte_perm(u, 0x47000000u, 0x7524u));
        const float f3 = __uint_as_float(__byte_perm(u, 0x47000000u, 0x7534u));
        o[2 * t] = pack_bf16x2(fmaf(d, f0, c), fmaf(d, f1, c));
        o[2 * t + 1] = pack_bf16x2(fmaf(d, f2, c), fmaf(d, f3, c));
    }
}

template <>
__device__ __forceinline__ void dequant32<Q4_K>(const uint8_t *rb, int sub, int h, uint32_t (&o)[16]) {
    const float d = f16_bits(*reinterpret_cast<const uint16_t *>(rb));
    const float dmin = f16_bits(*reinterpret_cast<const uint16_t *>(rb + 2));
    float sc, mn;
    q4k_sm(rb + 4, 2 * sub + h, sc, mn);
    const float a = d * sc;
    const float c = -(128.f * a + dmin * mn);
    const uint4 *qs = reinterpret_cast<const uint4 *>(rb + 16 + 32 * sub);
    const uint4 q0 = qs[0], q1 = qs[1];
    const uint32_t words[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
    const int sh = 4 * h;   // sub-block 2sub: low nibbles, 2sub+1: high nibbles
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        const uint32_t v = (words[t] >> sh) & 0x0F0F0F0Fu;
        o[2 * t] = pack_bf16x2(fmaf(a, byte_as_128_plus<0>(v), c), fmaf(a, byte_as_128_plus<1>(v), c));
        o[2 * t + 1] = pack_bf16x2(fmaf(a, byte_as_128_plus<2>(v), c), fmaf(a, byte_as_128_plus<3>(v), c));
    }
}

// Q5_K: as Q4_K, with bit s of qh[l] as bit 4 of sub-block s's element l.
template <>
__device__ __forceinline__ void dequant32<Q5_K>(const uint8_t *rb, int sub, int h, uint32_t (&o)[16]) {
    const float d = f16_bits(*reinterpret_cast<const uint16_t *>(rb));
    const float dmin = f16_bits(*reinterpret_cast<const uint16_t *>(rb + 2));
    const int s = 2 * sub + h;
    float sc, mn;
    q4k_sm(rb + 4, s, sc, mn);
    const float a = d * sc;
    const float c = -(128.f * a + dmin * mn);
    const uint4 *qh = reinterpret_cast<const uint4 *>(rb + 16);
    const uint4 *qs = reinterpret_cast<const uint4 *>(rb + 48 + 32 * sub);
    const uint4 h0 = qh[0], h1 = qh[1], q0 = qs[0], q1 = qs[1];
    const uint32_t words[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
    const uint32_t hw[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
    const int sh = 4 * h;   // sub-block 2sub: low nibbles, 2sub+1: high nibbles
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        const uint32_t v = ((words[t] >> sh) & 0x0F0F0F0Fu) | (((hw[t] >> s) & 0x01010101u) << 4);
        o[2 * t] = pack_bf16x2(fmaf(a, byte_as_128_plus<0>(v), c), fmaf(a, byte_as_128_plus<1>(v), c));
        o[2 * t + 1] = pack_bf16x2(fmaf(a, byte_as_128_plus<2>(v), c), fmaf(a, byte_as_128_plus<3>(v), c));
    }
}

// Q6_K: rb already points at the super-block (window offset applied).
template <>
__device__ __forceinline__ void dequant32<Q6_K>(const uint8_t *rb, int sub, int h, uint32_t (&o)[16]) {
    const int hh = sub >> 1, jp = sub & 1;
    const int J = 2 * jp + h;                    // e = 128 hh + 32 J + l
    const float d = f16_bits(*reinterpret_cast<const uint16_t *>(rb + 208));
    const int8_t *scl = reinterpret_cast<const int8_t *>(rb + 192);
    const uint8_t *ql = rb + 64 * hh + 32 * h;   // J % 2 == h
    const uint8_t *qh = rb + 128 + 32 * hh;
    const float ds0 = d * (float)scl[8 * hh + 2 * J], ds1 = d * (float)scl[8 * hh + 2 * J + 1];
    const float c0 = -160.f * ds0, c1 = -160.f * ds1;  // exact: ds (128 + q) - 160 ds = ds (q - 32)
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        const uint32_t lw = lds_u32_a2(ql + 4 * t), hw = lds_u32_a2(qh + 4 * t);
        const uint32_t q = ((lw >> (4 * jp)) & 0x0F0F0F0Fu) | (((hw >> (2 * J)) & 0x03030303u) << 4);
        const float a = t < 4 ? ds0 : ds1, c = t < 4 ? c0 : c1;
        o[2 * t] = pack_bf16x2(fmaf(a, byte_as_128_plus<0>(q), c), fmaf(a, byte_as_128_plus<1>(q), c));
        o[2 * t + 1] = pack_bf16x2(fmaf(a, byte_as_128_plus<2>(q), c), fmaf(a, byte_as_128_plus<3>(q), c));
    }
}

template <int F, int BN>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap wmap2,
                   const __grid_constant__ CUtensorMap xmap, int M, int K, int N, int mt0, float *__restrict__ Y1,
                   float *__restrict__ Y2, unsigned *status, uint64_t wait_limit) {
    using L = Layout<F, BN>;
    constexpr int SA = L::SA, SX = L::SX;
    constexpr int RAWB = Raw<F>::bytes;
    extern __shared__ uint8_t smem_dyn[];
    // 1024-byte aligned base derived from the shared array (keeps the
    // accesses below in the shared window)
    uint8_t *smem = smem_dyn + ((1024u - (smem_u32(smem_dyn) & 1023u)) & 1023u);
    uint8_t *sX = smem + L::OFF_X;
    uint8_t *sRaw = smem + L::OFF_RAW;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::OFF_BAR);
    constexpr int SR = L::SR;
    uint64_t *raw_full = bars, *raw_empty = bars + SR;
    uint64_t *x_full = bars + 2 * SR, *x_empty = x_full + SX;
    uint64_t *a_full = x_empty + SX, *ab_empty = a_full + SA;   // ab_empty: A slot consumed by the MMA
    uint64_t *acc_full = ab_empty + SA;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::OFF_MISC);
    unsigned *abort_flag = reinterpret_cast<unsigned *>(smem + L::OFF_MISC + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // With a second matrix (Y2 set: two projections of the same shape that
    // share X, e.g. gate and up), the second half of the grid's x range
    // takes it.
    const int tiles_m = (M + BM - 1) / BM;
    const int mt = mt0 + (int)blockIdx.x;   // this CTA's 128-row tile
    const bool second = Y2 != nullptr && mt >= tiles_m;
    const CUtensorMap *wm = second ? &wmap2 : &wmap;
    float *__restrict__ Y = second ? Y2 : Y1;
    const int m0 = (second ? mt - tiles_m : mt) * BM, n0 = blockIdx.y * BN;
    // K split: the KS CTAs of a (1, 1, KS) cluster take slices of the chunks;
    // rank 0 adds the other slices' partial sums (distributed shared memory,
    // rank order) in the epilogue.
    const int KS = (int)gridDim.z, zr = (int)blockIdx.z;
    const int nkc_all = K / KC;
    const int kc0 = nkc_all * zr / KS, nkc = nkc_all * (zr + 1) / KS - kc0;
    const int nsteps = nkc * (KC / BK);
    // Each CTA walks its chunks starting at its own offset (a rotation): CTAs
    // that run in lockstep then read different X tiles at any moment instead
    // of all hitting the same L2 lines at once.  The k-sum is the same set of
    // terms.
    const int koff = (int)(((unsigned)(m0 / BM) * 5u + blockIdx.y * 3u) % (unsigned)nkc);
    auto kchunk = [&](int c) { return kc0 + (c + koff < nkc ? c + koff : c + koff - nkc); };
    const Ctl ctl{abort_flag, wait_limit};
    const uint64_t drain_limit = wait_limit < (1ull << 31) ? (1ull << 31) : wait_limit;

    if (threadIdx.x == 0) {
        for (int r = 0; r < SR; ++r) {
            mbar_init(&raw_full[r], 1);
            mbar_init(&raw_empty[r], DQW);
        }
        for (int s = 0; s < SX; ++s) {
            mbar_init(&x_full[s], 1);
            mbar_init(&x_empty[s], 1);
        }
        for (int s = 0; s < SA; ++s) {
            mbar_init(&a_full[s], DQW);
            mbar_init(&ab_empty[s], 1);
        }
        mbar_init(acc_full, 1);
        *abort_flag = 0u;
        fence_barrier_init();
    }
    if (warp == WARP_WPROD && lane == 0) prefetch_tensormap(wm);
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
                    xb = (210 * kchunk(c)) & ~15;
                else
                    xb = kchunk(c) * RAWB;
                mbar_arrive_expect_tx(&raw_full[r], (uint32_t)L::RAW_BYTES);
                tma_load_2d(sRaw + r * L::RAW_BYTES, wm, &raw_full[r], xb >> 1, m0);
                issued = c + 1;
            }
            if (*abort_flag)   // drain: the last load issued into each stage
                for (int c = issued - SR < 0 ? 0 : issued - SR; c < issued; ++c)
                    drain(&raw_full[c % SR], (c / SR) & 1, drain_limit);
        }
    } else if (warp == WARP_XPROD) {
        // XL lanes may issue X copies side by side (lane l takes the rounds
        // u = l, l + XL, ...); XL must divide SX, so that every slot belongs to
        // exactly one lane and that lane's waits on it are in its own program
        // order (a parity wait can then never alias a phase two ahead).
        constexpr int XL = 1;   // several lanes were measured slower here; kept general for the lane split
        static_assert(SX % XL == 0, "each X slot owned by one issuing lane");
        if (lane < XL) {
            // Weights stream from the start; X (which may be written by the
            // preceding kernel, e.g. the bf16 conversion) only after it ends.
            pdl_wait();
            int issued = 0;   // X copies (rounds of XG stages) this lane issued: rounds lane + XL*i, i < issued
            constexpr int XG = L::XG;
            const int nrounds = nsteps / XG;
            for (int u = lane; u < nrounds; u += XL) {
                const int s = u % SX;
                if (u >= SX && !wait_ok(ctl, &x_empty[s], ((u / SX) - 1) & 1, wait_limit)) break;
                if (*abort_flag) break;
                mbar_arrive_expect_tx(&x_full[s], (uint32_t)L::XSLOT);   // this CTA's slot s: armed
                const int t0 = u * XG;                                    // first stage of the round
                const int kb = kchunk(t0 / (KC / BK)) * (KC / BK) + t0 % (KC / BK);   // its 64-k block
                tma_load_3d(sX + s * L::XSLOT, &xmap, &x_full[s], 0, n0, kb);
                ++issued;
            }
            if (*abort_flag)   // drain this lane's copies that may still be in flight
                for (int i = 0; i < issued; ++i) {
                    const int u = lane + XL * i;
                    if (u + SX >= lane + XL * issued) drain(&x_full[u % SX], (u / SX) & 1, drain_limit);
                }
        }
    } else if (warp == WARP_MMA) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(BM, BN);
            constexpr int XG = L::XG;
            for (int t = 0; t < nsteps; ++t) {
                const int u = t / XG, j = t % XG, sx = u % SX, sa = t % SA;
                if (j == 0 && !wait_ok(ctl, &x_full[sx], (u / SX) & 1, wait_limit)) break;
                if (!wait_ok(ctl, &a_full[sa], (t / SA) & 1, wait_limit)) break;
                tc_fence_after();
                const uint32_t a0 = tmem_d + (uint32_t)(L::A_COL0 + 32 * sa);   // lane 0, first column
                const uint32_t b0 = smem_u32(sX + sx * L::XSLOT + j * L::X_BYTES);
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk)   // 16 k = 8 columns of A, 32 bytes of a B row
                    umma_bf16_ts(tmem_d, a0 + 8 * kk, sdesc_k_sw128(b0 + 32 * kk), idesc, (t | kk) != 0);
                umma_commit(&ab_empty[sa]);                 // the A slot, for the dequantizers
                if (j == XG - 1) umma_commit(&x_empty[sx]);   // the X copy, for the X producer
            }
            umma_commit(acc_full);   // also on abort: lets the epilogue drain the MMAs
        }
    } else {
        // ---------------- dequantizers, then epilogue ----------------
        // Thread i: row i % 128 of the tile, half i / 128 of each 64-k stage.
        // G stages are decoded per step (one wait, fence and arrival round
        // per G stages).  Measured at N = 512 (14336 x 4096): one stage per
        // step (each stage goes to the MMA as soon as it is in tensor
        // memory) is 2-4% faster for Q4_K, Q5_K and Q8_0; four per step
        // (independent decode chains the scheduler interleaves) is 1% faster
        // for Q4_0 and 8% for Q6_K.
        constexpr int G = (F == Q4_0 || F == Q6_K) ? 4 : 1;
        // warp w may only write TMEM lanes 32 (w % 4) .. +31: row = lane of
        // that quarter; the two warps of a quarter take the two k halves
        const int row_t = 32 * (warp & 3) + lane, hk = (warp - WARP_DQ0) >> 2;
        const uint32_t a_lane = tmem_d + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)(L::A_COL0 + 16 * hk);
        bool ok = true;
        for (int c = 0; c < nkc && ok; ++c) {
            const int r = c % SR;
            // Every lane waits; the vote keeps the decision warp-uniform.
            if (!__all_sync(0xffffffffu, wait_ok(ctl, &raw_full[r], (c / SR) & 1, wait_limit))) {
                ok = false;
                break;
            }
            const uint8_t *rb = sRaw + r * L::RAW_BYTES + row_t * RAWB;
            if constexpr (F == Q6_K) rb += (210 * kchunk(c)) & 15;
#pragma unroll 1
            for (int sub0 = 0; sub0 < KC / BK; sub0 += G) {
                const int t0 = c * (KC / BK) + sub0;
                bool free_ok = true;
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const int t = t0 + g;
                    if (t >= SA) free_ok = free_ok && wait_ok(ctl, &ab_empty[t % SA], ((t / SA) - 1) & 1, wait_limit);
                }
                if (!__all_sync(0xffffffffu, free_ok)) {
                    ok = false;
                    break;
                }
                tc_fence_after();   // the MMAs that read these slots have completed
                uint32_t o[G][16];
#pragma unroll
                for (int g = 0; g < G; ++g) dequant32<F>(rb, sub0 + g, hk, o[g]);
#pragma unroll
                for (int g = 0; g < G; ++g) tmem_st_32x32b_x16(a_lane + 32u * (uint32_t)((t0 + g) % SA), o[g]);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
#pragma unroll
                    for (int g = 0; g < G; ++g) mbar_arrive(&a_full[(t0 + g) % SA]);
            }
            if (!ok) break;
            __syncwarp();
            if (lane == 0) mbar_arrive(&raw_empty[r]);
        }
        // Epilogue: TMEM lane = tile row.  Warp w may only touch lanes 32*(w%4)..+31.
        const bool acc_ok = mbar_wait(acc_full, 0, 2 * drain_limit);
        pdl_wait();   // Y: order after the preceding kernel
        tc_fence_after();
        const bool good = __all_sync(0xffffffffu, acc_ok && !*abort_flag);
        const int q = warp & 3;                      // TMEM lanes 32q .. 32q+31
        const int chalf = (warp - WARP_DQ0) >> 2;    // two warps per lane quarter split the columns
        const int rl = 32 * q + lane, row = m0 + rl;
        // K split: slice partials in shared memory [column / 4][row][4] (the
        // X stage area is free once every MMA has completed)
        float4 *red = reinterpret_cast<float4 *>(sX);
        if (good && (KS == 1 || zr != 0)) {
#pragma unroll 1
            for (int j = chalf * (BN / 32); j < (chalf + 1) * (BN / 32); ++j) {
                uint32_t v[16];
                tmem_ld_32x32b_x16(tmem_d + ((uint32_t)(32 * q) << 16) + 16 * j, v);
                tmem_ld_wait();
                if (KS > 1) {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        red[(4 * j + i) * BM + rl] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                                                 __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
                } else if (row < M) {
#pragma unroll
                    for (int cidx = 0; cidx < 16; ++cidx) {
                        const int n = n0 + 16 * j + cidx;
                        if (n < N) Y[(int64_t)n * M + row] = __uint_as_float(v[cidx]);
                    }
                }
            }
        }
        if (KS > 1) {
            // every CTA of the cluster reaches both barriers, aborted or not
            cluster_sync_epi();
            if (zr == 0 && good) {
#pragma unroll 1
                for (int j = chalf * (BN / 32); j < (chalf + 1) * (BN / 32); ++j) {
                    uint32_t v[16];
                    tmem_ld_32x32b_x16(tmem_d + ((uint32_t)(32 * q) << 16) + 16 * j, v);
                    tmem_ld_wait();
                    float acc[16];
#pragma unroll
                    for (int c = 0; c < 16; ++c) acc[c] = __uint_as_float(v[c]);
                    for (int r = 1; r < KS; ++r) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float4 p = ld_dsmem_f32x4(&red[(4 * j + i) * BM + rl], (uint32_t)r);
                            acc[4 * i] += p.x;
                            acc[4 * i + 1] += p.y;
                            acc[4 * i + 2] += p.z;
                            acc[4 * i + 3] += p.w;
                        }
                    }
                    if (row < M) {
#pragma unroll
                        for (int cidx = 0; cidx < 16; ++cidx) {
                            const int n = n0 + 16 * j + cidx;
                            if (n < N) Y[(int64_t)n * M + row] = acc[cidx];
                        }
                    }
                }
            }
            cluster_sync_epi();   // rank 0 has read every partial: the others may exit
        }
    }
    if (KS > 1 && warp < WARP_DQ0) {
        // the other warps take part in the epilogue's cluster barriers
        __syncwarp();
        cluster_sync_epi();
        cluster_sync_epi();
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
cudaError_t launch_one(const GemmArgs &a, const CUtensorMap &wmap, const CUtensorMap &wmap2, const CUtensorMap &xmap,
                       cudaStream_t st) {
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
    cfg.gridDim = dim3((unsigned)a.mtn, (unsigned)((a.N + BN - 1) / BN), 1);
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = L::SMEM;
    cfg.stream = st;
    cfg.gridDim.z = (unsigned)a.ks;
    cudaLaunchAttribute attr[2];
    unsigned na = 0;
    if (a.ks > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = 1;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = (unsigned)a.ks;
        ++na;
    }
    if (a.pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    e = cudaLaunchKernelEx(&cfg, kern, wmap, wmap2, xmap, (int)a.M, (int)a.K, a.N, a.mt0, a.Y, a.Y2, a.status,
                           a.wait_limit);
    if (e != cudaSuccess) return e;
    return launched(cudaGetLastError());
}

template <int F>
cudaError_t launch_fmt(const GemmArgs &a, const CUtensorMap &wmap, const CUtensorMap &wmap2, const CUtensorMap &xmap,
                       cudaStream_t st) {
    switch (a.bn) {
    case 64: return launch_one<F, 64>(a, wmap, wmap2, xmap, st);
    case 128: return launch_one<F, 128>(a, wmap, wmap2, xmap, st);
    case 256: return launch_one<F, 256>(a, wmap, wmap2, xmap, st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

int gemm_x_stages_per_copy(int) { return 1; }

namespace {
template <int F, int BN>
int cluster_slots_one(int ks) {
    using L = Layout<F, BN>;
    auto kern = gemm_tc_kernel<F, BN>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM) != cudaSuccess) return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, 1, (unsigned)ks);
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = L::SMEM;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = (unsigned)ks;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}
template <int F>
int cluster_slots_fmt(int bn, int ks) {
    switch (bn) {
    case 64: return cluster_slots_one<F, 64>(ks);
    case 128: return cluster_slots_one<F, 128>(ks);
    case 256: return cluster_slots_one<F, 256>(ks);
    default: return 0;
    }
}
}   // namespace

int gemm_max_clusters(int fmt, int bn, int ks) {
    switch (fmt) {
    case Q8_0: return cluster_slots_fmt<Q8_0>(bn, ks);
    case Q4_0: return cluster_slots_fmt<Q4_0>(bn, ks);
    case Q4_K: return cluster_slots_fmt<Q4_K>(bn, ks);
    case Q6_K: return cluster_slots_fmt<Q6_K>(bn, ks);
    case Q5_K: return cluster_slots_fmt<Q5_K>(bn, ks);
    default: return 0;
    }
}

int gemm_raw_window_bytes(int fmt) {
    switch (fmt) {
    case Q8_0: return Raw<Q8_0>::bytes;
    case Q4_0: return Raw<Q4_0>::bytes;
    case Q4_K: return Raw<Q4_K>::bytes;
    case Q6_K: return Raw<Q6_K>::bytes;
    case Q5_K: return Raw<Q5_K>::bytes;
    default: return 0;
    }
}

cudaError_t launch_gemm_tc(const GemmArgs &a, const CUtensorMap &wmap, const CUtensorMap &wmap2, const CUtensorMap &xmap,
                           cudaStream_t st) {
    switch (a.fmt) {
    case Q8_0: return launch_fmt<Q8_0>(a, wmap, wmap2, xmap, st);
    case Q4_0: return launch_fmt<Q4_0>(a, wmap, wmap2, xmap, st);
    case Q4_K: return launch_fmt<Q4_K>(a, wmap, wmap2, xmap, st);
    case Q6_K: return launch_fmt<Q6_K>(a, wmap, wmap2, xmap, st);
    case Q5_K: return launch_fmt<Q5_K>(a, wmap, wmap2, xmap, st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace qmm
