// gemv_shared.cuh -- pieces shared by the bf16 (gemv_fast.cu) and int8
// (gemv_i8.cu) tensor-core GEMV kernels: chunk geometry, the per-row scale
// table, bounded waits, small shared-memory loads, the end-of-tile
// reduction and store (plain, K-split through distributed shared memory, or
// argmax), and the cluster launch.  Everything sits in an unnamed namespace:
// each translation unit gets its own copy.
#pragma once
#include <atomic>

#include "amax.cuh"
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
template <> struct GWin<Q5_K> { static constexpr int bytes = 176; };

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
    const float2 r = __ffma2_rn(make_float2(s0, s1), make_float2(d0, d1), make_float2(a0, a1));
    a0 = r.x;
    a1 = r.y;
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
        if (mbar_try_wait_sleep(bar, parity, 2000u)) return true;
        if (*abort_flag) return false;
        if ((uint64_t)(clock64() - t0) > limit) {
            *abort_flag = 1u;
            return false;
        }
    }
}

// Entries e0..e0+NE-1 (e0 a multiple of 4) of row r of the scale table.
template <int NE>
__device__ __forceinline__ void ld_scales(float (&v)[NE], const float *sct, int r, int e0) {
#pragma unroll
    for (int i = 0; i < NE; i += 4) {
        const float4 a = *reinterpret_cast<const float4 *>(sct + sct_index(r, e0 + i));
        v[i] = a.x;
        v[i + 1] = a.y;
        v[i + 2] = a.z;
        v[i + 3] = a.w;
    }
}

// ---------------------------------------------------------------------------
// End of a tile: without a K split every compute thread stores its rows; with
// one, partials go to shared memory [row][token] and cluster rank 0 sums the
// KS slices in rank order (deterministic) and stores.
// ---------------------------------------------------------------------------
template <int NT, int P, int CW, int RG>
__device__ __forceinline__ void finish_tile(const float (&acc)[RG][NT][4], float *sred, float *__restrict__ Y, int M,
                                            int N, int m0, int KS, bool aborted, int warp, int lane,
                                            unsigned long long *amax) {
    constexpr int ROWS = 16 * CW * RG;
    if (KS == 1 && amax) {
        // argmax mode: Y is not written; each token's best (value, row)
        if (warp < CW && !aborted) {
            const int g = lane >> 2, t = lane & 3;
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                if constexpr (P == 2) {
                    const int n = 4 * j + t;
                    unsigned long long best = 0ull;
#pragma unroll
                    for (int q = 0; q < RG; ++q) {
                        const int r0 = m0 + 16 * (RG * warp + q) + g, r1 = r0 + 8;
                        if (n < N && r0 < M) amax_fold(best, acc[q][j][0] + acc[q][j][1], r0);
                        if (n < N && r1 < M) amax_fold(best, acc[q][j][2] + acc[q][j][3], r1);
                    }
                    amax_commit(amax, n, N, best, g);
                } else {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int n = 8 * j + 2 * t + h;
                        unsigned long long best = 0ull;
#pragma unroll
                        for (int q = 0; q < RG; ++q) {
                            const int r0 = m0 + 16 * (RG * warp + q) + g, r1 = r0 + 8;
                            if (n < N && r0 < M) amax_fold(best, acc[q][j][h], r0);
                            if (n < N && r1 < M) amax_fold(best, acc[q][j][2 + h], r1);
                        }
                        amax_commit(amax, n, N, best, g);
                    }
                }
            }
        }
    } else if (KS == 1) {
        if (warp < CW && !aborted) {
            const int g = lane >> 2, t = lane & 3;
#pragma unroll
            for (int q = 0; q < RG; ++q) {
                const int r0 = m0 + 16 * (RG * warp + q) + g, r1 = r0 + 8;
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    if constexpr (P == 2) {
                        const int n = 4 * j + t;
                        if (n < N) {
                            if (r0 < M) Y[(int64_t)n * M + r0] = acc[q][j][0] + acc[q][j][1];
                            if (r1 < M) Y[(int64_t)n * M + r1] = acc[q][j][2] + acc[q][j][3];
                        }
                    } else {
                        const int n0 = 8 * j + 2 * t;
                        if (n0 < N) {
                            if (r0 < M) Y[(int64_t)n0 * M + r0] = acc[q][j][0];
                            if (r1 < M) Y[(int64_t)n0 * M + r1] = acc[q][j][2];
                        }
                        if (n0 + 1 < N) {
                            if (r0 < M) Y[(int64_t)(n0 + 1) * M + r0] = acc[q][j][1];
                            if (r1 < M) Y[(int64_t)(n0 + 1) * M + r1] = acc[q][j][3];
                        }
                    }
                }
            }
        }
    } else {
        // partials -> shared memory [row][token] (aliases the X fragments:
        // wait until every warp of the CTA is done with them); rank 0 of the
        // cluster sums
        __syncthreads();
        if (warp < CW) {
            const int g = lane >> 2, t = lane & 3;
#pragma unroll
            for (int q = 0; q < RG; ++q) {
                const int r0 = 16 * (RG * warp + q) + g, r1 = r0 + 8;
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    if constexpr (P == 2) {
                        const int n = 4 * j + t;
                        if (n < 16) {
                            sred[r0 * 16 + n] = acc[q][j][0] + acc[q][j][1];
                            sred[r1 * 16 + n] = acc[q][j][2] + acc[q][j][3];
                        }
                    } else {
                        const int n0 = 8 * j + 2 * t;
                        if (n0 + 1 < 16) {
                            sred[r0 * 16 + n0] = acc[q][j][0];
                            sred[r0 * 16 + n0 + 1] = acc[q][j][1];
                            sred[r1 * 16 + n0] = acc[q][j][2];
                            sred[r1 * 16 + n0 + 1] = acc[q][j][3];
                        }
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
                if (m0 + row < M && !aborted) {
                    if (amax)
                        atomicMax(amax + n, amax_key(v, m0 + row));
                    else
                        Y[(int64_t)n * M + m0 + row] = v;
                }
            }
        }
        cluster_sync_all();
    }
}

// K split: the smallest power of two (<= 8, one cluster) that gives at
// least 1.5 CTAs per SM, and (max_cps > 0) few enough chunks per CTA for the
// resident fragments.  Returns 0 if the slice cannot be made small enough.
inline int plan_ks(int64_t tiles, int nchunks, int num_sms, int max_cps, int force) {
    int ks = 1;
    if (force > 0) {
        while (ks < force && ks < 8 && ks * 2 <= nchunks) ks *= 2;
    } else {
        while (ks < 8 && tiles * ks * 2 < (int64_t)num_sms * 3 && ks * 2 <= nchunks) ks *= 2;
    }
    while (max_cps > 0 && (nchunks + ks - 1) / ks > max_cps && ks < 8 && ks * 2 <= nchunks) ks *= 2;
    if (max_cps > 0 && (nchunks + ks - 1) / ks > max_cps) return 0;
    return ks;
}

template <typename Kern, typename XArg>
cudaError_t launch_cluster(Kern kern, int smem, int threads, int64_t tiles, int ks, int nchunks, cudaStream_t st,
                           bool pdl, const GemvSegs &segs, const XArg &x_arg, int64_t K, int N, unsigned *status,
                           uint64_t limit, const AmaxOut &amax) {
    const int cps = (nchunks + ks - 1) / ks;
    ks = (nchunks + cps - 1) / cps;   // no empty slices
    int ksp = 1;                      // cluster dims must divide the grid
    while (ksp < ks) ksp *= 2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)tiles, (unsigned)ksp, 1);
    cfg.blockDim = dim3((unsigned)threads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    unsigned na = 0;
    if (ksp > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = 1;
        attr[na].val.clusterDim.y = (unsigned)ksp;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    const cudaError_t e =
        cudaLaunchKernelEx(&cfg, kern, segs, x_arg, (int)K, N, cps, status, limit, amax);
    if (e != cudaSuccess) return e;
    return launched(cudaGetLastError());
}

template <typename Kern>
cudaError_t set_smem_once(Kern kern, int smem, std::atomic<uint64_t> &configured) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (!(configured.load() & (1ull << (dev & 63)))) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        configured.fetch_or(1ull << (dev & 63));
    }
    return cudaSuccess;
}

// First tile of every segment (tile0[nseg] = all tiles) for `rows`-row tiles.
inline int64_t set_tiles(GemvSegs &sg, int rows) {
    int64_t t = 0;
    for (int i = 0; i < sg.nseg; ++i) {
        sg.tile0[i] = (int)t;
        t += (sg.M[i] + rows - 1) / rows;
    }
    sg.tile0[sg.nseg] = (int)t;
    return t;
}

}  // namespace
}  // namespace qmm
