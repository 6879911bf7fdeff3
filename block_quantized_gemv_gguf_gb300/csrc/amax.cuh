// amax.cuh -- argmax mode of the GEMV kernels (the greedy-decode LM head):
// no output is stored; each token's largest output and its row are kept as
// an order-preserving 64-bit key, folded with atomicMax, and the last CTA to
// finish unpacks them.  Everything sits in an unnamed namespace: each
// translation unit gets its own copy.
#pragma once

#include "common.cuh"

namespace qmm {
namespace {

// Argmax-mode outputs: per-token keys (zeroed by the host with the counter),
// a counter of finished CTAs, and the unpacked results the last CTA writes.
struct AmaxOut {
    unsigned long long *keys;   // null: ordinary GEMV
    unsigned *counter;
    int32_t *idx;
    float *val;
};

// Order-preserving 64-bit key of (value, row): a larger value wins, then the
// lower row (the high word maps the float's bits to an unsigned order, the
// low word holds ~row).  0 is below every key.
__device__ __forceinline__ unsigned long long amax_key(float v, int row) {
    const uint32_t u = __float_as_uint(v);
    const uint32_t o = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((unsigned long long)o << 32) | (uint32_t)~(uint32_t)row;
}
__device__ __forceinline__ void amax_fold(unsigned long long &best, float v, int row) {
    const unsigned long long k = amax_key(v, row);
    best = k > best ? k : best;
}
// Maximum over the 8 lanes of a quad column (same t: same tokens, other
// rows), then one atomic per warp and token.
__device__ __forceinline__ void amax_commit(unsigned long long *keys, int n, int N, unsigned long long best, int g) {
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
        const unsigned long long x = __shfl_xor_sync(0xffffffffu, best, o);
        best = x > best ? x : best;
    }
    if (g == 0 && n < N && best != 0ull) atomicMax(keys + n, best);
}

// Argmax mode, after every CTA's keys are in: the last CTA to finish (a
// fenced counter) unpacks keys[n] into idx[n] (row) and val[n] (output).
__device__ __forceinline__ void amax_last_cta(const AmaxOut &a, int N) {
    __shared__ unsigned s_last;
    if (!a.keys) return;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned done = atomicAdd(a.counter, 1u);
        s_last = done == gridDim.x * gridDim.y - 1 ? 1u : 0u;
    }
    __syncthreads();
    if (s_last && (int)threadIdx.x < N) {
        __threadfence();
        const unsigned long long k = atomicAdd(a.keys + threadIdx.x, 0ull);   // coherent read
        const uint32_t o = (uint32_t)(k >> 32);
        const uint32_t u = (o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o;       // inverse of the key map
        a.idx[threadIdx.x] = (int32_t)~(uint32_t)k;
        a.val[threadIdx.x] = __uint_as_float(u);
    }
}


}  // namespace
}  // namespace qmm
