/*
 * qmm_oracle.c -- TEST INFRASTRUCTURE ONLY (see qmm_oracle.h).
 *
 * Plain C, IEEE double, no blocking, fusion or reordering beyond the
 * definition:  Y[n,m] = sum_k w(m,k) x(n,k).  Each weight row is expanded to
 * exact doubles, then every output is a straight sum over k.  Host threads
 * split the output rows; nothing else is parallel.
 */
#include "qmm_oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

int orc_block_info(int wtype, int *elems, int *bytes) {
    /* Block sizes: "cera 0.5.2 src/backend/cpu.rs" matmul_q4_0_f32 (18 B / 32),
     * matmul_q8_0_f32 (34 B / 32), matmul_q4km_f32 (144 B / 256);
     * "cera 0.3.1 src/model/gpu_lfm2.rs" weight upload (Q6_K 210 B / 256,
     * Q5_K 176 B / 256). */
    int e, b;
    switch (wtype) {
    case ORC_Q8_0: e = 32;  b = 34;  break;
    case ORC_Q4_0: e = 32;  b = 18;  break;
    case ORC_Q4_K: e = 256; b = 144; break;
    case ORC_Q6_K: e = 256; b = 210; break;
    case ORC_Q5_K: e = 256; b = 176; break;
    default: return -1;
    }
    if (elems) *elems = e;
    if (bytes) *bytes = b;
    return 0;
}

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double orc_f16_to_f64(uint16_t h) {
    int sign = (h >> 15) & 1;
    int ex = (h >> 10) & 0x1f;
    int fr = h & 0x3ff;
    double v;
    if (ex == 0) {
        v = ldexp((double)fr, -24);                 /* 0.fr x 2^-14 */
    } else if (ex == 31) {
        v = fr ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + fr), ex - 25);    /* 1.fr x 2^(ex-15) */
    }
    return sign ? -v : v;
}

static uint16_t rd16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }

/* Q8_0, 34 bytes: READING -- f16 d in bytes 0-1 (little endian), then 32
 * signed bytes q; w_e = d * q_e.  Only the 34-byte size is on the pages
 * ("cera 0.5.2 src/backend/cpu.rs" matmul_q8_0_f32); the d-first order is the
 * one the same page shows for Q4_0 (repack_q4_0_8x8) and the GGUF layout. */
static void deq_q8_0(const uint8_t *b, double *out) {
    double d = orc_f16_to_f64(rd16(b));
    for (int e = 0; e < 32; ++e) out[e] = d * (double)(int8_t)b[2 + e];
}

/* Q4_0, 18 bytes: f16 d in bytes 0-1, 16 bytes qs.  Element e < 16 is the low
 * nibble of qs[e], element e >= 16 the high nibble of qs[e-16]; w = (nib-8)*d.
 * "cera 0.5.2 src/backend/cpu.rs" repack_q4_0_8x8 (its per-element nibble
 * lookup and the f16 scale read from the first two bytes). */
static void deq_q4_0(const uint8_t *b, double *out) {
    double d = orc_f16_to_f64(rd16(b));
    const uint8_t *qs = b + 2;
    for (int e = 0; e < 32; ++e) {
        int nib = e < 16 ? (qs[e] & 0x0f) : (qs[e - 16] >> 4);
        out[e] = (double)(nib - 8) * d;
    }
}

/* Q4_K 6-bit scale/min of sub-block s from the 12 packed bytes S.
 * READING (the unpacking routine is named on the pages but not shown):
 * the GGUF K-quant packing.  Sub-blocks 0-3 keep their scale and min in the
 * low 6 bits of S[s] and S[s+4]; sub-blocks 4-7 take their low 4 bits from
 * the nibbles of S[s+4] and their top 2 bits from the top bits of S[s-4]
 * (scale) and S[s] (min). */
static void q4k_scale_min(const uint8_t *S, int s, int *sc, int *mn) {
    if (s < 4) {
        *sc = S[s] & 63;
        *mn = S[s + 4] & 63;
    } else {
        *sc = (S[s + 4] & 0x0f) | ((S[s - 4] >> 6) << 4);
        *mn = (S[s + 4] >> 4) | ((S[s] >> 6) << 4);
    }
}

/* Q4_K, 144 bytes: d (f16) @0, dmin (f16) @2, 12 scale bytes @4, qs[128] @16.
 * Field order: "cera 0.5.2 src/backend/cpu.rs" repack_q4_k_8x8 (d, dmin,
 * scales, qs); offsets follow from that order and the 144-byte size.
 * Sub-block s = e/32 reads qs[(s/2)*32 + e%32], low nibble for even s, high
 * nibble for odd s (the same function's nibble lookup).
 * w = d*sc_s*q - dmin*m_s (the products d*sc and dmin*m it precomputes). */
static void deq_q4_k(const uint8_t *b, double *out) {
    double d = orc_f16_to_f64(rd16(b));
    double dmin = orc_f16_to_f64(rd16(b + 2));
    const uint8_t *S = b + 4;
    const uint8_t *qs = b + 16;
    for (int e = 0; e < 256; ++e) {
        int s = e / 32, sc, mn;
        q4k_scale_min(S, s, &sc, &mn);
        uint8_t byte = qs[(s / 2) * 32 + e % 32];
        int q = (s % 2 == 0) ? (byte & 0x0f) : (byte >> 4);
        out[e] = d * (double)sc * (double)q - dmin * (double)mn;
    }
}

/* Q6_K, 210 bytes.  READING (only the 210-byte size is on the pages):
 * GGUF order ql[128] @0, qh[64] @128, int8 scales[16] @192, f16 d @208.
 * Element e = 128h + 32j + l (h in 0..1, j in 0..3, l in 0..31):
 *   low 4 bits : ql[64h + 32*(j%2) + l], low nibble for j < 2, high for j >= 2
 *   high 2 bits: bits 2j, 2j+1 of qh[32h + l]
 *   q = low | high << 4  (0..63),  w = d * scales[e/16] * (q - 32). */
static void deq_q6_k(const uint8_t *b, double *out) {
    const uint8_t *ql = b;
    const uint8_t *qh = b + 128;
    const int8_t *sc = (const int8_t *)(b + 192);
    double d = orc_f16_to_f64(rd16(b + 208));
    for (int e = 0; e < 256; ++e) {
        int h = e / 128, j = (e % 128) / 32, l = e % 32;
        uint8_t lb = ql[64 * h + 32 * (j % 2) + l];
        int lo = (j < 2) ? (lb & 0x0f) : (lb >> 4);
        int hi = (qh[32 * h + l] >> (2 * j)) & 3;
        int q = lo | (hi << 4);
        out[e] = d * (double)sc[e / 16] * (double)(q - 32);
    }
}

/* Q5_K, 176 bytes.  READING (only the 176-byte size is on the pages): GGUF
 * order d (f16) @0, dmin (f16) @2, 12 scale bytes @4 (the Q4_K packing),
 * qh[32] @16, qs[128] @48.  Sub-block s = e/32, l = e%32: the low 4 bits are
 * Q4_K's nibble (qs[(s/2)*32 + l], low for even s, high for odd s), bit 4 is
 * bit s of qh[l];  q = low | bit << 4 (0..31),  w = d*sc_s*q - dmin*m_s. */
static void deq_q5_k(const uint8_t *b, double *out) {
    double d = orc_f16_to_f64(rd16(b));
    double dmin = orc_f16_to_f64(rd16(b + 2));
    const uint8_t *S = b + 4;
    const uint8_t *qh = b + 16;
    const uint8_t *qs = b + 48;
    for (int e = 0; e < 256; ++e) {
        int s = e / 32, l = e % 32, sc, mn;
        q4k_scale_min(S, s, &sc, &mn);
        uint8_t byte = qs[(s / 2) * 32 + l];
        int lo = (s % 2 == 0) ? (byte & 0x0f) : (byte >> 4);
        int q = lo | (((qh[l] >> s) & 1) << 4);
        out[e] = d * (double)sc * (double)q - dmin * (double)mn;
    }
}

int orc_dequant_block(int wtype, const uint8_t *blk, double *out) {
    switch (wtype) {
    case ORC_Q8_0: deq_q8_0(blk, out); return 0;
    case ORC_Q4_0: deq_q4_0(blk, out); return 0;
    case ORC_Q4_K: deq_q4_k(blk, out); return 0;
    case ORC_Q6_K: deq_q6_k(blk, out); return 0;
    case ORC_Q5_K: deq_q5_k(blk, out); return 0;
    default: return -1;
    }
}

/* One row of K weights: K/elems consecutive blocks
 * ("cera 0.5.2 src/backend/cpu.rs" matmul_*_f32: row i starts at
 * i * blocks_per_row * block_bytes). */
static int dequant_row(int wtype, const uint8_t *w, int64_t m, int64_t K, double *out) {
    int E, B;
    if (orc_block_info(wtype, &E, &B)) return -1;
    int64_t nb = K / E;
    const uint8_t *row = w + m * nb * B;
    for (int64_t bi = 0; bi < nb; ++bi) orc_dequant_block(wtype, row + bi * B, out + bi * E);
    return 0;
}

static int check_shape(int wtype, int64_t M, int64_t K) {
    int E, B;
    if (orc_block_info(wtype, &E, &B)) return -1;
    if (M < 0 || K <= 0 || K % E) return -1;
    return 0;
}

int orc_dequant(int wtype, const uint8_t *w, int64_t M, int64_t K, double *out) {
    if (check_shape(wtype, M, K) || (M && (!w || !out))) return -1;
    for (int64_t m = 0; m < M; ++m) dequant_row(wtype, w, m, K, out + m * K);
    return 0;
}

int orc_dequant_f32(int wtype, const uint8_t *w, int64_t M, int64_t K, float *out) {
    if (check_shape(wtype, M, K) || (M && (!w || !out))) return -1;
    double *tmp = (double *)malloc(sizeof(double) * (size_t)K);
    if (!tmp) return -1;
    for (int64_t m = 0; m < M; ++m) {
        dequant_row(wtype, w, m, K, tmp);
        for (int64_t k = 0; k < K; ++k) out[m * K + k] = (float)tmp[k];
    }
    free(tmp);
    return 0;
}

static double x_at(const void *x, int xtype, int64_t i) {
    if (xtype == ORC_X_F32) return (double)((const float *)x)[i];
    /* bf16 = the top 16 bits of an IEEE binary32. */
    uint32_t bits = (uint32_t)((const uint16_t *)x)[i] << 16;
    float f;
    memcpy(&f, &bits, 4);
    return (double)f;
}

typedef struct {
    int wtype, xtype;
    const uint8_t *w;
    int64_t M, K, N;
    const double *xd;          /* x expanded to double, [N,K] */
    const int64_t *rows;
    int64_t nrows;
    double *Y, *S;
    int64_t j0, j1;
    int err;
} job_t;

static void *run_job(void *arg) {
    job_t *jb = (job_t *)arg;
    double *wrow = (double *)malloc(sizeof(double) * (size_t)jb->K);
    if (!wrow) { jb->err = -1; return NULL; }
    for (int64_t j = jb->j0; j < jb->j1; ++j) {
        int64_t m = jb->rows ? jb->rows[j] : j;
        dequant_row(jb->wtype, jb->w, m, jb->K, wrow);
        for (int64_t n = 0; n < jb->N; ++n) {
            const double *xr = jb->xd + n * jb->K;
            double y = 0.0, s = 0.0;
            for (int64_t k = 0; k < jb->K; ++k) {
                double p = wrow[k] * xr[k];
                y += p;
                s += fabs(p);
            }
            jb->Y[n * jb->nrows + j] = y;
            jb->S[n * jb->nrows + j] = s;
        }
    }
    free(wrow);
    return NULL;
}

int orc_matmul_rows(int wtype, const uint8_t *w, int64_t M, int64_t K,
                    const void *x, int xtype, int64_t N,
                    const int64_t *rows, int64_t nrows,
                    double *Y, double *S, int nthreads) {
    if (check_shape(wtype, M, K) || N < 0 || nrows < 0) return -1;
    if (xtype != ORC_X_F32 && xtype != ORC_X_BF16) return -1;
    if (nrows == 0 || N == 0) return 0;
    if (!w || !x || !Y || !S) return -1;
    for (int64_t j = 0; j < nrows; ++j) {
        int64_t m = rows ? rows[j] : j;
        if (m < 0 || m >= M) return -1;
    }
    double *xd = (double *)malloc(sizeof(double) * (size_t)(N * K));
    if (!xd) return -1;
    for (int64_t i = 0; i < N * K; ++i) xd[i] = x_at(x, xtype, i);

    if (nthreads <= 0) nthreads = (int)sysconf(_SC_NPROCESSORS_ONLN);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > nrows) nthreads = (int)nrows;
    job_t *jobs = (job_t *)calloc((size_t)nthreads, sizeof(job_t));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    int err = 0;
    if (!jobs || !th) { free(xd); free(jobs); free(th); return -1; }
    for (int t = 0; t < nthreads; ++t) {
        job_t *jb = &jobs[t];
        jb->wtype = wtype; jb->xtype = xtype; jb->w = w;
        jb->M = M; jb->K = K; jb->N = N; jb->xd = xd;
        jb->rows = rows; jb->nrows = nrows; jb->Y = Y; jb->S = S;
        jb->j0 = nrows * t / nthreads;
        jb->j1 = nrows * (t + 1) / nthreads;
    }
    int started = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&th[t], NULL, run_job, &jobs[t])) { err = -1; break; }
        started = t;
    }
    run_job(&jobs[0]);
    for (int t = 1; t <= started; ++t) pthread_join(th[t], NULL);
    if (err == 0 && started != nthreads - 1) err = -1;
    for (int t = 0; t < nthreads && !err; ++t) err = jobs[t].err;
    free(jobs);
    free(th);
    free(xd);
    return err;
}

/* ------------------------------------------------------------------------
 * Activation quantization (Q8_0 activations).
 * ------------------------------------------------------------------------ */

uint16_t orc_f32_to_f16(float f) {
    uint32_t bits;
    memcpy(&bits, &f, 4);
    const uint16_t sign = (uint16_t)((bits >> 16) & 0x8000u);
    if (isnan(f)) return (uint16_t)(sign | 0x7e00u);
    const double v = fabs((double)f);
    if (v >= 65520.0) return (uint16_t)(sign | 0x7c00u);   /* halfway above 65504 rounds up: infinity */
    if (v == 0.0) return sign;
    int ex;
    (void)frexp(v, &ex);                                   /* v = m 2^ex, m in [0.5, 1) */
    const int e = ex - 1;                                   /* floor(log2 v) */
    if (e < -14) {                                          /* subnormal: multiples of 2^-24 */
        const double r = nearbyint(ldexp(v, 24));           /* ties to even (default rounding) */
        return (uint16_t)(sign | (uint16_t)r);              /* r == 1024 is the smallest normal */
    }
    double r = nearbyint(ldexp(v, 10 - e));                 /* 11 significant bits: [1024, 2048] */
    int eb = e + 15;
    if (r == 2048.0) {
        r = 1024.0;
        eb += 1;
    }
    if (eb >= 31) return (uint16_t)(sign | 0x7c00u);
    return (uint16_t)(sign | (uint16_t)(eb << 10) | (uint16_t)(r - 1024.0));
}

int orc_quantize_q8_0(const float *x, int64_t n, float *scales, int8_t *quants) {
    if (n < 0 || n % 32 || (n && (!x || !scales || !quants))) return -1;
    for (int64_t b = 0; b < n / 32; ++b) {
        const float *blk = x + 32 * b;
        float amax = 0.0f;
        for (int e = 0; e < 32; ++e) amax = fmaxf(amax, fabsf(blk[e]));
        const float d = amax / 127.0f;
        const float r = 1.0f / d;
        const float id = (d != 0.0f && isfinite(r)) ? r : 0.0f;
        scales[b] = (float)orc_f16_to_f64(orc_f32_to_f16(d));
        for (int e = 0; e < 32; ++e) {
            float q = rintf(blk[e] * id);
            if (isnan(q)) q = 0.0f;
            q = q < -128.0f ? -128.0f : (q > 127.0f ? 127.0f : q);
            quants[32 * b + e] = (int8_t)q;
        }
    }
    return 0;
}
