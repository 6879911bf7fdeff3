// api.cu -- the extern "C" boundary declared in include/qmm.h: argument
// validation, the N-based dispatcher, TMA tensor-map construction and the
// per-device status word.
#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "../../include/qmm.h"
#include "kernels.h"

namespace qmm {
std::atomic<uint64_t> g_launches{0};

cudaError_t launched(cudaError_t e) {
    if (e == cudaSuccess) g_launches.fetch_add(1);
    return e;
}
}  // namespace qmm

namespace {

using namespace qmm;

// One status word per device, a static device variable (no allocation).
__device__ unsigned g_qmm_status_word;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned *g_status_ptr[kMaxDevices];
int g_num_sms[kMaxDevices];
std::atomic<uint64_t> g_wait_limit{1ull << 31};   // ~1 s at 2 GHz
// Static-weights mode (programmatic dependent launch): -1 = not set through
// the API, take QMM_STATIC_WEIGHTS from the environment.
std::atomic<int> g_static_weights{-1};
// Integer tensor-core GEMV for N <= 2 (exact int8 digits of X): -1 = not set
// through the API, take QMM_GEMV_I8 from the environment (default off: on
// this part it measures no faster than the bf16 kernel).
std::atomic<int> g_gemv_i8{-1};
// 16-row-tile tensor-core GEMV for 2 <= N <= QMM_TC_MAX_N: -1 = not set
// through the API, take QMM_GEMV_TC from the environment (default off).
std::atomic<int> g_gemv_tc{-1};
// Streaming GEMV plan parameters set through qmm_set_gemv_stream (rows per
// task, warps, slots, CTAs per SM, direct-load variant): -1 = not set, take
// the environment's.
std::atomic<int> g_stream_force[5] = {-1, -1, -1, -1, -1};
bool gemv_i8_on() {
    const int v = g_gemv_i8.load();
    if (v >= 0) return v != 0;
    static const bool env = [] {
        const char *e = std::getenv("QMM_GEMV_I8");
        return e && *e && std::atoi(e) != 0;
    }();
    return env;
}
// Set while qmm_matmul_host runs its compute call: that call follows a
// host-to-device copy, not a kernel, so it is launched the ordinary way.
thread_local bool t_after_copy = false;
bool static_weights() {
    if (t_after_copy) return false;
    const int v = g_static_weights.load();
    if (v >= 0) return v != 0;
    static const bool env = [] {
        const char *e = std::getenv("QMM_STATIC_WEIGHTS");
        return e && std::atoi(e) != 0;
    }();
    return env;
}

struct DevInfo {
    unsigned *status;
    int num_sms;
};

bool dev_info(DevInfo &out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_status_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_qmm_status_word) != cudaSuccess) return false;
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
        g_status_ptr[dev] = static_cast<unsigned *>(p);
        g_num_sms[dev] = sms;
    }
    out.status = g_status_ptr[dev];
    out.num_sms = g_num_sms[dev];
    return true;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no
// link-time dependency on the driver library).
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

bool block_geom(int wt, int &E, int &B) {
    switch (wt) {
    case QMM_Q8_0: E = 32; B = 34; return true;
    case QMM_Q4_0: E = 32; B = 18; return true;
    case QMM_Q4_K: E = 256; B = 144; return true;
    case QMM_Q6_K: E = 256; B = 210; return true;
    case QMM_Q5_K: E = 256; B = 176; return true;
    default: return false;
    }
}

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    const uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
    return a0 < b0 + nb && b0 < a0 + na;
}

int env_int(const char *name, int dflt) {
    const char *v = std::getenv(name);
    if (!v || !*v) return dflt;
    return std::atoi(v);
}

// Dispatcher settings, read once per process.
struct Settings {
    int gemv_max_n;   // QMM_GEMV_MAX_N: largest N qmm_matmul sends to the GEMV
    int force;        // QMM_FORCE_PATH: 0 none, 1 gemv, 2 gemm
    int gemm_bn;      // QMM_GEMM_BN: 0 = model-based choice
    int gemm_ks;      // QMM_GEMM_KS: K split of the GEMM (1, 2, 4); 0 = by tile count
    int gemv_rows;    // QMM_GEMV_ROWS: 64, 128 or 256 rows per GEMV tile; 0 = by M
    int gemv_rg;      // QMM_GEMV_RG: 16-row groups per warp (1 or 2) of the resident-X GEMV
    int gemv_ks;      // QMM_GEMV_KS: K split of the GEMV (1..8); 0 = automatic
    int gemv_res;     // QMM_GEMV_RESIDENT: 0 disables the resident-X GEMV
    int stream;       // QMM_GEMV_STREAM: 0 disables the streaming N = 1 GEMV
    int stream_warps; // QMM_STREAM_WARPS: warps per CTA of the streaming GEMV, 1..16 (0 = by shared memory)
    int stream_r;     // QMM_STREAM_R: rows per task of the streaming GEMV, 1, 2 or 4 (0 = by shape)
    int stream_slots; // QMM_STREAM_SLOTS: stage slots per warp, 1..3 (0 = by shared memory)
    int stream_cps;   // QMM_STREAM_CPS: CTAs per SM, 1 or 2 (0 = by shape)
    int stream_direct;// QMM_STREAM_DIRECT: 1 the direct-load variant, 2 the staged kernel (0 = planner's choice)
    int stream_stagger;// QMM_STREAM_STAGGER: 0 turns off the staggered stage issue of 2- and 3-slot plans
    int tc;           // QMM_GEMV_TC: 1 enables the 16-row-tile tensor-core GEMV (opt-in, see qmm_set_gemv_tc)
    int tc_warps;     // QMM_TC_WARPS: warps per CTA of that kernel (0 = by shared memory)
    int tc_max_n;     // QMM_TC_MAX_N: largest N it serves (default 4; above, the ring GEMV is faster)
};
const Settings &settings() {
    static Settings s = [] {
        Settings t;
        t.gemv_max_n = env_int("QMM_GEMV_MAX_N", QMM_MATMUL_GEMV_MAX_N);
        if (t.gemv_max_n < 0) t.gemv_max_n = 0;
        if (t.gemv_max_n > QMM_GEMV_MAX_N) t.gemv_max_n = QMM_GEMV_MAX_N;
        const char *f = std::getenv("QMM_FORCE_PATH");
        t.force = (f && !std::strcmp(f, "gemv")) ? 1 : (f && !std::strcmp(f, "gemm")) ? 2 : 0;
        t.gemm_bn = env_int("QMM_GEMM_BN", 0);
        if (t.gemm_bn != 64 && t.gemm_bn != 128 && t.gemm_bn != 256) t.gemm_bn = 0;
        t.gemm_ks = env_int("QMM_GEMM_KS", 0);
        if (t.gemm_ks != 1 && t.gemm_ks != 2 && t.gemm_ks != 4) t.gemm_ks = 0;
        t.gemv_rows = env_int("QMM_GEMV_ROWS", 0);
        if (t.gemv_rows != 64 && t.gemv_rows != 128 && t.gemv_rows != 256) t.gemv_rows = 0;
        t.gemv_rg = env_int("QMM_GEMV_RG", 0) == 2 ? 2 : 1;
        t.gemv_ks = env_int("QMM_GEMV_KS", 0);
        if (t.gemv_ks < 0 || t.gemv_ks > 8) t.gemv_ks = 0;
        t.gemv_res = env_int("QMM_GEMV_RESIDENT", 1) != 0;
        t.stream = env_int("QMM_GEMV_STREAM", 1) != 0;
        t.stream_warps = env_int("QMM_STREAM_WARPS", 0);
        if (t.stream_warps < 0 || t.stream_warps > 16) t.stream_warps = 0;
        t.stream_r = env_int("QMM_STREAM_R", 0);
        if (t.stream_r != 1 && t.stream_r != 2 && t.stream_r != 4) t.stream_r = 0;
        t.stream_slots = env_int("QMM_STREAM_SLOTS", 0);
        if (t.stream_slots < 0 || t.stream_slots > 3) t.stream_slots = 0;
        t.stream_cps = env_int("QMM_STREAM_CPS", 0);
        if (t.stream_cps != 1 && t.stream_cps != 2) t.stream_cps = 0;
        t.stream_direct = env_int("QMM_STREAM_DIRECT", 0);
        if (t.stream_direct != 1 && t.stream_direct != 2) t.stream_direct = 0;
        t.stream_stagger = env_int("QMM_STREAM_STAGGER", 1) == 0 ? 2 : 0;
        t.tc = env_int("QMM_GEMV_TC", 0) != 0;
        t.tc_warps = env_int("QMM_TC_WARPS", 0);
        if (t.tc_warps != 4 && t.tc_warps != 8 && t.tc_warps != 16) t.tc_warps = 0;
        t.tc_max_n = env_int("QMM_TC_MAX_N", 4);
        if (t.tc_max_n < 1) t.tc_max_n = 1;
        if (t.tc_max_n > 8) t.tc_max_n = 8;
        return t;
    }();
    return s;
}

StreamForce stream_force() {
    const Settings &t = settings();
    const int env[5] = {t.stream_r, t.stream_warps, t.stream_slots, t.stream_cps, t.stream_direct};
    int v[5];
    for (int i = 0; i < 5; ++i) {
        const int g = g_stream_force[i].load();
        v[i] = g >= 0 ? g : env[i];
    }
    return StreamForce{v[0], v[1], v[2], v[3], v[4], t.stream_stagger};
}

// Common validation of W, M, K, X, N, Y.
// ybytes_override: the size of the output actually written at Y (argmax
// mode writes N entries, not N x M); 0 means N * M * 4.
// xt == X_CODES: X holds int8 codes (N * K bytes, any alignment).
constexpr int X_CODES = 100;
qmm_status validate(int wt, const void *W, size_t w_bytes, int64_t M, int64_t K, const void *X, int xt,
                    int64_t N, const float *Y, int64_t max_n, int &E, int &B, size_t ybytes_override = 0) {
    if (!block_geom(wt, E, B)) return QMM_ERR_INVALID_ARG;
    if (xt != QMM_X_F32 && xt != QMM_X_BF16 && xt != X_CODES) return QMM_ERR_INVALID_ARG;
    if (!W || !X || !Y) return QMM_ERR_INVALID_ARG;
    if (M < 1 || K < 1 || M > (1ll << 30) || K > (1ll << 24)) return QMM_ERR_INVALID_ARG;
    if (N < 1 || N > max_n) return QMM_ERR_INVALID_ARG;
    if (K % E) return QMM_ERR_INVALID_ARG;
    const size_t need = (size_t)M * (size_t)(K / E) * (size_t)B;
    if (w_bytes < need) return QMM_ERR_INVALID_ARG;
    const size_t xs = xt == QMM_X_F32 ? 4 : (xt == QMM_X_BF16 ? 2 : 1);
    if (((uintptr_t)X) % xs || ((uintptr_t)Y) % 4) return QMM_ERR_INVALID_ARG;
    const size_t ybytes = ybytes_override ? ybytes_override : (size_t)N * (size_t)M * 4;
    if (overlaps(Y, ybytes, W, need) || overlaps(Y, ybytes, X, (size_t)N * (size_t)K * xs))
        return QMM_ERR_INVALID_ARG;
    return QMM_OK;
}

qmm_status from_cuda(cudaError_t e) { return e == cudaSuccess ? QMM_OK : QMM_ERR_CUDA; }

// Resident clusters of ks CTAs for (fmt, bn), per device (queried once).
int cluster_capacity(int fmt, int bn, int ks, int num_sms) {
    if (ks == 1) return num_sms;
    static std::atomic<int> cache[8][5][3][3];   // device, format, bn, ks; 0 = not queried
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 8 || fmt < 0 || fmt > 4) return num_sms / ks;
    const int bi = bn == 64 ? 0 : (bn == 128 ? 1 : 2), ki = ks == 2 ? 1 : 2;
    int v = cache[dev][fmt][bi][ki].load();
    if (v == 0) {
        v = gemm_max_clusters(fmt, bn, ks);
        if (v <= 0) v = -1;
        cache[dev][fmt][bi][ki].store(v);
    }
    return v > 0 ? v : num_sms / ks / 2;
}

// Token tile BN and K split KS of the GEMM, and how the 128-row tiles are
// divided between at most two launches.  A CTA spends about the same time on
// a 256-k chunk whatever BN is (weight copy, dequantization and MMA overlap),
// plus about two chunks' worth of set-up, drain and epilogue.  With fewer
// tiles than a wave, a K split over a cluster (2 or 4 CTAs) shortens each
// CTA's K range, as long as the split grid still fits one wave.  With more
// tiles than a wave, the whole waves run unsplit and the tiles of the last,
// partial wave run as a second launch, split when that is quicker.  Among
// the BNs, the fewest estimated chunk-times wins; on a tie the larger BN
// (less repeated dequantization).
struct TilePlan {
    int bn;
    int mt_a, ks_a;   // first launch: m-tiles 0 .. mt_a - 1, K split ks_a
    int ks_b;         // second launch (the remaining m-tiles, if any), K split ks_b
    double cost;
};

TilePlan plan_tiles(int fmt, int64_t total_mt, int64_t N, int64_t K, int num_sms) {
    const Settings &cfg = settings();
    const int64_t nkc = K / 256;
    TilePlan best{64, (int)total_mt, 1, 1, 1e30};
    auto chunks = [&](int ks) { return (double)((nkc + ks - 1) / ks) + (ks > 1 ? 2.0 : 1.5); };
    auto ks_ok = [&](int ks) {
        if (cfg.gemm_ks) return ks == cfg.gemm_ks && ks <= nkc;
        return ks == 1 || (nkc / ks >= 4);
    };
    for (int bn : {256, 128, 64}) {
        if (cfg.gemm_bn ? bn != cfg.gemm_bn : (bn > 64 && N <= bn / 2)) continue;   // a smaller tile covers N
        const int64_t tn = (N + bn - 1) / bn, tiles = total_mt * tn;
        // one launch, split within one wave or unsplit
        for (int ks : {1, 2, 4}) {
            if (!ks_ok(ks)) continue;
            const int64_t cap = cluster_capacity(fmt, bn, ks, num_sms);
            if (cap < 1 || (ks > 1 && tiles > cap)) continue;
            const double cost = (double)((tiles + cap - 1) / cap) * chunks(ks);
            if (cost < best.cost - 1e-9) best = TilePlan{bn, (int)total_mt, ks, ks, cost};
        }
        // whole waves unsplit, then the last wave's tiles split
        if (!cfg.gemm_ks && tiles > num_sms && tiles % num_sms) {
            const int64_t mt_a = tiles / num_sms * num_sms / tn;
            const int64_t tail = (total_mt - mt_a) * tn;
            if (mt_a < 1 || mt_a >= total_mt) continue;
            const double head = (double)((mt_a * tn + num_sms - 1) / num_sms) * chunks(1);
            for (int ks : {2, 4}) {
                if (!ks_ok(ks)) continue;
                const int64_t cap = cluster_capacity(fmt, bn, ks, num_sms);
                if (cap < 1 || tail > cap) continue;
                const double cost = head + chunks(ks);
                if (cost < best.cost - 1e-9) best = TilePlan{bn, (int)mt_a, 1, ks, cost};
            }
        }
    }
    return best;
}

// One GEMV launch over nseg weight matrices of format wt that share X (K,
// N): fused projections when nseg > 1.  amax != nullptr (nseg == 1): argmax
// mode (no Y; the fast path only, else QMM_ERR_UNSUPPORTED), launched the
// ordinary way.
struct SegIn {
    const void *W;
    size_t w_bytes;
    int64_t M;
    float *Y;
};

// Plan of the integer GEMV (mode 0: exact digits, 1: Q8_0 activations), or
// false when no variant holds the K slice.
bool plan_i8(int mode, int wt, int64_t m_total, int64_t K, int N, int xbf16, int num_sms, GemvPlan &p) {
    const Settings &cfg = settings();
    const int rows = cfg.gemv_rows ? (cfg.gemv_rows >= 128 ? 128 : 64) : gemv_tile_rows(m_total, num_sms);
    const int rg = mode == 0 && rows == 128 && cfg.gemv_rg == 2 ? 2 : 1;
    const int maxc = mode == 0 ? gemv_i8_exact_maxc(wt, N, xbf16, rows, rg) : gemv_i8_q8_maxc(wt, N, rows);
    if (maxc <= 0) return false;
    const int ks = plan_ks_host((m_total + rows - 1) / rows, (int)(K / 256), num_sms, maxc, cfg.gemv_ks);
    if (ks <= 0) return false;
    p.resident = 2;
    p.rows = rows;
    p.rg = rg;
    p.ks = ks;
    return true;
}

// xscales != nullptr: Q8_0-activation mode, X = quants int8 [N][K] and
// xscales f32 [N][K/32] (the fast path only, else QMM_ERR_UNSUPPORTED).
qmm_status gemv_segments(int wt, const SegIn *seg, int nseg, int64_t K, const void *X, int xt, int64_t N,
                         void *stream, unsigned long long *amax = nullptr, int32_t *idx = nullptr,
                         float *val = nullptr, const float *xscales = nullptr) {
    if (nseg < 1 || nseg > QMM_MAX_SEGS || (amax && nseg != 1)) return QMM_ERR_INVALID_ARG;
    const bool q8 = xscales != nullptr;
    if (q8 && (N < 1 || N > QMM_GEMV_MAX_N)) return QMM_ERR_INVALID_ARG;
    int E = 0, B = 0;
    int64_t m_total = 0;
    for (int i = 0; i < nseg; ++i) {
        const qmm_status s =
            validate(wt, seg[i].W, seg[i].w_bytes, seg[i].M, K, X, q8 ? X_CODES : xt, N,
                     amax ? reinterpret_cast<const float *>(amax) : seg[i].Y, QMM_GEMV_MAX_N, E, B,
                     amax ? (size_t)(N + 1) * 8 : (size_t)N * (size_t)seg[i].M * 4);
        if (s != QMM_OK) return s;
        if (q8 && (overlaps(amax ? static_cast<const void *>(amax) : seg[i].Y,
                            amax ? (size_t)(N + 1) * 8 : (size_t)N * (size_t)seg[i].M * 4, xscales,
                            (size_t)N * (size_t)(K / 32) * 4)))
            return QMM_ERR_INVALID_ARG;
        m_total += seg[i].M;
        for (int j = 0; j < nseg && !amax; ++j) {   // no output may overlap another matrix or output
            const size_t yi = (size_t)N * (size_t)seg[i].M * 4;
            if (j != i && (overlaps(seg[i].Y, yi, seg[j].W, (size_t)seg[j].M * (size_t)(K / E) * (size_t)B) ||
                           overlaps(seg[i].Y, yi, seg[j].Y, (size_t)N * (size_t)seg[j].M * 4)))
                return QMM_ERR_INVALID_ARG;
        }
    }
    DevInfo di;
    if (!dev_info(di)) return QMM_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int64_t row_bytes = K / E * B;
    // Tensor-core GEMV: whole 256-weight chunks, TMA-able rows (16-byte
    // aligned base and row pitch), 16-byte aligned X.  Anything else takes the
    // byte-addressed kernel, which computes the same sums.
    bool fast = K % 256 == 0 && row_bytes % 16 == 0 && (uintptr_t)X % 16 == 0 && m_total <= (1ll << 31) - 1;
    for (int i = 0; i < nseg; ++i) fast = fast && (uintptr_t)seg[i].W % 16 == 0;
    if (q8) fast = fast && (uintptr_t)xscales % 16 == 0;
    // an explicit request for the integer kernel (N <= 2) takes precedence
    const bool want_i8 = !q8 && gemv_i8_on() && N <= 2;
    if (fast && N == 1 && !q8 && !want_i8 && settings().stream) {
        // one token: the streaming kernel, when the shape fits it (several
        // matrices sharing X run in the same launch)
        const uint8_t *Ws[QMM_MAX_SEGS];
        float *Ys[QMM_MAX_SEGS];
        int64_t Ms[QMM_MAX_SEGS];
        for (int i = 0; i < nseg; ++i) {
            Ws[i] = static_cast<const uint8_t *>(seg[i].W);
            Ys[i] = seg[i].Y;
            Ms[i] = seg[i].M;
        }
        StreamPlan sp{};
        if (plan_gemv_stream(wt, Ms, nseg, K, di.num_sms, stream_force(), sp))
            return from_cuda(launch_gemv_stream(wt, sp, Ws, Ys, Ms, K, X, xt == QMM_X_BF16,
                                                !amax && static_weights(), di.status, g_wait_limit.load(), st,
                                                amax, idx, val));
    }
    const int tc_on = g_gemv_tc.load() >= 0 ? g_gemv_tc.load() : settings().tc;
    if (fast && nseg == 1 && N >= 2 && N <= settings().tc_max_n && !q8 && !want_i8 && tc_on &&
        gemv_tc_unit_bytes(wt)) {
        // several tokens: 16-row tiles on the tensor cores, when the shape fits
        TcPlan tp{};
        if (plan_gemv_tc(wt, seg[0].M, K, (int)N, di.num_sms, settings().tc_warps, tp)) {
            EncodeTiledFn enc = encode_fn();
            if (!enc) return QMM_ERR_CUDA;
            CUtensorMap wmap;
            cuuint64_t dims[2] = {(cuuint64_t)(row_bytes / 2), (cuuint64_t)seg[0].M};
            cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
            cuuint32_t box[2] = {(cuuint32_t)(gemv_tc_unit_bytes(wt) / 2), 16u};
            cuuint32_t estr[2] = {1u, 1u};
            if (enc(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void *>(seg[0].W), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
                return QMM_ERR_CUDA;
            return from_cuda(launch_gemv_tc(wt, tp, wmap, static_cast<const uint8_t *>(seg[0].W), seg[0].M, K, X,
                                            xt == QMM_X_BF16, (int)N, seg[0].Y, !amax && static_weights(), di.status,
                                            g_wait_limit.load(), st, amax, idx, val));
        }
    }
    if (fast) {
        EncodeTiledFn enc = encode_fn();
        if (!enc) return QMM_ERR_CUDA;
        const Settings &cfg = settings();
        const GemvTuning tun{cfg.gemv_rows, cfg.gemv_rg, cfg.gemv_ks, cfg.gemv_res};
        GemvPlan plan{};
        bool i8 = false;
        if (q8) {
            if (!plan_i8(1, wt, m_total, K, (int)N, 0, di.num_sms, plan)) return QMM_ERR_UNSUPPORTED;
            i8 = true;
        } else if (gemv_i8_on() && N <= 2) {
            i8 = plan_i8(0, wt, m_total, K, (int)N, xt == QMM_X_BF16, di.num_sms, plan);
        }
        if (!i8) plan = plan_gemv(m_total, K, (int)N, xt == QMM_X_BF16, di.num_sms, tun);
        GemvSegs segs{};
        segs.nseg = nseg;
        const int win = gemv_window_bytes(wt);
        for (int i = 0; i < nseg; ++i) {
            cuuint64_t dims[2] = {(cuuint64_t)(row_bytes / 2), (cuuint64_t)seg[i].M};
            cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
            cuuint32_t box[2] = {(cuuint32_t)(win / 2), (cuuint32_t)plan.rows};
            cuuint32_t estr[2] = {1u, 1u};
            if (enc(&segs.wmap[i], CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void *>(seg[i].W), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
                return QMM_ERR_CUDA;
            segs.Y[i] = seg[i].Y;
            segs.M[i] = (int)seg[i].M;
        }
        // Programmatic dependent launch in static-weights mode, except for the
        // resident-X and integer kernels (one CTA wave that holds its whole K
        // slice): there the early-launched dependents took slots and
        // bandwidth from the running grid (decode step 48.1 us with, 42.4 us
        // without, on GB300), while the ring GEMV gains 2%.
        const bool pdl = amax ? false : static_weights() && plan.resident == 0;
        if (q8)
            return from_cuda(launch_gemv_i8_q8(wt, plan, segs, static_cast<const int8_t *>(X), xscales, K, (int)N, pdl,
                                               di.status, g_wait_limit.load(), st, amax, idx, val));
        if (i8)
            return from_cuda(launch_gemv_i8_exact(wt, plan, segs, X, xt == QMM_X_BF16, K, (int)N, pdl, di.status,
                                                  g_wait_limit.load(), st, amax, idx, val));
        CUtensorMap xmap;
        const int xes = xt == QMM_X_F32 ? 4 : 2;
        cuuint64_t xdims[2] = {(cuuint64_t)K, (cuuint64_t)N};
        cuuint64_t xstrides[1] = {(cuuint64_t)K * xes};
        cuuint32_t xbox[2] = {256u, (cuuint32_t)N};
        cuuint32_t estr[2] = {1u, 1u};
        if (enc(&xmap, xt == QMM_X_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                const_cast<void *>(X), xdims, xstrides, xbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return QMM_ERR_CUDA;
        return from_cuda(launch_gemv_mma(wt, plan, segs, xmap, X, xt == QMM_X_BF16, K, (int)N,
                                         pdl, di.status, g_wait_limit.load(), st, amax,
                                         idx, val));
    }
    if (amax || q8) return QMM_ERR_UNSUPPORTED;
    for (int i = 0; i < nseg; ++i) {
        const qmm_status s = from_cuda(launch_gemv_generic(wt, static_cast<const uint8_t *>(seg[i].W), seg[i].M, K, X,
                                                           xt == QMM_X_BF16, (int)N, seg[i].Y, st));
        if (s != QMM_OK) return s;
    }
    return QMM_OK;
}

qmm_status gemv_impl(int wt, const void *W, size_t w_bytes, int64_t M, int64_t K, const void *X, int xt, int64_t N,
                     float *Y, void *stream, unsigned long long *amax = nullptr, int32_t *idx = nullptr,
                     float *val = nullptr) {
    const SegIn seg{W, w_bytes, M, Y};
    return gemv_segments(wt, &seg, 1, K, X, xt, N, stream, amax, idx, val);
}

// Every check qmm_gemm makes before it launches anything.
qmm_status gemm_check(int wt, const void *W, size_t w_bytes, int64_t M, int64_t K, const void *X, int xt, int64_t N,
                      const float *Y, const void *workspace, size_t ws_bytes, int &E, int &B) {
    qmm_status s = validate(wt, W, w_bytes, M, K, X, xt, N, Y, QMM_GEMM_MAX_N, E, B);
    if (s != QMM_OK) return s;
    const size_t ws_need = qmm_gemm_workspace_bytes(N, K, (qmm_xtype)xt);
    if (ws_need && (!workspace || ws_bytes < ws_need || ((uintptr_t)workspace % 16))) return QMM_ERR_INVALID_ARG;
    if (ws_need && (overlaps(workspace, ws_need, Y, (size_t)N * M * 4) ||
                    overlaps(workspace, ws_need, X, (size_t)N * K * 4) ||
                    overlaps(workspace, ws_need, W, (size_t)M * (K / E) * B)))
        return QMM_ERR_INVALID_ARG;
    // Tensor-core path geometry: 256-weight chunks, 16-byte aligned rows and
    // bases for the TMA descriptors.
    const int64_t row_bytes = K / E * B;
    if (K % 256 || row_bytes % 16 || (uintptr_t)W % 16 || (uintptr_t)X % 16) return QMM_ERR_UNSUPPORTED;
    if (M > (1ll << 31) - 1 || row_bytes / 2 > (1ll << 31)) return QMM_ERR_UNSUPPORTED;
    return QMM_OK;
}

// W2 / Y2 (optional): a second matrix of the same shape sharing X, computed
// in the same launch (checked by the caller).
qmm_status gemm_impl(int wt, const void *W, size_t w_bytes, int64_t M, int64_t K, const void *X, int xt, int64_t N,
                     float *Y, void *workspace, size_t ws_bytes, void *stream, const void *W2 = nullptr,
                     float *Y2 = nullptr) {
    int E, B;
    const qmm_status s = gemm_check(wt, W, w_bytes, M, K, X, xt, N, Y, workspace, ws_bytes, E, B);
    if (s != QMM_OK) return s;
    if (W2 && (uintptr_t)W2 % 16) return QMM_ERR_UNSUPPORTED;
    const int64_t row_bytes = K / E * B;
    DevInfo di;
    if (!dev_info(di)) return QMM_ERR_CUDA;
    EncodeTiledFn enc = encode_fn();
    if (!enc) return QMM_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    const void *xb = X;
    if (xt == QMM_X_F32) {
        cudaError_t e = launch_x_to_bf16(static_cast<const float *>(X), N * K, static_cast<uint16_t *>(workspace),
                                         static_weights(), st);
        if (e != cudaSuccess) return QMM_ERR_CUDA;
        xb = workspace;
    }
    const int64_t total_mt = (M + 127) / 128 * (W2 ? 2 : 1);
    const TilePlan plan = plan_tiles(wt, total_mt, N, K, di.num_sms);
    const int bn = plan.bn;

    CUtensorMap wmap, wmap2, xmap;
    for (int i = 0; i < (W2 ? 2 : 1); ++i) {
        const int win = gemm_raw_window_bytes(wt);
        cuuint64_t dims[2] = {(cuuint64_t)(row_bytes / 2), (cuuint64_t)M};
        cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
        cuuint32_t box[2] = {(cuuint32_t)(win / 2), 128u};
        cuuint32_t estr[2] = {1u, 1u};
        if (enc(i ? &wmap2 : &wmap, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void *>(i ? W2 : W), dims, strides,
                box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return QMM_ERR_CUDA;
    }
    if (!W2) wmap2 = wmap;
    {
        // {64 k within a block, token, 64-k block}: one copy = XG stages
        cuuint64_t dims[3] = {64u, (cuuint64_t)N, (cuuint64_t)(K / 64)};
        cuuint64_t strides[2] = {(cuuint64_t)K * 2, 128u};
        cuuint32_t box[3] = {64u, (cuuint32_t)bn, (cuuint32_t)gemm_x_stages_per_copy(bn)};
        cuuint32_t estr[3] = {1u, 1u, 1u};
        if (enc(&xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(xb), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return QMM_ERR_CUDA;
    }
    GemmArgs a;
    a.fmt = wt;
    a.M = M;
    a.K = K;
    a.N = (int)N;
    a.bn = bn;
    a.Y = Y;
    a.Y2 = W2 ? Y2 : nullptr;
    a.status = di.status;
    a.wait_limit = g_wait_limit.load();
    a.pdl = static_weights() ? 1 : 0;
    a.ks = plan.ks_a;
    a.mt0 = 0;
    a.mtn = plan.mt_a;
    cudaError_t e = launch_gemm_tc(a, wmap, wmap2, xmap, st);
    if (e == cudaSuccess && plan.mt_a < total_mt) {
        a.ks = plan.ks_b;
        a.mt0 = plan.mt_a;
        a.mtn = (int)(total_mt - plan.mt_a);
        e = launch_gemm_tc(a, wmap, wmap2, xmap, st);
    }
    return from_cuda(e);
}

}  // namespace

extern "C" {

qmm_status qmm_block_info(qmm_wtype wt, int *elems, int *bytes) {
    int E, B;
    if (!block_geom(wt, E, B)) return QMM_ERR_INVALID_ARG;
    if (elems) *elems = E;
    if (bytes) *bytes = B;
    return QMM_OK;
}

const char *qmm_status_str(qmm_status s) {
    switch (s) {
    case QMM_OK: return "QMM_OK";
    case QMM_ERR_INVALID_ARG: return "QMM_ERR_INVALID_ARG";
    case QMM_ERR_UNSUPPORTED: return "QMM_ERR_UNSUPPORTED";
    case QMM_ERR_CUDA: return "QMM_ERR_CUDA";
    case QMM_ERR_TIMEOUT: return "QMM_ERR_TIMEOUT";
    default: return "QMM_UNKNOWN_STATUS";
    }
}

size_t qmm_gemm_workspace_bytes(int64_t N, int64_t K, qmm_xtype xt) {
    if (xt != QMM_X_F32 || N < 1 || K < 1) return 0;
    return (size_t)N * (size_t)K * 2;
}

qmm_status qmm_gemv(qmm_wtype wt, const void *W, size_t w_bytes, int64_t M, int64_t K, const void *X, qmm_xtype xt,
                    int64_t N, float *Y, void *stream) {
    return gemv_impl(wt, W, w_bytes, M, K, X, xt, N, Y, stream);
}

static_assert(QMM_MAX_MATRICES == QMM_MAX_SEGS, "one launch holds every matrix of a fused call");

qmm_status qmm_gemv_multi(qmm_wtype wt, const qmm_matrix *mats, int nmat, int64_t K, const void *X, qmm_xtype xt,
                          int64_t N, void *stream) {
    if (!mats || nmat < 1 || nmat > QMM_MAX_MATRICES) return QMM_ERR_INVALID_ARG;
    SegIn seg[QMM_MAX_MATRICES];
    for (int i = 0; i < nmat; ++i) seg[i] = SegIn{mats[i].W, mats[i].w_bytes, mats[i].M, mats[i].Y};
    return gemv_segments(wt, seg, nmat, K, X, xt, N, stream);
}

qmm_status qmm_gemv_argmax(qmm_wtype wt, const void *W, size_t w_bytes, int64_t M, int64_t K, const void *X,
                           qmm_xtype xt, int64_t N, int32_t *idx, float *val, void *workspace, size_t ws_bytes,
                           void *stream) {
    if (!idx || !val || !workspace) return QMM_ERR_INVALID_ARG;
    if (N < 1 || N > QMM_GEMV_MAX_N || ws_bytes < (size_t)(N + 1) * 8 || ((uintptr_t)workspace % 8))
        return QMM_ERR_INVALID_ARG;
    if (M > (1ll << 31) - 1) return QMM_ERR_UNSUPPORTED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    auto *keys = static_cast<unsigned long long *>(workspace);
    // validate before anything is written (the outputs: idx, val, and the
    // workspace, none of which may overlap W or X)
    int E, B;
    qmm_status s = validate(wt, W, w_bytes, M, K, X, xt, N, val, QMM_GEMV_MAX_N, E, B, (size_t)N * 4);
    if (s != QMM_OK) return s;
    s = validate(wt, W, w_bytes, M, K, X, xt, N, reinterpret_cast<const float *>(idx), QMM_GEMV_MAX_N, E, B,
                 (size_t)N * 4);
    if (s != QMM_OK) return s;
    if (cudaMemsetAsync(keys, 0, (size_t)(N + 1) * 8, st) != cudaSuccess) return QMM_ERR_CUDA;   // keys + counter
    return gemv_impl(wt, W, w_bytes, M, K, X, xt, N, nullptr, stream, keys, idx, val);
}

qmm_status qmm_gemm(qmm_wtype wt, const void *W, size_t w_bytes, int64_t M, int64_t K, const void *X, qmm_xtype xt,
                    int64_t N, float *Y, void *workspace, size_t ws_bytes, void *stream) {
    return gemm_impl(wt, W, w_bytes, M, K, X, xt, N, Y, workspace, ws_bytes, stream);
}

// Whether qmm_matmul sends N tokens to the GEMV.
bool matmul_uses_gemv(int64_t N) {
    const Settings &cfg = settings();
    bool use_gemv = N <= cfg.gemv_max_n;
    if (cfg.force == 1) use_gemv = N <= QMM_GEMV_MAX_N;
    if (cfg.force == 2) use_gemv = false;
    return use_gemv;
}

qmm_status qmm_matmul(qmm_wtype wt, const void *W, size_t w_bytes, int64_t M, int64_t K, const void *X,
                      qmm_xtype xt, int64_t N, float *Y, void *workspace, size_t ws_bytes, void *stream) {
    if (matmul_uses_gemv(N)) return gemv_impl(wt, W, w_bytes, M, K, X, xt, N, Y, stream);
    return gemm_impl(wt, W, w_bytes, M, K, X, xt, N, Y, workspace, ws_bytes, stream);
}

qmm_status qmm_matmul_host(qmm_wtype wt, const void *W, size_t w_bytes, int64_t M, int64_t K, const void *X_host,
                           qmm_xtype xt, int64_t N, float *Y_host, void *x_dev, float *y_dev, void *workspace,
                           size_t ws_bytes, void *stream) {
    if (!X_host || !Y_host || !x_dev || !y_dev) return QMM_ERR_INVALID_ARG;
    if (N < 1 || N > QMM_GEMM_MAX_N || M < 1 || K < 1) return QMM_ERR_INVALID_ARG;
    if (xt != QMM_X_F32 && xt != QMM_X_BF16) return QMM_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t xbytes = (size_t)N * (size_t)K * (xt == QMM_X_F32 ? 4 : 2);
    const size_t ybytes = (size_t)N * (size_t)M * 4;
    // every check the compute call makes, before anything is copied: a bad
    // argument leaves x_dev, y_dev and Y_host untouched
    {
        int E = 0, B = 0;
        const qmm_status s =
            matmul_uses_gemv(N)
                ? validate(wt, W, w_bytes, M, K, x_dev, xt, N, y_dev, QMM_GEMV_MAX_N, E, B)
                : gemm_check(wt, W, w_bytes, M, K, x_dev, xt, N, y_dev, workspace, ws_bytes, E, B);
        if (s != QMM_OK) return s;
        if (overlaps(x_dev, xbytes, W, (size_t)M * (size_t)(K / E) * (size_t)B)) return QMM_ERR_INVALID_ARG;
    }
    if (cudaMemcpyAsync(x_dev, X_host, xbytes, cudaMemcpyHostToDevice, st) != cudaSuccess) return QMM_ERR_CUDA;
    t_after_copy = true;
    qmm_status s = qmm_matmul(wt, W, w_bytes, M, K, x_dev, xt, N, y_dev, workspace, ws_bytes, stream);
    t_after_copy = false;
    if (s != QMM_OK) return s;
    if (cudaMemcpyAsync(Y_host, y_dev, ybytes, cudaMemcpyDeviceToHost, st) != cudaSuccess) return QMM_ERR_CUDA;
    return QMM_OK;
}

qmm_status qmm_dequant(qmm_wtype wt, const void *W, size_t w_bytes, int64_t M, int64_t K, float *out,
                       void *stream) {
    int E, B;
    if (!block_geom(wt, E, B)) return QMM_ERR_INVALID_ARG;
    if (!W || !out || M < 1 || K < 1 || K % E || M > (1ll << 30) || K > (1ll << 24)) return QMM_ERR_INVALID_ARG;
    const size_t need = (size_t)M * (size_t)(K / E) * (size_t)B;
    if (w_bytes < need || ((uintptr_t)out % 16)) return QMM_ERR_INVALID_ARG;
    if (overlaps(out, (size_t)M * K * 4, W, need)) return QMM_ERR_INVALID_ARG;
    return from_cuda(launch_dequant(wt, static_cast<const uint8_t *>(W), M, K, out, static_cast<cudaStream_t>(stream)));
}

uint64_t qmm_kernel_launches(void) { return qmm::g_launches.load(); }

qmm_status qmm_last_device_error(void *stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return QMM_ERR_CUDA;
    DevInfo di;
    if (!dev_info(di)) return QMM_ERR_CUDA;
    unsigned v = 0, zero = 0;
    if (cudaMemcpy(&v, di.status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return QMM_ERR_CUDA;
    if (v && cudaMemcpy(di.status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return QMM_ERR_CUDA;
    return v == 0 ? QMM_OK : (qmm_status)v;
}

void qmm_set_static_weights(int on) { g_static_weights.store(on ? 1 : 0); }

qmm_status qmm_gemv_swiglu(qmm_wtype wt, const void *Wg, size_t wg_bytes, const void *Wu, size_t wu_bytes,
                           int64_t M, int64_t K, const void *X, qmm_xtype xt, int64_t N, float *Y, void *workspace,
                           size_t ws_bytes, void *stream) {
    int E, B;
    qmm_status s = validate(wt, Wg, wg_bytes, M, K, X, xt, N, Y, QMM_GEMV_MAX_N, E, B);
    if (s != QMM_OK) return s;
    s = validate(wt, Wu, wu_bytes, M, K, X, xt, N, Y, QMM_GEMV_MAX_N, E, B);
    if (s != QMM_OK) return s;
    const size_t ny = (size_t)N * (size_t)M;
    if (!workspace || ws_bytes < 2 * ny * 4 || (uintptr_t)workspace % 16) return QMM_ERR_INVALID_ARG;
    const size_t wb = (size_t)M * (size_t)(K / E) * (size_t)B;
    const size_t xs = xt == QMM_X_F32 ? 4 : 2;
    if (overlaps(workspace, 2 * ny * 4, Wg, wb) || overlaps(workspace, 2 * ny * 4, Wu, wb) ||
        overlaps(workspace, 2 * ny * 4, X, (size_t)N * K * xs) || overlaps(workspace, 2 * ny * 4, Y, ny * 4))
        return QMM_ERR_INVALID_ARG;
    float *g = static_cast<float *>(workspace);
    float *u = g + ny;
    const SegIn seg[2] = {{Wg, wg_bytes, M, g}, {Wu, wu_bytes, M, u}};
    s = gemv_segments(wt, seg, 2, K, X, xt, N, stream);
    if (s != QMM_OK) return s;
    return from_cuda(launch_swiglu(g, u, (int64_t)ny, Y, true, static_cast<cudaStream_t>(stream)));
}

void qmm_set_gemv_i8(int on) { g_gemv_i8.store(on < 0 ? -1 : (on ? 1 : 0)); }

void qmm_set_gemv_tc(int on) { g_gemv_tc.store(on < 0 ? -1 : (on ? 1 : 0)); }

void qmm_set_gemv_stream(int rows_per_task, int warps, int slots, int ctas_per_sm, int direct) {
    const int v[5] = {rows_per_task, warps, slots, ctas_per_sm, direct};
    for (int i = 0; i < 5; ++i) g_stream_force[i].store(v[i] < 0 ? -1 : v[i]);
}

qmm_status qmm_gemv_stream_plan(qmm_wtype wt, int64_t M, int64_t K, int32_t *plan) {
    if (!plan || M < 1 || K < 1) return QMM_ERR_INVALID_ARG;
    int E = 0, B = 0;
    if (!block_geom(wt, E, B)) return QMM_ERR_INVALID_ARG;
    DevInfo di;
    if (!dev_info(di)) return QMM_ERR_CUDA;
    StreamPlan sp{};
    if (!plan_gemv_stream(wt, M, K, di.num_sms, stream_force(), sp)) return QMM_ERR_UNSUPPORTED;
    plan[0] = sp.grid;
    plan[1] = sp.warps;
    plan[2] = sp.S;
    plan[3] = sp.R;
    plan[4] = sp.smem;
    plan[5] = sp.direct;
    return QMM_OK;
}

size_t qmm_q8act_workspace_bytes(int64_t N, int64_t K) {
    if (N < 1 || K < 1) return 0;
    return ((size_t)N * (size_t)K + 15) / 16 * 16 + (size_t)N * (size_t)(K / 32) * 4;
}

qmm_status qmm_quantize_q8_0(const void *X, qmm_xtype xt, int64_t N, int64_t K, float *scales, int8_t *quants,
                             void *stream) {
    if (!X || !scales || !quants || (xt != QMM_X_F32 && xt != QMM_X_BF16)) return QMM_ERR_INVALID_ARG;
    if (N < 1 || K < 32 || K % 32 || N > (1ll << 30) || K > (1ll << 24)) return QMM_ERR_INVALID_ARG;
    const size_t xs = xt == QMM_X_F32 ? 4 : 2;
    if ((uintptr_t)X % xs || (uintptr_t)scales % 4) return QMM_ERR_INVALID_ARG;
    const size_t nx = (size_t)N * (size_t)K;
    if (overlaps(scales, nx / 32 * 4, X, nx * xs) || overlaps(quants, nx, X, nx * xs) ||
        overlaps(quants, nx, scales, nx / 32 * 4))
        return QMM_ERR_INVALID_ARG;
    return from_cuda(launch_quantize_q8_0(X, xt == QMM_X_BF16, (int64_t)nx, scales, quants, static_weights(),
                                          static_cast<cudaStream_t>(stream)));
}

qmm_status qmm_gemv_preq(qmm_wtype wt, const void *W, size_t w_bytes, int64_t M, int64_t K, const float *scales,
                         const int8_t *quants, int64_t N, float *Y, void *stream) {
    if (!scales || !quants) return QMM_ERR_INVALID_ARG;
    const SegIn seg{W, w_bytes, M, Y};
    return gemv_segments(wt, &seg, 1, K, quants, QMM_X_F32, N, stream, nullptr, nullptr, nullptr, scales);
}

qmm_status qmm_gemv_q8act(qmm_wtype wt, const void *W, size_t w_bytes, int64_t M, int64_t K, const void *X,
                          qmm_xtype xt, int64_t N, float *Y, void *workspace, size_t ws_bytes, void *stream) {
    int E, B;
    qmm_status s = validate(wt, W, w_bytes, M, K, X, xt, N, Y, QMM_GEMV_MAX_N, E, B);
    if (s != QMM_OK) return s;
    const size_t need = qmm_q8act_workspace_bytes(N, K);
    if (!workspace || ws_bytes < need || (uintptr_t)workspace % 16) return QMM_ERR_INVALID_ARG;
    const size_t xs = xt == QMM_X_F32 ? 4 : 2;
    if (overlaps(workspace, need, Y, (size_t)N * M * 4) || overlaps(workspace, need, X, (size_t)N * K * xs) ||
        overlaps(workspace, need, W, (size_t)M * (K / E) * B))
        return QMM_ERR_INVALID_ARG;
    if (K % 256) return QMM_ERR_UNSUPPORTED;
    int8_t *q = static_cast<int8_t *>(workspace);
    float *sc = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + ((size_t)N * K + 15) / 16 * 16);
    s = qmm_quantize_q8_0(X, xt, N, K, sc, q, stream);
    if (s != QMM_OK) return s;
    return qmm_gemv_preq(wt, W, w_bytes, M, K, sc, q, N, Y, stream);
}

size_t qmm_gemm_q8act_workspace_bytes(int64_t N, int64_t K) {
    if (N < 1 || K < 1) return 0;
    return (size_t)N * (size_t)K * 2;
}

qmm_status qmm_gemm_q8act(qmm_wtype wt, const void *W, size_t w_bytes, int64_t M, int64_t K, const void *X,
                          qmm_xtype xt, int64_t N, float *Y, void *workspace, size_t ws_bytes, void *stream) {
    int E, B;
    // the checks of qmm_gemm on X as given, plus the activation workspace
    qmm_status s = validate(wt, W, w_bytes, M, K, X, xt, N, Y, QMM_GEMM_MAX_N, E, B);
    if (s != QMM_OK) return s;
    const size_t need = qmm_gemm_q8act_workspace_bytes(N, K);
    const size_t xs = xt == QMM_X_F32 ? 4 : 2;
    if (!workspace || ws_bytes < need || (uintptr_t)workspace % 16) return QMM_ERR_INVALID_ARG;
    if (overlaps(workspace, need, Y, (size_t)N * M * 4) || overlaps(workspace, need, X, (size_t)N * K * xs) ||
        overlaps(workspace, need, W, (size_t)M * (K / E) * B))
        return QMM_ERR_INVALID_ARG;
    s = gemm_check(wt, W, w_bytes, M, K, workspace, QMM_X_BF16, N, Y, nullptr, 0, E, B);
    if (s != QMM_OK) return s;
    if (launch_quantize_q8_0_bf16(X, xt == QMM_X_BF16, N * K, static_cast<uint16_t *>(workspace), static_weights(),
                                  static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return QMM_ERR_CUDA;
    return gemm_impl(wt, W, w_bytes, M, K, workspace, QMM_X_BF16, N, Y, nullptr, 0, stream);
}

size_t qmm_gemm_swiglu_workspace_bytes(int64_t N, int64_t M, int64_t K, qmm_xtype xt) {
    if (N < 1 || M < 1 || K < 1) return 0;
    return (qmm_gemm_workspace_bytes(N, K, xt) + 15) / 16 * 16 + 2 * (size_t)N * (size_t)M * 4;
}

qmm_status qmm_gemm_swiglu(qmm_wtype wt, const void *Wg, size_t wg_bytes, const void *Wu, size_t wu_bytes, int64_t M,
                           int64_t K, const void *X, qmm_xtype xt, int64_t N, float *Y, void *workspace,
                           size_t ws_bytes, void *stream) {
    int E, B;
    qmm_status s = validate(wt, Wg, wg_bytes, M, K, X, xt, N, Y, QMM_GEMM_MAX_N, E, B);
    if (s != QMM_OK) return s;
    s = validate(wt, Wu, wu_bytes, M, K, X, xt, N, Y, QMM_GEMM_MAX_N, E, B);
    if (s != QMM_OK) return s;
    const size_t need = qmm_gemm_swiglu_workspace_bytes(N, M, K, xt);
    if (!workspace || ws_bytes < need || (uintptr_t)workspace % 16) return QMM_ERR_INVALID_ARG;
    const size_t wb = (size_t)M * (size_t)(K / E) * (size_t)B, ny = (size_t)N * (size_t)M;
    const size_t xs = xt == QMM_X_F32 ? 4 : 2;
    if (overlaps(workspace, need, Wg, wb) || overlaps(workspace, need, Wu, wb) ||
        overlaps(workspace, need, X, (size_t)N * K * xs) || overlaps(workspace, need, Y, ny * 4))
        return QMM_ERR_INVALID_ARG;
    const size_t xws = (qmm_gemm_workspace_bytes(N, K, xt) + 15) / 16 * 16;
    float *g = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + xws);
    float *u = g + ny;
    s = gemm_check(wt, Wg, wg_bytes, M, K, X, xt, N, g, workspace, xws, E, B);
    if (s != QMM_OK) return s;
    s = gemm_impl(wt, Wg, wg_bytes, M, K, X, xt, N, g, workspace, xws, stream, Wu, u);
    if (s != QMM_OK) return s;
    return from_cuda(launch_swiglu(g, u, (int64_t)ny, Y, static_weights(), static_cast<cudaStream_t>(stream)));
}

void qmm_set_wait_limit(uint64_t cycles) {
    if (cycles < 1) cycles = 1;
    if (cycles > (1ull << 40)) cycles = 1ull << 40;
    g_wait_limit.store(cycles);
}

}  // extern "C"
