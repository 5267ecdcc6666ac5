// abi.cu -- the extern "C" entry points of libexl3 (declared in include/exl3.h):
// argument checks, workspace layout, and the orchestration of the quantize
// chain and of the device-resident golden-section search.
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "common.cuh"

namespace exl3 {

static thread_local char g_err[512] = "no error";

exl3_status set_error(exl3_status st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return st;
}

exl3_status cuda_check(cudaError_t e, const char *what) {
    if (e == cudaSuccess)
        return EXL3_OK;
    return set_error(EXL3_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

int device_sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        (void)cudaGetLastError();
        return 152;   // GB300 (two dies x 76 SMs) when no device can be queried
    }
    return n;
}

// ---- profiling ----------------------------------------------------------------
static std::atomic<bool> g_prof_on{false};
static std::atomic<int64_t> g_launches{0};
static std::mutex g_prof_mu;
struct EvPair { cudaEvent_t a, b; bool used; };
static std::vector<EvPair> g_ev;     // created lazily, reused
static size_t g_ev_next = 0;
static thread_local cudaEvent_t t_open = nullptr;
constexpr size_t kMaxEv = 4096;

void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

// kernel of the calling thread's most recent rotation launch (exl3_rotate_last_kernel)
static thread_local int t_rot_kernel = 0;
void note_rotate_kernel(int which) { t_rot_kernel = which; }
int last_rotate_kernel() { return t_rot_kernel; }

void profile_encode_begin(cudaStream_t s) {
    t_open = nullptr;
    if (!g_prof_on.load(std::memory_order_relaxed))
        return;
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (g_ev_next >= kMaxEv)
        return;
    if (g_ev_next == g_ev.size()) {
        EvPair e{nullptr, nullptr, false};
        if (cudaEventCreate(&e.a) != cudaSuccess || cudaEventCreate(&e.b) != cudaSuccess) {
            (void)cudaGetLastError();
            return;
        }
        g_ev.push_back(e);
    }
    EvPair &e = g_ev[g_ev_next];
    if (cudaEventRecord(e.a, s) != cudaSuccess) {
        (void)cudaGetLastError();
        return;
    }
    t_open = e.b;
}

void profile_encode_end(cudaStream_t s) {
    if (!t_open)
        return;
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (cudaEventRecord(t_open, s) == cudaSuccess && g_ev_next < g_ev.size() &&
        g_ev[g_ev_next].b == t_open) {
        g_ev[g_ev_next].used = true;
        g_ev_next++;
    } else {
        (void)cudaGetLastError();
    }
    t_open = nullptr;
}

namespace {

constexpr size_t kAlign = 256;

bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
    return x < y + nb && y < x + na;
}

bool k_ok(int K) { return K >= 1 && K <= 4; }

size_t dt_size(int dt) { return dt == EXL3_BF16 ? 2 : 4; }

// ---- workspace carving --------------------------------------------------
struct Carver {
    char *base;
    size_t off = 0;
    explicit Carver(void *b) : base((char *)b) {}
    void *take(size_t bytes) {
        void *p = base ? base + off : nullptr;
        off = align_up(off + bytes, kAlign);
        return p;
    }
};

// Persistent blocks for the whole machine: one per SM (one tile per block at
// a time; at K = 3 and 4 a pair of tiles).
int encode_grid_full(int64_t n_tiles, int K) {
    (void)K;
    const int64_t sm = device_sm_count();
    return (int)(n_tiles < sm ? n_tiles : sm);
}

// Grid that fits `cap` block slices; 0 if none fits.
int64_t fit_blocks(int64_t full, int64_t cap, int K) {
    (void)K;
    return full < cap ? full : cap;
}

struct QuantWs {
    float *R;
    double *tile_sums;
    double *tree_scr;
    double *scal;      // [0] sum R^2, [1] sum err^2
    float *fscal;      // [0] scale, [1] inv scale
    uint32_t *enc;     // encode scratch
    size_t enc_bytes;
    // gss extras
    uint32_t *eval_codes;
    double *gss_state;
    size_t total;
};

QuantWs carve_quant(void *ws, int64_t rows, int64_t cols, int K, bool gss, int grid) {
    const int64_t n_tiles = (rows / 16) * (cols / 16);
    Carver c(ws);
    QuantWs q{};
    q.R = (float *)c.take((size_t)rows * cols * sizeof(float));
    q.tile_sums = (double *)c.take((size_t)n_tiles * sizeof(double));
    q.tree_scr = (double *)c.take(tree_scratch_doubles(n_tiles) * sizeof(double));
    q.scal = (double *)c.take(8 * sizeof(double));
    q.fscal = (float *)c.take(8 * sizeof(float));
    if (gss) {
        q.eval_codes = (uint32_t *)c.take((size_t)n_tiles * 32 * K);
        q.gss_state = (double *)c.take(32 * sizeof(double));
    }
    q.enc_bytes = (size_t)grid * kEncodeBlockScratchBytes;
    q.enc = (uint32_t *)c.take(q.enc_bytes);
    q.total = c.off;
    return q;
}

// ---- scalar kernels --------------------------------------------------------

// sigma = sqrt(sum / n); s = fl32(g * sigma); inv = fl32(1 / s).
// g comes from *g_dev when non-null.
__global__ void scale_kernel(const double *sum, int64_t n, double g, const double *g_dev,
                             float *fscal, double *sigma_out, float *scale_out) {
    double sigma = __dsqrt_rn(__ddiv_rn(*sum, (double)n));
    if (sigma == 0.0)
        sigma = 1.0;   // all-zero matrix: any scale codes it; use g itself
    const double gg = g_dev ? *g_dev : g;
    float s = __double2float_rn(__dmul_rn(gg, sigma));
    float inv = __fdiv_rn(1.0f, s);
    if (!isfinite(sigma) || !isfinite(s) || !isfinite(inv)) {
        // a non-finite weight (or a scale out of binary32 range) is rejected:
        // NaN scale, and the encode kernels skip every tile when 1/s is not finite
        s = __int_as_float(0x7fffffff);
        inv = s;
    }
    fscal[0] = s;
    fscal[1] = inv;
    if (sigma_out) *sigma_out = sigma;
    if (scale_out) *scale_out = s;
}

__global__ void mse_kernel(const double *sum, int64_t n, double *mse_out) {
    *mse_out = __ddiv_rn(*sum, (double)n);
}

// Golden-section state (doubles): see exl3_gss_scale in include/exl3.h.
enum { GA = 0, GB, GX1, GX2, GF1, GF2, GPHI, GCUR, GBEST, GBESTF, GN, GWHICH, GIMPROVED, GNEVAL };

__global__ void gss_init_kernel(double *st, double lo, double hi, int n_eval) {
    const double phi = __ddiv_rn(__dsub_rn(__dsqrt_rn(5.0), 1.0), 2.0);
    st[GA] = lo;
    st[GB] = hi;
    st[GPHI] = phi;
    st[GX1] = __dsub_rn(hi, __dmul_rn(phi, __dsub_rn(hi, lo)));
    st[GX2] = __dadd_rn(lo, __dmul_rn(phi, __dsub_rn(hi, lo)));
    st[GCUR] = st[GX1];
    st[GBEST] = 0.0;
    st[GBESTF] = __longlong_as_double(0x7ff0000000000000ll);
    st[GN] = 0.0;
    st[GWHICH] = 1.0;
    st[GIMPROVED] = 0.0;
    st[GNEVAL] = (double)n_eval;
}

// Record f at the current point, update the best, choose the next point.
__global__ void gss_update_kernel(double *st, const double *sum, int64_t n, const float *fscal,
                                  float *best_scale, double *best_g, double *best_mse,
                                  double *history) {
    const double f = __ddiv_rn(*sum, (double)n);
    const double x = st[GCUR];
    const int e = (int)st[GN];
    const int n_eval = (int)st[GNEVAL];
    if (history) {
        history[2 * e] = x;
        history[2 * e + 1] = f;
    }
    const bool better = f < st[GBESTF] || (f == st[GBESTF] && x < st[GBEST]);
    st[GIMPROVED] = better ? 1.0 : 0.0;
    if (better) {
        st[GBEST] = x;
        st[GBESTF] = f;
        *best_scale = fscal[0];
        *best_g = x;
        *best_mse = f;
    }
    if (e == 0) {
        st[GF1] = f;
        st[GCUR] = st[GX2];
    } else {
        if (e == 1 || st[GWHICH] == 2.0)
            st[GF2] = f;
        else
            st[GF1] = f;
        if (e + 1 < n_eval) {
            const double phi = st[GPHI];
            if (st[GF1] <= st[GF2]) {
                st[GB] = st[GX2];
                st[GX2] = st[GX1];
                st[GF2] = st[GF1];
                st[GX1] = __dsub_rn(st[GB], __dmul_rn(phi, __dsub_rn(st[GB], st[GA])));
                st[GCUR] = st[GX1];
                st[GWHICH] = 1.0;
            } else {
                st[GA] = st[GX1];
                st[GX1] = st[GX2];
                st[GF1] = st[GF2];
                st[GX2] = __dadd_rn(st[GA], __dmul_rn(phi, __dsub_rn(st[GB], st[GA])));
                st[GCUR] = st[GX2];
                st[GWHICH] = 2.0;
            }
        }
    }
    st[GN] = (double)(e + 1);
}

__global__ void copy_if_kernel(const double *flag, const uint4 *__restrict__ src, uint4 *__restrict__ dst,
                               int64_t n16) {
    if (*flag == 0.0)
        return;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16;
         i += (int64_t)gridDim.x * blockDim.x)
        dst[i] = src[i];
}

// ---- shared checks ----------------------------------------------------------

exl3_status check_matrix(const void *p, const char *name, int dt, int64_t rows, int64_t cols,
                         int64_t mult) {
    if (!p)
        return set_error(EXL3_ERR_INVALID_ARG, "%s is NULL", name);
    if (dt != EXL3_F32 && dt != EXL3_BF16)
        return set_error(EXL3_ERR_INVALID_ARG, "%s: dtype %d is not EXL3_F32/EXL3_BF16", name, dt);
    if (!aligned(p, dt_size(dt)))
        return set_error(EXL3_ERR_INVALID_ARG, "%s is not %zu-byte aligned", name, dt_size(dt));
    if (rows <= 0 || cols <= 0)
        return set_error(EXL3_ERR_INVALID_ARG, "rows=%lld cols=%lld must be positive",
                         (long long)rows, (long long)cols);
    if (rows % mult || cols % mult)
        return set_error(EXL3_ERR_UNSUPPORTED, "rows=%lld cols=%lld must be multiples of %lld",
                         (long long)rows, (long long)cols, (long long)mult);
    if (rows > (1ll << 24) || cols > (1ll << 24) || rows * cols > (1ll << 34))
        return set_error(EXL3_ERR_INVALID_ARG, "matrix %lldx%lld is too large", (long long)rows,
                         (long long)cols);
    return EXL3_OK;
}

exl3_status check_signs(const float *su, const float *sv) {
    if (!su || !sv)
        return set_error(EXL3_ERR_INVALID_ARG, "su/sv must not be NULL");
    if (!aligned(su, 4) || !aligned(sv, 4))
        return set_error(EXL3_ERR_INVALID_ARG, "su/sv must be 4-byte aligned");
    return EXL3_OK;
}

exl3_status check_k(int K) {
    if (!k_ok(K))
        return set_error(EXL3_ERR_UNSUPPORTED, "K=%d: this build encodes K in {1,2,3,4}", K);
    return EXL3_OK;
}

exl3_status check_ptr(const void *p, const char *name, size_t al) {
    if (!p)
        return set_error(EXL3_ERR_INVALID_ARG, "%s is NULL", name);
    if (!aligned(p, al))
        return set_error(EXL3_ERR_INVALID_ARG, "%s is not %zu-byte aligned", name, al);
    return EXL3_OK;
}

// ---- the quantize chain ------------------------------------------------------

exl3_status run_quantize(const QuantWs &q, int grid, const void *W, int dt, int64_t rows,
                         int64_t cols, const float *su, const float *sv, int K, double g,
                         const double *g_dev, uint32_t *codes, float *scale_out, double *mse_out,
                         double *sigma_out, float *What, cudaStream_t s) {
    const int64_t n_tiles = (rows / 16) * (cols / 16);
    exl3_status st;
    RotateLaunch rf{};
    rf.inverse = 0;
    rf.src = dt == EXL3_BF16 ? SRC_BF16 : SRC_F32;
    rf.in = W;
    rf.su = su;
    rf.sv = sv;
    rf.rows = rows;
    rf.cols = cols;
    rf.out = q.R;
    rf.tile_sums = q.tile_sums;
    if ((st = launch_rotate(rf, s)) != EXL3_OK) return st;
    if ((st = launch_tree_sum(q.tile_sums, n_tiles, q.tree_scr, &q.scal[0], s)) != EXL3_OK) return st;
    scale_kernel<<<1, 1, 0, s>>>(&q.scal[0], rows * cols, g, g_dev, q.fscal, sigma_out, scale_out);
    note_launch();
    if ((st = cuda_check(cudaGetLastError(), "scale launch")) != EXL3_OK) return st;

    EncodeLaunch el{};
    el.Y = q.R;
    el.rows = rows;
    el.cols = cols;
    el.K = K;
    el.T = 256;
    el.row_tiles = 0;
    el.inv_scale = 1.0f;
    el.inv_scale_dev = &q.fscal[1];
    el.codes = codes;
    el.tile_cost = nullptr;
    el.scratch = q.enc;
    el.grid = grid;
    if ((st = launch_encode(el, s)) != EXL3_OK) return st;

    RotateLaunch ri{};
    ri.inverse = 1;
    ri.src = SRC_CODES;
    ri.in = codes;
    ri.K = K;
    ri.scale_dev = &q.fscal[0];
    ri.su = su;
    ri.sv = sv;
    ri.rows = rows;
    ri.cols = cols;
    ri.out = What;
    ri.ref = W;
    ri.ref_dt = dt;
    ri.tile_sums = q.tile_sums;
    if ((st = launch_rotate(ri, s)) != EXL3_OK) return st;
    if ((st = launch_tree_sum(q.tile_sums, n_tiles, q.tree_scr, &q.scal[1], s)) != EXL3_OK) return st;
    if (mse_out) {
        mse_kernel<<<1, 1, 0, s>>>(&q.scal[1], rows * cols, mse_out);
    note_launch();
        if ((st = cuda_check(cudaGetLastError(), "mse launch")) != EXL3_OK) return st;
    }
    return EXL3_OK;
}

}  // namespace
}  // namespace exl3

using namespace exl3;

extern "C" {

const char *exl3_status_str(int status) {
    switch (status) {
    case EXL3_OK: return "EXL3_OK";
    case EXL3_ERR_INVALID_ARG: return "EXL3_ERR_INVALID_ARG";
    case EXL3_ERR_UNSUPPORTED: return "EXL3_ERR_UNSUPPORTED";
    case EXL3_ERR_WORKSPACE: return "EXL3_ERR_WORKSPACE";
    case EXL3_ERR_CUDA: return "EXL3_ERR_CUDA";
    case EXL3_ERR_NUMERIC: return "EXL3_ERR_NUMERIC";
    case EXL3_ERR_TIMEOUT: return "EXL3_ERR_TIMEOUT";
    default: return "EXL3_ERR_UNKNOWN";
    }
}

const char *exl3_last_error(void) { return g_err; }

int exl3_rotate_last_kernel(void) { return exl3::last_rotate_kernel(); }

int exl3_version(void) { return 100; }

int exl3_supports_k(int K) { return k_ok(K) ? 1 : 0; }

exl3_status exl3_rotate(const void *W, int dt, int64_t rows, int64_t cols, const float *su,
                        const float *sv, int inverse, float *out, void *stream) {
    exl3_status st;
    if ((st = check_matrix(W, "W", dt, rows, cols, 128)) != EXL3_OK) return st;
    if ((st = check_signs(su, sv)) != EXL3_OK) return st;
    if ((st = check_ptr(out, "out", 4)) != EXL3_OK) return st;
    if (inverse != 0 && inverse != 1)
        return set_error(EXL3_ERR_INVALID_ARG, "inverse must be 0 or 1");
    if (inverse && dt != EXL3_F32)
        return set_error(EXL3_ERR_INVALID_ARG, "the inverse rotation takes fp32 input");
    const size_t nin = (size_t)rows * cols * dt_size(dt), nout = (size_t)rows * cols * 4;
    if (overlaps(W, nin, out, nout) && !((const void *)out == W && dt == EXL3_F32))
        return set_error(EXL3_ERR_INVALID_ARG, "out overlaps W (only exact in-place fp32 is allowed)");
    RotateLaunch r{};
    r.inverse = inverse;
    r.src = dt == EXL3_BF16 ? SRC_BF16 : SRC_F32;
    r.in = W;
    r.su = su;
    r.sv = sv;
    r.rows = rows;
    r.cols = cols;
    r.out = out;
    return launch_rotate(r, (cudaStream_t)stream);
}

size_t exl3_encode_workspace_bytes(int64_t n_tiles, int K) {
    if (!k_ok(K) || n_tiles < 0)
        return 0;
    const int64_t g = encode_grid_full(n_tiles, K);
    return (size_t)(g > 0 ? g : 1) * kEncodeBlockScratchBytes;
}

size_t exl3_encode_workspace_min_bytes(int K) {
    return k_ok(K) ? kEncodeBlockScratchBytes : 0;
}

exl3_status exl3_encode_tiles(const float *Y, int64_t rows, int64_t cols, int K, float scale,
                              uint16_t *codes, float *tile_cost, void *ws, size_t ws_bytes,
                              void *stream) {
    exl3_status st;
    if ((st = check_matrix(Y, "Y", EXL3_F32, rows, cols, 16)) != EXL3_OK) return st;
    if ((st = check_k(K)) != EXL3_OK) return st;
    if ((st = check_ptr(codes, "codes", 4)) != EXL3_OK) return st;
    if (tile_cost && !aligned(tile_cost, 4))
        return set_error(EXL3_ERR_INVALID_ARG, "tile_cost is not 4-byte aligned");
    if (!(scale > 0.0f) || !std::isfinite(scale) || !std::isfinite(1.0f / scale))
        return set_error(EXL3_ERR_INVALID_ARG, "scale and 1 / scale must be positive and finite");
    if (!ws || !aligned(ws, kAlign))
        return set_error(EXL3_ERR_INVALID_ARG, "workspace must be non-NULL and 256-byte aligned");
    const int64_t n_tiles = (rows / 16) * (cols / 16);
    const int64_t grid = fit_blocks(encode_grid_full(n_tiles, K),
                                    (int64_t)(ws_bytes / kEncodeBlockScratchBytes), K);
    if (grid < 1)
        return set_error(EXL3_ERR_WORKSPACE, "workspace %zu bytes < minimum %zu", ws_bytes,
                         exl3_encode_workspace_min_bytes(K));
    EncodeLaunch el{};
    el.Y = Y;
    el.rows = rows;
    el.cols = cols;
    el.K = K;
    el.T = 256;
    el.row_tiles = 0;
    el.inv_scale = 1.0f / scale;   // IEEE binary32 division, round to nearest
    el.inv_scale_dev = nullptr;
    el.codes = reinterpret_cast<uint32_t *>(codes);
    el.tile_cost = tile_cost;
    el.scratch = reinterpret_cast<uint32_t *>(ws);
    el.grid = (int)grid;
    return launch_encode(el, (cudaStream_t)stream);
}

static exl3_status check_rows(int64_t n_rows, int T, int K) {
    exl3_status st;
    if ((st = check_k(K)) != EXL3_OK) return st;
    if (n_rows <= 0 || n_rows > (1ll << 26))
        return set_error(EXL3_ERR_INVALID_ARG, "n_rows=%lld outside [1, 2^26]", (long long)n_rows);
    if (T < 16 || T > 256 || (T & 1) || (T * K) % 32)
        return set_error(EXL3_ERR_UNSUPPORTED,
                         "T=%d: need an even T in [16, 256] with T*K a multiple of 32 (K=%d)", T, K);
    return EXL3_OK;
}

exl3_status exl3_encode_rows(const float *Y, int64_t n_rows, int T, int K, float scale,
                             uint16_t *codes, float *row_cost, void *ws, size_t ws_bytes,
                             void *stream) {
    exl3_status st;
    if ((st = check_rows(n_rows, T, K)) != EXL3_OK) return st;
    if ((st = check_ptr(Y, "Y", 4)) != EXL3_OK) return st;
    if ((st = check_ptr(codes, "codes", 4)) != EXL3_OK) return st;
    if (row_cost && !aligned(row_cost, 4))
        return set_error(EXL3_ERR_INVALID_ARG, "row_cost is not 4-byte aligned");
    if (!(scale > 0.0f) || !std::isfinite(scale) || !std::isfinite(1.0f / scale))
        return set_error(EXL3_ERR_INVALID_ARG, "scale and 1 / scale must be positive and finite");
    if (!ws || !aligned(ws, kAlign))
        return set_error(EXL3_ERR_INVALID_ARG, "workspace must be non-NULL and 256-byte aligned");
    const int64_t grid = fit_blocks(encode_grid_full(n_rows, K),
                                    (int64_t)(ws_bytes / kEncodeBlockScratchBytes), K);
    if (grid < 1)
        return set_error(EXL3_ERR_WORKSPACE, "workspace %zu bytes < minimum %zu", ws_bytes,
                         exl3_encode_workspace_min_bytes(K));
    EncodeLaunch el{};
    el.Y = Y;
    el.rows = n_rows;
    el.cols = T;
    el.K = K;
    el.T = T;
    el.row_tiles = 1;
    el.inv_scale = 1.0f / scale;
    el.inv_scale_dev = nullptr;
    el.codes = reinterpret_cast<uint32_t *>(codes);
    el.tile_cost = row_cost;
    el.scratch = reinterpret_cast<uint32_t *>(ws);
    el.grid = (int)grid;
    return launch_encode(el, (cudaStream_t)stream);
}

exl3_status exl3_decode_rows(const uint16_t *codes, int64_t n_rows, int T, int K, float scale,
                             float *Yhat, void *stream) {
    exl3_status st;
    if ((st = check_rows(n_rows, T, K)) != EXL3_OK) return st;
    if ((st = check_ptr(codes, "codes", 4)) != EXL3_OK) return st;
    if ((st = check_ptr(Yhat, "Yhat", 4)) != EXL3_OK) return st;
    if (!std::isfinite(scale))
        return set_error(EXL3_ERR_INVALID_ARG, "scale must be finite");
    return launch_decode_rows(reinterpret_cast<const uint32_t *>(codes), n_rows, T, K, scale, Yhat,
                              (cudaStream_t)stream);
}

exl3_status exl3_decode_tiles(const uint16_t *codes, int64_t rows, int64_t cols, int K, float scale,
                              float *Yhat, void *stream) {
    exl3_status st;
    if ((st = check_ptr(codes, "codes", 4)) != EXL3_OK) return st;
    if ((st = check_matrix(Yhat, "Yhat", EXL3_F32, rows, cols, 16)) != EXL3_OK) return st;
    if ((st = check_k(K)) != EXL3_OK) return st;
    if (!std::isfinite(scale))
        return set_error(EXL3_ERR_INVALID_ARG, "scale must be finite");
    return launch_decode(reinterpret_cast<const uint32_t *>(codes), rows, cols, K, scale, nullptr,
                         Yhat, (cudaStream_t)stream);
}

size_t exl3_mse_workspace_bytes(int64_t rows, int64_t cols) {
    if (rows <= 0 || cols <= 0) return 0;
    const int64_t n = (rows / 16) * (cols / 16);
    return align_up((size_t)n * sizeof(double), kAlign) +
           align_up(tree_scratch_doubles(n) * sizeof(double), kAlign) + kAlign;
}

exl3_status exl3_mse(const void *W, int dt, const float *What, int64_t rows, int64_t cols,
                     double *mse_out, void *ws, size_t ws_bytes, void *stream) {
    exl3_status st;
    if ((st = check_matrix(W, "W", dt, rows, cols, 16)) != EXL3_OK) return st;
    if ((st = check_matrix(What, "What", EXL3_F32, rows, cols, 16)) != EXL3_OK) return st;
    if ((st = check_ptr(mse_out, "mse_out", 8)) != EXL3_OK) return st;
    if (!ws || !aligned(ws, kAlign))
        return set_error(EXL3_ERR_INVALID_ARG, "workspace must be non-NULL and 256-byte aligned");
    if (ws_bytes < exl3_mse_workspace_bytes(rows, cols))
        return set_error(EXL3_ERR_WORKSPACE, "workspace %zu bytes < %zu", ws_bytes,
                         exl3_mse_workspace_bytes(rows, cols));
    const int64_t n = (rows / 16) * (cols / 16);
    Carver c(ws);
    double *ts = (double *)c.take((size_t)n * sizeof(double));
    double *scr = (double *)c.take(tree_scratch_doubles(n) * sizeof(double));
    double *sum = (double *)c.take(sizeof(double));
    cudaStream_t s = (cudaStream_t)stream;
    if ((st = launch_tile_sumsq(W, dt, What, rows, cols, ts, s)) != EXL3_OK) return st;
    if ((st = launch_tree_sum(ts, n, scr, sum, s)) != EXL3_OK) return st;
    mse_kernel<<<1, 1, 0, s>>>(sum, rows * cols, mse_out);
    note_launch();
    return cuda_check(cudaGetLastError(), "mse launch");
}

size_t exl3_quantize_workspace_bytes(int64_t rows, int64_t cols, int K) {
    if (!k_ok(K) || rows <= 0 || cols <= 0) return 0;
    const int64_t n_tiles = (rows / 16) * (cols / 16);
    return carve_quant(nullptr, rows, cols, K, false, encode_grid_full(n_tiles, K)).total;
}

static exl3_status quant_common_checks(const void *W, int dt, int64_t rows, int64_t cols,
                                       const float *su, const float *sv, int K) {
    exl3_status st;
    if ((st = check_matrix(W, "W", dt, rows, cols, 128)) != EXL3_OK) return st;
    if ((st = check_signs(su, sv)) != EXL3_OK) return st;
    return check_k(K);
}

// grid that fits the workspace (returns 0 when even one block does not fit)
static int fit_grid(void *ws, size_t ws_bytes, int64_t rows, int64_t cols, int K, bool gss) {
    const int64_t n_tiles = (rows / 16) * (cols / 16);
    int g = encode_grid_full(n_tiles, K);
    const size_t fixed = carve_quant(nullptr, rows, cols, K, gss, 0).total;
    if (ws_bytes < fixed + kEncodeBlockScratchBytes)
        return 0;
    const int64_t cap = (int64_t)((ws_bytes - fixed) / kEncodeBlockScratchBytes);
    (void)ws;
    return (int)fit_blocks(g, cap, K);
}

exl3_status exl3_quantize(const void *W, int dt, int64_t rows, int64_t cols, const float *su,
                          const float *sv, int K, double g, uint16_t *codes, float *scale_out,
                          double *mse_out, double *sigma_out, float *What, void *ws,
                          size_t ws_bytes, void *stream) {
    exl3_status st;
    if ((st = quant_common_checks(W, dt, rows, cols, su, sv, K)) != EXL3_OK) return st;
    if ((st = check_ptr(codes, "codes", 4)) != EXL3_OK) return st;
    if ((st = check_ptr(scale_out, "scale_out", 4)) != EXL3_OK) return st;
    if ((st = check_ptr(mse_out, "mse_out", 8)) != EXL3_OK) return st;
    if (sigma_out && !aligned(sigma_out, 8))
        return set_error(EXL3_ERR_INVALID_ARG, "sigma_out is not 8-byte aligned");
    if (What && !aligned(What, 4))
        return set_error(EXL3_ERR_INVALID_ARG, "What is not 4-byte aligned");
    if (!(g > 0.0) || !std::isfinite(g))
        return set_error(EXL3_ERR_INVALID_ARG, "g must be positive and finite");
    if (!ws || !aligned(ws, kAlign))
        return set_error(EXL3_ERR_INVALID_ARG, "workspace must be non-NULL and 256-byte aligned");
    const int grid = fit_grid(ws, ws_bytes, rows, cols, K, false);
    if (grid < 1)
        return set_error(EXL3_ERR_WORKSPACE, "workspace %zu bytes is below the minimum", ws_bytes);
    QuantWs q = carve_quant(ws, rows, cols, K, false, grid);
    return run_quantize(q, grid, W, dt, rows, cols, su, sv, K, g, nullptr,
                        reinterpret_cast<uint32_t *>(codes), scale_out, mse_out, sigma_out, What,
                        (cudaStream_t)stream);
}

size_t exl3_gss_workspace_bytes(int64_t rows, int64_t cols, int K) {
    if (!k_ok(K) || rows <= 0 || cols <= 0) return 0;
    const int64_t n_tiles = (rows / 16) * (cols / 16);
    return carve_quant(nullptr, rows, cols, K, true, encode_grid_full(n_tiles, K)).total;
}

exl3_status exl3_gss_scale(const void *W, int dt, int64_t rows, int64_t cols, const float *su,
                           const float *sv, int K, double lo, double hi, int n_eval,
                           uint16_t *best_codes, float *best_scale_out, double *best_g_out,
                           double *best_mse_out, double *history_out, void *ws, size_t ws_bytes,
                           void *stream) {
    exl3_status st;
    if ((st = quant_common_checks(W, dt, rows, cols, su, sv, K)) != EXL3_OK) return st;
    if ((st = check_ptr(best_codes, "best_codes", 16)) != EXL3_OK) return st;
    if ((st = check_ptr(best_scale_out, "best_scale_out", 4)) != EXL3_OK) return st;
    if ((st = check_ptr(best_g_out, "best_g_out", 8)) != EXL3_OK) return st;
    if ((st = check_ptr(best_mse_out, "best_mse_out", 8)) != EXL3_OK) return st;
    if (history_out && !aligned(history_out, 8))
        return set_error(EXL3_ERR_INVALID_ARG, "history_out is not 8-byte aligned");
    if (!(lo > 0.0) || !(hi > lo) || !std::isfinite(hi))
        return set_error(EXL3_ERR_INVALID_ARG, "bracket must satisfy 0 < lo < hi < inf");
    if (n_eval < 2 || n_eval > 64)
        return set_error(EXL3_ERR_INVALID_ARG, "n_eval=%d outside [2, 64]", n_eval);
    if (!ws || !aligned(ws, kAlign))
        return set_error(EXL3_ERR_INVALID_ARG, "workspace must be non-NULL and 256-byte aligned");
    const int grid = fit_grid(ws, ws_bytes, rows, cols, K, true);
    if (grid < 1)
        return set_error(EXL3_ERR_WORKSPACE, "workspace %zu bytes is below the minimum", ws_bytes);
    QuantWs q = carve_quant(ws, rows, cols, K, true, grid);
    cudaStream_t s = (cudaStream_t)stream;
    const int64_t n = rows * cols;
    const int64_t n16 = (rows / 16) * (cols / 16) * 32 * K / 16;
    gss_init_kernel<<<1, 1, 0, s>>>(q.gss_state, lo, hi, n_eval);
    note_launch();
    if ((st = cuda_check(cudaGetLastError(), "gss init")) != EXL3_OK) return st;
    for (int e = 0; e < n_eval; e++) {
        if ((st = run_quantize(q, grid, W, dt, rows, cols, su, sv, K, 0.0, &q.gss_state[GCUR],
                               q.eval_codes, nullptr, nullptr, nullptr, nullptr, s)) != EXL3_OK)
            return st;
        gss_update_kernel<<<1, 1, 0, s>>>(q.gss_state, &q.scal[1], n, q.fscal, best_scale_out,
                                          best_g_out, best_mse_out, history_out);
        note_launch();
        if ((st = cuda_check(cudaGetLastError(), "gss update")) != EXL3_OK) return st;
        copy_if_kernel<<<256, 256, 0, s>>>(&q.gss_state[GIMPROVED],
                                           reinterpret_cast<const uint4 *>(q.eval_codes),
                                           reinterpret_cast<uint4 *>(best_codes), n16);
        note_launch();
        if ((st = cuda_check(cudaGetLastError(), "gss copy")) != EXL3_OK) return st;
    }
    return EXL3_OK;
}

// ---- grid-and-parabola scale search -------------------------------------------

static size_t grid_search_carve(void *ws, int64_t rows, int64_t cols, int K, int grid,
                                GridSearchLaunch *out) {
    const int64_t n_tiles = (rows / 16) * (cols / 16);
    const int max_rows = grid_search_max_rows(rows, cols);
    Carver c(ws);
    GridSearchLaunch g{};
    g.R = (float *)c.take((size_t)rows * cols * sizeof(float));
    g.tile_sums = (double *)c.take((size_t)n_tiles * sizeof(double));
    g.tree_scr = (double *)c.take(tree_scratch_doubles(n_tiles) * sizeof(double));
    g.sum = (double *)c.take(sizeof(double));
    g.sigma = (double *)c.take(sizeof(double));
    g.extremes = (int *)c.take(2 * sizeof(int));
    g.sample = (int *)c.take(grid_search_sample_max(rows, cols) * sizeof(int));
    g.count = (int *)c.take(sizeof(int));
    g.state = (double *)c.take(grid_search_state_doubles() * sizeof(double));
    g.rows_buf = (float *)c.take((size_t)max_rows * 256 * sizeof(float));
    g.codes_buf = (uint32_t *)c.take((size_t)max_rows * 8 * K * sizeof(uint32_t));
    g.row_sum = (double *)c.take((size_t)max_rows * sizeof(double));
    g.s_per_g = (float *)c.take(32 * sizeof(float));
    g.enc = (uint32_t *)c.take((size_t)grid * kEncodeBlockScratchBytes);
    g.grid = grid;
    if (out)
        *out = g;
    return c.off;
}

size_t exl3_scale_search_workspace_bytes(int64_t rows, int64_t cols, int K) {
    if (!k_ok(K) || rows <= 0 || cols <= 0)
        return 0;
    const int max_rows = grid_search_max_rows(rows, cols);
    return grid_search_carve(nullptr, rows, cols, K, encode_grid_full(max_rows, K), nullptr);
}

exl3_status exl3_scale_search(const void *W, int dt, int64_t rows, int64_t cols, const float *su,
                              const float *sv, int K, double *g_out, float *scale_out,
                              double *history_out, void *ws, size_t ws_bytes, void *stream) {
    exl3_status st;
    if ((st = quant_common_checks(W, dt, rows, cols, su, sv, K)) != EXL3_OK) return st;
    if ((st = check_ptr(g_out, "g_out", 8)) != EXL3_OK) return st;
    if (scale_out && !aligned(scale_out, 4))
        return set_error(EXL3_ERR_INVALID_ARG, "scale_out is not 4-byte aligned");
    if (history_out && !aligned(history_out, 8))
        return set_error(EXL3_ERR_INVALID_ARG, "history_out is not 8-byte aligned");
    if (grid_search_sample_max(rows, cols) > 2048)
        return set_error(EXL3_ERR_UNSUPPORTED, "rows/16 and cols/16 must be at most 2046");
    if (!ws || !aligned(ws, kAlign))
        return set_error(EXL3_ERR_INVALID_ARG, "workspace must be non-NULL and 256-byte aligned");
    const size_t fixed = grid_search_carve(nullptr, rows, cols, K, 0, nullptr);
    if (ws_bytes < fixed)
        return set_error(EXL3_ERR_WORKSPACE, "workspace %zu bytes is below the minimum", ws_bytes);
    const int grid = (int)fit_blocks(encode_grid_full(grid_search_max_rows(rows, cols), K),
                                     (int64_t)((ws_bytes - fixed) / kEncodeBlockScratchBytes), K);
    if (grid < 1)
        return set_error(EXL3_ERR_WORKSPACE, "workspace %zu bytes is below the minimum", ws_bytes);
    GridSearchLaunch g{};
    grid_search_carve(ws, rows, cols, K, grid, &g);
    g.W = W;
    g.dt = dt;
    g.rows = rows;
    g.cols = cols;
    g.su = su;
    g.sv = sv;
    g.K = K;
    g.g_out = g_out;
    g.scale_out = scale_out;
    g.history = history_out;
    return run_grid_search(g, (cudaStream_t)stream);
}

// ---- block LDL and LDLQ -------------------------------------------------------

static size_t block_ldl_carve(void *ws, int64_t n, BlockLdlLaunch *out) {
    Carver c(ws);
    BlockLdlLaunch b{};
    b.A = (double *)c.take((size_t)n * n * sizeof(double));
    b.LD = (double *)c.take((size_t)(n / 16) * 256 * sizeof(double));
    b.delta = (double *)c.take(sizeof(double));
    b.flag = (int *)c.take(sizeof(int));
    if (out)
        *out = b;
    return c.off;
}

static bool ldl_dim_ok(int64_t n) { return n >= 16 && n % 16 == 0 && n <= 32768; }

size_t exl3_block_ldl_workspace_bytes(int64_t n) {
    if (!ldl_dim_ok(n))
        return 0;
    return block_ldl_carve(nullptr, n, nullptr);
}

exl3_status exl3_block_ldl(const double *H, int64_t n, double sigma_reg, int max_retries, float *M,
                           int *retries_out, void *ws, size_t ws_bytes, void *stream) {
    exl3_status st;
    if ((st = check_ptr(H, "H", 8)) != EXL3_OK) return st;
    if (!ldl_dim_ok(n))
        return set_error(EXL3_ERR_UNSUPPORTED, "n=%lld: must be a multiple of 16 in [16, 32768]",
                         (long long)n);
    if (!(sigma_reg >= 0.0) || !std::isfinite(sigma_reg))
        return set_error(EXL3_ERR_INVALID_ARG, "sigma_reg must be finite and >= 0");
    if (max_retries < 0 || max_retries > 100)
        return set_error(EXL3_ERR_INVALID_ARG, "max_retries=%d outside [0, 100]", max_retries);
    if ((st = check_ptr(M, "M", 16)) != EXL3_OK) return st;
    if (!ws || !aligned(ws, kAlign))
        return set_error(EXL3_ERR_INVALID_ARG, "workspace must be non-NULL and 256-byte aligned");
    const size_t need = block_ldl_carve(nullptr, n, nullptr);
    if (ws_bytes < need)
        return set_error(EXL3_ERR_WORKSPACE, "workspace %zu bytes < %zu", ws_bytes, need);
    BlockLdlLaunch b{};
    block_ldl_carve(ws, n, &b);
    b.H = H;
    b.n = n;
    b.sigma_reg = sigma_reg;
    b.max_retries = max_retries;
    b.M = M;
    b.retries_out = retries_out;
    return run_block_ldl(b, (cudaStream_t)stream);
}

static size_t ldlq_carve(void *ws, int64_t rows, int64_t cols, int grid, LdlqLaunch *out) {
    Carver c(ws);
    LdlqLaunch l{};
    l.acc = (float *)c.take((size_t)rows * cols * sizeof(float));
    l.U = (float *)c.take((size_t)32 * cols * sizeof(float));          // two span rows
    l.E = (float *)c.take((size_t)16 * cols * sizeof(float));          // cols / 16 tiles
    l.ring = (uint32_t *)c.take((size_t)2 * (cols / 16) * 32 * sizeof(uint32_t));   // K <= 4
    l.enc = (uint32_t *)c.take((size_t)grid * kEncodeBlockScratchBytes);
    l.grid = grid;
    if (out)
        *out = l;
    return c.off;
}

size_t exl3_ldlq_workspace_bytes(int64_t rows, int64_t cols, int K) {
    if (!k_ok(K) || rows < 16 || cols < 16 || rows % 16 || cols % 16 || rows > (1ll << 24) ||
        cols > (1ll << 24) || rows * cols > (1ll << 34))
        return 0;
    return ldlq_carve(nullptr, rows, cols, encode_grid_full(cols / 16, K), nullptr);
}

exl3_status exl3_ldlq(const float *R, int64_t rows, int64_t cols, const float *M, int K, float scale,
                      uint16_t *codes, float *Q, void *ws, size_t ws_bytes, void *stream) {
    exl3_status st;
    if ((st = check_ptr(R, "R", 4)) != EXL3_OK) return st;
    if (rows < 16 || cols < 16 || rows % 16 || cols % 16)
        return set_error(EXL3_ERR_UNSUPPORTED, "rows and cols must be positive multiples of 16");
    if (rows > (1ll << 24) || cols > (1ll << 24) || rows * cols > (1ll << 34))
        return set_error(EXL3_ERR_INVALID_ARG, "matrix %lldx%lld is too large", (long long)rows,
                         (long long)cols);
    if ((st = check_ptr(M, "M", 4)) != EXL3_OK) return st;
    if ((st = check_k(K)) != EXL3_OK) return st;
    if (!(scale > 0.0f) || !std::isfinite(scale) || !std::isfinite(1.0f / scale))
        return set_error(EXL3_ERR_INVALID_ARG, "scale and 1 / scale must be positive and finite");
    if ((st = check_ptr(codes, "codes", 4)) != EXL3_OK) return st;
    if (Q && !aligned(Q, 4))
        return set_error(EXL3_ERR_INVALID_ARG, "Q is not 4-byte aligned");
    if (!ws || !aligned(ws, kAlign))
        return set_error(EXL3_ERR_INVALID_ARG, "workspace must be non-NULL and 256-byte aligned");
    const size_t fixed = ldlq_carve(nullptr, rows, cols, 0, nullptr);
    const int64_t cap = ws_bytes > fixed ? (int64_t)((ws_bytes - fixed) / kEncodeBlockScratchBytes) : 0;
    const int grid = (int)fit_blocks(encode_grid_full(cols / 16, K), cap, K);
    if (grid < 1)
        return set_error(EXL3_ERR_WORKSPACE, "workspace %zu bytes is below the minimum", ws_bytes);
    LdlqLaunch l{};
    ldlq_carve(ws, rows, cols, grid, &l);
    l.R = R;
    l.rows = rows;
    l.cols = cols;
    l.M = M;
    l.K = K;
    l.scale = scale;
    l.codes = reinterpret_cast<uint32_t *>(codes);
    l.Q = Q;
    return run_ldlq(l, (cudaStream_t)stream);
}

// ---- output-channel regularisation ----------------------------------------------

static size_t regularize_carve(void *ws, int64_t rows, int64_t cols, RegularizeLaunch *out) {
    Carver c(ws);
    RegularizeLaunch r{};
    r.part = (double *)c.take((size_t)32 * cols * sizeof(double));
    r.S = (double *)c.take((size_t)cols * sizeof(double));
    r.tree_scr = (double *)c.take(tree_scratch_doubles(rows > cols ? rows : cols) * sizeof(double));
    r.total = (double *)c.take(sizeof(double));
    r.sortbuf = (double *)c.take((size_t)regularize_sort_len(rows) * sizeof(double));
    r.hsum = (double *)c.take(2 * sizeof(double));
    r.info = (double *)c.take(4 * sizeof(double));
    r.g_rms = (float *)c.take(sizeof(float));
    r.scale = (float *)c.take((size_t)cols * sizeof(float));
    if (out)
        *out = r;
    return c.off;
}

static bool reg_dims_ok(int64_t rows, int64_t cols) {
    return rows >= 1 && cols >= 1 && rows <= 65536 && cols <= (int64_t)1 << 24;
}

size_t exl3_regularize_workspace_bytes(int64_t rows, int64_t cols) {
    if (!reg_dims_ok(rows, cols))
        return 0;
    return regularize_carve(nullptr, rows, cols, nullptr);
}

exl3_status exl3_regularize(const void *W, int dt, int64_t rows, int64_t cols, const float *h,
                            const float *sv, int apply_out, float *W_out, float *sv_out,
                            double *info_out, void *ws, size_t ws_bytes, void *stream) {
    exl3_status st;
    if (dt != EXL3_F32 && dt != EXL3_BF16)
        return set_error(EXL3_ERR_INVALID_ARG, "dt=%d is not EXL3_F32 or EXL3_BF16", dt);
    if ((st = check_ptr(W, "W", dt == EXL3_BF16 ? 2 : 4)) != EXL3_OK) return st;
    if (!reg_dims_ok(rows, cols))
        return set_error(EXL3_ERR_UNSUPPORTED, "rows in [1, 65536] and cols in [1, 2^24] required");
    if ((st = check_ptr(h, "h", 4)) != EXL3_OK) return st;
    if ((st = check_ptr(sv, "sv", 4)) != EXL3_OK) return st;
    if (apply_out < -1 || apply_out > 1)
        return set_error(EXL3_ERR_INVALID_ARG, "apply_out=%d is not -1, 0 or 1", apply_out);
    if ((st = check_ptr(W_out, "W_out", 4)) != EXL3_OK) return st;
    if ((st = check_ptr(sv_out, "sv_out", 4)) != EXL3_OK) return st;
    if (info_out && !aligned(info_out, 8))
        return set_error(EXL3_ERR_INVALID_ARG, "info_out is not 8-byte aligned");
    if (dt == EXL3_BF16 && (const void *)W_out == W)
        return set_error(EXL3_ERR_INVALID_ARG, "in-place regularisation needs an fp32 W");
    if (!ws || !aligned(ws, kAlign))
        return set_error(EXL3_ERR_INVALID_ARG, "workspace must be non-NULL and 256-byte aligned");
    const size_t need = regularize_carve(nullptr, rows, cols, nullptr);
    if (ws_bytes < need)
        return set_error(EXL3_ERR_WORKSPACE, "workspace %zu bytes < %zu", ws_bytes, need);
    RegularizeLaunch r{};
    regularize_carve(ws, rows, cols, &r);
    r.W = W;
    r.dt = dt;
    r.rows = rows;
    r.cols = cols;
    r.h = h;
    r.sv = sv;
    r.apply_out = apply_out;
    r.W_out = W_out;
    r.sv_out = sv_out;
    r.info_out = info_out;
    return run_regularize(r, (cudaStream_t)stream);
}

void exl3_profile_enable(int on) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    g_prof_on.store(on != 0);
    g_ev_next = 0;
    g_launches.store(0);
}

exl3_status exl3_profile_read(double *encode_ms, int64_t *encode_launches, int64_t *kernel_launches) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    double tot = 0.0;
    int64_t n = 0;
    exl3_status st = EXL3_OK;
    for (size_t i = 0; i < g_ev_next; i++) {
        if (!g_ev[i].used)
            continue;
        float ms = 0.0f;
        cudaError_t e = cudaEventSynchronize(g_ev[i].b);
        if (e == cudaSuccess)
            e = cudaEventElapsedTime(&ms, g_ev[i].a, g_ev[i].b);
        if (e != cudaSuccess) {
            st = cuda_check(e, "profile event");
            break;
        }
        tot += ms;
        n++;
        g_ev[i].used = false;
    }
    g_ev_next = 0;
    if (encode_ms) *encode_ms = tot;
    if (encode_launches) *encode_launches = n;
    if (kernel_launches) *kernel_launches = g_launches.exchange(0);
    return st;
}

}  // extern "C"

exl3_status exl3_wait_timeouts(unsigned int *count_out) {
    unsigned int n = 0, r = 0;
    exl3_status st = exl3::cuda_check(cudaDeviceSynchronize(), "device synchronise (wait timeouts)");
    if (st == EXL3_OK)
        st = exl3::rot_take_wait_timeouts(&r);
    n += r;
    if (count_out)
        *count_out = n;
    if (st != EXL3_OK)
        return st;
    return n ? exl3::set_error(EXL3_ERR_TIMEOUT, "%u device waits expired", n) : EXL3_OK;
}
