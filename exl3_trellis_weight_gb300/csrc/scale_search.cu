// scale_search.cu -- grid-and-parabola global-scale search on a tile sample
// (page "EXL3 Intel Arc Quantizer", Core Implemented Architecture item 8:
// wrapped-diagonal tile sample with the highest/lowest-RMS tiles, coarse grid
// 0.1..1.9 on a strided subsample, fine grid within 0.075 of the coarse minimum
// on the full sample, parabolic refinement with a 0.01 floor).
//
// Readings of the parts the page leaves open (the oracle implements the same):
//   sample   : tiles (i mod TR, i mod TC), i < max(TR, TC), then the highest-
//              and lowest-RMS tiles (ties to the lower index) if not yet in;
//   objective: rotated-domain MSE of a tile subset at s = fl32(g * sigma_R):
//              sum (r - fl(v * s))^2 in fp64, row-major per tile, tiles added as
//              a pairwise tree in sample order, / (256 * tiles);
//   coarse   : g = k/10, k = 1..19, on sample entries 0, 2, 4, ...;
//   fine     : g_c + 0.025 k, k = -3..3, on the full sample;
//   refine   : vertex of the parabola through the fine minimum and its grid
//              neighbours (interior minimum only), floored at 0.01, kept when
//              strictly better on the full sample.
// Every grid level is one batch: gather the sampled tiles scaled per g into
// rows, encode all rows in one launch (row mode, T = 256), one error kernel,
// one segmented tree.  Selection kernels pick the next grid on the device; the
// host never waits.
#include "common.cuh"

namespace exl3 {

namespace {

constexpr int kCoarse = 19;
constexpr int kFine = 7;
constexpr int kSegMax = 2048;   // tiles per sample (one tree block per grid point)

// highest / lowest per-tile sum of squares, ties to the lower tile index
__global__ void __launch_bounds__(1024) extreme_tiles_kernel(const double *__restrict__ ts,
                                                             int64_t n, int *out) {
    __shared__ double shv[2][32];
    __shared__ int64_t shi[2][32];
    double vmax = -1.0, vmin = __longlong_as_double(0x7ff0000000000000ll);
    int64_t imax = 0, imin = 0;
    for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
        const double v = ts[i];
        if (v > vmax) { vmax = v; imax = i; }          // ascending i: first max kept
        if (v < vmin) { vmin = v; imin = i; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const double v1 = __shfl_xor_sync(0xffffffffu, vmax, o);
        const int64_t i1 = __shfl_xor_sync(0xffffffffu, imax, o);
        if (v1 > vmax || (v1 == vmax && i1 < imax)) { vmax = v1; imax = i1; }
        const double v2 = __shfl_xor_sync(0xffffffffu, vmin, o);
        const int64_t i2 = __shfl_xor_sync(0xffffffffu, imin, o);
        if (v2 < vmin || (v2 == vmin && i2 < imin)) { vmin = v2; imin = i2; }
    }
    const int w = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) {
        shv[0][w] = vmax; shi[0][w] = imax;
        shv[1][w] = vmin; shi[1][w] = imin;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const int nw = (blockDim.x + 31) / 32;
        for (int k = 1; k < nw; k++) {
            if (shv[0][k] > shv[0][0] || (shv[0][k] == shv[0][0] && shi[0][k] < shi[0][0])) {
                shv[0][0] = shv[0][k]; shi[0][0] = shi[0][k];
            }
            if (shv[1][k] < shv[1][0] || (shv[1][k] == shv[1][0] && shi[1][k] < shi[1][0])) {
                shv[1][0] = shv[1][k]; shi[1][0] = shi[1][k];
            }
        }
        out[0] = (int)shi[0][0];
        out[1] = (int)shi[1][0];
    }
}

// sample list: wrapped diagonal, then the extremes if new; slots >= count are
// padding (tile 0, weight 0) kept at the end
__global__ void build_sample_kernel(int TR, int TC, const int *extremes, int n_max, int *S,
                                    int *count) {
    if (threadIdx.x != 0 || blockIdx.x != 0)
        return;
    const int nd = TR > TC ? TR : TC;
    for (int i = 0; i < nd; i++)
        S[i] = (i % TR) * TC + (i % TC);
    int c = nd;
    for (int e = 0; e < 2; e++) {
        const int t = extremes[e];
        const int tr = t / TC, tc = t % TC;
        bool on_diag = false;   // tile (tr, tc) is S[i] iff i = tr (mod TR) and i = tc (mod TC)
        for (int i = tr; i < nd; i += TR)
            if (i % TC == tc) { on_diag = true; break; }
        for (int k = nd; k < c; k++)
            if (S[k] == t) on_diag = true;
        if (!on_diag)
            S[c++] = t;
    }
    for (int k = c; k < n_max; k++)
        S[k] = 0;
    *count = c;
}

// row (gi, j): sample entry idx = j * stride of the sample, scaled by fl32(1/s_g)
__global__ void gather_rows_kernel(const float *__restrict__ R, int64_t cols, const int *S,
                                   int n_slots, int stride, const double *gvals, const double *sigma,
                                   float *__restrict__ rows_out, float *__restrict__ s_out) {
    const int row = blockIdx.x;               // gi * n_slots + j
    const int gi = row / n_slots, j = row % n_slots;
    double sg = *sigma;
    if (sg == 0.0)
        sg = 1.0;
    const float s = __double2float_rn(__dmul_rn(gvals[gi], sg));
    const float inv = __fdiv_rn(1.0f, s);
    if (threadIdx.x == 0 && j == 0)
        s_out[gi] = s;
    const int t = S[j * stride];
    const int64_t TC = cols / 16;
    const int64_t tr = t / TC, tc = t % TC;
    const int i = threadIdx.x;                // 256 threads: element i of the tile
    const float r = R[(size_t)(tr * 16 + (i >> 4)) * (size_t)cols + tc * 16 + (i & 15)];
    rows_out[(size_t)row * 256 + i] = __fmul_rn(r, inv);
}

// per-row fp64 error: sum_i (r_i - fl(v(state_i) * s_g))^2 in row-major order;
// padding rows (j >= valid count) give 0
__global__ void row_error_kernel(const uint32_t *__restrict__ codes, int K, const float *__restrict__ R,
                                 int64_t cols, const int *S, int n_slots, int stride,
                                 const int *count, int half_count, const float *s_per_g,
                                 double *__restrict__ row_sum) {
    __shared__ float yh[256];
    __shared__ uint32_t cw[32];
    const int row = blockIdx.x;
    const int gi = row / n_slots, j = row % n_slots;
    const int valid = half_count ? (*count + 1) / 2 : *count;
    const int NW = 8 * K;
    if (threadIdx.x < NW)
        cw[threadIdx.x] = codes[(size_t)row * NW + threadIdx.x];
    __syncthreads();
    const int i = threadIdx.x;
    yh[i] = __fmul_rn(mul1_value(window_state_k(cw, i, K)), s_per_g[gi]);
    __syncthreads();
    if (threadIdx.x == 0) {
        double acc = 0.0;
        if (j < valid) {
            const int t = S[j * stride];
            const int64_t TC = cols / 16;
            const int64_t tr = t / TC, tc = t % TC;
            for (int e = 0; e < 256; e++) {
                const float r = R[(size_t)(tr * 16 + (e >> 4)) * (size_t)cols + tc * 16 + (e & 15)];
                const double d = __dsub_rn((double)r, (double)yh[e]);
                acc = __dadd_rn(acc, __dmul_rn(d, d));
            }
        }
        row_sum[row] = acc;
    }
}

// one block per grid point: pairwise tree over its n_slots row sums (level by
// level, neighbours (2i, 2i+1), odd last moves up), / (256 * valid tiles)
__global__ void __launch_bounds__(1024) segment_mse_kernel(const double *__restrict__ row_sum,
                                                           int n_slots, const int *count,
                                                           int half_count, double *f_out) {
    __shared__ double v[kSegMax];
    const int gi = blockIdx.x;
    for (int i = threadIdx.x; i < n_slots; i += blockDim.x)
        v[i] = row_sum[(size_t)gi * n_slots + i];
    __syncthreads();
    int m = n_slots;
    while (m > 1) {
        const int h = m >> 1;
        double r0 = 0.0, r1 = 0.0;
        const int i0 = threadIdx.x, i1 = threadIdx.x + 1024;
        if (i0 < h) r0 = __dadd_rn(v[2 * i0], v[2 * i0 + 1]);
        if (i1 < h) r1 = __dadd_rn(v[2 * i1], v[2 * i1 + 1]);
        const bool odd = (m & 1) != 0;
        double carry = 0.0;
        if (odd && threadIdx.x == 0) carry = v[m - 1];
        __syncthreads();
        if (i0 < h) v[i0] = r0;
        if (i1 < h) v[i1] = r1;
        if (odd && threadIdx.x == 0) v[h] = carry;
        __syncthreads();
        m = h + (odd ? 1 : 0);
    }
    if (threadIdx.x == 0) {
        const int valid = half_count ? (*count + 1) / 2 : *count;
        f_out[gi] = __ddiv_rn(v[0], __dmul_rn(256.0, (double)valid));
    }
}

// state (doubles): [0..19) coarse g, [19..38) coarse f, [38..45) fine g, [45..52) fine f,
// [52] refine g, [53] refine f, [54] refine valid, [55] final g
enum { SC_G = 0, SC_F = 19, SF_G = 38, SF_F = 45, SR_G = 52, SR_F = 53, SR_OK = 54, S_FINAL = 55, S_LEN = 56 };

__global__ void init_coarse_kernel(double *st) {
    const int k = threadIdx.x;
    if (k < kCoarse)
        st[SC_G + k] = (double)(k + 1) / 10.0;
}

__global__ void select_coarse_kernel(double *st) {
    int b = 0;
    for (int k = 1; k < kCoarse; k++)
        if (st[SC_F + k] < st[SC_F + b]) b = k;
    const double gc = st[SC_G + b];
    for (int k = 0; k < kFine; k++)
        st[SF_G + k] = __dadd_rn(gc, __dmul_rn(0.025, (double)(k - 3)));
}

__global__ void select_fine_kernel(double *st) {
    int b = 0;
    for (int k = 1; k < kFine; k++)
        if (st[SF_F + k] < st[SF_F + b]) b = k;
    st[S_FINAL] = st[SF_G + b];
    st[SR_OK] = 0.0;
    st[SR_G] = st[SF_G + b];   // evaluated anyway; ignored unless valid
    if (b > 0 && b < kFine - 1) {
        const double a = st[SF_G + b - 1], fa = st[SF_F + b - 1];
        const double x = st[SF_G + b], fx = st[SF_F + b];
        const double c = st[SF_G + b + 1], fc = st[SF_F + b + 1];
        const double p = __dmul_rn(__dsub_rn(x, a), __dsub_rn(fx, fc));
        const double q = __dmul_rn(__dsub_rn(x, c), __dsub_rn(fx, fa));
        const double den = __dsub_rn(p, q);
        if (den != 0.0) {
            const double num = __dsub_rn(__dmul_rn(__dsub_rn(x, a), p), __dmul_rn(__dsub_rn(x, c), q));
            double v = __dsub_rn(x, __dmul_rn(0.5, __ddiv_rn(num, den)));
            if (v < 0.01) v = 0.01;
            st[SR_G] = v;
            st[SR_OK] = 1.0;
        }
    }
}

__global__ void select_final_kernel(double *st, const double *sigma, double *g_out, float *scale_out,
                                    double *history) {
    int b = 0;
    for (int k = 1; k < kFine; k++)
        if (st[SF_F + k] < st[SF_F + b]) b = k;
    double g = st[SF_G + b];
    if (st[SR_OK] != 0.0 && st[SR_F] < st[SF_F + b])
        g = st[SR_G];
    st[S_FINAL] = g;
    *g_out = g;
    if (scale_out) {
        double sg = *sigma;
        if (sg == 0.0) sg = 1.0;
        *scale_out = __double2float_rn(__dmul_rn(g, sg));
    }
    if (history) {
        for (int k = 0; k < kCoarse; k++) {
            history[2 * k] = st[SC_G + k];
            history[2 * k + 1] = st[SC_F + k];
        }
        for (int k = 0; k < kFine; k++) {
            history[2 * (kCoarse + k)] = st[SF_G + k];
            history[2 * (kCoarse + k) + 1] = st[SF_F + k];
        }
        history[2 * (kCoarse + kFine)] = st[SR_OK] != 0.0 ? st[SR_G] : -1.0;
        history[2 * (kCoarse + kFine) + 1] = st[SR_OK] != 0.0 ? st[SR_F] : -1.0;
    }
}

__global__ void sigma_kernel(const double *sum, int64_t n, double *sigma) {
    *sigma = __dsqrt_rn(__ddiv_rn(*sum, (double)n));
}

}  // namespace

size_t grid_search_sample_max(int64_t rows, int64_t cols) {
    const int64_t TR = rows / 16, TC = cols / 16;
    return (size_t)((TR > TC ? TR : TC) + 2);
}

exl3_status run_grid_search(const GridSearchLaunch &p, cudaStream_t s) {
    const int64_t TR = p.rows / 16, TC = p.cols / 16;
    const int64_t n_tiles = TR * TC;
    const int n_max = (int)grid_search_sample_max(p.rows, p.cols);
    if (n_max > kSegMax)
        return set_error(EXL3_ERR_UNSUPPORTED, "sample of %d tiles exceeds %d", n_max, kSegMax);
    const int n_c = (n_max + 1) / 2;
    exl3_status st;
    RotateLaunch rf{};
    rf.inverse = 0;
    rf.src = p.dt == EXL3_BF16 ? SRC_BF16 : SRC_F32;
    rf.in = p.W;
    rf.su = p.su;
    rf.sv = p.sv;
    rf.rows = p.rows;
    rf.cols = p.cols;
    rf.out = p.R;
    rf.tile_sums = p.tile_sums;
    if ((st = launch_rotate(rf, s)) != EXL3_OK) return st;
    if ((st = launch_tree_sum(p.tile_sums, n_tiles, p.tree_scr, p.sum, s)) != EXL3_OK) return st;
    sigma_kernel<<<1, 1, 0, s>>>(p.sum, p.rows * p.cols, p.sigma);
    note_launch();
    extreme_tiles_kernel<<<1, 1024, 0, s>>>(p.tile_sums, n_tiles, p.extremes);
    note_launch();
    build_sample_kernel<<<1, 1, 0, s>>>((int)TR, (int)TC, p.extremes, n_max, p.sample, p.count);
    note_launch();
    init_coarse_kernel<<<1, 32, 0, s>>>(p.state);
    note_launch();

    // one grid level: gather -> encode rows -> error -> segmented MSE
    auto level = [&](const double *gvals, int n_g, int n_slots, int stride, int half_count,
                     double *f_out) -> exl3_status {
        const int n_rows = n_g * n_slots;
        gather_rows_kernel<<<n_rows, 256, 0, s>>>(p.R, p.cols, p.sample, n_slots, stride, gvals,
                                                  p.sigma, p.rows_buf, p.s_per_g);
        note_launch();
        exl3_status e2 = cuda_check(cudaGetLastError(), "gather launch");
        if (e2 != EXL3_OK) return e2;
        EncodeLaunch el{};
        el.Y = p.rows_buf;
        el.rows = n_rows;
        el.cols = 256;
        el.K = p.K;
        el.T = 256;
        el.row_tiles = 1;
        el.inv_scale = 1.0f;
        el.inv_scale_dev = nullptr;
        el.codes = p.codes_buf;
        el.tile_cost = nullptr;
        el.scratch = p.enc;
        el.grid = p.grid < n_rows ? p.grid : n_rows;
        if ((e2 = launch_encode(el, s)) != EXL3_OK) return e2;
        row_error_kernel<<<n_rows, 256, 0, s>>>(p.codes_buf, p.K, p.R, p.cols, p.sample, n_slots,
                                                stride, p.count, half_count, p.s_per_g, p.row_sum);
        note_launch();
        segment_mse_kernel<<<n_g, 1024, 0, s>>>(p.row_sum, n_slots, p.count, half_count, f_out);
        note_launch();
        return cuda_check(cudaGetLastError(), "grid level launch");
    };
    if ((st = level(p.state + SC_G, kCoarse, n_c, 2, 1, p.state + SC_F)) != EXL3_OK) return st;
    select_coarse_kernel<<<1, 1, 0, s>>>(p.state);
    note_launch();
    if ((st = level(p.state + SF_G, kFine, n_max, 1, 0, p.state + SF_F)) != EXL3_OK) return st;
    select_fine_kernel<<<1, 1, 0, s>>>(p.state);
    note_launch();
    if ((st = level(p.state + SR_G, 1, n_max, 1, 0, p.state + SR_F)) != EXL3_OK) return st;
    select_final_kernel<<<1, 1, 0, s>>>(p.state, p.sigma, p.g_out, p.scale_out, p.history);
    note_launch();
    return cuda_check(cudaGetLastError(), "grid search launch");
}

size_t grid_search_state_doubles() { return S_LEN; }
int grid_search_max_rows(int64_t rows, int64_t cols) {
    const int n_max = (int)grid_search_sample_max(rows, cols);
    const int n_c = (n_max + 1) / 2;
    return kCoarse * n_c > kFine * n_max ? kCoarse * n_c : kFine * n_max;
}

}  // namespace exl3
