// ldlq.cu -- block LDL factorisation of a Hessian and LDLQ error feedback
// around the trellis tile encoder (page "EXL3 Intel Arc Quantizer", Core
// Implemented Architecture item 3: blockwise Cholesky/LDL with the inverse of
// the 16x16 block diagonal folded in, diagonal damping of
// 2 sigma_reg mean(diag H) retried up to 10 times, and bottom-up error
// feedback from the strictly lower factor into the targets of the 16-row
// spans not yet quantised).
//
// Arithmetic (the same sequence of IEEE operations as the textbook
// definitions):
//   Cholesky, binary64: L[i][j] = (H[i][j] - sum_{k<j} L[i][k] L[j][k]) / L[j][j]
//     and L[j][j] = sqrt(H[j][j] - sum_{k<j} L[j][k]^2), each term one
//     rounded product then one rounded difference, k ascending.  The blocked
//     right-looking schedule below (panels of 16 columns) applies exactly that
//     sequence to every entry: panel p's 16 terms in ascending k after panel
//     p-1's, then the entry's own panel.
//   Fold: X = inverse of each 16x16 diagonal block by forward substitution,
//     M[i][16b+c] = fl32(sum_{k=c..15} L[i][16b+k] X[k][c]), k ascending.
//   Feedback, binary32: after span j is coded, every row r above it gets
//     acc[r][c] = fmaf(M[i][r], E[i][c], acc[r][c]) for i = 16j+15 down to 16j,
//     E = fl32(R - Q); span b is coded from U = fl32(R + acc).
// Since column c's accumulators take only column c's errors, the feedback is
// applied per tile (16 columns) as soon as a tile is coded, with the same
// per-accumulator order; see run_ldlq for the launch schedule.
#include "common.cuh"

namespace exl3 {

namespace {

constexpr int kUpdTile = 64;     // trailing-update tile (64 x 64 entries, 4 x 4 per thread)
constexpr int kFbRows = 256;     // rows per feedback block

// delta = (2 sigma_reg) * (sum of the diagonal, ascending / n)
__global__ void __launch_bounds__(1024) diag_delta_kernel(const double *__restrict__ H, int64_t n,
                                                          double sigma_reg, double *delta) {
    __shared__ double d[1024];
    double sum = 0.0;
    for (int64_t base = 0; base < n; base += 1024) {
        const int64_t j = base + threadIdx.x;
        d[threadIdx.x] = j < n ? H[j * n + j] : 0.0;
        __syncthreads();
        if (threadIdx.x == 0) {
            const int m = (int)((n - base) < 1024 ? (n - base) : 1024);
            for (int t = 0; t < m; t++)
                sum = __dadd_rn(sum, d[t]);
        }
        __syncthreads();
    }
    if (threadIdx.x == 0)
        *delta = __dmul_rn(__dmul_rn(2.0, sigma_reg), __ddiv_rn(sum, (double)n));
}

// A = lower triangle of H with a * delta added to the diagonal; clears the flag
__global__ void chol_init_kernel(const double *__restrict__ H, double *__restrict__ A, int64_t n,
                                 int a, const double *delta, int *flag) {
    const int64_t i = blockIdx.y;
    if (i == 0 && blockIdx.x == 0 && threadIdx.x == 0)
        *flag = 0;
    const double add = __dmul_rn((double)a, *delta);
    for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j <= i;
         j += (int64_t)gridDim.x * blockDim.x) {
        double v = H[i * n + j];
        if (j == i)
            v = __dadd_rn(v, add);
        A[i * n + j] = v;
    }
}

// Panel p0 (columns p0 .. p0+15), one warp per block so that the rows spread
// over many SMs (the FP64 units are few per SM).  Every block factors the
// 16x16 diagonal block in shared memory (identically); block 0 stores it to
// LD (the rows of A inside the diagonal block are left as they are, so no
// block reads a value another one has overwritten).  Then one row
// i >= p0 + 16 per thread:
// L[i][p0+j] = (A[i][p0+j] - sum_{k<j} L[i][p0+k] L[p0+j][p0+k]) / L[p0+j][p0+j].
constexpr int kPanelThreads = 32;

__global__ void __launch_bounds__(kPanelThreads) chol_panel_kernel(double *__restrict__ A,
                                                                   double *__restrict__ LD,
                                                                   int64_t n, int64_t p0, int *flag) {
    __shared__ double D[16][17];
    const int t = threadIdx.x;
    for (int e = t; e < 256; e += kPanelThreads) {
        const int r = e >> 4, c = e & 15;
        D[r][c] = (c <= r) ? A[(p0 + r) * n + p0 + c] : 0.0;
    }
    __syncthreads();
    {
        const int r = t & 15;     // lanes 16..31 repeat lanes 0..15 and never store
        for (int j = 0; j < 16; j++) {
            double acc = D[r][j];
            for (int k = 0; k < j; k++)
                acc = __dsub_rn(acc, __dmul_rn(D[r][k], D[j][k]));
            __syncwarp();
            if (t == j) {
                double d = 1.0;
                if (acc > 0.0)
                    d = __dsqrt_rn(acc);
                else
                    *flag = 1;           // not positive definite: the attempt fails
                D[j][j] = d;
            }
            __syncwarp();
            if (t < 16 && r > j)
                D[r][j] = __ddiv_rn(acc, D[j][j]);
            __syncwarp();
        }
    }
    __syncthreads();
    if (blockIdx.x == 0) {
        for (int e = t; e < 256; e += kPanelThreads)
            LD[e] = D[e >> 4][e & 15];
    }
    const int64_t i = p0 + 16 + (int64_t)blockIdx.x * blockDim.x + t;
    if (i >= n)
        return;
    double *row = A + i * n + p0;
    double l[16];
#pragma unroll
    for (int c = 0; c < 16; c++)
        l[c] = row[c];
#pragma unroll
    for (int j = 0; j < 16; j++) {
        double acc = l[j];
#pragma unroll
        for (int k = 0; k < j; k++)
            acc = __dsub_rn(acc, __dmul_rn(l[k], D[j][k]));
        l[j] = __ddiv_rn(acc, D[j][j]);
    }
#pragma unroll
    for (int c = 0; c < 16; c++)
        row[c] = l[c];
}

// Trailing update after panel p0: A[i][j] -= L[i][p0+k] L[j][p0+k], k = 0..15
// ascending, for start <= j <= i < n (start = p0 + 32: the next panel's 16
// columns get the same terms from chol_strip_kernel).  64 x 64 tiles on or
// below the diagonal; thread (ty, tx) owns entries (ty + 16a, tx + 16b).
__global__ void __launch_bounds__(256) chol_update_kernel(double *__restrict__ A, int64_t n,
                                                          int64_t p0, int64_t start) {
    const int ti = blockIdx.y, tj = blockIdx.x;
    if (tj > ti)
        return;
    __shared__ double Li[kUpdTile][17], Lj[kUpdTile][17];
    const int t = threadIdx.x;
    const int64_t p1 = start;
    const int64_t i0 = p1 + (int64_t)kUpdTile * ti, j0 = p1 + (int64_t)kUpdTile * tj;
    for (int e = t; e < kUpdTile * 16; e += 256) {
        const int r = e >> 4, k = e & 15;
        Li[r][k] = (i0 + r < n) ? A[(i0 + r) * n + p0 + k] : 0.0;
        Lj[r][k] = (j0 + r < n) ? A[(j0 + r) * n + p0 + k] : 0.0;
    }
    __syncthreads();
    const int tx = t & 15, ty = t >> 4;
    double acc[4][4];
#pragma unroll
    for (int a = 0; a < 4; a++)
#pragma unroll
        for (int b = 0; b < 4; b++) {
            const int64_t gi = i0 + ty + 16 * a, gj = j0 + tx + 16 * b;
            acc[a][b] = (gi < n && gj <= gi) ? A[gi * n + gj] : 0.0;
        }
#pragma unroll
    for (int k = 0; k < 16; k++) {
        double lj[4];
#pragma unroll
        for (int b = 0; b < 4; b++)
            lj[b] = Lj[tx + 16 * b][k];
#pragma unroll
        for (int a = 0; a < 4; a++) {
            const double li = Li[ty + 16 * a][k];
#pragma unroll
            for (int b = 0; b < 4; b++)
                acc[a][b] = __dsub_rn(acc[a][b], __dmul_rn(li, lj[b]));
        }
    }
#pragma unroll
    for (int a = 0; a < 4; a++)
#pragma unroll
        for (int b = 0; b < 4; b++) {
            const int64_t gi = i0 + ty + 16 * a, gj = j0 + tx + 16 * b;
            if (gi < n && gj <= gi)
                A[gi * n + gj] = acc[a][b];
        }
}

// The same update for the next panel's columns only: A[i][j] -= L[i][p0+k] L[j][p0+k],
// k = 0..15 ascending, for p0 + 16 <= j < p0 + 32, j <= i < n; one entry per thread.
__global__ void __launch_bounds__(256) chol_strip_kernel(double *__restrict__ A, int64_t n,
                                                         int64_t p0) {
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t i = p0 + 16 + (idx >> 4);
    const int64_t j = p0 + 16 + (idx & 15);
    if (i >= n || j > i)
        return;
    const double *li = A + i * n + p0;
    const double *lj = A + j * n + p0;
    double acc = A[i * n + j];
#pragma unroll
    for (int k = 0; k < 16; k++)
        acc = __dsub_rn(acc, __dmul_rn(li[k], lj[k]));
    A[i * n + j] = acc;
}

// M[i][16b + c] = fl32(sum_{k=c..15} L[i][16b+k] X[k][c]) for rows i >= 16(b+1),
// X the inverse of diagonal block b (forward substitution by 16 lanes, one
// column each: X[c][c] = 1 / B[c][c]; X[r][c] = -(sum_{k=c..r-1} B[r][k] X[k][c]) / B[r][r]).
__global__ void __launch_bounds__(256) ldl_fold_kernel(const double *__restrict__ A,
                                                       const double *__restrict__ LD, int64_t n,
                                                       float *__restrict__ M) {
    const int64_t b = blockIdx.y;
    __shared__ double X[16][17];
    const int t = threadIdx.x;
    const double *B = LD + b * 256;
    if (t < 16) {
        const int c = t;
        for (int r = 0; r < 16; r++)
            X[r][c] = 0.0;
        X[c][c] = __ddiv_rn(1.0, B[c * 16 + c]);
        for (int r = c + 1; r < 16; r++) {
            double acc = 0.0;
            for (int k = c; k < r; k++)
                acc = __dadd_rn(acc, __dmul_rn(B[r * 16 + k], X[k][c]));
            X[r][c] = __ddiv_rn(-acc, B[r * 16 + r]);
        }
    }
    __syncthreads();
    const int64_t i = 16 * (b + 1) + (int64_t)blockIdx.x * blockDim.x + t;
    if (i >= n)
        return;
    double l[16];
#pragma unroll
    for (int k = 0; k < 16; k++)
        l[k] = A[i * n + 16 * b + k];
    float out[16];
#pragma unroll
    for (int c = 0; c < 16; c++) {
        double acc = 0.0;
#pragma unroll
        for (int k = c; k < 16; k++)
            acc = __dadd_rn(acc, __dmul_rn(l[k], X[k][c]));
        out[c] = __double2float_rn(acc);
    }
    float4 *dst = reinterpret_cast<float4 *>(M + i * n + 16 * b);
#pragma unroll
    for (int q = 0; q < 4; q++)
        dst[q] = make_float4(out[4 * q], out[4 * q + 1], out[4 * q + 2], out[4 * q + 3]);
}

// targets of the first (bottom) span: U = fl32(R + 0)
__global__ void ldlq_first_target_kernel(const float *__restrict__ R, int64_t cols, int64_t row0,
                                         float *__restrict__ U) {
    const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (e < 16 * cols)
        U[e] = __fadd_rn(R[row0 * cols + e], 0.0f);
}

// Tiles in coding order: position p = sigma * TC + c is tile column c of span
// j = B - 1 - sigma (spans bottom-up); its targets and codes sit in ring slot
// sigma & 1 (ring tile p mod 2 TC).
struct SpanTile {
    int64_t j, c, slot;
    __device__ SpanTile(int64_t p, int64_t TC, int64_t B) {
        const int64_t sigma = p / TC;
        j = B - 1 - sigma;
        c = p - sigma * TC;
        slot = sigma & 1;
    }
};

// one block (256 threads) per tile coded by the launch (tiles p0 + blockIdx.x):
// the codes move from the ring to their place, q = fl32(v(state) * s),
// E = fl32(R - q); Q optional
__global__ void __launch_bounds__(256) ldlq_error_kernel(const uint32_t *__restrict__ ring,
                                                         uint32_t *__restrict__ codes, int K,
                                                         const float *__restrict__ R, int64_t cols,
                                                         int64_t TC, int64_t B, int64_t p0, float s,
                                                         float *__restrict__ E, float *__restrict__ Q) {
    __shared__ uint32_t cw[32];
    const SpanTile tl(p0 + blockIdx.x, TC, B);
    const int NW = 8 * K;
    if (threadIdx.x < NW) {
        const uint32_t w = ring[(tl.slot * TC + tl.c) * NW + threadIdx.x];
        cw[threadIdx.x] = w;
        codes[(tl.j * TC + tl.c) * NW + threadIdx.x] = w;
    }
    __syncthreads();
    const int i = threadIdx.x;
    const int64_t r = 16 * tl.j + (i >> 4), c = 16 * tl.c + (i & 15);
    const float q = __fmul_rn(mul1_value(window_state_k(cw, i, K)), s);
    E[(int64_t)blockIdx.x * 256 + i] = __fsub_rn(R[r * cols + c], q);
    if (Q)
        Q[r * cols + c] = q;
}

// after tile (j, c) is coded: rows r < 16 j of its 16 columns get
// acc = fmaf(M[i][r], E[i - 16j][x], acc) for i = 16j+15 down to 16j; the rows
// of span j-1 get their targets U = fl32(R + acc) in the next ring slot (their
// accumulator is not needed any more).  Block (tile, 256-row chunk); thread =
// (column x, row lane): rows chunk + lane + 16 k.
__global__ void __launch_bounds__(256) ldlq_feedback_kernel(float *__restrict__ ACC,
                                                            const float *__restrict__ M, int64_t n,
                                                            int64_t cols, int64_t TC, int64_t B,
                                                            int64_t p0, const float *__restrict__ E,
                                                            const float *__restrict__ R,
                                                            float *__restrict__ U) {
    __shared__ float Ms[16][kFbRows];
    const SpanTile tl(p0 + blockIdx.x, TC, B);
    const int64_t above = 16 * tl.j;
    const int64_t r0 = (int64_t)blockIdx.y * kFbRows;
    if (r0 >= above)
        return;
    for (int e = threadIdx.x; e < 16 * kFbRows; e += blockDim.x) {
        const int ii = e / kFbRows, rr = e % kFbRows;
        Ms[ii][rr] = (r0 + rr < above) ? M[(above + ii) * n + r0 + rr] : 0.0f;
    }
    const int x = threadIdx.x & 15, lane = threadIdx.x >> 4;
    float e[16];
#pragma unroll
    for (int ii = 0; ii < 16; ii++)
        e[ii] = E[(int64_t)blockIdx.x * 256 + ii * 16 + x];
    __syncthreads();
    const int64_t c = 16 * tl.c + x;
    const int64_t span_lo = above - 16;
    float *const Un = U + (1 - tl.slot) * 16 * cols;
    for (int rr = lane; rr < kFbRows; rr += 16) {
        const int64_t r = r0 + rr;
        if (r >= above)
            break;
        float a = ACC[r * cols + c];
#pragma unroll
        for (int ii = 15; ii >= 0; ii--)
            a = __fmaf_rn(Ms[ii][rr], e[ii], a);
        if (r >= span_lo)
            Un[(r - span_lo) * cols + c] = __fadd_rn(R[r * cols + c], a);
        else
            ACC[r * cols + c] = a;
    }
}

}  // namespace

namespace {

// A second stream and the events that order it against the caller's stream,
// created for one factorisation and released on every return path.
struct Lookahead {
    cudaStream_t side = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr, panel[2] = {}, rest[2] = {};
    exl3_status init() {
        exl3_status st;
        if ((st = cuda_check(cudaStreamCreateWithFlags(&side, cudaStreamNonBlocking),
                             "look-ahead stream")) != EXL3_OK)
            return st;
        cudaEvent_t *evs[6] = {&fork, &join, &panel[0], &panel[1], &rest[0], &rest[1]};
        for (cudaEvent_t *e : evs)
            if ((st = cuda_check(cudaEventCreateWithFlags(e, cudaEventDisableTiming),
                                 "look-ahead event")) != EXL3_OK)
                return st;
        return EXL3_OK;
    }
    ~Lookahead() {
        for (cudaEvent_t e : {fork, join, panel[0], panel[1], rest[0], rest[1]})
            if (e)
                cudaEventDestroy(e);
        if (side)
            cudaStreamDestroy(side);
    }
};

}  // namespace

// One attempt, with look-ahead: panel p + 1 (and the update of its own 16
// columns by panel p) runs on a second stream while the caller's stream applies
// panel p to everything to the right of them.  Each entry still receives its
// terms in ascending k, so the factor is the same as without look-ahead.
//   side:  panel(0) | strip(0) panel(1) | strip(1) panel(2) | ...
//   main:           rest(0)             | rest(1)          | ...
// rest(p) waits for panel(p); strip(p) waits for rest(p - 1), the last writer of
// the columns it updates.
static exl3_status cholesky_attempt(const BlockLdlLaunch &p, int a, Lookahead &la, cudaStream_t s) {
    const int64_t n = p.n;
    exl3_status st;
    const int ix = (int)((n + 255) / 256 < 64 ? (n + 255) / 256 : 64);
    chol_init_kernel<<<dim3(ix, (unsigned)n), 256, 0, s>>>(p.H, p.A, n, a, p.delta, p.flag);
    note_launch();
    if ((st = cuda_check(cudaEventRecord(la.fork, s), "fork")) != EXL3_OK) return st;
    if ((st = cuda_check(cudaStreamWaitEvent(la.side, la.fork, 0), "fork wait")) != EXL3_OK) return st;
    auto panel = [&](int64_t p0) {
        const int64_t below = n - p0 - 16;
        const unsigned gp = below > 0 ? (unsigned)((below + kPanelThreads - 1) / kPanelThreads) : 1u;
        chol_panel_kernel<<<gp, kPanelThreads, 0, la.side>>>(p.A, p.LD + (p0 / 16) * 256, n, p0,
                                                              p.flag);
        note_launch();
    };
    panel(0);
    if ((st = cuda_check(cudaEventRecord(la.panel[0], la.side), "panel event")) != EXL3_OK) return st;
    for (int64_t q = 0; 16 * q + 16 < n; q++) {
        const int64_t p0 = 16 * q;
        const int64_t below = n - p0 - 16;             // rows under panel q (>= 16)
        // main: panel q applied to the columns right of panel q + 1
        if ((st = cuda_check(cudaStreamWaitEvent(s, la.panel[q & 1], 0), "panel wait")) != EXL3_OK)
            return st;
        if (below > 16) {
            const unsigned T = (unsigned)((below - 16 + kUpdTile - 1) / kUpdTile);
            chol_update_kernel<<<dim3(T, T), 256, 0, s>>>(p.A, n, p0, p0 + 32);
            note_launch();
        }
        if ((st = cuda_check(cudaEventRecord(la.rest[q & 1], s), "rest event")) != EXL3_OK) return st;
        // side: panel q applied to panel q + 1's columns, then panel q + 1
        if (q > 0 && (st = cuda_check(cudaStreamWaitEvent(la.side, la.rest[(q - 1) & 1], 0),
                                      "rest wait")) != EXL3_OK)
            return st;
        chol_strip_kernel<<<(unsigned)((below * 16 + 255) / 256), 256, 0, la.side>>>(p.A, n, p0);
        note_launch();
        panel(p0 + 16);
        if ((st = cuda_check(cudaEventRecord(la.panel[(q + 1) & 1], la.side), "panel event")) != EXL3_OK)
            return st;
    }
    if ((st = cuda_check(cudaEventRecord(la.join, la.side), "join")) != EXL3_OK) return st;
    if ((st = cuda_check(cudaStreamWaitEvent(s, la.join, 0), "join wait")) != EXL3_OK) return st;
    return cuda_check(cudaGetLastError(), "cholesky launch");
}

exl3_status run_block_ldl(const BlockLdlLaunch &p, cudaStream_t s) {
    const int64_t n = p.n;
    exl3_status st;
    Lookahead la;
    if ((st = la.init()) != EXL3_OK) return st;
    diag_delta_kernel<<<1, 1024, 0, s>>>(p.H, n, p.sigma_reg, p.delta);
    note_launch();
    for (int a = 0; a <= p.max_retries; a++) {
        if ((st = cholesky_attempt(p, a, la, s)) != EXL3_OK) return st;
        int failed = 0;
        if ((st = cuda_check(cudaMemcpyAsync(&failed, p.flag, sizeof(int), cudaMemcpyDeviceToHost, s),
                             "pivot flag copy")) != EXL3_OK)
            return st;
        if ((st = cuda_check(cudaStreamSynchronize(s), "pivot flag wait")) != EXL3_OK) return st;
        if (!failed) {
            if ((st = cuda_check(cudaMemsetAsync(p.M, 0, (size_t)n * n * sizeof(float), s),
                                 "M clear")) != EXL3_OK)
                return st;
            if (n > 16) {
                const unsigned gx = (unsigned)((n - 16 + 255) / 256);
                ldl_fold_kernel<<<dim3(gx, (unsigned)(n / 16 - 1)), 256, 0, s>>>(p.A, p.LD, n, p.M);
                note_launch();
            }
            if (p.retries_out)
                *p.retries_out = a;
            return cuda_check(cudaGetLastError(), "fold launch");
        }
    }
    if (p.retries_out)
        *p.retries_out = -1;
    return set_error(EXL3_ERR_NUMERIC, "H is not positive definite after %d damping retries",
                     p.max_retries);
}

exl3_status run_ldlq(const LdlqLaunch &p, cudaStream_t s) {
    const int64_t n = p.rows, cols = p.cols;
    const int64_t B = n / 16, TC = cols / 16;
    const float inv = 1.0f / p.scale;
    // Tile (j, c) depends only on the tiles below it in column c, so the tiles
    // are coded in span-major order, bottom-up, one round of the persistent grid
    // per launch (K >= 3: a pair per block) and at most one span row (TC tiles)
    // per launch: a tile's nearest dependency, TC positions back, then always
    // lies in an earlier launch, whose feedback has written its targets.
    const int64_t round = (int64_t)p.grid * (p.K >= 3 ? 2 : 1);
    const int64_t G = round < TC ? round : TC;
    const int64_t total = B * TC;
    exl3_status st;
    if ((st = cuda_check(cudaMemsetAsync(p.acc, 0, (size_t)n * cols * sizeof(float), s),
                         "feedback clear")) != EXL3_OK)
        return st;
    ldlq_first_target_kernel<<<(unsigned)((16 * cols + 255) / 256), 256, 0, s>>>(p.R, cols,
                                                                                  16 * (B - 1), p.U);
    note_launch();
    for (int64_t p0 = 0; p0 < total; p0 += G) {
        const int64_t cnt = total - p0 < G ? total - p0 : G;
        EncodeLaunch el{};
        el.Y = p.U;                  // the ring: 2 span rows of targets
        el.rows = 32;
        el.cols = cols;
        el.K = p.K;
        el.T = 256;
        el.row_tiles = 0;
        el.inv_scale = inv;
        el.inv_scale_dev = nullptr;
        el.codes = p.ring;
        el.tile_cost = nullptr;
        el.scratch = p.enc;
        el.grid = (int)(p.grid < cnt ? p.grid : cnt);
        el.tile0 = (int)(p0 % (2 * TC));
        el.n_work = (int)cnt;
        el.ring = (int)(2 * TC);
        if ((st = launch_encode(el, s)) != EXL3_OK) return st;
        ldlq_error_kernel<<<(unsigned)cnt, 256, 0, s>>>(p.ring, p.codes, p.K, p.R, cols, TC, B, p0,
                                                        p.scale, p.E, p.Q);
        note_launch();
        const int64_t j_top = B - 1 - p0 / TC;       // the launch's highest span
        if (j_top > 0) {
            const dim3 g((unsigned)cnt, (unsigned)((16 * j_top + kFbRows - 1) / kFbRows));
            ldlq_feedback_kernel<<<g, 256, 0, s>>>(p.acc, p.M, n, cols, TC, B, p0, p.E, p.R, p.U);
            note_launch();
        }
        if ((st = cuda_check(cudaGetLastError(), "ldlq launch")) != EXL3_OK) return st;
    }
    return EXL3_OK;
}

}  // namespace exl3
