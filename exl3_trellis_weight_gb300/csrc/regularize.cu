// regularize.cu -- output-channel regularisation of a weight before rotation
// (page "EXL3 Intel Arc Quantizer", Core Implemented Architecture item 8:
// block_rms with a 32-slice accumulation order, the output-scale skew
// heuristic on the top 2 % of sqrt(H_diag) against a 15 % cutoff, output-channel
// RMS normalisation with sign and scale folded into sv, the zero-channel floor
// 0.1 with sv = 0).
//
// Readings (the oracle implements the same):
//   S_c   = sum over 32 consecutive row slices (ceil(rows / 32) rows each), in
//           slice order, of each slice's binary64 sum of w^2 in row order;
//   skew  = tree(the m = max(1, rows / 50) largest sqrt(h)) / tree(all of
//           them), binary64 pairwise trees over the values sorted descending;
//   scale = 0.1 for S_c = 0 (and sv = 0); else fl32(sqrt(S_c / rows)) when
//           skew < 0.15 (or forced), else the global fl32(sqrt(tree(S) / n));
//   W_out = fl32(W / scale_c), sv_out = sv * scale_c.
#include "common.cuh"

namespace exl3 {

namespace {

constexpr int kSlices = 32;
constexpr double kCutoff = 0.15;
constexpr float kZeroFloor = 0.1f;

__device__ __forceinline__ float load_w(const void *p, int dt, size_t idx) {
    if (dt == EXL3_BF16)
        return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p)[idx]);
    return reinterpret_cast<const float *>(p)[idx];
}

// part[s][c] = sum_{r in slice s} w[r][c]^2 (binary64, ascending r)
__global__ void __launch_bounds__(256) slice_sumsq_kernel(const void *__restrict__ W, int dt,
                                                          int64_t rows, int64_t cols,
                                                          double *__restrict__ part) {
    const int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int s = blockIdx.y;
    if (c >= cols)
        return;
    const int64_t len = (rows + kSlices - 1) / kSlices;
    const int64_t r0 = (int64_t)s * len;
    const int64_t r1 = r0 + len < rows ? r0 + len : rows;
    double acc = 0.0;
    for (int64_t r = r0; r < r1; r++) {
        const double w = (double)load_w(W, dt, (size_t)(r * cols + c));
        acc = __dadd_rn(acc, __dmul_rn(w, w));
    }
    part[(int64_t)s * cols + c] = acc;
}

// S[c] = slice sums added in slice order
__global__ void slice_combine_kernel(const double *__restrict__ part, int64_t cols,
                                     double *__restrict__ S) {
    const int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= cols)
        return;
    double t = 0.0;
    for (int s = 0; s < kSlices; s++)
        t = __dadd_rn(t, part[(int64_t)s * cols + c]);
    S[c] = t;
}

// d = sqrt(h) (binary64, -0 turned into +0) padded to P (a power of two) with
// -1; stored as the int64 bit patterns, whose signed order is the numeric
// order of non-negative doubles with the padding last.
__global__ void skew_sqrt_kernel(const float *__restrict__ h, int64_t rows, int64_t P,
                                 long long *__restrict__ d) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < P)
        d[i] = __double_as_longlong(i < rows ? __dadd_rn(__dsqrt_rn((double)h[i]), 0.0) : -1.0);
}

// One block: bitonic sort of the bit patterns into descending order, in
// shared memory when P <= kSortSmem (then copied back), else in place in d.
constexpr int64_t kSortSmem = 16384;

__global__ void __launch_bounds__(1024) skew_sort_kernel(int64_t P, long long *__restrict__ dg) {
    extern __shared__ long long dsm[];
    const bool in_smem = P <= kSortSmem;
    long long *d = in_smem ? dsm : dg;
    if (in_smem) {
        for (int64_t i = threadIdx.x; i < P; i += blockDim.x)
            dsm[i] = dg[i];
        __syncthreads();
    }
    for (int64_t k = 2; k <= P; k <<= 1) {
        for (int64_t j = k >> 1; j > 0; j >>= 1) {
            for (int64_t i = threadIdx.x; i < P; i += blockDim.x) {
                const int64_t ixj = i ^ j;
                if (ixj > i) {
                    const long long a = d[i], b = d[ixj];
                    const bool desc = (i & k) == 0;
                    if (desc ? (a < b) : (a > b)) {
                        d[i] = b;
                        d[ixj] = a;
                    }
                }
            }
            __syncthreads();
        }
    }
    if (in_smem)
        for (int64_t i = threadIdx.x; i < P; i += blockDim.x)
            dg[i] = dsm[i];
}

// hs = {tree of the top m, tree of all}: skew, the decision and the global RMS.
// info: [0] skew, [1] apply (0/1), [2] zeros (0/1), [3] global rms
__global__ void skew_decide_kernel(const double *hs, const double *total, int64_t n_elems,
                                   int apply_out, double *__restrict__ info,
                                   float *__restrict__ g_rms) {
    const double skew = hs[1] == 0.0 ? 0.0 : __ddiv_rn(hs[0], hs[1]);
    const bool app = apply_out < 0 ? (skew < kCutoff) : (apply_out != 0);
    const double t = *total;
    const float g = __double2float_rn(__dsqrt_rn(__ddiv_rn(t, (double)n_elems)));
    info[0] = skew;
    info[1] = app ? 1.0 : 0.0;
    info[2] = t == 0.0 ? 1.0 : 0.0;
    info[3] = (double)g;
    *g_rms = g;
}

// per-channel scale and sv_out
__global__ void channel_scale_kernel(const double *__restrict__ S, int64_t rows, int64_t cols,
                                     const double *__restrict__ info, const float *__restrict__ g_rms,
                                     const float *__restrict__ sv, float *__restrict__ scale,
                                     float *__restrict__ sv_out) {
    const int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= cols)
        return;
    const double s = S[c];
    float sc;
    if (s == 0.0)
        sc = kZeroFloor;
    else if (info[1] != 0.0)
        sc = __double2float_rn(__dsqrt_rn(__ddiv_rn(s, (double)rows)));
    else
        sc = *g_rms;
    scale[c] = sc;
    sv_out[c] = s == 0.0 ? 0.0f : __fmul_rn(sv[c], sc);
}

// W_out = fl32(W / scale_c); thread per column, blocks stride over rows; may
// run in place on an fp32 W (each element is read and written by one thread)
__global__ void normalise_kernel(const void *W, int dt, int64_t rows, int64_t cols,
                                 const float *__restrict__ scale, float *W_out) {
    const int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= cols)
        return;
    const float sc = scale[c];
    for (int64_t r = blockIdx.y; r < rows; r += gridDim.y)
        W_out[r * cols + c] = __fdiv_rn(load_w(W, dt, (size_t)(r * cols + c)), sc);
}

// the same with four consecutive columns per thread (cols % 4 == 0): one
// 8- or 16-byte load and one 16-byte store per row
__global__ void normalise4_kernel(const void *W, int dt, int64_t rows, int64_t cols,
                                  const float *__restrict__ scale, float *W_out) {
    const int64_t c4 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (4 * c4 >= cols)
        return;
    const float4 sc = reinterpret_cast<const float4 *>(scale)[c4];
    const int64_t q = cols / 4;
    for (int64_t r = blockIdx.y; r < rows; r += gridDim.y) {
        float4 w;
        if (dt == EXL3_BF16) {
            const uint2 b = reinterpret_cast<const uint2 *>(W)[r * q + c4];
            w.x = __uint_as_float(b.x << 16);
            w.y = __uint_as_float(b.x & 0xFFFF0000u);
            w.z = __uint_as_float(b.y << 16);
            w.w = __uint_as_float(b.y & 0xFFFF0000u);
        } else {
            w = reinterpret_cast<const float4 *>(W)[r * q + c4];
        }
        float4 o;
        o.x = __fdiv_rn(w.x, sc.x);
        o.y = __fdiv_rn(w.y, sc.y);
        o.z = __fdiv_rn(w.z, sc.z);
        o.w = __fdiv_rn(w.w, sc.w);
        reinterpret_cast<float4 *>(W_out)[r * q + c4] = o;
    }
}

bool aligned_to(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

}  // namespace

int64_t regularize_sort_len(int64_t rows) {
    int64_t P = 1;
    while (P < rows)
        P <<= 1;
    return P;
}

exl3_status run_regularize(const RegularizeLaunch &p, cudaStream_t s) {
    exl3_status st;
    const unsigned gc = (unsigned)((p.cols + 255) / 256);
    slice_sumsq_kernel<<<dim3(gc, kSlices), 256, 0, s>>>(p.W, p.dt, p.rows, p.cols, p.part);
    note_launch();
    slice_combine_kernel<<<gc, 256, 0, s>>>(p.part, p.cols, p.S);
    note_launch();
    if ((st = cuda_check(cudaGetLastError(), "block_rms launch")) != EXL3_OK) return st;
    if ((st = launch_tree_sum(p.S, p.cols, p.tree_scr, p.total, s)) != EXL3_OK) return st;
    const int64_t P = regularize_sort_len(p.rows);
    const size_t smem = P <= kSortSmem ? (size_t)P * sizeof(long long) : 0;
    skew_sqrt_kernel<<<(unsigned)((P + 255) / 256), 256, 0, s>>>(p.h, p.rows, P,
                                                                  (long long *)p.sortbuf);
    note_launch();
    if ((st = cuda_check(cudaFuncSetAttribute(skew_sort_kernel,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              (int)(kSortSmem * sizeof(long long))),
                         "cudaFuncSetAttribute(skew)")) != EXL3_OK)
        return st;
    skew_sort_kernel<<<1, 1024, smem, s>>>(P, (long long *)p.sortbuf);
    note_launch();
    if ((st = cuda_check(cudaGetLastError(), "skew sort launch")) != EXL3_OK) return st;
    const int64_t m = p.rows / 50 > 1 ? p.rows / 50 : 1;
    if ((st = launch_tree_sum(p.sortbuf, m, p.tree_scr, p.hsum, s)) != EXL3_OK) return st;
    if ((st = launch_tree_sum(p.sortbuf, p.rows, p.tree_scr, p.hsum + 1, s)) != EXL3_OK) return st;
    skew_decide_kernel<<<1, 1, 0, s>>>(p.hsum, p.total, p.rows * p.cols, p.apply_out, p.info,
                                       p.g_rms);
    note_launch();
    channel_scale_kernel<<<gc, 256, 0, s>>>(p.S, p.rows, p.cols, p.info, p.g_rms, p.sv, p.scale,
                                            p.sv_out);
    note_launch();
    const bool vec = p.cols % 4 == 0 && aligned_to(p.W, p.dt == EXL3_BF16 ? 8 : 16) &&
                     aligned_to(p.W_out, 16);
    const unsigned gx = vec ? (unsigned)((p.cols / 4 + 255) / 256) : gc;
    const int64_t ry = (152 * 16 + gx - 1) / gx;       // about 16 blocks of 256 per SM
    const unsigned gy = (unsigned)(p.rows < ry ? p.rows : ry);
    if (vec)
        normalise4_kernel<<<dim3(gx, gy), 256, 0, s>>>(p.W, p.dt, p.rows, p.cols, p.scale, p.W_out);
    else
        normalise_kernel<<<dim3(gx, gy), 256, 0, s>>>(p.W, p.dt, p.rows, p.cols, p.scale, p.W_out);
    note_launch();
    if (p.info_out) {
        if ((st = cuda_check(cudaMemcpyAsync(p.info_out, p.info, 4 * sizeof(double),
                                             cudaMemcpyDeviceToDevice, s),
                             "info copy")) != EXL3_OK)
            return st;
    }
    return cuda_check(cudaGetLastError(), "regularize launch");
}

}  // namespace exl3
