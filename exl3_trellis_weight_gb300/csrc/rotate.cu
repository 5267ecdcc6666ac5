// rotate.cu -- blockwise Sylvester Hadamard rotation, tile decode and the
// fixed-order fp64 reductions (page "EXL3 Intel Arc Quantizer", Core
// Implemented Architecture items 5, 7 and 10).
//
// Rotation: one 512-thread block per 128x128 block of the matrix, staged in
// shared memory (pitch 129 floats: column reads are bank-conflict free).
// A 128-point transform is held by one warp, lane l owning elements
// l, l+32, l+64, l+96: butterfly spans 1..16 are lane exchanges (shfl.xor),
// spans 32 and 64 are inside the lane.  The stage order is always 1,2,...,64
// and each butterfly is (a, b) -> (a+b, a-b) with a the lower index, so the
// result is bit-identical to a plain in-place transform.
#include "common.cuh"

namespace exl3 {

namespace {

constexpr int kRotThreads = 512;
constexpr int kPitch = 129;

// x[i] holds element lane + 32*i of a 128-vector; in-place x <- H x.
__device__ __forceinline__ void fwht128_warp(float (&x)[4], const int lane) {
#pragma unroll
    for (int h = 1; h < 32; h <<= 1) {
        const bool upper = (lane & h) != 0;   // this lane holds the "b" element
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const float o = __shfl_xor_sync(0xffffffffu, x[i], h);
            x[i] = upper ? __fsub_rn(o, x[i]) : __fadd_rn(x[i], o);
        }
    }
    // span 32: (x0, x1), (x2, x3); span 64: (x0, x2), (x1, x3)
    float a0 = __fadd_rn(x[0], x[1]), a1 = __fsub_rn(x[0], x[1]);
    float a2 = __fadd_rn(x[2], x[3]), a3 = __fsub_rn(x[2], x[3]);
    x[0] = __fadd_rn(a0, a2);
    x[2] = __fsub_rn(a0, a2);
    x[1] = __fadd_rn(a1, a3);
    x[3] = __fsub_rn(a1, a3);
}

__device__ __forceinline__ float load_elem(const void *p, int dt, size_t idx) {
    if (dt == EXL3_BF16)
        return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p)[idx]);
    return reinterpret_cast<const float *>(p)[idx];
}

__global__ void __launch_bounds__(kRotThreads) rotate_kernel(const RotateLaunch a) {
    extern __shared__ __align__(16) unsigned char smem[];
    float *tile = reinterpret_cast<float *>(smem);                  // [128][kPitch]
    uint32_t *cw = reinterpret_cast<uint32_t *>(tile + 128 * kPitch); // codes of 64 tiles

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t nbc = a.cols / 128;
    const int64_t rb = blockIdx.x / nbc, cb = blockIdx.x % nbc;
    const int64_t r0 = rb * 128, c0 = cb * 128;
    const int64_t tiles_c = a.cols / 16;
    const float two_m7 = 0x1p-7f;

    if (!a.inverse) {
        // x sv (columns), rows x H, x su (rows)
        float sv[4];
#pragma unroll
        for (int i = 0; i < 4; i++)
            sv[i] = a.sv[c0 + lane + 32 * i];
        for (int rr = 0; rr < 8; rr++) {
            const int r = warp * 8 + rr;
            const size_t base = (size_t)(r0 + r) * a.cols + c0;
            float x[4];
#pragma unroll
            for (int i = 0; i < 4; i++)
                x[i] = __fmul_rn(load_elem(a.in, a.src, base + lane + 32 * i), sv[i]);
            fwht128_warp(x, lane);
            const float su = a.su[r0 + r];
#pragma unroll
            for (int i = 0; i < 4; i++)
                tile[r * kPitch + lane + 32 * i] = __fmul_rn(x[i], su);
        }
        __syncthreads();
        // H x columns, x 2^-7
        for (int cc = 0; cc < 8; cc++) {
            const int c = warp * 8 + cc;
            float x[4];
#pragma unroll
            for (int i = 0; i < 4; i++)
                x[i] = tile[(lane + 32 * i) * kPitch + c];
            fwht128_warp(x, lane);
#pragma unroll
            for (int i = 0; i < 4; i++)
                tile[(lane + 32 * i) * kPitch + c] = __fmul_rn(x[i], two_m7);
        }
        __syncthreads();
    } else {
        // source rows into shared memory
        if (a.src == SRC_CODES) {
            const int NW = 8 * a.K;
            const uint32_t *codes = reinterpret_cast<const uint32_t *>(a.in);
            for (int q = threadIdx.x; q < 64 * NW; q += kRotThreads) {
                const int t = q / NW, w = q % NW;
                const int64_t gt = (rb * 8 + t / 8) * tiles_c + cb * 8 + (t % 8);
                cw[q] = codes[(size_t)gt * NW + w];
            }
            __syncthreads();
            const float sc = *a.scale_dev;
            for (int rr = 0; rr < 8; rr++) {
                const int r = warp * 8 + rr;
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    const int c = lane + 32 * i;
                    const int t = (r >> 4) * 8 + (c >> 4);
                    const uint32_t st = window_state_k(cw + t * NW, (r & 15) * 16 + (c & 15), a.K);
                    tile[r * kPitch + c] = __fmul_rn(mul1_value(st), sc);
                }
            }
        } else {
            for (int rr = 0; rr < 8; rr++) {
                const int r = warp * 8 + rr;
                const size_t base = (size_t)(r0 + r) * a.cols + c0;
#pragma unroll
                for (int i = 0; i < 4; i++)
                    tile[r * kPitch + lane + 32 * i] = load_elem(a.in, a.src, base + lane + 32 * i);
            }
        }
        __syncthreads();
        // H x columns, x su (rows)
        float su[4];
#pragma unroll
        for (int i = 0; i < 4; i++)
            su[i] = a.su[r0 + lane + 32 * i];
        for (int cc = 0; cc < 8; cc++) {
            const int c = warp * 8 + cc;
            float x[4];
#pragma unroll
            for (int i = 0; i < 4; i++)
                x[i] = tile[(lane + 32 * i) * kPitch + c];
            fwht128_warp(x, lane);
#pragma unroll
            for (int i = 0; i < 4; i++)
                tile[(lane + 32 * i) * kPitch + c] = __fmul_rn(x[i], su[i]);
        }
        __syncthreads();
        // rows x H, x sv (columns), x 2^-7
        float sv[4];
#pragma unroll
        for (int i = 0; i < 4; i++)
            sv[i] = a.sv[c0 + lane + 32 * i];
        for (int rr = 0; rr < 8; rr++) {
            const int r = warp * 8 + rr;
            float x[4];
#pragma unroll
            for (int i = 0; i < 4; i++)
                x[i] = tile[r * kPitch + lane + 32 * i];
            fwht128_warp(x, lane);
#pragma unroll
            for (int i = 0; i < 4; i++)
                tile[r * kPitch + lane + 32 * i] = __fmul_rn(__fmul_rn(x[i], sv[i]), two_m7);
        }
        __syncthreads();
    }

    // store (coalesced rows)
    if (a.out) {
        for (int rr = 0; rr < 8; rr++) {
            const int r = warp * 8 + rr;
            const size_t base = (size_t)(r0 + r) * a.cols + c0;
#pragma unroll
            for (int i = 0; i < 4; i++)
                a.out[base + lane + 32 * i] = tile[r * kPitch + lane + 32 * i];
        }
    }
    // per-tile fp64 sums, sequential in row-major order inside each 16x16 tile
    if (a.tile_sums && threadIdx.x < 64) {
        const int ti = threadIdx.x >> 3, tj = threadIdx.x & 7;
        double s = 0.0;
        for (int i = 0; i < 16; i++) {
            const int r = ti * 16 + i;
            for (int j = 0; j < 16; j++) {
                const int c = tj * 16 + j;
                double v = (double)tile[r * kPitch + c];
                if (a.ref)
                    v = __dsub_rn((double)load_elem(a.ref, a.ref_dt, (size_t)(r0 + r) * a.cols + c0 + c), v);
                s = __dadd_rn(s, __dmul_rn(v, v));
            }
        }
        a.tile_sums[(rb * 8 + ti) * tiles_c + cb * 8 + tj] = s;
    }
}

// Decode: one 128-thread block per 16-row strip of 8 tiles.
__global__ void __launch_bounds__(128) decode_kernel(const uint32_t *__restrict__ codes, int64_t rows,
                                                     int64_t cols, int K, float scale,
                                                     const float *scale_dev, float *__restrict__ out) {
    __shared__ uint32_t cw[8 * 32];
    const int64_t tiles_c = cols / 16;
    const int64_t groups = (tiles_c + 7) / 8;
    const int64_t tr = blockIdx.x / groups, tg = blockIdx.x % groups;
    const int NW = 8 * K;
    const int64_t t0 = tr * tiles_c + tg * 8;
    const int nt = (int)((tiles_c - tg * 8) < 8 ? (tiles_c - tg * 8) : 8);
    for (int q = threadIdx.x; q < nt * NW; q += 128)
        cw[q] = codes[(size_t)t0 * NW + q];
    __syncthreads();
    const float sc = scale_dev ? *scale_dev : scale;
    const int c = threadIdx.x;
    const int t = c >> 4;
    if (t >= nt)
        return;
    const int64_t col = (tg * 8 + t) * 16 + (c & 15);
    for (int r = 0; r < 16; r++) {
        const uint32_t st = window_state_k(cw + t * NW, r * 16 + (c & 15), K);
        out[(size_t)(tr * 16 + r) * cols + col] = __fmul_rn(mul1_value(st), sc);
    }
}

// Rows of T targets: one thread per element; state i is the 16-bit window of
// the row's circular T*K-bit stream ending with the last bit of code i.
__global__ void decode_rows_kernel(const uint32_t *__restrict__ codes, int64_t n_rows, int T, int K,
                                   float scale, float *__restrict__ out) {
    const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= n_rows * T)
        return;
    const int64_t r = e / T;
    const int i = (int)(e % T);
    const int NB = T * K, NW = T * K / 32;
    const uint32_t *w = codes + (size_t)r * NW;
    int p = (i + 1) * K - 16;
    while (p < 0)
        p += NB;
    const int wi = p >> 5;
    const int wj = (wi + 1 == NW) ? 0 : wi + 1;
    const unsigned long long cat = ((unsigned long long)__ldg(w + wi) << 32) | __ldg(w + wj);
    const uint32_t st = (uint32_t)(cat >> (48 - (p & 31))) & 0xFFFFu;
    out[e] = __fmul_rn(mul1_value(st), scale);
}

// Per-tile fp64 sum of x^2 or (x - ref)^2, one thread per tile.
__global__ void tile_sumsq_kernel(const void *x, int x_dt, const float *ref, int64_t rows,
                                  int64_t cols, double *out) {
    const int64_t tiles_c = cols / 16;
    const int64_t n = (rows / 16) * tiles_c;
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= n)
        return;
    const int64_t tr = t / tiles_c, tc = t % tiles_c;
    double s = 0.0;
    for (int i = 0; i < 16; i++)
        for (int j = 0; j < 16; j++) {
            const size_t idx = (size_t)(tr * 16 + i) * cols + tc * 16 + j;
            double v = (double)load_elem(x, x_dt, idx);
            if (ref)
                v = __dsub_rn(v, (double)ref[idx]);
            s = __dadd_rn(s, __dmul_rn(v, v));
        }
    out[t] = s;
}

// Pairwise tree over an aligned block of up to 2048 values (level by level:
// neighbours (2i, 2i+1), an odd last element moves up).  Block b reduces
// in[b*2048, min((b+1)*2048, n)).  Aligned power-of-two blocks reproduce the
// whole-array tree exactly.
constexpr int kTreeBlock = 2048;
__global__ void __launch_bounds__(1024) tree_kernel(const double *__restrict__ in, int64_t n,
                                                    double *__restrict__ out) {
    __shared__ double v[kTreeBlock];
    const int64_t base = (int64_t)blockIdx.x * kTreeBlock;
    int m = (int)((n - base) < kTreeBlock ? (n - base) : kTreeBlock);
    for (int i = threadIdx.x; i < m; i += blockDim.x)
        v[i] = in[base + i];
    __syncthreads();
    while (m > 1) {
        const int h = m >> 1;
        double r0 = 0.0, r1 = 0.0;
        const int i0 = threadIdx.x, i1 = threadIdx.x + 1024;
        if (i0 < h) r0 = __dadd_rn(v[2 * i0], v[2 * i0 + 1]);
        if (i1 < h) r1 = __dadd_rn(v[2 * i1], v[2 * i1 + 1]);
        double carry = 0.0;
        const bool odd = (m & 1) != 0;
        if (odd && threadIdx.x == 0) carry = v[m - 1];
        __syncthreads();
        if (i0 < h) v[i0] = r0;
        if (i1 < h) v[i1] = r1;
        if (odd && threadIdx.x == 0) v[h] = carry;
        __syncthreads();
        m = h + (odd ? 1 : 0);
    }
    if (threadIdx.x == 0)
        out[blockIdx.x] = v[0];
}

}  // namespace

exl3_status launch_rotate(const RotateLaunch &p, cudaStream_t s) {
    const int64_t nblk = (p.rows / 128) * (p.cols / 128);
    if (nblk == 0)
        return EXL3_OK;
    if (rotate_fwd_eligible(p))
        return launch_rotate_fwd(p, s);
    const size_t smem = (size_t)128 * kPitch * sizeof(float) + (size_t)64 * 32 * sizeof(uint32_t);
    cudaError_t e = cudaFuncSetAttribute(rotate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess)
        return cuda_check(e, "cudaFuncSetAttribute(rotate)");
    rotate_kernel<<<(unsigned)nblk, kRotThreads, smem, s>>>(p);
    note_launch();
    note_rotate_kernel(3);
    return cuda_check(cudaGetLastError(), "rotate launch");
}

exl3_status launch_decode(const uint32_t *codes, int64_t rows, int64_t cols, int K, float scale,
                          const float *scale_dev, float *out, cudaStream_t s) {
    const int64_t tiles_c = cols / 16;
    const int64_t nblk = (rows / 16) * ((tiles_c + 7) / 8);
    if (nblk == 0)
        return EXL3_OK;
    decode_kernel<<<(unsigned)nblk, 128, 0, s>>>(codes, rows, cols, K, scale, scale_dev, out);
    note_launch();
    return cuda_check(cudaGetLastError(), "decode launch");
}

exl3_status launch_decode_rows(const uint32_t *codes, int64_t n_rows, int T, int K, float scale,
                               float *out, cudaStream_t s) {
    const int64_t n = n_rows * T;
    if (n == 0)
        return EXL3_OK;
    decode_rows_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(codes, n_rows, T, K, scale, out);
    note_launch();
    return cuda_check(cudaGetLastError(), "decode_rows launch");
}

exl3_status launch_tile_sumsq(const void *x, int x_dt, const float *ref, int64_t rows, int64_t cols,
                              double *tile_sums, cudaStream_t s) {
    const int64_t n = (rows / 16) * (cols / 16);
    if (n == 0)
        return EXL3_OK;
    tile_sumsq_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(x, x_dt, ref, rows, cols, tile_sums);
    note_launch();
    return cuda_check(cudaGetLastError(), "tile_sumsq launch");
}

size_t tree_scratch_doubles(int64_t n) {
    size_t tot = 0;
    while (n > kTreeBlock) {
        n = (n + kTreeBlock - 1) / kTreeBlock;
        tot += (size_t)n;
    }
    return tot + 1;
}

exl3_status launch_tree_sum(const double *in, int64_t n, double *scratch, double *out,
                            cudaStream_t s) {
    if (n <= 0) {
        cudaError_t e = cudaMemsetAsync(out, 0, sizeof(double), s);
        return cuda_check(e, "tree memset");
    }
    const double *cur = in;
    double *nxt = scratch;
    while (n > kTreeBlock) {
        const int64_t m = (n + kTreeBlock - 1) / kTreeBlock;
        tree_kernel<<<(unsigned)m, 1024, 0, s>>>(cur, n, nxt);
        note_launch();
        cur = nxt;
        nxt += m;
        n = m;
    }
    tree_kernel<<<1, 1024, 0, s>>>(cur, n, out);
    note_launch();
    return cuda_check(cudaGetLastError(), "tree launch");
}

}  // namespace exl3
