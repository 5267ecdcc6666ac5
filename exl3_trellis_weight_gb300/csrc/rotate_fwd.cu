// rotate_fwd.cu -- forward blockwise Sylvester Hadamard rotation without lane
// exchanges (page "EXL3 Intel Arc Quantizer", Core Implemented Architecture
// item 7: R = H (su . W . sv) H per 128 x 128 block, unnormalised butterflies
// then one exact 2^-7).
//
// The 2-D transform of a 128 x 128 block is 14 butterfly stages over the 2^14
// element index (i, j): the seven stages along j (within a row, spans 1..64
// ascending), then the seven along i.  Each thread of the 512-thread block holds
// 32 elements whose index differs in five bits, so five stages run in registers;
// two transposes through shared memory bring the next bits into registers:
//   phase 1: j bits 0..4        -> j spans 1, 2, 4, 8, 16
//   phase 2: j bits 5, 6, i 0..2 -> j spans 32, 64; x su; i spans 1, 2, 4
//   phase 3: i bits 3..6, j bit 0 -> i spans 8, 16, 32, 64; x 2^-7
// Every butterfly is (a, b) -> (a + b, a - b) with a at the lower index and the
// stages keep the order above, so the result is bit-identical to the plain
// in-place transform (and to the shuffle-based kernel in rotate.cu).
//
// Shared memory holds the block row-major, each row's 16-byte groups permuted
// inside every run of eight by an XOR (offset function blk_off), so that the
// 16-byte stores of phase 1, the 4-byte loads of phase 2 and the 8-byte loads
// of phase 3 all touch 32 distinct banks per wavefront.
#include "common.cuh"

namespace exl3 {

namespace {

constexpr int kFwdThreads = 512;

__device__ __forceinline__ int blk_off(int i, int j) {
    const int g = j >> 2;                              // 16-byte group, 0..31
    const int h = ((g >> 3) | ((i & 1) << 2)) & 7;     // permutes g's low three bits
    return i * 128 + ((g ^ h) << 2) + (j & 3);
}

template <int SPAN, int N>
__device__ __forceinline__ void bfly(float (&x)[N]) {
#pragma unroll
    for (int e = 0; e < N; e++) {
        if ((e & SPAN) == 0) {
            const float a = x[e], b = x[e + SPAN];
            x[e] = __fadd_rn(a, b);
            x[e + SPAN] = __fsub_rn(a, b);
        }
    }
}

// One block per 128 x 128 block (two resident per SM).
__global__ void __launch_bounds__(kFwdThreads, 2) rotate_fwd_kernel(const RotateLaunch a) {
    extern __shared__ __align__(16) float sblk[];      // [128 * 128], swizzled rows
    const int t = threadIdx.x;
    const int nbc = (int)(a.cols / 128);
    const size_t cols = (size_t)a.cols;
    {
        const int blk = blockIdx.x;
        const int rb = blk / nbc, cb = blk % nbc;
        const int r0 = rb * 128, c0 = cb * 128;

        // ---- phase 1: row i, columns 32 jh .. 32 jh + 31 -------------------
        {
            const int i = t >> 2, jh = t & 3;
            float x[32];
            const size_t base = (size_t)(r0 + i) * cols + (size_t)(c0 + 32 * jh);
            const float4 *svp = reinterpret_cast<const float4 *>(a.sv + c0 + 32 * jh);
            if (a.src == SRC_BF16) {
                const uint4 *p = reinterpret_cast<const uint4 *>(
                    reinterpret_cast<const __nv_bfloat16 *>(a.in) + base);
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    const uint4 w = p[q];
                    const float4 s0 = __ldg(svp + 2 * q), s1 = __ldg(svp + 2 * q + 1);
                    x[8 * q + 0] = __fmul_rn(__uint_as_float(w.x << 16), s0.x);
                    x[8 * q + 1] = __fmul_rn(__uint_as_float(w.x & 0xFFFF0000u), s0.y);
                    x[8 * q + 2] = __fmul_rn(__uint_as_float(w.y << 16), s0.z);
                    x[8 * q + 3] = __fmul_rn(__uint_as_float(w.y & 0xFFFF0000u), s0.w);
                    x[8 * q + 4] = __fmul_rn(__uint_as_float(w.z << 16), s1.x);
                    x[8 * q + 5] = __fmul_rn(__uint_as_float(w.z & 0xFFFF0000u), s1.y);
                    x[8 * q + 6] = __fmul_rn(__uint_as_float(w.w << 16), s1.z);
                    x[8 * q + 7] = __fmul_rn(__uint_as_float(w.w & 0xFFFF0000u), s1.w);
                }
            } else {
                const float4 *p =
                    reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(a.in) + base);
#pragma unroll
                for (int q = 0; q < 8; q++) {
                    const float4 w = p[q];
                    const float4 sq = __ldg(svp + q);
                    x[4 * q] = __fmul_rn(w.x, sq.x);
                    x[4 * q + 1] = __fmul_rn(w.y, sq.y);
                    x[4 * q + 2] = __fmul_rn(w.z, sq.z);
                    x[4 * q + 3] = __fmul_rn(w.w, sq.w);
                }
            }
            bfly<1>(x);
            bfly<2>(x);
            bfly<4>(x);
            bfly<8>(x);
            bfly<16>(x);
#pragma unroll
            for (int q = 0; q < 8; q++)
                *reinterpret_cast<float4 *>(sblk + blk_off(i, 32 * jh + 4 * q)) =
                    make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
        }
        __syncthreads();

        // ---- phase 2: rows 8 ib .. 8 ib + 7, columns jlo + 32 jh -----------
        {
            const int ib = t >> 5, jlo = t & 31;
            float x[32];                               // x[8 jh + il]
#pragma unroll
            for (int jh = 0; jh < 4; jh++)
#pragma unroll
                for (int il = 0; il < 8; il++)
                    x[8 * jh + il] = sblk[blk_off(8 * ib + il, jlo + 32 * jh)];
            bfly<8>(x);                                // j span 32 (jh bit 0)
            bfly<16>(x);                               // j span 64 (jh bit 1)
#pragma unroll
            for (int il = 0; il < 8; il++) {
                const float su = __ldg(a.su + r0 + 8 * ib + il);
#pragma unroll
                for (int jh = 0; jh < 4; jh++)
                    x[8 * jh + il] = __fmul_rn(x[8 * jh + il], su);
            }
            bfly<1>(x);                                // i span 1
            bfly<2>(x);                                // i span 2
            bfly<4>(x);                                // i span 4
#pragma unroll
            for (int jh = 0; jh < 4; jh++)
#pragma unroll
                for (int il = 0; il < 8; il++)
                    sblk[blk_off(8 * ib + il, jlo + 32 * jh)] = x[8 * jh + il];
        }
        __syncthreads();

        // ---- phase 3: rows ilo + 8 ih, columns 2 jp, 2 jp + 1 ---------------
        {
            const int ilo = t >> 6, jp = t & 63;
            float x[32];                               // x[2 ih + jb]
#pragma unroll
            for (int ih = 0; ih < 16; ih++) {
                const float2 v =
                    *reinterpret_cast<const float2 *>(sblk + blk_off(ilo + 8 * ih, 2 * jp));
                x[2 * ih] = v.x;
                x[2 * ih + 1] = v.y;
            }
            bfly<2>(x);                                // i span 8  (ih bit 0)
            bfly<4>(x);                                // i span 16
            bfly<8>(x);                                // i span 32
            bfly<16>(x);                               // i span 64
#pragma unroll
            for (int e = 0; e < 32; e++)
                x[e] = __fmul_rn(x[e], 0x1p-7f);
            if (a.out) {
                float *op = a.out + (size_t)(r0 + ilo) * cols + (size_t)(c0 + 2 * jp);
#pragma unroll
                for (int ih = 0; ih < 16; ih++)
                    *reinterpret_cast<float2 *>(op + (size_t)(8 * ih) * cols) =
                        make_float2(x[2 * ih], x[2 * ih + 1]);
            }
            if (a.tile_sums) {
#pragma unroll
                for (int ih = 0; ih < 16; ih++)
                    *reinterpret_cast<float2 *>(sblk + blk_off(ilo + 8 * ih, 2 * jp)) =
                        make_float2(x[2 * ih], x[2 * ih + 1]);
            }
        }
        if (a.tile_sums) {
            __syncthreads();
            // per-tile fp64 sums of R^2, sequential in row-major order inside each 16x16 tile
            if (t < 64) {
                const int ti = t >> 3, tj = t & 7;
                double s = 0.0;
                for (int i = 0; i < 16; i++)
                    for (int j = 0; j < 16; j++) {
                        const double v = (double)sblk[blk_off(ti * 16 + i, tj * 16 + j)];
                        s = __dadd_rn(s, __dmul_rn(v, v));
                    }
                a.tile_sums[(size_t)(rb * 8 + ti) * (size_t)(a.cols / 16) + cb * 8 + tj] = s;
            }
        }
    }
}

}  // namespace

bool rotate_fwd_eligible(const RotateLaunch &p) {
    auto al16 = [](const void *q) { return ((uintptr_t)q & 15u) == 0; };
    return !p.inverse && (p.src == SRC_F32 || p.src == SRC_BF16) && !p.ref && al16(p.in) &&
           al16(p.sv) && (!p.out || al16(p.out));
}

exl3_status launch_rotate_fwd(const RotateLaunch &p, cudaStream_t s) {
    const int64_t nblk = (p.rows / 128) * (p.cols / 128);
    if (nblk == 0)
        return EXL3_OK;
    if (rotate_fwd_tma_eligible(p)) {
        const exl3_status st = launch_rotate_fwd_tma(p, s);
        if (st != EXL3_ERR_UNSUPPORTED)
            return st;
    }
    const size_t smem = (size_t)128 * 128 * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(rotate_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess)
        return cuda_check(e, "cudaFuncSetAttribute(rotate_fwd)");
    rotate_fwd_kernel<<<(unsigned)nblk, kFwdThreads, smem, s>>>(p);
    note_launch();
    note_rotate_kernel(2);
    return cuda_check(cudaGetLastError(), "rotate_fwd launch");
}

}  // namespace exl3
