// rotate_fwd_tma.cu -- forward blockwise Sylvester Hadamard rotation of a bf16
// matrix with TMA staging (page "EXL3 Intel Arc Quantizer", Core Implemented
// Architecture item 7: R = H (su . W . sv) H per 128 x 128 block, unnormalised
// butterflies then one exact 2^-7).
//
// Same arithmetic and stage order as rotate_fwd.cu (bit-identical results);
// what differs is the data movement.  Persistent 128-thread blocks, two per SM,
// walk the 128 x 128 blocks blockIdx.x, + gridDim.x, ...:
//   - the bf16 block arrives by two TMA loads (64-column boxes, 128-byte
//     swizzle) into the input stage, with its 128 column signs sv and 128 row
//     signs su (two 512-byte bulk copies on the same transaction barrier); the
//     next block's load is issued as soon as every thread has read the stage;
//   - phase A: thread t holds row t (128 values in registers): the column signs,
//     all seven column spans, the row sign; the rows go to a transpose buffer
//     whose element (j, r) sits at j * 128 + (r ^ 4 (j & 7)), so the scalar
//     writes (one j, 32 consecutive r per warp) and the 16-byte reads of phase B
//     (4 consecutive r of 32 consecutive j) are conflict-free;
//   - phase B: thread t holds column t: all seven row spans and the 2^-7 scale;
//     the result is written row-major over the same buffer (after every column
//     has been read) and leaves by one 128 x 128 TMA store, which overlaps the
//     next block until the next transpose write.
// Two arrangements instead of three move about 288 KiB of shared memory per
// block instead of 416 KiB (4096 x 4096: 22.45 -> 20.95 us).  Shared memory:
// a 33 KiB input stage and a 64 KiB transpose/output buffer.
//
// Each wait for a TMA load is bounded in time: on expiry the block stops
// waiting, issues no further load, waits (bounded) for the loads it issued,
// its results are void, and a device counter records it (exl3_wait_timeouts).
//
// The kernel is launched with programmatic stream serialization: its prologue
// (barrier set-up) may overlap the tail of the previous kernel in the stream,
// `griddepcontrol.wait` holds every global access until that kernel has
// completed, and each block allows the next kernel to launch once it has
// started its last 128 x 128 block (4096 x 4096: 25.0 -> 22.4 us).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"

namespace exl3 {

namespace {

constexpr int kTmaThreads = 128;                        // one row, then one column, per thread
constexpr uint32_t kBlockBytes = 128 * 128 * 2;        // one bf16 block (two 16 KiB boxes)
constexpr uint32_t kSignBytes = 2 * 128 * 4;           // sv[c0 .. c0+127], su[r0 .. r0+127]
constexpr uint32_t kStageBytes = kBlockBytes + 1024;   // keeps the transpose buffer 1024-byte aligned
constexpr uint32_t kTOff = kStageBytes;                // transpose buffer, then the output stage
constexpr uint32_t kSmemBytes = kTOff + 128 * 128 * 4; // 97 KiB: two blocks per SM
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

__device__ unsigned int g_rot_wait_timeouts;

__device__ __forceinline__ uint32_t saddr(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

// transpose buffer: element (j, r) -- column j of the rotated rows, row r -- at
// j * 128 + (r ^ 4 (j & 7)): a warp writing one j for 32 consecutive r and a warp
// reading 4 consecutive r of 32 consecutive j (16 bytes each) are both conflict-free
__device__ __forceinline__ int tr_off(int j, int r) {
    return j * 128 + (r ^ ((j & 7) << 2));
}

__device__ __forceinline__ void bfly_pair(float &a0, float &a1, float &b0, float &b1) {
    asm("{\n\t.reg .b64 a, b, s, d;\n\t"
        "mov.b64 a, {%0, %1};\n\t"
        "mov.b64 b, {%2, %3};\n\t"
        "add.rn.f32x2 s, a, b;\n\t"
        "sub.rn.f32x2 d, a, b;\n\t"
        "mov.b64 {%0, %1}, s;\n\t"
        "mov.b64 {%2, %3}, d;\n\t}"
        : "+f"(a0), "+f"(a1), "+f"(b0), "+f"(b1));
}

// one butterfly stage of span SPAN over all N elements (unnormalised)
template <int SPAN, int N>
__device__ __forceinline__ void bfly(float (&x)[N]) {
    if constexpr (SPAN == 1) {
#pragma unroll
        for (int e = 0; e < N; e += 2) {
            const float a = x[e], b = x[e + 1];
            x[e] = __fadd_rn(a, b);
            x[e + 1] = __fsub_rn(a, b);
        }
    } else {
#pragma unroll
        for (int e = 0; e < N; e += 2)
            if ((e & SPAN) == 0)
                bfly_pair(x[e], x[e + 1], x[e + SPAN], x[e + SPAN + 1]);
    }
}

template <int N>
__device__ __forceinline__ void fwht(float (&x)[N]) {
    bfly<1>(x);
    bfly<2>(x);
    bfly<4>(x);
    bfly<8>(x);
    bfly<16>(x);
    bfly<32>(x);
    bfly<64>(x);
}

__device__ __forceinline__ bool bar_test(uint32_t a, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(a), "r"(parity) : "memory");
    return ok != 0u;
}

__device__ __noinline__ void bar_wait_slow(uint32_t a, uint32_t parity, volatile int *gave_up) {
    unsigned long long t0;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t0));
    while (!bar_test(a, parity)) {
        if (*gave_up)
            return;
        unsigned long long t1;
        asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t1));
        if (t1 - t0 > kWaitLimitNs) {
            *gave_up = 1;
            atomicAdd(&g_rot_wait_timeouts, 1u);
            return;
        }
    }
}

__device__ __forceinline__ void bar_wait(uint32_t a, uint32_t parity, volatile int *gave_up) {
    if (!bar_test(a, parity))
        bar_wait_slow(a, parity, gave_up);
}

// thread 0: both 64-column boxes of block blk and its sign slices into input
// stage `stage` (block at +0, sv at +kBlockBytes, su at +kBlockBytes + 512)
__device__ __forceinline__ void issue_load(const CUtensorMap *map, const float *su, const float *sv,
                                           uint32_t stage_addr, uint32_t bar, int blk, int nbc) {
    const int r0 = (blk / nbc) * 128, c0 = (blk % nbc) * 128;
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(bar), "r"(kBlockBytes + kSignBytes) : "memory");
#pragma unroll
    for (int h = 0; h < 2; h++)
        asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
                     "[%0], [%1, {%2, %3}], [%4];"
                     :: "r"(stage_addr + (uint32_t)h * (kBlockBytes / 2)), "l"((uint64_t)map),
                        "r"(c0 + 64 * h), "r"(r0), "r"(bar)
                     : "memory");
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], 512, [%2];"
                 :: "r"(stage_addr + kBlockBytes), "l"((uint64_t)(sv + c0)), "r"(bar) : "memory");
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], 512, [%2];"
                 :: "r"(stage_addr + kBlockBytes + 512u), "l"((uint64_t)(su + r0)), "r"(bar) : "memory");
}

__global__ void __launch_bounds__(kTmaThreads, 2)
    rotate_fwd_tma_kernel(const __grid_constant__ CUtensorMap in_map,
                          const __grid_constant__ CUtensorMap out_map, const float *__restrict__ su,
                          const float *__restrict__ sv, const int rows, const int cols,
                          double *tile_sums) {
    extern __shared__ unsigned char smem_raw[];
    __shared__ __align__(8) unsigned long long full;
    __shared__ int gave_up;
    // the swizzled TMA destination wants 1024-byte alignment
    const uint32_t raw = saddr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    unsigned char *const sb = smem_raw + (base - raw);
    float *const T = reinterpret_cast<float *>(sb + kTOff);
    const int t = threadIdx.x;
    const int nbc = cols / 128;
    const int nblk = (rows / 128) * nbc;
    const uint32_t bar = saddr(&full);

    if (t == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(bar) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        gave_up = 0;
    }
    __syncthreads();
    // loads issued (thread 0's count); each is waited on before the next is issued,
    // so the barrier is at most one phase behind
    int issued = 0;
    // programmatic dependent launch: everything above overlaps the previous
    // kernel's tail; global memory is read only after it has completed
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (t == 0 && (int)blockIdx.x < nblk) {
        issue_load(&in_map, su, sv, base, bar, (int)blockIdx.x, nbc);
        issued = 1;
    }

    int it = 0;
    for (int blk = (int)blockIdx.x; blk < nblk; blk += (int)gridDim.x, it++) {
        const int r0 = (blk / nbc) * 128, c0 = (blk % nbc) * 128;
        bar_wait(bar, (uint32_t)it & 1u, &gave_up);
        if (blk + (int)gridDim.x >= nblk)
            asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

        // ---- phase A: row t, every column span (1 .. 64), then the row sign ----
        float x[128];
        float s_row;
        {
            const float4 *svp = reinterpret_cast<const float4 *>(sb + kBlockBytes);
#pragma unroll
            for (int h = 0; h < 2; h++)
#pragma unroll
                for (int g = 0; g < 8; g++) {
                    // 16-byte group g of the 128-byte row of box h, swizzled by the row
                    const uint4 w = *reinterpret_cast<const uint4 *>(sb + h * (kBlockBytes / 2) + t * 128 +
                                                                     ((g ^ (t & 7)) << 4));
                    const int j = 64 * h + 8 * g;
                    const float4 s0 = svp[j / 4], s1 = svp[j / 4 + 1];
                    x[j + 0] = __fmul_rn(__uint_as_float(w.x << 16), s0.x);
                    x[j + 1] = __fmul_rn(__uint_as_float(w.x & 0xFFFF0000u), s0.y);
                    x[j + 2] = __fmul_rn(__uint_as_float(w.y << 16), s0.z);
                    x[j + 3] = __fmul_rn(__uint_as_float(w.y & 0xFFFF0000u), s0.w);
                    x[j + 4] = __fmul_rn(__uint_as_float(w.z << 16), s1.x);
                    x[j + 5] = __fmul_rn(__uint_as_float(w.z & 0xFFFF0000u), s1.y);
                    x[j + 6] = __fmul_rn(__uint_as_float(w.w << 16), s1.z);
                    x[j + 7] = __fmul_rn(__uint_as_float(w.w & 0xFFFF0000u), s1.w);
                }
            s_row = reinterpret_cast<const float *>(sb + kBlockBytes + 512u)[t];
        }
        __syncthreads();                 // the input stage is free: load the next block
        if (t == 0 && blk + (int)gridDim.x < nblk && !gave_up) {
            issue_load(&in_map, su, sv, base, bar, blk + (int)gridDim.x, nbc);
            issued++;
        }
        fwht(x);
#pragma unroll
        for (int j = 0; j < 128; j++)
            x[j] = __fmul_rn(x[j], s_row);
        // the previous block's store must have finished reading the buffer
        if (t == 0)
            asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
        __syncthreads();
#pragma unroll
        for (int j = 0; j < 128; j++)
            T[tr_off(j, t)] = x[j];
        __syncthreads();

        // ---- phase B: column t, every row span (1 .. 64), then 2^-7 ----
#pragma unroll
        for (int q = 0; q < 32; q++) {
            const float4 v = *reinterpret_cast<const float4 *>(T + t * 128 + ((q ^ (t & 7)) << 2));
            x[4 * q] = v.x;
            x[4 * q + 1] = v.y;
            x[4 * q + 2] = v.z;
            x[4 * q + 3] = v.w;
        }
        __syncthreads();                 // every column is read: the buffer takes the output
        fwht(x);
#pragma unroll
        for (int i = 0; i < 128; i++)
            T[i * 128 + t] = __fmul_rn(x[i], 0x1p-7f);
        // generic-proxy writes of the output stage, then one TMA store of it
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();
        if (t == 0) {
            asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];"
                         :: "l"((uint64_t)&out_map), "r"(c0), "r"(r0), "r"(base + kTOff)
                         : "memory");
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        }
        if (tile_sums && t < 64) {
            // per-tile fp64 sums of R^2, sequential in row-major order inside each 16x16 tile
            const int ti = t >> 3, tj = t & 7;
            double s = 0.0;
            for (int i = 0; i < 16; i++)
                for (int j = 0; j < 16; j++) {
                    const double v = (double)T[(ti * 16 + i) * 128 + tj * 16 + j];
                    s = __dadd_rn(s, __dmul_rn(v, v));
                }
            tile_sums[(size_t)((r0 >> 4) + ti) * (size_t)(cols / 16) + (c0 >> 4) + tj] = s;
        }
    }
    if (t == 0) {
        // after a wait gave up, the last load issued may still be in flight: wait
        // (bounded) for it before the block exits, so that no copy lands in shared
        // memory of a block that is gone (n loads issued: phase n - 1 completes it)
        if (gave_up && issued > 0) {
            const uint32_t parity = (uint32_t)(issued - 1) & 1u;
            unsigned long long t0, t1;
            asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t0));
            do {
                asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t1));
            } while (!bar_test(bar, parity) && t1 - t0 < kWaitLimitNs);
        }
        asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    }
}

}  // namespace

namespace {

// cuTensorMapEncodeTiled, looked up once through the runtime (no link against
// the driver library).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            (void)cudaGetLastError();
    });
    return fn;
}

// row-major [rows, cols] matrix, box of box_c columns x box_r rows
bool encode_map(CUtensorMap *m, CUtensorMapDataType dt, uint32_t esize, const void *ptr, int64_t rows,
                int64_t cols, uint32_t box_c, uint32_t box_r, CUtensorMapSwizzle swizzle) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = tensor_map_encoder();
    if (!fn)
        return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * esize};
    const cuuint32_t box[2] = {box_c, box_r};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool rotate_fwd_tma_eligible(const RotateLaunch &p) {
    auto al16 = [](const void *q) { return ((uintptr_t)q & 15u) == 0; };
    return !p.inverse && p.src == SRC_BF16 && !p.ref && p.out && al16(p.in) && al16(p.out) &&
           al16(p.sv) && al16(p.su) && p.rows % 128 == 0 && p.cols % 128 == 0 && p.rows < (1ll << 30) &&
           p.cols < (1ll << 30) && tensor_map_encoder() != nullptr;
}

// EXL3_OK when launched; EXL3_ERR_UNSUPPORTED when a tensor map cannot be
// encoded for these pointers (the caller then uses rotate_fwd_kernel).
exl3_status launch_rotate_fwd_tma(const RotateLaunch &p, cudaStream_t s) {
    const int64_t nblk = (p.rows / 128) * (p.cols / 128);
    if (nblk == 0)
        return EXL3_OK;
    CUtensorMap in_map, out_map;
    if (!encode_map(&in_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.in, p.rows, p.cols, 64, 128,
                    CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_map(&out_map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, p.out, p.rows, p.cols, 128, 128,
                    CU_TENSOR_MAP_SWIZZLE_NONE))
        return EXL3_ERR_UNSUPPORTED;
    const size_t smem = kSmemBytes + 1024;   // + alignment slack
    cudaError_t e = cudaFuncSetAttribute(rotate_fwd_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess)
        return cuda_check(e, "cudaFuncSetAttribute(rotate_fwd_tma)");
    const int64_t slots = 2 * (int64_t)device_sm_count();     // two blocks per SM
    const int64_t grid = nblk < slots ? nblk : slots;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kTmaThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const float *su_ = p.su, *sv_ = p.sv;
    int rows_ = (int)p.rows, cols_ = (int)p.cols;
    double *ts_ = p.tile_sums;
    e = cudaLaunchKernelEx(&cfg, rotate_fwd_tma_kernel, in_map, out_map, su_, sv_, rows_, cols_, ts_);
    if (e != cudaSuccess)
        return cuda_check(e, "rotate_fwd_tma launch");
    note_launch();
    note_rotate_kernel(1);
    return cuda_check(cudaGetLastError(), "rotate_fwd_tma launch");
}

exl3_status rot_take_wait_timeouts(unsigned int *n) {
    *n = 0;
    unsigned int v = 0;
    const unsigned int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_rot_wait_timeouts, sizeof v);
    if (e == cudaSuccess && v != 0)
        e = cudaMemcpyToSymbol(g_rot_wait_timeouts, &zero, sizeof zero);
    if (e != cudaSuccess)
        return cuda_check(e, "wait timeout count");
    *n = v;
    return EXL3_OK;
}

}  // namespace exl3
