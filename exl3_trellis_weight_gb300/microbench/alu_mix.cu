// alu_mix.cu -- issue rate of the instruction kinds the trellis encoder uses,
// per SM per clock, on the running GPU.  One 1024-thread block per SM, eight
// independent dependency chains per thread, operands that change every
// iteration (so no chain can be hoisted or folded), cycles from clock64().
//
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 alu_mix.cu -o alu_mix
#include <cuda_fp16.h>
#include <cstdio>
#include <cstdint>

#define ITERS 2048

__device__ __forceinline__ float sub_h_f(unsigned short h, float y) {
    float r;
    asm volatile("sub.rn.f32.f16 %0, %1, %2;" : "=f"(r) : "h"(h), "f"(y));
    return r;
}
__device__ __forceinline__ unsigned long long mul2(unsigned long long a, unsigned long long b) {
    unsigned long long r;
    asm volatile("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ unsigned long long add2(unsigned long long a, unsigned long long b) {
    unsigned long long r;
    asm volatile("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

template <int KIND>
__global__ void __launch_bounds__(1024, 1) kern(const int *in, unsigned *out, unsigned long long *cyc) {
    // per-chain operands, unknown to the compiler and loop-invariant (no
    // per-iteration operand arithmetic in the timed loop)
    int x[8], op[8];
    float f[8], fo[8];
    unsigned b[8];
    unsigned long long u[8], uo[8];
    unsigned short h[8];
    const int t = threadIdx.x;
    for (int i = 0; i < 8; i++) {
        x[i] = in[(t + i) & 15];
        op[i] = in[(t + 3 * i + 1) & 15];
        f[i] = __int_as_float((x[i] & 0x0fffffff) | 0x30000000);
        fo[i] = __int_as_float((op[i] & 0x0fffffff) | 0x20000000);
        b[i] = (unsigned)x[i];
        u[i] = ((unsigned long long)(unsigned)x[i] << 32) | (unsigned)(x[i] + 7);
        uo[i] = ((unsigned long long)(unsigned)op[i] << 32) | (unsigned)(op[i] + 9);
        h[i] = (unsigned short)(op[i] >> 3);
    }
    __syncthreads();
    const unsigned long long c0 = clock64();
    // the trip count depends on c0 and every result is consumed before c1, so
    // the compiler cannot move work out of the timed region
    int n = ITERS;
    asm volatile("" : "+r"(n) : "l"(c0));
#pragma unroll 4
    for (int it = 0; it < n; it++) {
#pragma unroll
        for (int i = 0; i < 8; i++) {
            if (KIND == 0) f[i] = __fadd_rn(f[i], fo[i]);
            if (KIND == 1) u[i] = mul2(u[i], uo[i]);
            if (KIND == 2) u[i] = add2(u[i], uo[i]);
            if (KIND == 3) f[i] = sub_h_f(h[i], f[i]);
            if (KIND == 4) x[i] = min(x[i] + op[i], op[i ^ 1]);                       // iadd + imnmx
            if (KIND == 5) f[i] = fminf(__fadd_rn(f[i], fo[i]), fo[i ^ 1]);           // fadd + fmnmx
            if (KIND == 6) { bool p; x[i] = __vibmin_s32(x[i] + op[i], op[i ^ 1], &p); b[i] = p ? b[i] : (unsigned)x[i]; } // iadd + dpx min + select
            if (KIND == 7) { const bool p = f[i] < fo[i]; b[i] = p ? b[i] : (unsigned)i; f[i] = __fadd_rn(f[i], fo[i ^ 1]); } // compare + select + fadd
            if (KIND == 8) b[i] = b[i] * (unsigned)op[i] + (unsigned)op[i ^ 1];
            if (KIND == 10) b[i] = __byte_perm(b[i], (unsigned)op[i], 0x5410);
            if (KIND == 11) f[i] = fminf(fminf(__fadd_rn(f[i], fo[i]), fo[i ^ 1]), fo[i ^ 2]);  // fadd + 2 fmnmx
            if (KIND == 15) {                                                             // fadd + fsetp + fmnmx + sel
                const float v = __fadd_rn(f[i], fo[i]);
                const bool p = v < fo[i ^ 1];
                f[i] = fminf(v, fo[i ^ 1]);
                b[i] = p ? (unsigned)i : b[i];
            }
        }
    }
    unsigned acc = 0;
    for (int i = 0; i < 8; i++)
        acc ^= (unsigned)x[i] ^ __float_as_uint(f[i]) ^ b[i] ^ (unsigned)u[i] ^ (unsigned)(u[i] >> 32);
    asm volatile("" : "+r"(acc));
    const unsigned long long c1 = clock64();
    out[blockIdx.x * 1024 + t] = acc;
    if (t == 0)
        cyc[blockIdx.x] = c1 - c0;
}

template <int KIND>
static void run(const char *name, int per_iter, int sms, const int *din, unsigned *dout,
                unsigned long long *dcyc) {
    kern<KIND><<<sms, 1024>>>(din, dout, dcyc);
    cudaDeviceSynchronize();
    kern<KIND><<<sms, 1024>>>(din, dout, dcyc);
    const cudaError_t e = cudaDeviceSynchronize();
    unsigned long long cyc[4096];
    cudaMemcpy(cyc, dcyc, (size_t)sms * 8, cudaMemcpyDeviceToHost);
    double mean = 0;
    for (int i = 0; i < sms; i++)
        mean += (double)cyc[i];
    mean /= sms;
    const double bodies = 1024.0 * ITERS * 8 / mean;   // includes the short epilogue
    printf("%-34s %-8s %7.1f bodies/clk/SM  (%d instr per body: %6.1f thread-instr/clk/SM)\n", name,
           e == cudaSuccess ? "ok" : cudaGetErrorString(e), bodies, per_iter, bodies * per_iter);
}

int main() {
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
    if (sms <= 0 || sms > 4096) {
        printf("no device\n");
        return 1;
    }
    int hin[16];
    for (int i = 0; i < 16; i++)
        hin[i] = 0x12345 * (i + 1);
    int *din;
    unsigned *dout;
    unsigned long long *dcyc;
    cudaMalloc(&din, sizeof(hin));
    cudaMalloc(&dout, (size_t)sms * 1024 * 4);
    cudaMalloc(&dcyc, (size_t)sms * 8);
    cudaMemcpy(din, hin, sizeof(hin), cudaMemcpyHostToDevice);
    printf("SMs: %d; issue limit 128 thread-instr/clk/SM\n", sms);
    run<0>("FADD (fp32 add)", 1, sms, din, dout, dcyc);
    run<1>("mul.rn.f32x2", 1, sms, din, dout, dcyc);
    run<2>("add.rn.f32x2", 1, sms, din, dout, dcyc);
    run<3>("sub.rn.f32.f16 (mixed)", 1, sms, din, dout, dcyc);
    run<4>("int add + int min", 2, sms, din, dout, dcyc);
    run<5>("fp32 add + fp32 min", 2, sms, din, dout, dcyc);
    run<6>("int add + DPX min-pred + select", 3, sms, din, dout, dcyc);
    run<7>("fp32 compare + select + fp32 add", 3, sms, din, dout, dcyc);
    run<8>("integer multiply-add", 1, sms, din, dout, dcyc);
    run<10>("byte permute", 1, sms, din, dout, dcyc);
    // fp32 min: 42.7 bodies/clk if it issues to the FMA pipe (3 FMA-pipe instructions),
    // 32 if to the 64-lane ALU pipe (2 ALU slots)
    run<11>("fp32 add + 2 fp32 min", 3, sms, din, dout, dcyc);
    // 32 bodies/clk if fp32 min is on the FMA pipe (compare + select = 2 ALU slots), 21.3 if on the ALU
    run<15>("fp32 add + compare + min + select", 4, sms, din, dout, dcyc);
    cudaFree(din);
    cudaFree(dout);
    cudaFree(dcyc);
    return 0;
}
