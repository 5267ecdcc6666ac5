// encode_common.cuh -- device helpers of the trellis encode kernels (encode.cu).
#pragma once

#include "common.cuh"

namespace exl3 {
namespace {


template <int K>
__device__ __forceinline__ void put_code(uint32_t *bs, int t, uint32_t e) {
    const int p = t * K;
    const int w = p >> 5;
    const int sh = 32 - K - (p & 31);
    if (sh >= 0) {
        bs[w] |= e << sh;
    } else {
        bs[w] |= e >> (-sh);
        bs[w + 1] |= e << (32 + sh);
    }
}

__device__ __forceinline__ unsigned long long warp_min_u64(unsigned long long v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
        v = w < v ? w : v;
    }
    return v;
}

// Two candidates: fl(m + fl(fl(v - y)^2)) for the two fp16 levels packed in vw
// and the two predecessor costs packed in mm, as one 64-bit pair.  The two
// mixed-precision subtracts (exact widening of v, one binary32 rounding) write
// the halves of a 64-bit operand; the square is a packed FMA with a +0 addend --
// exactly fl(d*d), since d*d is never -0 -- and the add is packed too.  A plain
// packed multiply would not do: the compiler contracts a packed multiply feeding
// a packed add into a fused multiply-add whatever the rounding qualifiers, and a
// fused result differs from the two-rounding definition (measured: 3.4 % of
// random candidates; none with the FMA form).
__device__ __forceinline__ unsigned long long cand2(const uint32_t vw, const float y,
                                                    const unsigned long long mm) {
    unsigned long long c;
    asm("{\n\t.reg .b16 hl, hh;\n\t.reg .f32 a, b;\n\t.reg .b64 d, q, z;\n\t"
        "mov.b32 {hl, hh}, %1;\n\t"
        "sub.rn.f32.f16 a, hl, %2;\n\t"
        "sub.rn.f32.f16 b, hh, %2;\n\t"
        "mov.b64 d, {a, b};\n\t"
        "mov.b64 z, 0;\n\t"
        "fma.rn.f32x2 q, d, d, z;\n\t"
        "add.rn.f32x2 %0, %3, q;\n\t}"
        : "=l"(c) : "r"(vw), "f"(y), "l"(mm));
    return c;
}

__device__ __forceinline__ unsigned long long pack_costs(const float lo, const float hi) {
    return (unsigned long long)__float_as_uint(lo) | ((unsigned long long)__float_as_uint(hi) << 32);
}

// Candidate k of two entries (predecessor costs packed in mm), then the running
// minima (ties keep the lower k).
__device__ __forceinline__ void acs2(const unsigned long long mm, const uint32_t vw, const float y,
                                     const int k, int &best0, int &best1, uint32_t &bk0,
                                     uint32_t &bk1) {
    const unsigned long long c = cand2(vw, y, mm);
    const int c0 = (int)(uint32_t)(c & 0xffffffffull), c1 = (int)(uint32_t)(c >> 32);
    if (k == 0) {
        best0 = c0;
        best1 = c1;
        bk0 = 0u;
        bk1 = 0u;
    } else {
        bool keep0, keep1;
        best0 = __vibmin_s32(best0, c0, &keep0);   // keep0: best0 <= c0
        best1 = __vibmin_s32(best1, c1, &keep1);
        bk0 = keep0 ? bk0 : (uint32_t)k;
        bk1 = keep1 ? bk1 : (uint32_t)k;
    }
}

template <int K, bool ARGMIN>
__device__ __forceinline__ void finish_pair(const int u, const int jp, const int hp, const int j0,
                                            const int best0, const int best1, const uint32_t bk0,
                                            const uint32_t bk1, float *outv,
                                            uint32_t (&word)[Geo<K>::DW],
                                            unsigned long long &key) {
    using Gm = Geo<K>;
    outv[jp] = __int_as_float(best0);
    outv[jp + 1] = __int_as_float(best1);
    word[u / Gm::UPW] |= (bk0 << Gm::dec_bit(u, jp)) | (bk1 << Gm::dec_bit(u, jp + 1));
    if (ARGMIN) {
        const uint32_t g0 = ((uint32_t)hp << K) | (uint32_t)(j0 + jp);
        const unsigned long long k0 =
            ((unsigned long long)(uint32_t)best0 << 32) | ((bk0 << Gm::KR) | g0);
        const unsigned long long k1 =
            ((unsigned long long)(uint32_t)best1 << 32) | ((bk1 << Gm::KR) | (g0 + 1u));
        key = k0 < key ? k0 : key;
        key = k1 < key ? k1 : key;
    }
}

struct Tb {          // traceback state, kept in shared memory, used by thread 0 only
    const uint32_t *rows;
    int tile;
    uint32_t s;       // full state at step t
    uint32_t pending; // decision word in flight
    int t, stop, row0, pass, slot;
    bool on;
};

}  // namespace
}  // namespace exl3
