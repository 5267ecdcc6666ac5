// common.cuh -- shared definitions for the libexl3 CUDA kernels (sm_103a).
//
// Everything on the encode/decode/rotation path is IEEE binary32 with
// round-to-nearest and no contraction: the library is compiled with
// -fmad=false and the hot arithmetic uses the explicit __f*_rn intrinsics.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/exl3.h"

namespace exl3 {

// ---------------------------------------------------------------------------
// mul1 codebook (page "EXL3 Intel Arc Quantizer", Core Implemented
// Architecture item 5: a procedural codebook with fp16 levels).  The
// multiplier and scale are this library's reading of that passage:
//   v(s) = fp16_rn( fl32( (bytesum(u32(s * 0x9E3779B1)) - 510) * c ) ),
//   c = fl32(1 / 147.9146802...), the inverse population standard deviation
//   of that byte sum over the 65536 states.
// ---------------------------------------------------------------------------
constexpr uint32_t kMul1Mult = 0x9E3779B1u;
constexpr float kMul1C = 0x1.bb10f4p-8f;

__host__ __device__ __forceinline__ int mul1_bytesum(uint32_t state) {
    uint32_t x = state * kMul1Mult;
    return (int)(x & 0xFFu) + (int)((x >> 8) & 0xFFu) + (int)((x >> 16) & 0xFFu) +
           (int)(x >> 24);
}

__device__ __forceinline__ __half mul1_half(uint32_t state) {
    float f = __fmul_rn((float)(mul1_bytesum(state) - 510), kMul1C);
    return __float2half_rn(f);
}

__device__ __forceinline__ float mul1_value(uint32_t state) {
    return __half2float(mul1_half(state));
}

// 16-bit window of a tile's circular code stream ending with the last bit of
// code i (stream bits [(i+1)K - 16, (i+1)K) modulo 256K, MSB first).
template <int K>
__device__ __forceinline__ uint32_t window_state(const uint32_t *w, int i) {
    constexpr int NB = 256 * K;
    constexpr int NW = 8 * K;
    int p = (i + 1) * K - 16;
    if (p < 0)
        p += NB;
    const int wi = p >> 5;
    const int wj = (wi + 1 == NW) ? 0 : wi + 1;
    const unsigned long long cat = ((unsigned long long)w[wi] << 32) | w[wj];
    return (uint32_t)(cat >> (48 - (p & 31))) & 0xFFFFu;
}

__device__ __forceinline__ uint32_t window_state_k(const uint32_t *w, int i, int K) {
    switch (K) {
    case 1: return window_state<1>(w, i);
    case 2: return window_state<2>(w, i);
    case 3: return window_state<3>(w, i);
    default: return window_state<4>(w, i);
    }
}

// ---------------------------------------------------------------------------
// Trellis geometry for K bits per step on the 16-bit bitshift trellis.
//   tracked row:   G = 2^(16-K) entries, index g = low 16-K bits of a state
//   candidates:    sigma_k = (k << (16-K)) | g,  k in [0, 2^K)
//   predecessor:   sigma_k >> K = (k << (16-2K)) | (g >> K)
// A "unit" h' = g >> K groups the 2^K tracked entries g = (h' << K) | j that
// read the same 2^K predecessor costs M((k << (16-2K)) | h').  Each of the
// 512 threads of an encode block owns 128 candidate states:
//   K=2: 8 units x 4 groups x 4 candidates   (units h' = u*512 + tid)
//   K=3: 2 units x 8 groups x 8 candidates   (units h' = u*512 + tid)
//   K=4: 1/2 unit: 8 groups x 16 candidates  (unit h' = tid >> 1,
//                                             groups 8*(tid & 1) .. +7)
// The K-bit decisions of a thread's entries fill UPW units per 32-bit word
// (K=2: 4, K=3: 1, K=4: 1), DW words per thread and step (2, 2, 1).
// ---------------------------------------------------------------------------
// Encode block size (K >= 2): 512 threads x 128 candidate states, up to 128
// registers each (1024 x 64 at 64 registers measured 3 % slower at K=2, 12 %
// at K=4).
constexpr int kThreads = 512;

template <int K>
struct Geo {
    static constexpr int KR = 16 - K;
    static constexpr int NK = 1 << K;
    static constexpr int G = 1 << KR;
    static constexpr int UNITS = 1 << (16 - 2 * K);
    static constexpr int NU = UNITS >= kThreads ? UNITS / kThreads : 1;  // units per thread
    static constexpr int TPU = UNITS >= kThreads ? 1 : kThreads / UNITS; // threads per unit
    static constexpr int NJ = NK / TPU;                                  // groups per thread-unit
    static constexpr int STATES = NU * NJ * NK;                          // candidate states per thread
    static constexpr int UPW = 32 / (NJ * K);                            // units per decision word
    static constexpr int DW = (NU + UPW - 1) / UPW;                      // decision words per thread
    static_assert(STATES * kThreads == 65536, "the threads own all 2^16 candidate states");
    static_assert(UPW >= 1, "a unit's decisions fit one 32-bit word");

    __device__ __forceinline__ static int unit(int u, int tid) {
        return TPU == 1 ? u * kThreads + tid : (tid / TPU);
    }
    __device__ __forceinline__ static int j0(int tid) {
        return TPU == 1 ? 0 : (tid % TPU) * NJ;
    }
    // Bit of entry j (0..NJ-1 of the thread's share) of unit u in decision word u / UPW.
    __host__ __device__ __forceinline__ static constexpr int dec_bit(int u, int j) {
        return ((u % UPW) * NJ + j) * K;
    }
    // Location of D_t(g) inside a decision row: (word index, bit position).
    // Word w of thread tid is row word tid + w * kThreads.
    __host__ __device__ __forceinline__ static void dec_locate(uint32_t g, int &word, int &bit) {
        uint32_t hp = g >> K;
        uint32_t j = g & (NK - 1);
        if (TPU == 1) {
            const int tid = (int)(hp % kThreads);
            const int u = (int)(hp / kThreads);
            word = tid + kThreads * (u / UPW);
            bit = dec_bit(u, (int)j);
        } else {
            word = (int)(hp * TPU + j / NJ);
            bit = (int)(j % NJ) * K;
        }
    }
};

// Decision rows: 1024 32-bit words per step (4 KiB per row); an encode thread
// writes words tid + w * kThreads, w < Geo<K>::DW.
constexpr int kRowWords = 1024;
constexpr int kRowsPass1 = 128;   // steps 127..254 of the rolled pass
constexpr int kRowsPass2 = 255;   // steps 0..254 of the constrained pass
constexpr size_t kEncodeBlockScratchBytes =
    (size_t)2 * (kRowsPass1 + kRowsPass2) * kRowWords * sizeof(uint32_t);

// ---------------------------------------------------------------------------
// host-side helpers
// ---------------------------------------------------------------------------
exl3_status set_error(exl3_status st, const char *fmt, ...);
exl3_status cuda_check(cudaError_t e, const char *what);
int device_sm_count();

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// launch accounting for exl3_profile_* (abi.cu)
void note_launch();
// records which kernel a rotation launched: 1 TMA forward, 2 shared-memory
// forward, 3 warp-shuffle (inverse, decode-fused or unaligned)
void note_rotate_kernel(int which);
int last_rotate_kernel();
void profile_encode_begin(cudaStream_t s);
void profile_encode_end(cudaStream_t s);

// internal launchers (no argument checks; the ABI layer checks)
struct EncodeLaunch {
    const float *Y;
    int64_t rows, cols;
    int K;
    int T;                       // steps per tile (256 for 16x16 tiles)
    int row_tiles;               // 0: 16x16 tiles of Y[rows, cols]; 1: each row of Y[rows, T] is a tile
    float inv_scale;             // used when inv_scale_dev == nullptr
    const float *inv_scale_dev;  // device scalar or nullptr
    uint32_t *codes;             // [n_tiles][8K] uint32
    float *tile_cost;            // nullable
    uint32_t *scratch;           // grid * kEncodeBlockScratchBytes
    int grid;
    // tiles coded: n_work tiles (0: all) from tile tile0 on; with ring > 0 the
    // tile index wraps at ring (the matrix's tile count); codes and costs go to
    // the tiles' own positions
    int tile0;
    int n_work;
    int ring;
};
exl3_status launch_encode(const EncodeLaunch &p, cudaStream_t s);
// same launch without the profiling hooks (creates no CUDA events)
exl3_status launch_encode_unprofiled(const EncodeLaunch &p, cudaStream_t s);

exl3_status launch_decode(const uint32_t *codes, int64_t rows, int64_t cols, int K,
                          float scale, const float *scale_dev, float *out, cudaStream_t s);
exl3_status launch_decode_rows(const uint32_t *codes, int64_t n_rows, int T, int K, float scale,
                               float *out, cudaStream_t s);

// rotation modes
enum RotSrc { SRC_F32 = 0, SRC_BF16 = 1, SRC_CODES = 2 };
struct RotateLaunch {
    int inverse;
    int src;                  // RotSrc
    const void *in;           // fp32/bf16 matrix or uint32 codes
    int K;                    // SRC_CODES only
    const float *scale_dev;   // SRC_CODES only: decode scale (device)
    const float *su, *sv;
    int64_t rows, cols;
    float *out;               // nullable: skip the store
    const void *ref;          // nullable: per-tile fp64 sum of (ref - out)^2
    int ref_dt;
    double *tile_sums;        // per-tile sums: of out^2 (ref == null) or of (ref-out)^2
};
exl3_status launch_rotate(const RotateLaunch &p, cudaStream_t s);
// forward path without lane exchanges (rotate_fwd.cu): fp32/bf16 source, no ref,
// 16-byte aligned in / sv / out; launch_rotate picks it when eligible
bool rotate_fwd_eligible(const RotateLaunch &p);
exl3_status launch_rotate_fwd(const RotateLaunch &p, cudaStream_t s);
// the same with TMA staging (rotate_fwd_tma.cu): bf16 source, fp32 output, 16-byte
// aligned; EXL3_ERR_UNSUPPORTED when no tensor map can be encoded for the pointers
bool rotate_fwd_tma_eligible(const RotateLaunch &p);
exl3_status launch_rotate_fwd_tma(const RotateLaunch &p, cudaStream_t s);
// reads and clears the TMA rotation's expired-wait count (no synchronisation)
exl3_status rot_take_wait_timeouts(unsigned int *n);

// grid-and-parabola scale search (scale_search.cu)
struct GridSearchLaunch {
    const void *W;
    int dt;
    int64_t rows, cols;
    const float *su, *sv;
    int K;
    float *R;               // [rows, cols]
    double *tile_sums;      // [n_tiles]
    double *tree_scr;       // tree_scratch_doubles(n_tiles)
    double *sum, *sigma;    // scalars
    int *extremes;          // [2]
    int *sample;            // [sample_max]
    int *count;             // [1]
    double *state;          // [grid_search_state_doubles()]
    float *rows_buf;        // [max_rows, 256]
    uint32_t *codes_buf;    // [max_rows, 8K]
    double *row_sum;        // [max_rows]
    float *s_per_g;         // [19]
    uint32_t *enc;          // encode scratch, grid blocks
    int grid;
    double *g_out;
    float *scale_out;       // nullable
    double *history;        // nullable, [2 * 27]
};
size_t grid_search_sample_max(int64_t rows, int64_t cols);
size_t grid_search_state_doubles();
int grid_search_max_rows(int64_t rows, int64_t cols);
exl3_status run_grid_search(const GridSearchLaunch &p, cudaStream_t s);

// block LDL and LDLQ (ldlq.cu)
struct BlockLdlLaunch {
    const double *H;        // [n, n], lower triangle read
    int64_t n;
    double sigma_reg;
    int max_retries;
    float *M;               // [n, n] out
    int *retries_out;       // host, nullable
    double *A;              // [n, n] work (lower triangle)
    double *LD;             // [n / 16, 16, 16] diagonal blocks of L
    double *delta;          // scalar
    int *flag;              // device pivot-failure flag
};
exl3_status run_block_ldl(const BlockLdlLaunch &p, cudaStream_t s);

struct LdlqLaunch {
    const float *R;         // [rows, cols]
    int64_t rows, cols;
    const float *M;         // [rows, rows]
    int K;
    float scale;
    uint32_t *codes;        // [rows/16, cols/16, 8K words]
    float *Q;               // nullable [rows, cols]
    float *acc;             // [rows, cols]
    float *U;               // [2][16, cols]: targets of two span rows (a ring)
    float *E;               // [cols / 16][256]: errors of one launch's tiles
    uint32_t *ring;         // [2][cols / 16][8K words]: codes of two span rows
    uint32_t *enc;          // encode scratch, grid blocks
    int grid;
};
exl3_status run_ldlq(const LdlqLaunch &p, cudaStream_t s);

// output-channel regularisation (regularize.cu)
struct RegularizeLaunch {
    const void *W;
    int dt;
    int64_t rows, cols;
    const float *h;         // [rows]
    const float *sv;        // [cols]
    int apply_out;          // -1 heuristic, 0 / 1 forced
    float *W_out;           // [rows, cols]
    float *sv_out;          // [cols]
    double *info_out;       // nullable, [4]
    double *part;           // [32, cols]
    double *S;              // [cols]
    double *tree_scr;       // tree_scratch_doubles(max(rows, cols))
    double *total;          // scalar
    double *sortbuf;        // [regularize_sort_len(rows)]
    double *hsum;           // [2]: trees of the top sqrt(h) and of all
    double *info;           // [4]
    float *g_rms;           // scalar
    float *scale;           // [cols]
};
int64_t regularize_sort_len(int64_t rows);
exl3_status run_regularize(const RegularizeLaunch &p, cudaStream_t s);

exl3_status launch_tile_sumsq(const void *x, int x_dt, const float *ref, int64_t rows,
                              int64_t cols, double *tile_sums, cudaStream_t s);
// tree sum of n doubles; scratch >= tree_scratch_doubles(n) doubles; result -> *out
size_t tree_scratch_doubles(int64_t n);
exl3_status launch_tree_sum(const double *in, int64_t n, double *scratch, double *out,
                            cudaStream_t s);

}  // namespace exl3
