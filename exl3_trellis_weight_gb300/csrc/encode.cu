// encode.cu -- persistent trellis tile encoder (page "EXL3 Intel Arc
// Quantizer", Core Implemented Architecture items 1, 4 and 5).
//
// One 512-thread block per SM walks its share of the tiles (K = 1, 2 here; K =
// 3, 4 in encode2_kernel below, two tiles at a time).  A tile is T
// targets: the 256 elements of a 16x16 tile (row-major), or one row of T
// elements (even T in [16, 256]).  For each tile:
//   pass 1: targets rolled left by T/2, free start, T add-compare-select
//           steps; decisions of steps T/2-1..T-2 are kept; the lowest-index
//           minimal final state is traced back to step T/2-1 -> end_state.
//   pass 2: unrolled targets, first predecessor fixed to end_state, T-1 steps
//           (the last step of the constrained pass is never needed: its path
//           is forced to end at end_state); traced back from end_state; the
//           low K bits of each state are packed MSB first.
//
// The tracked cost row M (2^(16-K) fp32) is double-buffered in shared memory
// (K = 1: one row, updated in place; see acs_step_k1);
// the mul1 level of each of a thread's 128 candidate states is fixed for the
// whole launch and is kept in registers as packed fp16.  Decisions (K bits per
// tracked entry per step, one or two 32-bit words per thread per step) go to
// the block's slice of the workspace.
//
// The traceback is a chain of dependent loads, so it is overlapped with the
// forward pass of another tile: the block keeps two tiles A and B in flight
// and cycles through four phases
//     fwd1(A) | tb2(prev B);  fwd1(B) | tb1(A);  fwd2(A) | tb1(B);  fwd2(B) | tb2(A)
// where thread 0 performs one traceback step per forward step, issuing the
// load at the start of the step and consuming it at the end.
//
// At K = 3 and 4 the cost rows of two tiles fit one SM's shared memory, and
// encode2_kernel runs the same pipeline on pairs of tiles: every barrier
// interval holds the step of both tiles of a pair (6-7 % faster than one tile
// per interval on 4096 x 4096), with the decision rows packed so that the two
// pairs in flight use the same per-block workspace slice.
//
// A traceback with no forward pass beside it (a block's last tile, launches of
// one tile or pair per block) reads its rows from shared memory, streamed in
// ahead by its warp (tb_drain_streamed).  A launch may code a run of tiles
// from an offset, wrapping over the matrix (tile_at), as LDLQ does.
#include "encode_common.cuh"

namespace exl3 {

namespace {
// One add-compare-select step of a thread's units.  The NK predecessor costs of
// a unit are loaded once and each is duplicated into both halves of a 64-bit
// register pair; the entries are taken a pair at a time, so every candidate
// pair is one packed square (an FMA with a +0 addend) and one packed add.
// Measured against the alternatives at 512 threads: scalar adds 4-6 % slower
// (K=2..4); pairing the same (k, j) of two units instead of two entries of one
// unit (the two costs then load straight into a pair) 1-9 % slower; reloading
// the cost for every entry pair the same speed; keeping all running minima
// live while the costs stream 6 % slower at K=2 and 77 % at K=4.
template <int K, bool ARGMIN>
__device__ __forceinline__ void acs_step(const float *__restrict__ Mp, float *__restrict__ Mn,
                                         const float y, const uint32_t (&vpk)[Geo<K>::STATES / 2],
                                         const int tid, uint32_t (&word)[Geo<K>::DW],
                                         unsigned long long &key) {
    using Gm = Geo<K>;
#pragma unroll
    for (int w = 0; w < Gm::DW; w++)
        word[w] = 0u;
#pragma unroll
    for (int u = 0; u < Gm::NU; u++) {
        const int hp = Gm::unit(u, tid);
        const int j0 = Gm::j0(tid);
        float outv[Gm::NJ];
        unsigned long long mm[Gm::NK];
#pragma unroll
        for (int k = 0; k < Gm::NK; k++) {
            const float m = Mp[(k << (16 - 2 * K)) + hp];
            mm[k] = pack_costs(m, m);
        }
#pragma unroll
        for (int jp = 0; jp < Gm::NJ; jp += 2) {
            int best0 = 0, best1 = 0;
            uint32_t bk0 = 0u, bk1 = 0u;
#pragma unroll
            for (int k = 0; k < Gm::NK; k++)
                acs2(mm[k], vpk[((u * Gm::NK + k) * Gm::NJ + jp) >> 1], y, k, best0, best1, bk0, bk1);
            finish_pair<K, ARGMIN>(u, jp, hp, j0, best0, best1, bk0, bk1, outv, word, key);
        }
        if (!ARGMIN) {
            float *dst = Mn + (hp << K) + j0;
#pragma unroll
            for (int q = 0; q < Gm::NJ; q += 4)
                *reinterpret_cast<float4 *>(dst + q) =
                    make_float4(outv[q], outv[q + 1], outv[q + 2], outv[q + 3]);
        }
    }
}

// Candidates of one entry pair (two entries j, j + 1 of one unit) for the NK
// predecessors: c[k] = fl(M(k) + fl(fl(v - y)^2)), two packed per 64 bits.
template <int K>
__device__ __forceinline__ void cands_pair(const unsigned long long (&mm)[1 << K], const uint32_t *vp,
                                           const float y, unsigned long long (&c)[1 << K]) {
#pragma unroll
    for (int k = 0; k < (1 << K); k++)
        c[k] = cand2(vp[k * (Geo<K>::NJ / 2)], y, mm[k]);
}

// Running minimum over k with the lowest k on ties, as a balanced tournament
// (pairs (0,1), (2,3), ... then their winners): the same result as the
// sequential scan, with log2 NK dependent levels instead of NK - 1.
template <int K>
__device__ __forceinline__ void tour_pair(const unsigned long long (&c)[1 << K], int &best0, int &best1,
                                          uint32_t &bk0, uint32_t &bk1) {
    constexpr int NK = 1 << K;
    int v0[NK], v1[NK];
    uint32_t i0[NK], i1[NK];
#pragma unroll
    for (int k = 0; k < NK; k++) {
        v0[k] = (int)(uint32_t)(c[k] & 0xffffffffull);
        v1[k] = (int)(uint32_t)(c[k] >> 32);
        i0[k] = (uint32_t)k;
        i1[k] = (uint32_t)k;
    }
#pragma unroll
    for (int w = 1; w < NK; w <<= 1) {
#pragma unroll
        for (int k = 0; k < NK; k += 2 * w) {
            bool keep0, keep1;      // keep: the lower group is no worse
            v0[k] = __vibmin_s32(v0[k], v0[k + w], &keep0);
            v1[k] = __vibmin_s32(v1[k], v1[k + w], &keep1);
            i0[k] = keep0 ? i0[k] : i0[k + w];
            i1[k] = keep1 ? i1[k] : i1[k + w];
        }
    }
    best0 = v0[0];
    best1 = v1[0];
    bk0 = i0[0];
    bk1 = i1[0];
}
// The single-tile kernel's step (K = 2): the same candidates and results as
// acs_step, with two changes that measured 8.7 % faster at 4096 x 4096
// (384.6 -> 351.3 ms): the minimum over k is a balanced tournament (lowest k
// on ties, like the scan, with log2 NK dependent levels instead of NK - 1), and
// the candidates of the next entry pair are formed before the current pair's
// comparisons.  At K = 3 and 4 the same form spilled and ran slower.
template <int K, bool ARGMIN>
__device__ __forceinline__ void acs_step_sp(const float *__restrict__ Mp, float *__restrict__ Mn,
                                         const float y, const uint32_t (&vpk)[Geo<K>::STATES / 2],
                                         const int tid, uint32_t (&word)[Geo<K>::DW],
                                         unsigned long long &key) {
    using Gm = Geo<K>;
    constexpr int NP = Gm::NJ / 2;                 // entry pairs per unit
    constexpr int NE = Gm::NU * NP;                // entry pairs per thread
#pragma unroll
    for (int w = 0; w < Gm::DW; w++)
        word[w] = 0u;
    const int j0 = Gm::j0(tid);
    unsigned long long mm[Gm::NK];
#pragma unroll
    for (int k = 0; k < Gm::NK; k++) {
        const float m = Mp[(k << (16 - 2 * K)) + Gm::unit(0, tid)];
        mm[k] = pack_costs(m, m);
    }
    // software pipeline: the candidates (loads, squares, adds) of entry pair
    // e + 1 are formed before the comparisons of entry pair e, so that each
    // warp's instruction stream alternates FMA-pipe and ALU-pipe work
    unsigned long long cn[Gm::NK];
    cands_pair<K>(mm, &vpk[0], y, cn);
    float outv[Gm::NJ];
#pragma unroll
    for (int e = 0; e < NE; e++) {
        const int u = e / NP, jp = 2 * (e % NP);
        const int hp = Gm::unit(u, tid);
        unsigned long long cc[Gm::NK];
#pragma unroll
        for (int k = 0; k < Gm::NK; k++)
            cc[k] = cn[k];
        if (e + 1 < NE) {
            const int u1 = (e + 1) / NP, jp1 = 2 * ((e + 1) % NP);
            if (jp1 == 0) {
#pragma unroll
                for (int k = 0; k < Gm::NK; k++) {
                    const float m = Mp[(k << (16 - 2 * K)) + Gm::unit(u1, tid)];
                    mm[k] = pack_costs(m, m);
                }
            }
            cands_pair<K>(mm, &vpk[((u1 * Gm::NK) * Gm::NJ + jp1) >> 1], y, cn);
        }
        int best0 = 0, best1 = 0;
        uint32_t bk0 = 0u, bk1 = 0u;
        tour_pair<K>(cc, best0, best1, bk0, bk1);
        finish_pair<K, ARGMIN>(u, jp, hp, j0, best0, best1, bk0, bk1, outv, word, key);
        if (!ARGMIN && jp + 2 == Gm::NJ) {
            float *dst = Mn + (hp << K) + j0;
#pragma unroll
            for (int q = 0; q < Gm::NJ; q += 4)
                *reinterpret_cast<float4 *>(dst + q) =
                    make_float4(outv[q], outv[q + 1], outv[q + 2], outv[q + 3]);
        }
    }
}

// ---------------------------------------------------------------------------
// K = 1: one block per tile, the 2^15-entry cost row updated in place in one
// buffer (two would not fit one SM).  Unit h (14 bits) owns the tracked
// entries 2h and 2h + 1; both read the predecessor costs M(h) (k = 0) and
// M(h | 2^14) (k = 1).  M_t(g) is kept at position f(rotr^(t+1)(g)), where rotr
// rotates the 15-bit index right by one and f(p) = p + (p >> 5) + (p >> 10):
// then f(rotr^(t+1)(2h)) = f(rotr^t(h)) and f(rotr^(t+1)(2h + 1)) =
// f(rotr^t(h | 2^14)), so the two new costs of unit h land exactly where its
// two predecessor costs were read.  Each position is read and rewritten by the
// one thread that owns it at that step, and one barrier per step orders the
// steps.  The padding f sends the 32 lanes of a warp (units differing in the
// five low bits, which the rotation moves to any five cyclically adjacent bit
// positions) to 32 distinct banks at every step; the row takes 33,822 floats.
// Thread tid owns units h = (i << 9) | tid, i < 32.  The positions split as
// f(rotr^s(tid)) + f(rotr^s(i << 9)) (+ f(rotr^s(2^14)) for k = 1), s = t mod
// 15, the middle term a sum of five per-step values; the units are walked in
// Gray-code order of i, so each unit's address is one add from the previous
// one's, and their loads are issued BATCH units at a time ahead of the
// comparisons.
// ---------------------------------------------------------------------------
constexpr int kK1RowFloats = 33822;   // f(2^15 - 1) + 1

__host__ __device__ __forceinline__ uint32_t rotr15(uint32_t x, int s) {
    return ((x >> s) | (x << (15 - s))) & 0x7FFFu;
}
__host__ __device__ __forceinline__ uint32_t k1_pad(uint32_t p) { return p + (p >> 5) + (p >> 10); }

// per-step values of acs_step_k1 for s = 0..14: the five Gray-walk steps
// k1_pad(rotr^s(2^(9+b))) and the k = 1 offset k1_pad(rotr^s(2^14))
struct K1Tab {
    uint32_t v[15][6];
};
constexpr K1Tab k1_make_tab() {
    K1Tab t{};
    for (int s = 0; s < 15; s++) {
        for (int b = 0; b < 6; b++) {
            const uint32_t x = 1u << (9 + b);
            const uint32_t r = ((x >> s) | (x << (15 - s))) & 0x7FFFu;
            t.v[s][b] = r + (r >> 5) + (r >> 10);
        }
    }
    return t;
}
__constant__ K1Tab k1_tab = k1_make_tab();

// D_t(g) of entry g (15 bits): thread h & 511 of unit h = g >> 1, word i >> 4,
// bit 2 (i & 15) + (g & 1), with i = h >> 9
__host__ __device__ __forceinline__ void k1_dec_locate(uint32_t g, int &word, int &bit) {
    const uint32_t h = g >> 1, i = h >> 9;
    word = (int)((h & 511u) + 512u * (i >> 4));
    bit = (int)(((i & 15u) << 1) | (g & 1u));
}

template <int K>
__device__ __forceinline__ void dec_loc(uint32_t g, int &w, int &b) {
    if constexpr (K == 1)
        k1_dec_locate(g, w, b);
    else
        Geo<K>::dec_locate(g, w, b);
}

// One step at K = 1 (s = t mod 15: M_{t-1}(x) sits at k1_pad(rotr^s(x))).
template <bool ARGMIN>
__device__ __forceinline__ void acs_step_k1(float *M, const float y, const uint32_t (&vpk)[64],
                                            const int tid, const int s, uint32_t (&word)[2],
                                            unsigned long long &key) {
    constexpr int BATCH = 4;
    word[0] = 0u;
    word[1] = 0u;
    const uint32_t E0 = k1_tab.v[s][0], E1 = k1_tab.v[s][1], E2 = k1_tab.v[s][2],
                   E3 = k1_tab.v[s][3], E4 = k1_tab.v[s][4], D = k1_tab.v[s][5];
    uint32_t a0 = k1_pad(rotr15((uint32_t)tid, s));
    // every position is read, then rewritten, by the one unit that owns it at
    // this step, and different units' positions never coincide: loads go
    // through Mr and stores through Mw so that a later unit's loads may move
    // above an earlier unit's stores (a unit's stores depend on its own loads)
    const float *__restrict__ Mr = M;
    float *__restrict__ Mw = M;
#pragma unroll
    for (int n0 = 0; n0 < 32; n0 += BATCH) {
        uint32_t ad0[BATCH], ad1[BATCH];
        float m0[BATCH], m1[BATCH];
#pragma unroll
        for (int q = 0; q < BATCH; q++) {
            const int n = n0 + q;
            const int i = n ^ (n >> 1);
            if (n > 0) {
                const int b = __ffs(n) - 1;          // the Gray-code bit that flips
                const uint32_t Eb = b == 0 ? E0 : b == 1 ? E1 : b == 2 ? E2 : b == 3 ? E3 : E4;
                if (i & (1 << b))
                    a0 += Eb;
                else
                    a0 -= Eb;
            }
            ad0[q] = a0;
            ad1[q] = a0 + D;
            m0[q] = Mr[ad0[q]];
            m1[q] = Mr[ad1[q]];
        }
#pragma unroll
        for (int q = 0; q < BATCH; q++) {
            const int n = n0 + q;
            const int i = n ^ (n >> 1);
            const unsigned long long c0 = cand2(vpk[2 * i], y, pack_costs(m0[q], m0[q]));
            const unsigned long long c1 = cand2(vpk[2 * i + 1], y, pack_costs(m1[q], m1[q]));
            bool keep0, keep1;   // keep: k = 0 is no worse (ties keep the lower k)
            const int b0 = __vibmin_s32((int)(uint32_t)(c0 & 0xffffffffull),
                                        (int)(uint32_t)(c1 & 0xffffffffull), &keep0);
            const int b1 = __vibmin_s32((int)(uint32_t)(c0 >> 32), (int)(uint32_t)(c1 >> 32), &keep1);
            const uint32_t bk0 = keep0 ? 0u : 1u, bk1 = keep1 ? 0u : 1u;
            word[i >> 4] |= (bk0 << ((i & 15) * 2)) | (bk1 << ((i & 15) * 2 + 1));
            if (ARGMIN) {
                const uint32_t g0 = 2u * (((uint32_t)i << 9) | (uint32_t)tid);
                const unsigned long long k0 =
                    ((unsigned long long)(uint32_t)b0 << 32) | ((bk0 << 15) | g0);
                const unsigned long long k1 =
                    ((unsigned long long)(uint32_t)b1 << 32) | ((bk1 << 15) | (g0 + 1u));
                key = k0 < key ? k0 : key;
                key = k1 < key ? k1 : key;
            } else {
                Mw[ad0[q]] = __int_as_float(b0);
                Mw[ad1[q]] = __int_as_float(b1);
            }
        }
    }
}

// Matrix tile of a block's l-th tile: the launch's tiles tile0, tile0 + 1, ...
// (wrapping at a.ring when that is set) are dealt to the blocks round-robin.  It
// reads only launch parameters, so nothing extra stays live through the forward
// loop (a wrap against a kept tile count cost 2.6 % at K=2).
__device__ __forceinline__ int tile_at(const EncodeLaunch &a, const int l, const int grid) {
    const int t = a.tile0 + (int)blockIdx.x + l * grid;
    return (a.ring > 0 && t >= a.ring) ? t - a.ring : t;
}

template <int K>
__device__ __forceinline__ void tb_issue(Tb &tb) {
    int w, b;
    dec_loc<K>(tb.s >> K, w, b);
    tb.pending = __ldcg(tb.rows + (size_t)(tb.t - 1 - tb.row0) * kRowWords + w);
}

template <int K>
__device__ __forceinline__ void tb_advance(Tb &tb, uint32_t *bs) {
    using Gm = Geo<K>;
    const uint32_t g = tb.s >> K;
    int w, b;
    dec_loc<K>(g, w, b);
    const uint32_t k = (tb.pending >> b) & (uint32_t)(Gm::NK - 1);
    tb.s = (k << Gm::KR) | g;
    tb.t -= 1;
    if (tb.pass == 2)
        put_code<K>(bs, tb.t, tb.s & (uint32_t)(Gm::NK - 1));
    if (tb.t == tb.stop)
        tb.on = false;
}

// ---------------------------------------------------------------------------
// A traceback with no forward pass beside it (a block's last tile, or launches
// of one tile per block, as in LDLQ) would expose its chain of dependent L2
// loads, about 0.4 us a step.  There warp 0 streams the decision rows t-1,
// t-2, ... into shared memory kTbAhead rows ahead (cp.async, 16 bytes a lane
// per copy, one commit group per row; the rows do not depend on the path) and
// lane 0 walks the chain from shared memory.
// ---------------------------------------------------------------------------
constexpr int kTbAhead = 16;
constexpr size_t kTbStreamBytes = (size_t)kTbAhead * kRowWords * sizeof(uint32_t);

__device__ __forceinline__ void tb_copy_row(uint32_t *dst, const uint32_t *src, const int lane) {
#pragma unroll
    for (int i = 0; i < kRowWords / 128; i++) {       // 8 x 16 bytes per lane
        const int c = (lane + 32 * i) * 4;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
                     ::"r"((uint32_t)__cvta_generic_to_shared(dst + c)), "l"(src + c) : "memory");
    }
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Called by all of warp 0; the traceback state is lane 0's.  Out of line: inlined
// into the kernel, its code changed the forward loop's and cost it 17 % at K=2.
template <int K>
__device__ __noinline__ Tb tb_drain_streamed(Tb tb, uint32_t *bs, uint32_t *pf, const int lane) {
    const unsigned long long rp = __shfl_sync(0xffffffffu, (unsigned long long)(uintptr_t)tb.rows, 0);
    const int t0 = __shfl_sync(0xffffffffu, tb.t, 0);
    const int n = t0 - __shfl_sync(0xffffffffu, tb.stop, 0);
    const int row0 = __shfl_sync(0xffffffffu, tb.row0, 0);
    // the row of the q-th step back is first - q rows
    const uint32_t *first = reinterpret_cast<const uint32_t *>((uintptr_t)rp) + (size_t)(t0 - 1 - row0) * kRowWords;
#pragma unroll 1
    for (int q = 0; q < kTbAhead; q++) {
        if (q < n)
            tb_copy_row(pf + q * kRowWords, first - (size_t)q * kRowWords, lane);
        cp_async_commit();
    }
#pragma unroll 1
    for (int q = 0; q < n; q++) {
        cp_async_wait<kTbAhead - 1>();      // this lane's copies of row q have landed
        __syncwarp();                       // and every lane's
        if (lane == 0) {
            int w, b;
            dec_loc<K>(tb.s >> K, w, b);
            tb.pending = pf[(q % kTbAhead) * kRowWords + w];
            tb_advance<K>(tb, bs);
        }
        __syncwarp();                       // the slot is read before it is refilled
        if (q + kTbAhead < n)
            tb_copy_row(pf + (q % kTbAhead) * kRowWords, first - (size_t)(q + kTbAhead) * kRowWords, lane);
        cp_async_commit();
    }
    cp_async_wait<0>();
    __syncwarp();
    return tb;
}

// TT: tile length fixed at compile time (256 for 16x16 tiles) or 0 (rows of
// a.T targets).
template <int K, int TT>
__global__ void __launch_bounds__(kThreads, 1) encode_kernel(const EncodeLaunch a) {
    using Gm = Geo<K>;
    extern __shared__ __align__(16) unsigned char smem[];
    float *M0 = reinterpret_cast<float *>(smem);
    float *M1 = M0 + Gm::G;
    // K = 1: one row of kK1RowFloats (+ 2 for alignment); M1 is not used
    float *ys = K == 1 ? M0 + kK1RowFloats + 2 : M1 + Gm::G;     // up to 256 targets
    uint32_t *bs = reinterpret_cast<uint32_t *>(ys + 256);         // packed codes (tb2)
    unsigned long long *red = reinterpret_cast<unsigned long long *>(bs + 32);
    uint32_t *pf = reinterpret_cast<uint32_t *>(red + 32);          // kTbAhead streamed rows
    __shared__ uint32_t sh_sstar[2], sh_end[2];
    // traceback state, used by thread 0 only: registers at K = 1 (1.7 % faster),
    // shared memory at K = 2 (in registers it spilled and ran 4 % slower)
    __shared__ Tb tb_shared;
    Tb tb_local;
    Tb &tb = K == 1 ? tb_local : tb_shared;

    const int tid = threadIdx.x;

    // mul1 levels of this thread's candidate states, packed two per register
    uint32_t vpk[Gm::STATES / 2];
    if constexpr (K == 1) {
        // vpk[2 i + k] = (v((k << 15) | 2h), v((k << 15) | 2h + 1)), h = (i << 9) | tid
#pragma unroll
        for (int i = 0; i < 32; i++)
#pragma unroll
            for (int k = 0; k < 2; k++) {
                const uint32_t s0 = ((uint32_t)k << 15) | (2u * (((uint32_t)i << 9) | (uint32_t)tid));
                vpk[2 * i + k] = (uint32_t)__half_as_ushort(mul1_half(s0)) |
                                 ((uint32_t)__half_as_ushort(mul1_half(s0 + 1u)) << 16);
            }
    } else
#pragma unroll
    for (int u = 0; u < Gm::NU; u++)
#pragma unroll
        for (int k = 0; k < Gm::NK; k++)
#pragma unroll
            for (int jj = 0; jj < Gm::NJ; jj += 2) {
                const uint32_t g = ((uint32_t)Gm::unit(u, tid) << K) | (uint32_t)(Gm::j0(tid) + jj);
                const uint32_t s0 = ((uint32_t)k << Gm::KR) | g;
                const unsigned short h0 = __half_as_ushort(mul1_half(s0));
                const unsigned short h1 = __half_as_ushort(mul1_half(s0 + 1u));
                vpk[((u * Gm::NK + k) * Gm::NJ + jj) >> 1] = (uint32_t)h0 | ((uint32_t)h1 << 16);
            }

    const float inv_s = a.inv_scale_dev ? __ldg(a.inv_scale_dev) : a.inv_scale;
    // tile bookkeeping fits 32 bits: the ABI bounds a matrix to 2^34 elements
    const int T = TT ? TT : a.T;       // even, 16..256
    const int half = T / 2;
    const int code_words = T * K / 32;
    const bool row_tiles = TT == 0;
    const int tiles_c = row_tiles ? 1 : (int)(a.cols / 16);
    const int n_tiles = row_tiles ? (int)a.rows : (int)(a.rows / 16) * tiles_c;
    const int grid = (int)gridDim.x;
    // a non-finite inverse scale (a rejected weight, see scale_kernel) codes no tile
    const int n_work = a.n_work > 0 ? a.n_work : n_tiles;
    const int n_my = (isfinite(inv_s) && n_work > (int)blockIdx.x)
                         ? (n_work - (int)blockIdx.x + grid - 1) / grid : 0;
    // decision buffers of this block: pass-1 slots 0/1, then pass-2 slots 0/1
    uint32_t *const scr = a.scratch + (size_t)blockIdx.x * (kEncodeBlockScratchBytes / sizeof(uint32_t));
    constexpr size_t kP1 = (size_t)kRowsPass1 * kRowWords, kP2 = (size_t)kRowsPass2 * kRowWords;

    if (tid == 0) {
        tb.on = false;
        tb.rows = nullptr;
        tb.tile = 0;
        tb.s = tb.pending = 0u;
        tb.t = tb.stop = tb.row0 = tb.pass = tb.slot = 0;
    }

    const int npairs = (n_my + 1) / 2;
    for (int ph = 0; ph <= npairs * 4; ph++) {
        const int p = ph >> 2;
        const int sub = ph & 3;
        int f_slot = 0, f_pass = 0, b_slot = 0, b_pass = 0;
        int f_loc = -1, b_loc = -1;
        if (p < npairs) {
            const int A = 2 * p, B = 2 * p + 1;
            const bool hasB = B < n_my;
            if (sub == 0) {
                f_slot = 0; f_pass = 1; f_loc = A;
                if (p > 0) { b_slot = 1; b_pass = 2; b_loc = 2 * p - 1; }
            } else if (sub == 1) {
                if (hasB) { f_slot = 1; f_pass = 1; f_loc = B; }
                b_slot = 0; b_pass = 1; b_loc = A;
            } else if (sub == 2) {
                f_slot = 0; f_pass = 2; f_loc = A;
                if (hasB) { b_slot = 1; b_pass = 1; b_loc = B; }
            } else {
                if (hasB) { f_slot = 1; f_pass = 2; f_loc = B; }
                b_slot = 0; b_pass = 2; b_loc = A;
            }
        } else if (p > 0 && 2 * p - 1 < n_my) {
            b_slot = 1; b_pass = 2; b_loc = 2 * p - 1;   // drain: last B's traceback
        }
        const bool fwd = f_loc >= 0;
        const int f_tile = tile_at(a, f_loc, grid);

        if (fwd) {
            if (tid < T) {
                const int i = (f_pass == 1) ? (tid + half < T ? tid + half : tid + half - T) : tid;
                const float *src;
                if (row_tiles) {
                    src = a.Y + (size_t)f_tile * (size_t)T + i;
                } else {
                    const int tr = f_tile / tiles_c, tc = f_tile % tiles_c;
                    src = a.Y + (size_t)(tr * 16 + (i >> 4)) * (size_t)a.cols + tc * 16 + (i & 15);
                }
                ys[tid] = __fmul_rn(__ldg(src), inv_s);
            }
            if (K == 1 && f_pass == 1) {
                for (int g = tid; g < kK1RowFloats; g += kThreads)
                    M0[g] = 0.0f;
            } else if (K == 1) {
                // M_{-1}(g) at k1_pad(g)
                const uint32_t ge = sh_end[f_slot] & 0x7FFFu;
                for (int g = tid; g < Gm::G; g += kThreads)
                    M0[k1_pad((uint32_t)g)] = ((uint32_t)g == ge) ? 0.0f : __int_as_float(0x7f800000);
            } else if (f_pass == 1) {
                for (int g = tid; g < Gm::G; g += kThreads)
                    M0[g] = 0.0f;
            } else {
                const int ge = (int)(sh_end[f_slot] & (uint32_t)(Gm::G - 1));
                for (int g = tid; g < Gm::G; g += kThreads)
                    M0[g] = (g == ge) ? 0.0f : __int_as_float(0x7f800000);
            }
        }
        if (tid == 0 && b_loc >= 0) {
            tb.on = true;
            tb.pass = b_pass;
            tb.slot = b_slot;
            tb.tile = tile_at(a, b_loc, grid);
            tb.t = T - 1;
            if (b_pass == 1) {
                tb.s = sh_sstar[b_slot];
                tb.stop = half - 1;
                tb.rows = scr + (size_t)b_slot * kP1;
                tb.row0 = half - 1;
            } else {
                tb.s = sh_end[b_slot];
                tb.stop = 0;
                tb.rows = scr + 2 * kP1 + (size_t)b_slot * kP2;
                tb.row0 = 0;
                for (int w = 0; w < code_words; w++)
                    bs[w] = 0u;
                put_code<K>(bs, T - 1, tb.s & (uint32_t)(Gm::NK - 1));
            }
        }
        __syncthreads();

        if (fwd) {
            uint32_t *rows = (f_pass == 1) ? scr + (size_t)f_slot * kP1
                                           : scr + 2 * kP1 + (size_t)f_slot * kP2;
            const int row0 = (f_pass == 1) ? half - 1 : 0;
            for (int t = 0; t < T - 1; t++) {
                if (tid == 0 && tb.on)
                    tb_issue<K>(tb);
                const float *Mp = (t & 1) ? M1 : M0;
                float *Mn = (t & 1) ? M0 : M1;
                uint32_t word[Gm::DW];
                unsigned long long key = 0ull;
                if constexpr (K == 1)
                    acs_step_k1<false>(M0, ys[t], vpk, tid, t % 15, word, key);
                else
                    acs_step_sp<K, false>(Mp, Mn, ys[t], vpk, tid, word, key);
                if (t >= row0) {
#pragma unroll
                    for (int w = 0; w < Gm::DW; w++)
                        rows[(size_t)(t - row0) * kRowWords + tid + w * kThreads] = word[w];
                }
                if (tid == 0 && tb.on)
                    tb_advance<K>(tb, bs);
                __syncthreads();
            }
            if (f_pass == 1) {
                // step T-1 (T even: reads M_{T-2} from M1): lowest full state with minimal cost
                if (tid == 0 && tb.on)
                    tb_issue<K>(tb);
                uint32_t word[Gm::DW];
                unsigned long long key = ~0ull;
                if constexpr (K == 1)
                    acs_step_k1<true>(M0, ys[T - 1], vpk, tid, (T - 1) % 15, word, key);
                else
                    acs_step_sp<K, true>(M1, nullptr, ys[T - 1], vpk, tid, word, key);
                if (tid == 0 && tb.on)
                    tb_advance<K>(tb, bs);
                key = warp_min_u64(key);
                if ((tid & 31) == 0)
                    red[tid >> 5] = key;
                __syncthreads();
                if (tid < 32) {
                    key = warp_min_u64(tid < kThreads / 32 ? red[tid] : ~0ull);
                    if (tid == 0)
                        sh_sstar[f_slot] = (uint32_t)(key & 0xffffffffull);
                }
            } else if (tid == 0 && a.tile_cost) {
                // path forced to end at end_state: fl(M_{T-2}(end >> K) + q_{T-1}(end))
                const uint32_t e = sh_end[f_slot];
                const float d = __fsub_rn(ys[T - 1], mul1_value(e));
                const float mprev = K == 1 ? M0[k1_pad(rotr15(e >> 1, (T - 1) % 15))] : M1[e >> K];
                a.tile_cost[f_tile] = __fadd_rn(mprev, __fmul_rn(d, d));
            }
        }
        if (b_loc >= 0 && !fwd && tid < 32) {
            const Tb r = tb_drain_streamed<K>(tb, bs, pf, tid);
            if (tid == 0)
                tb = r;
        }
        if (tid == 0 && b_loc >= 0) {
            while (tb.on) {
                tb_issue<K>(tb);
                tb_advance<K>(tb, bs);
            }
            if (tb.pass == 1) {
                sh_end[tb.slot] = tb.s;
            } else {
                uint32_t *dst = a.codes + (size_t)tb.tile * code_words;
                for (int w = 0; w < code_words; w++)
                    dst[w] = bs[w];
            }
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// K = 3, 4: two tiles per forward pass.  The cost rows of both fit one SM's
// shared memory (2 tiles x 2 buffers x 2^(16-K) fp32), so each barrier
// interval runs the step of tile x = 0 and then of tile x = 1: twice the work
// per barrier, and one tile's comparisons overlap the other's loads and
// squares.  The pipeline is the one above with "unit" = a pair of tiles:
//     fwd1(P) | tb2(prev Q);  fwd1(Q) | tb1(P);  fwd2(P) | tb1(Q);  fwd2(Q) | tb2(P)
// with the two tracebacks of a pair run by threads 0 and 32.  Decision rows
// are packed to the bits a step produces (K = 4: one word per thread, 512 per
// row; K = 3: two 24-bit fields per thread, 768 words per row) so that the two
// pairs in flight (one region of 2 x 255 rows each) fit the same per-block
// workspace slice as the single-tile pipeline.
// ---------------------------------------------------------------------------
template <int K>
struct Dual {
    static constexpr int RW = K == 3 ? 768 : 512;        // words per decision row
    static constexpr size_t SLOT = (size_t)kRowsPass2 * RW; // one tile's rows
    static_assert(4 * SLOT * sizeof(uint32_t) <= kEncodeBlockScratchBytes, "rows fit the slice");
    // bit offset of D_t(g) in a row
    __device__ __forceinline__ static uint32_t bit_of(uint32_t g) {
        const uint32_t hp = g >> K, j = g & (uint32_t)((1 << K) - 1);
        if (K == 3) {
            const uint32_t tid = hp & 511u, u = hp >> 9;
            return 48u * tid + 24u * u + 3u * j;
        }
        // K = 4: word hp * 2 + j / 8, bit (j % 8) * 4
        return 32u * (hp * 2u + (j >> 3)) + 4u * (j & 7u);
    }
};

template <int K>
__device__ __forceinline__ void dual_store_row(uint32_t *row, const uint32_t (&word)[Geo<K>::DW],
                                               const int tid) {
    if constexpr (K == 4) {
        row[tid] = word[0];
    } else {
        // 48 bits per thread: unit 0 at bits 0..23, unit 1 at 24..47; thread pair
        // (2m, 2m + 1) fills words 3m .. 3m + 2 (the odd thread's low 16 bits
        // complete the even thread's second word)
        const unsigned long long v = (unsigned long long)word[0] | ((unsigned long long)word[1] << 24);
        const uint32_t recv = __shfl_xor_sync(0xffffffffu, (uint32_t)v & 0xFFFFu, 1);
        const int m = tid >> 1;
        if ((tid & 1) == 0) {
            row[3 * m] = (uint32_t)v;
            row[3 * m + 1] = (uint32_t)(v >> 32) | (recv << 16);
        } else {
            row[3 * m + 2] = (uint32_t)(v >> 16);
        }
    }
}

struct Tb2 {         // one traceback of the dual pipeline (threads 0 and 32)
    const uint32_t *rows;
    int tile;
    uint32_t s;
    unsigned long long pending;
    int t, stop, row0, pass;
    bool on;
};

template <int K>
__device__ __forceinline__ void tb2_issue(Tb2 &tb) {
    const uint32_t off = Dual<K>::bit_of(tb.s >> K);
    const uint32_t *r = tb.rows + (size_t)(tb.t - 1 - tb.row0) * Dual<K>::RW + (off >> 5);
    if (K == 3) {
        const uint32_t lo = __ldcg(r);
        const uint32_t hi = ((off & 31u) > 29u) ? __ldcg(r + 1) : 0u;
        tb.pending = (unsigned long long)lo | ((unsigned long long)hi << 32);
    } else {
        tb.pending = __ldcg(r);
    }
}

template <int K>
__device__ __forceinline__ void tb2_advance(Tb2 &tb, uint32_t *bs) {
    using Gm = Geo<K>;
    const uint32_t g = tb.s >> K;
    const uint32_t off = Dual<K>::bit_of(g);
    const uint32_t k = (uint32_t)(tb.pending >> (off & 31u)) & (uint32_t)(Gm::NK - 1);
    tb.s = (k << Gm::KR) | g;
    tb.t -= 1;
    if (tb.pass == 2)
        put_code<K>(bs, tb.t, tb.s & (uint32_t)(Gm::NK - 1));
    if (tb.t == tb.stop)
        tb.on = false;
}

// The pair kernel's streamed traceback (see tb_drain_streamed): warps 0 and 1
// each stream the packed rows of their own tile, kTb2Ahead<K> rows ahead.
template <int K>
constexpr int kTb2Ahead = K == 3 ? 12 : 16;
template <int K>
constexpr size_t kTb2StreamBytes = (size_t)2 * kTb2Ahead<K> * Dual<K>::RW * sizeof(uint32_t);

template <int K>
__device__ __forceinline__ void tb2_copy_row(uint32_t *dst, const uint32_t *src, const int lane) {
#pragma unroll
    for (int i = 0; i < Dual<K>::RW / 128; i++) {     // RW / 4 chunks of 16 bytes
        const int c = (lane + 32 * i) * 4;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
                     ::"r"((uint32_t)__cvta_generic_to_shared(dst + c)), "l"(src + c) : "memory");
    }
}

template <int K>
__device__ __noinline__ Tb2 tb2_drain_streamed(Tb2 tb, uint32_t *bs, uint32_t *pf, const int lane) {
    constexpr int RW = Dual<K>::RW, A = kTb2Ahead<K>;
    const unsigned long long rp = __shfl_sync(0xffffffffu, (unsigned long long)(uintptr_t)tb.rows, 0);
    const int t0 = __shfl_sync(0xffffffffu, tb.t, 0);
    const int n = t0 - __shfl_sync(0xffffffffu, tb.stop, 0);
    const int row0 = __shfl_sync(0xffffffffu, tb.row0, 0);
    const uint32_t *first = reinterpret_cast<const uint32_t *>((uintptr_t)rp) + (size_t)(t0 - 1 - row0) * RW;
#pragma unroll 1
    for (int q = 0; q < A; q++) {
        if (q < n)
            tb2_copy_row<K>(pf + q * RW, first - (size_t)q * RW, lane);
        cp_async_commit();
    }
#pragma unroll 1
    for (int q = 0; q < n; q++) {
        cp_async_wait<A - 1>();
        __syncwarp();
        if (lane == 0) {
            const uint32_t off = Dual<K>::bit_of(tb.s >> K);
            const uint32_t *r = pf + (q % A) * RW + (off >> 5);
            const uint32_t hi = (K == 3 && (off & 31u) > 29u) ? r[1] : 0u;
            tb.pending = (unsigned long long)r[0] | ((unsigned long long)hi << 32);
            tb2_advance<K>(tb, bs);
        }
        __syncwarp();
        if (q + A < n)
            tb2_copy_row<K>(pf + (q % A) * RW, first - (size_t)(q + A) * RW, lane);
        cp_async_commit();
    }
    cp_async_wait<0>();
    __syncwarp();
    return tb;
}

// ST: launches in which every block codes at most one pair (LDLQ rounds, small
// matrices), whose tracebacks run with no forward pass beside them, stream their
// rows (tb2_drain_streamed); other launches take an instantiation without that
// code (at K = 4 its call site alone cost the forward loop 1.3 %).
template <int K, int TT, bool ST>
__global__ void __launch_bounds__(kThreads, 1) encode2_kernel(const EncodeLaunch a) {
    using Gm = Geo<K>;
    using Du = Dual<K>;
    extern __shared__ __align__(16) unsigned char smem[];
    float *Mb = reinterpret_cast<float *>(smem);                  // [x][buffer][G]
    float *ysb = Mb + 4 * Gm::G;                                   // [x][256]
    uint32_t *bsb = reinterpret_cast<uint32_t *>(ysb + 512);       // [x][32]
    unsigned long long *red = reinterpret_cast<unsigned long long *>(bsb + 64);   // [32]
    uint32_t *pf = reinterpret_cast<uint32_t *>(red + 32);        // [warp][kTb2Ahead][RW]
    __shared__ uint32_t sh_sstar[2][2], sh_end[2][2];             // [unit slot][x]
    // this thread's traceback (threads 0 and 32 only): registers at K = 4 (1.7 %
    // faster), shared memory at K = 3 (2.5 % slower in registers)
    __shared__ Tb2 tbs[2];
    Tb2 tb_local;

    const int tid = threadIdx.x;
    const int my_tb = tid == 0 ? 0 : (tid == 32 ? 1 : -1);

    uint32_t vpk[Gm::STATES / 2];
#pragma unroll
    for (int u = 0; u < Gm::NU; u++)
#pragma unroll
        for (int k = 0; k < Gm::NK; k++)
#pragma unroll
            for (int jj = 0; jj < Gm::NJ; jj += 2) {
                const uint32_t g = ((uint32_t)Gm::unit(u, tid) << K) | (uint32_t)(Gm::j0(tid) + jj);
                const uint32_t s0 = ((uint32_t)k << Gm::KR) | g;
                const unsigned short h0 = __half_as_ushort(mul1_half(s0));
                const unsigned short h1 = __half_as_ushort(mul1_half(s0 + 1u));
                vpk[((u * Gm::NK + k) * Gm::NJ + jj) >> 1] = (uint32_t)h0 | ((uint32_t)h1 << 16);
            }

    const float inv_s = a.inv_scale_dev ? __ldg(a.inv_scale_dev) : a.inv_scale;
    const int T = TT ? TT : a.T;
    const int half = T / 2;
    const int code_words = T * K / 32;
    const bool row_tiles = TT == 0;
    const int tiles_c = row_tiles ? 1 : (int)(a.cols / 16);
    const int n_tiles = row_tiles ? (int)a.rows : (int)(a.rows / 16) * tiles_c;
    const int grid = (int)gridDim.x;
    const int n_work = a.n_work > 0 ? a.n_work : n_tiles;
    const int n_my = (isfinite(inv_s) && n_work > (int)blockIdx.x)
                         ? (n_work - (int)blockIdx.x + grid - 1) / grid : 0;
    const int n_units = (n_my + 1) / 2;                  // pairs of tiles
    uint32_t *const scr = a.scratch + (size_t)blockIdx.x * (kEncodeBlockScratchBytes / sizeof(uint32_t));

    if (my_tb >= 0) {
        Tb2 &tb = K == 4 ? tb_local : tbs[my_tb & 1];
        tb.on = false;
        tb.rows = nullptr;
        tb.tile = 0;
        tb.s = 0u;
        tb.pending = 0ull;
        tb.t = tb.stop = tb.row0 = tb.pass = 0;
    }

    const int nq = (n_units + 1) / 2;
    for (int ph = 0; ph <= nq * 4; ph++) {
        const int p = ph >> 2;
        const int sub = ph & 3;
        int f_slot = 0, f_pass = 0, b_slot = 0, b_pass = 0;
        int f_loc = -1, b_loc = -1;
        if (p < nq) {
            const int A = 2 * p, B = 2 * p + 1;
            const bool hasB = B < n_units;
            if (sub == 0) {
                f_slot = 0; f_pass = 1; f_loc = A;
                if (p > 0) { b_slot = 1; b_pass = 2; b_loc = 2 * p - 1; }
            } else if (sub == 1) {
                if (hasB) { f_slot = 1; f_pass = 1; f_loc = B; }
                b_slot = 0; b_pass = 1; b_loc = A;
            } else if (sub == 2) {
                f_slot = 0; f_pass = 2; f_loc = A;
                if (hasB) { b_slot = 1; b_pass = 1; b_loc = B; }
            } else {
                if (hasB) { f_slot = 1; f_pass = 2; f_loc = B; }
                b_slot = 0; b_pass = 2; b_loc = A;
            }
        } else if (p > 0 && 2 * p - 1 < n_units) {
            b_slot = 1; b_pass = 2; b_loc = 2 * p - 1;
        }
        const bool fwd = f_loc >= 0;
        // tiles of a unit: local indices 2 * unit + x
        const bool has1 = fwd && 2 * f_loc + 1 < n_my;

        if (fwd) {
            for (int x = 0; x < (has1 ? 2 : 1); x++) {
                const int f_tile = tile_at(a, 2 * f_loc + x, grid);
                float *ys = ysb + 256 * x;
                if (tid < T) {
                    const int i = (f_pass == 1) ? (tid + half < T ? tid + half : tid + half - T) : tid;
                    const float *src;
                    if (row_tiles) {
                        src = a.Y + (size_t)f_tile * (size_t)T + i;
                    } else {
                        const int tr = f_tile / tiles_c, tc = f_tile % tiles_c;
                        src = a.Y + (size_t)(tr * 16 + (i >> 4)) * (size_t)a.cols + tc * 16 + (i & 15);
                    }
                    ys[tid] = __fmul_rn(__ldg(src), inv_s);
                }
                float *M0 = Mb + (size_t)(2 * x) * Gm::G;
                if (f_pass == 1) {
                    for (int g = tid; g < Gm::G; g += kThreads)
                        M0[g] = 0.0f;
                } else {
                    const int ge = (int)(sh_end[f_slot][x] & (uint32_t)(Gm::G - 1));
                    for (int g = tid; g < Gm::G; g += kThreads)
                        M0[g] = (g == ge) ? 0.0f : __int_as_float(0x7f800000);
                }
            }
        }
        const bool has_b1 = b_loc >= 0 && 2 * b_loc + 1 < n_my;
        if (my_tb >= 0 && b_loc >= 0 && (my_tb == 0 || has_b1)) {
            Tb2 &tb = K == 4 ? tb_local : tbs[my_tb & 1];
            uint32_t *bs = bsb + 32 * my_tb;
            tb.on = true;
            tb.pass = b_pass;
            tb.tile = tile_at(a, 2 * b_loc + my_tb, grid);
            tb.t = T - 1;
            tb.rows = scr + (size_t)(2 * b_slot + my_tb) * Du::SLOT;
            if (b_pass == 1) {
                tb.s = sh_sstar[b_slot][my_tb];
                tb.stop = half - 1;
                tb.row0 = half - 1;
            } else {
                tb.s = sh_end[b_slot][my_tb];
                tb.stop = 0;
                tb.row0 = 0;
                for (int w = 0; w < code_words; w++)
                    bs[w] = 0u;
                put_code<K>(bs, T - 1, tb.s & (uint32_t)(Gm::NK - 1));
            }
        }
        __syncthreads();

        if (fwd) {
            const int row0 = (f_pass == 1) ? half - 1 : 0;
            uint32_t *rows0 = scr + (size_t)(2 * f_slot) * Du::SLOT;
            uint32_t *rows1 = rows0 + Du::SLOT;
            float *const A0 = Mb, *const A1 = Mb + Gm::G;             // tile 0 buffers
            float *const B0 = Mb + 2 * Gm::G, *const B1 = Mb + 3 * Gm::G;   // tile 1 buffers
            for (int t = 0; t < T - 1; t++) {
                if (my_tb >= 0 && (K == 4 ? tb_local : tbs[my_tb & 1]).on)
                    tb2_issue<K>(K == 4 ? tb_local : tbs[my_tb & 1]);
                uint32_t word[Gm::DW];
                unsigned long long key = 0ull;
                acs_step<K, false>((t & 1) ? A1 : A0, (t & 1) ? A0 : A1, ysb[t], vpk, tid, word, key);
                if (t >= row0)
                    dual_store_row<K>(rows0 + (size_t)(t - row0) * Du::RW, word, tid);
                if (has1) {
                    uint32_t word1[Gm::DW];
                    acs_step<K, false>((t & 1) ? B1 : B0, (t & 1) ? B0 : B1, ysb[256 + t], vpk, tid, word1, key);
                    if (t >= row0)
                        dual_store_row<K>(rows1 + (size_t)(t - row0) * Du::RW, word1, tid);
                }
                if (my_tb >= 0 && (K == 4 ? tb_local : tbs[my_tb & 1]).on)
                    tb2_advance<K>(K == 4 ? tb_local : tbs[my_tb & 1], bsb + 32 * my_tb);
                __syncthreads();
            }
            if (f_pass == 1) {
                // step T-1: lowest full state with minimal cost, per tile
                if (my_tb >= 0 && (K == 4 ? tb_local : tbs[my_tb & 1]).on)
                    tb2_issue<K>(K == 4 ? tb_local : tbs[my_tb & 1]);
                uint32_t word[Gm::DW];
                unsigned long long key0 = ~0ull, key1 = ~0ull;
                acs_step<K, true>(A1, nullptr, ysb[T - 1], vpk, tid, word, key0);
                if (has1)
                    acs_step<K, true>(B1, nullptr, ysb[256 + T - 1], vpk, tid, word, key1);
                if (my_tb >= 0 && (K == 4 ? tb_local : tbs[my_tb & 1]).on)
                    tb2_advance<K>(K == 4 ? tb_local : tbs[my_tb & 1], bsb + 32 * my_tb);
                key0 = warp_min_u64(key0);
                key1 = warp_min_u64(key1);
                if ((tid & 31) == 0) {
                    red[tid >> 5] = key0;
                    red[16 + (tid >> 5)] = key1;
                }
                __syncthreads();
                if (tid < 32) {
                    unsigned long long k = red[tid];   // lanes 0..15: tile 0, 16..31: tile 1
#pragma unroll
                    for (int o = 8; o > 0; o >>= 1) {
                        const unsigned long long w = __shfl_xor_sync(0xffffffffu, k, o);
                        k = w < k ? w : k;
                    }
                    if (tid == 0)
                        sh_sstar[f_slot][0] = (uint32_t)(k & 0xffffffffull);
                    if (tid == 16)
                        sh_sstar[f_slot][1] = (uint32_t)(k & 0xffffffffull);
                }
            } else if (a.tile_cost && (tid == 0 || (tid == 32 && has1))) {
                const int x = tid == 0 ? 0 : 1;
                const uint32_t e = sh_end[f_slot][x];
                const float d = __fsub_rn(ysb[256 * x + T - 1], mul1_value(e));
                const float *M1x = x ? B1 : A1;
                a.tile_cost[tile_at(a, 2 * f_loc + x, grid)] = __fadd_rn(M1x[e >> K], __fmul_rn(d, d));
            }
        }
        if constexpr (ST) {
            // no forward pass beside the tracebacks: warps 0 and 1 stream their rows
            if (b_loc >= 0 && !fwd && (tid < 32 || (tid < 64 && has_b1))) {
                const int w = tid >> 5;
                const Tb2 r = tb2_drain_streamed<K>(K == 4 ? tb_local : tbs[w], bsb + 32 * w,
                                                    pf + (size_t)w * kTb2Ahead<K> * Du::RW, tid & 31);
                if ((tid & 31) == 0) {
                    if (K == 4)
                        tb_local = r;
                    else
                        tbs[w] = r;
                }
            }
        }
        if (my_tb >= 0 && b_loc >= 0 && (my_tb == 0 || has_b1)) {
            Tb2 &tb = K == 4 ? tb_local : tbs[my_tb & 1];
            uint32_t *bs = bsb + 32 * my_tb;
            while (tb.on) {
                tb2_issue<K>(tb);
                tb2_advance<K>(tb, bs);
            }
            if (tb.pass == 1) {
                sh_end[b_slot][my_tb] = tb.s;
            } else {
                uint32_t *dst = a.codes + (size_t)tb.tile * code_words;
                for (int w = 0; w < code_words; w++)
                    dst[w] = bs[w];
            }
        }
        __syncthreads();
    }
}

template <int K, int TT, bool ST>
exl3_status launch_dual_st(const EncodeLaunch &p, cudaStream_t s, bool profiled) {
    using Gm = Geo<K>;
    const size_t smem = (size_t)(4 * Gm::G + 512 + 64) * sizeof(float) + 32 * sizeof(unsigned long long) +
                        (ST ? kTb2StreamBytes<K> : 0);
    cudaError_t e = cudaFuncSetAttribute(encode2_kernel<K, TT, ST>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return cuda_check(e, "cudaFuncSetAttribute(encode2)");
    if (profiled)
        profile_encode_begin(s);
    encode2_kernel<K, TT, ST><<<p.grid, kThreads, smem, s>>>(p);
    if (profiled) {
        note_launch();
        profile_encode_end(s);
    }
    return cuda_check(cudaGetLastError(), "encode launch");
}

template <int K, int TT>
exl3_status launch_dual(const EncodeLaunch &p, cudaStream_t s, bool profiled) {
    const int64_t n_tiles = p.row_tiles ? p.rows : (p.rows / 16) * (p.cols / 16);
    const int64_t work = p.n_work > 0 ? p.n_work : n_tiles;
    if (work <= 2 * (int64_t)p.grid)          // at most one pair per block
        return launch_dual_st<K, TT, true>(p, s, profiled);
    return launch_dual_st<K, TT, false>(p, s, profiled);
}

template <int K, int TT>
exl3_status launch_kt(const EncodeLaunch &p, cudaStream_t s, bool profiled) {
    using Gm = Geo<K>;
    const size_t smem = (size_t)((K == 1 ? kK1RowFloats + 2 : 2 * Gm::G) + 256 + 32) * sizeof(float) +
                        32 * sizeof(unsigned long long) + kTbStreamBytes;
    cudaError_t e = cudaFuncSetAttribute(encode_kernel<K, TT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return cuda_check(e, "cudaFuncSetAttribute(encode)");
    if (profiled)
        profile_encode_begin(s);
    encode_kernel<K, TT><<<p.grid, kThreads, smem, s>>>(p);
    if (profiled) {
        note_launch();
        profile_encode_end(s);
    }
    return cuda_check(cudaGetLastError(), "encode launch");
}

template <int K>
exl3_status launch_k(const EncodeLaunch &p, cudaStream_t s, bool profiled) {
    if constexpr (K >= 3) {
        if (p.row_tiles)
            return launch_dual<K, 0>(p, s, profiled);
        return launch_dual<K, 256>(p, s, profiled);
    } else {
        if (p.row_tiles)
            return launch_kt<K, 0>(p, s, profiled);
        return launch_kt<K, 256>(p, s, profiled);
    }
}

}  // namespace

static exl3_status check_work(const EncodeLaunch &p) {
    const int64_t n_tiles = p.row_tiles ? p.rows : (p.rows / 16) * (p.cols / 16);
    const int64_t work = p.n_work > 0 ? p.n_work : n_tiles;
    const bool ok = p.tile0 >= 0 && p.n_work >= 0 && work <= n_tiles &&
                    (p.ring == 0 ? p.tile0 + work <= n_tiles : (p.ring == n_tiles && p.tile0 < n_tiles));
    if (!ok)
        return set_error(EXL3_ERR_INVALID_ARG, "tile range %d + %d (ring %d) outside %lld tiles",
                         p.tile0, p.n_work, p.ring, (long long)n_tiles);
    return EXL3_OK;
}

exl3_status launch_encode_unprofiled(const EncodeLaunch &p, cudaStream_t s) {
    if (exl3_status st = check_work(p); st != EXL3_OK)
        return st;
    switch (p.K) {
    case 1: return launch_k<1>(p, s, false);
    case 2: return launch_k<2>(p, s, false);
    case 3: return launch_k<3>(p, s, false);
    case 4: return launch_k<4>(p, s, false);
    default: return set_error(EXL3_ERR_UNSUPPORTED, "K=%d is not built", p.K);
    }
}

exl3_status launch_encode(const EncodeLaunch &p, cudaStream_t s) {
    if (exl3_status st = check_work(p); st != EXL3_OK)
        return st;
    switch (p.K) {
    case 1: return launch_k<1>(p, s, true);
    case 2: return launch_k<2>(p, s, true);
    case 3: return launch_k<3>(p, s, true);
    case 4: return launch_k<4>(p, s, true);
    default: return set_error(EXL3_ERR_UNSUPPORTED, "K=%d is not built", p.K);
    }
}

}  // namespace exl3
