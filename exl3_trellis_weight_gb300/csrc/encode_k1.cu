// encode_k1.cu -- trellis tile encoder at K = 1 bit per weight (page "EXL3 Intel
// Arc Quantizer", Core Implemented Architecture items 1, 4 and 5: K in {1..4}).
//
// At K = 1 the tracked cost row has 2^15 fp32 entries (128 KiB); two copies do
// not fit one SM's shared memory.  A tile is therefore encoded by a cluster of
// two 512-thread blocks on two SMs.  Unit h' (tracked entries 2h', 2h'+1)
// reads M(h') and M(16384 + h'); block r handles the 8192 units
// h' = r*8192 + u3*1024 + 2*tid + m (u3 = 0..7, m = 0, 1: adjacent pairs, so
// the two costs each array read are one 8-byte load; 64 candidate states per
// thread) and keeps, in three rotating buffers in its shared memory, exactly
// the costs its units read:
//   A[i] = M(r*8192 + i),  B[i] = M(16384 + r*8192 + i),  i in [0, 8192).
// The writer pushes: a unit pair yields the four entries
// g = 4 (r*4096 + u3*512 + tid) + 0..3, read next step by block (g >> 13) & 1
// (= u3 >> 2) as its A (r = 0) or B (r = 1) values at g & 8191 -- one 16-byte
// store, a plain shared store into the own block or an st.async into the
// peer's that completes 16 bytes of the transaction count of the peer's
// barrier for that buffer (no multicast).  Every read is local.
//
// Step t reads buffer t mod 3 and writes buffer (t+1) mod 3; it ends with the
// block barrier (own stores) and a wait on the own transaction barrier of the
// written buffer (the peer's 32 KiB).  No fence is needed: the buffer a push
// of step t overwrites was last read at step t-2, and the pusher only got to
// step t after the peer's step t-1 pushes had all arrived, each made after
// the peer's block barrier that closed step t-2.  Each wait is bounded in time;
// on expiry the block stops waiting, the results are void and a device flag
// records it (exl3_k1_wait_timeouts).
//
// Everything else follows encode.cu: the same two passes, tie rules, packing,
// decision rows (each block writes the rows of its own entries into its own
// workspace slice: word tid of each 1024-word row, bit 4 u3 + 2 m + j; words
// 512..1023 unused), and the same two-tile
// pipeline with an interleaved traceback run by thread 0 of block 0; cluster
// barriers separate the pipeline's phases.
#include <cooperative_groups.h>

#include "encode_common.cuh"

namespace cg = cooperative_groups;

namespace exl3 {

namespace {

constexpr size_t kBlockWords = kEncodeBlockScratchBytes / sizeof(uint32_t);

constexpr int kBufFloats = 16384;                    // one buffer: A[8192], B[8192]
// 512 threads x 64 candidate states (256 x 128 is bit-exact too, and 9 % slower)
constexpr int kK1Threads = 512;
constexpr int kPairs = 4096 / kK1Threads;               // unit pairs per thread
constexpr int kHalfPairs = kPairs / 2;                  // pairs bound for one block
constexpr int kDecWords = kPairs / 8;                   // decision words per thread and step
constexpr uint32_t kPushBytes = kK1Threads * kHalfPairs * 16u; // bytes a block receives per step
static_assert(kK1Threads == 512 || kK1Threads == 256, "K=1 block size");
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

// number of K=1 barrier waits that gave up (read and cleared by the host)
__device__ unsigned int g_k1_wait_timeouts;

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
// the same shared-memory offset in block `rank` of the cluster
__device__ __forceinline__ uint32_t cluster_addr(uint32_t a, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}
// 16-byte store into a peer block, completing 16 bytes of its barrier's transaction
__device__ __forceinline__ void push_peer(uint32_t dst, float4 v, uint32_t bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];"
                 :: "r"(dst), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(bar) : "memory");
}
__device__ __forceinline__ void bar_init(uint32_t a) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(a) : "memory");
}
// the single arrival of a phase, announcing the bytes the phase waits for
__device__ __forceinline__ void bar_expect(uint32_t a, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(a), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool bar_test(uint32_t a, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(a), "r"(parity) : "memory");
    return ok != 0u;
}
__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}
// Wait for the phase of parity `parity` of the barrier at a.  Gives up after
// kWaitLimitNs, or at once when another thread of the block already gave up.
__device__ __noinline__ void bar_wait_slow(uint32_t a, uint32_t parity, volatile int *gave_up) {
    const unsigned long long t0 = global_ns();
    while (!bar_test(a, parity)) {
        if (*gave_up)
            return;
        if (global_ns() - t0 > kWaitLimitNs) {
            *gave_up = 1;
            atomicAdd(&g_k1_wait_timeouts, 1u);
            return;
        }
    }
}
__device__ __forceinline__ void bar_wait(uint32_t a, uint32_t parity, volatile int *gave_up) {
    if (!bar_test(a, parity))
        bar_wait_slow(a, parity, gave_up);
}

// Where D_t(g) of tracked entry g (15 bits) lives: owner block, word, bit.
__device__ __forceinline__ void k1_locate(uint32_t g, int &owner, int &word, int &bit) {
    const uint32_t hp = g >> 1;
    const uint32_t i = hp & 8191u;               // up * 2 NT + 2 tid + m
    const uint32_t up = i / (2u * kK1Threads);
    owner = (int)(hp >> 13);
    word = (int)(((i >> 1) % kK1Threads) + kK1Threads * (up >> 3));
    bit = (int)((up & 7u) * 4u + (i & 1u) * 2u + (g & 1u));
}

// traceback step helpers (thread 0 of block 0); tb.rows = slot rows in block 0's slice
__device__ __forceinline__ void k1_tb_issue(Tb &tb) {
    int owner, w, b;
    k1_locate(tb.s >> 1, owner, w, b);
    tb.pending = __ldcg(tb.rows + (size_t)owner * kBlockWords +
                        (size_t)(tb.t - 1 - tb.row0) * kRowWords + w);
}

__device__ __forceinline__ void k1_tb_advance(Tb &tb, uint32_t *bs) {
    const uint32_t g = tb.s >> 1;
    int owner, w, b;
    k1_locate(g, owner, w, b);
    const uint32_t k = (tb.pending >> b) & 1u;
    tb.s = (k << 15) | g;
    tb.t -= 1;
    if (tb.pass == 2)
        put_code<1>(bs, tb.t, tb.s & 1u);
    if (tb.t == tb.stop)
        tb.on = false;
}

// One step of block r: kPairs unit pairs x 2 units x 2 entries x 2 candidates
// per thread (pair up: units h' = r*8192 + up*2NT + 2 tid + m; unit u = 2 up + m;
// the levels of candidate k of unit u are vpk[u*2 + k]).  A, B: this block's
// read buffer.  own: the array this block writes in its own next buffer;
// peer / peer_bar: the same array in the peer's next buffer and the peer's
// barrier for it (shared::cluster addresses).
// FIRST: the pair processed first (kHalfPairs for block 0, 0 for block 1), so
// the pairs whose costs go to the peer block (sidx < kHalfPairs) are computed
// and pushed first and have the longest time to land.
template <bool ARGMIN, int FIRST>
__device__ __forceinline__ void k1_step(const float *__restrict__ A, const float *__restrict__ B,
                                        float *own, const uint32_t peer, const uint32_t peer_bar,
                                        const uint32_t (&vpk)[4 * kPairs], const float y,
                                        const int r, const int tid, uint32_t (&word)[kDecWords],
                                        unsigned long long &key) {
#pragma unroll
    for (int w = 0; w < kDecWords; w++)
        word[w] = 0u;
#pragma unroll
    for (int sidx = 0; sidx < kPairs; sidx++) {
        const int up = (sidx + FIRST) % kPairs;
        const int i = up * (2 * kK1Threads) + 2 * tid;   // units h' = r*8192 + i, i + 1
        const float2 ma = *reinterpret_cast<const float2 *>(A + i);
        const float2 mb = *reinterpret_cast<const float2 *>(B + i);
        float out[4];
#pragma unroll
        for (int m = 0; m < 2; m++) {
            const float m0 = m ? ma.y : ma.x;      // M(h')
            const float m1 = m ? mb.y : mb.x;      // M(16384 + h')
            const int u = 2 * up + m;
            const unsigned long long q0 = sq_pair(vpk[u * 2 + 0], y);
            const unsigned long long q1 = sq_pair(vpk[u * 2 + 1], y);
            int best0 = __float_as_int(__fadd_rn(m0, __uint_as_float((uint32_t)(q0 & 0xffffffffull))));
            int best1 = __float_as_int(__fadd_rn(m0, __uint_as_float((uint32_t)(q0 >> 32))));
            const int c0 = __float_as_int(__fadd_rn(m1, __uint_as_float((uint32_t)(q1 & 0xffffffffull))));
            const int c1 = __float_as_int(__fadd_rn(m1, __uint_as_float((uint32_t)(q1 >> 32))));
            bool keep0, keep1;
            best0 = __vibmin_s32(best0, c0, &keep0);   // ties keep k = 0
            best1 = __vibmin_s32(best1, c1, &keep1);
            const uint32_t bk0 = keep0 ? 0u : 1u, bk1 = keep1 ? 0u : 1u;
            const int bit = 4 * (up & 7) + 2 * m;
            word[up >> 3] |= (bk0 << bit) | (bk1 << (bit + 1));
            if (ARGMIN) {
                const uint32_t g0 = 2u * (uint32_t)(r * 8192 + i + m);
                const unsigned long long k0 =
                    ((unsigned long long)(uint32_t)best0 << 32) | ((bk0 << 15) | g0);
                const unsigned long long k1 =
                    ((unsigned long long)(uint32_t)best1 << 32) | ((bk1 << 15) | (g0 + 1u));
                key = k0 < key ? k0 : key;
                key = k1 < key ? k1 : key;
            }
            out[2 * m] = __int_as_float(best0);
            out[2 * m + 1] = __int_as_float(best1);
        }
        if (!ARGMIN) {
            // entries 4 (r*4096 + up*NT + tid) + 0..3: read next step by block
            // up / kHalfPairs at array offset 4 ((up % kHalfPairs) * NT + tid)
            const int off = 4 * ((up % kHalfPairs) * kK1Threads + tid);
            const float4 v = make_float4(out[0], out[1], out[2], out[3]);
            if (sidx < kHalfPairs)
                push_peer(peer + 4u * (uint32_t)off, v, peer_bar);
            else
                *reinterpret_cast<float4 *>(own + off) = v;
        }
    }
}

template <int TT>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kK1Threads, 1)
    encode_k1_kernel(const EncodeLaunch a) {
    cg::cluster_group cluster = cg::this_cluster();
    const int r = (int)cluster.block_rank();
    extern __shared__ __align__(16) unsigned char smem[];
    // cost buffers b = 0, 1, 2: A_b[8192] then B_b[8192]
    float *const buf = reinterpret_cast<float *>(smem);
    float *const A0 = buf;
    float *const B0 = buf + 8192;
    float *ys = buf + 3 * kBufFloats;
    uint32_t *bs = reinterpret_cast<uint32_t *>(ys + 256);
    unsigned long long *red = reinterpret_cast<unsigned long long *>(bs + 32);
    __shared__ uint32_t sh_sstar[2], sh_end[2];
    __shared__ unsigned long long sh_key;
    __shared__ Tb tb;
    __shared__ __align__(8) unsigned long long bars[3];   // transaction barrier per buffer
    __shared__ int gave_up;
    // the array this block writes (its A for r = 0, B for r = 1) in its own
    // buffer 0, the same array in the peer's buffer 0, the barriers
    const int own_off = r == 0 ? 0 : 8192;
    const uint32_t peer_rank = (uint32_t)(r ^ 1);
    const uint32_t peer0 = cluster_addr(smem_addr(buf + own_off), peer_rank);
    const uint32_t bar0 = smem_addr(&bars[0]);
    const uint32_t peer_bar0 = cluster_addr(bar0, peer_rank);

    const int tid = threadIdx.x;
    uint32_t vpk[4 * kPairs];
#pragma unroll
    for (int u = 0; u < 2 * kPairs; u++)
#pragma unroll
        for (int k = 0; k < 2; k++) {
            const uint32_t hp = (uint32_t)(r * 8192 + (u >> 1) * (2 * kK1Threads) + 2 * tid + (u & 1));
            const uint32_t s0 = ((uint32_t)k << 15) | (2u * hp);
            vpk[u * 2 + k] = (uint32_t)__half_as_ushort(mul1_half(s0)) |
                             ((uint32_t)__half_as_ushort(mul1_half(s0 + 1u)) << 16);
        }

    const float inv_s = a.inv_scale_dev ? __ldg(a.inv_scale_dev) : a.inv_scale;
    const int T = TT ? TT : a.T;
    const int half = T / 2;
    const int code_words = T / 32;
    const bool row_tiles = TT == 0;
    const int tiles_c = row_tiles ? 1 : (int)(a.cols / 16);
    const int n_tiles = row_tiles ? (int)a.rows : (int)(a.rows / 16) * tiles_c;
    const int cid = (int)blockIdx.x >> 1;
    const int n_clusters = (int)gridDim.x >> 1;
    // a non-finite inverse scale (a rejected weight) codes no tile; both blocks
    // of a cluster read the same scalar, so they skip the same barriers
    const int n_my = (isfinite(inv_s) && n_tiles > cid)
                         ? (n_tiles - cid + n_clusters - 1) / n_clusters : 0;
    uint32_t *const scr = a.scratch + (size_t)blockIdx.x * kBlockWords;       // own slice
    uint32_t *const scr0 = a.scratch + (size_t)(2 * cid) * kBlockWords;       // block 0's slice
    constexpr size_t kP1 = (size_t)kRowsPass1 * kRowWords, kP2 = (size_t)kRowsPass2 * kRowWords;

    if (tid == 0) {
        tb.on = false;
        tb.rows = nullptr;
        tb.tile = 0;
        tb.s = tb.pending = 0u;
        tb.t = tb.stop = tb.row0 = tb.pass = tb.slot = 0;
        sh_end[0] = sh_end[1] = sh_sstar[0] = sh_sstar[1] = 0u;
        gave_up = 0;
        for (int b = 0; b < 3; b++)
            bar_init(bar0 + 8u * (uint32_t)b);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // the peer's barriers are initialised before any push reaches them
    cluster_sync();
    uint32_t parity = 0u;   // bit b: parity of the next phase of barrier b

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
            b_slot = 1; b_pass = 2; b_loc = 2 * p - 1;
        }
        const bool fwd = f_loc >= 0;
        const int f_tile = cid + f_loc * n_clusters;

        // block 1 takes end_state from block 0 (written before the last cluster barrier)
        if (r == 1 && tid == 0) {
            const uint32_t *rend = cluster.map_shared_rank(sh_end, 0);
            sh_end[0] = rend[0];
            sh_end[1] = rend[1];
        }
        __syncthreads();

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
            if (f_pass == 1) {
                for (int i = tid; i < 8192; i += kK1Threads) {
                    A0[i] = 0.0f;
                    B0[i] = 0.0f;
                }
            } else {
                const int ge = (int)(sh_end[f_slot] & 0x7FFFu);
                for (int i = tid; i < 8192; i += kK1Threads) {
                    A0[i] = (r * 8192 + i == ge) ? 0.0f : __int_as_float(0x7f800000);
                    B0[i] = (16384 + r * 8192 + i == ge) ? 0.0f : __int_as_float(0x7f800000);
                }
            }
        }
        if (r == 0 && tid == 0 && b_loc >= 0) {
            tb.on = true;
            tb.pass = b_pass;
            tb.slot = b_slot;
            tb.tile = cid + b_loc * n_clusters;
            tb.t = T - 1;
            if (b_pass == 1) {
                tb.s = sh_sstar[b_slot];
                tb.stop = half - 1;
                tb.rows = scr0 + (size_t)b_slot * kP1;
                tb.row0 = half - 1;
            } else {
                tb.s = sh_end[b_slot];
                tb.stop = 0;
                tb.rows = scr0 + 2 * kP1 + (size_t)b_slot * kP2;
                tb.row0 = 0;
                for (int w = 0; w < code_words; w++)
                    bs[w] = 0u;
                put_code<1>(bs, T - 1, tb.s & 1u);
            }
        }
        cluster_sync();

        if (fwd) {
            uint32_t *rows = (f_pass == 1) ? scr + (size_t)f_slot * kP1
                                           : scr + 2 * kP1 + (size_t)f_slot * kP2;
            const int row0 = (f_pass == 1) ? half - 1 : 0;
            int cur = 0;            // buffer read by step t: t mod 3
            for (int t = 0; t < T - 1; t++) {
                const int nxt = cur == 2 ? 0 : cur + 1;
                const uint32_t bar = bar0 + 8u * (uint32_t)nxt;
                if (tid == 0)
                    bar_expect(bar, kPushBytes);
                if (r == 0 && tid == 0 && tb.on)
                    k1_tb_issue(tb);
                const float *Ap = buf + cur * kBufFloats;
                float *own = buf + nxt * kBufFloats + own_off;
                const uint32_t peer = peer0 + (uint32_t)(nxt * kBufFloats * 4);
                const uint32_t peer_bar = peer_bar0 + 8u * (uint32_t)nxt;
                uint32_t word[kDecWords];
                unsigned long long key = 0ull;
                const float y = ys[t];
                if (r == 0)
                    k1_step<false, kHalfPairs>(Ap, Ap + 8192, own, peer, peer_bar, vpk, y, r, tid, word, key);
                else
                    k1_step<false, 0>(Ap, Ap + 8192, own, peer, peer_bar, vpk, y, r, tid, word, key);
                // work that needs no new costs: decision store, traceback
                if (t >= row0) {
#pragma unroll
                    for (int w = 0; w < kDecWords; w++)
                        rows[(size_t)(t - row0) * kRowWords + tid + w * kK1Threads] = word[w];
                }
                if (r == 0 && tid == 0 && tb.on)
                    k1_tb_advance(tb, bs);
                __syncthreads();                                  // own stores
                bar_wait(bar, (parity >> nxt) & 1u, &gave_up);    // the peer's pushes
                parity ^= 1u << nxt;
                cur = nxt;
            }
            if (f_pass == 1) {
                // last step (reads M_{T-2} from buffer cur)
                if (r == 0 && tid == 0 && tb.on)
                    k1_tb_issue(tb);
                uint32_t word[kDecWords];
                unsigned long long key = ~0ull;
                const float *Ap = buf + cur * kBufFloats;
                k1_step<true, 0>(Ap, Ap + 8192, nullptr, 0u, 0u, vpk, ys[T - 1], r, tid, word, key);
                if (r == 0 && tid == 0 && tb.on)
                    k1_tb_advance(tb, bs);
                key = warp_min_u64(key);
                if ((tid & 31) == 0)
                    red[tid >> 5] = key;
                __syncthreads();
                if (tid < 32) {
                    key = warp_min_u64(tid < kK1Threads / 32 ? red[tid] : ~0ull);
                    if (tid == 0)
                        sh_key = key;
                }
                cluster_sync();
                if (r == 0 && tid == 0) {
                    const unsigned long long k1 = *cluster.map_shared_rank(&sh_key, 1);
                    const unsigned long long kk = sh_key < k1 ? sh_key : k1;
                    sh_sstar[f_slot] = (uint32_t)(kk & 0xffffffffull);
                }
            } else if (a.tile_cost) {
                // fl(M_{T-2}(end >> 1) + q_{T-1}(end)); M_{T-2} is in buffer cur of the
                // block that reads it: block (ge >> 13) & 1, array A/B by ge >> 14.
                // The cluster barrier makes both blocks' last stores visible.
                cluster_sync();
                if (r == 0 && tid == 0) {
                    const uint32_t e = sh_end[f_slot];
                    const uint32_t ge = e >> 1;
                    const float *Ac = buf + cur * kBufFloats;
                    const float *arr =
                        cluster.map_shared_rank((ge >> 14) ? Ac + 8192 : Ac, (int)((ge >> 13) & 1u));
                    const float d = __fsub_rn(ys[T - 1], mul1_value(e));
                    a.tile_cost[f_tile] = __fadd_rn(arr[ge & 8191u], __fmul_rn(d, d));
                }
            }
        }
        if (r == 0 && tid == 0 && b_loc >= 0) {
            while (tb.on) {
                k1_tb_issue(tb);
                k1_tb_advance(tb, bs);
            }
            if (tb.pass == 1) {
                sh_end[tb.slot] = tb.s;
            } else {
                uint32_t *dst = a.codes + (size_t)tb.tile * code_words;
                for (int w = 0; w < code_words; w++)
                    dst[w] = bs[w];
            }
        }
        cluster_sync();
    }
}

template <int TT>
exl3_status launch_k1_t(const EncodeLaunch &p, cudaStream_t s, bool profiled) {
    const size_t smem = (size_t)(3 * kBufFloats + 256 + 32) * sizeof(float) + 32 * sizeof(unsigned long long);
    cudaError_t e = cudaFuncSetAttribute(encode_k1_kernel<TT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return cuda_check(e, "cudaFuncSetAttribute(encode k1)");
    // tiles are assigned statically to clusters: launch only as many clusters as
    // can be resident at once, so none starts its share late
    EncodeLaunch q = p;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.grid);
    cfg.blockDim = dim3(kK1Threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    int n_clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&n_clusters, (void *)encode_k1_kernel<TT>, &cfg);
    if (e != cudaSuccess)
        return cuda_check(e, "cudaOccupancyMaxActiveClusters(encode k1)");
    if (n_clusters < 1)
        return set_error(EXL3_ERR_CUDA, "no two-block cluster of the K=1 encoder fits this GPU");
    if (2 * n_clusters < q.grid)
        q.grid = 2 * n_clusters;
    if (profiled)
        profile_encode_begin(s);
    encode_k1_kernel<TT><<<q.grid, kK1Threads, smem, s>>>(q);
    if (profiled) {
        note_launch();
        profile_encode_end(s);
    }
    return cuda_check(cudaGetLastError(), "encode k1 launch");
}

}  // namespace

exl3_status k1_take_wait_timeouts(unsigned int *n) {
    *n = 0;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess)
        return cuda_check(e, "device synchronise (wait timeouts)");
    unsigned int v = 0;
    const unsigned int zero = 0;
    e = cudaMemcpyFromSymbol(&v, g_k1_wait_timeouts, sizeof v);
    if (e == cudaSuccess && v != 0)
        e = cudaMemcpyToSymbol(g_k1_wait_timeouts, &zero, sizeof zero);
    if (e != cudaSuccess)
        return cuda_check(e, "wait timeout count");
    *n = v;
    return EXL3_OK;
}

exl3_status launch_encode_k1(const EncodeLaunch &p, cudaStream_t s, bool profiled) {
    if (p.grid < 2 || (p.grid & 1))
        return set_error(EXL3_ERR_WORKSPACE, "K=1 needs an even number (>= 2) of blocks, got %d",
                         p.grid);
    if (p.row_tiles)
        return launch_k1_t<0>(p, s, profiled);
    return launch_k1_t<256>(p, s, profiled);
}

}  // namespace exl3
