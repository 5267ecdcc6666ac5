/*
 * exl3_oracle.c -- plain, slow CPU oracle for the EXL3 trellis tile encoder.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark do.  It shares no code, header, table or constant
 * generator with the CUDA path.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -shared -fPIC.
 * Every float operation below is one IEEE-754 binary32 (or binary64 where
 * stated) operation rounded to nearest-even; contraction into FMA is off.
 *
 * Sources (page "EXL3 Intel Arc Quantizer", section "Core Implemented
 * Architecture", by item):
 *   [Enc]   item 1, "SYCL XPU Tile Encoder": add-compare-select dynamic
 *           programming, two-pass tail-biting closure (pass 1 rolled by 128
 *           with a free start finds end_state; pass 2 unrolled, constrained by
 *           pre_state = end_state, emits the path).
 *   [Ref]   item 4, "Contract-Conformant CPU Reference Encoder": 65536 >> K
 *           tracked states, Kr = 16 - K, candidate branch states
 *           sigma = (k << Kr) | e, predecessor sigma >> K, strict-< first-branch
 *           tie-breaking.
 *   [Fmt]   item 5, "Format Primitives & Bitpacking": procedural mul1
 *           codebook (fp16 levels), MSB-first packing with the SWAP16
 *           half-word swap.
 *   [Had]   item 7, "Sylvester Hadamard Transform": natural-order Sylvester
 *           H_128, blockwise H@x per 128 rows and x@H per 128 columns; decode
 *           order H_l -> x su -> H_r -> x sv.
 *   [Qual]  item 10, "Single-Layer Quantization & Distortion Metrics":
 *           reconstruction MSE.
 *   [LDL]   item 3, "Block LDLQ Decomposition & Preprocessing": blockwise
 *           Cholesky/LDL with the block-diagonal inverse folded in
 *           (M = L * blockdiag(L_bb)^-1), damping retries of
 *           2 * sigma_reg * mean(diag H) up to 10 times, bottom-up error
 *           feedback from the strictly lower part of M into the targets of the
 *           rows not yet quantised.
 *   [Reg]   item 8, "Weight Regularization & Global-Scale Search": block_rms
 *           accumulated over 32 slices, output-channel RMS normalisation
 *           folded into sv.
 *
 * Readings fixed where the pages are silent (each also listed in the design
 * notes of the repository):
 *   - mul1 decode: v(s) = fp16_rn( fl32( (bytesum(u32(s * 0x9E3779B1)) - 510)
 *     * MUL1_C ) ), MUL1_C = fl32(1 / population sd of that byte sum over all
 *     65536 states).  0x9E3779B1 = 2654435761, the multiplicative-hashing
 *     prime near 2^32/phi.
 *   - branch metric in fp32 without contraction: d = y - v, q = d*d, and the
 *     tracked cost update c = M + q (add, then compare-select over k).
 *   - ties inside a group: lowest k (strict < over ascending k).
 *   - pass-1 final choice: lowest full state index with minimal cost.
 *   - pass 2 forces the last state to end_state (ring closure).
 *   - Hadamard rounding order: radix-2 butterflies (a,b)->(a+b,a-b), stage
 *     span 1,2,...,64; one exact final multiplication by 2^-7.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define MUL1_MULT 0x9E3779B1u
/* fl32(1 / 147.9146802...) -- pinned by the test suite against an independent
 * numpy recomputation of the byte-sum standard deviation. */
#define MUL1_C 0x1.bb10f4p-8f

/* ------------------------------------------------------------------------ */
/* fp16 rounding                                                             */
/* ------------------------------------------------------------------------ */

/* Round a finite binary32 value to the nearest binary16 value (ties to even)
 * and return it as binary32.  Written from the format definition: binary16 has
 * an 11-bit significand, exponent range [-14, 15], subnormal spacing 2^-24.
 * The scaling and nearbyint() below are exact in binary64. */
float ora_round_fp16(float x)
{
    if (x == 0.0f || isnan(x) || isinf(x))
        return x;
    int e2;
    (void)frexp((double)x, &e2);   /* |x| = m * 2^e2, m in [0.5, 1) */
    int e = e2 - 1;                /* |x| in [2^e, 2^(e+1)) */
    if (e < -14)
        e = -14;                   /* subnormal range: fixed spacing */
    double ulp = ldexp(1.0, e - 10);
    double r = nearbyint((double)x / ulp) * ulp;  /* default mode: ties even */
    if (fabs(r) > 65504.0)
        return x > 0 ? INFINITY : -INFINITY;
    return (float)r;
}

void ora_round_fp16_array(const float *in, float *out, int64_t n)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = ora_round_fp16(in[i]);
}

/* ------------------------------------------------------------------------ */
/* mul1 codebook [Fmt]                                                       */
/* ------------------------------------------------------------------------ */

float ora_mul1_value(uint32_t state)
{
    uint32_t x = state * MUL1_MULT;            /* mod 2^32 */
    int b = (int)(x & 0xFFu) + (int)((x >> 8) & 0xFFu) +
            (int)((x >> 16) & 0xFFu) + (int)((x >> 24) & 0xFFu);
    float f = (float)(b - 510) * MUL1_C;       /* one fp32 multiply */
    return ora_round_fp16(f);
}

void ora_mul1_table(float *out, int n_states)
{
    for (int s = 0; s < n_states; s++)
        out[s] = ora_mul1_value((uint32_t)s);
}

float ora_mul1_constant(void) { return MUL1_C; }
uint32_t ora_mul1_multiplier(void) { return MUL1_MULT; }

/* ------------------------------------------------------------------------ */
/* Viterbi forward pass [Enc], [Ref]                                         */
/* ------------------------------------------------------------------------ */

/*
 * One forward pass over T targets y[0..T) on the L-bit bitshift trellis with K
 * bits per step, codebook cb[2^L].
 *
 * Tracked row: G = 2^(L-K) entries, index g = low L-K bits of a full state.
 * Step t, tracked g: candidates sigma_k = (k << (L-K)) | g, k = 0..2^K-1,
 * whose predecessor tracked index is sigma_k >> K.
 *     cost_t(g) = min over k of fl( cost_{t-1}(sigma_k >> K) + fl(d*d) ),
 *     d = fl(y[t] - cb[sigma_k]),
 * with the first (lowest) k kept on ties; dec[t*G + g] = that k.
 *
 * Initial row cost_{-1}: all zero when constrained == 0 (free start); else
 * zero only at g == (pre_state & (G-1)) and +inf elsewhere, so the first
 * state's predecessor is pre_state.
 *
 * final_cost[G] receives cost_{T-1}; penult_cost[G] (may be NULL) receives
 * cost_{T-2}, the initial row when T == 1.
 */
void ora_viterbi_forward(const float *y, int T, int L, int K, const float *cb,
                         int constrained, uint32_t pre_state,
                         uint8_t *dec, float *final_cost, float *penult_cost)
{
    const int G = 1 << (L - K);
    const int NK = 1 << K;
    float *prev = (float *)malloc(sizeof(float) * (size_t)G);
    float *cur = (float *)malloc(sizeof(float) * (size_t)G);
    for (int g = 0; g < G; g++)
        prev[g] = constrained ? ((g == (int)(pre_state & (uint32_t)(G - 1))) ? 0.0f : INFINITY)
                              : 0.0f;
    for (int t = 0; t < T; t++) {
        if (t == T - 1 && penult_cost)
            memcpy(penult_cost, prev, sizeof(float) * (size_t)G);
        for (int g = 0; g < G; g++) {
            float best = INFINITY;
            int best_k = 0;
            for (int k = 0; k < NK; k++) {
                uint32_t sigma = ((uint32_t)k << (L - K)) | (uint32_t)g;
                float d = y[t] - cb[sigma];
                float q = d * d;
                float c = prev[sigma >> K] + q;
                if (k == 0 || c < best) {   /* strict <: first branch wins ties */
                    best = c;
                    best_k = k;
                }
            }
            cur[g] = best;
            dec[(size_t)t * (size_t)G + (size_t)g] = (uint8_t)best_k;
        }
        float *tmp = prev; prev = cur; cur = tmp;
    }
    memcpy(final_cost, prev, sizeof(float) * (size_t)G);
    free(prev);
    free(cur);
}

/*
 * Traceback: given the full state at step t_last, recover the full states at
 * steps t_last, t_last-1, ..., t_first into states[t] using
 *     s_{t-1} = (dec[t-1][s_t >> K] << (L-K)) | (s_t >> K).
 */
void ora_traceback(const uint8_t *dec, int L, int K, int t_last, int t_first,
                   uint32_t last_state, uint32_t *states)
{
    const int G = 1 << (L - K);
    uint32_t s = last_state;
    states[t_last] = s;
    for (int t = t_last; t > t_first; t--) {
        uint32_t g = s >> K;
        uint32_t k = dec[(size_t)(t - 1) * (size_t)G + g];
        s = (k << (L - K)) | g;
        states[t - 1] = s;
    }
}

/*
 * Lowest full state index with minimal final cost: the final full state of
 * tracked g is (dec[T-1][g] << (L-K)) | g with cost final_cost[g].
 */
uint32_t ora_final_argmin(const uint8_t *dec_last_row, const float *final_cost,
                          int L, int K)
{
    const int G = 1 << (L - K);
    uint32_t best_state = 0;
    float best = INFINITY;
    int have = 0;
    for (int g = 0; g < G; g++) {
        uint32_t s = ((uint32_t)dec_last_row[g] << (L - K)) | (uint32_t)g;
        float c = final_cost[g];
        if (!have || c < best || (c == best && s < best_state)) {
            best = c;
            best_state = s;
            have = 1;
        }
    }
    return best_state;
}

/* ------------------------------------------------------------------------ */
/* Two-pass tail-biting tile encode [Enc]                                    */
/* ------------------------------------------------------------------------ */

/*
 * Encode one tile of T targets.  Pass 1 runs on y rotated left by T/2 with a
 * free start, takes the lowest-index minimal final state and traces back to
 * rotated position T/2 - 1 (original position T-1): that state is end_state.
 * Pass 2 runs on y unrotated with the first predecessor fixed to end_state and
 * traces back from end_state at position T-1.  states[T] receives the pass-2
 * path; *cost receives its final cost fl(cost_{T-2}(end_state >> K) + q), the
 * fp32 left-to-right sum of its branch metrics.
 */
void ora_encode_tile(const float *y, int T, int L, int K, const float *cb,
                     uint32_t *states, float *cost, uint32_t *end_state_out)
{
    const int G = 1 << (L - K);
    const int half = T / 2;
    float *yr = (float *)malloc(sizeof(float) * (size_t)T);
    uint8_t *dec = (uint8_t *)malloc((size_t)T * (size_t)G);
    float *fc = (float *)malloc(sizeof(float) * (size_t)G);
    float *pen = (float *)malloc(sizeof(float) * (size_t)G);
    uint32_t *tmp_states = (uint32_t *)malloc(sizeof(uint32_t) * (size_t)T);

    for (int j = 0; j < T; j++)
        yr[j] = y[(j + half) % T];
    ora_viterbi_forward(yr, T, L, K, cb, 0, 0u, dec, fc, NULL);
    uint32_t s_star = ora_final_argmin(dec + (size_t)(T - 1) * (size_t)G, fc, L, K);
    ora_traceback(dec, L, K, T - 1, half - 1, s_star, tmp_states);
    uint32_t end_state = tmp_states[half - 1];

    ora_viterbi_forward(y, T, L, K, cb, 1, end_state, dec, fc, pen);
    ora_traceback(dec, L, K, T - 1, 0, end_state, states);

    /* cost of the path that ends exactly at end_state */
    {
        float d = y[T - 1] - cb[end_state];
        float q = d * d;
        *cost = pen[end_state >> K] + q;
    }
    if (end_state_out)
        *end_state_out = end_state;
    free(yr);
    free(dec);
    free(fc);
    free(pen);
    free(tmp_states);
}

/* Encode tiles [tile_begin, tile_end) of a [rows, cols] fp32 matrix, 16x16
 * tiles in row-major tile order, elements row-major inside a tile.  Targets
 * are y = fl(Y * inv_scale).  states[(tile_end-tile_begin)*256], costs[...]. */
void ora_encode_matrix(const float *Y, int64_t rows, int64_t cols, int K,
                       float inv_scale, const float *cb,
                       int64_t tile_begin, int64_t tile_end,
                       uint32_t *states, float *costs)
{
    const int64_t tiles_c = cols / 16;
    float y[256];
    (void)rows;
    for (int64_t t = tile_begin; t < tile_end; t++) {
        int64_t tr = t / tiles_c, tc = t % tiles_c;
        for (int i = 0; i < 16; i++)
            for (int j = 0; j < 16; j++)
                y[i * 16 + j] = Y[(tr * 16 + i) * cols + tc * 16 + j] * inv_scale;
        ora_encode_tile(y, 256, 16, K, cb, states + (t - tile_begin) * 256,
                        costs + (t - tile_begin), NULL);
    }
}

/* ------------------------------------------------------------------------ */
/* Packing [Fmt]                                                             */
/* ------------------------------------------------------------------------ */

/*
 * Pack the low K bits of states[0..T) as one MSB-first bitstream
 * e_0 || e_1 || ... (each code most-significant bit first), cut into 16-bit
 * words (first bit of each word = its MSB), then swap the two half-words of
 * every 32-bit pair (SWAP16).  out has T*K/16 uint16 words.
 */
void ora_pack(const uint32_t *states, int T, int K, uint16_t *out)
{
    const int n_words = T * K / 16;
    uint16_t *w = (uint16_t *)calloc((size_t)n_words, sizeof(uint16_t));
    for (int i = 0; i < T; i++) {
        uint32_t e = states[i] & ((1u << K) - 1u);
        for (int b = 0; b < K; b++) {
            int bit = (int)((e >> (K - 1 - b)) & 1u);      /* MSB of the code first */
            int pos = i * K + b;                            /* position in the stream */
            if (bit)
                w[pos / 16] |= (uint16_t)(1u << (15 - (pos % 16)));
        }
    }
    for (int m = 0; m + 1 < n_words; m += 2) {
        out[m] = w[m + 1];
        out[m + 1] = w[m];
    }
    if (n_words % 2)
        out[n_words - 1] = w[n_words - 1];
    free(w);
}

/*
 * Decode states from a packed stream: undo SWAP16, then state i is the
 * L-bit window of the circular bitstream that ends with the last bit of code i,
 * i.e. bits [(i+1)K - L, (i+1)K) modulo T*K, read MSB first.
 */
void ora_unpack_states(const uint16_t *in, int T, int K, int L, uint32_t *states)
{
    const int n_words = T * K / 16;
    const int n_bits = T * K;
    uint16_t *w = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)n_words);
    for (int m = 0; m + 1 < n_words; m += 2) {
        w[m] = in[m + 1];
        w[m + 1] = in[m];
    }
    if (n_words % 2)
        w[n_words - 1] = in[n_words - 1];
    for (int i = 0; i < T; i++) {
        uint32_t s = 0;
        int start = (i + 1) * K - L;
        for (int b = 0; b < L; b++) {
            int pos = ((start + b) % n_bits + n_bits) % n_bits;
            int bit = (w[pos / 16] >> (15 - (pos % 16))) & 1;
            s = (s << 1) | (uint32_t)bit;
        }
        states[i] = s;
    }
    free(w);
}

/* Reconstructed tile values: fl(v(s_i) * scale). */
void ora_decode_values(const uint32_t *states, int T, const float *cb, float scale,
                       float *out)
{
    for (int i = 0; i < T; i++)
        out[i] = cb[states[i]] * scale;
}

/* ------------------------------------------------------------------------ */
/* Blockwise Sylvester Hadamard rotation [Had]                               */
/* ------------------------------------------------------------------------ */

/* In-place unnormalised Sylvester transform of 128 values with stride
 * `stride`: stages with span h = 1, 2, ..., 64, butterfly (a, b) -> (a+b, a-b).
 * Result: x <- H x with H[i][j] = (-1)^popcount(i & j). */
static void fwht128(float *x, int64_t stride)
{
    for (int h = 1; h < 128; h <<= 1)
        for (int i = 0; i < 128; i++)
            if ((i & h) == 0) {
                float a = x[i * stride];
                float b = x[(i + h) * stride];
                x[i * stride] = a + b;
                x[(i + h) * stride] = a - b;
            }
}

/*
 * Forward rotation (encoder side), the mirror of the page's decode order:
 *   X = W x sv (per column) -> rows: X H (per 128 columns) -> x su (per row)
 *   -> columns: H X (per 128 rows) -> x 2^-7.
 * R = 2^-7 H (su . W . sv) H for +-1 sign vectors.  W is fp32 here (a bf16
 * input is widened exactly before the call).
 */
void ora_rotate_forward(const float *W, int64_t rows, int64_t cols,
                        const float *su, const float *sv, float *out)
{
    for (int64_t r = 0; r < rows; r++)
        for (int64_t c = 0; c < cols; c++)
            out[r * cols + c] = W[r * cols + c] * sv[c];
    for (int64_t r = 0; r < rows; r++)
        for (int64_t cb = 0; cb < cols; cb += 128)
            fwht128(out + r * cols + cb, 1);
    for (int64_t r = 0; r < rows; r++)
        for (int64_t c = 0; c < cols; c++)
            out[r * cols + c] = out[r * cols + c] * su[r];
    for (int64_t rb = 0; rb < rows; rb += 128)
        for (int64_t c = 0; c < cols; c++)
            fwht128(out + rb * cols + c, cols);
    for (int64_t i = 0; i < rows * cols; i++)
        out[i] = out[i] * 0x1p-7f;
}

/*
 * Inverse rotation (decoder side), the page's order:
 *   columns: H Q (per 128 rows) -> x su (per row) -> rows: (.) H (per 128
 *   columns) -> x sv (per column) -> x 2^-7.
 */
void ora_rotate_inverse(const float *Q, int64_t rows, int64_t cols,
                        const float *su, const float *sv, float *out)
{
    memcpy(out, Q, sizeof(float) * (size_t)(rows * cols));
    for (int64_t rb = 0; rb < rows; rb += 128)
        for (int64_t c = 0; c < cols; c++)
            fwht128(out + rb * cols + c, cols);
    for (int64_t r = 0; r < rows; r++)
        for (int64_t c = 0; c < cols; c++)
            out[r * cols + c] = out[r * cols + c] * su[r];
    for (int64_t r = 0; r < rows; r++)
        for (int64_t cb = 0; cb < cols; cb += 128)
            fwht128(out + r * cols + cb, 1);
    for (int64_t r = 0; r < rows; r++)
        for (int64_t c = 0; c < cols; c++)
            out[r * cols + c] = (out[r * cols + c] * sv[c]) * 0x1p-7f;
}

/* ------------------------------------------------------------------------ */
/* Fixed-order binary64 reductions [Qual]                                    */
/* ------------------------------------------------------------------------ */

/* Per-tile sums of squares: for tile t (16x16, row-major tile order), the
 * sequential binary64 sum over its 256 elements in row-major order of
 * fl64(a*a) where a = x, or a = fl64(x - ref) when ref != NULL. */
void ora_tile_sumsq(const float *x, const float *ref, int64_t rows, int64_t cols,
                    double *tile_sums)
{
    const int64_t tiles_c = cols / 16, tiles_r = rows / 16;
    for (int64_t tr = 0; tr < tiles_r; tr++)
        for (int64_t tc = 0; tc < tiles_c; tc++) {
            double s = 0.0;
            for (int i = 0; i < 16; i++)
                for (int j = 0; j < 16; j++) {
                    int64_t idx = (tr * 16 + i) * cols + tc * 16 + j;
                    double a = ref ? ((double)x[idx] - (double)ref[idx]) : (double)x[idx];
                    s = s + a * a;
                }
            tile_sums[tr * tiles_c + tc] = s;
        }
}

/* Pairwise tree over n values: each level adds neighbours (2i, 2i+1); an odd
 * last element moves up unchanged; repeat until one value remains. */
double ora_tree_sum(const double *v, int64_t n)
{
    if (n <= 0)
        return 0.0;
    double *a = (double *)malloc(sizeof(double) * (size_t)n);
    memcpy(a, v, sizeof(double) * (size_t)n);
    while (n > 1) {
        int64_t m = n / 2;
        for (int64_t i = 0; i < m; i++)
            a[i] = a[2 * i] + a[2 * i + 1];
        if (n % 2) {
            a[m] = a[n - 1];
            m++;
        }
        n = m;
    }
    double r = a[0];
    free(a);
    return r;
}

/* ------------------------------------------------------------------------ */
/* Block LDL and LDLQ error feedback  [LDL]                                  */
/* ------------------------------------------------------------------------ */

/* Textbook Cholesky H = L L^T in binary64.  Only the lower triangle of H
 * (row-major n x n) is read; L is written row-major with its upper triangle
 * set to zero.  Column by column, each entry is
 *     acc = H[i][j];  for k = 0 .. j-1:  acc = acc - L[i][k] * L[j][k]
 * (one rounded product and one rounded difference per term, ascending k),
 * then L[j][j] = sqrt(acc) and L[i][j] = acc / L[j][j] for i > j.  diag_add
 * is added to every diagonal entry of H first (0 for none).  Returns 0, or
 * j + 1 for the first column whose pivot acc is not > 0. */
int ora_cholesky(const double *H, int64_t n, double diag_add, double *L)
{
    memset(L, 0, sizeof(double) * (size_t)n * (size_t)n);
    for (int64_t j = 0; j < n; j++) {
        double acc = H[j * n + j] + diag_add;
        for (int64_t k = 0; k < j; k++)
            acc = acc - L[j * n + k] * L[j * n + k];
        if (!(acc > 0.0))
            return (int)(j + 1);
        const double d = sqrt(acc);
        L[j * n + j] = d;
        for (int64_t i = j + 1; i < n; i++) {
            double a = H[i * n + j];
            for (int64_t k = 0; k < j; k++)
                a = a - L[i * n + k] * L[j * n + k];
            L[i * n + j] = a / d;
        }
    }
    return 0;
}

/* Retry schedule: attempt a = 0, 1, ..., max_retries factors
 * H + a * delta * I with delta = (2 * sigma_reg) * mean, mean = (sum of the
 * diagonal in ascending order) / n, and the diagonal addend a * delta rounded
 * once.  Returns the number of retries used (0 = undamped), or -1 when every
 * attempt failed. */
int ora_cholesky_damped(const double *H, int64_t n, double sigma_reg, int max_retries, double *L)
{
    double sum = 0.0;
    for (int64_t j = 0; j < n; j++)
        sum = sum + H[j * n + j];
    const double delta = (2.0 * sigma_reg) * (sum / (double)n);
    for (int a = 0; a <= max_retries; a++) {
        if (ora_cholesky(H, n, (double)a * delta, L) == 0)
            return a;
    }
    return -1;
}

/* Inverse of a 16x16 lower-triangular block (row stride ld) by forward
 * substitution, binary64:  X[c][c] = 1 / B[c][c];  for r > c:
 *     acc = 0;  for k = c .. r-1:  acc = acc + B[r][k] * X[k][c];
 *     X[r][c] = -acc / B[r][r]. */
static void lower16_inverse(const double *B, int64_t ld, double X[16][16])
{
    for (int r = 0; r < 16; r++)
        for (int c = 0; c < 16; c++)
            X[r][c] = 0.0;
    for (int c = 0; c < 16; c++) {
        X[c][c] = 1.0 / B[c * ld + c];
        for (int r = c + 1; r < 16; r++) {
            double acc = 0.0;
            for (int k = c; k < r; k++)
                acc = acc + B[r * ld + k] * X[k][c];
            X[r][c] = -acc / B[r * ld + r];
        }
    }
}

/* Block LDL fold: with Lambda = blockdiag of the 16x16 diagonal blocks of
 * L, M = L * Lambda^-1 is unit block-lower-triangular and
 * H = M * (Lambda Lambda^T) * M^T.  Writes fl32 of the strictly lower block
 * part of M (row-major n x n):  for block column b, rows i >= 16 (b + 1),
 *     M[i][16b + c] = sum_{k = c .. 15} L[i][16b + k] * X[k][c]
 * (ascending k, binary64, X = inverse of the diagonal block); the diagonal
 * blocks (identity) and everything above them are written as zero. */
void ora_block_fold(const double *L, int64_t n, float *M)
{
    memset(M, 0, sizeof(float) * (size_t)n * (size_t)n);
    for (int64_t b = 0; b < n / 16; b++) {
        double X[16][16];
        lower16_inverse(L + (16 * b) * n + 16 * b, n, X);
        for (int64_t i = 16 * (b + 1); i < n; i++) {
            for (int c = 0; c < 16; c++) {
                double acc = 0.0;
                for (int k = c; k < 16; k++)
                    acc = acc + L[i * n + 16 * b + k] * X[k][c];
                M[i * n + 16 * b + c] = (float)acc;
            }
        }
    }
}

/* Error feedback of one quantised block-row j (rows 16j .. 16j+15, errors
 * E[16][cols] = fl32(R - Q) of that block-row) into the accumulated target
 * corrections acc[r][c] of every row r < 16 j:
 *     for i = 16 j + 15 down to 16 j:  acc[r][c] = fmaf(M[i][r], E[i - 16 j][c], acc[r][c])
 * Rows are quantised bottom-up, so over the whole sweep each correction is
 * the fp32 fused-multiply-add chain over i = n-1 down to 16 (b + 1). */
void ora_ldlq_feedback(float *acc, const float *M, int64_t n, int64_t cols, int64_t j,
                       const float *E)
{
    for (int64_t r = 0; r < 16 * j; r++) {
        for (int64_t c = 0; c < cols; c++) {
            float a = acc[r * cols + c];
            for (int64_t i = 16 * j + 15; i >= 16 * j; i--)
                a = fmaf(M[i * n + r], E[(i - 16 * j) * cols + c], a);
            acc[r * cols + c] = a;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Output-channel regularisation  [Reg]                                      */
/* ------------------------------------------------------------------------ */

/* block_rms accumulation of every column of W [rows, cols] (fp32): the rows
 * are cut into `slices` consecutive slices of ceil(rows / slices) rows (the
 * last may be shorter or empty); each slice's sum of squares is accumulated
 * in binary64 in ascending row order starting from 0, and the slice sums are
 * added in slice order.  out[c] = that total (the caller takes
 * sqrt(out[c] / rows)). */
void ora_block_sumsq_cols(const float *W, int64_t rows, int64_t cols, int slices, double *out)
{
    const int64_t len = (rows + slices - 1) / slices;
    for (int64_t c = 0; c < cols; c++) {
        double total = 0.0;
        for (int s = 0; s < slices; s++) {
            double part = 0.0;
            const int64_t r0 = (int64_t)s * len;
            const int64_t r1 = r0 + len < rows ? r0 + len : rows;
            for (int64_t r = r0; r < r1; r++) {
                const double w = (double)W[r * cols + c];
                part = part + w * w;
            }
            total = total + part;
        }
        out[c] = total;
    }
}
