/*
 * exl3.h -- C ABI of libexl3: the EXL3 trellis tile encoder on GB300 (sm_103a).
 *
 * Pipeline (page "EXL3 Intel Arc Quantizer", section "Core Implemented
 * Architecture", items 1, 4, 5, 7, 10; page "alpha2beta/JEV-9B-EXL3-K2",
 * section 2):
 *   W --exl3_rotate--> R = 2^-7 H (su.W.sv) H      (blockwise 128x128)
 *     --exl3_encode_tiles(scale s)--> packed K-bit codes per 16x16 tile
 *     --exl3_decode_tiles--> Yhat = v(state) * s
 *     --exl3_rotate(inverse)--> What;  MSE(W, What)
 *   exl3_quantize runs the whole chain at one relative scale g (s = g * rms(R));
 *   exl3_gss_scale runs it inside a golden-section search over g.
 *
 * Conventions shared by every entry point
 *   - Pointers marked (device) are CUDA device pointers owned by the caller;
 *     the library never frees or retains them after the call returns.
 *   - Matrices are dense row-major with no padding: element (r, c) at r*cols+c.
 *   - Tiles are 16x16; tile (tr, tc) has index tr*(cols/16)+tc and its 256
 *     elements are taken row-major.  Codes are uint16 [rows/16][cols/16][16*K]
 *     (see exl3_encode_tiles for the bit layout).
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  All work
 *     is enqueued on it; no entry point synchronises the host with the device,
 *     except exl3_block_ldl, whose damping retries depend on a device result,
 *     and the exl3_wait_timeouts query.
 *   - The library allocates no device memory at run time.  Scratch comes from
 *     the caller's workspace `ws` (device, 256-byte aligned) of `ws_bytes`
 *     bytes, sized with the matching *_workspace_bytes query.  The workspace
 *     must not be used by anything else until the enqueued work has finished.
 *     The one exception is the static scratch array of
 *     exl3_encode_tiles_noalloc (about 24 MiB, see there): it is part of the
 *     library's device code, reserved on a device when that code is loaded
 *     there (with lazy module loading, at the first call that needs it) and
 *     held until the process exits.
 *   - Every argument is checked before anything is enqueued; on a non-OK
 *     status nothing was enqueued (except EXL3_ERR_CUDA, which reports a
 *     failed launch) and no output is promised.  exl3_last_error() returns a
 *     message for the calling thread's last failure.
 *   - Inputs must be finite.  exl3_quantize and exl3_gss_scale detect a
 *     non-finite weight on the device and code nothing (see exl3_quantize);
 *     elsewhere non-finite inputs produce unspecified codes and values but
 *     never an out-of-bounds access: every data-dependent index in the kernels
 *     is masked to its table.
 *   - Arithmetic: IEEE binary32 with round-to-nearest and no FMA contraction
 *     on the encode/decode/rotation path; binary64 for reductions and the
 *     search.  Results are bit-for-bit reproducible run to run.
 */
#ifndef EXL3_H
#define EXL3_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define EXL3_API __attribute__((visibility("default")))
#else
#define EXL3_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    EXL3_OK = 0,
    EXL3_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size, bad bracket */
    EXL3_ERR_UNSUPPORTED = 2,  /* K outside the built set, dims not multiples of 16/128 */
    EXL3_ERR_WORKSPACE = 3,    /* ws_bytes below the minimum for this call */
    EXL3_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
    EXL3_ERR_TIMEOUT = 5,      /* a bounded device-side wait expired (exl3_wait_timeouts) */
    EXL3_ERR_NUMERIC = 6       /* the input has no factorisation (exl3_block_ldl) */
} exl3_status;

typedef enum { EXL3_F32 = 0, EXL3_BF16 = 1 } exl3_dtype;

/* Static string for a status code (never NULL). */
EXL3_API const char *exl3_status_str(int status);

/* Message for the calling thread's most recent non-OK status (never NULL). */
EXL3_API const char *exl3_last_error(void);

/* Library version, major*10000 + minor*100 + patch. */
EXL3_API int exl3_version(void);

/* 1 if this build encodes at K bits per weight, else 0.  K in {1, 2, 3, 4}. */
EXL3_API int exl3_supports_k(int K);

/*
 * Blockwise randomized Hadamard rotation (page "EXL3 Intel Arc Quantizer",
 * Core item 7: natural-order Sylvester H_128, applied per 128 rows and per 128
 * columns; decode order H_l -> x su -> H_r -> x sv).
 *
 *   inverse = 0:  out = 2^-7 * H (su . W . sv) H, in the order
 *                 x sv (columns), rows x H, x su (rows), H x columns, x 2^-7.
 *   inverse = 1:  out = 2^-7 * su . (H W H) . sv, in the page's decode order
 *                 H x columns, x su, rows x H, x sv, x 2^-7.
 * H is the unnormalised Sylvester matrix, applied as radix-2 butterflies
 * (a,b) -> (a+b, a-b) with spans 1, 2, ..., 64.  su/sv are multiplied as given;
 * with +-1 entries the two directions are exact inverses up to rounding.
 *
 *   W    (device) [rows, cols], dtype `dt` (inverse = 1 requires EXL3_F32).
 *   su   (device) fp32 [rows];  sv (device) fp32 [cols].
 *   out  (device) fp32 [rows, cols]; must not overlap W.
 * rows, cols: positive multiples of 128.  Pointers 16-byte aligned.
 */
EXL3_API exl3_status exl3_rotate(const void *W, int dt, int64_t rows, int64_t cols,
                        const float *su, const float *sv, int inverse,
                        float *out, void *stream);

/*
 * Workspace bytes exl3_encode_tiles needs to run n_tiles tiles at K bits with
 * the full machine (one persistent block per SM of the current device).  A
 * smaller workspace (at least exl3_encode_workspace_min_bytes) also works,
 * with fewer blocks.  Returns 0 for unsupported K or n_tiles < 0.
 */
EXL3_API size_t exl3_encode_workspace_bytes(int64_t n_tiles, int K);
EXL3_API size_t exl3_encode_workspace_min_bytes(int K);

/*
 * Trellis-encode every 16x16 tile of Y (page "EXL3 Intel Arc Quantizer",
 * Core item 1: two-pass tail-biting Viterbi; item 4: 65536 >> K tracked
 * states, candidates sigma = (k<<(16-K))|e, predecessor sigma >> K, strict-<
 * first-branch ties; item 5: mul1 codebook,
 * MSB-first packing with SWAP16).
 *
 *   Y      (device) fp32 [rows, cols], the rotated matrix; targets are
 *          y = fl(Y * fl32(1/scale)).
 *   rows, cols: positive multiples of 16.   K in {1, 2, 3, 4}.   scale > 0, finite.
 *   codes  (device, 4-byte aligned) uint16 [rows/16][cols/16][16*K].  For each
 *          tile the codes e_i (low K bits of the chosen state at element i)
 *          form the bitstream e_0 || e_1 || ... || e_255, each code MSB first.
 *          Stream 16-bit word j holds bits [16j, 16j+16) (first bit = MSB) and
 *          is stored at index j^1 (SWAP16).  Equivalently, the tile's codes
 *          read as little-endian uint32 word m are stream bits [32m, 32m+32)
 *          MSB first.  State i is the 16-bit window of the circular stream
 *          ending with the last bit of e_i.
 *   tile_cost (device) fp32 [n_tiles] or NULL: the chosen path's squared error
 *          sum(y_i - v(s_i))^2, accumulated left to right in fp32.
 *   ws/ws_bytes: workspace (see exl3_encode_workspace_bytes).
 */
EXL3_API exl3_status exl3_encode_tiles(const float *Y, int64_t rows, int64_t cols, int K,
                              float scale, uint16_t *codes, float *tile_cost,
                              void *ws, size_t ws_bytes, void *stream);

/*
 * Decode packed codes back to tile values (page "EXL3 Intel Arc Quantizer", Core
 * item 5: state = circular
 * 16-bit window, mul1 decode; item 7: values x scale before the inverse
 * rotation).  Yhat[r, c] = fl(v(s) * scale), v the fp16 mul1 level of s.
 *   codes (device, 4-byte aligned) as produced by exl3_encode_tiles.
 *   Yhat  (device) fp32 [rows, cols].   rows, cols multiples of 16.
 */
EXL3_API exl3_status exl3_decode_tiles(const uint16_t *codes, int64_t rows, int64_t cols, int K,
                              float scale, float *Yhat, void *stream);

/*
 * Row-wise variants for tiles that are not 16x16: every row of Y[n_rows, T]
 * is one tile of T targets (page "EXL3 Intel Arc Quantizer", Core item 1,
 * Shape Support: standard 256-element tiles and 160-element n-gram rows).  Same two-pass search, codebook and packing as
 * exl3_encode_tiles, with the pass-1 roll T/2 and a T*K-bit circular stream
 * per row stored as T*K/16 uint16 words (MSB first, SWAP16).
 *   T even, 16 <= T <= 256, (T*K) % 32 == 0 (e.g. T = 160 for K = 2, 3, 4).
 *   codes (device, 4-byte aligned) uint16 [n_rows][T*K/16];
 *   row_cost (device) fp32 [n_rows] or NULL.
 *   ws: exl3_encode_workspace_bytes(n_rows, K) (same per-block scratch).
 * exl3_decode_rows writes Yhat[n_rows, T] = fl(v(state) * scale).
 */
EXL3_API exl3_status exl3_encode_rows(const float *Y, int64_t n_rows, int T, int K, float scale,
                                      uint16_t *codes, float *row_cost, void *ws, size_t ws_bytes,
                                      void *stream);
EXL3_API exl3_status exl3_decode_rows(const uint16_t *codes, int64_t n_rows, int T, int K,
                                      float scale, float *Yhat, void *stream);

/*
 * Reconstruction MSE (page "EXL3 Intel Arc Quantizer", Core item 10): sum over
 * tiles of the fp64 squared error sum((double)W - (double)What)^2, each tile summed sequentially in
 * row-major order and the tile sums added as a pairwise tree (neighbours
 * (2i, 2i+1) per level, an odd last element moving up), divided by rows*cols.
 *   W (device) dtype dt [rows, cols];  What (device) fp32 [rows, cols].
 *   mse_out (device) one double.   rows, cols multiples of 16.
 *   ws: at least exl3_mse_workspace_bytes(rows, cols) bytes.
 */
EXL3_API size_t exl3_mse_workspace_bytes(int64_t rows, int64_t cols);
EXL3_API exl3_status exl3_mse(const void *W, int dt, const float *What, int64_t rows, int64_t cols,
                     double *mse_out, void *ws, size_t ws_bytes, void *stream);

/*
 * One full quantization at relative scale g (all of the above in order):
 * R = rotate(W); sigma = sqrt(tree(tile sums of R^2) / n) in fp64, taken as
 * 1 when it is 0 (an all-zero matrix); s = fl32(g * sigma); codes = encode(R, s);
 * What = inverse(decode(codes, s));
 * mse = MSE(W, What).
 *   W (device) bf16 or fp32 [rows, cols]; su, sv (device) fp32 sign vectors.
 *   rows, cols multiples of 128; K in {1, 2, 3, 4}; g > 0.
 *   codes (device) uint16 [rows/16][cols/16][16*K].
 *   scale_out (device) float, the absolute scale s (decode with it).
 *   mse_out (device) double.   sigma_out (device) double or NULL.
 *   What (device) fp32 [rows, cols] or NULL to skip writing it.
 *   ws: exl3_quantize_workspace_bytes(rows, cols, K) for the full machine.
 * A non-finite weight is rejected on the device (the call does not
 * synchronise, so the status stays EXL3_OK): when sigma, s or 1/s is not
 * finite, scale_out is NaN, no tile is coded (codes keep their previous
 * contents), and mse_out and What are NaN; sigma_out shows the cause.
 * exl3_gss_scale inherits this for every evaluation.
 */
EXL3_API size_t exl3_quantize_workspace_bytes(int64_t rows, int64_t cols, int K);
EXL3_API exl3_status exl3_quantize(const void *W, int dt, int64_t rows, int64_t cols,
                          const float *su, const float *sv, int K, double g,
                          uint16_t *codes, float *scale_out, double *mse_out,
                          double *sigma_out, float *What,
                          void *ws, size_t ws_bytes, void *stream);

/*
 * Golden-section search over the relative scale g in [lo, hi] (page
 * "alpha2beta/JEV-9B-EXL3-K2", section 2: "Golden Section Search (GSS) scale
 * optimization"), every
 * evaluation a full exl3_quantize.  With phi = (sqrt 5 - 1)/2 in fp64:
 * x1 = b - phi(b-a), x2 = a + phi(b-a), both evaluated; then while fewer than
 * n_eval evaluations: if f(x1) <= f(x2) {b = x2; x2 = x1; x1 = b - phi(b-a);
 * evaluate x1} else {a = x1; x1 = x2; x2 = a + phi(b-a); evaluate x2}.  The
 * result is the evaluated g with least MSE (smaller g on ties).  The search
 * state lives on the device: the host enqueues n_eval evaluations and never
 * waits.
 *   lo < hi, both > 0 and finite; n_eval in [2, 64].
 *   best_codes (device) uint16 [rows/16][cols/16][16*K]: codes at best g.
 *   best_scale_out (device) float; best_g_out, best_mse_out (device) double.
 *   history_out (device) double [2*n_eval] or NULL: (g, mse) per evaluation.
 */
EXL3_API size_t exl3_gss_workspace_bytes(int64_t rows, int64_t cols, int K);
EXL3_API exl3_status exl3_gss_scale(const void *W, int dt, int64_t rows, int64_t cols,
                           const float *su, const float *sv, int K,
                           double lo, double hi, int n_eval,
                           uint16_t *best_codes, float *best_scale_out,
                           double *best_g_out, double *best_mse_out,
                           double *history_out,
                           void *ws, size_t ws_bytes, void *stream);

/*
 * Grid-and-parabola global-scale search on a tile sample (page "EXL3 Intel Arc
 * Quantizer", Core item 8:
 * wrapped-diagonal tile sampling with the highest/lowest-RMS tiles, coarse grid
 * 0.1..1.9 on a strided subsample, fine grid within 0.075 of the coarse
 * minimum on the full sample, parabolic refinement with a 0.01 floor).  The
 * page leaves the details open; this library reads them as follows.
 *   sample   : tiles (i mod TR, i mod TC) for i < max(TR, TC) (TR x TC 16x16
 *              tiles of R = rotate(W)), then the highest- and lowest-RMS tiles
 *              (ties to the lower index) when not already in the sample;
 *   objective: rotated-domain MSE of a subset at s = fl32(g * sigma_R): codes
 *              from y = fl(r * fl32(1/s)); sum (r - fl(v * s))^2 in fp64,
 *              row-major per tile, tiles added as a pairwise tree in sample
 *              order, divided by 256 * tiles;
 *   coarse   : g = k/10, k = 1..19, on sample entries 0, 2, 4, ...;
 *   fine     : g_c + 0.025 k, k = -3..3 (g_c the coarse minimum), full sample;
 *   refine   : when the fine minimum is interior, the vertex of the parabola
 *              through it and its two neighbours, floored at 0.01, evaluated on
 *              the full sample and kept if strictly better.
 * Ties between grid points go to the smaller g.  Everything runs on the device.
 *   W bf16/fp32 [rows, cols], rows and cols multiples of 128 and at most 32736;
 *   su, sv fp32 signs; K in {1, 2, 3, 4}.
 *   g_out (device) double: the chosen relative scale; scale_out (device) float
 *   or NULL: fl32(g * sigma_R); history_out (device) double [54] or NULL:
 *   (g, mse) for the 19 coarse points, the 7 fine points and the refinement
 *   (-1, -1 when it was not valid).
 *   ws: exl3_scale_search_workspace_bytes(rows, cols, K).
 */
EXL3_API size_t exl3_scale_search_workspace_bytes(int64_t rows, int64_t cols, int K);
EXL3_API exl3_status exl3_scale_search(const void *W, int dt, int64_t rows, int64_t cols,
                                       const float *su, const float *sv, int K, double *g_out,
                                       float *scale_out, double *history_out, void *ws,
                                       size_t ws_bytes, void *stream);

/*
 * Block LDL factorisation of a Hessian (page "EXL3 Intel Arc Quantizer", Core
 * item 3: blockwise Cholesky/LDL, the inverse of the 16x16 block diagonal folded in, retry-only damping of
 * 2 sigma_reg mean(diag H) up to 10 times).
 *   H = L L^T (binary64 Cholesky in the textbook order: each entry
 *   H[i][j] - sum_{k<j} L[i][k] L[j][k], k ascending, one rounded product and
 *   one rounded difference per term; sqrt / divide correctly rounded).  With
 *   Lambda = blockdiag of L's 16x16 diagonal blocks, M = L Lambda^-1 is unit
 *   block-lower-triangular and H = M (Lambda Lambda^T) M^T.
 *   Attempt a = 0, 1, ..., max_retries factors H + a * delta * I,
 *   delta = (2 sigma_reg) * (ascending sum of diag H / n); the first attempt
 *   whose pivots are all > 0 is kept.
 *   H (device) double [n, n] row-major, symmetric: only the lower triangle is
 *     read; n a multiple of 16 in [16, 32768].
 *   sigma_reg >= 0 and finite (0.01 in the page's damping); max_retries in
 *     [0, 100] (10 on the page).
 *   M (device, 16-byte aligned) float [n, n] out: fl32 of M's strictly lower
 *     block part (the entries below the 16x16 diagonal blocks); the diagonal
 *     blocks (identity) and everything above them are written as 0.  Each
 *     entry M[i][16b+c] = fl32(sum_{k=c..15} L[i][16b+k] X[k][c]) with X the
 *     inverse of diagonal block b by forward substitution.
 *   retries_out (host) int or NULL: the number of retries used, -1 on failure.
 *   ws: exl3_block_ldl_workspace_bytes(n).
 * Returns EXL3_ERR_NUMERIC when every attempt has a non-positive pivot (M is
 * then not written).  The call synchronises `stream` once per attempt: it
 * reads the pivot flag back to decide whether to retry.
 */
EXL3_API size_t exl3_block_ldl_workspace_bytes(int64_t n);
EXL3_API exl3_status exl3_block_ldl(const double *H, int64_t n, double sigma_reg, int max_retries,
                                    float *M, int *retries_out, void *ws, size_t ws_bytes,
                                    void *stream);

/*
 * LDLQ: trellis-code the 16-row spans of R bottom-up with error feedback
 * (page "EXL3 Intel Arc Quantizer", Core item 3: one-sided LDLQ error
 * feedback, the tile encoder as the callback on each span).  With E = fl32(R - Q) for the spans already coded
 * (Q = fl32(v * scale)), span b (rows 16b .. 16b+15) is coded from the
 * targets U_b = fl32(R_b + acc_b), where acc_b[r][c] is the binary32 chain
 * acc = fmaf(M[i][16b + r], E[i][c], acc) over i = rows-1 down to 16(b+1)
 * (starting from 0), i.e. the correction sum_{i below the span} M[i, span]^T E_i
 * that minimises the Hessian-weighted error tr(E^T H E) span by span.
 * Codes come from fl32(U * fl32(1 / scale)), as in exl3_encode_tiles.
 *   R (device) float [rows, cols]: rotated weights with the input channels (the
 *     Hessian's index) down the rows; rows and cols multiples of 16, each at
 *     most 2^24, rows * cols at most 2^34.
 *   M (device) float [rows, rows]: from exl3_block_ldl (only the strictly
 *     lower block part is read).
 *   K in {1, 2, 3, 4}; scale > 0 and finite (e.g. fl32(g * sigma_R)).
 *   codes (device) uint16 [rows/16, cols/16, 16K] out, the layout of
 *     exl3_encode_tiles; Q (device) float [rows, cols] out or NULL: the
 *     reconstruction fl32(v * scale) of every span.
 *   ws: exl3_ldlq_workspace_bytes(rows, cols, K); a smaller workspace (at least
 *     the K's encode minimum on top of the fixed part) runs fewer encode blocks.
 * A tile depends on the errors of the tiles below it in its own tile column,
 * so the tiles are coded bottom-up in span-major order, one round of the
 * encode grid per launch and at most one span row (cols / 16 tiles) per
 * launch; each launch's errors are fed back before the next one starts.
 */
EXL3_API size_t exl3_ldlq_workspace_bytes(int64_t rows, int64_t cols, int K);
EXL3_API exl3_status exl3_ldlq(const float *R, int64_t rows, int64_t cols, const float *M, int K,
                               float scale, uint16_t *codes, float *Q, void *ws, size_t ws_bytes,
                               void *stream);

/*
 * Output-channel regularisation of a weight before rotation (page "EXL3 Intel Arc
 * Quantizer", Core item 8:
 * block_rms with a 32-slice accumulation order, the output-scale skew
 * heuristic on the top 2 % of sqrt(H_diag) against a 15 % cutoff, output-channel
 * RMS normalisation with sign and scale folded into sv, and the zero-channel
 * floor 0.1 with sv = 0).  The page names the parts only; this library reads
 * them as follows.
 *   S_c      : the rows cut into 32 consecutive slices of ceil(rows / 32) rows;
 *              each slice's binary64 sum of w^2 in row order; the slice sums
 *              added in slice order (block_rms of channel c = sqrt(S_c / rows));
 *   skew     : d = sqrt(h) (binary64) sorted descending; skew = tree(the first
 *              max(1, rows / 50)) / tree(all), binary64 pairwise trees over the
 *              sorted values (neighbours (2i, 2i+1) per level, an odd last
 *              element moves up), 0 when the total is 0;
 *   scale_c  : 0.1 when S_c = 0 (sv_out[c] = 0: the channel decodes to zero);
 *              otherwise fl32(sqrt(S_c / rows)) when the output scales apply,
 *              else the global fl32(sqrt(T / (rows * cols))), T = the S_c added
 *              as a pairwise tree; the output scales apply when skew < 0.15
 *              (apply_out = -1) or when forced (apply_out = 1; 0 forces off);
 *   W_out    : fl32(W[r][c] / scale_c); sv_out[c] = sv[c] * scale_c.
 * The inverse rotation with sv_out in place of the signs sv undoes the
 * normalisation (the decode multiplies by sv as given).
 *   W bf16/fp32 [rows, cols]: input channels down the rows, output channels
 *     across; rows in [1, 65536], cols in [1, 2^24].  W_out (device) float
 *     [rows, cols] may equal W when W is fp32.
 *   h (device) float [rows]: the Hessian's diagonal, >= 0; sv (device) float
 *     [cols]: output-channel signs.
 *   sv_out (device) float [cols] out; info_out (device) double [4] or NULL:
 *     {skew, output scales applied (0/1), all-zero weight (0/1), global RMS}.
 *   ws: exl3_regularize_workspace_bytes(rows, cols).
 */
EXL3_API size_t exl3_regularize_workspace_bytes(int64_t rows, int64_t cols);
EXL3_API exl3_status exl3_regularize(const void *W, int dt, int64_t rows, int64_t cols,
                                     const float *h, const float *sv, int apply_out,
                                     float *W_out, float *sv_out, double *info_out, void *ws,
                                     size_t ws_bytes, void *stream);

/*
 * exl3_encode_tiles without a workspace, for callers that cannot allocate
 * device memory (no counterpart on the pages: an interface addition of this
 * library).  Such callers include plug-ins running inside an application that
 * owns all device memory through its own pool, and latency-critical loops that
 * cannot afford an allocation (cudaMalloc may synchronise the whole device).
 *
 * Same inputs, outputs, layout and results as exl3_encode_tiles (K in
 * {1, 2, 3, 4}).  The decision rows live in a static device array inside the
 * library instead of a caller workspace.  That array holds at
 * most EXL3_NOALLOC_MAX_BLOCKS persistent blocks (8 blocks x 3,137,536 bytes,
 * about 24 MiB) and stays allocated on every device that loads the library's
 * device code until the process exits.
 *   blocks: number of persistent blocks to run, 1..EXL3_NOALLOC_MAX_BLOCKS, or
 *           0 for the maximum.  More is rejected with EXL3_ERR_WORKSPACE.
 *           With at most 8 of the GPU's SMs busy this is slower than
 *           exl3_encode_tiles with a full-machine workspace.
 * Set-up: the first call on each device (and the first after that device's
 * context was destroyed, e.g. by cudaDeviceReset) looks up the array's device
 * address with that device current; with lazy module loading that first call
 * also loads the library's device code.  Make that first call before any
 * stream capture.  The function allocates nothing and creates no CUDA events.
 * All calls share the one array: calls whose work overlaps on the GPU (for
 * example on two streams without ordering) race and produce wrong codes.
 * Nothing in the array needs clearing between calls: each call writes every
 * decision row before reading it.
 */
#define EXL3_NOALLOC_MAX_BLOCKS 8
EXL3_API exl3_status exl3_encode_tiles_noalloc(const float *Y, int64_t rows, int64_t cols, int K,
                                               float scale, uint16_t *codes, float *tile_cost,
                                               int blocks, void *stream);

/*
 * Which kernel the calling thread's most recent exl3_rotate (or the rotation
 * inside exl3_quantize) launched (no counterpart on the pages; a test hook):
 * 1 the TMA forward kernel (bf16 weights, 16-byte aligned pointers), 2 the
 * shared-memory forward kernel (fp32 weights, or when no tensor map could be
 * encoded), 3 the warp-shuffle kernel (inverse, decode-fused, or pointers that
 * are not 16-byte aligned), 0 none yet.  Thread-local; no synchronisation.
 */
EXL3_API int exl3_rotate_last_kernel(void);

/*
 * Profiling (no counterpart on the pages; used by the benchmark).  While
 * enabled, each launch of the encode kernel is bracketed by two CUDA events
 * recorded on its stream, and every kernel launch made by the library is
 * counted.  exl3_profile_read waits for the recorded events, returns the
 * summed encode-kernel time in milliseconds, the number of encode launches
 * and of all kernel launches since the last read or enable, and clears them.
 * Up to 4096 encode launches are recorded between reads.  The events belong
 * to the device that was current at the launch.
 */
EXL3_API void exl3_profile_enable(int on);
EXL3_API exl3_status exl3_profile_read(double *encode_ms, int64_t *encode_launches,
                              int64_t *kernel_launches);

/*
 * Device-side wait accounting (no counterpart on the pages).  One kernel waits
 * on asynchronous arrivals: the forward rotation of bf16 weights waits for its
 * TMA tile loads.  Each such wait gives up after one second, after which the
 * block issues no further loads, waits (bounded) for the loads it already
 * issued, and the launch's results are void.  exl3_wait_timeouts synchronises the device,
 * stores in *count_out (may be NULL) the number of expired waits since the
 * previous call and resets it; it returns EXL3_ERR_TIMEOUT when that number is
 * nonzero, EXL3_ERR_CUDA when the device could not be read, else EXL3_OK.  The
 * count is global to the process and the current device.
 */
EXL3_API exl3_status exl3_wait_timeouts(unsigned int *count_out);

#ifdef __cplusplus
}
#endif

#endif /* EXL3_H */
