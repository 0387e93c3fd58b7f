/*
 * tm_oracle.c -- plain, slow, single-threaded CPU oracle for the tiled fp32 maps.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library includes, links
 * or calls this file; only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg load it.  It shares no code, header, table or helper with
 * the CUDA path.
 *
 * Build: gcc -O2 -std=c11 -fno-fast-math -ffp-contract=off -fPIC -shared
 * (no FTZ, no contraction: every float operation rounds once, as written).
 *
 * Sources (cited by page title and section):
 *   [AL]  Phobos docs, "@aligned" -- "A minimal kernel", "When the promise is broken".
 *   [PZ]  Mojo GPU puzzles, "Aligned Load & Store" -- "The exercise", "Solution".
 *   [SB]  Phobos docs, "Slicing, bounds and masking" -- "Masking",
 *         "Loops over a dynamic extent", "Promising whole tiles with @aligned",
 *         "Reductions over a ragged tile".
 *   [MC]  teenygrad, "Memory Coalescing and Tensor Layout" -- "What it actually
 *         costs", "Strides, and reading an index expression".
 *
 * Layout convention everywhere: row-major [M, N] with an explicit leading
 * dimension ld >= N (element (i, j) lives at i*ld + j), per [MC] "The alignment
 * constraint": use the passed row stride, never the shape's last extent.
 *
 * Parity status: every function here is pinned by the CPU test suite (closed
 * forms, the pages' printed examples, brute force, library routines); none is
 * "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Tile walk over a runtime extent.                                          */
/* [SB] "Loops over a dynamic extent": a loop `for kt in range(0, K, T)` over  */
/* a runtime extent is split into whole tiles, which need no mask, and one     */
/* masked iteration over the remainder.  Written as the walk itself: visit     */
/* kt = 0, T, 2T, ... < K and classify each visit.                             */
/* out[0] = whole (unmasked) iterations, out[1] = masked iterations (0 or 1),  */
/* out[2] = columns covered by the masked iteration, out[3] = all iterations.  */
/* Returns -1 for T <= 0 or K < 0 ([AL]: a tile divisor must be positive).     */
/* ------------------------------------------------------------------------ */
int oracle_tile_walk(int64_t K, int64_t T, int64_t out[4])
{
    int64_t kt, whole = 0, masked = 0, rem = 0, iters = 0;
    if (T <= 0 || K < 0)
        return -1;
    for (kt = 0; kt < K; kt += T) {
        if (kt + T <= K) {
            whole += 1;
        } else {
            masked += 1;
            rem = K - kt;
        }
        iters += 1;
    }
    out[0] = whole;
    out[1] = masked;
    out[2] = rem;
    out[3] = iters;
    return 0;
}

/* ------------------------------------------------------------------------ */
/* In-bounds elements of tile (pm, pn) in a TM x TN tiling of [M, N].         */
/* [SB] "Masking": a slice X[pm*TM :+ TM, pn*TN :+ TN] may run past the end;  */
/* elements past the end are masked.  Counted element by element.             */
/* ------------------------------------------------------------------------ */
int64_t oracle_tile_valid(int64_t M, int64_t N, int64_t TM, int64_t TN,
                          int64_t pm, int64_t pn)
{
    int64_t r, c, valid = 0;
    for (r = 0; r < TM; ++r)
        for (c = 0; c < TN; ++c) {
            int64_t i = pm * TM + r, j = pn * TN + c;
            if (i < M && j < N)
                valid += 1;
        }
    return valid;
}

/* ------------------------------------------------------------------------ */
/* The @aligned promise.  [AL] "When the promise is broken" and [SB]          */
/* "Promising whole tiles with @aligned": the host promises that M and N are  */
/* whole numbers of tiles.  Returns 1 when the promise holds, 0 when broken,  */
/* -1 when a tile is not positive.                                            */
/* ------------------------------------------------------------------------ */
int oracle_promise_kept(int64_t M, int64_t N, int64_t TM, int64_t TN)
{
    if (TM <= 0 || TN <= 0)
        return -1;
    return (M % TM == 0 && N % TN == 0) ? 1 : 0;
}

/* ------------------------------------------------------------------------ */
/* a1: the memory-bound map of [PZ] "The exercise": out[i] = a[i]*SCALE+BIAS  */
/* with SCALE = 2 and BIAS = 1, over every one of the n elements.  The three  */
/* kernels of the puzzle differ only in memory access and give identical      */
/* output, so one definition covers them all.                                 */
/* ------------------------------------------------------------------------ */
void oracle_affine(const float *a, float *out, int64_t n)
{
    const float SCALE = 2.0f, BIAS = 1.0f;
    int64_t i;
    for (i = 0; i < n; ++i) {
        float v = a[i] * SCALE;   /* rounds once (exact: power-of-two scale) */
        out[i] = v + BIAS;        /* rounds once */
    }
}

/* ------------------------------------------------------------------------ */
/* a2: Y = alpha * X of [AL] "A minimal kernel" (kernel `scale`), restricted  */
/* to the in-bounds elements of [M, N]: [SB] "Masking" skips every store past */
/* the end, so words in the ld gap (j >= N) and past row M are never written. */
/* ------------------------------------------------------------------------ */
void oracle_scale2d(const float *X, int64_t ldx, float *Y, int64_t ldy,
                    int64_t M, int64_t N, float alpha)
{
    int64_t i, j;
    for (i = 0; i < M; ++i)
        for (j = 0; j < N; ++j)
            Y[i * ldy + j] = alpha * X[i * ldx + j];
}

/* ------------------------------------------------------------------------ */
/* a3: B = A of [SB] "Promising whole tiles with @aligned" (kernel copy2d),  */
/* in-bounds only, as raw 32-bit words so NaN payloads survive bit for bit.   */
/* ------------------------------------------------------------------------ */
void oracle_copy2d(const uint32_t *A, int64_t lda, uint32_t *B, int64_t ldb,
                   int64_t M, int64_t N)
{
    int64_t i, j;
    for (i = 0; i < M; ++i)
        for (j = 0; j < N; ++j)
            B[i * ldb + j] = A[i * lda + j];
}

/* ------------------------------------------------------------------------ */
/* a5: per-row sums of a row-major matrix -- the stride-1 walk of [MC] "What  */
/* it actually costs" (the page fixes the access order, not the arithmetic;   */
/* the reading is a sum).  Accumulated in fp64: r[i] = sum_j X[i, j].         */
/* ------------------------------------------------------------------------ */
void oracle_rowsum(const float *X, int64_t ldx, int64_t M, int64_t N, double *r)
{
    int64_t i, j;
    for (i = 0; i < M; ++i) {
        double s = 0.0;
        for (j = 0; j < N; ++j)
            s += (double)X[i * ldx + j];
        r[i] = s;
    }
}

/* ------------------------------------------------------------------------ */
/* a6: per-column sums -- the stride-COLS walk of [MC] "What it actually      */
/* costs", the row walk's data read in column order: c[j] = sum_i X[i, j] in  */
/* fp64, rows added in ascending order.                                       */
/* ------------------------------------------------------------------------ */
void oracle_colsum(const float *X, int64_t ldx, int64_t M, int64_t N, double *c)
{
    int64_t i, j;
    for (j = 0; j < N; ++j)
        c[j] = 0.0;
    for (i = 0; i < M; ++i)
        for (j = 0; j < N; ++j)
            c[j] += (double)X[i * ldx + j];
}

/* ------------------------------------------------------------------------ */
/* a8: masked row-max over ragged column tiles, following [SB] "Reductions    */
/* over a ragged tile" step by step for each row i:                            */
/*   for kt in range(0, N, BC):                                               */
/*     s[c] = S[i, kt + c] when kt + c < N, else 0  (a masked load reads 0,   */
/*            [SB] "Masking")                                                 */
/*     fill_mode 0: s[c] = (c < N - kt) ? s[c] : -inf  (the where/iota mask;  */
/*            -inf can never be a row's maximum)                             */
/*     fill_mode 1: no where step -- the zero-fill pitfall the page warns of  */
/*     m = max(m, max_c s[c])                                                 */
/* m starts at -inf, the identity of max, so N = 0 gives -inf.  max follows   */
/* C's fmaxf: a NaN operand is ignored unless both are NaN.                   */
/* Returns -1 for BC <= 0 or an unknown fill_mode.                            */
/* ------------------------------------------------------------------------ */
int oracle_rowmax_masked(const float *S, int64_t lds, int64_t M, int64_t N,
                         int64_t BC, int fill_mode, float *m)
{
    int64_t i, kt, c;
    if (BC <= 0 || (fill_mode != 0 && fill_mode != 1))
        return -1;
    for (i = 0; i < M; ++i) {
        float mi = -INFINITY;
        for (kt = 0; kt < N; kt += BC) {
            for (c = 0; c < BC; ++c) {
                float s = (kt + c < N) ? S[i * lds + kt + c] : 0.0f;
                if (fill_mode == 0)
                    s = (c < N - kt) ? s : -INFINITY;
                mi = fmaxf(mi, s);
            }
        }
        m[i] = mi;
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* f1: softmax row statistics over ragged column tiles.  [SB] "Reductions    */
/* over a ragged tile" names the softmax as the second reduction the zero    */
/* fill breaks; its statistics are the row maximum m and the normaliser      */
/* l = sum_j exp(s_j - m).  Per row i, over the tile walk of the row-max     */
/* oracle above (masked load reading 0, then the where step unless           */
/* fill_mode == 1), every tile value v enters the definition:                */
/*   m = max over all tile values (fmaxf; starts at -inf)                    */
/*   l = sum over all tile values of exp(v - m), in fp64; a value of -inf    */
/*       contributes exp(-inf) = 0; when m = -inf the sum is empty: l = 0.   */
/* With fill -inf this is the plain definition over the N real scores.       */
/* ------------------------------------------------------------------------ */
int oracle_softmax_rowstats(const float *S, int64_t lds, int64_t M, int64_t N,
                            int64_t BC, int fill_mode, float *m, double *l)
{
    int64_t i, kt, c;
    if (BC <= 0 || (fill_mode != 0 && fill_mode != 1))
        return -1;
    for (i = 0; i < M; ++i) {
        float mi = -INFINITY;
        double li = 0.0;
        /* first pass: the maximum over the masked tiles */
        for (kt = 0; kt < N; kt += BC)
            for (c = 0; c < BC; ++c) {
                float s = (kt + c < N) ? S[i * lds + kt + c] : 0.0f;
                if (fill_mode == 0)
                    s = (c < N - kt) ? s : -INFINITY;
                mi = fmaxf(mi, s);
            }
        /* second pass: the sum of exponentials relative to it */
        if (mi != -INFINITY)
            for (kt = 0; kt < N; kt += BC)
                for (c = 0; c < BC; ++c) {
                    float s = (kt + c < N) ? S[i * lds + kt + c] : 0.0f;
                    if (fill_mode == 0)
                        s = (c < N - kt) ? s : -INFINITY;
                    if (s != -INFINITY)
                        li += exp((double)s - (double)mi);
                }
        m[i] = mi;
        l[i] = li;
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* f3: per-channel scale and bias.  [MC] "NCHW versus NHWC": a per-channel   */
/* scale and bias wants the channel to be the fast dimension, which a         */
/* [B, C, H, W] tensor reinterpreted as [N, C] with N = B*H*W gives without  */
/* moving data (channels last, layout 0: channel = column j); with channels  */
/* first the same tensor is [B*C, H*W] and the channel of row i is i mod C   */
/* (layout 1).  Y[i, j] = X[i, j] * scale[ch] + bias[ch], rounded once (a    */
/* fused multiply-add, C's fmaf); a NULL scale means x + bias and a NULL     */
/* bias x * scale, each rounded once.  In-bounds elements only.              */
/* ------------------------------------------------------------------------ */
int oracle_channel_affine(const float *X, int64_t ldx, int64_t R, int64_t K,
                          const float *scale, const float *bias, int64_t C,
                          int layout, float *Y, int64_t ldy)
{
    int64_t i, j;
    if (C <= 0 || (layout != 0 && layout != 1) || (layout == 0 && K > C))
        return -1;
    for (i = 0; i < R; ++i)
        for (j = 0; j < K; ++j) {
            int64_t ch = layout == 0 ? j : i % C;
            float x = X[i * ldx + j], y;
            if (scale != NULL && bias != NULL)
                y = fmaf(x, scale[ch], bias[ch]);
            else if (scale != NULL)
                y = x * scale[ch];
            else if (bias != NULL)
                y = x + bias[ch];
            else
                y = x;
            Y[i * ldy + j] = y;
        }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* f2: keeping the promise by padding.  [AL] "Interactions": when the tile   */
/* sizes come from a tuner, the promise has to hold for every candidate, so  */
/* the host pads (or picks) extents that every candidate divides.  [MC] "The  */
/* alignment constraint": rows that must start on 16 bytes get a padded row  */
/* stride, and kernels use that stride.  Written as the searches they are.   */
/* ------------------------------------------------------------------------ */

/* Smallest e >= extent that every tile divides; -1 on bad input. */
int64_t oracle_padded_extent(int64_t extent, const int32_t *tiles, int32_t ntiles)
{
    int64_t e;
    int32_t k;
    if (extent < 0 || ntiles <= 0)
        return -1;
    for (k = 0; k < ntiles; ++k)
        if (tiles[k] <= 0)
            return -1;
    for (e = extent;; ++e) {
        int ok = 1;
        for (k = 0; k < ntiles && ok; ++k)
            if (e % tiles[k] != 0)
                ok = 0;
        if (ok)
            return e;
    }
}

/* Smallest row stride ld >= N (in floats) whose byte length is a multiple */
/* of align_bytes; -1 on bad input.                                         */
int64_t oracle_row_stride(int64_t N, int32_t align_bytes)
{
    int64_t ld;
    if (N < 0 || align_bytes <= 0 || align_bytes % 4 != 0)
        return -1;
    for (ld = N;; ++ld)
        if ((ld * 4) % align_bytes == 0)
            return ld;
}

/* B[i, j] = A[i, j] inside [M, N], 0 in the rest of [Mp, Np] (the value a   */
/* masked load reads); words of B outside [Mp, Np] are not written.          */
void oracle_pad2d(const uint32_t *A, int64_t lda, int64_t M, int64_t N,
                  uint32_t *B, int64_t ldb, int64_t Mp, int64_t Np)
{
    int64_t i, j;
    for (i = 0; i < Mp; ++i)
        for (j = 0; j < Np; ++j)
            B[i * ldb + j] = (i < M && j < N) ? A[i * lda + j] : 0u;
}

/* ------------------------------------------------------------------------ */
/* f4: the gemm of [AL] "A minimal kernel"'s companion example (kernel gemm, */
/* "without @aligned" / "with @aligned"): C = alpha * (A B) + beta * C_old   */
/* over row-major A [M, K], B [K, N], C [M, N].  The tiled kernel walks K in */
/* whole tiles plus one masked remainder whose missing columns read 0 ([SB]  */
/* "Loops over a dynamic extent"), and masks its M and N edges; both leave   */
/* the plain definition, computed here in fp64 and rounded once to fp32,     */
/* for the rows listed in rows[0 .. nrows) (out is [nrows, N], ld = N).      */
/* ------------------------------------------------------------------------ */
void oracle_gemm_rows(const float *A, int64_t lda, const float *B, int64_t ldb,
                      const float *Cin, int64_t ldc, const int64_t *rows, int64_t nrows,
                      int64_t N, int64_t K, float alpha, float beta, float *out)
{
    int64_t r, j, k;
    for (r = 0; r < nrows; ++r) {
        const int64_t i = rows[r];
        for (j = 0; j < N; ++j) {
            double acc = 0.0;
            for (k = 0; k < K; ++k)
                acc += (double)A[i * lda + k] * (double)B[k * ldb + j];
            acc = (double)alpha * acc;
            if (beta != 0.0f)
                acc += (double)beta * (double)Cin[i * ldc + j];
            out[r * N + j] = (float)acc;
        }
    }
}
