/*
 * tm.h -- C ABI of libtm: memory-bound tiled maps over fp32 tensors, each with
 * a whole-tile fast path (unmasked 16/32-byte vector access, taken only under
 * an explicit promise that the extents are whole numbers of tiles) and a
 * ragged-edge path (out-of-bounds loads read 0, out-of-bounds stores are
 * skipped).  Hand-written CUDA for sm_103a (GB300).
 *
 * Sources, cited by page title and section:
 *   "@aligned" (Phobos docs): "A minimal kernel", "What it changes",
 *       "When the promise is broken", "Interactions".
 *   "Aligned Load & Store" (Mojo GPU puzzles, puzzle 35): "The exercise",
 *       "Key API", "Tips", "Solution".
 *   "Slicing, bounds and masking" (Phobos docs): "Subscript forms", "Masking",
 *       "Loops over a dynamic extent", "Promising whole tiles with @aligned",
 *       "Reductions over a ragged tile".
 *   "Memory Coalescing and Tensor Layout" (teenygrad): "Coalescing",
 *       "What it actually costs", "Seeing it in a real kernel", "Strides",
 *       "Block pointers and descriptors", "The alignment constraint".
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Layout.   2-D tensors are row-major [M, N] fp32 with an explicit leading
 *           dimension (row stride, in elements) ld >= N: element (i, j) is at
 *           base[i*ld + j].  The stride is always the passed one, never N
 *           ("Memory Coalescing and Tensor Layout", "The alignment constraint").
 * Pointers. Every pointer (except `workspace` sizes and host-side out-params
 *           of the probes, which say so) is a DEVICE pointer on the current
 *           CUDA device.  The caller owns all memory; libtm allocates nothing
 *           and keeps no pointer after the call returns.  Its only state is one
 *           status word per device (see tm_check).
 * Streams.  `stream` is a cudaStream_t passed as void*; NULL selects the legacy
 *           default stream.  Every call is asynchronous on that stream: the
 *           return value covers host-side validation and the launch itself.
 * Errors.   No call prints, aborts or throws.  A call that returns anything but
 *           TM_OK has launched nothing and written nothing.  A promise broken
 *           on the device side is reported by the next tm_check, mirroring
 *           the page's failing host synchronize ("@aligned", "When the
 *           promise is broken").
 * Empty.    M == 0, N == 0 or n == 0 is legal.  Maps then do nothing; a
 *           reduction still writes its outputs (sum of nothing = 0, max of
 *           nothing = -inf).
 * Overlap.  The maps may run in place (out == a; Y == X with ldy == ldx;
 *           B == A with ldb == lda).  Any other overlap of inputs and outputs
 *           is rejected with TM_ERR_INVALID_ARG.
 * Tiles.    Tile extents must be positive ("@aligned": a divisor must be
 *           positive) and one of the shapes each entry point lists (the
 *           kernels are instantiated per shape); anything else returns
 *           TM_ERR_UNSUPPORTED_TILE.
 */
#ifndef TM_H_
#define TM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum tm_status {
    TM_OK = 0,
    TM_ERR_INVALID_ARG = 1,      /* negative extent, ld < N, NULL pointer with work, bad overlap, unknown flag or variant */
    TM_ERR_UNSUPPORTED_TILE = 2, /* tile not positive, or not an instantiated shape */
    TM_ERR_MISALIGNED = 3,       /* a vector path or TM_ALIGNED with a pointer or ld that breaks 16-byte alignment */
    TM_ERR_BROKEN_PROMISE = 4,   /* TM_ALIGNED while M % TM != 0 or N % TN != 0 */
    TM_ERR_CUDA = 5,             /* a CUDA runtime call or kernel launch failed */
    TM_ERR_WORKSPACE = 6,        /* workspace NULL, too small or misaligned (colsum: 16 bytes, gemm: 1024) */
    TM_ERR_TIMEOUT = 7           /* a bounded device-side wait gave up (reported by tm_check) */
} tm_status;

/* A cudaStream_t, passed as an opaque pointer; NULL = legacy default stream. */
typedef void *tm_stream_t;

/* flags (bitwise OR) */
/* The @aligned promise: M % TM == 0 and N % TN == 0 (and, implied by the
 * 16-byte access it unlocks, every base pointer 16-byte aligned and every ld a
 * multiple of 4).  Masks are dropped.  Checked on the host before launch
 * (TM_ERR_MISALIGNED / TM_ERR_BROKEN_PROMISE, nothing launched) and once more
 * at kernel entry ("@aligned", "When the promise is broken"; "Slicing, bounds
 * and masking", "Promising whole tiles with @aligned"). */
#define TM_ALIGNED 0x1u
/* Path forcing, for tests and ablations; at most one may be set.  Without
 * them the library picks the fastest path the arguments allow. */
#define TM_PATH_SCALAR 0x10u /* per-element accesses with per-element masks */
#define TM_PATH_VEC 0x20u    /* 16-byte register accesses (needs the vector alignment) */
#define TM_PATH_TMA 0x40u    /* TMA tile copies through shared memory (needs 16-byte rows) */
/* Overlapped launch (programmatic dependent launch): the call's kernel may
 * start while the previous kernel in the stream is still draining.  Its loads
 * of the inputs may then run ahead of that kernel; every store, and the
 * kernel's completion, still wait for it, so writes stay in stream order and a
 * chain of such calls completes in order.  Use it only when no kernel still
 * pending on the stream writes this call's inputs (for example independent
 * maps of one resident tensor, back to back).  Accepted by every entry point
 * that takes flags except tm_gemm, and by tm_affine OR-ed into its variant. */
#define TM_PDL 0x200u

typedef enum tm_variant {
    TM_VAR_AUTO = 0,
    /* tm_affine ("Aligned Load & Store", "The exercise") */
    TM_VAR_SCALAR = 1,        /* one element per thread, one 4-byte load and store */
    TM_VAR_VEC_UNALIGNED = 2, /* 4 elements per thread through 4 scalar 4-byte loads and stores */
    TM_VAR_VEC4 = 3,          /* 4 elements per access, one 16-byte load and store (needs 16-byte pointers) */
    TM_VAR_VEC8 = 4,          /* 8 elements per access, one 32-byte load and store (needs 32-byte pointers) */
    /* tm_colsum ("Memory Coalescing and Tensor Layout", "What it actually costs",
     * "Seeing it in a real kernel") */
    TM_VAR_NAIVE = 5,     /* the column walk: 256-lane programs over rows, stride ld between lanes */
    TM_VAR_STAGED = 6,    /* TMA tiles staged in shared memory, columns reduced from there; a cluster per strip
                             adds the partials over distributed shared memory (no workspace) */
    TM_VAR_REGDIRECT = 7, /* lanes over columns: coalesced row segments straight into registers */
    TM_VAR_CLUSTER = 8    /* REGDIRECT's layout in one pass: clusters of 8 or 16 CTAs split a strip's rows and add
                             their partials over distributed shared memory (no workspace) */
} tm_variant;

typedef enum tm_fill {
    TM_FILL_NEG_INF = 0, /* where(iota < N - kt, s, -inf): padding never wins the max */
    TM_FILL_ZERO = 1     /* no where step: padding reads as 0 (the pitfall, kept as a foil) */
} tm_fill;

/* Human-readable name of a status code (static string, never NULL). */
const char *tm_status_string(tm_status st);

/* Library version, major*10000 + minor*100 + patch. */
int tm_version(void);

/*
 * tm_affine -- out[i] = a[i]*2 + 1 for 0 <= i < n.
 * "Aligned Load & Store", "The exercise" and "Solution": the same map through
 * three access patterns.  Every variant writes every element (the puzzle's
 * vector kernels skip the n % 4 tail; here a scalar tail finishes it) and all
 * variants are bit-identical: 2a is exact, so the result is 2a + 1 rounded once.
 *   a, out   device pointers to n floats (out == a allowed, no other overlap)
 *   n        element count, >= 0
 *   variant  TM_VAR_AUTO (widest access the alignment allows), _SCALAR,
 *            _VEC_UNALIGNED, _VEC4 (a, out 16-byte aligned), _VEC8 (32-byte);
 *            may be OR-ed with TM_PDL (an overlapped launch).  This is the one
 *            place in the ABI where a flag bit rides in an enum argument:
 *            tm_affine keeps the boundary's signature, which has no flags
 *            word.  C callers OR the two; C++ callers cast the result back,
 *            e.g. (tm_variant)(TM_VAR_VEC4 | TM_PDL).  No other enum value
 *            has the TM_PDL bit set, and no other entry point reads it there.
 * Errors: INVALID_ARG (n < 0, NULL with n > 0, bad variant, partial overlap),
 *         MISALIGNED (VEC4/VEC8 with misaligned pointers), CUDA.
 */
tm_status tm_affine(const float *a, float *out, int64_t n, tm_variant variant, tm_stream_t stream);

/*
 * tm_scale2d -- Y[i, j] = alpha * X[i, j] for i < M, j < N, one TM x TN tile
 * per work unit.  "@aligned", "A minimal kernel" (kernel `scale`, TM = 32,
 * TN = 128).  Words of Y outside [M, N] (the ld gap, past row M) are never
 * written ("Slicing, bounds and masking", "Masking").
 *   X, ldx   device input [M, ldx]     Y, ldy   device output [M, ldy]
 *   TM, TN   tile: (8,8) (16,16) (32,32) (64,64) (32,128) (128,128)
 *   flags    TM_ALIGNED and/or one TM_PATH_* bit, and/or TM_PDL
 * Errors: INVALID_ARG, UNSUPPORTED_TILE, MISALIGNED, BROKEN_PROMISE, CUDA.
 */
tm_status tm_scale2d(const float *X, int64_t ldx, float *Y, int64_t ldy, int64_t M, int64_t N,
                     float alpha, int32_t TM, int32_t TN, uint32_t flags, tm_stream_t stream);

/*
 * tm_copy2d -- B[i, j] = A[i, j] bit for bit, for i < M, j < N.
 * "Slicing, bounds and masking", "Promising whole tiles with @aligned"
 * (kernel copy2d, TM = TN = 64).  Same tiles, flags, masking and errors as
 * tm_scale2d.  NaN payloads are preserved.
 */
tm_status tm_copy2d(const float *A, int64_t lda, float *B, int64_t ldb, int64_t M, int64_t N,
                    int32_t TM, int32_t TN, uint32_t flags, tm_stream_t stream);

/*
 * tm_channel_affine -- per-channel scale and bias over a [B, C, H, W] tensor,
 * Y = X * scale[ch] + bias[ch] rounded once (fused multiply-add); a NULL scale
 * gives X + bias, a NULL bias X * scale (each rounded once).  "Memory
 * Coalescing and Tensor Layout", "NCHW versus NHWC": the operation wants the
 * channel as the fast dimension, which reinterpreting the tensor (no data
 * moved) provides:
 *   layout TM_CHANNELS_LAST  -- X is [R, K] = [B*H*W, C]: channel = column j
 *                               (requires K <= C);
 *   layout TM_CHANNELS_FIRST -- X is [R, K] = [B*C, H*W]: channel = i mod C
 *                               (requires R < 2^31).
 * Same tiles, flags, paths, masking and in-place rule as tm_scale2d.
 *   scale, bias   device vectors of C floats, or NULL; never overlapping Y.
 *                 With channels last, the vector paths need 16-byte aligned
 *                 parameter vectors (otherwise the scalar path is taken).
 * Errors: INVALID_ARG (also C <= 0, unknown layout), UNSUPPORTED_TILE,
 *         MISALIGNED, BROKEN_PROMISE, CUDA.
 */
#define TM_CHANNELS_LAST 0
#define TM_CHANNELS_FIRST 1
tm_status tm_channel_affine(const float *X, int64_t ldx, int64_t R, int64_t K, const float *scale,
                            const float *bias, int64_t C, int32_t layout, float *Y, int64_t ldy, int32_t TM,
                            int32_t TN, uint32_t flags, tm_stream_t stream);

/*
 * Keeping the promise by padding.  "@aligned", "Interactions": when tiles come
 * from a tuner the promise must hold for every candidate, so the host pads the
 * extents; "Memory Coalescing and Tensor Layout", "The alignment constraint":
 * rows that must start on 16 bytes get a padded stride, and that stride -- not
 * the shape -- is what kernels are given.
 *
 * tm_padded_extent -- the smallest extent >= `extent` that every one of the
 * ntiles candidate tiles (a HOST array of positive ints) divides: `extent`
 * rounded up to their least common multiple.  -1 on bad input or overflow.
 * Host only, no CUDA call.
 *
 * tm_row_stride -- the smallest row stride >= N (in floats) whose rows are a
 * whole multiple of align_bytes (a power of two, >= 4): 16 gives N rounded up
 * to a multiple of 4.  -1 on bad input.  Host only.
 *
 * tm_pad2d -- B[i, j] = A[i, j] for i < M, j < N and B[i, j] = 0 for the rest
 * of [Mp, Np] (the value a masked load reads, so sums over B equal sums over A
 * and the aligned path can run on B).  Words of B outside [Mp, Np] are not
 * written.  A and B must not overlap.  Requires Mp >= M, Np >= N, lda >= N,
 * ldb >= Np.  16-byte vectors when B, ldb, Np (and A, lda, N) allow.
 * Errors: INVALID_ARG, MISALIGNED (a pointer not 4-byte aligned), CUDA.
 */
int64_t tm_padded_extent(int64_t extent, const int32_t *tiles, int32_t ntiles);
int64_t tm_row_stride(int64_t N, int32_t align_bytes);
tm_status tm_pad2d(const float *A, int64_t lda, int64_t M, int64_t N, float *B, int64_t ldb, int64_t Mp,
                   int64_t Np, tm_stream_t stream);

/*
 * tm_rowsum -- r[i] = sum_j X[i, j] (fp32 accumulation), the stride-1 walk of
 * "Memory Coalescing and Tensor Layout", "What it actually costs".  Each row
 * is walked in TN-column tiles: the whole tiles unmasked, then one masked
 * remainder tile whose missing columns read 0 ("Slicing, bounds and masking",
 * "Loops over a dynamic extent").  One warp per row, TM rows per block.
 *   X, ldx   device input [M, ldx]     r   device output, M floats
 *   TM       rows per block: 1, 2, 4, 8, 16, 32
 *   TN       columns per tile: 128, 256, 512, 1024
 *   flags    TM_ALIGNED (no remainder tile and no row mask), TM_PATH_SCALAR, TM_PATH_VEC,
 *            TM_PDL
 * Errors: INVALID_ARG, UNSUPPORTED_TILE, MISALIGNED, BROKEN_PROMISE, CUDA.
 */
tm_status tm_rowsum(const float *X, int64_t ldx, int64_t M, int64_t N, float *r, int32_t TM,
                    int32_t TN, uint32_t flags, tm_stream_t stream);

/*
 * tm_colsum_workspace_bytes -- bytes of scratch tm_colsum needs for these
 * arguments (a partial sum per column per row chunk).  0 for invalid
 * arguments or when no scratch is needed (M == 0 or N == 0).
 */
size_t tm_colsum_workspace_bytes(int64_t M, int64_t N, int32_t TM, int32_t TN, tm_variant variant);

/*
 * tm_colsum -- c[j] = sum_i X[i, j] (fp32 accumulation), the stride-COLS walk
 * of "Memory Coalescing and Tensor Layout", "What it actually costs", and its
 * fix from "Seeing it in a real kernel" (stage a tile in fast on-chip memory
 * and read it there in any order).
 * Row chunks write partial sums to `workspace`; a second pass adds them in a
 * fixed order, so the result is deterministic run to run.  When every
 * TN-column strip is a single row chunk -- tm_colsum_workspace_bytes returns
 * 0: at most max(64, TM) rows, or 8192 strips and more -- the first pass
 * writes c itself and needs no workspace.
 * TM_VAR_CLUSTER and TM_VAR_STAGED instead add the partials of a strip's row
 * chunks on chip (a thread-block cluster's distributed shared memory), also
 * in a fixed order, in one pass; with the 16-byte path both give the same
 * bits.
 *   X, ldx      device input [M, ldx]        c   device output, N floats
 *   workspace   device scratch of >= tm_colsum_workspace_bytes(...) bytes,
 *               16-byte aligned (128-byte alignment lets the second pass drop
 *               the partials from L2 without writing them back), owned by the
 *               caller; its contents on entry do not matter and on exit are
 *               unspecified.  NULL allowed when tm_colsum_workspace_bytes is 0
 *               (TM_VAR_CLUSTER and TM_VAR_STAGED always, the others for
 *               single-chunk strips)
 *   TM, TN      row tile x column strip: TM in 8..256 (powers of two),
 *               TN in 64, 128, 256; TM*TN <= 8192 for STAGED
 *               (NAIVE ignores them: its programs are 256 rows x 1 column)
 *   variant     TM_VAR_AUTO (the fastest measured: CLUSTER whenever all its
 *               clusters fit on the GPU at once -- e.g. [4096, 4096] and
 *               [8192, 8192] at TN 128 -- else REGDIRECT), _NAIVE,
 *               _REGDIRECT, _CLUSTER and _STAGED (16 CTAs per strip when there
 *               are few strips, else 8); the workspace AUTO sizes is passed
 *               either way
 *   flags       TM_ALIGNED (whole row tiles and strips: no masks), TM_PATH_SCALAR,
 *               TM_PDL (the first pass overlaps the previous kernel; the
 *               finish pass of a two-pass variant always overlaps the first)
 * Errors: INVALID_ARG, UNSUPPORTED_TILE, MISALIGNED, BROKEN_PROMISE,
 *         WORKSPACE, CUDA; a stalled TMA pipeline (STAGED) or partial sums
 *         that never reach their cluster peer (CLUSTER, STAGED; each wait is
 *         bounded) are reported by tm_check as TM_ERR_TIMEOUT, with the
 *         affected columns of c left unwritten.
 */
tm_status tm_colsum(const float *X, int64_t ldx, int64_t M, int64_t N, float *c, void *workspace,
                    size_t ws_bytes, int32_t TM, int32_t TN, tm_variant variant, uint32_t flags,
                    tm_stream_t stream);

/*
 * tm_rowmax_masked -- m[i] = max_{j < N} S[i, j] over ragged BC-column tiles.
 * "Slicing, bounds and masking", "Reductions over a ragged tile": whole tiles
 * are read unmasked; the remainder tile's missing columns read 0 and are then
 * replaced by where(iota < N - kt, s, fill).  fill = TM_FILL_NEG_INF gives the
 * true row maximum (the fill can never win); TM_FILL_ZERO skips the
 * where step and reproduces the pitfall (max(0, true max) when N % BC != 0).
 * N == 0 gives -inf.  max ignores a NaN operand unless both are NaN.
 *   S, lds   device input [M, lds]     m   device output, M floats
 *   BR       rows per block (one warp per row): 1, 2, 4, 8, 16, 32
 *   BC       columns per tile: 16, 32, 64, 128, 256, 512
 *   flags    TM_ALIGNED (M % BR == 0, N % BC == 0: no remainder, no row mask),
 *            TM_PATH_SCALAR, TM_PATH_VEC, TM_PDL
 * Errors: INVALID_ARG, UNSUPPORTED_TILE, MISALIGNED, BROKEN_PROMISE, CUDA.
 */
tm_status tm_rowmax_masked(const float *S, int64_t lds, int64_t M, int64_t N, float *m, int32_t BR,
                           int32_t BC, tm_fill fill, uint32_t flags, tm_stream_t stream);

/*
 * tm_softmax_rowstats -- the softmax row statistics over ragged BC-column
 * tiles: m[i] = max_{j < N} S[i, j] and l[i] = sum_{j < N} exp(S[i, j] - m[i]).
 * "Slicing, bounds and masking", "Reductions over a ragged tile": the softmax
 * is the second reduction a zero fill breaks; the remainder tile takes the
 * masked load and the where(iota < N - kt, s, -inf) step, so padding is never
 * the maximum and adds exp(-inf) = 0 to l.  TM_FILL_ZERO skips the where step
 * (the pitfall: padding zeros enter both m and l).  N == 0 gives m = -inf and
 * l = 0.  fp32 with CUDA's expf; l is within 1e-5 relative of the exact sum,
 * m is exact.
 *   S, lds   device input [M, lds]     m, l   device outputs, M floats each
 *   BR, BC, flags   as tm_rowmax_masked
 * Errors: INVALID_ARG, UNSUPPORTED_TILE, MISALIGNED, BROKEN_PROMISE, CUDA.
 */
tm_status tm_softmax_rowstats(const float *S, int64_t lds, int64_t M, int64_t N, float *m, float *l,
                              int32_t BR, int32_t BC, tm_fill fill, uint32_t flags, tm_stream_t stream);

/*
 * tm_colsum_noalloc -- tm_colsum for callers that cannot allocate device
 * memory (no counterpart in the pages: a convenience of this library).  Code
 * running inside another framework that owns all device memory, under a fixed
 * memory budget, or on a path where cudaMalloc's implicit device-wide
 * synchronization is not allowed can still take column sums: the partial sums
 * live in a static device array of TM_NOALLOC_SCRATCH_BYTES that the library
 * holds on every GPU that loads it, for the life of the process.  This call
 * allocates nothing and calls no allocating routine.
 *   Same arguments, variants, flags, results and errors as tm_colsum, minus
 *   the workspace.  Returns TM_ERR_WORKSPACE (nothing launched) when the
 *   arguments need more scratch than TM_NOALLOC_SCRATCH_BYTES, i.e. when
 *   tm_colsum_workspace_bytes(M, N, TM, TN, variant) exceeds it.
 *   TM_VAR_CLUSTER and TM_VAR_STAGED need no scratch and so run at any
 *   shape.
 *   The first call on each device that needs scratch looks up the array's
 *   device address with cudaGetSymbolAddress while that device is current,
 *   and keeps it for the life of the process; make that first call before
 *   any stream capture.  The cached address (like the status word's) belongs
 *   to the device's primary context: the library assumes the runtime API's
 *   primary contexts and no cudaDeviceReset while it is loaded.
 *   All calls share the one array: calls whose kernels may overlap on the GPU
 *   (different streams, no ordering between them) race and give wrong sums;
 *   serialize them.  The array keeps the last call's partial sums; every word
 *   a call reads it wrote first, so no clearing is needed.
 */
#define TM_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20) /* 8 MiB per device */
tm_status tm_colsum_noalloc(const float *X, int64_t ldx, int64_t M, int64_t N, float *c, int32_t TM,
                            int32_t TN, tm_variant variant, uint32_t flags, tm_stream_t stream);

/*
 * tm_gemm -- the fp32 gemm of the pages' @aligned example:
 *   C = alpha * (A B) + beta * C     A [M, K], B [K, N], C [M, N], row-major.
 * "@aligned", the gemm example (acc += dot(a, b) over TILE_K-wide tiles of K,
 * then alpha * acc + beta * c_old per TILE_M x TILE_N output tile, with and
 * without the promise); "Slicing, bounds and masking", "Loops over a dynamic
 * extent" (K known only at run time: whole tiles plus one masked remainder
 * whose missing columns read 0).
 * On GB300 the contraction runs on the tensor cores (tcgen05, tf32 inputs,
 * fp32 accumulation in tensor memory).  By default each operand is split as
 * x = hi + lo (both tf32) and the product takes hi*hi + hi*lo + lo*hi, which
 * keeps fp32-level accuracy; TM_GEMM_TF32 keeps only hi*hi (tf32 accuracy,
 * about 3x the speed).  A first pass writes the split operands, K-major and
 * zero-padded to whole tiles, into the caller's workspace; the zero padding
 * is the masked remainder tile's fill, so the tensor-core loop itself runs
 * over whole tiles only.  When the tiles fill at most half of the last round
 * of CTAs (pairs) and K is long enough, each of that round's tiles is cut
 * along K into parts run side by side (split-K): the later parts go to the
 * workspace and the CTA that ran the first part adds them in K order before
 * the output, so results stay deterministic.  beta == 0 does not read C (NaN
 * in C stays out).
 * K == 0 gives C = beta * C.
 *   A, lda   device input [M, lda]    B, ldb   device input [K, ldb]
 *   C, ldc   device in/out [M, ldc]; C must not overlap A, B or the workspace
 *   TM, TN, TK   the output tile and K tile: TM = 128 (one CTA per tile) or
 *            256 (a pair of CTAs on neighbouring SMs shares each tile: each
 *            stages 128 rows of A and half of the B tile, cutting operand
 *            traffic per flop by a third), TN = 128 or 256, TK = 16 or 32 (the
 *            K width of one pipeline stage: TK 16 gives twice as many,
 *            half-size stages in the same shared memory)
 *   flags    TM_ALIGNED (M % TM == 0, N % TN == 0, K % TK == 0: the output
 *            tiles store without masks), TM_GEMM_TF32
 *   The output moves through TMA copies when C is 16-byte aligned and
 *   ldc % 4 == 0 and N % 4 == 0, else by direct stores; either way nothing
 *   outside [M, N] (the ld gap included) is written.
 *   workspace, ws_bytes   device scratch of at least
 *            tm_gemm_workspace_bytes(M, N, K, TN) bytes, 1024-byte aligned,
 *            overlapping no operand; contents on entry do not matter.  It holds
 *            the split operands and the split-K partial tiles, and is in use
 *            until the call's kernels finish on `stream`: calls that may run
 *            at the same time need separate workspaces.
 * Accuracy: |C - exact| <= (3*2^-22 + 3*K*2^-23) * |alpha| * sum_k |a_ik||b_kj|
 *   + 2^-23 * (|alpha * (A B)_ij| + |beta c_ij|) (3xTF32; tensor-core
 *   accumulation is taken as fp32 with truncation, one rounding per k, which
 *   also covers the few additions of split-K parts).  Integer-valued inputs
 *   whose partial sums stay below 2^24 give exact results.
 * Errors: INVALID_ARG (extents, NULL, ld, overlap, unknown flag, a padded
 *   extent or the tile count beyond 2^31 - 1), UNSUPPORTED_TILE, MISALIGNED
 *   (a pointer not 4-byte aligned), BROKEN_PROMISE (host check of
 *   TM_ALIGNED), WORKSPACE, CUDA;
 *   TIMEOUT through tm_check if the tensor-core pipeline stalls (its waits
 *   are bounded; C is then left partly written).
 */
#define TM_GEMM_TF32 0x100u
size_t tm_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t TN);
tm_status tm_gemm(const float *A, int64_t lda, const float *B, int64_t ldb, float *C, int64_t ldc,
                  int64_t M, int64_t N, int64_t K, float alpha, float beta, int32_t TM, int32_t TN,
                  int32_t TK, uint32_t flags, void *workspace, size_t ws_bytes, tm_stream_t stream);

/*
 * tm_check -- synchronize `stream`, then read and clear this device's status
 * word.  Returns TM_ERR_BROKEN_PROMISE if a kernel's entry check found the
 * aligned promise broken (that kernel stored nothing), TM_ERR_MISALIGNED if it
 * found a misaligned pointer or ld, TM_ERR_TIMEOUT if a bounded wait gave up,
 * TM_ERR_CUDA if the stream reports a CUDA error, else TM_OK.
 */
tm_status tm_check(tm_stream_t stream);

/*
 * Diagnostic entry points (used by the test suite; safe for any caller).
 *
 * tm_tile_walk_probe -- runs, on the device, the tile-walk planner every
 * kernel uses for a loop over a runtime extent K in steps of T ("Slicing,
 * bounds and masking", "Loops over a dynamic extent") and writes four int64 to
 * the DEVICE pointer out4: whole (unmasked) tiles, masked tiles (0 or 1),
 * columns in the masked tile, total iterations.
 * Errors: INVALID_ARG (K < 0, T <= 0, out4 NULL), CUDA.
 */
tm_status tm_tile_walk_probe(int64_t K, int32_t T, int64_t *out4, tm_stream_t stream);

/*
 * tm_wait_timeout_probe -- exercises the failure path of the pipelined kernels
 * (the gemm and the staged column sum), which has no counterpart in the
 * pages: one thread waits, with the same bounded mbarrier wait those kernels
 * use, on a barrier that nothing arrives at.  After the limit (about 2e9 SM
 * cycles, ~1 s) the wait gives up, the kernel records the timeout in the
 * device's status word and ends normally; the next tm_check returns
 * TM_ERR_TIMEOUT and the context stays usable.
 * Errors: CUDA.
 */
tm_status tm_wait_timeout_probe(tm_stream_t stream);

/*
 * tm_read_probe -- the plain streaming read the reductions are measured
 * against ("Memory Coalescing and Tensor Layout", "What it actually costs":
 * the row walk's bandwidth is the ceiling to compare any kernel with).  The n
 * floats of x (n % 4 == 0, x 16-byte aligned) are read once by a flat grid of
 * 256-thread blocks, each thread issuing per_thread (1, 2, 4, 8 or 16)
 * independent 16-byte loads together; block b writes out[b], the fp32 sum of
 * elements [b*1024*per_thread, (b+1)*1024*per_thread) in a fixed order.  out
 * holds tm_read_probe_blocks(n, per_thread) floats and must not overlap x.
 * tm_read_probe_blocks returns -1 for a bad n or per_thread.
 * Errors: INVALID_ARG, MISALIGNED, CUDA.
 */
int64_t tm_read_probe_blocks(int64_t n, int32_t per_thread);
tm_status tm_read_probe(const float *x, int64_t n, float *out, int32_t per_thread, tm_stream_t stream);

/*
 * tm_read_probe_fixed -- the same plain read with every block's share fixed
 * before it starts: the floor of a one-pass walk that cannot hand work from a
 * slow block to a fast one (the column sums' one-pass forms give each CTA a
 * fixed part of a strip; "Memory Coalescing and Tensor Layout", "Seeing it in
 * a real kernel").  Exactly `blocks` blocks (1 .. 65535) of 256 threads; with
 * share = tm_read_probe_fixed_share(n, blocks) floats (a multiple of 8192:
 * each step of a block is 256 threads x 8 16-byte loads), block b sums floats
 * [b*share, min((b+1)*share, n)) of x into out[b] in a fixed order (0 for a
 * block wholly past n).  n % 4 == 0, x 16-byte aligned, out holds `blocks`
 * floats and must not overlap x.  tm_read_probe_fixed_share returns -1 for a
 * bad n or blocks.  Errors: INVALID_ARG, MISALIGNED, CUDA.
 */
int64_t tm_read_probe_fixed_share(int64_t n, int32_t blocks);
tm_status tm_read_probe_fixed(const float *x, int64_t n, float *out, int32_t blocks, tm_stream_t stream);

/*
 * tm_scale2d_unchecked -- tm_scale2d on its TM_ALIGNED path without the host
 * promise check, so the kernel's own entry check is what stands between a
 * broken promise and the tensor's end.  With a broken promise no element is
 * read or written and the next tm_check returns TM_ERR_BROKEN_PROMISE (or
 * TM_ERR_MISALIGNED).  Still validates everything except the promise and the
 * alignment.  Tiles as tm_scale2d.
 */
tm_status tm_scale2d_unchecked(const float *X, int64_t ldx, float *Y, int64_t ldy, int64_t M,
                               int64_t N, float alpha, int32_t TM, int32_t TN, tm_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* TM_H_ */
