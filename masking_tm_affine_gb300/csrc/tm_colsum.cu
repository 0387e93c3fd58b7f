// tm_colsum.cu -- c[j] = sum_i X[i, j]: the column walk and its fixes.
//
// Source: "Memory Coalescing and Tensor Layout".  "What it actually costs":
// the column-order walk of a row-major matrix (offsets rows*COLS + col, 65536
// programs of 256 elements over 4096 x 4096, neighbouring programs on
// neighbouring columns) moves the row walk's bytes yet ran 2.4x slower
// on the page's GPU.  "Seeing it in a real kernel": the way out is to load a
// tile once into fast memory and read it there in any order.
//
// Variants:
//   NAIVE     -- the page's walk: a 256-lane program per (256-row block,
//                column); lanes step down a column, ld apart.  Kept as the foil.
//                Its partials go to the workspace and colsum_finish adds them
//                (two passes).
//   REGDIRECT -- lanes over columns: a warp reads a contiguous row segment of a
//                TN-column strip with 16-byte loads and walks down the rows,
//                accumulating in registers, one block per (strip, row chunk);
//                the units' partials go to the workspace, strip-major, and
//                colsum_finish_strips adds each column's partials in ascending
//                chunk order (a fixed order: the same bits run to run) and
//                drops their lines from L2 without writing them back.  A strip
//                of one chunk writes c itself, with no second pass.
//   CLUSTER   -- REGDIRECT's layout in one pass: the CTAs of a thread-block
//                cluster split a strip's row tiles, and their partials meet in
//                distributed shared memory (cluster_push_partials); no
//                workspace.
//   STAGED    -- the page's fix on GB300 hardware: the TMA engine copies
//                TM x TN tiles into a ring of shared-memory stages (mbarrier
//                completion, bounded waits); threads read the columns back out
//                of shared memory.  Ragged edges come free: TMA fills
//                out-of-bounds elements with 0, the masked-load value of
//                "Slicing, bounds and masking" ("Masking").  The cluster
//                form's grid and end: one pass, the same bits as CLUSTER.
//   AUTO      -- CLUSTER when every cluster fits on the GPU at once, else
//                REGDIRECT.
//
// (A one-pass REGDIRECT, in which the block that brought a strip's last
// partial added them all, measured slower: every block then waited for a
// counter round trip before it could leave its SM.)
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "tm_host.h"

namespace libtm {
namespace {

constexpr int kNaiveRows = 256;        // the page's program length
constexpr int64_t kTargetUnits = 8192; // (strip, chunk) work units aimed for: one block each
constexpr int64_t kMinChunkRows = 64;  // rows per chunk at least: 8 row lanes x 8 loads in flight
constexpr int kFinishPG = 8;           // chunk groups per column in the finish pass

struct ColPlan {
    int64_t S;      // column strips: ceil(N / TN)
    int64_t RT;     // row tiles: ceil(M / TM)
    int64_t CT;     // row tiles per chunk
    int64_t P;      // chunks (partials per column)
    int64_t units;  // S * P
};

ColPlan plan_chunks(int64_t M, int64_t N, int64_t TM, int64_t TN)
{
    ColPlan pl;
    pl.S = (N + TN - 1) / TN;
    pl.RT = (M + TM - 1) / TM;
    int64_t P = (kTargetUnits + pl.S - 1) / pl.S;
    if (P > pl.RT) P = pl.RT;
    if (P < 1) P = 1;
    pl.CT = (pl.RT + P - 1) / P;
    const int64_t min_ct = (kMinChunkRows + TM - 1) / TM;
    if (pl.CT < min_ct) pl.CT = min_ct;
    pl.P = (pl.RT + pl.CT - 1) / pl.CT;
    pl.units = pl.S * pl.P;
    return pl;
}

// Scratch of REGDIRECT and STAGED: [S][P][TN] partials; none when each strip
// is a single chunk (the unit's sums are c itself).
int64_t partial_bytes(const ColPlan &pl, int64_t TN)
{
    return pl.P <= 1 ? 0 : pl.S * pl.P * TN * (int64_t)sizeof(float);
}

struct ColArgs {
    const float *X;
    int64_t ldx, M, N;
    float *part;  // [S][P][TN] partial sums, strip-major (unused when P == 1)
    float *c;     // [N] the result
    int64_t S, RT, CT, P, units;
    int TM;
    unsigned *status;
};

__device__ __forceinline__ void report(unsigned *status, unsigned bit)
{
    atomicOr(status, bit);
}

// The end of unit (strip s, chunk p): red[0 .. RL) holds each row lane's
// column sums.  Threads 0 .. TN/4 - 1 add the row lanes in order, 4 columns
// each, into c when every strip is one chunk, else into the unit's TN-wide
// partial (columns past N hold 0 there).
template <int TN, int RL>
__device__ __forceinline__ void store_unit(const ColArgs &a, int64_t s, int64_t p, const float (*red)[TN])
{
    const int t = threadIdx.x;
    if (t >= TN / 4) return;
    float4 v = *reinterpret_cast<const float4 *>(&red[0][t * 4]);
#pragma unroll
    for (int q = 1; q < RL; ++q) {
        const float4 w = *reinterpret_cast<const float4 *>(&red[q][t * 4]);
        v.x += w.x;
        v.y += w.y;
        v.z += w.z;
        v.w += w.w;
    }
    pdl_wait();  // the loads may run ahead of the previous kernel, the stores may not
    if (a.P == 1) {
        const float tv[4] = {v.x, v.y, v.z, v.w};
        const int64_t j = s * TN + t * 4;
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (j + e < a.N) a.c[j + e] = tv[e];
    } else {
        const u32x4 w = {{as_u(v.x), as_u(v.y), as_u(v.z), as_u(v.w)}};
        st_v4(a.part + (s * a.P + p) * TN + t * 4, w);
    }
}

// ------------------------------------------------------------------ finish (strip-major partials)
// c[j] = sum over chunks p (ascending) of REGDIRECT's partials.
// A block takes 32 columns: 8 lanes of 4 columns by 32 row lanes; row lane r
// adds chunks r, r + 32, r + 64, ..., issuing its loads together (one L2 round
// trip for up to 128 chunks), then the 32 lane sums are added in order.  The
// partials are read once: with 128-byte aligned lines they are then dropped
// from L2, so they never cost a DRAM write.
constexpr int kFinCL = 8, kFinRL = 32;
__global__ void __launch_bounds__(256, 6) colsum_finish_strips(const float *__restrict__ part, int64_t P, int64_t TN,
                                                            int64_t N, float *__restrict__ c, int discard)
{
    __shared__ float4 lane[kFinRL][kFinCL];
    pdl_trigger();  // a dependent next call may launch once every block has started
    pdl_wait();     // launched as a dependent of the partial-sum pass: its writes first
    const int cl = threadIdx.x % kFinCL, r = threadIdx.x / kFinCL;
    const int64_t blocks = (N + 31) / 32;
    for (int64_t b = blockIdx.x; b < blocks; b += gridDim.x) {
        const int64_t j0 = b * 32, s = j0 / TN;
        const float *col = part + s * P * TN + (j0 - s * TN);  // this block's 32 columns of chunk 0
        // a strip's partials span P * TN < 2^23 floats (P > 1 only below 8192
        // strips, and S * P stays under 16384 units): 32-bit offsets suffice
        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        const uint32_t step = kFinRL * (uint32_t)TN;       // from chunk p to chunk p + 32
        uint32_t off = (uint32_t)r * (uint32_t)TN + cl * 4;  // chunk r, this lane's 4 columns
        int n = r < P ? (int)((P - 1 - r) / kFinRL) + 1 : 0;  // chunks of this row lane
        for (; n >= 4; n -= 4, off += 4 * step) {
            const u32x4 w0 = ld_l2_v4(col + off), w1 = ld_l2_v4(col + off + step);
            const u32x4 w2 = ld_l2_v4(col + off + 2 * step), w3 = ld_l2_v4(col + off + 3 * step);
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[e] += as_f(w0.v[e]);
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[e] += as_f(w1.v[e]);
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[e] += as_f(w2.v[e]);
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[e] += as_f(w3.v[e]);
        }
        for (; n > 0; --n, off += step) {
            const u32x4 w = ld_l2_v4(col + off);
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[e] += as_f(w.v[e]);
        }
        lane[r][cl] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        __syncthreads();  // every partial of these columns has been read
        if (r == 0) {
            float4 t = lane[0][cl];
#pragma unroll 8
            for (int q = 1; q < kFinRL; ++q) {
                const float4 v = lane[q][cl];
                t.x += v.x;
                t.y += v.y;
                t.z += v.z;
                t.w += v.w;
            }
            const float tv[4] = {t.x, t.y, t.z, t.w};
            const int64_t j = j0 + cl * 4;
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (j + e < N) c[j + e] = tv[e];
        }
        if (discard)  // one 128-byte line per chunk: nothing reads it again
            for (int64_t q = threadIdx.x; q < P; q += 256) discard_l2_line(col + q * TN);
        __syncthreads();
    }
}

// ------------------------------------------------------------------ NAIVE
__global__ void __launch_bounds__(kNaiveRows) colsum_naive(const float *__restrict__ X, int64_t ldx, int64_t M,
                                                           int64_t N, float *__restrict__ part, int64_t npad,
                                                           int64_t programs)
{
    pdl_trigger();  // the finish may launch once every block has started
    __shared__ float warp_sums[kNaiveRows / 32];
    for (int64_t pid = blockIdx.x; pid < programs; pid += gridDim.x) {
        const int64_t col = pid % N;  // neighbouring programs read neighbouring columns
        const int64_t rb = pid / N;
        const int64_t row = rb * kNaiveRows + threadIdx.x;
        float v = row < M ? as_f(ld_nc_b32(X + row * ldx + col)) : 0.0f;  // lane stride: ld words
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if ((threadIdx.x & 31) == 0) warp_sums[threadIdx.x >> 5] = v;
        __syncthreads();
        if (threadIdx.x == 0) {
            float t = warp_sums[0];
#pragma unroll
            for (int w = 1; w < kNaiveRows / 32; ++w) t += warp_sums[w];
            pdl_wait();  // the loads may run ahead of the previous kernel, the stores may not
            part[rb * npad + col] = t;
        }
        __syncthreads();
    }
    pdl_wait();  // threads that stored nothing: the grid completes only after the one before it
}

// ------------------------------------------------------------------ finish
// c[j] = sum over chunks p (ascending) of part[p][j].  A block covers 32
// columns; its 8 warps each add a contiguous group of chunks, and the groups
// are added in order.
__global__ void __launch_bounds__(256) colsum_finish(const float *__restrict__ part, int64_t npad, int64_t P,
                                                     int64_t N, float *__restrict__ c)
{
    __shared__ float grp[kFinishPG][33];
    pdl_trigger();  // a dependent next call may launch once every block has started
    pdl_wait();     // launched as a dependent of the partial-sum pass: its writes first
    const int cx = threadIdx.x & 31, py = threadIdx.x >> 5;
    const int64_t per = (P + kFinishPG - 1) / kFinishPG;
    const int64_t p_lo = py * per;
    const int64_t p_hi = p_lo + per < P ? p_lo + per : P;
    for (int64_t j0 = (int64_t)blockIdx.x * 32; j0 < N; j0 += (int64_t)gridDim.x * 32) {
        const int64_t j = j0 + cx;
        float s = 0.0f;
        if (j < N) {
            int64_t p = p_lo;
            for (; p + 4 <= p_hi; p += 4) {
                const float a0 = part[(p + 0) * npad + j], a1 = part[(p + 1) * npad + j];
                const float a2 = part[(p + 2) * npad + j], a3 = part[(p + 3) * npad + j];
                s += a0;
                s += a1;
                s += a2;
                s += a3;
            }
            for (; p < p_hi; ++p) s += part[p * npad + j];
        }
        grp[py][cx] = s;
        __syncthreads();
        if (py == 0 && j < N) {
            float t = grp[0][cx];
#pragma unroll
            for (int q = 1; q < kFinishPG; ++q) t += grp[q][cx];
            c[j] = t;
        }
        __syncthreads();
    }
}

// ------------------------------------------------------------------ REGDIRECT
// Four blocks per SM: room for all UNR vector loads of a batch in registers
// (at eight blocks and 32 registers part of every batch was serialised).
template <int TN, bool VEC, bool ALIGNED>
__global__ void __launch_bounds__(kThreads, 4) colsum_regdirect(const ColArgs a)
{
    constexpr int EW = VEC ? 4 : 1;
    constexpr int CL = TN / EW;           // column lanes
    constexpr int RL = kThreads / CL;     // row lanes
    constexpr int UNR = 8;                // rows in flight per thread
    static_assert(CL * RL == kThreads, "strip does not fit the block");
    __shared__ __align__(16) float red[RL][TN];
    pdl_trigger();  // the finish may launch once every block has started

    if constexpr (ALIGNED) {
        const bool whole = (a.M % a.TM == 0) && (a.N % TN == 0);
        const bool grid_ok = !VEC || ((a.ldx % 4 == 0) && (reinterpret_cast<uintptr_t>(a.X) & 15) == 0);
        if (!whole || !grid_ok) {
            if (blockIdx.x == 0 && threadIdx.x == 0) report(a.status, whole ? kStatusMisaligned : kStatusBrokenPromise);
            pdl_wait();
            return;
        }
    }
    const int cl = threadIdx.x % CL, rl = threadIdx.x / CL;
    const int64_t CR = a.CT * a.TM;  // rows per chunk
    for (int64_t u = blockIdx.x; u < a.units; u += gridDim.x) {
        const int64_t s = u % a.S, p = u / a.S;
        const int64_t j = s * TN + (int64_t)cl * EW;
        const bool col_in = ALIGNED || j < a.N;  // column mask of a ragged last strip
        const int64_t r0 = p * CR;
        const int64_t r1 = r0 + CR < a.M ? r0 + CR : a.M;  // rows past M are not visited
        float acc[EW];
#pragma unroll
        for (int e = 0; e < EW; ++e) acc[e] = 0.0f;
        if (col_in) {
            const float *xp = a.X + j;
            int64_t row = r0 + rl;
            for (; row + (UNR - 1) * RL < r1; row += UNR * RL) {
                uint32_t v[UNR][EW];
#pragma unroll
                for (int q = 0; q < UNR; ++q) {
                    const float *ptr = xp + (row + (int64_t)q * RL) * a.ldx;
                    if constexpr (VEC) {
                        u32x4 w = ld_nc_v4(ptr);
#pragma unroll
                        for (int e = 0; e < 4; ++e) v[q][e] = w.v[e];
                    } else {
                        v[q][0] = ld_nc_b32(ptr);
                    }
                }
#pragma unroll
                for (int q = 0; q < UNR; ++q)
#pragma unroll
                    for (int e = 0; e < EW; ++e) acc[e] += as_f(v[q][e]);
            }
            for (; row < r1; row += RL) {
                const float *ptr = xp + row * a.ldx;
                if constexpr (VEC) {
                    u32x4 w = ld_nc_v4(ptr);
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[e] += as_f(w.v[e]);
                } else {
                    acc[0] += as_f(ld_nc_b32(ptr));
                }
            }
        }
#pragma unroll
        for (int e = 0; e < EW; ++e) red[rl][cl * EW + e] = acc[e];
        __syncthreads();
        store_unit<TN, RL>(a, s, p, red);
        __syncthreads();
    }
    pdl_wait();  // threads that stored nothing: the grid completes only after the one before it
}

// The end of both one-pass forms.  Every CTA holds the TN partial sums of its
// rows of the strip; rank r owns columns [r*TN/CS, (r+1)*TN/CS) and adds the
// CS partials of each in rank order from 0 (the order one thread adding all
// of them would take).  The partials travel by push: thread (q, k) of each
// CTA stores its partial of rank q's column k straight into rank q's inbox
// with st.async, and every such store counts its 4 bytes on that inbox's
// mbarrier, so an owner starts adding as soon as its TN floats have landed,
// with no cluster barrier and no round trip of remote reads before it.
template <int TN, int CS>
struct Inbox {
    uint64_t bar;          // counts TN * 4 bytes in, once per launch
    float v[CS][TN / CS];  // v[q][k]: rank q's partial of this rank's column k
};

// At kernel start, in every thread (after any early return, which all CTAs
// take together): thread 0 sets the inbox up, then every thread arrives at
// the cluster barrier that cluster_push_partials waits on before its first
// remote store, so no store can reach an inbox not yet set up.
template <int TN, int CS>
__device__ __forceinline__ void inbox_open(Inbox<TN, CS> &in)
{
    if (threadIdx.x == 0) {
        const uint32_t bar = smem_u32(&in.bar);
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar) : "memory");
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                     "r"((uint32_t)(TN * sizeof(float)))
                     : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

// part[0 .. TN) holds this CTA's partials (written before the call by some
// threads; every thread calls).  Pushes them, waits (bounded) for its own
// inbox, adds and writes its columns of c.  The closing cluster barrier is
// passed only once every CTA's inbox is full, so no store is still in flight
// to a CTA that leaves.  A wait that gives up records kStatusTimeout and
// writes nothing.
template <int TN, int CS>
__device__ __forceinline__ void cluster_push_partials(const float *part, Inbox<TN, CS> &in, float *c, int64_t N,
                                                      int64_t strip, unsigned *status)
{
    constexpr int SL = TN / CS;  // columns per rank
    static_assert(SL >= 1 && SL * CS == TN, "the ranks split the strip evenly");
    __syncthreads();                                                       // part[] complete
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");  // every peer's inbox is set up
    const uint32_t me = cluster_rank();
    if (threadIdx.x < TN) {
        const uint32_t q = threadIdx.x / SL, k = threadIdx.x % SL;
        const uint32_t dst = cluster_addr(smem_u32(&in.v[me][k]), q);
        const uint32_t bar = cluster_addr(smem_u32(&in.bar), q);
        asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(dst),
                     "r"(as_u(part[q * SL + k])), "r"(bar)
                     : "memory");
    }
    const bool ok = mbar_wait_bounded(smem_u32(&in.bar), 0);
    if (!ok && threadIdx.x == 0) report(status, kStatusTimeout);
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");  // this inbox is full
    if (ok && threadIdx.x < SL) {
        float t = 0.0f;
#pragma unroll
        for (int q = 0; q < CS; ++q) t += in.v[q][threadIdx.x];
        const int64_t col = strip * TN + (int64_t)me * SL + threadIdx.x;
        pdl_wait();  // the loads may run ahead of the previous kernel, the stores may not
        if (col < N) c[col] = t;
    }
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");  // every inbox is full
}

// ------------------------------------------------------------------ CLUSTER (one pass)
// The register-direct layout, with the partial sums reduced on chip: the CS
// CTAs of a cluster split the rows of one TN-column strip, each adds its rows
// into a TN-wide partial in its shared memory, and the CTAs then push each
// rank its slice of the columns over distributed shared memory, where the
// rank adds the CS partials in rank order and writes them to c (see
// cluster_push_partials).  No workspace and no second pass.  IT is the type of element
// offsets: uint32_t when (M + 128) * ldx fits 32 bits (host-checked), which
// saves registers.  Four CTAs per SM, each free to hold all UNR loads of a
// batch in flight (at eight CTAs, capped at 32 registers, the compiler
// serialised part of every batch: [8192, 8192] 41.1 against 39.7 us).
template <int TN, int CS, bool VEC, bool ALIGNED, typename IT>
__global__ void __launch_bounds__(kThreads, 4) colsum_cluster(const ColArgs a, int64_t rows_per_cta)
{
    constexpr int EW = VEC ? 4 : 1;
    constexpr int CL = TN / EW;           // column lanes
    constexpr int RL = kThreads / CL;     // row lanes
    constexpr int UNR = 8;                // rows in flight per thread
    static_assert(CL * RL == kThreads && TN <= kThreads, "strip does not fit the block");
    __shared__ float red[RL][TN];
    __shared__ float part[TN];

    pdl_trigger();
    if constexpr (ALIGNED) {
        // a pure function of the arguments: every CTA of every cluster returns
        // together, so no CTA is left waiting at a cluster barrier
        const bool whole = (a.M % a.TM == 0) && (a.N % TN == 0);
        const bool grid_ok = !VEC || ((a.ldx % 4 == 0) && (reinterpret_cast<uintptr_t>(a.X) & 15) == 0);
        if (!whole || !grid_ok) {
            if (blockIdx.x == 0 && threadIdx.x == 0) report(a.status, whole ? kStatusMisaligned : kStatusBrokenPromise);
            pdl_wait();
            return;
        }
    }
    __shared__ Inbox<TN, CS> inbox;
    inbox_open(inbox);
    const int cl = threadIdx.x % CL, rl = threadIdx.x / CL;
    float acc[EW];
#pragma unroll
    for (int e = 0; e < EW; ++e) acc[e] = 0.0f;
    {
        const int64_t j = (int64_t)(blockIdx.x / CS) * TN + (int64_t)cl * EW;
        const int64_t r0 = (int64_t)cluster_rank() * rows_per_cta;
        if ((ALIGNED || j < a.N) && r0 < a.M) {
            const float *xp = a.X + j;
            const IT ld = (IT)a.ldx;
            const IT nrows = (IT)((r0 + rows_per_cta < a.M ? r0 + rows_per_cta : a.M) - r0);
            IT off = ((IT)r0 + (IT)rl) * ld;        // element offset of this lane's next row
            const IT end = ((IT)r0 + nrows) * ld;   // one row past the CTA's last
            const IT step = (IT)RL * ld;
            for (; off + (IT)(UNR - 1) * step < end; off += (IT)UNR * step) {
                uint32_t v[UNR][EW];
#pragma unroll
                for (int q = 0; q < UNR; ++q) {
                    const float *ptr = xp + (off + (IT)q * step);
                    if constexpr (VEC) {
                        u32x4 w = ld_nc_v4(ptr);
#pragma unroll
                        for (int e = 0; e < 4; ++e) v[q][e] = w.v[e];
                    } else {
                        v[q][0] = ld_nc_b32(ptr);
                    }
                }
#pragma unroll
                for (int q = 0; q < UNR; ++q)
#pragma unroll
                    for (int e = 0; e < EW; ++e) acc[e] += as_f(v[q][e]);
            }
            for (; off < end; off += step) {
                const float *ptr = xp + off;
                if constexpr (VEC) {
                    u32x4 w = ld_nc_v4(ptr);
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[e] += as_f(w.v[e]);
                } else {
                    acc[0] += as_f(ld_nc_b32(ptr));
                }
            }
        }
    }
#pragma unroll
    for (int e = 0; e < EW; ++e) red[rl][cl * EW + e] = acc[e];
    __syncthreads();
    if (rl == 0) {
#pragma unroll
        for (int e = 0; e < EW; ++e) {
            float t = red[0][cl * EW + e];
#pragma unroll
            for (int q = 1; q < RL; ++q) t += red[q][cl * EW + e];
            part[cl * EW + e] = t;
        }
    }
    cluster_push_partials(part, inbox, a.c, a.N, (int64_t)(blockIdx.x / CS), a.status);
    pdl_wait();  // threads that stored nothing: the grid completes only after the one before it
}

// ------------------------------------------------------------------ STAGED (TMA)
// The page's fix on GB300: tiles are loaded once into fast on-chip memory and
// read there in any order.  The CS CTAs of a cluster split the row tiles of
// one TN-column strip; each streams its TM x TN tiles through a ring of
// `stages` shared-memory stages filled by the TMA engine (one thread issues
// cp.async.bulk.tensor copies into this CTA's own shared memory, an mbarrier
// per stage counts the bytes in), and the threads read columns back out: lane
// (cl, rl) adds rows rl, rl + RL, ... of every tile, in order.  TMA fills rows
// past M and columns past N with 0, the masked-load value of "Slicing, bounds
// and masking" ("Masking").  The CTAs' partials then meet over distributed
// shared memory as in the cluster form (cluster_push_partials): one pass, no
// workspace.  With the same tile-aligned row split, lanes and order as
// colsum_cluster's 16-byte path, the two give the same bits.  Every wait is
// bounded; a CTA whose wait gives up records TM_ERR_TIMEOUT, drains the
// copies it started (bounded) and still takes its part in the cluster's end,
// so its peers are not left waiting.
template <int TN, int CS, bool ALIGNED>
__global__ void __launch_bounds__(kThreads) colsum_staged(const __grid_constant__ CUtensorMap tmap, const ColArgs a,
                                                          int TM, int64_t tiles_per_cta, int stages)
{
    constexpr int CL = TN / 4;         // column lanes, 4 columns each
    constexpr int RL = kThreads / CL;  // row lanes
    extern __shared__ __align__(128) unsigned char smem[];
    const int tile = TM * TN;          // floats per stage
    float *tiles = reinterpret_cast<float *>(smem);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)stages * tile * sizeof(float));
    __shared__ __align__(16) float red[RL][TN];
    __shared__ float part[TN];
    __shared__ int abort_flag;

    pdl_trigger();
    if constexpr (ALIGNED) {
        // a pure function of the arguments: every CTA of every cluster returns
        // together, so no CTA is left waiting at a cluster barrier
        const bool whole = (a.M % TM == 0) && (a.N % TN == 0);
        if (!whole) {
            if (blockIdx.x == 0 && threadIdx.x == 0) report(a.status, kStatusBrokenPromise);
            pdl_wait();
            return;
        }
    }
    const int tid = threadIdx.x;
    const int cl = tid % CL, rl = tid / CL;
    const int64_t strip = blockIdx.x / CS;
    const int64_t t0 = (int64_t)cluster_rank() * tiles_per_cta;  // this CTA's first row tile
    const int64_t t1 = t0 + tiles_per_cta < a.RT ? t0 + tiles_per_cta : a.RT;
    const int n = t1 > t0 ? (int)(t1 - t0) : 0;

    __shared__ Inbox<TN, CS> inbox;
    // the tiles are read once: evict-first, so that loading them does not
    // push out (and force the write-back of) lines an earlier kernel left
    // dirty in L2 ([8192, 8192] after a 512 MiB write: 49.8 against 58.0 us)
    const uint64_t pol = tid == 0 ? l2_evict_first_policy() : 0;
    if (tid == 0) {
        abort_flag = 0;
        for (int st = 0; st < stages; ++st)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&full[st])) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    inbox_open(inbox);
    __syncthreads();
    auto issue = [&](int k) {
        if (k >= n) return;
        const int st = k % stages;
        const uint32_t bar = smem_u32(&full[st]);
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                     "r"((uint32_t)(tile * sizeof(float)))
                     : "memory");
        asm volatile(
            "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
            " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(tiles + (size_t)st * tile)),
            "l"(&tmap), "r"((int)(strip * TN)), "r"((int)((t0 + k) * TM)), "r"(bar), "l"(pol)
            : "memory");
    };
    if (tid == 0)
        for (int k = 0; k < stages; ++k) issue(k);

    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    uint32_t phase = 0;  // bit st: parity of the next completion of stage st
    int k = 0;
    for (; k < n; ++k) {
        const int st = k % stages;
        if (!mbar_wait_bounded(smem_u32(&full[st]), (phase >> st) & 1u)) {
            report(a.status, kStatusTimeout);
            abort_flag = 1;
        } else {
            const float *t = tiles + (size_t)st * tile;
            for (int rr = rl; rr < TM; rr += RL) {
                const float4 v = *reinterpret_cast<const float4 *>(t + rr * TN + cl * 4);
                acc[0] += v.x;
                acc[1] += v.y;
                acc[2] += v.z;
                acc[3] += v.w;
            }
        }
        phase ^= 1u << st;
        __syncthreads();  // every read of stage st is done
        if (abort_flag) break;
        if (tid == 0) issue(k + stages);
    }
    if (k < n && tid == 0) {
        // a wait gave up at tile k: the copies of tiles k .. k + stages - 1
        // may still be in flight; let them land before the block's shared
        // memory goes away (tile j is use j / stages of its stage, whose
        // completion has that parity; each wait bounded as well)
        for (int j = k; j < n && j < k + stages; ++j)
            mbar_wait_bounded(smem_u32(&full[j % stages]), (uint32_t)((j / stages) & 1));
    }

#pragma unroll
    for (int e = 0; e < 4; ++e) red[rl][cl * 4 + e] = acc[e];
    __syncthreads();
    if (rl == 0) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            float t = red[0][cl * 4 + e];
#pragma unroll
            for (int q = 1; q < RL; ++q) t += red[q][cl * 4 + e];
            part[cl * 4 + e] = t;
        }
    }
    cluster_push_partials(part, inbox, a.c, a.N, strip, a.status);
    pdl_wait();  // threads that stored nothing: the grid completes only after the one before it
}

// ------------------------------------------------------------------ host side

bool staged_tile(int TM, int TN)
{
    if (!(TN == 64 || TN == 128 || TN == 256)) return false;
    if (TM * TN > 8192) return false;
    return TM >= 1024 / TN && TM <= 256;
}

// The ring of the staged form: about 32 KB per CTA (at least two stages),
// which leaves room for five or six CTAs per SM; a TMA streaming experiment
// on this GPU found many CTAs with shallow rings faster than few CTAs with
// deep ones ([4096, 4096]: 14.1 us with two 16 KB stages at five CTAs per SM
// against 16.1 us with twelve stages at one).
int staged_stages(int TM, int TN)
{
    const int bytes = TM * TN * 4;
    int s = (32 * 1024) / bytes;
    if (s < 2) s = 2;
    if (s > 8) s = 8;
    return s;
}

bool pow2_in(int v, int lo, int hi)
{
    return v >= lo && v <= hi && (v & (v - 1)) == 0;
}

template <int TN, int CS>
const void *staged_kernel(bool aligned)
{
    return aligned ? (const void *)colsum_staged<TN, CS, true> : (const void *)colsum_staged<TN, CS, false>;
}

template <int TN>
tm_status launch_regdirect_t(bool vec, bool aligned, const ColArgs &a, cudaStream_t s, bool pdl)
{
    const void *k;
    if (vec) k = aligned ? (const void *)colsum_regdirect<TN, true, true> : (const void *)colsum_regdirect<TN, true, false>;
    else k = aligned ? (const void *)colsum_regdirect<TN, false, true> : (const void *)colsum_regdirect<TN, false, false>;
    void *args[] = {const_cast<ColArgs *>(&a)};
    return launch_kernel(k, dim3(flat_grid(a.units)), dim3(kThreads), args, 0, s, pdl);
}

// NAIVE's second pass (and the whole of an M == 0 call, P = 0: c = 0), run as
// a programmatic dependent of the partial-sum pass, which releases it as soon
// as its last block has started: the finish's blocks are resident and waiting
// (pdl_wait) when the partial sums land.
tm_status launch_finish(const float *part, int64_t npad, int64_t P, int64_t N, float *c, cudaStream_t s)
{
    void *args[] = {const_cast<float **>(&part), &npad, &P, &N, &c};
    return launch_dependent((const void *)colsum_finish, dim3(flat_grid((N + 31) / 32)), dim3(256), args, 0, s);
}

// The second pass of REGDIRECT and STAGED, also a programmatic dependent of
// the partial-sum pass.
tm_status launch_finish_strips(const float *part, int64_t P, int64_t TN, int64_t N, float *c, cudaStream_t s)
{
    int discard = aligned_to(part, 128) ? 1 : 0;
    void *args[] = {const_cast<float **>(&part), &P, &TN, &N, &c, &discard};
    return launch_dependent((const void *)colsum_finish_strips, dim3(flat_grid((N + 31) / 32)), dim3(256), args, 0,
                            s);
}

// The cluster variant: CS CTAs per TN-column strip (8-CTA clusters are
// portable; 16 needs the non-portable cluster size, set once per kernel).
template <int TN, int CS>
const void *cluster_kernel(bool vec, bool aligned, bool narrow)
{
    if (narrow) {
        if (vec) return aligned ? (const void *)colsum_cluster<TN, CS, true, true, uint32_t>
                                : (const void *)colsum_cluster<TN, CS, true, false, uint32_t>;
        return aligned ? (const void *)colsum_cluster<TN, CS, false, true, uint32_t>
                       : (const void *)colsum_cluster<TN, CS, false, false, uint32_t>;
    }
    if (vec) return aligned ? (const void *)colsum_cluster<TN, CS, true, true, int64_t>
                            : (const void *)colsum_cluster<TN, CS, true, false, int64_t>;
    return aligned ? (const void *)colsum_cluster<TN, CS, false, true, int64_t>
                   : (const void *)colsum_cluster<TN, CS, false, false, int64_t>;
}

const void *pick_cluster_kernel(int TN, int CS, bool vec, bool aligned, bool narrow)
{
    switch (TN) {
    case 64: return CS == 16 ? cluster_kernel<64, 16>(vec, aligned, narrow) : cluster_kernel<64, 8>(vec, aligned, narrow);
    case 128:
        return CS == 16 ? cluster_kernel<128, 16>(vec, aligned, narrow) : cluster_kernel<128, 8>(vec, aligned, narrow);
    default:
        return CS == 16 ? cluster_kernel<256, 16>(vec, aligned, narrow) : cluster_kernel<256, 8>(vec, aligned, narrow);
    }
}

// Per device and kernel: the non-portable cluster size allowed (16-CTA
// kernels), and how many clusters of CS CTAs can be resident at once (the
// occupancy API's answer; -1 if it could not answer).
struct ClusterSlot {
    const void *kernel;
    int max_active;
};
std::mutex g_cluster_mu;
ClusterSlot g_cluster_slots[kMaxDevices][64];

tm_status cluster_prepare(const void *k, int CS, int *max_active)
{
    int devno = 0;
    if (cudaGetDevice(&devno) != cudaSuccess || devno < 0 || devno >= kMaxDevices) {
        cudaGetLastError();
        return TM_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_cluster_mu);
    ClusterSlot *slots = g_cluster_slots[devno];
    for (int i = 0; i < 64 && slots[i].kernel; ++i)
        if (slots[i].kernel == k) {
            *max_active = slots[i].max_active;
            return TM_OK;
        }
    if (CS > 8 && cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
        cudaGetLastError();
        return TM_ERR_CUDA;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(CS * 64));
    cfg.blockDim = dim3(kThreads);
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = (unsigned)CS;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = -1;
    if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) != cudaSuccess) {
        cudaGetLastError();
        n = -1;
    }
    for (int i = 0; i < 64; ++i)
        if (!slots[i].kernel) {
            slots[i].kernel = k;
            slots[i].max_active = n;
            break;
        }
    *max_active = n;
    return TM_OK;
}

// 32-bit element offsets in the cluster kernel when they cannot wrap: the row
// loop looks up to UNR * RL <= 128 rows past the CTA's range before it
// compares, so every offset it forms is below (M + 128) * ldx.
bool cluster_narrow(int64_t M, int64_t ldx) { return ldx <= (int64_t)UINT32_MAX / (M + 128); }

tm_status launch_cluster(int TN, int CS, bool vec, bool aligned, const ColArgs &a, cudaStream_t s, bool pdl)
{
    const void *k = pick_cluster_kernel(TN, CS, vec, aligned, cluster_narrow(a.M, a.ldx));
    int max_active;
    const tm_status st = cluster_prepare(k, CS, &max_active);
    if (st != TM_OK) return st;
    // whole row tiles per CTA (the split the staged form uses too)
    int64_t rows_per_cta = (a.RT + CS - 1) / CS * a.TM;
    const int64_t strips = (a.N + TN - 1) / TN;
    void *args[] = {const_cast<ColArgs *>(&a), &rows_per_cta};
    return launch_kernel(k, dim3((unsigned)(strips * CS)), dim3(kThreads), args, 0, s, pdl, (unsigned)CS);
}

// The staged form: clusters of CS CTAs per strip, each streaming whole row
// tiles through its TMA ring.  Per kernel and device, once: the largest ring
// (two 32 KB stages) and, for 16-CTA clusters, the non-portable cluster size.
tm_status launch_staged(int TM, int TN, int CS, bool aligned, const CUtensorMap &map, const ColArgs &a,
                        cudaStream_t s, bool pdl)
{
    const int kidx = (TN == 64 ? 0 : TN == 128 ? 1 : 2) * 4 + (CS == 16 ? 2 : 0) + (aligned ? 1 : 0);
    const void *k;
    switch (TN) {
    case 64: k = CS == 16 ? staged_kernel<64, 16>(aligned) : staged_kernel<64, 8>(aligned); break;
    case 128: k = CS == 16 ? staged_kernel<128, 16>(aligned) : staged_kernel<128, 8>(aligned); break;
    default: k = CS == 16 ? staged_kernel<256, 16>(aligned) : staged_kernel<256, 8>(aligned); break;
    }
    static std::once_flag once[kMaxDevices][12];
    int devno = 0;
    if (cudaGetDevice(&devno) != cudaSuccess || devno < 0 || devno >= kMaxDevices) {
        cudaGetLastError();
        return TM_ERR_CUDA;
    }
    bool ok = true;
    std::call_once(once[devno][kidx], [&] {
        const int most = 2 * 8192 * (int)sizeof(float) + 2 * (int)sizeof(uint64_t);
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, most) != cudaSuccess ||
            (CS > 8 && cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)) {
            cudaGetLastError();
            ok = false;
        }
    });
    if (!ok) return TM_ERR_CUDA;
    int stages = staged_stages(TM, TN);
    int64_t tiles_per_cta = (a.RT + CS - 1) / CS;
    if (tiles_per_cta < stages) stages = tiles_per_cta > 2 ? (int)tiles_per_cta : 2;  // no deeper than its tiles
    const size_t smem = (size_t)stages * TM * TN * sizeof(float) + (size_t)stages * sizeof(uint64_t);
    const int64_t strips = (a.N + TN - 1) / TN;
    void *args[] = {const_cast<CUtensorMap *>(&map), const_cast<ColArgs *>(&a), &TM, &tiles_per_cta, &stages};
    return launch_kernel(k, dim3((unsigned)(strips * CS)), dim3(kThreads), args, smem, s, pdl, (unsigned)CS);
}

// CTAs per strip in the cluster variant: 16 (non-portable clusters) when there
// are few strips -- half the rows per CTA, half the dependent load batches
// ([4096, 4096]: 17.9 against 19.2 us per call) -- else 8 ([8192, 8192]: 16
// per strip measured 47.2 against 46.2 us, 38.1 against 36.2 chained).
constexpr int kClusterCTAs = 8;
constexpr int kClusterCTAsTall = 16;

int cluster_ctas(int64_t strips, int sms)
{
    return strips * kClusterCTAsTall <= 4LL * sms ? kClusterCTAsTall : kClusterCTAs;
}

enum class Variant { Naive, RegDirect, Staged, Cluster };

}  // namespace
}  // namespace libtm

using namespace libtm;

extern "C" size_t tm_colsum_workspace_bytes(int64_t M, int64_t N, int32_t TM, int32_t TN, tm_variant variant)
{
    if (M <= 0 || N <= 0) return 0;
    if (variant == TM_VAR_CLUSTER || variant == TM_VAR_STAGED) return 0;  // partials meet on chip
    if (variant == TM_VAR_NAIVE) {
        const int64_t rb = (M + kNaiveRows - 1) / kNaiveRows;
        return (size_t)(rb * ((N + 3) & ~int64_t(3)) * (int64_t)sizeof(float));
    }
    if (variant != TM_VAR_AUTO && variant != TM_VAR_REGDIRECT) return 0;
    if (!pow2_in(TM, 8, 256) || !(TN == 64 || TN == 128 || TN == 256)) return 0;
    return (size_t)partial_bytes(plan_chunks(M, N, TM, TN), TN);
}

extern "C" tm_status tm_colsum(const float *X, int64_t ldx, int64_t M, int64_t N, float *c, void *workspace,
                               size_t ws_bytes, int32_t TM, int32_t TN, tm_variant variant, uint32_t flags,
                               tm_stream_t stream)
{
    if (!valid2d(X, ldx, M, N)) return TM_ERR_INVALID_ARG;
    if (N > 0 && c == nullptr) return TM_ERR_INVALID_ARG;
    if (!flags_ok(flags, TM_ALIGNED | TM_PATH_SCALAR | TM_PATH_VEC | TM_PDL)) return TM_ERR_INVALID_ARG;
    if (variant != TM_VAR_AUTO && variant != TM_VAR_NAIVE && variant != TM_VAR_STAGED &&
        variant != TM_VAR_REGDIRECT && variant != TM_VAR_CLUSTER)
        return TM_ERR_INVALID_ARG;
    if (variant != TM_VAR_NAIVE && (!pow2_in(TM, 8, 256) || !(TN == 64 || TN == 128 || TN == 256)))
        return TM_ERR_UNSUPPORTED_TILE;
    if (variant == TM_VAR_STAGED && !staged_tile(TM, TN)) return TM_ERR_UNSUPPORTED_TILE;
    if (N > 0 && !aligned_to(c, 4)) return TM_ERR_MISALIGNED;
    if (M > 0 && N > 0 && !aligned_to(X, 4)) return TM_ERR_MISALIGNED;
    const bool aligned = (flags & TM_ALIGNED) != 0;
    const bool vec16 = aligned_to(X, 16) && ldx % 4 == 0;
    if (aligned) {
        if (!vec16) return TM_ERR_MISALIGNED;
        if (variant == TM_VAR_NAIVE) return TM_ERR_INVALID_ARG;  // the foil has no whole-tile path
        if (M % TM != 0 || N % TN != 0) return TM_ERR_BROKEN_PROMISE;
    }
    if ((flags & TM_PATH_VEC) && !(vec16 && N % 4 == 0)) return TM_ERR_MISALIGNED;

    const bool vec = !(flags & TM_PATH_SCALAR) && vec16 && (aligned || N % 4 == 0);

    // scratch: the requested variant's (AUTO sizes for REGDIRECT even when it
    // then runs CLUSTER); X, c and the scratch must not overlap
    const int64_t npad = (N + 3) & ~int64_t(3);
    ColPlan pl{};
    size_t need = 0;
    if (M > 0 && N > 0) {
        uintptr_t xlo, xhi;
        span2d(X, ldx, M, N, &xlo, &xhi);
        const uintptr_t clo = reinterpret_cast<uintptr_t>(c), chi = clo + (uintptr_t)N * 4;
        if (!(xhi <= clo || chi <= xlo)) return TM_ERR_INVALID_ARG;
        need = tm_colsum_workspace_bytes(M, N, TM, TN, variant);
        if (need > 0) {
            if (workspace == nullptr || ws_bytes < need || !aligned_to(workspace, 16)) return TM_ERR_WORKSPACE;
            const uintptr_t wlo = reinterpret_cast<uintptr_t>(workspace), whi = wlo + need;
            if (!(xhi <= wlo || whi <= xlo) || !(chi <= wlo || whi <= clo)) return TM_ERR_INVALID_ARG;
        }
        if (variant != TM_VAR_NAIVE) pl = plan_chunks(M, N, TM, TN);
        if ((variant == TM_VAR_CLUSTER || variant == TM_VAR_STAGED) && (N + TN - 1) / TN * kClusterCTAsTall > INT32_MAX)
            return TM_ERR_INVALID_ARG;
    }
    const bool tma_shape = vec16 && M <= INT32_MAX && N <= INT32_MAX && staged_tile(TM, TN) &&
                           !(flags & (TM_PATH_SCALAR | TM_PATH_VEC));
    if (variant == TM_VAR_STAGED && !tma_shape) return TM_ERR_MISALIGNED;
    if (N == 0) return TM_OK;

    const DevInfo *dev;
    tm_status st = device_info(&dev);
    if (st != TM_OK) return st;
    cudaStream_t s = as_stream(stream);
    const bool pdl = (flags & TM_PDL) != 0;
    if (M == 0) return launch_finish(nullptr, npad, 0, N, c, s);  // the sum of nothing: c = 0

    // pick the variant (the TMA encoder comes from the driver on first use)
    Variant v;
    if (variant == TM_VAR_NAIVE) v = Variant::Naive;
    else if (variant == TM_VAR_REGDIRECT) v = Variant::RegDirect;
    else if (variant == TM_VAR_CLUSTER) v = Variant::Cluster;
    else if (variant == TM_VAR_STAGED) {
        if (tensor_map_encoder() == nullptr) return TM_ERR_CUDA;
        v = Variant::Staged;
    } else {
        // AUTO: the one-pass cluster form whenever all its clusters fit on the
        // GPU at once (one wave), else the register-direct pass and its finish.
        // [8192, 8192] at 32 x 128: 64 strips of 8-CTA clusters, all resident
        // at four CTAs per SM (one pass: 41.9 us by kernel time, against 41.1
        // for the register-direct pass plus its second launch and the 4 MiB
        // of partials it writes and reads back); [4096, 4096]: 32 strips of
        // 16-CTA clusters.
        const int CS = cluster_ctas(pl.S, dev->sms);
        int max_active = -1;
        st = cluster_prepare(pick_cluster_kernel(TN, CS, vec, aligned, cluster_narrow(M, ldx)), CS, &max_active);
        if (st != TM_OK) return st;
        v = (max_active > 0 && pl.S <= max_active) ? Variant::Cluster : Variant::RegDirect;
    }

    if (v == Variant::Naive) {
        float *part = static_cast<float *>(workspace);
        const int64_t P = (M + kNaiveRows - 1) / kNaiveRows;
        int64_t programs = P * N;
        void *args[] = {(void *)&X, (void *)&ldx, (void *)&M, (void *)&N, (void *)&part, (void *)&npad,
                        (void *)&programs};
        st = launch_kernel((const void *)colsum_naive, dim3(flat_grid(programs)), dim3(kNaiveRows), args, 0, s, pdl);
        if (st != TM_OK) return st;
        return launch_finish(part, npad, P, N, c, s);
    }

    ColArgs a;
    a.X = X;
    a.ldx = ldx;
    a.M = M;
    a.N = N;
    a.c = c;
    a.S = pl.S;
    a.RT = pl.RT;
    a.CT = pl.CT;
    a.P = pl.P;
    a.units = pl.units;
    a.TM = TM;
    a.status = dev->status;
    a.part = pl.P > 1 ? static_cast<float *>(workspace) : nullptr;
    if (v == Variant::Cluster) return launch_cluster(TN, cluster_ctas(pl.S, dev->sms), vec, aligned, a, s, pdl);

    if (v == Variant::Staged) {
        CUtensorMap map;
        const cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)M};
        const cuuint64_t strides[1] = {(cuuint64_t)ldx * sizeof(float)};
        const cuuint32_t box[2] = {(cuuint32_t)TN, (cuuint32_t)TM};
        const cuuint32_t estr[2] = {1, 1};
        if (tensor_map_encoder()(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(X), dims, strides, box,
                                 estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return TM_ERR_CUDA;
        return launch_staged(TM, TN, cluster_ctas(pl.S, dev->sms), aligned, map, a, s, pdl);
    }
    switch (TN) {
    case 64: st = launch_regdirect_t<64>(vec, aligned, a, s, pdl); break;
    case 128: st = launch_regdirect_t<128>(vec, aligned, a, s, pdl); break;
    default: st = launch_regdirect_t<256>(vec, aligned, a, s, pdl); break;
    }
    if (st != TM_OK || pl.P == 1) return st;  // one chunk per strip: the pass wrote c itself
    return launch_finish_strips(a.part, pl.P, TN, N, c, s);
}

// ------------------------------------------------------------------ no-allocation entry point
// Some callers cannot allocate device memory at the point where they need a
// column sum: code hosted inside another framework whose allocator owns every
// device byte, loops with a fixed memory budget that must not fail with
// out-of-memory halfway through, or latency-critical paths where cudaMalloc
// (which may synchronize the whole device) is not allowed.  For them
// tm_colsum_noalloc keeps the partial sums in this file-scope array instead of
// a caller-provided workspace.  Every GPU that loads the library holds the
// array until the process exits.
namespace libtm {
namespace {

static __device__ __align__(256) float g_colsum_scratch[TM_NOALLOC_SCRATCH_BYTES / sizeof(float)];

struct ScratchSlot {
    std::atomic<bool> ready{false};
    void *addr = nullptr;
};
ScratchSlot g_scratch_slots[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of g_colsum_scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so the real address is asked of
// the runtime once per device, with that device current.
tm_status scratch_address(void **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return TM_ERR_CUDA;
    }
    ScratchSlot &s = g_scratch_slots[dev];
    if (!s.ready.load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lock(g_scratch_mu);
        if (!s.ready.load(std::memory_order_relaxed)) {
            void *p = nullptr;
            if (cudaGetSymbolAddress(&p, g_colsum_scratch) != cudaSuccess || p == nullptr) {
                cudaGetLastError();
                return TM_ERR_CUDA;
            }
            s.addr = p;
            s.ready.store(true, std::memory_order_release);
        }
    }
    *out = s.addr;
    return TM_OK;
}

}  // namespace
}  // namespace libtm

extern "C" tm_status tm_colsum_noalloc(const float *X, int64_t ldx, int64_t M, int64_t N, float *c, int32_t TM,
                                       int32_t TN, tm_variant variant, uint32_t flags, tm_stream_t stream)
{
    // The requested variant's own requirement: CLUSTER keeps its partials on
    // chip and needs none, so it runs at any shape; the others are limited by
    // the array's size.  (0 also for arguments tm_colsum itself rejects.)
    const size_t need = tm_colsum_workspace_bytes(M, N, TM, TN, variant);
    if (need > TM_NOALLOC_SCRATCH_BYTES) return TM_ERR_WORKSPACE;  // beyond the built-in scratch
    void *scratch = nullptr;
    if (need > 0) {
        const tm_status st = scratch_address(&scratch);
        if (st != TM_OK) return st;
    }
    // Every partial-sum word the second pass reads is written earlier in the
    // same call, so the array's leftover contents never need clearing.
    return tm_colsum(X, ldx, M, N, c, scratch, need > 0 ? TM_NOALLOC_SCRATCH_BYTES : 0, TM, TN, variant, flags,
                     stream);
}
