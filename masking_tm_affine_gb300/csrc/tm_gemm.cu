// tm_gemm.cu -- the ragged fp32 gemm: C = alpha * (A B) + beta * C on tcgen05.
//
// Source: "@aligned" -- the gemm example (C = alpha * acc + beta * c_old over
// TILE_M x TILE_N output tiles, acc += dot(a, b) over K tiles), shown with and
// without the promise; "Slicing, bounds and masking", "Loops over a dynamic
// extent": a K loop over a runtime extent is whole tiles plus one masked
// remainder whose missing columns read 0.
//
// GB300 design.  A dense contraction, so it runs on the 5th-generation tensor
// cores: tcgen05.mma kind::tf32 from shared-memory operands into a TMEM
// accumulator.  fp32 accuracy comes from the 3xTF32 split: each operand x is
// hi + lo with hi = x rounded to tf32 and lo = (x - hi) rounded to tf32, and
// the product is hi*hi + hi*lo + lo*hi (the lo*lo term is below fp32
// resolution); TM_GEMM_TF32 keeps the single hi*hi pass instead.
//   1. split pass (one launch, memory-bound): A [M, K] and B [K, N] become
//      K-major hi/lo operands zero-padded to whole tiles -- the zero padding
//      is exactly the masked remainder tile's fill -- with B transposed on
//      the way.
//   2. gemm (a programmatic dependent of the split): persistent 192-thread
//      CTAs walking the output tiles -- by default CTA pairs (2-CTA clusters,
//      256-row tiles, tcgen05 cta_group::2: each CTA stages 128 rows of A and
//      half of the B tile, and the even CTA issues the MMAs for both), else
//      one CTA per 128-row tile.  Warp 0 issues TMA copies (K-major, 64- or
//      128-byte swizzle) into a ring of STAGES shared-memory stages; warp 1
//      owns the TMEM accumulators (two buffers of BN columns) and one of its
//      threads issues the MMAs (K = 8 each, three per K step for 3xTF32),
//      committing each stage back to the producers and each finished tile to
//      the epilogues through mbarriers; warps 2-5 read the other accumulator
//      buffer out of TMEM (32x32b loads) and write alpha * acc + beta * C
//      (through TMA when C's layout allows), while the next tile accumulates.
//      Every wait is bounded; a stalled pipeline sets the status word and the
//      CTA drains and frees its TMEM before it exits.  When the output tiles
//      fill at most half of the last round of units and K is long, each of
//      that round's tiles is cut along K into parts run side by side
//      (split-K); the unit that ran part 0 adds the others, read back from the
//      workspace in K order, before its epilogue.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "tm_host.h"

namespace libtm {
namespace {

constexpr int GBM = 128;  // UMMA M (one CTA)
constexpr int GBK = 32;   // K padding granule of the split operands (a multiple of both stage widths)

// ------------------------------------------------------------------ split pass
__device__ __forceinline__ uint32_t to_tf32(float x)
{
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

// One launch splits both operands.  Blocks [0, blocks_a) walk A's rows
// (threads over k, both sides coalesced) into hi/lo [Mp, Kp]; the rest walk
// 32 x 32 tiles of B through shared memory into the transposed hi/lo
// [Np, Kp].  Everything outside [M, K] (resp. [K, N]) is written as zero.
// With alo == blo == nullptr (the single-pass mode) only hi is written.
struct SplitArgs {
    const float *A, *B;
    int64_t lda, ldb, M, N, K, Mp, Np, Kp;
    float *ahi, *alo, *bhi, *blo;
    unsigned blocks_a, blocks_b;
    unsigned *flags;  // the gemm's split-K flags, zeroed here (the gemm starts after this pass)
    int nflags;
};

__device__ __forceinline__ void split_store(float *hi, float *lo, int64_t at, float x)
{
    const uint32_t h = to_tf32(x);
    hi[at] = as_f(h);
    if (lo != nullptr) lo[at] = as_f(to_tf32(x - as_f(h)));
}

__global__ void __launch_bounds__(256) split_operands(const SplitArgs a)
{
    __shared__ float t[32][33];
    pdl_trigger();  // the gemm's prologue may start once every block has started
    if (blockIdx.x == 0)
        for (int i = threadIdx.x; i < a.nflags; i += blockDim.x) a.flags[i] = 0u;
    if (blockIdx.x < a.blocks_a) {
        for (int64_t i = blockIdx.x; i < a.Mp; i += a.blocks_a)
            for (int64_t k = threadIdx.x; k < a.Kp; k += blockDim.x) {
                const float x = (i < a.M && k < a.K) ? as_f(ld_nc_b32(a.A + i * a.lda + k)) : 0.0f;
                split_store(a.ahi, a.alo, i * a.Kp + k, x);
            }
        return;
    }
    const int64_t tiles_k = a.Kp / 32, tiles_n = a.Np / 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
    for (int64_t tile = blockIdx.x - a.blocks_a; tile < tiles_k * tiles_n; tile += a.blocks_b) {
        const int64_t k0 = (tile / tiles_n) * 32, n0 = (tile % tiles_n) * 32;
#pragma unroll
        for (int r = ty; r < 32; r += 8) {
            const int64_t k = k0 + r, n = n0 + tx;
            t[r][tx] = (k < a.K && n < a.N) ? as_f(ld_nc_b32(a.B + k * a.ldb + n)) : 0.0f;
        }
        __syncthreads();
#pragma unroll
        for (int r = ty; r < 32; r += 8) split_store(a.bhi, a.blo, (n0 + r) * a.Kp + k0 + tx, t[tx][r]);
        __syncthreads();
    }
}

// ------------------------------------------------------------------ gemm
// Shared-memory matrix descriptor: start >> 4 in [0, 14), leading byte offset
// >> 4 in [16, 30), stride byte offset >> 4 in [32, 46), descriptor version 1
// at bit 46, layout in [61, 64): 2 = 128-byte swizzle, 4 = 64-byte swizzle.
// K-major rows of BK fp32 (BK * 4 bytes, the swizzle width): consecutive
// 8-row groups are 8 * BK * 4 bytes apart.
template <int BK>
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr)
{
    static_assert(BK == 16 || BK == 32, "stage K must fill one 64- or 128-byte swizzle row");
    constexpr uint64_t kSbo = 8 * BK * 4, kLayout = BK == 32 ? 2 : 4;
    return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)1 << 16) | ((kSbo >> 4) << 32) | ((uint64_t)1 << 46) |
           (kLayout << 61);
}

// Instruction descriptor, kind::tf32: D fp32 (bits 4-5 = 1), A and B tf32
// (bits 7-9, 10-12 = 2), both K-major, N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N)
{
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// tcgen05 operations of one CTA (PAIR = false) or of a CTA pair (PAIR = true:
// cta_group::2, issued by the even CTA of a 2-CTA cluster; A is split by rows
// between the two CTAs' shared memory, B by its N rows, and each CTA's TMEM
// holds its 128 rows of the 256-row accumulator).  A kernel uses one group
// throughout.
template <bool PAIR>
__device__ __forceinline__ void umma_tf32(uint32_t tmem, uint64_t da, uint64_t db, uint32_t id, uint32_t acc)
{
    if constexpr (PAIR)
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem),
            "l"(da), "l"(db), "r"(id), "r"(acc)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem),
            "l"(da), "l"(db), "r"(id), "r"(acc)
            : "memory");
}

// Arrive on `bar` (same offset in both CTAs of a pair) once every MMA issued
// so far by this thread has completed.
template <bool PAIR>
__device__ __forceinline__ void umma_commit(uint32_t bar)
{
    if constexpr (PAIR)
        asm volatile(
            "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
                bar),
            "h"((uint16_t)3)
            : "memory");
    else
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                     : "memory");
}

template <bool PAIR>
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t cols)
{
    if constexpr (PAIR) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst), "r"(cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    } else {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst), "r"(cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
}

template <bool PAIR>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t cols)
{
    if constexpr (PAIR)
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols) : "memory");
    else
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols) : "memory");
}

// TMA load into this CTA's shared memory whose completion is signalled on the
// even CTA's barrier `bar` (a cluster address): a pair's operand copies.
__device__ __forceinline__ void tma_load_pair(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(map), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_load(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(map), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

struct GemmArgs {
    float *C;
    int64_t ldc, M, N;
    float alpha, beta;
    int KT;       // pipeline stages per output tile: Kp / BK
    int tiles_m;  // output tiles along M (tile order: tile_coords)
    int ntiles;   // tiles_m * tiles along N
    int vec_c;    // C base 16-byte aligned, ldc % 4 == 0 and N % 4 == 0: the epilogue moves C by TMA
    unsigned *status;
    // split-K of the last round: tiles [0, dp_tiles) run whole, round-robin
    // over the units; each later tile is cut along K into sk_split equal
    // parts, part q of tile dp_tiles + j run by unit j * sk_split + q, all
    // parts at the same time (0: no split)
    int dp_tiles;
    int sk_split;
    float *part;      // a unit's partial accumulator: rows [unit * tile rows, + tile rows) x BN
    unsigned *flags;  // per unit: epilogue warps that have written its partial
};

constexpr int kMaxSms = 256;     // split-K partial rows: at most this many 128-row accumulators
constexpr int kSkMinSaved = 48;  // split-K only when it takes this many K stages off the critical path

// The work of one unit (CTA or CTA pair), in order: its data-parallel tiles
// (every units-th tile from its own index), then its part of a split tile, as
// items [kb, ke) of one tile.  Producer, MMA issuer and epilogues all walk
// the same sequence.  Part 0 finishes the tile: it adds the other parts,
// written by the next sk_split - 1 units, in K order.
struct Items {
    int next_dp, step, dp_tiles, KT, sk_tile, sk_kb, sk_ke;
    bool sk_left;
    __device__ Items(const GemmArgs &g, int unit, int units)
        : next_dp(unit), step(units), dp_tiles(g.dp_tiles), KT(g.KT), sk_tile(0), sk_kb(0), sk_ke(0),
          sk_left(g.sk_split > 0 && unit < (g.ntiles - g.dp_tiles) * g.sk_split)
    {
        if (sk_left) {
            const int q = unit % g.sk_split;
            sk_tile = g.dp_tiles + unit / g.sk_split;
            sk_kb = q * g.KT / g.sk_split;
            sk_ke = (q + 1) * g.KT / g.sk_split;
        }
    }
    __device__ bool next(int &tile, int &kb, int &ke)
    {
        if (next_dp < dp_tiles) {
            tile = next_dp;
            kb = 0;
            ke = KT;
            next_dp += step;
            return true;
        }
        if (!sk_left) return false;
        sk_left = false;
        tile = sk_tile;
        kb = sk_kb;
        ke = sk_ke;
        return true;
    }
};

template <int BN, int BK, bool THREE>
struct GemmStage {
    static constexpr int kLo = THREE ? 1 : 0;  // the single-pass mode keeps no lo operands
    alignas(1024) float a_hi[GBM * BK];
    alignas(1024) float b_hi[BN * BK];
    alignas(1024) float a_lo[kLo * GBM * BK + (1 - kLo)];
    alignas(1024) float b_lo[kLo * BN * BK + (1 - kLo)];
};

// Stages that fit the 192 KB of shared memory given to the ring (the C
// staging buffers take 32 KB more, inside the 227 KB a CTA may have).
template <int BN, int BK, bool THREE>
constexpr int gemm_stages()
{
    return (int)((192u * 1024u) / sizeof(GemmStage<BN, BK, THREE>));
}

template <int BN, int BK, int STAGES, bool THREE>
struct GemmSmem {
    using Stage = GemmStage<BN, BK, THREE>;
    Stage st[STAGES];
    // epilogue staging: per epilogue warp two 32 x 32 fp32 chunks of C in the
    // TMA 128-byte-swizzled layout (row r's 16-byte piece j at j ^ (r % 8))
    alignas(1024) float cbuf[4][2][32 * 32];
    alignas(8) uint64_t cbar[4][2];     // TMA -> epilogue warp: the chunk of C has landed
    alignas(8) uint64_t full[STAGES];   // TMA -> MMA: the stage's operands have landed
    alignas(8) uint64_t empty[STAGES];  // MMA -> TMA: the MMAs reading the stage are done
    alignas(8) uint64_t acc_full[2];    // MMA -> epilogue: accumulator buffer holds a finished tile
    alignas(8) uint64_t acc_empty[2];   // epilogue -> MMA: accumulator buffer has been read out
    alignas(8) uint64_t done;           // every MMA issued has completed
    uint32_t tmem;
    int abort;
};

constexpr int kGemmThreads = 192;  // warp 0 TMA, warp 1 MMA (and TMEM owner), warps 2-5 epilogue

__device__ __forceinline__ bool gemm_aborted(const int *flag) { return *(volatile const int *)flag != 0; }

// The epilogue waits a whole tile's K loop for its accumulator, so its limit
// grows with K (a stage takes a few microseconds at most; 40000 cycles are
// allowed per stage on top of the fixed limit).  A stall inside the pipeline
// is caught sooner by the producer's and the MMA issuer's own waits, which set
// the abort flag that this wait also watches.
__device__ __forceinline__ bool acc_wait(uint32_t bar, uint32_t parity, int KT, const int *abort_flag)
{
    if (mbar_try_wait(bar, parity)) return true;
    const long long limit = kWaitCycles + 40000LL * KT;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (*(volatile const int *)abort_flag != 0 || clock64() - t0 > limit) return false;
    }
    return true;
}

__device__ __forceinline__ void gemm_fail(int *flag, unsigned *status)
{
    atomicOr(status, kStatusTimeout);
    *(volatile int *)flag = 1;
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
          "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
          "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Stream-K partials: written and read at L2 (other SMs produce and consume
// them), published with a release add and observed with an acquire load.
__device__ __forceinline__ void st_cg_v4(float *p, const u32x4 &x)
{
    asm volatile("st.global.cg.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(x.v[0]), "r"(x.v[1]), "r"(x.v[2]),
                 "r"(x.v[3])
                 : "memory");
}

__device__ __forceinline__ u32x4 ld_cg_v4(const float *p)
{
    u32x4 r;
    asm volatile("ld.global.cg.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.v[0]), "=r"(r.v[1]), "=r"(r.v[2]), "=r"(r.v[3])
                 : "l"(p)
                 : "memory");
    return r;
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned *p)
{
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_release_add_u32(unsigned *p, unsigned v)
{
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void tma_store(const CUtensorMap *map, int x, int y, uint32_t src)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(map), "r"(x),
                 "r"(y), "r"(src)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// The calling thread's bulk stores have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// The calling thread's bulk stores have completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Output tile t -> (m0, n0): groups of kGroupM tile rows, M-fastest inside a
// group, so the CTAs running at the same time share a compact block of A and
// B tiles in L2 (the page's pm = block.x, pn = block.y order within a group).
constexpr int kGroupM = 16;

__device__ __forceinline__ void tile_coords(int tile, int tiles_m, int tiles_n, int BM, int BN, int &m0, int &n0)
{
    const int64_t per_group = (int64_t)kGroupM * tiles_n;
    const int group = (int)(tile / per_group);
    const int first = group * kGroupM;
    const int gm = tiles_m - first < kGroupM ? tiles_m - first : kGroupM;
    const int local = (int)(tile - group * per_group);
    m0 = (first + local % gm) * BM;
    n0 = (local / gm) * BN;
}

// Persistent over the output tiles in tile_coords order: one CTA per SM
// (PAIR = false, 128-row tiles) or one 2-CTA cluster per SM pair (PAIR = true,
// 256-row tiles: each CTA stages its 128 rows of A and half of B's BN rows, so
// a pair moves a third fewer operand bytes per flop than two single CTAs).
// The accumulator is double-buffered in TMEM (2 x BN columns): the epilogue of
// one tile runs while the MMAs of the next accumulate into the other buffer.
template <int BN, int BK, int STAGES, bool THREE, bool ALIGNED, bool PAIR>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_tf32_kernel(const __grid_constant__ CUtensorMap m_ahi, const __grid_constant__ CUtensorMap m_alo,
                     const __grid_constant__ CUtensorMap m_bhi, const __grid_constant__ CUtensorMap m_blo,
                     const __grid_constant__ CUtensorMap m_c, const GemmArgs g)
{
    constexpr int BH = PAIR ? BN / 2 : BN;   // B rows staged per CTA
    constexpr int TMR = PAIR ? 2 * GBM : GBM;  // output tile rows
    using Smem = GemmSmem<BH, BK, STAGES, THREE>;
    extern __shared__ __align__(1024) unsigned char raw[];
    Smem &s = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tiles_n = g.ntiles / g.tiles_m;
    const uint32_t rank = PAIR ? cluster_rank() : 0u;  // 0: this CTA issues the MMAs
    const int unit = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
    const int units = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;
    constexpr uint32_t kStageBytes = (uint32_t)((THREE ? 2 : 1) * (GBM + BH) * BK * sizeof(float));  // per CTA
    constexpr uint32_t kCols = 2 * BN;  // TMEM columns: two accumulator buffers

    if (warp == 1) tmem_alloc<PAIR>(smem_u32(&s.tmem), kCols);
    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&s.full[i])));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&s.empty[i])));
        }
        for (int i = 0; i < 2; ++i) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&s.acc_full[i])));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(&s.acc_empty[i])),
                         "r"(PAIR ? 256 : 128));
        }
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&s.done)));
        for (int i = 0; i < 4; ++i)
            for (int j = 0; j < 2; ++j) asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&s.cbar[i][j])));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        s.abort = 0;
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if constexpr (PAIR) cluster_sync();  // both CTAs' barriers exist before any remote signal
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = s.tmem;
    pdl_wait();  // launched as a dependent of the split pass: its operands first

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer: this CTA's operand tiles of every K stage
            uint32_t it = 0;
            bool ok = true;
            Items items(g, unit, units);
            int tile, kb, ke;
            while (ok && items.next(tile, kb, ke)) {
                int m0, n0;
                tile_coords(tile, g.tiles_m, tiles_n, TMR, BN, m0, n0);
                const int am = m0 + (int)rank * GBM, bn = n0 + (int)rank * BH;
                for (int kt = kb; kt < ke; ++kt, ++it) {
                    const uint32_t st = it % STAGES;
                    if (it >= STAGES && !mbar_wait_bounded(smem_u32(&s.empty[st]), ((it / STAGES) - 1) & 1u)) {
                        gemm_fail(&s.abort, g.status);
                        ok = false;
                        break;
                    }
                    if (gemm_aborted(&s.abort)) {
                        ok = false;
                        break;
                    }
                    const int kx = kt * BK;
                    if constexpr (PAIR) {
                        // the even CTA's barrier counts both CTAs' bytes
                        if (rank == 0)
                            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
                                             smem_u32(&s.full[st])),
                                         "r"(2 * kStageBytes)
                                         : "memory");
                        const uint32_t bar = cluster_addr(smem_u32(&s.full[st]), 0);
                        tma_load_pair(smem_u32(s.st[st].a_hi), &m_ahi, kx, am, bar);
                        tma_load_pair(smem_u32(s.st[st].b_hi), &m_bhi, kx, bn, bar);
                        if (THREE) {
                            tma_load_pair(smem_u32(s.st[st].a_lo), &m_alo, kx, am, bar);
                            tma_load_pair(smem_u32(s.st[st].b_lo), &m_blo, kx, bn, bar);
                        }
                    } else {
                        const uint32_t bar = smem_u32(&s.full[st]);
                        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                                     "r"(kStageBytes)
                                     : "memory");
                        tma_load(smem_u32(s.st[st].a_hi), &m_ahi, kx, am, bar);
                        tma_load(smem_u32(s.st[st].b_hi), &m_bhi, kx, bn, bar);
                        if (THREE) {
                            tma_load(smem_u32(s.st[st].a_lo), &m_alo, kx, am, bar);
                            tma_load(smem_u32(s.st[st].b_lo), &m_blo, kx, bn, bar);
                        }
                    }
                }
            }
            // Nothing may still be landing in shared memory when the CTA (or
            // its pair) leaves: the barriers this CTA armed see every byte.
            // After a normal run they have all completed already.
            if (!ok || PAIR) {
                if (rank == 0)
                    for (uint32_t j = (it > STAGES ? it - STAGES : 0); j < it; ++j)
                        mbar_wait_bounded(smem_u32(&s.full[j % STAGES]), (j / STAGES) & 1u);
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            // ---------------- MMA issuer: 3 (or 1) tf32 MMAs per 8-wide K step
            constexpr uint32_t id = idesc_tf32(TMR, BN);
            uint32_t it = 0;
            bool ok = true;
            Items items(g, unit, units);
            int tile, kb, ke;
            for (int t = 0; ok && items.next(tile, kb, ke); ++t) {
                const uint32_t ab = (uint32_t)t & 1u;
                if (t >= 2 && !mbar_wait_bounded(smem_u32(&s.acc_empty[ab]), ((uint32_t)(t / 2) - 1) & 1u)) {
                    gemm_fail(&s.abort, g.status);
                    break;
                }
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t d = tmem + ab * BN;
                for (int kt = kb; kt < ke; ++kt, ++it) {
                    const uint32_t st = it % STAGES;
                    if (!mbar_wait_bounded(smem_u32(&s.full[st]), (it / STAGES) & 1u) || gemm_aborted(&s.abort)) {
                        if (!gemm_aborted(&s.abort)) gemm_fail(&s.abort, g.status);
                        ok = false;
                        break;
                    }
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    const uint32_t ahi = smem_u32(s.st[st].a_hi), alo = smem_u32(s.st[st].a_lo);
                    const uint32_t bhi = smem_u32(s.st[st].b_hi), blo = smem_u32(s.st[st].b_lo);
#pragma unroll
                    for (int k = 0; k < BK / 8; ++k) {
                        const uint32_t off = (uint32_t)k * 32;  // 8 tf32 = 32 bytes inside the swizzled row
                        umma_tf32<PAIR>(d, smem_desc<BK>(ahi + off), smem_desc<BK>(bhi + off), id,
                                        (kt != kb || k != 0) ? 1u : 0u);  // the item's first MMA overwrites
                        if (THREE) {
                            umma_tf32<PAIR>(d, smem_desc<BK>(ahi + off), smem_desc<BK>(blo + off), id, 1u);
                            umma_tf32<PAIR>(d, smem_desc<BK>(alo + off), smem_desc<BK>(bhi + off), id, 1u);
                        }
                    }
                    umma_commit<PAIR>(smem_u32(&s.empty[st]));  // the stage (in both CTAs) is free once these are done
                }
                if (ok) umma_commit<PAIR>(smem_u32(&s.acc_full[ab]));
            }
            umma_commit<PAIR>(smem_u32(&s.done));  // tracks every MMA issued, also after an abort
            if (!mbar_wait_bounded(smem_u32(&s.done), 0u)) gemm_fail(&s.abort, g.status);
        }
    } else {
        // ---------------- epilogue: TMEM rows -> alpha * acc + beta * C
        const int eg = warp & 3;  // TMEM lane group this warp may access (rows 32 eg .. 32 eg + 31)
        const bool use_c = g.beta != 0.0f;
        // the MMA issuer's "accumulator free" barrier (in the even CTA of a pair)
        const uint32_t acc_empty0 = PAIR ? cluster_addr(smem_u32(&s.acc_empty[0]), 0) : smem_u32(&s.acc_empty[0]);
        const uint32_t acc_empty1 = PAIR ? cluster_addr(smem_u32(&s.acc_empty[1]), 0) : smem_u32(&s.acc_empty[1]);
        uint32_t cpar = 0;        // bit j: parity of the next completion of cbar[eg][j]
        uint32_t loads_out = 0;   // bit j: a load into cbuf[eg][j] is in flight
        constexpr unsigned kEpiWarps = PAIR ? 8u : 4u;  // epilogue warps of a unit: a partial's arrivals
        Items items(g, unit, units);
        int tile, kb, ke;
        for (int t = 0; items.next(tile, kb, ke); ++t) {
            const uint32_t ab = (uint32_t)t & 1u;
            const bool contrib = kb != 0;              // a later part of a tile another unit finishes
            const bool finish = kb == 0 && ke < g.KT;  // this unit finishes the tile with the later parts
            const int last = unit + g.sk_split;        // (finish) the later parts' units: unit + 1 .. last - 1
            // Unit u's partial accumulator is laid out as this thread sees it: for
            // each CTA rank, epilogue warp and 32-column chunk c, eight 512-byte
            // pieces, piece j holding columns c + 4j .. c + 4j + 3 of the warp's
            // 32 rows, lane after lane -- every warp access is 512 contiguous bytes.
            auto part_chunk = [&](int u, int c) {
                return g.part + ((((int64_t)u * (TMR / GBM) + rank) * 4 + eg) * (BN / 32) + c / 32) * 1024 + lane * 4;
            };
            auto add4 = [](uint32_t(&r)[32], const u32x4 (&v)[8]) {
#pragma unroll
                for (int j = 0; j < 8; ++j)
#pragma unroll
                    for (int e = 0; e < 4; ++e) r[4 * j + e] = as_u(as_f(r[4 * j + e]) + as_f(v[j].v[e]));
            };
            auto load_chunk = [&](int u, int c, u32x4 (&v)[8]) {
                const float *q = part_chunk(u, c);
#pragma unroll
                for (int j = 0; j < 8; ++j) v[j] = ld_cg_v4(q + 128 * j);
            };
            // add the partials of the units after this one (their stages follow
            // in K order); from the second one on when the first is prefetched
            auto add_partials = [&](uint32_t(&r)[32], int c, int first) {
                for (int u2 = first; u2 < last; ++u2) {
                    u32x4 v[8];
                    load_chunk(u2, c, v);
                    add4(r, v);
                }
            };
            int m0i, n0i;
            tile_coords(tile, g.tiles_m, tiles_n, TMR, BN, m0i, n0i);
            const int64_t m0 = m0i + (int64_t)rank * GBM, n0 = n0i;  // this CTA's 128 rows
            const int64_t row0 = m0 + eg * 32, row = row0 + lane;
            const bool rows_in = ALIGNED || row0 < g.M;  // warp-uniform: any row of this warp inside C
            const bool row_in = ALIGNED || row < g.M;
            float *crow = g.C + row * g.ldc + n0;
            const int ncols = ALIGNED ? BN : (int)(g.N - n0 < BN ? g.N - n0 : BN);
            const bool tma_path = g.vec_c && rows_in;
            const int nchunks = (ncols + 31) / 32;
            // C of chunks 0 and 1 heads for this warp's staging buffers (both
            // free: the last tile ended with its stores' reads complete), the
            // rest into L2, while this tile's MMAs run
            if (use_c && !contrib && tma_path && lane == 0) {
                for (int ci = 0; ci < 2 && ci < nchunks; ++ci) {
                    const uint32_t bar = smem_u32(&s.cbar[eg][ci]);
                    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], 4096;" ::"r"(bar) : "memory");
                    tma_load(smem_u32(s.cbuf[eg][ci]), &m_c, (int)n0 + 32 * ci, (int)row0, bar);
                    loads_out |= 1u << ci;
                }
            }
            if (use_c && !contrib && row_in) {
                for (int c = tma_path ? 64 : 0; c < ncols; c += 32)
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(crow + c));
            }
            if (!acc_wait(smem_u32(&s.acc_full[ab]), ((uint32_t)t / 2) & 1u, g.KT, &s.abort) || gemm_aborted(&s.abort)) {
                if (!gemm_aborted(&s.abort)) gemm_fail(&s.abort, g.status);
                break;
            }
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const uint32_t tbase = tmem + ((uint32_t)(eg * 32) << 16) + ab * BN;
            bool ok = true;
            if (finish) {
                // wait until every later unit's epilogue warps have written their partials
                bool good = true;
                if (lane == 0) {
                    for (int u2 = unit + 1; good && u2 < last; ++u2) {
                        const long long w0 = clock64();
                        while (ld_acquire_u32(&g.flags[u2]) < kEpiWarps) {
                            if (gemm_aborted(&s.abort) || clock64() - w0 > kWaitCycles) {
                                good = false;
                                break;
                            }
                        }
                    }
                    if (!good && !gemm_aborted(&s.abort)) gemm_fail(&s.abort, g.status);
                }
                ok = __shfl_sync(0xffffffffu, good ? 1 : 0, 0) != 0;
                __threadfence();
            }
            if (contrib) {
                // the raw accumulator rows into this unit's partial slot (all rows and
                // columns: padding included), then this warp counts itself in
                for (int c = 0; c < BN; c += 32) {
                    uint32_t r[32];
                    tmem_ld32(tbase + (uint32_t)c, r);
                    float *q = part_chunk(unit, c);
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        st_cg_v4(q + 128 * j, {{r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]}});
                }
                __threadfence();
                __syncwarp();
                if (lane == 0) red_release_add_u32(&g.flags[unit], 1u);
            } else if (!ok) {
                // a partial never came: leave C alone
            } else if (tma_path) {
                // TMA path: C moves in 32 x 32 chunks through this warp's two
                // staging buffers; TMA clips rows >= M and columns >= N on the
                // store and reads them as 0 on the load.  A finishing unit
                // loads the next chunk of the first later unit's partial while
                // it adds the current one.
                u32x4 nxt[8];
                if (finish) load_chunk(unit + 1, 0, nxt);
                for (int ci = 0; ci < nchunks; ++ci) {
                    const int bsel = ci & 1;
                    if (ci >= 1 && lane == 0) {
                        bulk_wait_read();  // chunk ci-1's store has read its buffer (and ci-2's, this one)
                        if (use_c && ci + 1 < nchunks) {
                            const uint32_t bar = smem_u32(&s.cbar[eg][bsel ^ 1]);
                            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], 4096;" ::"r"(bar)
                                         : "memory");
                            tma_load(smem_u32(s.cbuf[eg][bsel ^ 1]), &m_c, (int)n0 + 32 * (ci + 1), (int)row0, bar);
                            loads_out |= 1u << (bsel ^ 1);
                        }
                    }
                    uint32_t r[32];
                    tmem_ld32(tbase + (uint32_t)(32 * ci), r);
                    if (finish) {
                        u32x4 cur[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j) cur[j] = nxt[j];
                        if (ci + 1 < nchunks) load_chunk(unit + 1, 32 * (ci + 1), nxt);
                        add4(r, cur);
                        add_partials(r, 32 * ci, unit + 2);
                    }
                    if (use_c) {
                        if (!mbar_wait_bounded(smem_u32(&s.cbar[eg][bsel]), (cpar >> bsel) & 1u)) {
                            gemm_fail(&s.abort, g.status);
                            ok = false;
                            break;
                        }
                        cpar ^= 1u << bsel;
                        loads_out &= ~(1u << bsel);
                    }
                    __syncwarp();
                    float *rowp = s.cbuf[eg][bsel] + lane * 32;
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        float4 *slot = reinterpret_cast<float4 *>(rowp + 4 * (q ^ (lane & 7)));
                        float4 v;
                        v.x = g.alpha * as_f(r[4 * q]);
                        v.y = g.alpha * as_f(r[4 * q + 1]);
                        v.z = g.alpha * as_f(r[4 * q + 2]);
                        v.w = g.alpha * as_f(r[4 * q + 3]);
                        if (use_c) {
                            const float4 cv = *slot;
                            v.x = __fmaf_rn(g.beta, cv.x, v.x);
                            v.y = __fmaf_rn(g.beta, cv.y, v.y);
                            v.z = __fmaf_rn(g.beta, cv.z, v.z);
                            v.w = __fmaf_rn(g.beta, cv.w, v.w);
                        }
                        *slot = v;
                    }
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the TMA store
                    __syncwarp();
                    if (lane == 0) tma_store(&m_c, (int)n0 + 32 * ci, (int)row0, smem_u32(s.cbuf[eg][bsel]));
                }
                if (lane == 0) bulk_wait_read();  // both buffers free for the next tile
                __syncwarp();
            } else if (rows_in) {
                // direct path (C not 16-byte aligned or ldc % 4 != 0): one row per lane
                for (int c = 0; c < ncols; c += 32) {  // warp-uniform: the TMEM load is .sync.aligned
                    uint32_t r[32];
                    tmem_ld32(tbase + (uint32_t)c, r);
                    if (finish) add_partials(r, c, unit + 1);
                    if (!row_in) continue;
                    float *p = crow + c;
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        if (c + e < ncols) {
                            float v = g.alpha * as_f(r[e]);
                            if (use_c) v = __fmaf_rn(g.beta, p[e], v);
                            p[e] = v;
                        }
                    }
                }
            }
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            const uint32_t freed = ab ? acc_empty1 : acc_empty0;
            if constexpr (PAIR)
                asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(freed) : "memory");
            else
                asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(freed) : "memory");
            if (!ok) break;
        }
        if (lane == 0) {
            bulk_wait_all();  // stores complete before the CTA (and its shared memory) goes away
            for (int j = 0; j < 2; ++j)  // a load still in flight after an abort lands first
                if (loads_out & (1u << j)) mbar_wait_bounded(smem_u32(&s.cbar[eg][j]), (cpar >> j) & 1u);
        }
        __syncwarp();
    }

    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if constexpr (PAIR) cluster_sync();  // the pair's MMAs, copies and remote arrivals are over
    if (warp == 1) {
        __syncwarp();
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        tmem_dealloc<PAIR>(tmem, kCols);
    }
}

// One thread waits, with the pipeline's own bounded wait, on an mbarrier that
// nothing arrives at; when the limit runs out it records the timeout exactly
// as a stalled gemm role does, and the kernel ends normally.
__global__ void __launch_bounds__(32) wait_timeout_probe(unsigned *status)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bar)));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        abort_flag = 0;
        if (!mbar_wait_bounded(smem_u32(&bar), 0u)) gemm_fail(&abort_flag, status);
    }
}

// ------------------------------------------------------------------ host

bool kmajor_map(CUtensorMap *m, float *base, int64_t rows, int64_t Kp, int box_rows, int BK)
{
    const cuuint64_t dims[2] = {(cuuint64_t)Kp, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)Kp * sizeof(float)};
    const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
    const cuuint32_t es[2] = {1, 1};
    return tensor_map_encoder()(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, es,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, BK == 32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct GemmPlan {
    int64_t Mp, Np, Kp;
    size_t bytes;     // workspace
    size_t off[6];    // a_hi, a_lo, b_hi, b_lo, split-K partials, split-K flags
};

GemmPlan gemm_plan(int64_t M, int64_t N, int64_t K, int TN)
{
    GemmPlan p;
    p.Mp = (M + 2 * GBM - 1) / (2 * GBM) * (2 * GBM);  // whole 256-row tiles: either TM fits
    p.Np = (N + TN - 1) / TN * TN;
    p.Kp = K > 0 ? (K + GBK - 1) / GBK * GBK : GBK;  // K = 0: one zero tile, acc = 0
    const size_t a = (size_t)(p.Mp * p.Kp) * sizeof(float), b = (size_t)(p.Np * p.Kp) * sizeof(float);
    auto up = [](size_t x) { return (x + 1023) & ~size_t(1023); };
    p.off[0] = 0;
    p.off[1] = up(a);
    p.off[2] = p.off[1] + up(a);
    p.off[3] = p.off[2] + up(b);
    // split-K partials: one accumulator per unit (units x tile rows <= the
    // 128-row tiles of C, and <= kMaxSms 128-row accumulators); one flag per unit
    // (none when K is too short for split-K: s parts save KT (s - 1) / s
    // stages, fewer than kSkMinSaved unless KT > kSkMinSaved)
    const int64_t n128 = (p.Mp / GBM) * (p.Np / TN);
    const size_t part = p.Kp / 16 > kSkMinSaved
                            ? (size_t)((n128 < kMaxSms ? n128 : kMaxSms) * GBM * TN) * sizeof(float)
                            : 0;
    p.off[4] = p.off[3] + up(b);
    p.off[5] = p.off[4] + up(part);
    p.bytes = p.off[5] + up(kMaxSms * sizeof(unsigned));
    return p;
}

template <int BN, int BK, bool THREE, bool ALIGNED, bool PAIR>
tm_status launch_gemm(const CUtensorMap *maps, const GemmArgs &g, unsigned grid, cudaStream_t s)
{
    constexpr int BH = PAIR ? BN / 2 : BN;
    constexpr int STAGES = gemm_stages<BH, BK, THREE>();
    static_assert(STAGES >= 2, "shared-memory ring needs two stages");
    const void *k = (const void *)gemm_tf32_kernel<BN, BK, STAGES, THREE, ALIGNED, PAIR>;
    const size_t smem = sizeof(GemmSmem<BH, BK, STAGES, THREE>) + 1024;
    static std::once_flag once[kMaxDevices];
    int dev = 0;
    cudaGetDevice(&dev);
    bool attr_ok = true;
    std::call_once(once[dev < 0 || dev >= kMaxDevices ? 0 : dev], [&] {
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) {
            cudaGetLastError();
            attr_ok = false;
        }
    });
    if (!attr_ok) return TM_ERR_CUDA;
    void *args[] = {const_cast<CUtensorMap *>(&maps[0]), const_cast<CUtensorMap *>(&maps[1]),
                    const_cast<CUtensorMap *>(&maps[2]), const_cast<CUtensorMap *>(&maps[3]),
                    const_cast<CUtensorMap *>(&maps[4]), const_cast<GemmArgs *>(&g)};
    // a programmatic dependent of the split pass; CTA pairs as 2-CTA clusters
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kGemmThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = PAIR ? 2 : 1;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = PAIR ? 2 : 1;
    if (cudaLaunchKernelExC(&cfg, k, args) != cudaSuccess) {
        cudaGetLastError();
        return TM_ERR_CUDA;
    }
    return TM_OK;
}

// Stages fill about 192 KB of shared memory: 3xTF32 stages hold hi and lo of
// both operands (96 KB at TN 256 and TK 32, 48 KB at TK 16, ...; a pair's CTA
// holds half of B), single-pass stages only hi, so that mode runs twice as many.
template <int BN, int BK, bool PAIR>
tm_status launch_gemm_cfg(bool three, bool aligned, const CUtensorMap *maps, const GemmArgs &g, unsigned grid,
                          cudaStream_t s)
{
    if (three)
        return aligned ? launch_gemm<BN, BK, true, true, PAIR>(maps, g, grid, s)
                       : launch_gemm<BN, BK, true, false, PAIR>(maps, g, grid, s);
    return aligned ? launch_gemm<BN, BK, false, true, PAIR>(maps, g, grid, s)
                   : launch_gemm<BN, BK, false, false, PAIR>(maps, g, grid, s);
}

template <bool PAIR>
tm_status launch_gemm_tiles(int TN, int TK, bool three, bool aligned, const CUtensorMap *maps, const GemmArgs &g,
                            unsigned grid, cudaStream_t s)
{
    if (TK == 32) {
        if (TN == 128) return launch_gemm_cfg<128, 32, PAIR>(three, aligned, maps, g, grid, s);
        return launch_gemm_cfg<256, 32, PAIR>(three, aligned, maps, g, grid, s);
    }
    if (TN == 128) return launch_gemm_cfg<128, 16, PAIR>(three, aligned, maps, g, grid, s);
    return launch_gemm_cfg<256, 16, PAIR>(three, aligned, maps, g, grid, s);
}

bool disjoint_bytes(const void *a, size_t na, const void *b, size_t nb)
{
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x + na <= y || y + nb <= x;
}

}  // namespace
}  // namespace libtm

using namespace libtm;

extern "C" size_t tm_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t TN)
{
    if (M <= 0 || N <= 0 || K < 0 || !(TN == 128 || TN == 256)) return 0;
    return gemm_plan(M, N, K, TN).bytes;
}

extern "C" tm_status tm_gemm(const float *A, int64_t lda, const float *B, int64_t ldb, float *C, int64_t ldc,
                             int64_t M, int64_t N, int64_t K, float alpha, float beta, int32_t TM, int32_t TN,
                             int32_t TK, uint32_t flags, void *workspace, size_t ws_bytes, tm_stream_t stream)
{
    if (M < 0 || N < 0 || K < 0) return TM_ERR_INVALID_ARG;
    if (!flags_ok(flags, TM_ALIGNED | TM_GEMM_TF32)) return TM_ERR_INVALID_ARG;
    if (!(TM == GBM || TM == 2 * GBM) || !(TK == 16 || TK == 32) || !(TN == 128 || TN == 256))
        return TM_ERR_UNSUPPORTED_TILE;
    if (!valid2d(C, ldc, M, N) || !valid2d(A, lda, M, K) || !valid2d(B, ldb, K, N)) return TM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return TM_OK;
    if (!aligned_to(C, 4) || (K > 0 && (!aligned_to(A, 4) || !aligned_to(B, 4)))) return TM_ERR_MISALIGNED;
    if (flags & TM_ALIGNED) {
        if (M % TM != 0 || N % TN != 0 || K % TK != 0) return TM_ERR_BROKEN_PROMISE;
    }
    const GemmPlan pl = gemm_plan(M, N, K, TN);
    if (pl.Mp > INT32_MAX || pl.Np > INT32_MAX || pl.Kp > INT32_MAX || (pl.Mp / TM) * (pl.Np / TN) > INT32_MAX)
        return TM_ERR_INVALID_ARG;
    if (workspace == nullptr || ws_bytes < pl.bytes || !aligned_to(workspace, 1024)) return TM_ERR_WORKSPACE;
    {
        uintptr_t clo, chi;
        span2d(C, ldc, M, N, &clo, &chi);
        const void *cp = reinterpret_cast<const void *>(clo);
        if (!disjoint_bytes(cp, chi - clo, workspace, pl.bytes)) return TM_ERR_INVALID_ARG;
        if (K > 0) {
            uintptr_t lo, hi;
            span2d(A, lda, M, K, &lo, &hi);
            if (!disjoint_bytes(cp, chi - clo, reinterpret_cast<const void *>(lo), hi - lo) ||
                !disjoint_bytes(workspace, pl.bytes, reinterpret_cast<const void *>(lo), hi - lo))
                return TM_ERR_INVALID_ARG;
            span2d(B, ldb, K, N, &lo, &hi);
            if (!disjoint_bytes(cp, chi - clo, reinterpret_cast<const void *>(lo), hi - lo) ||
                !disjoint_bytes(workspace, pl.bytes, reinterpret_cast<const void *>(lo), hi - lo))
                return TM_ERR_INVALID_ARG;
        }
    }

    const DevInfo *dev;
    tm_status st = device_info(&dev);
    if (st != TM_OK) return st;
    if (tensor_map_encoder() == nullptr) return TM_ERR_CUDA;
    cudaStream_t s = as_stream(stream);
    char *ws = static_cast<char *>(workspace);
    float *ahi = reinterpret_cast<float *>(ws + pl.off[0]), *alo = reinterpret_cast<float *>(ws + pl.off[1]);
    float *bhi = reinterpret_cast<float *>(ws + pl.off[2]), *blo = reinterpret_cast<float *>(ws + pl.off[3]);

    // 1. split (and transpose B) into zero-padded K-major tf32 hi/lo operands
    SplitArgs sa;
    sa.A = A;
    sa.B = B;
    sa.lda = lda;
    sa.ldb = ldb;
    sa.M = M;
    sa.N = N;
    sa.K = K;
    sa.Mp = pl.Mp;
    sa.Np = pl.Np;
    sa.Kp = pl.Kp;
    const bool three = !(flags & TM_GEMM_TF32);
    sa.ahi = ahi;
    sa.alo = three ? alo : nullptr;
    sa.bhi = bhi;
    sa.blo = three ? blo : nullptr;
    sa.flags = reinterpret_cast<unsigned *>(ws + pl.off[5]);
    sa.nflags = kMaxSms;
    {
        // A: up to 8 blocks per SM over rows (each streams whole padded rows);
        // B: up to 32 per SM over 32 x 32 tiles (each tile is a short
        // load-transpose-store round trip, so more blocks keep more in flight)
        const int64_t tiles_b = (pl.Kp / 32) * (pl.Np / 32);
        const int64_t na = pl.Mp < 8LL * dev->sms ? pl.Mp : 8LL * dev->sms;
        const int64_t nb = tiles_b < 32LL * dev->sms ? tiles_b : 32LL * dev->sms;
        sa.blocks_a = (unsigned)na;
        sa.blocks_b = (unsigned)nb;
    }
    split_operands<<<sa.blocks_a + sa.blocks_b, 256, 0, s>>>(sa);
    if ((st = launch_status()) != TM_OK) return st;

    // 2. the tensor-core gemm over whole tiles
    CUtensorMap maps[5] = {};
    // each CTA copies 128 rows of A and its TN (one CTA) or TN / 2 (a pair) rows of B per stage
    const int b_rows = TM == 2 * GBM ? TN / 2 : TN;
    if (!kmajor_map(&maps[0], ahi, pl.Mp, pl.Kp, GBM, TK) || !kmajor_map(&maps[1], alo, pl.Mp, pl.Kp, GBM, TK) ||
        !kmajor_map(&maps[2], bhi, pl.Np, pl.Kp, b_rows, TK) || !kmajor_map(&maps[3], blo, pl.Np, pl.Kp, b_rows, TK))
        return TM_ERR_CUDA;
    // C as 32 x 32 TMA chunks (the epilogue's staging unit), when its rows
    // start on 16-byte boundaries and N % 4 == 0: a TMA store clips the inner
    // dimension only at 16-byte granularity (measured: with N = 1 it wrote
    // columns 1-3 of the row's padding), so a row end inside a 16-byte piece
    // would be overrun.  Otherwise the epilogue writes C directly.
    const bool vec_c = aligned_to(C, 16) && ldc % 4 == 0 && N % 4 == 0;
    if (vec_c) {
        const cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)M};
        const cuuint64_t strides[1] = {(cuuint64_t)ldc * sizeof(float)};
        const cuuint32_t box[2] = {32, 32};
        const cuuint32_t es[2] = {1, 1};
        if (tensor_map_encoder()(&maps[4], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, C, dims, strides, box, es,
                             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return TM_ERR_CUDA;
    }
    GemmArgs g;
    g.C = C;
    g.ldc = ldc;
    g.M = M;
    g.N = N;
    g.alpha = alpha;
    g.beta = beta;
    g.KT = (int)(pl.Kp / TK);
    g.tiles_m = (int)(pl.Mp / TM);
    g.ntiles = (int)((pl.Mp / TM) * (pl.Np / TN));
    g.vec_c = vec_c;
    g.status = dev->status;
    const bool aligned = (flags & TM_ALIGNED) != 0;
    // persistent: one CTA per SM, or one 2-CTA cluster per SM pair
    const bool pair = TM == 2 * GBM;
    const int sms = dev->sms < kMaxSms ? dev->sms : kMaxSms;
    const int slots = pair ? sms / 2 : sms;
    const int units = g.ntiles < slots ? g.ntiles : slots;
    // split-K of the last round: when its rem tiles would leave at least
    // half of the units idle, each is cut along K into s = units / rem parts
    // run side by side (so the units that share A or B rows read them at the
    // same K, as in the whole rounds).  The round then takes KT / s stages
    // instead of KT; it pays when that saves at least kSkMinSaved stages
    // (the parts' cost -- partials written and read back, a finishing
    // epilogue that waits for them -- measured ~10 stages of 3xTF32, ~30 of
    // the single pass).  gemm_8192: 36 tiles on 76 pairs, s = 2, 128 stages
    // saved; gemm_4100: 61 tiles on 76 pairs, no split.
    const int rem = g.ntiles % units;
    g.dp_tiles = g.ntiles;
    g.sk_split = 0;
    if (g.ntiles > units && rem != 0) {
        const int split = units / rem;
        if (split >= 2 && (int64_t)g.KT * (split - 1) >= (int64_t)kSkMinSaved * split) {
            g.dp_tiles = g.ntiles - rem;
            g.sk_split = split;
        }
    }
    g.part = reinterpret_cast<float *>(ws + pl.off[4]);
    g.flags = reinterpret_cast<unsigned *>(ws + pl.off[5]);
    if (pair) return launch_gemm_tiles<true>(TN, TK, three, aligned, maps, g, 2u * (unsigned)units, s);
    return launch_gemm_tiles<false>(TN, TK, three, aligned, maps, g, (unsigned)units, s);
}

extern "C" tm_status tm_wait_timeout_probe(tm_stream_t stream)
{
    const DevInfo *dev;
    tm_status st = device_info(&dev);
    if (st != TM_OK) return st;
    wait_timeout_probe<<<1, 32, 0, as_stream(stream)>>>(dev->status);
    return launch_status();
}
