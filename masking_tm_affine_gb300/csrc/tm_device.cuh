// tm_device.cuh -- device-side building blocks shared by the libtm kernels.
//
// Global accesses are written as inline PTX so the instruction each path
// issues is fixed by the source, not left to the vectoriser: the puzzle
// "Aligned Load & Store" ("Solution") is exactly about the gap between four
// scalar `ld.global.nc.f32` and one `ld.global.nc.v4.f32` per 4-element chunk.
// Loads of read-only inputs use the non-coherent path with L1::no_allocate
// (each byte is read once); values move as raw 32-bit words so a copy keeps
// NaN payloads bit for bit.
#pragma once

#include <cstdint>

namespace libtm {

// Status word bits (one word per device; read and cleared by tm_check).
enum : unsigned {
    kStatusBrokenPromise = 1u,  // aligned path entered with M % TM or N % TN != 0
    kStatusMisaligned = 2u,     // aligned path entered with a pointer or ld off the vector grid
    kStatusTimeout = 4u,        // a bounded wait gave up
};

struct u32x4 {
    uint32_t v[4];
};
struct u32x8 {
    uint32_t v[8];
};

// ---------------------------------------------------------------- loads
__device__ __forceinline__ uint32_t ld_nc_b32(const void *p)
{
    uint32_t r;
    asm volatile("ld.global.nc.L1::no_allocate.b32 %0, [%1];" : "=r"(r) : "l"(p));
    return r;
}

__device__ __forceinline__ u32x4 ld_nc_v4(const void *p)
{
    u32x4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.v[0]), "=r"(r.v[1]), "=r"(r.v[2]), "=r"(r.v[3])
                 : "l"(p));
    return r;
}

// 32-byte access: sm_100-class GPUs accept .v8 for 32-bit types in .global.
__device__ __forceinline__ u32x8 ld_nc_v8(const void *p)
{
    u32x8 r;
    asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r.v[0]), "=r"(r.v[1]), "=r"(r.v[2]), "=r"(r.v[3]), "=r"(r.v[4]),
                   "=r"(r.v[5]), "=r"(r.v[6]), "=r"(r.v[7])
                 : "l"(p));
    return r;
}

// Cached read-only loads for small vectors every row reuses (per-channel
// parameters): these keep the default L1 allocation.
__device__ __forceinline__ uint32_t ldg_b32(const void *p)
{
    uint32_t r;
    asm volatile("ld.global.nc.b32 %0, [%1];" : "=r"(r) : "l"(p));
    return r;
}

__device__ __forceinline__ u32x4 ldg_v4(const void *p)
{
    u32x4 r;
    asm volatile("ld.global.nc.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.v[0]), "=r"(r.v[1]), "=r"(r.v[2]), "=r"(r.v[3])
                 : "l"(p));
    return r;
}

// ---------------------------------------------------------------- stores
__device__ __forceinline__ void st_b32(void *p, uint32_t x)
{
    asm volatile("st.global.b32 [%0], %1;" ::"l"(p), "r"(x) : "memory");
}

__device__ __forceinline__ void st_v4(void *p, const u32x4 &x)
{
    asm volatile("st.global.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(x.v[0]), "r"(x.v[1]),
                 "r"(x.v[2]), "r"(x.v[3])
                 : "memory");
}

__device__ __forceinline__ void st_v8(void *p, const u32x8 &x)
{
    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(x.v[0]),
                 "r"(x.v[1]), "r"(x.v[2]), "r"(x.v[3]), "r"(x.v[4]), "r"(x.v[5]), "r"(x.v[6]),
                 "r"(x.v[7])
                 : "memory");
}

__device__ __forceinline__ float as_f(uint32_t u) { return __uint_as_float(u); }

// Data written earlier by other blocks of the same grid (partial sums): read
// at L2, the point of coherence, never from a possibly stale L1 line.
__device__ __forceinline__ u32x4 ld_l2_v4(const void *p)
{
    u32x4 r;
    asm volatile("ld.global.cg.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.v[0]), "=r"(r.v[1]), "=r"(r.v[2]), "=r"(r.v[3])
                 : "l"(p)
                 : "memory");
    return r;
}

// Drop the 128-byte L2 line at p (128-byte aligned) without writing it back:
// for scratch that nothing reads again, so its dirty lines cost no DRAM write.
__device__ __forceinline__ void discard_l2_line(const void *p)
{
    asm volatile("discard.global.L2 [%0], 128;" ::"l"(p) : "memory");
}

// ---------------------------------------------------------------- mbarriers
// Bounded waits on shared-memory mbarriers (the TMA pipelines of the staged
// column sum and the gemm).  A wait gives up after kWaitCycles SM clock cycles
// (~1 s at full clock): the caller then records kStatusTimeout, drains what it
// started and exits, so a stalled pipeline never hangs the GPU.
constexpr long long kWaitCycles = 2000000000LL;

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the completion of phase `parity` of the mbarrier at shared address
// `bar`; false if it has not completed within `limit` cycles.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, long long limit = kWaitCycles)
{
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > limit) return false;
    return true;
}

// An L2 cache policy that marks lines evict-first: for data read once (a TMA
// copy of a streamed tile), so that it, and not older lines still to be
// written back, is what L2 gives up first.
__device__ __forceinline__ uint64_t l2_evict_first_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// ---------------------------------------------------------------- clusters
// Rank of this CTA in its cluster, the address of a shared variable in CTA
// `rank` of the cluster (distributed shared memory), and a full cluster
// barrier with release/acquire ordering of shared-memory accesses.
__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_addr(uint32_t a, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}

__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- dependent launch
// Programmatic dependent launch: a kernel launched with the programmatic
// stream-serialization attribute may start (and run its prologue) while the
// kernel before it in the stream finishes; pdl_wait() then blocks the calling
// thread until that kernel has completed and its writes are visible.  In a
// normally launched kernel both are no-ops.  pdl_trigger() lets the dependent
// launch begin once every block of this grid has issued it or exited.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// The library's streaming kernels all follow one rule so that any of them may
// be launched as a dependent (TM_PDL): pdl_trigger() at entry, pdl_wait() in
// every thread before its first global store, and pdl_wait() before exit in a
// thread that stored nothing.  Loads of the inputs may therefore run ahead of
// the previous kernel; no write may, and no grid completes before the grid it
// depends on, which keeps a chain of dependent launches in stream order.
__device__ __forceinline__ uint32_t as_u(float f) { return __float_as_uint(f); }

// ---------------------------------------------------------------- tile walk
// The split of a loop over a runtime extent K in steps of T into whole tiles
// (no mask) and at most one masked remainder tile ("Slicing, bounds and
// masking", "Loops over a dynamic extent": K = 1000, T = 16 gives 62 + 1 over
// 8 columns).  Every kernel that walks a runtime extent takes its bounds from
// here; tm_tile_walk_probe exposes it to the tests.
struct TileWalk {
    int64_t whole;   // tiles that lie entirely inside [0, K)
    int64_t masked;  // 1 if a partial tile remains, else 0
    int64_t rem;     // extent of that partial tile (K - whole*T)
    int64_t iters;   // whole + masked
};

__host__ __device__ __forceinline__ TileWalk tile_walk(int64_t K, int64_t T)
{
    TileWalk w;
    w.whole = K / T;
    w.rem = K - w.whole * T;
    w.masked = w.rem > 0 ? 1 : 0;
    w.iters = w.whole + w.masked;
    return w;
}

// ---------------------------------------------------------------- division
// n / d for 0 <= n < 2^31 and 1 <= d < 2^31 by multiply-high and shift (the
// round-up method of Granlund and Montgomery, "Division by invariant integers
// using multiplication", PLDI 1994).  Built on the host, used per element on
// the device where a runtime divisor would otherwise cost a division loop.
struct FastDiv {
    uint32_t d, mul, shift;
};

__device__ __forceinline__ uint32_t fdiv(uint32_t n, const FastDiv &f)
{
    return (__umulhi(n, f.mul) + n) >> f.shift;
}

}  // namespace libtm
