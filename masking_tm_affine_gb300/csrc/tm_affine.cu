// tm_affine.cu -- the 1-D map out[i] = a[i]*2 + 1 through four access patterns.
//
// Source: "Aligned Load & Store" (Mojo GPU puzzles, puzzle 35).  "The
// exercise": SCALE = 2, BIAS = 1 over a 1M-element float32 buffer, computed by
// a scalar kernel, a vector kernel whose alignment is under-stated (four scalar
// loads and stores per 4-element chunk) and an aligned vector kernel (one
// 16-byte load and store per chunk).  "Solution": the vector kernels guard with
// base + 4 <= size, which leaves the size % 4 tail unwritten; here a scalar
// tail writes it, so every variant writes all n elements and all are
// bit-identical (2a is exact, so 2a + 1 is one rounding, with or without FMA).
//
// GB300 design: the fast variants give every thread U independent vector
// loads in flight and run one block per 256*U-vector chunk (a flat grid the
// block scheduler balances); VEC8 uses the 32-byte global access sm_100-class
// GPUs provide.  SCALAR and VEC_UNALIGNED keep the puzzle's
// one-unit-per-thread grids: they are the instruction-mix foils.
#include "tm_host.h"

namespace libtm {
namespace {

__device__ __forceinline__ uint32_t affine1(uint32_t a)
{
    return as_u(fmaf(as_f(a), 2.0f, 1.0f));  // SCALE = 2, BIAS = 1
}

// SCALAR: one element per thread.
__global__ void __launch_bounds__(kThreads) affine_scalar(const float *a, float *out, int64_t n)
{
    pdl_trigger();
    pdl_wait();
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < n; i += stride)
        st_b32(out + i, affine1(ld_nc_b32(a + i)));
}

// VEC_UNALIGNED: a 4-element chunk per thread, moved by four 4-byte accesses
// each way (the under-stated alignment of the puzzle), then the scalar tail.
__global__ void __launch_bounds__(kThreads) affine_vec_unaligned(const float *a, float *out, int64_t n)
{
    pdl_trigger();
    pdl_wait();
    const int64_t chunks = n / 4;
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    for (int64_t c = (int64_t)blockIdx.x * kThreads + threadIdx.x; c < chunks; c += stride) {
        const int64_t base = c * 4;  // base + 4 <= n holds for every chunk
        const uint32_t v0 = ld_nc_b32(a + base + 0);
        const uint32_t v1 = ld_nc_b32(a + base + 1);
        const uint32_t v2 = ld_nc_b32(a + base + 2);
        const uint32_t v3 = ld_nc_b32(a + base + 3);
        st_b32(out + base + 0, affine1(v0));
        st_b32(out + base + 1, affine1(v1));
        st_b32(out + base + 2, affine1(v2));
        st_b32(out + base + 3, affine1(v3));
    }
    const int64_t t = chunks * 4 + threadIdx.x;
    if (blockIdx.x == 0 && t < n) st_b32(out + t, affine1(ld_nc_b32(a + t)));
}

// VEC4 / VEC8: U vectors of VW elements in flight per thread, one chunk of
// kThreads*U vectors per block (grid-stride beyond the grid limit).
// Elements [0, head) are a scalar prologue that brings `a + head` and
// `out + head` onto the vector grid (both have the same misalignment); the
// vector body covers [head, head + nvec*VW); the rest is the scalar tail.
template <int VW, int U>
__global__ void __launch_bounds__(kThreads) affine_vec(const float *a, float *out, int64_t n, int64_t head)
{
    pdl_trigger();
    const float *va = a + head;
    float *vo = out + head;
    const int64_t nvec = (n - head) / VW;
    constexpr int64_t kPerIter = (int64_t)kThreads * U;
    const int64_t iters = nvec / kPerIter;
    bool waited = false;
    for (int64_t it = blockIdx.x; it < iters; it += gridDim.x) {
        const int64_t v0 = it * kPerIter + threadIdx.x;
        uint32_t r[U][VW];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const float *src = va + (v0 + (int64_t)u * kThreads) * VW;
            if constexpr (VW == 4) {
                u32x4 t = ld_nc_v4(src);
#pragma unroll
                for (int e = 0; e < 4; ++e) r[u][e] = t.v[e];
            } else {
                u32x8 t = ld_nc_v8(src);
#pragma unroll
                for (int e = 0; e < 8; ++e) r[u][e] = t.v[e];
            }
        }
        if (!waited) {  // the loads above may run ahead of the previous kernel, the stores may not
            pdl_wait();
            waited = true;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            float *dst = vo + (v0 + (int64_t)u * kThreads) * VW;
            if constexpr (VW == 4) {
                u32x4 t;
#pragma unroll
                for (int e = 0; e < 4; ++e) t.v[e] = affine1(r[u][e]);
                st_v4(dst, t);
            } else {
                u32x8 t;
#pragma unroll
                for (int e = 0; e < 8; ++e) t.v[e] = affine1(r[u][e]);
                st_v8(dst, t);
            }
        }
    }
    if (!waited) pdl_wait();
    // vectors left over after the whole iterations: one per thread
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    for (int64_t v = iters * kPerIter + (int64_t)blockIdx.x * kThreads + threadIdx.x; v < nvec; v += stride) {
        const float *src = va + v * VW;
        float *dst = vo + v * VW;
        if constexpr (VW == 4) {
            u32x4 t = ld_nc_v4(src);
#pragma unroll
            for (int e = 0; e < 4; ++e) t.v[e] = affine1(t.v[e]);
            st_v4(dst, t);
        } else {
            u32x8 t = ld_nc_v8(src);
#pragma unroll
            for (int e = 0; e < 8; ++e) t.v[e] = affine1(t.v[e]);
            st_v8(dst, t);
        }
    }
    // scalar prologue and tail, on the last block
    if (blockIdx.x == gridDim.x - 1) {
        if (threadIdx.x < head) st_b32(out + threadIdx.x, affine1(ld_nc_b32(a + threadIdx.x)));
        const int64_t t = head + nvec * VW + threadIdx.x;
        if (t < n) st_b32(out + t, affine1(ld_nc_b32(a + t)));
    }
}

constexpr int kUnroll4 = 4;
constexpr int kUnroll8 = 2;

}  // namespace
}  // namespace libtm

using namespace libtm;

extern "C" tm_status tm_affine(const float *a, float *out, int64_t n, tm_variant variant_pdl, tm_stream_t stream)
{
    const bool pdl = ((uint32_t)variant_pdl & TM_PDL) != 0;
    const tm_variant variant = (tm_variant)((uint32_t)variant_pdl & ~TM_PDL);
    if (n < 0) return TM_ERR_INVALID_ARG;
    if (n > 0 && (a == nullptr || out == nullptr)) return TM_ERR_INVALID_ARG;
    if (variant != TM_VAR_AUTO && variant != TM_VAR_SCALAR && variant != TM_VAR_VEC_UNALIGNED &&
        variant != TM_VAR_VEC4 && variant != TM_VAR_VEC8)
        return TM_ERR_INVALID_ARG;
    if (!overlap_ok(a, n, out, n, 1, n)) return TM_ERR_INVALID_ARG;
    if (n > 0 && (!aligned_to(a, 4) || !aligned_to(out, 4))) return TM_ERR_MISALIGNED;
    if (n > INT64_MAX / 8) return TM_ERR_INVALID_ARG;

    const uintptr_t pa = reinterpret_cast<uintptr_t>(a), po = reinterpret_cast<uintptr_t>(out);
    int vw = 0;        // 0 = scalar kernel
    int64_t head = 0;  // scalar prologue length
    switch (variant) {
    case TM_VAR_VEC4:
        if (!aligned_to(a, 16) || !aligned_to(out, 16)) return TM_ERR_MISALIGNED;
        vw = 4;
        break;
    case TM_VAR_VEC8:
        if (!aligned_to(a, 32) || !aligned_to(out, 32)) return TM_ERR_MISALIGNED;
        vw = 8;
        break;
    case TM_VAR_AUTO:
        // widest access both pointers reach after the same scalar prologue
        if ((pa & 31) == (po & 31)) {
            vw = 8;
            head = (int64_t)(((32 - (pa & 31)) & 31) / 4);
        } else if ((pa & 15) == (po & 15)) {
            vw = 4;
            head = (int64_t)(((16 - (pa & 15)) & 15) / 4);
        }
        if (head > n) head = n;
        break;
    default:
        break;
    }
    if (n == 0) return TM_OK;

    const DevInfo *dev;
    tm_status st = device_info(&dev);
    if (st != TM_OK) return st;
    cudaStream_t s = as_stream(stream);

    if (variant == TM_VAR_SCALAR || (variant == TM_VAR_AUTO && vw == 0)) {
        int64_t grid = (n + kThreads - 1) / kThreads;
        if (grid > INT32_MAX) grid = INT32_MAX;
        void *args[] = {(void *)&a, (void *)&out, (void *)&n};
        return launch_kernel((const void *)affine_scalar, dim3((unsigned)grid), dim3(kThreads), args, 0, s, pdl);
    }
    if (variant == TM_VAR_VEC_UNALIGNED) {
        int64_t grid = (n / 4 + kThreads - 1) / kThreads;
        if (grid < 1) grid = 1;
        if (grid > INT32_MAX) grid = INT32_MAX;
        void *args[] = {(void *)&a, (void *)&out, (void *)&n};
        return launch_kernel((const void *)affine_vec_unaligned, dim3((unsigned)grid), dim3(kThreads), args, 0, s,
                             pdl);
    }
    const int64_t nvec = (n - head) / vw;
    const int64_t chunks = nvec / (kThreads * (vw == 4 ? kUnroll4 : kUnroll8));
    const unsigned grid = flat_grid(chunks > 0 ? chunks : (nvec + kThreads - 1) / kThreads);
    const void *k = vw == 4 ? (const void *)affine_vec<4, kUnroll4> : (const void *)affine_vec<8, kUnroll8>;
    void *args[] = {(void *)&a, (void *)&out, (void *)&n, (void *)&head};
    return launch_kernel(k, dim3(grid), dim3(kThreads), args, 0, s, pdl);
}
