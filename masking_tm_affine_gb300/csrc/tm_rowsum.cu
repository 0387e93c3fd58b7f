// tm_rowsum.cu -- r[i] = sum_j X[i, j], the stride-1 walk.
//
// Source: "Memory Coalescing and Tensor Layout" ("What it actually costs": the
// row-order walk of a row-major matrix, consecutive lanes on consecutive
// addresses).  The row is walked in TN-column tiles as "Slicing, bounds and
// masking" ("Loops over a dynamic extent") splits any loop over a runtime
// extent: the whole tiles carry no mask, then one masked remainder tile whose
// missing columns read 0, the right fill for a sum ("Reductions over a ragged
// tile").
//
// GB300 design: one warp per row, TM warps per block, persistent grid over
// row blocks.  In the vector path each lane takes TN/128 16-byte vectors per
// tile and several tiles are in flight per step (8 vectors = 128 bytes per
// lane); the warp's partial sums meet in a butterfly of shuffles, so the
// summation order is fixed and the result is identical run to run.
#include "tm_host.h"

namespace libtm {
namespace {

template <int TN, bool VEC, bool ALIGNED>
__global__ void __launch_bounds__(1024, 1) rowsum_kernel(const float *__restrict__ X, int64_t ldx, int64_t M,
                                                      int64_t N, float *__restrict__ r, int TM, unsigned *status)
{
    constexpr int EW = VEC ? 4 : 1;                   // elements per access
    constexpr int PER_TILE = TN / (32 * EW);          // accesses per lane per tile
    constexpr int TPS = PER_TILE >= 8 ? 1 : 8 / PER_TILE;  // tiles per unrolled step
    static_assert(PER_TILE >= 1, "tile narrower than a warp's access");

    if constexpr (ALIGNED) {
        const bool whole = (M % TM == 0) && (N % TN == 0);
        const bool grid_ok = !VEC || ((ldx % 4 == 0) && (reinterpret_cast<uintptr_t>(X) & 15) == 0);
        if (!whole || !grid_ok) {
            if (blockIdx.x == 0 && threadIdx.x == 0)
                atomicOr(status, whole ? kStatusMisaligned : kStatusBrokenPromise);
            return;
        }
    }

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const TileWalk walk = tile_walk(N, TN);
    const int64_t row_blocks = (M + TM - 1) / TM;

    for (int64_t rb = blockIdx.x; rb < row_blocks; rb += gridDim.x) {
        const int64_t row = rb * TM + warp;
        if (!ALIGNED && row >= M) continue;  // row mask (warp-uniform)
        const float *xr = X + row * ldx;
        float acc[EW];
#pragma unroll
        for (int e = 0; e < EW; ++e) acc[e] = 0.0f;

        // whole tiles, TPS at a time, no mask
        int64_t t = 0;
        for (; t + TPS <= walk.whole; t += TPS) {
            uint32_t v[TPS * PER_TILE][EW];
#pragma unroll
            for (int q = 0; q < TPS * PER_TILE; ++q) {
                const float *p = xr + t * TN + ((int64_t)q * 32 + lane) * EW;
                if constexpr (VEC) {
                    u32x4 w = ld_nc_v4(p);
#pragma unroll
                    for (int e = 0; e < 4; ++e) v[q][e] = w.v[e];
                } else {
                    v[q][0] = ld_nc_b32(p);
                }
            }
#pragma unroll
            for (int q = 0; q < TPS * PER_TILE; ++q)
#pragma unroll
                for (int e = 0; e < EW; ++e) acc[e] += as_f(v[q][e]);
        }
        // leftover whole tiles, one at a time, no mask
        for (; t < walk.whole; ++t) {
#pragma unroll
            for (int q = 0; q < PER_TILE; ++q) {
                const float *p = xr + t * TN + ((int64_t)q * 32 + lane) * EW;
                if constexpr (VEC) {
                    u32x4 w = ld_nc_v4(p);
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[e] += as_f(w.v[e]);
                } else {
                    acc[0] += as_f(ld_nc_b32(p));
                }
            }
        }
        // the masked remainder tile: columns past N read as 0
        if (!ALIGNED && walk.masked) {
            const int64_t kt = walk.whole * TN;
#pragma unroll
            for (int q = 0; q < PER_TILE; ++q) {
                const int64_t j = kt + ((int64_t)q * 32 + lane) * EW;
                if constexpr (VEC) {
                    u32x4 w = {{0u, 0u, 0u, 0u}};
                    if (j < N) w = ld_nc_v4(xr + j);  // N % 4 == 0: a vector is wholly in or out
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[e] += as_f(w.v[e]);
                } else {
                    acc[0] += j < N ? as_f(ld_nc_b32(xr + j)) : 0.0f;
                }
            }
        }
        float s = acc[0];
#pragma unroll
        for (int e = 1; e < EW; ++e) s += acc[e];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) r[row] = s;
    }
}

template <int TN>
tm_status launch(bool vec, bool aligned, const float *X, int64_t ldx, int64_t M, int64_t N, float *r, int TM,
                 const DevInfo *dev, cudaStream_t s)
{
    const void *k;
    if (vec) k = aligned ? (const void *)rowsum_kernel<TN, true, true> : (const void *)rowsum_kernel<TN, true, false>;
    else k = aligned ? (const void *)rowsum_kernel<TN, false, true> : (const void *)rowsum_kernel<TN, false, false>;
    const int threads = 32 * TM;
    const int64_t grid = persistent_grid(dev, k, (M + TM - 1) / TM, 0, threads);
    unsigned *status = dev->status;
    void *args[] = {(void *)&X, (void *)&ldx, (void *)&M, (void *)&N, (void *)&r, (void *)&TM, (void *)&status};
    if (cudaLaunchKernel(k, dim3((unsigned)grid), dim3(threads), args, 0, s) != cudaSuccess) {
        cudaGetLastError();
        return TM_ERR_CUDA;
    }
    return TM_OK;
}

}  // namespace
}  // namespace libtm

using namespace libtm;

extern "C" tm_status tm_rowsum(const float *X, int64_t ldx, int64_t M, int64_t N, float *r, int32_t TM,
                               int32_t TN, uint32_t flags, tm_stream_t stream)
{
    if (!valid2d(X, ldx, M, N)) return TM_ERR_INVALID_ARG;
    if (M > 0 && r == nullptr) return TM_ERR_INVALID_ARG;
    if (!flags_ok(flags, TM_ALIGNED | TM_PATH_SCALAR | TM_PATH_VEC)) return TM_ERR_INVALID_ARG;
    if (!(TM == 1 || TM == 2 || TM == 4 || TM == 8 || TM == 16 || TM == 32)) return TM_ERR_UNSUPPORTED_TILE;
    if (!(TN == 128 || TN == 256 || TN == 512 || TN == 1024)) return TM_ERR_UNSUPPORTED_TILE;
    if (M > 0 && !aligned_to(r, 4)) return TM_ERR_MISALIGNED;
    if (M > 0 && N > 0 && !aligned_to(X, 4)) return TM_ERR_MISALIGNED;
    if (M > 0 && N > 0) {
        uintptr_t xlo, xhi, rlo = reinterpret_cast<uintptr_t>(r), rhi = rlo + (uintptr_t)M * 4;
        span2d(X, ldx, M, N, &xlo, &xhi);
        if (!(xhi <= rlo || rhi <= xlo)) return TM_ERR_INVALID_ARG;
    }
    const bool vec16 = aligned_to(X, 16) && ldx % 4 == 0;
    const bool aligned = (flags & TM_ALIGNED) != 0;
    bool vec;
    if (aligned) {
        if (!vec16 && !(flags & TM_PATH_SCALAR)) return TM_ERR_MISALIGNED;
        if (M % TM != 0 || N % TN != 0) return TM_ERR_BROKEN_PROMISE;
        vec = !(flags & TM_PATH_SCALAR);
    } else if (flags & TM_PATH_SCALAR) {
        vec = false;
    } else if (vec16 && N % 4 == 0) {
        vec = true;
    } else if (flags & TM_PATH_VEC) {
        return TM_ERR_MISALIGNED;
    } else {
        vec = false;
    }
    if (M == 0) return TM_OK;

    const DevInfo *dev;
    tm_status st = device_info(&dev);
    if (st != TM_OK) return st;
    cudaStream_t s = as_stream(stream);
    switch (TN) {
    case 128: return launch<128>(vec, aligned, X, ldx, M, N, r, TM, dev, s);
    case 256: return launch<256>(vec, aligned, X, ldx, M, N, r, TM, dev, s);
    case 512: return launch<512>(vec, aligned, X, ldx, M, N, r, TM, dev, s);
    default: return launch<1024>(vec, aligned, X, ldx, M, N, r, TM, dev, s);
    }
}
