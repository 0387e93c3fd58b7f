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
// GB300 design: a block of 256 threads takes TM rows, L = 256/TM lanes per
// row.  The whole tiles of a row form one contiguous unmasked prefix, which
// the row's lanes stride through with U independent 16-byte loads in flight
// each; then the lanes cover the remainder tile with masked loads.  The L
// partial sums of a row meet in a shuffle butterfly (plus shared memory when
// L > 32), so the summation order is fixed and the result identical run to
// run.  The grid is flat -- one block per TM-row band -- for the block
// scheduler to balance (TM = 1, a block per row, measured fastest on long rows).
// Four blocks per SM, so that a lane's U vector loads all fit in registers
// and go out together: without the bound the compiler chose 32 registers and
// serialised part of every batch ([8192, 8192]: 40.1 against 37.9 us by
// kernel time; [4096, 4096]: 12.6 against 12.0 us).
#include "tm_host.h"

namespace libtm {
namespace {

template <int TM, bool VEC, bool ALIGNED>
__global__ void __launch_bounds__(kThreads, 4) rowsum_kernel(const float *__restrict__ X, int64_t ldx, int64_t M,
                                                          int64_t N, float *__restrict__ r, int TN, unsigned *status)
{
    constexpr int L = kThreads / TM;   // lanes sharing a row
    constexpr int EW = VEC ? 4 : 1;    // elements per access
    constexpr int U = VEC ? 8 : 16;    // accesses in flight per lane
    constexpr int W = L > 32 ? L / 32 : 1;  // warps per row
    __shared__ float part[TM][W];

    pdl_trigger();
    if constexpr (ALIGNED) {
        const bool whole = (M % TM == 0) && (N % TN == 0);
        const bool grid_ok = !VEC || ((ldx % 4 == 0) && (reinterpret_cast<uintptr_t>(X) & 15) == 0);
        if (!whole || !grid_ok) {
            if (blockIdx.x == 0 && threadIdx.x == 0)
                atomicOr(status, whole ? kStatusMisaligned : kStatusBrokenPromise);
            pdl_wait();
            return;
        }
    }
    const int lr = threadIdx.x / L, ln = threadIdx.x % L;
    const TileWalk walk = tile_walk(N, TN);
    const int64_t prefix = walk.whole * TN / EW;  // accesses in the whole tiles
    const int64_t row_blocks = (M + TM - 1) / TM;

    for (int64_t rb = blockIdx.x; rb < row_blocks; rb += gridDim.x) {
        const int64_t row = rb * TM + lr;
        const bool live = ALIGNED || row < M;  // row mask
        float acc[EW];
#pragma unroll
        for (int e = 0; e < EW; ++e) acc[e] = 0.0f;
        if (live) {
            const float *xr = X + row * ldx;
            // whole tiles: no mask.  U loads in flight per lane; the last batch
            // of a row may be partial (lanes past the prefix add nothing), but
            // it still issues all its loads before the first add
            for (int64_t v = ln; v < prefix; v += (int64_t)L * U) {
                const bool full = v + (int64_t)L * (U - 1) < prefix;
                uint32_t w[U][EW];
#pragma unroll
                for (int q = 0; q < U; ++q) {
                    const float *p = xr + (v + (int64_t)L * q) * EW;
#pragma unroll
                    for (int e = 0; e < EW; ++e) w[q][e] = 0u;
                    if (full || v + (int64_t)L * q < prefix) {
                        if constexpr (VEC) {
                            const u32x4 t = ld_nc_v4(p);
#pragma unroll
                            for (int e = 0; e < 4; ++e) w[q][e] = t.v[e];
                        } else {
                            w[q][0] = ld_nc_b32(p);
                        }
                    }
                }
#pragma unroll
                for (int q = 0; q < U; ++q)
#pragma unroll
                    for (int e = 0; e < EW; ++e) acc[e] += as_f(w[q][e]);
            }
            // the masked remainder tile: columns past N read as 0
            if (!ALIGNED && walk.masked) {
                const int64_t kt = walk.whole * TN;
                for (int iota = ln * EW; iota < TN; iota += L * EW) {
                    const int64_t j = kt + iota;
                    if constexpr (VEC) {
                        u32x4 t = {{0u, 0u, 0u, 0u}};
                        if (j < N) t = ld_nc_v4(xr + j);  // N % 4 == 0: a vector is wholly in or out
#pragma unroll
                        for (int e = 0; e < 4; ++e) acc[e] += as_f(t.v[e]);
                    } else {
                        acc[0] += j < N ? as_f(ld_nc_b32(xr + j)) : 0.0f;
                    }
                }
            }
        }
        float s = acc[0];
#pragma unroll
        for (int e = 1; e < EW; ++e) s += acc[e];
#pragma unroll
        for (int o = (L < 32 ? L : 32) / 2; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if constexpr (W > 1) {
            if ((ln & 31) == 0) part[lr][ln >> 5] = s;
            __syncthreads();
            if (ln == 0) {
                s = part[lr][0];
#pragma unroll
                for (int w = 1; w < W; ++w) s += part[lr][w];
            }
            __syncthreads();
        }
        if (ln == 0 && live) {
            pdl_wait();  // the loads above may run ahead of the previous kernel, the store may not
            r[row] = s;
        }
    }
    pdl_wait();  // threads that stored nothing: the grid completes only after the one before it
}

template <int TM>
tm_status launch(bool vec, bool aligned, const float *X, int64_t ldx, int64_t M, int64_t N, float *r, int TN,
                 unsigned *status, cudaStream_t s, bool pdl)
{
    const void *k;
    if (vec) k = aligned ? (const void *)rowsum_kernel<TM, true, true> : (const void *)rowsum_kernel<TM, true, false>;
    else k = aligned ? (const void *)rowsum_kernel<TM, false, true> : (const void *)rowsum_kernel<TM, false, false>;
    void *args[] = {(void *)&X, (void *)&ldx, (void *)&M, (void *)&N, (void *)&r, (void *)&TN, (void *)&status};
    return launch_kernel(k, dim3(flat_grid((M + TM - 1) / TM)), dim3(kThreads), args, 0, s, pdl);
}

bool pow2_in(int v, int lo, int hi) { return v >= lo && v <= hi && (v & (v - 1)) == 0; }

}  // namespace
}  // namespace libtm

using namespace libtm;

extern "C" tm_status tm_rowsum(const float *X, int64_t ldx, int64_t M, int64_t N, float *r, int32_t TM,
                               int32_t TN, uint32_t flags, tm_stream_t stream)
{
    if (!valid2d(X, ldx, M, N)) return TM_ERR_INVALID_ARG;
    if (M > 0 && r == nullptr) return TM_ERR_INVALID_ARG;
    if (!flags_ok(flags, TM_ALIGNED | TM_PATH_SCALAR | TM_PATH_VEC | TM_PDL)) return TM_ERR_INVALID_ARG;
    if (!pow2_in(TM, 1, 32) || !pow2_in(TN, 16, 4096)) return TM_ERR_UNSUPPORTED_TILE;
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
    const bool pdl = (flags & TM_PDL) != 0;
    switch (TM) {
    case 1: return launch<1>(vec, aligned, X, ldx, M, N, r, TN, dev->status, s, pdl);
    case 2: return launch<2>(vec, aligned, X, ldx, M, N, r, TN, dev->status, s, pdl);
    case 4: return launch<4>(vec, aligned, X, ldx, M, N, r, TN, dev->status, s, pdl);
    case 8: return launch<8>(vec, aligned, X, ldx, M, N, r, TN, dev->status, s, pdl);
    case 16: return launch<16>(vec, aligned, X, ldx, M, N, r, TN, dev->status, s, pdl);
    default: return launch<32>(vec, aligned, X, ldx, M, N, r, TN, dev->status, s, pdl);
    }
}
