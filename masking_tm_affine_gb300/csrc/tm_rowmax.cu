// tm_rowmax.cu -- m[i] = max_{j < N} S[i, j] over ragged BC-column tiles.
//
// Source: "Slicing, bounds and masking", "Reductions over a ragged tile".  A
// masked load reads 0, which is right for a sum and wrong for a maximum: a row
// of negative scores padded with zeros has a maximum of 0.  The fix is a
// second mask written with where and iota: in the column tile starting at kt,
// the column index iota (0 .. BC-1) is kept where iota < N - kt and replaced
// otherwise by a fill that can never be a row's maximum.  That fill is -inf (the
// page prints -1.0e30; -inf is the same for every finite score above -1e30 and
// still correct below it).  TM_FILL_ZERO skips the where step: the foil.
//
// The row is walked as "Loops over a dynamic extent" splits it: the whole
// tiles form an unmasked prefix of whole*BC columns, then the one remainder
// tile takes the masked load and the where.  A block of 256 threads takes BR
// rows, L = 256/BR lanes per row, flat grid (one block per BR-row band); the
// row's lanes stride through the prefix with U independent loads in flight,
// and a shuffle butterfly of fmaxf (plus shared memory when L > 32) ends the
// row.  max is exact and order-free, so the result equals the oracle's bit
// for bit.  Four blocks per SM, so that a lane's U vector loads fit in
// registers and go out together (eight blocks at 32 registers serialised
// part of each batch: [8192, 8192] 46.3 against 38.1 us by kernel time).
#include "tm_host.h"

namespace libtm {
namespace {

template <int BR, bool VEC, bool ALIGNED>
__global__ void __launch_bounds__(kThreads, 4) rowmax_kernel(const float *__restrict__ S, int64_t lds, int64_t M,
                                                          int64_t N, float *__restrict__ m, int BC, int fill_zero,
                                                          unsigned *status)
{
    constexpr int L = kThreads / BR;   // lanes sharing a row
    constexpr int EW = VEC ? 4 : 1;
    constexpr int U = VEC ? 8 : 16;    // accesses in flight per lane
    constexpr int W = L > 32 ? L / 32 : 1;
    constexpr int kPre = 2;  // remainder-tile vectors a lane loads up front
    __shared__ float part[BR][W];

    pdl_trigger();
    if constexpr (ALIGNED) {
        const bool whole = (M % BR == 0) && (N % BC == 0);
        const bool grid_ok = !VEC || ((lds % 4 == 0) && (reinterpret_cast<uintptr_t>(S) & 15) == 0);
        if (!whole || !grid_ok) {
            if (blockIdx.x == 0 && threadIdx.x == 0)
                atomicOr(status, whole ? kStatusMisaligned : kStatusBrokenPromise);
            pdl_wait();
            return;
        }
    }
    const int lr = threadIdx.x / L, ln = threadIdx.x % L;
    const TileWalk walk = tile_walk(N, BC);
    const int64_t prefix = walk.whole * BC / EW;  // accesses in the whole tiles
    const int64_t row_blocks = (M + BR - 1) / BR;

    for (int64_t rb = blockIdx.x; rb < row_blocks; rb += gridDim.x) {
        const int64_t row = rb * BR + lr;
        const bool live = ALIGNED || row < M;  // row mask
        float mx = -INFINITY;
        if (live) {
            const float *sr = S + row * lds;
            // The remainder tile's loads go out first, with the whole tiles'
            // (when they fit kPre vectors per lane): a short row is then one
            // DRAM round trip, not two.
            const int64_t kt = walk.whole * BC;
            const bool pre = !ALIGNED && walk.masked && BC <= kPre * L * EW;
            uint32_t rw[kPre][EW];
            if (pre) {
#pragma unroll
                for (int r = 0; r < kPre; ++r) {
                    const int iota = (ln + r * L) * EW;
                    const int64_t j = kt + iota;
#pragma unroll
                    for (int e = 0; e < EW; ++e) rw[r][e] = 0u;  // a masked load reads 0
                    if (iota < BC && j < N) {
                        if constexpr (VEC) {
                            const u32x4 t = ld_nc_v4(sr + j);  // N % 4 == 0: a vector is wholly in or out
#pragma unroll
                            for (int e = 0; e < 4; ++e) rw[r][e] = t.v[e];
                        } else {
                            rw[r][0] = ld_nc_b32(sr + j);
                        }
                    }
                }
            }
            // whole tiles: no mask.  U loads in flight per lane; in a partial
            // last batch the lanes past the prefix hold -inf, the max identity
            for (int64_t v = ln; v < prefix; v += (int64_t)L * U) {
                const bool full = v + (int64_t)L * (U - 1) < prefix;
                uint32_t w[U][EW];
#pragma unroll
                for (int q = 0; q < U; ++q) {
                    const float *p = sr + (v + (int64_t)L * q) * EW;
#pragma unroll
                    for (int e = 0; e < EW; ++e) w[q][e] = as_u(-INFINITY);
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
                    for (int e = 0; e < EW; ++e) mx = fmaxf(mx, as_f(w[q][e]));
            }
            // the remainder tile: masked load (reads 0), then where(iota < N - kt, s, -inf)
            if (pre) {
#pragma unroll
                for (int r = 0; r < kPre; ++r) {
                    const int iota = (ln + r * L) * EW;
                    if (iota >= BC) continue;
#pragma unroll
                    for (int e = 0; e < EW; ++e) {
                        float v = as_f(rw[r][e]);
                        if (!fill_zero) v = (iota + e < N - kt) ? v : -INFINITY;
                        mx = fmaxf(mx, v);
                    }
                }
            } else if (!ALIGNED && walk.masked) {
                for (int iota = ln * EW; iota < BC; iota += L * EW) {
                    const int64_t j = kt + iota;
                    float s[EW];
                    if constexpr (VEC) {
                        u32x4 t = {{0u, 0u, 0u, 0u}};
                        if (j < N) t = ld_nc_v4(sr + j);  // N % 4 == 0: a vector is wholly in or out
#pragma unroll
                        for (int e = 0; e < 4; ++e) s[e] = as_f(t.v[e]);
                    } else {
                        s[0] = j < N ? as_f(ld_nc_b32(sr + j)) : 0.0f;
                    }
#pragma unroll
                    for (int e = 0; e < EW; ++e) {
                        if (!fill_zero) s[e] = (iota + e < N - kt) ? s[e] : -INFINITY;
                        mx = fmaxf(mx, s[e]);
                    }
                }
            }
        }
#pragma unroll
        for (int o = (L < 32 ? L : 32) / 2; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if constexpr (W > 1) {
            if ((ln & 31) == 0) part[lr][ln >> 5] = mx;
            __syncthreads();
            if (ln == 0) {
#pragma unroll
                for (int w = 1; w < W; ++w) mx = fmaxf(mx, part[lr][w]);
            }
            __syncthreads();
        }
        if (ln == 0 && live) {
            pdl_wait();  // the loads above may run ahead of the previous kernel, the store may not
            m[row] = mx;
        }
    }
    pdl_wait();  // threads that stored nothing: the grid completes only after the one before it
}

template <int BR>
tm_status launch(bool vec, bool aligned, const float *S, int64_t lds, int64_t M, int64_t N, float *m, int BC,
                 int fill_zero, unsigned *status, cudaStream_t s, bool pdl)
{
    const void *k;
    if (vec) k = aligned ? (const void *)rowmax_kernel<BR, true, true> : (const void *)rowmax_kernel<BR, true, false>;
    else k = aligned ? (const void *)rowmax_kernel<BR, false, true> : (const void *)rowmax_kernel<BR, false, false>;
    void *args[] = {(void *)&S, (void *)&lds, (void *)&M, (void *)&N, (void *)&m,
                    (void *)&BC, (void *)&fill_zero, (void *)&status};
    return launch_kernel(k, dim3(flat_grid((M + BR - 1) / BR)), dim3(kThreads), args, 0, s, pdl);
}

bool pow2_in(int v, int lo, int hi) { return v >= lo && v <= hi && (v & (v - 1)) == 0; }

}  // namespace
}  // namespace libtm

using namespace libtm;

extern "C" tm_status tm_rowmax_masked(const float *S, int64_t lds, int64_t M, int64_t N, float *m, int32_t BR,
                                      int32_t BC, tm_fill fill, uint32_t flags, tm_stream_t stream)
{
    if (!valid2d(S, lds, M, N)) return TM_ERR_INVALID_ARG;
    if (M > 0 && m == nullptr) return TM_ERR_INVALID_ARG;
    if (fill != TM_FILL_NEG_INF && fill != TM_FILL_ZERO) return TM_ERR_INVALID_ARG;
    if (!flags_ok(flags, TM_ALIGNED | TM_PATH_SCALAR | TM_PATH_VEC | TM_PDL)) return TM_ERR_INVALID_ARG;
    if (!pow2_in(BR, 1, 32) || !pow2_in(BC, 16, 4096)) return TM_ERR_UNSUPPORTED_TILE;
    if (M > 0 && !aligned_to(m, 4)) return TM_ERR_MISALIGNED;
    if (M > 0 && N > 0 && !aligned_to(S, 4)) return TM_ERR_MISALIGNED;
    if (M > 0 && N > 0) {
        uintptr_t slo, shi, mlo = reinterpret_cast<uintptr_t>(m), mhi = mlo + (uintptr_t)M * 4;
        span2d(S, lds, M, N, &slo, &shi);
        if (!(shi <= mlo || mhi <= slo)) return TM_ERR_INVALID_ARG;
    }
    const bool vec16 = aligned_to(S, 16) && lds % 4 == 0;
    const bool aligned = (flags & TM_ALIGNED) != 0;
    bool vec;
    if (aligned) {
        if (!vec16 && !(flags & TM_PATH_SCALAR)) return TM_ERR_MISALIGNED;
        if (M % BR != 0 || N % BC != 0) return TM_ERR_BROKEN_PROMISE;
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
    const int fz = fill == TM_FILL_ZERO ? 1 : 0;
    const bool pdl = (flags & TM_PDL) != 0;
    switch (BR) {
    case 1: return launch<1>(vec, aligned, S, lds, M, N, m, BC, fz, dev->status, s, pdl);
    case 2: return launch<2>(vec, aligned, S, lds, M, N, m, BC, fz, dev->status, s, pdl);
    case 4: return launch<4>(vec, aligned, S, lds, M, N, m, BC, fz, dev->status, s, pdl);
    case 8: return launch<8>(vec, aligned, S, lds, M, N, m, BC, fz, dev->status, s, pdl);
    case 16: return launch<16>(vec, aligned, S, lds, M, N, m, BC, fz, dev->status, s, pdl);
    default: return launch<32>(vec, aligned, S, lds, M, N, m, BC, fz, dev->status, s, pdl);
    }
}
