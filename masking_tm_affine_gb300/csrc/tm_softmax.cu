// tm_softmax.cu -- softmax row statistics over ragged BC-column tiles:
// m[i] = max_j S[i, j] and l[i] = sum_j exp(S[i, j] - m[i]).
//
// Source: "Slicing, bounds and masking", "Reductions over a ragged tile": the
// zero fill of a masked load is right for a sum and wrong for a maximum or a
// softmax, and the fix is the where/iota mask that replaces the columns past
// the end of the remainder tile with a fill that can never matter -- here
// -inf, which is never the maximum and whose exponential is exactly 0.  The
// page's fragment stops at the new row maximum; the softmax it names also
// needs the normaliser l, which this kernel carries alongside.
//
// GB300 design: the row-max kernel's layout (256-thread blocks of BR rows x
// 256/BR lanes, flat grid, whole-tile prefix unmasked with 8 loads in flight,
// then the masked remainder tile).  Each lane keeps an online pair (m, l):
// a batch with maximum b moves m to m' = max(m, b) and l to
// l * exp(m - m') + sum exp(v - m'), one exponential per element plus one per
// batch, each taken as CUDA's exp2f of (v - m') * log2(e): the difference is
// formed first (exact when v and m' are within a factor of two), and the one
// extra rounding of the product costs at most |v - m'| * 2^-24 relative in
// the term -- a few 1e-7 for the terms that carry the sum -- against expf's
// roughly twice the instruction count.  Lanes merge pairs in a shuffle butterfly (partners compute the same
// commutative sums, so every lane ends with identical values), warps through
// shared memory in a fixed order: the result is the same run to run.  All
// arithmetic is fp32; the normaliser matches the fp64 oracle to 1e-5 relative.
#include "tm_host.h"

namespace libtm {
namespace {

constexpr float kLog2e = 1.4426950408889634f;  // log2(e), rounded to fp32

// exp(d) for d <= 0 (or -inf): 2^(d log2 e).  exp(-inf) = 0.
__device__ __forceinline__ float exp_nonpos(float d) { return exp2f(d * kLog2e); }

// l * exp(m - mn) with the empty state (m = -inf, l = 0) mapped to 0.
__device__ __forceinline__ float rescale(float l, float m, float mn)
{
    return m == -INFINITY ? 0.0f : l * exp_nonpos(m - mn);
}

// Merge (m2, l2) into (m, l).
__device__ __forceinline__ void merge(float &m, float &l, float m2, float l2)
{
    const float mn = fmaxf(m, m2);
    if (mn == -INFINITY) return;  // both empty
    l = rescale(l, m, mn) + rescale(l2, m2, mn);
    m = mn;
}

// Absorb K values into (m, l).
template <int K>
__device__ __forceinline__ void absorb(float &m, float &l, const float (&v)[K])
{
    float b = -INFINITY;
#pragma unroll
    for (int k = 0; k < K; ++k) b = fmaxf(b, v[k]);
    const float mn = fmaxf(m, b);
    if (mn == -INFINITY) return;  // nothing but -inf so far
    float acc = rescale(l, m, mn);
#pragma unroll
    for (int k = 0; k < K; ++k) acc += exp_nonpos(v[k] - mn);  // exp(-inf) = 0
    l = acc;
    m = mn;
}

// Four blocks per SM, each lane holding 8 vector loads (32 values) in flight
// per batch: at [8192, 8192] 44.5 against 48.1 us with 4 (16 values) and no
// bound; a batch still takes one exponential per value plus one.
template <int BR, bool VEC, bool ALIGNED>
__global__ void __launch_bounds__(kThreads, 4) softmax_rowstats_kernel(const float *__restrict__ S, int64_t lds,
                                                                    int64_t M, int64_t N, float *__restrict__ m_out,
                                                                    float *__restrict__ l_out, int BC, int fill_zero,
                                                                    unsigned *status)
{
    constexpr int L = kThreads / BR;   // lanes sharing a row
    constexpr int EW = VEC ? 4 : 1;
    constexpr int U = VEC ? 8 : 16;    // accesses in flight per lane (32 vector values or 16 scalars per batch)
    constexpr int W = L > 32 ? L / 32 : 1;
    constexpr int kPre = 1;  // remainder-tile vectors a lane loads up front
    __shared__ float part_m[BR][W], part_l[BR][W];

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
        float mx = -INFINITY, sum = 0.0f;
        if (live) {
            const float *sr = S + row * lds;
            // The remainder tile's loads go out first, with the whole tiles'
            // (when they fit kPre vectors per lane): one DRAM round trip fewer.
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
            // last batch the lanes past the prefix hold -inf, which is never the
            // maximum and adds exp(-inf) = 0
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
                float vals[U * EW];
#pragma unroll
                for (int q = 0; q < U; ++q)
#pragma unroll
                    for (int e = 0; e < EW; ++e) vals[q * EW + e] = as_f(w[q][e]);
                absorb(mx, sum, vals);
            }
            // the remainder tile: masked load (reads 0), then where(iota < N - kt, s, -inf)
            if (pre) {
#pragma unroll
                for (int r = 0; r < kPre; ++r) {
                    const int iota = (ln + r * L) * EW;
                    if (iota >= BC) continue;
                    float sv[EW];
#pragma unroll
                    for (int e = 0; e < EW; ++e) {
                        sv[e] = as_f(rw[r][e]);
                        if (!fill_zero) sv[e] = (iota + e < N - kt) ? sv[e] : -INFINITY;
                    }
                    absorb(mx, sum, sv);
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
                    if (!fill_zero) {
#pragma unroll
                        for (int e = 0; e < EW; ++e) s[e] = (iota + e < N - kt) ? s[e] : -INFINITY;
                    }
                    absorb(mx, sum, s);
                }
            }
        }
#pragma unroll
        for (int o = (L < 32 ? L : 32) / 2; o > 0; o >>= 1) {
            const float m2 = __shfl_xor_sync(0xffffffffu, mx, o);
            const float l2 = __shfl_xor_sync(0xffffffffu, sum, o);
            merge(mx, sum, m2, l2);
        }
        if constexpr (W > 1) {
            if ((ln & 31) == 0) {
                part_m[lr][ln >> 5] = mx;
                part_l[lr][ln >> 5] = sum;
            }
            __syncthreads();
            if (ln == 0) {
                mx = part_m[lr][0];
                sum = part_l[lr][0];
#pragma unroll
                for (int w = 1; w < W; ++w) merge(mx, sum, part_m[lr][w], part_l[lr][w]);
            }
            __syncthreads();
        }
        if (ln == 0 && live) {
            pdl_wait();  // the loads above may run ahead of the previous kernel, the stores may not
            m_out[row] = mx;
            l_out[row] = sum;
        }
    }
    pdl_wait();  // threads that stored nothing: the grid completes only after the one before it
}

template <int BR>
tm_status launch(bool vec, bool aligned, const float *S, int64_t lds, int64_t M, int64_t N, float *m, float *l,
                 int BC, int fill_zero, unsigned *status, cudaStream_t s, bool pdl)
{
    const void *k;
    if (vec)
        k = aligned ? (const void *)softmax_rowstats_kernel<BR, true, true>
                    : (const void *)softmax_rowstats_kernel<BR, true, false>;
    else
        k = aligned ? (const void *)softmax_rowstats_kernel<BR, false, true>
                    : (const void *)softmax_rowstats_kernel<BR, false, false>;
    void *args[] = {(void *)&S, (void *)&lds, (void *)&M, (void *)&N, (void *)&m,
                    (void *)&l, (void *)&BC, (void *)&fill_zero, (void *)&status};
    return launch_kernel(k, dim3(flat_grid((M + BR - 1) / BR)), dim3(kThreads), args, 0, s, pdl);
}

bool pow2_in(int v, int lo, int hi) { return v >= lo && v <= hi && (v & (v - 1)) == 0; }

bool disjoint(const void *a, size_t abytes, const void *b, size_t bbytes)
{
    const uintptr_t alo = reinterpret_cast<uintptr_t>(a), blo = reinterpret_cast<uintptr_t>(b);
    return alo + abytes <= blo || blo + bbytes <= alo;
}

}  // namespace
}  // namespace libtm

using namespace libtm;

extern "C" tm_status tm_softmax_rowstats(const float *S, int64_t lds, int64_t M, int64_t N, float *m, float *l,
                                         int32_t BR, int32_t BC, tm_fill fill, uint32_t flags, tm_stream_t stream)
{
    if (!valid2d(S, lds, M, N)) return TM_ERR_INVALID_ARG;
    if (M > 0 && (m == nullptr || l == nullptr)) return TM_ERR_INVALID_ARG;
    if (fill != TM_FILL_NEG_INF && fill != TM_FILL_ZERO) return TM_ERR_INVALID_ARG;
    if (!flags_ok(flags, TM_ALIGNED | TM_PATH_SCALAR | TM_PATH_VEC | TM_PDL)) return TM_ERR_INVALID_ARG;
    if (!pow2_in(BR, 1, 32) || !pow2_in(BC, 16, 4096)) return TM_ERR_UNSUPPORTED_TILE;
    if (M > 0 && (!aligned_to(m, 4) || !aligned_to(l, 4))) return TM_ERR_MISALIGNED;
    if (M > 0 && N > 0 && !aligned_to(S, 4)) return TM_ERR_MISALIGNED;
    if (M > 0) {
        const size_t ob = (size_t)M * sizeof(float);
        if (!disjoint(m, ob, l, ob)) return TM_ERR_INVALID_ARG;
        if (N > 0) {
            uintptr_t slo, shi;
            span2d(S, lds, M, N, &slo, &shi);
            const void *sp = reinterpret_cast<const void *>(slo);
            if (!disjoint(sp, shi - slo, m, ob) || !disjoint(sp, shi - slo, l, ob)) return TM_ERR_INVALID_ARG;
        }
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
    case 1: return launch<1>(vec, aligned, S, lds, M, N, m, l, BC, fz, dev->status, s, pdl);
    case 2: return launch<2>(vec, aligned, S, lds, M, N, m, l, BC, fz, dev->status, s, pdl);
    case 4: return launch<4>(vec, aligned, S, lds, M, N, m, l, BC, fz, dev->status, s, pdl);
    case 8: return launch<8>(vec, aligned, S, lds, M, N, m, l, BC, fz, dev->status, s, pdl);
    case 16: return launch<16>(vec, aligned, S, lds, M, N, m, l, BC, fz, dev->status, s, pdl);
    default: return launch<32>(vec, aligned, S, lds, M, N, m, l, BC, fz, dev->status, s, pdl);
    }
}
