// tm_map2d.cu -- tiled 2-D maps: Y = alpha*X (tm_scale2d) and B = A (tm_copy2d).
//
// Sources: "@aligned" ("A minimal kernel": kernel `scale`, one TM x TN tile per
// work unit; "What it changes": no masks and 16-byte row access under the
// promise; "When the promise is broken": the promise is checked once at kernel
// entry); "Slicing, bounds and masking" ("Masking": loads past the end read 0,
// stores past the end are skipped; "Promising whole tiles with @aligned":
// kernel copy2d with 64 x 64 tiles).
//
// GB300 design.  The pages launch one CTA per tile.  Here one block takes a
// group of G consecutive tiles (row-major tile order) so that every thread has
// U independent loads in flight (G = 1 for tiles of >= 1024 vectors), and the
// grid is flat -- one block per group -- so the block scheduler balances the
// load (a persistent grid-stride loop measured ~9% slower on GB300).  Within a
// group, consecutive threads take consecutive vectors of a tile row, so a warp
// reads whole 128-byte lines.  Three paths:
//   Aligned   -- the promise holds: no predicate on any access, 16- or 32-byte
//                vectors.  Entry check first; on failure no block touches memory.
//   RaggedVec -- N, ld multiples of 4 and 16-byte bases: 16-byte vectors, one
//                predicate per vector (a vector is wholly in or wholly out).
//   Scalar    -- anything else: 4-byte accesses, one predicate per element.
#include "tm_host.h"

namespace libtm {
namespace {

enum class Op { Scale, Copy, Channel, Pad };
enum class Path { Aligned, RaggedVec, Scalar };

struct Map2dArgs {
    const float *X;
    float *Y;
    int64_t ldx, ldy, M, N;
    float alpha;
    uint32_t tiles_n;  // ceil(N / TN)
    uint32_t ntiles;   // ceil(M / TM) * tiles_n
    FastDiv div_tiles_n;
    unsigned *status;
    // Op::Channel only: per-channel parameters (either may be NULL)
    const float *scale, *bias;
    int layout;       // 0: channel = column j; 1: channel = row i mod C
    uint32_t C;
    FastDiv div_C;
    // Op::Pad only: the source extents inside the padded [M, N]
    int64_t Msrc, Nsrc;
};

template <Op OP>
__device__ __forceinline__ uint32_t apply(uint32_t x, float alpha)
{
    if (OP == Op::Copy || OP == Op::Pad) return x;  // bitwise: no arithmetic touches the word
    return as_u(__fmul_rn(alpha, as_f(x)));       // one rounding, like the oracle
}

// y = x*s + b rounded once (fused), or x*s / x + b when a vector is absent.
__device__ __forceinline__ uint32_t apply_channel(uint32_t x, float s, float b, bool has_s, bool has_b)
{
    if (has_s && has_b) return as_u(__fmaf_rn(as_f(x), s, b));
    if (has_s) return as_u(__fmul_rn(as_f(x), s));
    if (has_b) return as_u(__fadd_rn(as_f(x), b));
    return x;
}

// EW consecutive per-channel parameters starting at channel ch (16-byte
// aligned when EW >= 4: the host picks a scalar path otherwise).
template <int EW>
__device__ __forceinline__ void load_params(const float *v, uint32_t ch, float (&out)[EW])
{
    if constexpr (EW == 1) {
        out[0] = as_f(ldg_b32(v + ch));
    } else {
#pragma unroll
        for (int h = 0; h < EW; h += 4) {
            const u32x4 t = ldg_v4(v + ch + h);
#pragma unroll
            for (int e = 0; e < 4; ++e) out[h + e] = as_f(t.v[e]);
        }
    }
}

template <int EW>
struct Vec {
    uint32_t v[EW];
};

template <int EW>
__device__ __forceinline__ Vec<EW> load_vec(const float *p)
{
    Vec<EW> r;
    if constexpr (EW == 1) {
        r.v[0] = ld_nc_b32(p);
    } else if constexpr (EW == 4) {
        u32x4 t = ld_nc_v4(p);
#pragma unroll
        for (int e = 0; e < 4; ++e) r.v[e] = t.v[e];
    } else {
        u32x8 t = ld_nc_v8(p);
#pragma unroll
        for (int e = 0; e < 8; ++e) r.v[e] = t.v[e];
    }
    return r;
}

template <int EW>
__device__ __forceinline__ void store_vec(float *p, const Vec<EW> &x)
{
    if constexpr (EW == 1) {
        st_b32(p, x.v[0]);
    } else if constexpr (EW == 4) {
        u32x4 t;
#pragma unroll
        for (int e = 0; e < 4; ++e) t.v[e] = x.v[e];
        st_v4(p, t);
    } else {
        u32x8 t;
#pragma unroll
        for (int e = 0; e < 8; ++e) t.v[e] = x.v[e];
        st_v8(p, t);
    }
}

// IT: the index type of element offsets -- uint32_t when every offset the
// walk dereferences is below 2^31 (host-checked), int64_t otherwise.  The
// narrower arithmetic frees registers: the ragged 64 x 64 map drops from 38
// to fit 8 blocks per SM, so a ragged tensor of a few tens of MB runs in one
// wave instead of 1.14.
template <int TM, int TN, Op OP, Path P, int EW, typename IT = int64_t>
__global__ void __launch_bounds__(kThreads) map2d_kernel(const Map2dArgs p)
{
    constexpr int VPR = TN / EW;                       // accesses per tile row
    constexpr int V = TM * VPR;                        // accesses per tile
    constexpr int G = V >= 4 * kThreads ? 1 : (4 * kThreads) / V;  // tiles per group
    constexpr int A = G * V;                           // accesses per group
    constexpr int U = A / kThreads;                    // accesses per thread per group
    constexpr int UB = U < 4 ? U : 4;                  // accesses in flight per batch
    static_assert(A % kThreads == 0 && U % UB == 0, "tile shape does not fit the block");

    pdl_trigger();
    if constexpr (P == Path::Aligned) {
        // The promise, checked once at entry ("@aligned", "When the promise is
        // broken").  A pure function of the arguments, so every block takes the
        // same branch: on failure nothing is read or written anywhere.
        const bool whole = (p.M % TM == 0) && (p.N % TN == 0);
        const bool grid_ok = (p.ldx % EW == 0) && (p.ldy % EW == 0) &&
                             ((reinterpret_cast<uintptr_t>(p.X) | reinterpret_cast<uintptr_t>(p.Y)) &
                              (EW * sizeof(float) - 1)) == 0;
        if (!whole || !grid_ok) {
            if (blockIdx.x == 0 && threadIdx.x == 0)
                atomicOr(p.status, whole ? kStatusMisaligned : kStatusBrokenPromise);
            pdl_wait();
            return;
        }
    }

    const uint32_t ngroups = (p.ntiles + G - 1) / G;
    for (uint32_t g = blockIdx.x; g < ngroups; g += gridDim.x) {
#pragma unroll(U / UB <= 4 ? U / UB : 1)
        for (int b = 0; b < U; b += UB) {
            Vec<EW> val[UB];
            IT yoff[UB];
            uint32_t chan[UB];  // Op::Channel: the first element's channel (C < 2^31)
            bool live[UB];
#pragma unroll
            for (int u = 0; u < UB; ++u) {
                const uint32_t k = (uint32_t)(b + u) * kThreads + threadIdx.x;  // access within group
                const uint32_t tile = g * G + k / V;
                const uint32_t v = k % V;
                const uint32_t r = v / VPR;
                const uint32_t c = (v % VPR) * EW;
                const uint32_t pm = fdiv(tile, p.div_tiles_n);
                const uint32_t pn = tile - pm * p.tiles_n;
                const IT i = (IT)pm * TM + r;
                const IT j = (IT)pn * TN + c;
                bool in = (G == 1) || (tile < p.ntiles);
                if constexpr (P != Path::Aligned) in = in && ((int64_t)i < p.M) && ((int64_t)j < p.N);
                live[u] = in;
                yoff[u] = i * (IT)p.ldy + j;  // (wraps harmlessly for masked elements when IT is 32-bit)
                if constexpr (OP == Op::Channel)
                    chan[u] = p.layout == 0 ? (uint32_t)j : (uint32_t)i - fdiv((uint32_t)i, p.div_C) * p.C;
                // Op::Pad: the walk covers the padded extents; the source is read
                // only inside [Msrc, Nsrc] (vectors there are whole: Nsrc % EW == 0)
                const bool src = OP != Op::Pad || ((int64_t)i < p.Msrc && (int64_t)j < p.Nsrc);
                if (in && src) {
                    val[u] = load_vec<EW>(p.X + (i * (IT)p.ldx + j));
                } else {
#pragma unroll
                    for (int e = 0; e < EW; ++e) val[u].v[e] = 0u;  // a masked load reads 0
                }
            }
            pdl_wait();  // the loads above may run ahead of the previous kernel, the stores may not
#pragma unroll
            for (int u = 0; u < UB; ++u) {
                if (!live[u]) continue;                              // a masked store is skipped
                Vec<EW> o;
                if constexpr (OP == Op::Channel) {
                    // per-channel scale and bias: along the row (channels last)
                    // or one pair per row (channels first)
                    const bool hs = p.scale != nullptr, hb = p.bias != nullptr;
                    float sv[EW], bv[EW];
                    if (p.layout == 0) {
                        if (hs) load_params<EW>(p.scale, chan[u], sv);
                        if (hb) load_params<EW>(p.bias, chan[u], bv);
                    } else {
                        const float s1 = hs ? as_f(ldg_b32(p.scale + chan[u])) : 0.0f;
                        const float b1 = hb ? as_f(ldg_b32(p.bias + chan[u])) : 0.0f;
#pragma unroll
                        for (int e = 0; e < EW; ++e) {
                            sv[e] = s1;
                            bv[e] = b1;
                        }
                    }
#pragma unroll
                    for (int e = 0; e < EW; ++e) o.v[e] = apply_channel(val[u].v[e], sv[e], bv[e], hs, hb);
                } else {
#pragma unroll
                    for (int e = 0; e < EW; ++e) o.v[e] = apply<OP>(val[u].v[e], p.alpha);
                }
                store_vec<EW>(p.Y + yoff[u], o);
            }
        }
    }
    pdl_wait();
}

// Every element offset the ragged walk dereferences fits 31 bits: the last
// element of X (of the source region for Op::Pad) and of Y.
template <Op OP>
bool offsets_fit_i32(const Map2dArgs &a)
{
    const int64_t xm = OP == Op::Pad ? a.Msrc : a.M, xn = OP == Op::Pad ? a.Nsrc : a.N;
    const auto last = [](int64_t rows, int64_t ld, int64_t cols) { return rows > 0 ? (rows - 1) * ld + cols : 0; };
    return last(xm, a.ldx, xn) <= INT32_MAX && last(a.M, a.ldy, a.N) <= INT32_MAX;
}

template <int TM, int TN, Op OP>
tm_status launch_tile(Path path, int ew, const Map2dArgs &a, cudaStream_t s, bool pdl)
{
    const void *k = nullptr;
    if (path == Path::Aligned && ew == 8) k = (const void *)map2d_kernel<TM, TN, OP, Path::Aligned, 8>;
    else if (path == Path::Aligned) k = (const void *)map2d_kernel<TM, TN, OP, Path::Aligned, 4>;
    else if (path == Path::RaggedVec)
        // 32 x 32 tiles already fit 32 registers with 64-bit offsets (and need more with 32-bit ones)
        k = (!(TM == 32 && TN == 32) && offsets_fit_i32<OP>(a))
                ? (const void *)map2d_kernel<TM, TN, OP, Path::RaggedVec, 4, uint32_t>
                : (const void *)map2d_kernel<TM, TN, OP, Path::RaggedVec, 4>;
    else k = (const void *)map2d_kernel<TM, TN, OP, Path::Scalar, 1>;
    const int EW = path == Path::Scalar ? 1 : ew;
    const int64_t V = (int64_t)TM * TN / EW;
    const int64_t G = V >= 4 * kThreads ? 1 : (4 * kThreads) / V;
    const int64_t groups = ((int64_t)a.ntiles + G - 1) / G;
    void *args[] = {const_cast<Map2dArgs *>(&a)};
    return launch_kernel(k, dim3(flat_grid(groups)), dim3(kThreads), args, 0, s, pdl);
}

template <Op OP>
tm_status dispatch(int TM, int TN, Path path, int ew, const Map2dArgs &a, cudaStream_t s, bool pdl)
{
#define TM_TILE(tm_, tn_) \
    if (TM == tm_ && TN == tn_) return launch_tile<tm_, tn_, OP>(path, ew, a, s, pdl);
    TM_TILE(8, 8)
    TM_TILE(16, 16)
    TM_TILE(32, 32)
    TM_TILE(64, 64)
    TM_TILE(32, 128)
    TM_TILE(128, 128)
#undef TM_TILE
    return TM_ERR_UNSUPPORTED_TILE;
}

bool tile_supported(int TM, int TN)
{
    return (TM == 8 && TN == 8) || (TM == 16 && TN == 16) || (TM == 32 && TN == 32) ||
           (TM == 64 && TN == 64) || (TM == 32 && TN == 128) || (TM == 128 && TN == 128);
}

// Per-channel parameters of Op::Channel (see tm_channel_affine).
struct ChannelParams {
    const float *scale, *bias;
    int64_t C;
    int layout;
};

tm_status map2d(Op op, const float *X, int64_t ldx, float *Y, int64_t ldy, int64_t M, int64_t N,
                float alpha, int32_t TM, int32_t TN, uint32_t flags, tm_stream_t stream, bool check_promise,
                const ChannelParams *ch = nullptr)
{
    if (!valid2d(X, ldx, M, N) || !valid2d(Y, ldy, M, N)) return TM_ERR_INVALID_ARG;
    bool params16 = true;  // every present parameter vector is 16-byte aligned
    if (op == Op::Channel) {
        if (ch->C <= 0 || ch->C > INT32_MAX || (ch->layout != 0 && ch->layout != 1)) return TM_ERR_INVALID_ARG;
        if (ch->layout == 0 && N > ch->C) return TM_ERR_INVALID_ARG;
        if (ch->layout == 1 && M > INT32_MAX) return TM_ERR_INVALID_ARG;
        for (const float *v : {ch->scale, ch->bias}) {
            if (v == nullptr) continue;
            if (!aligned_to(v, 4)) return TM_ERR_MISALIGNED;
            params16 = params16 && aligned_to(v, 16);
            if (M > 0 && N > 0) {
                uintptr_t ylo, yhi, vlo = reinterpret_cast<uintptr_t>(v), vhi = vlo + (uintptr_t)ch->C * 4;
                span2d(Y, ldy, M, N, &ylo, &yhi);
                if (!(yhi <= vlo || vhi <= ylo)) return TM_ERR_INVALID_ARG;
            }
        }
        if (ch->layout == 1) params16 = true;  // one scalar parameter per row: no vector loads
    }
    if (!flags_ok(flags, TM_ALIGNED | kPathBits | TM_PDL)) return TM_ERR_INVALID_ARG;
    if (TM <= 0 || TN <= 0 || !tile_supported(TM, TN)) return TM_ERR_UNSUPPORTED_TILE;
    if (!overlap_ok(X, ldx, Y, ldy, M, N)) return TM_ERR_INVALID_ARG;
    if (M > 0 && N > 0 && (!aligned_to(X, 4) || !aligned_to(Y, 4))) return TM_ERR_MISALIGNED;
    if (flags & TM_PATH_TMA) return TM_ERR_INVALID_ARG;  // no TMA variant of the 2-D maps yet

    const bool vec16 = aligned_to(X, 16) && aligned_to(Y, 16) && ldx % 4 == 0 && ldy % 4 == 0;
    const bool vec32 = aligned_to(X, 32) && aligned_to(Y, 32) && ldx % 8 == 0 && ldy % 8 == 0 && TN % 8 == 0;
    if (!params16) flags |= TM_PATH_SCALAR;  // parameters read per element
    Path path;
    int ew = 4;
    if (flags & TM_ALIGNED) {
        if (check_promise) {
            if (!vec16) return TM_ERR_MISALIGNED;
            if (M % TM != 0 || N % TN != 0) return TM_ERR_BROKEN_PROMISE;
        }
        if (flags & TM_PATH_SCALAR) {
            if (flags & TM_PATH_VEC) return TM_ERR_MISALIGNED;
            path = Path::Scalar;
        } else {
            path = Path::Aligned;
            ew = (vec32 && !(flags & TM_PATH_VEC) && check_promise) ? 8 : 4;
        }
    } else if (flags & TM_PATH_SCALAR) {
        if (flags & TM_PATH_VEC) return TM_ERR_MISALIGNED;
        path = Path::Scalar;
    } else if (vec16 && N % 4 == 0) {
        path = Path::RaggedVec;
    } else if (flags & TM_PATH_VEC) {
        return TM_ERR_MISALIGNED;
    } else {
        path = Path::Scalar;
    }
    if (M == 0 || N == 0) return TM_OK;

    const DevInfo *dev;
    tm_status st = device_info(&dev);
    if (st != TM_OK) return st;

    const int64_t tiles_m = (M + TM - 1) / TM, tiles_n = (N + TN - 1) / TN;
    if (tiles_n > INT32_MAX || tiles_m > INT32_MAX / tiles_n) return TM_ERR_INVALID_ARG;
    Map2dArgs a;
    a.X = X;
    a.Y = Y;
    a.ldx = ldx;
    a.ldy = ldy;
    a.M = M;
    a.N = N;
    a.alpha = alpha;
    a.tiles_n = (uint32_t)tiles_n;
    a.ntiles = (uint32_t)(tiles_m * tiles_n);
    a.div_tiles_n = make_fastdiv((uint32_t)tiles_n);
    a.status = dev->status;
    a.scale = op == Op::Channel ? ch->scale : nullptr;
    a.bias = op == Op::Channel ? ch->bias : nullptr;
    a.layout = op == Op::Channel ? ch->layout : 0;
    a.C = op == Op::Channel ? (uint32_t)ch->C : 1u;
    a.div_C = make_fastdiv(a.C);
    cudaStream_t s = as_stream(stream);
    const bool pdl = (flags & TM_PDL) != 0;
    if (op == Op::Channel) return dispatch<Op::Channel>(TM, TN, path, ew, a, s, pdl);
    return op == Op::Scale ? dispatch<Op::Scale>(TM, TN, path, ew, a, s, pdl)
                           : dispatch<Op::Copy>(TM, TN, path, ew, a, s, pdl);
}

}  // namespace
}  // namespace libtm

using namespace libtm;

extern "C" tm_status tm_scale2d(const float *X, int64_t ldx, float *Y, int64_t ldy, int64_t M, int64_t N,
                                float alpha, int32_t TM, int32_t TN, uint32_t flags, tm_stream_t stream)
{
    return map2d(Op::Scale, X, ldx, Y, ldy, M, N, alpha, TM, TN, flags, stream, true);
}

extern "C" tm_status tm_copy2d(const float *A, int64_t lda, float *B, int64_t ldb, int64_t M, int64_t N,
                               int32_t TM, int32_t TN, uint32_t flags, tm_stream_t stream)
{
    return map2d(Op::Copy, A, lda, B, ldb, M, N, 1.0f, TM, TN, flags, stream, true);
}

extern "C" tm_status tm_scale2d_unchecked(const float *X, int64_t ldx, float *Y, int64_t ldy, int64_t M,
                                          int64_t N, float alpha, int32_t TM, int32_t TN, tm_stream_t stream)
{
    return map2d(Op::Scale, X, ldx, Y, ldy, M, N, alpha, TM, TN, TM_ALIGNED, stream, false);
}

extern "C" tm_status tm_channel_affine(const float *X, int64_t ldx, int64_t R, int64_t K, const float *scale,
                                       const float *bias, int64_t C, int32_t layout, float *Y, int64_t ldy,
                                       int32_t TM, int32_t TN, uint32_t flags, tm_stream_t stream)
{
    const ChannelParams ch{scale, bias, C, layout};
    return map2d(Op::Channel, X, ldx, Y, ldy, R, K, 0.0f, TM, TN, flags, stream, true, &ch);
}

extern "C" tm_status tm_pad2d(const float *A, int64_t lda, int64_t M, int64_t N, float *B, int64_t ldb, int64_t Mp,
                              int64_t Np, tm_stream_t stream)
{
    if (M < 0 || N < 0 || Mp < M || Np < N) return TM_ERR_INVALID_ARG;
    if (!valid2d(A, lda, M, N) || !valid2d(B, ldb, Mp, Np)) return TM_ERR_INVALID_ARG;
    if (Mp == 0 || Np == 0) return TM_OK;
    if (M > 0 && N > 0) {
        uintptr_t alo, ahi, blo, bhi;
        span2d(A, lda, M, N, &alo, &ahi);
        span2d(B, ldb, Mp, Np, &blo, &bhi);
        if (!(ahi <= blo || bhi <= alo)) return TM_ERR_INVALID_ARG;  // no in-place padding
        if (!aligned_to(A, 4)) return TM_ERR_MISALIGNED;
    }
    if (!aligned_to(B, 4)) return TM_ERR_MISALIGNED;
    const bool vec = aligned_to(B, 16) && ldb % 4 == 0 && Np % 4 == 0 &&
                     (M == 0 || N == 0 || (aligned_to(A, 16) && lda % 4 == 0 && N % 4 == 0));
    constexpr int TM = 32, TN = 128;
    const DevInfo *dev;
    tm_status st = device_info(&dev);
    if (st != TM_OK) return st;
    const int64_t tiles_m = (Mp + TM - 1) / TM, tiles_n = (Np + TN - 1) / TN;
    if (tiles_n > INT32_MAX || tiles_m > INT32_MAX / tiles_n) return TM_ERR_INVALID_ARG;
    Map2dArgs a{};
    a.X = A;
    a.Y = B;
    a.ldx = lda;
    a.ldy = ldb;
    a.M = Mp;
    a.N = Np;
    a.tiles_n = (uint32_t)tiles_n;
    a.ntiles = (uint32_t)(tiles_m * tiles_n);
    a.div_tiles_n = make_fastdiv((uint32_t)tiles_n);
    a.status = dev->status;
    a.C = 1u;
    a.div_C = make_fastdiv(1u);
    a.Msrc = M;
    a.Nsrc = N;
    return launch_tile<TM, TN, Op::Pad>(vec ? Path::RaggedVec : Path::Scalar, 4, a, as_stream(stream), false);
}

extern "C" int64_t tm_padded_extent(int64_t extent, const int32_t *tiles, int32_t ntiles)
{
    if (extent < 0 || ntiles <= 0 || tiles == nullptr) return -1;
    int64_t L = 1;
    for (int32_t k = 0; k < ntiles; ++k) {
        const int64_t t = tiles[k];
        if (t <= 0) return -1;
        int64_t a = L, b = t;  // L = lcm(L, t)
        while (b) {
            const int64_t r = a % b;
            a = b;
            b = r;
        }
        if (L / a > INT64_MAX / t) return -1;
        L = L / a * t;
    }
    const int64_t q = extent / L + (extent % L ? 1 : 0);
    if (q > INT64_MAX / L) return -1;
    return q * L;
}

extern "C" int64_t tm_row_stride(int64_t N, int32_t align_bytes)
{
    if (N < 0 || align_bytes <= 0 || align_bytes % 4 != 0 || (align_bytes & (align_bytes - 1)) != 0) return -1;
    const int64_t q = align_bytes / 4;  // elements per aligned unit
    if (N > INT64_MAX - q) return -1;
    return (N + q - 1) / q * q;
}
