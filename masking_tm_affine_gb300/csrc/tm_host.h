// tm_host.h -- host-side internals shared by the libtm translation units.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "../../include/tm.h"
#include "tm_device.cuh"

namespace libtm {

constexpr int kMaxDevices = 64;
constexpr int kThreads = 256;  // block size of the streaming kernels

// Per-device facts, filled once per device on first use (tm_core.cu).
struct DevInfo {
    int sms;           // multiprocessor count
    unsigned *status;  // device address of this device's status word
};

// Current device's info; TM_ERR_CUDA if the runtime cannot answer.
tm_status device_info(const DevInfo **out);

// The driver's cuTensorMapEncodeTiled, looked up once through the runtime
// (no link against libcuda); nullptr if the driver does not provide it.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// Flat grid: one block per work unit, capped at the 2^31-1 grid limit (the
// kernels keep a grid-stride loop for anything beyond it).  On GB300 the block
// scheduler's dynamic balancing beats a persistent grid-stride loop for these
// streaming kernels: static round-robin assignment left about 9% of the time
// in the imbalanced tail (2-D map at 8192 x 8192: 89.8 us persistent, 81.6 us flat).
inline unsigned flat_grid(int64_t units)
{
    if (units < 1) return 1;
    if (units > INT32_MAX) return (unsigned)INT32_MAX;
    return (unsigned)units;
}

// Map the last launch's outcome to a status.
inline tm_status launch_status()
{
    return cudaGetLastError() == cudaSuccess ? TM_OK : TM_ERR_CUDA;
}

inline cudaStream_t as_stream(tm_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

// Launch `kernel`; with pdl, as a programmatic dependent of the previous
// kernel in the stream (see pdl_wait in tm_device.cuh): its blocks may start
// while that kernel drains, and each must pdl_wait() before it reads what that
// kernel produced or writes anything.  cluster > 1 adds a cluster dimension.
inline tm_status launch_kernel(const void *kernel, dim3 grid, dim3 block, void **args, size_t smem, cudaStream_t s,
                               bool pdl, unsigned cluster = 1)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (cluster > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = cluster;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = n ? attr : nullptr;
    cfg.numAttrs = n;
    if (cudaLaunchKernelExC(&cfg, kernel, args) != cudaSuccess) {
        cudaGetLastError();
        return TM_ERR_CUDA;
    }
    return TM_OK;
}

inline tm_status launch_dependent(const void *kernel, dim3 grid, dim3 block, void **args, size_t smem,
                                  cudaStream_t s)
{
    return launch_kernel(kernel, grid, block, args, smem, s, true);
}

inline bool aligned_to(const void *p, uintptr_t bytes)
{
    return (reinterpret_cast<uintptr_t>(p) & (bytes - 1)) == 0;
}

// Byte extent [lo, hi) touched by a row-major [M, N] tensor with leading dimension ld.
inline void span2d(const void *base, int64_t ld, int64_t M, int64_t N, uintptr_t *lo, uintptr_t *hi)
{
    *lo = reinterpret_cast<uintptr_t>(base);
    *hi = *lo + (uintptr_t)(((M - 1) * ld + N) * (int64_t)sizeof(float));
}

// Shared argument checks of a 2-D [M, N] operand: extents >= 0, ld >= N,
// no int64 overflow of the addressed span, non-NULL when there is work.
inline bool valid2d(const void *p, int64_t ld, int64_t M, int64_t N)
{
    if (M < 0 || N < 0 || ld < N || ld < 0) return false;
    if (M == 0 || N == 0) return true;
    if (p == nullptr) return false;
    if (ld > 0 && M > (INT64_MAX / 4) / ld) return false;
    return true;
}

// Two 2-D operands may alias only exactly (same base, same ld): in-place maps.
inline bool overlap_ok(const void *a, int64_t lda, const void *b, int64_t ldb, int64_t M, int64_t N)
{
    if (M == 0 || N == 0) return true;
    if (a == b) return lda == ldb;
    uintptr_t alo, ahi, blo, bhi;
    span2d(a, lda, M, N, &alo, &ahi);
    span2d(b, ldb, M, N, &blo, &bhi);
    return ahi <= blo || bhi <= alo;
}

// Multiply-high divider for 1 <= d < 2^31 (see FastDiv in tm_device.cuh).
inline FastDiv make_fastdiv(uint32_t d)
{
    FastDiv f;
    f.d = d;
    uint32_t l = 0;
    while ((1ull << l) < d) ++l;
    f.shift = l;
    f.mul = (uint32_t)((((1ull << l) - d) << 32) / d + 1);
    return f;
}

constexpr uint32_t kPathBits = TM_PATH_SCALAR | TM_PATH_VEC | TM_PATH_TMA;

// At most one path bit, no unknown bits.
inline bool flags_ok(uint32_t flags, uint32_t allowed)
{
    if (flags & ~allowed) return false;
    uint32_t p = flags & kPathBits;
    return (p & (p - 1)) == 0;
}

}  // namespace libtm
