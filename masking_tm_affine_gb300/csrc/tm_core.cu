// tm_core.cu -- per-device state, status reporting and the diagnostic probes.
//
// The pages' broken-promise behaviour is a trap that makes the host's next
// synchronize fail ("@aligned", "When the promise is broken").  Here the
// kernel's entry check instead sets a bit in a per-device status word and
// every block returns before its first access; tm_check is that "next
// synchronize": it waits on the stream and reports the bit.
#include <atomic>
#include <mutex>

#include "tm_host.h"

namespace libtm {

// One status word per device (the module is loaded once per device context).
__device__ unsigned g_status_word;

namespace {

struct DevSlot {
    std::atomic<bool> ready{false};
    DevInfo info{};
};

DevSlot g_slots[kMaxDevices];
std::mutex g_init_mu;

}  // namespace

tm_status device_info(const DevInfo **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return TM_ERR_CUDA;
    }
    DevSlot &s = g_slots[dev];
    if (!s.ready.load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lock(g_init_mu);
        if (!s.ready.load(std::memory_order_relaxed)) {
            int sms = 0;
            void *addr = nullptr;
            if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
                cudaGetSymbolAddress(&addr, g_status_word) != cudaSuccess || sms <= 0) {
                cudaGetLastError();
                return TM_ERR_CUDA;
            }
            s.info.sms = sms;
            s.info.status = static_cast<unsigned *>(addr);
            s.ready.store(true, std::memory_order_release);
        }
    }
    *out = &s.info;
    return TM_OK;
}

namespace {

__global__ void tile_walk_probe_kernel(int64_t K, int64_t T, int64_t *out4)
{
    TileWalk w = tile_walk(K, T);
    out4[0] = w.whole;
    out4[1] = w.masked;
    out4[2] = w.rem;
    out4[3] = w.iters;
}

// The plain streaming read tm_read_probe times: a flat grid, each thread U
// independent 16-byte loads issued together, one sum per block.
template <int U>
__global__ void __launch_bounds__(kThreads) read_probe_kernel(const float *__restrict__ x, int64_t n4,
                                                              float *__restrict__ out)
{
    __shared__ float wsum[kThreads / 32];
    const int64_t base = (int64_t)blockIdx.x * kThreads * U + threadIdx.x;
    u32x4 v[U];
#pragma unroll
    for (int q = 0; q < U; ++q) {
        const int64_t i = base + (int64_t)q * kThreads;
        v[q] = i < n4 ? ld_nc_v4(x + 4 * i) : u32x4{{0u, 0u, 0u, 0u}};
    }
    float s = 0.0f;
#pragma unroll
    for (int q = 0; q < U; ++q) s += (as_f(v[q].v[0]) + as_f(v[q].v[1])) + (as_f(v[q].v[2]) + as_f(v[q].v[3]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if ((threadIdx.x & 31) == 0) wsum[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = wsum[0];
#pragma unroll
        for (int w = 1; w < kThreads / 32; ++w) t += wsum[w];
        out[blockIdx.x] = t;
    }
}

// The same read with each block's share fixed at launch: block b walks its
// own contiguous range [b0, b1) of 16-byte vectors, 256 threads x 8 loads per
// step, and writes one sum.  No block can take over another's work, as in
// the column sums' one-pass forms, whose CTAs each own a fixed part of a
// strip.
__global__ void __launch_bounds__(kThreads) read_probe_fixed_kernel(const float *__restrict__ x, int64_t n4,
                                                                    int64_t share4, float *__restrict__ out)
{
    constexpr int U = 8;
    __shared__ float wsum[kThreads / 32];
    const int64_t b0 = (int64_t)blockIdx.x * share4;
    const int64_t b1 = b0 + share4 < n4 ? b0 + share4 : n4;
    float s = 0.0f;
    for (int64_t c = b0; c < b1; c += (int64_t)kThreads * U) {
        u32x4 v[U];
#pragma unroll
        for (int q = 0; q < U; ++q) {
            const int64_t i = c + threadIdx.x + (int64_t)q * kThreads;
            v[q] = i < b1 ? ld_nc_v4(x + 4 * i) : u32x4{{0u, 0u, 0u, 0u}};
        }
#pragma unroll
        for (int q = 0; q < U; ++q) s += (as_f(v[q].v[0]) + as_f(v[q].v[1])) + (as_f(v[q].v[2]) + as_f(v[q].v[3]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if ((threadIdx.x & 31) == 0) wsum[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = wsum[0];
#pragma unroll
        for (int w = 1; w < kThreads / 32; ++w) t += wsum[w];
        out[blockIdx.x] = t;
    }
}

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

}  // namespace libtm

using namespace libtm;

extern "C" const char *tm_status_string(tm_status st)
{
    switch (st) {
    case TM_OK: return "TM_OK";
    case TM_ERR_INVALID_ARG: return "TM_ERR_INVALID_ARG: invalid argument";
    case TM_ERR_UNSUPPORTED_TILE: return "TM_ERR_UNSUPPORTED_TILE: tile not positive or not instantiated";
    case TM_ERR_MISALIGNED: return "TM_ERR_MISALIGNED: pointer or leading dimension breaks vector alignment";
    case TM_ERR_BROKEN_PROMISE: return "TM_ERR_BROKEN_PROMISE: aligned promise broken (an extent is not a multiple of its tile)";
    case TM_ERR_CUDA: return "TM_ERR_CUDA: CUDA runtime error";
    case TM_ERR_WORKSPACE: return "TM_ERR_WORKSPACE: workspace missing, too small or misaligned";
    case TM_ERR_TIMEOUT: return "TM_ERR_TIMEOUT: a bounded device wait gave up";
    }
    return "TM_ERR_UNKNOWN";
}

extern "C" int tm_version(void) { return 10000; }

extern "C" tm_status tm_check(tm_stream_t stream)
{
    const DevInfo *dev;
    tm_status st = device_info(&dev);
    if (st != TM_OK) return st;
    cudaStream_t s = as_stream(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return TM_ERR_CUDA;
    }
    unsigned word = 0;
    const unsigned zero = 0;
    if (cudaMemcpyAsync(&word, dev->status, sizeof word, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemcpyAsync(dev->status, &zero, sizeof zero, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return TM_ERR_CUDA;
    }
    if (word & kStatusBrokenPromise) return TM_ERR_BROKEN_PROMISE;
    if (word & kStatusMisaligned) return TM_ERR_MISALIGNED;
    if (word & kStatusTimeout) return TM_ERR_TIMEOUT;
    return TM_OK;
}

extern "C" tm_status tm_tile_walk_probe(int64_t K, int32_t T, int64_t *out4, tm_stream_t stream)
{
    if (K < 0 || T <= 0 || out4 == nullptr) return TM_ERR_INVALID_ARG;
    const DevInfo *dev;
    tm_status st = device_info(&dev);
    if (st != TM_OK) return st;
    tile_walk_probe_kernel<<<1, 1, 0, as_stream(stream)>>>(K, T, out4);
    return launch_status();
}

extern "C" int64_t tm_read_probe_blocks(int64_t n, int32_t per_thread)
{
    if (n < 0 || n % 4 != 0 || !(per_thread == 1 || per_thread == 2 || per_thread == 4 || per_thread == 8 ||
                                  per_thread == 16))
        return -1;
    const int64_t per_block = (int64_t)kThreads * per_thread * 4;
    return (n + per_block - 1) / per_block;
}

extern "C" int64_t tm_read_probe_fixed_share(int64_t n, int32_t blocks)
{
    if (n < 0 || n % 4 != 0 || blocks < 1 || blocks > 65535) return -1;
    const int64_t step = (int64_t)kThreads * 8 * 4;  // floats per block step
    const int64_t steps = (n + step * blocks - 1) / (step * blocks);
    return steps * step;
}

extern "C" tm_status tm_read_probe_fixed(const float *x, int64_t n, float *out, int32_t blocks, tm_stream_t stream)
{
    const int64_t share = tm_read_probe_fixed_share(n, blocks);
    if (share < 0) return TM_ERR_INVALID_ARG;
    if (n == 0) return TM_OK;
    if (x == nullptr || out == nullptr) return TM_ERR_INVALID_ARG;
    if (!aligned_to(x, 16) || !aligned_to(out, 4)) return TM_ERR_MISALIGNED;
    const uintptr_t xlo = reinterpret_cast<uintptr_t>(x), xhi = xlo + (uintptr_t)n * 4;
    const uintptr_t olo = reinterpret_cast<uintptr_t>(out), ohi = olo + (uintptr_t)blocks * 4;
    if (!(xhi <= olo || ohi <= xlo)) return TM_ERR_INVALID_ARG;
    const DevInfo *dev;
    tm_status st = device_info(&dev);
    if (st != TM_OK) return st;
    read_probe_fixed_kernel<<<(unsigned)blocks, kThreads, 0, as_stream(stream)>>>(x, n / 4, share / 4, out);
    return launch_status();
}

extern "C" tm_status tm_read_probe(const float *x, int64_t n, float *out, int32_t per_thread, tm_stream_t stream)
{
    const int64_t blocks = tm_read_probe_blocks(n, per_thread);
    if (blocks < 0 || blocks > INT32_MAX) return TM_ERR_INVALID_ARG;
    if (n == 0) return TM_OK;
    if (x == nullptr || out == nullptr) return TM_ERR_INVALID_ARG;
    if (!aligned_to(x, 16) || !aligned_to(out, 4)) return TM_ERR_MISALIGNED;
    const uintptr_t xlo = reinterpret_cast<uintptr_t>(x), xhi = xlo + (uintptr_t)n * 4;
    const uintptr_t olo = reinterpret_cast<uintptr_t>(out), ohi = olo + (uintptr_t)blocks * 4;
    if (!(xhi <= olo || ohi <= xlo)) return TM_ERR_INVALID_ARG;
    const DevInfo *dev;
    tm_status st = device_info(&dev);
    if (st != TM_OK) return st;
    const int64_t n4 = n / 4;
    cudaStream_t s = as_stream(stream);
    switch (per_thread) {
    case 1: read_probe_kernel<1><<<(unsigned)blocks, kThreads, 0, s>>>(x, n4, out); break;
    case 2: read_probe_kernel<2><<<(unsigned)blocks, kThreads, 0, s>>>(x, n4, out); break;
    case 4: read_probe_kernel<4><<<(unsigned)blocks, kThreads, 0, s>>>(x, n4, out); break;
    case 8: read_probe_kernel<8><<<(unsigned)blocks, kThreads, 0, s>>>(x, n4, out); break;
    default: read_probe_kernel<16><<<(unsigned)blocks, kThreads, 0, s>>>(x, n4, out); break;
    }
    return launch_status();
}
