// runtime.cuh -- host-side device facts and per-kernel launch set-up, cached.
#pragma once

#include <cuda_runtime.h>
#include <cstdint>
#include <atomic>
#include <mutex>
#include <utility>

namespace qmv {

constexpr int kMaxDevices = 64;

inline int current_device()
{
    int d = 0;
    cudaGetDevice(&d);
    return d;
}

inline int num_sms()
{
    static std::atomic<int> cache[kMaxDevices];
    const int d = current_device();
    int v = (d >= 0 && d < kMaxDevices) ? cache[d].load(std::memory_order_relaxed) : 0;
    if (v == 0) {
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, d);
        if (v <= 0) v = 1;
        if (d >= 0 && d < kMaxDevices) cache[d].store(v, std::memory_order_relaxed);
    }
    return v;
}

// Token tile width of the plain bf16 prefill GEMM (k_gemm_bf16): true for
// 128-token tiles, false for 256.  The width with the larger expected
// throughput: the useful fraction of the padded tokens, times the fraction of
// the SMs busy over the waves of tiles, times 0.8 for 128-token tiles (their
// measured throughput against 256-token tiles when both fill whole waves: 1241
// against 1545 TFLOP/s at 14336 x 4096 x 2048).
inline bool gemm_bf16_narrow(int64_t rows, int64_t m, int64_t sms)
{
    const int64_t n_rt = (rows + 127) / 128;
    auto score = [&](int64_t bn) {
        const int64_t nt = (m + bn - 1) / bn, tiles = n_rt * nt;
        const int64_t waves = (tiles + sms - 1) / sms;
        return (double)m / (double)(nt * bn) * (double)tiles / (double)(waves * sms) * (bn == 128 ? 0.8 : 1.0);
    };
    return score(128) > score(256);
}

// Device address of the library's status word (defined in api.cu).
unsigned* status_word();

// The limit of the bounded waits of the decode and expert matvec kernels
// launched on device d: the default, or a diagnostic override
// (qmv_set_wait_limit; 0 restores the default).
inline std::atomic<unsigned long long>* wait_limit_slots()
{
    static std::atomic<unsigned long long> slots[kMaxDevices];
    return slots;
}
inline void set_wait_limit_ns(int d, unsigned ns) { wait_limit_slots()[d].store(ns, std::memory_order_relaxed); }
inline unsigned long long wait_limit_ns(unsigned long long dflt)
{
    const int d = current_device();
    const unsigned long long v =
        (d >= 0 && d < kMaxDevices) ? wait_limit_slots()[d].load(std::memory_order_relaxed) : 0ull;
    return v ? v : dflt;
}

// Opt a kernel into `bytes` of dynamic shared memory (once per kernel and
// device) and return how many of its blocks fit on one SM with that much.
template <typename K>
inline int prepare_kernel(K* kernel, int threads, size_t bytes)
{
    struct Entry {
        const void* fn;
        int dev;
        int threads;
        size_t bytes;
        int occ;
    };
    static std::mutex mu;
    static Entry cache[64];
    static int n = 0;
    const int dev = current_device();
    const void* fn = reinterpret_cast<const void*>(kernel);
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n; ++i)
        if (cache[i].fn == fn && cache[i].dev == dev && cache[i].threads == threads && cache[i].bytes == bytes)
            return cache[i].occ;
    // The limit is per kernel, not per launch: raise it to the device's opt-in
    // maximum once, so launches of the same kernel with other sizes stay valid.
    int max_optin = 0;
    cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         max_optin > (int)bytes ? max_optin : (int)bytes);
    // Prefer shared memory over L1 so that two ~100 KB blocks fit on one SM.
    cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, threads, bytes) != cudaSuccess || occ < 1) occ = 1;
    Entry e{fn, dev, threads, bytes, occ};
    if (n < 64) cache[n++] = e;
    else cache[(reinterpret_cast<uintptr_t>(fn) >> 4) % 64] = e;
    return occ;
}

// Launch `kernel` with an optional programmatic-dependent-launch attribute.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_ex(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                             bool pdl, Args&&... args)
{
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// As launch_ex, with thread-block clusters of `cluster` CTAs along x (grid.x a
// multiple of it); cluster 1 is a plain launch.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_ex_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                     bool pdl, int cluster, Args&&... args)
{
    if (cluster <= 1) return launch_ex(kernel, grid, block, smem, st, pdl, std::forward<Args>(args)...);
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace qmv
