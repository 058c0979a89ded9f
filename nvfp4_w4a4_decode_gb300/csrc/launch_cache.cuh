// launch_cache.cuh -- per-device cache of launch facts that cost a driver
// round trip to query (SM count, occupancy, the dynamic shared memory limit
// already granted to a kernel), so that a launch from the host costs only the
// launch itself after the first call with a given configuration.
#pragma once

#include <cuda_runtime.h>

#include <mutex>
#include <unordered_map>

namespace nvfp4 {

struct LaunchKey {
    const void* fn;
    int device, threads;
    size_t smem;
    int cluster;
    bool operator==(const LaunchKey& o) const
    {
        return fn == o.fn && device == o.device && threads == o.threads && smem == o.smem &&
               cluster == o.cluster;
    }
};

struct LaunchKeyHash {
    size_t operator()(const LaunchKey& k) const
    {
        size_t h = reinterpret_cast<size_t>(k.fn);
        h = h * 1000003u ^ (size_t)k.device;
        h = h * 1000003u ^ (size_t)k.threads;
        h = h * 1000003u ^ k.smem;
        h = h * 1000003u ^ (size_t)k.cluster;
        return h;
    }
};

inline int current_device()
{
    int dev = 0;
    cudaGetDevice(&dev);
    return dev;
}

inline int device_sm_count(int dev)
{
    static std::mutex mu;
    static std::unordered_map<int, int> cache;
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(dev);
    if (it != cache.end())
        return it->second;
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = sms;
    return sms;
}

// Raise a kernel's dynamic shared memory limit to `smem` on this device once
// (the limit only permits; each launch still states its own size).
template <typename Kern>
cudaError_t ensure_smem_limit(Kern kern, size_t smem, int dev)
{
    static std::mutex mu;
    static std::unordered_map<size_t, size_t> granted;  // (fn ^ device) -> bytes
    const size_t key = reinterpret_cast<size_t>(reinterpret_cast<const void*>(kern)) ^
                       ((size_t)dev << 48);
    std::lock_guard<std::mutex> lock(mu);
    auto it = granted.find(key);
    if (it != granted.end() && it->second >= smem)
        return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e == cudaSuccess)
        granted[key] = smem;
    return e;
}

// Resident CTAs per SM (cluster == 0) or resident clusters on the device
// (cluster > 0, via cudaOccupancyMaxActiveClusters), cached.
template <typename Kern>
cudaError_t cached_occupancy(Kern kern, int threads, size_t smem, int cluster, int dev, int* out)
{
    static std::mutex mu;
    static std::unordered_map<LaunchKey, int, LaunchKeyHash> cache;
    const LaunchKey key{reinterpret_cast<const void*>(kern), dev, threads, smem, cluster};
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = cache.find(key);
        if (it != cache.end()) {
            *out = it->second;
            return cudaSuccess;
        }
    }
    int v = 0;
    cudaError_t e;
    if (cluster <= 0) {
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, kern, threads, smem);
    } else {
        cudaLaunchConfig_t q = {};
        q.gridDim = dim3((unsigned)cluster, 1, 1);
        q.blockDim = dim3((unsigned)threads, 1, 1);
        q.dynamicSmemBytes = smem;
        cudaLaunchAttribute ca;
        ca.id = cudaLaunchAttributeClusterDimension;
        ca.val.clusterDim.x = (unsigned)cluster;
        ca.val.clusterDim.y = 1;
        ca.val.clusterDim.z = 1;
        q.attrs = &ca;
        q.numAttrs = 1;
        e = cudaOccupancyMaxActiveClusters(&v, kern, &q);
    }
    if (e != cudaSuccess)
        return e;
    std::lock_guard<std::mutex> lock(mu);
    cache[key] = v;
    *out = v;
    return cudaSuccess;
}

}  // namespace nvfp4
