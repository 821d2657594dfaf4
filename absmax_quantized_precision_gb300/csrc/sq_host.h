// Host-side helpers shared by the launchers (internal to libsq).
#pragma once

#include <cuda_runtime.h>

#include <map>
#include <mutex>
#include <utility>

namespace sq {

// Per-device, per-kernel results computed once: kernel attributes and
// occupancy belong to the device the kernel runs on, so a process that
// drives several GPUs sets and queries them for each one.  `make` runs under
// a lock the first time (device, key) is seen; the pair (error, value) is
// cached.
template <typename Fn>
inline std::pair<cudaError_t, int> per_device_once(const void* key, Fn make) {
    static std::mutex mu;
    static std::map<std::pair<int, const void*>, std::pair<cudaError_t, int>> done;
    int dev = 0;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return {e, 0};
    std::lock_guard<std::mutex> lock(mu);
    const auto k = std::make_pair(dev, key);
    const auto it = done.find(k);
    if (it != done.end()) return it->second;
    const std::pair<cudaError_t, int> r = make();
    done.emplace(k, r);
    return r;
}

// The dynamic shared-memory limit of a kernel, raised once per device.
inline cudaError_t set_max_dynamic_smem(const void* kernel, int bytes) {
    return per_device_once(kernel, [&] {
               return std::make_pair(
                   cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes), 0);
           })
        .first;
}

// Launch with programmatic stream serialization (the kernel must start with
// pdl_begin()), and as clusters of cluster_x CTAs when cluster_x > 1.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, unsigned cluster_x, Args&&... args) {
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
    if (cluster_x > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = cluster_x;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

}  // namespace sq
