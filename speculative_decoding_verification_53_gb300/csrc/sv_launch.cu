// sv_launch.cu -- per-device launch facts of the kernels (function attributes and
// occupancy answers), shared by every launcher and safe to use from several host
// threads and on several devices.
#include "sv_internal.h"

namespace sv {

cudaError_t KernelLaunchCache::device(const void* kern, Device** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kDevices) return cudaErrorInvalidDevice;
    Device& d = dev_[dev];
    if (!d.ready) {
        int optin = 0;
        cudaFuncAttributes fa;
        e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, kern);
        if (e != cudaSuccess) return e;
        const int m = optin - (int)fa.sharedSizeBytes;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, m);
        if (e != cudaSuccess) return e;
        d.max_dyn = m;
        d.used = 0;
        d.ready = true;
    }
    *out = &d;
    return cudaSuccess;
}

cudaError_t KernelLaunchCache::setup(const void* kern, int* max_dyn) {
    std::lock_guard<std::mutex> lock(mu_);
    Device* d = nullptr;
    const cudaError_t e = device(kern, &d);
    if (e != cudaSuccess) return e;
    *max_dyn = d->max_dyn;
    return cudaSuccess;
}

static cudaError_t occupancy_query(const void* kern, const cudaLaunchConfig_t& cfg_in, int G, int* out) {
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = cfg_in.blockDim;
    cfg.dynamicSmemBytes = cfg_in.dynamicSmemBytes;
    if (G == 0) {
        cfg.gridDim = dim3(16, 1, 1);
        return cudaOccupancyMaxPotentialClusterSize(out, kern, &cfg);
    }
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)G;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)G, 1, 1);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(out, kern, &cfg);
}

cudaError_t KernelLaunchCache::max_cluster(const void* kern, const cudaLaunchConfig_t& cfg, int* out) {
    return active_clusters(kern, cfg, 0, out);
}

cudaError_t KernelLaunchCache::active_clusters(const void* kern, const cudaLaunchConfig_t& cfg, int G, int* out) {
    std::lock_guard<std::mutex> lock(mu_);
    Device* d = nullptr;
    cudaError_t e = device(kern, &d);
    if (e != cudaSuccess) return e;
    if (cfg.dynamicSmemBytes > (size_t)d->max_dyn) {
        *out = 0;
        return cudaSuccess;
    }
    const unsigned threads = cfg.blockDim.x * cfg.blockDim.y * cfg.blockDim.z;
    const int n = d->used < kEntries ? d->used : kEntries;
    for (int i = 0; i < n; ++i) {
        const Entry& x = d->e[i];
        if (x.smem == cfg.dynamicSmemBytes && x.threads == threads && x.G == G) {
            *out = x.value;
            return cudaSuccess;
        }
    }
    int v = 0;
    e = occupancy_query(kern, cfg, G, &v);
    if (e != cudaSuccess) return e;
    d->e[d->used % kEntries] = Entry{cfg.dynamicSmemBytes, threads, G, v};
    ++d->used;
    *out = v;
    return cudaSuccess;
}

}  // namespace sv
