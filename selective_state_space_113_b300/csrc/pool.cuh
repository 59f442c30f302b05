// pool.cuh -- the stream-ordered memory pool the library's workspaces come
// from.
//
// The calls that need a workspace (unit summaries, flags, carried states,
// the backward's unit states) allocate it on the caller's stream and free it
// there after their last launch.  From the device's default pool, whose
// release threshold is 0, such an allocation after any synchronisation maps
// its pages again: about 0.09 ms for 4 MB and 0.37 ms for 168 MB on a B300,
// against 0.01 ms from a pool that keeps its memory.  So the library makes one
// pool of its own per device, which keeps up to kKeepBytes reserved across
// synchronisations (more is returned at the next one), until the process
// ends.  An explicit pool is a device's, not a context's: it stays usable
// after cudaDeviceReset.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

namespace ssm {
namespace pool {

constexpr uint64_t kKeepBytes = 1ull << 30;
constexpr int kMaxDevices = 128;

// The pool of the current device, made the first time a workspace is needed
// there.
inline cudaError_t current(cudaMemPool_t* out) {
    static std::mutex mu;
    static cudaMemPool_t pools[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!pools[dev]) {
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t p = nullptr;
        e = cudaMemPoolCreate(&p, &props);
        if (e != cudaSuccess) return e;
        uint64_t keep = kKeepBytes;
        e = cudaMemPoolSetAttribute(p, cudaMemPoolAttrReleaseThreshold, &keep);
        if (e != cudaSuccess) {
            cudaMemPoolDestroy(p);
            return e;
        }
        pools[dev] = p;
    }
    *out = pools[dev];
    return cudaSuccess;
}

}  // namespace pool
}  // namespace ssm
