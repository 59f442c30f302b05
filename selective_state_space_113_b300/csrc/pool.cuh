// pool.cuh -- the stream-ordered memory pool the library's workspaces come
// from.
//
// The calls that need a workspace (unit summaries, flags, carried states,
// the backward's unit states) allocate it on the caller's stream and free it
// there after their last launch.  From the device's default pool, whose
// release threshold is 0, such an allocation after any synchronisation maps
// its pages again: about 0.09 ms for 4 MB and 0.37 ms for 168 MB on a B300,
// against 0.01 ms from a pool that keeps its memory.  So the library makes one
// pool of its own per device and context, which keeps up to kKeepBytes
// reserved across synchronisations (more is returned at the next one).  The
// memory stays reserved until the process ends or the context is destroyed.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

namespace ssm {
namespace pool {

constexpr uint64_t kKeepBytes = 1ull << 30;
constexpr int kMaxDevices = 128;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

// cuCtxGetCurrent from the driver, found once through the runtime (the
// library does not link libcuda).
inline CtxGetCurrentFn ctx_get_current() {
    static CtxGetCurrentFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(f);
    });
    return fn;
}

// The pool of the current device in its current context, made the first time
// a workspace is needed there (and again after that context was destroyed and
// another made current, so that a pool is never used from a context that is
// gone).
inline cudaError_t current(cudaMemPool_t* out) {
    static std::mutex mu;
    struct Slot {
        CUcontext ctx;
        cudaMemPool_t pool;
    };
    static Slot slots[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    CtxGetCurrentFn get_ctx = ctx_get_current();
    if (!get_ctx) return cudaErrorNotSupported;
    std::lock_guard<std::mutex> lock(mu);
    CUcontext ctx = nullptr;
    if (get_ctx(&ctx) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
    Slot& s = slots[dev];
    if (ctx && s.ctx == ctx && s.pool) {
        *out = s.pool;
        return cudaSuccess;
    }
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t p = nullptr;
    e = cudaMemPoolCreate(&p, &props);   // makes the primary context current if none was
    if (e != cudaSuccess) return e;
    uint64_t keep = kKeepBytes;
    e = cudaMemPoolSetAttribute(p, cudaMemPoolAttrReleaseThreshold, &keep);
    if (e != cudaSuccess || get_ctx(&ctx) != CUDA_SUCCESS || !ctx) {
        cudaMemPoolDestroy(p);
        return e != cudaSuccess ? e : cudaErrorDeviceUninitialized;
    }
    s.ctx = ctx;
    s.pool = p;
    *out = p;
    return cudaSuccess;
}

}  // namespace pool
}  // namespace ssm
