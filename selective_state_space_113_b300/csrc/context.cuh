// context.cuh -- which CUDA context a call runs in, for the caches that
// belong to one (a kernel's shared-memory limit, a device symbol's address).
//
// A context destroyed and made again -- cudaDeviceReset, then any runtime
// call -- can come back with the same CUcontext handle (the primary context
// does), so the handle cannot tell the two apart.  cuCtxGetId gives every
// context a new ID, which can.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

namespace ssm {
namespace context {

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

template <typename F>
inline F driver_fn(const char* name) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        return reinterpret_cast<F>(f);
    return nullptr;
}

// The ID of the calling thread's current context, or 0 when there is none
// (or the driver does not say).  Found through the runtime: the library does
// not link libcuda.
inline unsigned long long current_id() {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
        get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
    });
    if (!get_current || !get_id) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

}  // namespace context
}  // namespace ssm
