// faults.cuh -- host-side fault injection, for tests of the library's error
// paths, and NVTX ranges around the entry points.
//
// SSM_FAULT_INJECT=alloc   every stream-ordered workspace allocation fails as
//                          if the device were out of memory (SSM_ERR_NOMEM);
// SSM_FAULT_INJECT=launch  every kernel launch fails before anything of it is
//                          enqueued (SSM_ERR_CUDA).
// Any other value, or none, injects nothing.  The failures are made on the
// host only: no kernel is started, so nothing can fault or hang on the GPU,
// and the CUDA context carries no error afterwards.
#pragma once

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <cstdlib>
#include <cstring>

#include "pool.cuh"

namespace ssm {
namespace fault {

inline bool injected(const char* kind) {
    const char* v = std::getenv("SSM_FAULT_INJECT");
    return v && std::strcmp(v, kind) == 0;
}

// A stream-ordered workspace allocation from the library's pool (pool.cuh),
// freed by the caller with cudaFreeAsync; cudaErrorMemoryAllocation under
// SSM_FAULT_INJECT=alloc.
inline cudaError_t malloc_async(void** p, size_t bytes, cudaStream_t s) {
    *p = nullptr;
    if (injected("alloc")) return cudaErrorMemoryAllocation;
    cudaMemPool_t pl = nullptr;
    const cudaError_t e = pool::current(&pl);
    if (e != cudaSuccess) return e;
    return cudaMallocFromPoolAsync(p, bytes, pl, s);
}

// True when the launch about to be made must fail (SSM_FAULT_INJECT=launch);
// the caller then returns cudaErrorLaunchFailure without launching.
inline bool launch_refused() { return injected("launch"); }

// An NVTX range for the lifetime of the object (a no-op unless a profiler
// that listens to NVTX is attached).
struct Range {
    explicit Range(const char* name) { nvtxRangePushA(name); }
    ~Range() { nvtxRangePop(); }
    Range(const Range&) = delete;
    Range& operator=(const Range&) = delete;
};

}  // namespace fault
}  // namespace ssm
