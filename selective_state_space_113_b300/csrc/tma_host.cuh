// tma_host.cuh -- host-side encoding of TMA tensor maps (cuTensorMapEncodeTiled
// from the driver, found once through the runtime, so that the library does
// not link libcuda).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

namespace ssm {
namespace tma {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_tiled() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Row-major tensor of `rank` dimensions, dims[0] innermost; strides (bytes)
// of dims 1..rank-1; box extents; element type; swizzle.  Out-of-range
// elements of a box are read as zero.  Returns false if the driver refuses.
inline bool make_map(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base,
                     const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                     CUtensorMapSwizzle swizzle) {
    EncodeTiledFn fn = encode_tiled();
    if (!fn) return false;
    const cuuint32_t estr[5] = {1u, 1u, 1u, 1u, 1u};
    return fn(m, dt, (cuuint32_t)rank, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tma
}  // namespace ssm
