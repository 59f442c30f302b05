// tma_host.cuh -- host-side encoding of TMA tensor maps (cuTensorMapEncodeTiled
// from the driver, found once through the runtime, so that the library does
// not link libcuda).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
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

// make_map through a cache keyed by every argument (direct-mapped, 4096
// entries, one lock): a decode loop that reuses its buffers encodes each
// map once instead of at every call.
inline bool cached_map(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base,
                       const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                       CUtensorMapSwizzle swizzle) {
    struct Key {
        const void* base;
        int dt, rank, swizzle;
        cuuint64_t dims[5], strides[4];
        cuuint32_t box[5];
        bool operator==(const Key& o) const {
            if (base != o.base || dt != o.dt || rank != o.rank || swizzle != o.swizzle) return false;
            for (int i = 0; i < 5; ++i)
                if (dims[i] != o.dims[i] || box[i] != o.box[i]) return false;
            for (int i = 0; i < 4; ++i)
                if (strides[i] != o.strides[i]) return false;
            return true;
        }
    };
    struct Entry {
        Key key;
        CUtensorMap map;
        bool valid;
    };
    constexpr int kSlots = 4096;
    static std::mutex mu;
    static Entry table[kSlots];
    if (rank < 1 || rank > 5) return false;
    Key k{};
    k.base = base;
    k.dt = (int)dt;
    k.rank = rank;
    k.swizzle = (int)swizzle;
    for (int i = 0; i < rank; ++i) {
        k.dims[i] = dims[i];
        k.box[i] = box[i];
        if (i + 1 < rank) k.strides[i] = strides[i];
    }
    uint64_t h = reinterpret_cast<uintptr_t>(base) * 0x9E3779B97F4A7C15ull;
    for (int i = 0; i < rank; ++i) h = (h ^ dims[i] ^ ((uint64_t)box[i] << 32)) * 0x100000001B3ull;
    h ^= (uint64_t)dt * 131 + (uint64_t)swizzle;
    Entry& e = table[(h >> 24) % kSlots];
    {
        std::lock_guard<std::mutex> lock(mu);
        if (e.valid && e.key == k) {
            *m = e.map;
            return true;
        }
    }
    if (!make_map(m, dt, rank, base, dims, strides, box, swizzle)) return false;
    std::lock_guard<std::mutex> lock(mu);
    e.key = k;
    e.map = *m;
    e.valid = true;
    return true;
}

}  // namespace tma
}  // namespace ssm
