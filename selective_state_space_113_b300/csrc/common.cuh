// common.cuh -- element access and the plain float32 forms of the scan's
// scalar functions, shared by the libssmscan kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ssm {

using bf16 = __nv_bfloat16;

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(bf16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_f32<bf16>(float x) { return __float2bfloat16_rn(x); }

// softplus(v) = log(1 + exp(v)); above 20 it equals v to float32 precision.
__device__ __forceinline__ float softplus_ref(float v) {
    return v > 20.0f ? v : log1pf(expf(v));
}

// SiLU(z) = z * sigmoid(z) = z / (1 + exp(-z)); tends to -0 as z -> -inf.
__device__ __forceinline__ float silu_ref(float z) { return z / (1.0f + expf(-z)); }

// exp(x) - 1 given ex = 2^(x log2 e) (an approximate exp(x)): below |x| =
// 1/32 a degree-4 Taylor polynomial (truncation below 1e-9 relative), since
// ex - 1 there keeps only the few bits of x that survive the rounding of ex
// to a number near 1; elsewhere ex - 1, which loses no significant digits.
__device__ __forceinline__ float em1_near0(float x, float ex) {
    if (fabsf(x) < 0.03125f)
        return x * fmaf(x, fmaf(x, fmaf(x, 1.0f / 24.0f, 1.0f / 6.0f), 0.5f), 1.0f);
    return ex - 1.0f;
}

// Device-wide error word (one per device that loads the library).  Bounded
// waits that give up OR their code in; ssm_device_status() reads and clears it.
// The library is one translation unit (api.cu includes every kernel file), so
// this definition is seen exactly once.
__device__ unsigned int g_error_word = 0;
constexpr unsigned int kErrTimeout = 1u;

}  // namespace ssm
