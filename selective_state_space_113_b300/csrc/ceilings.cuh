// ceilings.cuh -- microbenchmarks of the three execution units that bound
// the scan kernels: the fp32 FMA pipes, the special-function unit (ex2) and
// instruction issue.  Used by ssm_unit_ceilings() so that a benchmark can put
// its measured throughput beside rates measured on the same GPU in the same
// process, instead of rates derived from a clock and a unit count.
#pragma once

#include <cuda_runtime.h>

#include "ptx.cuh"

namespace ssm {
namespace ceil {

constexpr int kChains = 8;          // independent dependency chains per thread
constexpr int kThreads = 512;       // 16 warps per CTA: four per SM sub-partition
constexpr float kMagic = 1234567.0f;

// Written only when a result equals kMagic (never, in practice); it keeps the
// compiler from removing the measured arithmetic.
__device__ float g_ceiling_sink;

// Packed f32x2 fused multiply-adds: kChains independent chains per thread.
__global__ void __launch_bounds__(kThreads) fma2_kernel(int iters, float m) {
    float2 a[kChains];
#pragma unroll
    for (int k = 0; k < kChains; ++k) a[k] = make_float2(threadIdx.x * 1e-3f + k, k * 0.5f);
    const float2 M = make_float2(m, m), C = make_float2(0.5f, 0.25f);
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int k = 0; k < kChains; ++k) a[k] = __ffma2_rn(a[k], M, C);
    }
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < kChains; ++k) s += a[k].x + a[k].y;
    if (s == kMagic) g_ceiling_sink = s;
}

// Scalar fused multiply-adds: one warp instruction each, so the rate of
// warp instructions issued when nothing else limits.
__global__ void __launch_bounds__(kThreads) fma1_kernel(int iters, float m) {
    float a[kChains];
#pragma unroll
    for (int k = 0; k < kChains; ++k) a[k] = threadIdx.x * 1e-3f + k;
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int k = 0; k < kChains; ++k) a[k] = fmaf(a[k], m, 0.5f);
    }
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < kChains; ++k) s += a[k];
    if (s == kMagic) g_ceiling_sink = s;
}

// 2^x on the special-function unit: x <- 2^(-x) keeps every value in
// [0.5, 1], so no chain overflows or reaches a denormal.
__global__ void __launch_bounds__(kThreads) ex2_kernel(int iters) {
    float a[kChains];
#pragma unroll
    for (int k = 0; k < kChains; ++k) a[k] = (threadIdx.x & 31) * (1.0f / 32.0f) + k * 0.01f;
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int k = 0; k < kChains; ++k) a[k] = ptx::ex2(-a[k]);
    }
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < kChains; ++k) s += a[k];
    if (s == kMagic) g_ceiling_sink = s;
}

// Best-of-`reps` rate (operations per second) of one kernel: `ops` operations
// per launch of `grid` CTAs.  Returns a CUDA error.
template <typename Launch>
inline cudaError_t best_rate(Launch launch, double ops, int reps, cudaStream_t s, double* rate) {
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    cudaError_t e = cudaEventCreate(&e0);
    if (e == cudaSuccess) e = cudaEventCreate(&e1);
    double best = 0.0;
    if (e == cudaSuccess) {
        launch();   // warm-up
        e = cudaGetLastError();
    }
    for (int r = 0; r < reps && e == cudaSuccess; ++r) {
        e = cudaEventRecord(e0, s);
        if (e == cudaSuccess) launch();
        if (e == cudaSuccess) e = cudaGetLastError();
        if (e == cudaSuccess) e = cudaEventRecord(e1, s);
        if (e == cudaSuccess) e = cudaEventSynchronize(e1);
        float ms = 0.f;
        if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
        if (e == cudaSuccess && ms > 0.f) {
            const double r_ = ops / (ms * 1e-3);
            if (r_ > best) best = r_;
        }
    }
    if (e0) cudaEventDestroy(e0);
    if (e1) cudaEventDestroy(e1);
    *rate = best;
    return e;
}

// out[0]: fp32 multiply-adds per second (packed), out[1]: ex2 per second,
// out[2]: warp instructions issued per second (scalar FMA stream); every
// rate is the sum over all SMs of the current device.
inline cudaError_t measure(double* out, int reps, cudaStream_t s) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int grid = 2 * sms;
    const double threads = (double)grid * kThreads;
    const int it_fma = 20000, it_ex2 = 4000;
    e = best_rate([&] { fma2_kernel<<<grid, kThreads, 0, s>>>(it_fma, 0.999f); },
                  threads * it_fma * kChains * 2.0, reps, s, &out[0]);
    if (e != cudaSuccess) return e;
    e = best_rate([&] { ex2_kernel<<<grid, kThreads, 0, s>>>(it_ex2); },
                  threads * it_ex2 * kChains, reps, s, &out[1]);
    if (e != cudaSuccess) return e;
    return best_rate([&] { fma1_kernel<<<grid, kThreads, 0, s>>>(it_fma, 0.999f); },
                     threads / 32.0 * it_fma * kChains, reps, s, &out[2]);
}

}  // namespace ceil
}  // namespace ssm
