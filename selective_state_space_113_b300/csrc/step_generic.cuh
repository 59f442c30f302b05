// step_generic.cuh -- the generic decode-step kernel: one thread per (b, d)
// channel, any N <= 256, any element alignment.  The same per-token update as
// one step of the scan (ta-paperlens page, S4 section: the recurrent form runs
// at constant cost per token), applied to the stored float32 state in place.
#pragma once

#include "common.cuh"
#include "faults.cuh"

namespace ssm {

template <typename T>
__global__ void __launch_bounds__(128)
step_generic_kernel(float* __restrict__ state, const T* __restrict__ u,
                    const T* __restrict__ delta, const float* __restrict__ dt_bias,
                    const float* __restrict__ A, const T* __restrict__ Bm,
                    const T* __restrict__ Cm, const float* __restrict__ Dskip,
                    const T* __restrict__ z, T* __restrict__ y,
                    int64_t batch, int64_t D, int N) {
    const int64_t ch = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (ch >= batch * D) return;
    const int64_t b = ch / D, d = ch - b * D;
    const float ut = to_f32(u[ch]);
    const float dt = softplus_ref(to_f32(delta[ch]) + (dt_bias ? dt_bias[d] : 0.0f));
    float* h = state + ch * N;
    const T* Bt = Bm + b * N;
    const T* Ct = Cm + b * N;
    float acc = 0.0f;
    for (int n = 0; n < N; ++n) {
        const float a = A[d * N + n];
        const float x = dt * a;
        const float abar = expf(x);
        const float bcoef = (a != 0.0f) ? expm1f(x) / a : dt;
        const float hn = fmaf(abar, h[n], bcoef * to_f32(Bt[n]) * ut);
        h[n] = hn;
        acc = fmaf(to_f32(Ct[n]), hn, acc);
    }
    acc = fmaf(Dskip ? Dskip[d] : 0.0f, ut, acc);
    if (z) acc *= silu_ref(to_f32(z[ch]));
    y[ch] = from_f32<T>(acc);
}

template <typename T>
static cudaError_t launch_step_generic(float* state, const T* u, const T* delta,
                                       const float* dt_bias, const float* A, const T* Bm,
                                       const T* Cm, const float* Dskip, const T* z, T* y,
                                       int64_t batch, int64_t D, int N, cudaStream_t stream) {
    const int64_t channels = batch * D;
    const int threads = 128;
    const int64_t blocks = (channels + threads - 1) / threads;
    if (fault::launch_refused()) return cudaErrorLaunchFailure;
    step_generic_kernel<T><<<(unsigned)blocks, threads, 0, stream>>>(
        state, u, delta, dt_bias, A, Bm, Cm, Dskip, z, y, batch, D, N);
    return cudaGetLastError();
}

}  // namespace ssm
