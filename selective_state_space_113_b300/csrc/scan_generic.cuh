// scan_generic.cuh -- the generic selective-scan kernel: any N <= 256, any
// element alignment, any D.  One thread owns one (b, d) channel and walks the
// sequence; the state stays in registers (N <= 32) or thread-local memory.
//
// Arithmetic is the definition written out in float32 (ultralytics page,
// "SSMの仕組み": A_bar = exp(dt A), B_bar = (A_bar - 1)/A * B with expm1 for
// accuracy; ta-paperlens page, Mamba pseudocode: dt = softplus(delta + bias),
// h = A_bar h + B_bar u, y = C h; D skip from the output equation y = C h + D x;
// SiLU(z) gate from the Mamba block diagram).  `disc` selects the input term:
// 0 zero-order hold as above, 1 Euler dt B_t u_t (the ta-paperlens
// pseudocode), 2 trapezoid dt/2 (B_t u_t + A_bar B_{t-1} u_{t-1}) (the
// news.han.ihouse.idv.tw Mamba-3 article, weight 1/2).  With conv_w given,
// u is x after the causal depthwise width-4 convolution in front of the SSM
// (ta-paperlens, "現場ではこう使う": d_conv; agenticai-flow: d_conv=4),
// u_t = act(conv_b + sum_k conv_w[d, k] x_{t-3+k}), zero x before step 0.
#pragma once

#include "common.cuh"
#include "faults.cuh"

namespace ssm {

template <typename T, int NMAX>
__global__ void __launch_bounds__(128)
scan_generic_kernel(const T* __restrict__ u, const T* __restrict__ delta,
                    const float* __restrict__ dt_bias, const float* __restrict__ A,
                    const T* __restrict__ Bm, const T* __restrict__ Cm,
                    const float* __restrict__ Dskip, const T* __restrict__ z,
                    T* __restrict__ y, float* __restrict__ h_last,
                    int64_t batch, int64_t L, int64_t D, int N, int disc,
                    const float* __restrict__ conv_w, const float* __restrict__ conv_b,
                    int act) {
    const int64_t ch = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (ch >= batch * D) return;
    const int64_t b = ch / D, d = ch - b * D;

    float h[NMAX];
    float a[NMAX];
    float q[NMAX];   // B_{t-1} u_{t-1} (trapezoid)
#pragma unroll
    for (int n = 0; n < NMAX; ++n) {
        h[n] = 0.0f;
        q[n] = 0.0f;
        a[n] = (n < N) ? A[d * N + n] : 0.0f;
    }
    const float bias = dt_bias ? dt_bias[d] : 0.0f;
    const float dsk = Dskip ? Dskip[d] : 0.0f;
    float cw[4] = {0.f, 0.f, 0.f, 0.f};
    float xh[3] = {0.f, 0.f, 0.f};   // x_{t-3}, x_{t-2}, x_{t-1}
    const float cb = (conv_w && conv_b) ? conv_b[d] : 0.0f;
    if (conv_w)
        for (int k = 0; k < 4; ++k) cw[k] = conv_w[d * 4 + k];

    for (int64_t t = 0; t < L; ++t) {
        const int64_t i = (b * L + t) * D + d;
        float ut = to_f32(u[i]);
        if (conv_w) {
            const float x = ut;
            float v = cb;
            v = fmaf(cw[0], xh[0], v);
            v = fmaf(cw[1], xh[1], v);
            v = fmaf(cw[2], xh[2], v);
            v = fmaf(cw[3], x, v);
            ut = act ? silu_ref(v) : v;
            xh[0] = xh[1];
            xh[1] = xh[2];
            xh[2] = x;
        }
        const float dt = softplus_ref(to_f32(delta[i]) + bias);
        const T* Bt = Bm + (b * L + t) * N;
        const T* Ct = Cm + (b * L + t) * N;
        float acc = 0.0f;
#pragma unroll
        for (int n = 0; n < NMAX; ++n) {
            if (n < N) {
                const float x = dt * a[n];
                const float abar = expf(x);
                const float qt = to_f32(Bt[n]) * ut;
                if (disc == 0) {
                    const float bcoef = (a[n] != 0.0f) ? expm1f(x) / a[n] : dt;
                    h[n] = fmaf(abar, h[n], bcoef * qt);
                } else if (disc == 1) {
                    h[n] = fmaf(abar, h[n], dt * qt);
                } else {
                    h[n] = fmaf(abar, fmaf(0.5f * dt, q[n], h[n]), 0.5f * dt * qt);
                }
                q[n] = qt;
                acc = fmaf(to_f32(Ct[n]), h[n], acc);
            }
        }
        acc = fmaf(dsk, ut, acc);
        if (z) acc *= silu_ref(to_f32(z[i]));
        y[i] = from_f32<T>(acc);
    }
    if (h_last) {
#pragma unroll
        for (int n = 0; n < NMAX; ++n)
            if (n < N) h_last[ch * N + n] = h[n];
    }
}

template <typename T, int NMAX>
static cudaError_t launch_scan_generic_n(const T* u, const T* delta, const float* dt_bias,
                                         const float* A, const T* Bm, const T* Cm,
                                         const float* Dskip, const T* z, T* y, float* h_last,
                                         int64_t batch, int64_t L, int64_t D, int N,
                                         int disc, cudaStream_t stream, const float* conv_w,
                                         const float* conv_b, int act) {
    const int64_t channels = batch * D;
    const int threads = 128;
    const int64_t blocks = (channels + threads - 1) / threads;
    if (fault::launch_refused()) return cudaErrorLaunchFailure;
    scan_generic_kernel<T, NMAX><<<(unsigned)blocks, threads, 0, stream>>>(
        u, delta, dt_bias, A, Bm, Cm, Dskip, z, y, h_last, batch, L, D, N, disc, conv_w, conv_b,
        act);
    return cudaGetLastError();
}

template <typename T>
static cudaError_t launch_scan_generic(const T* u, const T* delta, const float* dt_bias,
                                       const float* A, const T* Bm, const T* Cm,
                                       const float* Dskip, const T* z, T* y, float* h_last,
                                       int64_t batch, int64_t L, int64_t D, int N,
                                       cudaStream_t stream, int disc = 0,
                                       const float* conv_w = nullptr,
                                       const float* conv_b = nullptr, int act = 0) {
    if (N <= 16)
        return launch_scan_generic_n<T, 16>(u, delta, dt_bias, A, Bm, Cm, Dskip, z, y, h_last,
                                            batch, L, D, N, disc, stream, conv_w, conv_b, act);
    if (N <= 32)
        return launch_scan_generic_n<T, 32>(u, delta, dt_bias, A, Bm, Cm, Dskip, z, y, h_last,
                                            batch, L, D, N, disc, stream, conv_w, conv_b, act);
    if (N <= 64)
        return launch_scan_generic_n<T, 64>(u, delta, dt_bias, A, Bm, Cm, Dskip, z, y, h_last,
                                            batch, L, D, N, disc, stream, conv_w, conv_b, act);
    return launch_scan_generic_n<T, 256>(u, delta, dt_bias, A, Bm, Cm, Dskip, z, y, h_last,
                                         batch, L, D, N, disc, stream, conv_w, conv_b, act);
}

}  // namespace ssm
