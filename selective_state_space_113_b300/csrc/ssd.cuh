// ssd.cuh -- the Mamba-2 form of the scan (structured state-space duality)
// for the inputs the tensor-core kernel (ssd_tc.cuh) does not take: any dtype,
// any head dimension P and any state size N <= 256, one thread per channel.
//
// What it computes (news.han.ihouse.idv.tw article 1304: Mamba-2 reduced A to
// a scalar per head and discretises with Euler's rule), per batch b, head h,
// channel p of the head, step t, state n:
//   dt_t = softplus(dt[b,t,h] + dt_bias[h]);  h_t[n] = exp(dt_t A[h]) h_{t-1}[n]
//          + dt_t B_t[n] x_t[p];   y_t[p] = sum_n C_t[n] h_t[n] + Dskip[h] x_t[p]
// from h = 0, sequentially in t, in float32.
#pragma once

#include "common.cuh"
#include "faults.cuh"
#include "ptx.cuh"

namespace ssm {
namespace ssd {

// Any dtype, P and N <= 256: one thread per channel (b, t-walk, h, p), the
// recurrence in float32.  Correct, not tuned.
template <typename T, int NMAX>
__global__ void __launch_bounds__(128)
ssd_generic_kernel(const T* __restrict__ x, const T* __restrict__ dtr,
                   const float* __restrict__ dt_bias, const float* __restrict__ A,
                   const T* __restrict__ Bm, const T* __restrict__ Cm,
                   const float* __restrict__ Dskip, T* __restrict__ y, float* __restrict__ h_last,
                   long long batch, long long L, long long H, long long P, int N) {
    const long long ch = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (ch >= batch * H * P) return;
    const long long b = ch / (H * P), hp = ch % (H * P), hh = hp / P;
    const float a = A[hh];
    const float bias = dt_bias ? dt_bias[hh] : 0.0f;
    const float dsk = Dskip ? Dskip[hh] : 0.0f;
    float h[NMAX];
#pragma unroll
    for (int n = 0; n < NMAX; ++n) h[n] = 0.0f;
    for (long long t = 0; t < L; ++t) {
        const float dt = softplus_ref(to_f32(dtr[(b * L + t) * H + hh]) + bias);
        const float ab = expf(dt * a);
        const float xt = to_f32(x[(b * L + t) * H * P + hp]);
        float acc = dsk * xt;
#pragma unroll
        for (int n = 0; n < NMAX; ++n) {
            if (n < N) {
                h[n] = fmaf(ab, h[n], dt * to_f32(Bm[(b * L + t) * N + n]) * xt);
                acc = fmaf(to_f32(Cm[(b * L + t) * N + n]), h[n], acc);
            }
        }
        y[(b * L + t) * H * P + hp] = from_f32<T>(acc);
    }
    if (h_last) {
#pragma unroll
        for (int n = 0; n < NMAX; ++n)
            if (n < N) h_last[ch * N + n] = h[n];
    }
}

template <typename T>
inline cudaError_t launch_ssd_generic(const T* x, const T* dt, const float* dt_bias,
                                      const float* A, const T* Bm, const T* Cm,
                                      const float* Dskip, T* y, float* h_last, long long batch,
                                      long long L, long long H, long long P, int N,
                                      cudaStream_t s) {
    const long long nch = batch * H * P;
    const unsigned blocks = (unsigned)((nch + 127) / 128);
#define SSM_SSDG(NM)                                                                            \
    ssd_generic_kernel<T, NM><<<blocks, 128, 0, s>>>(x, dt, dt_bias, A, Bm, Cm, Dskip, y, h_last, \
                                                     batch, L, H, P, N)
    if (fault::launch_refused()) return cudaErrorLaunchFailure;
    if (N <= 16) SSM_SSDG(16);
    else if (N <= 64) SSM_SSDG(64);
    else if (N <= 128) SSM_SSDG(128);
    else SSM_SSDG(256);
#undef SSM_SSDG
    return cudaGetLastError();
}

}  // namespace ssd
}  // namespace ssm
