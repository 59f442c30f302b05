// scan_bwd_generic.cuh -- the generic backward kernel of the zero-order-hold
// scan: any N <= 256, any element alignment, any D.  One thread owns one
// (b, d) channel.  A forward walk stores the state every KC steps in a global
// checkpoint array; then, chunk by chunk from the last, the chunk's states
// are recomputed into a global history array and walked backward (the
// derivatives are those listed at the top of scan_bwd.cuh, in the plain
// per-state form).  dB and dC are summed over channels with atomic adds, dA,
// dDskip and ddt_bias over the batch.  Correct, not tuned: it exists so that
// no shape needs a CPU path.
#pragma once

#include "common.cuh"
#include "faults.cuh"

namespace ssm {
namespace bwdg {

constexpr int KC = 16;   // steps per checkpoint

__device__ __forceinline__ float psi_ref(float x) {
    if (fabsf(x) < 0.25f)
        return fmaf(x, fmaf(x, fmaf(x, fmaf(x, fmaf(x, 1.0f / 5040.0f, 1.0f / 720.0f),
                                               1.0f / 120.0f), 1.0f / 24.0f), 1.0f / 6.0f), 0.5f);
    return (expm1f(x) - x) / (x * x);
}

template <typename T, int NMAX>
__global__ void __launch_bounds__(128)
scan_bwd_generic_kernel(const T* __restrict__ u, const T* __restrict__ delta,
                        const float* __restrict__ dt_bias, const float* __restrict__ A,
                        const T* __restrict__ Bm, const T* __restrict__ Cm,
                        const float* __restrict__ Dskip, const T* __restrict__ z,
                        const T* __restrict__ dy, const float* __restrict__ dh_last,
                        T* __restrict__ du, T* __restrict__ ddelta, float* __restrict__ ddt_bias,
                        float* __restrict__ dA, float* __restrict__ dB, float* __restrict__ dC,
                        float* __restrict__ dDskip, T* __restrict__ dz,
                        float* __restrict__ ck, float* __restrict__ hist,
                        int64_t batch, int64_t L, int64_t D, int N) {
    const int64_t ch = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t nch = batch * D;
    if (ch >= nch) return;
    const int64_t b = ch / D, d = ch - b * D;
    const float bias = dt_bias ? dt_bias[d] : 0.0f;
    const float dsk = Dskip ? Dskip[d] : 0.0f;
    float a[NMAX], h[NMAX], lam[NMAX], dacc[NMAX];
#pragma unroll
    for (int n = 0; n < NMAX; ++n) {
        a[n] = n < N ? A[d * N + n] : 0.0f;
        h[n] = 0.0f;
        dacc[n] = 0.0f;
        lam[n] = (n < N && dh_last) ? dh_last[ch * N + n] : 0.0f;
    }
    const int64_t nck = (L + KC - 1) / KC;
    // forward: the state entering every chunk
    for (int64_t c = 0; c < nck; ++c) {
#pragma unroll
        for (int n = 0; n < NMAX; ++n)
            if (n < N) ck[(c * nch + ch) * N + n] = h[n];
        const int64_t te = (c + 1) * KC < L ? (c + 1) * KC : L;
        for (int64_t t = c * KC; t < te; ++t) {
            const int64_t i = (b * L + t) * D + d;
            const float ut = to_f32(u[i]);
            const float dt = softplus_ref(to_f32(delta[i]) + bias);
#pragma unroll
            for (int n = 0; n < NMAX; ++n) {
                if (n < N) {
                    const float x = dt * a[n];
                    const float q = a[n] != 0.0f ? expm1f(x) / a[n] : dt;
                    h[n] = fmaf(expf(x), h[n], q * to_f32(Bm[(b * L + t) * N + n]) * ut);
                }
            }
        }
    }
    float dsk_acc = 0.0f, dtb_acc = 0.0f;
    for (int64_t c = nck - 1; c >= 0; --c) {
        const int64_t t0 = c * KC, te = (c + 1) * KC < L ? (c + 1) * KC : L;
#pragma unroll
        for (int n = 0; n < NMAX; ++n)
            if (n < N) h[n] = ck[(c * nch + ch) * N + n];
        for (int64_t t = t0; t < te; ++t) {
            const int64_t i = (b * L + t) * D + d;
            const float ut = to_f32(u[i]);
            const float dt = softplus_ref(to_f32(delta[i]) + bias);
#pragma unroll
            for (int n = 0; n < NMAX; ++n) {
                if (n < N) {
                    const float x = dt * a[n];
                    const float q = a[n] != 0.0f ? expm1f(x) / a[n] : dt;
                    h[n] = fmaf(expf(x), h[n], q * to_f32(Bm[(b * L + t) * N + n]) * ut);
                    hist[((t - t0) * nch + ch) * N + n] = h[n];
                }
            }
        }
        for (int64_t t = te - 1; t >= t0; --t) {
            const int64_t i = (b * L + t) * D + d;
            const float ut = to_f32(u[i]);
            const float v = to_f32(delta[i]) + bias;
            const float dt = softplus_ref(v);
            const float dyt = to_f32(dy[i]);
            float g = 1.0f, sg = 0.0f, zt = 0.0f;
            if (z) {
                zt = to_f32(z[i]);
                sg = 1.0f / (1.0f + expf(-zt));
                g = zt * sg;
            }
            const float ds = dyt * g;
            float s = dsk * ut, dut = ds * dsk, ddt = 0.0f;
#pragma unroll
            for (int n = 0; n < NMAX; ++n) {
                if (n < N) {
                    const int64_t r = (b * L + t) * N + n;
                    const float x = dt * a[n];
                    const float ab = expf(x);
                    const float q = a[n] != 0.0f ? expm1f(x) / a[n] : dt;
                    const float ht = hist[((t - t0) * nch + ch) * N + n];
                    const float bt = to_f32(Bm[r]), ct = to_f32(Cm[r]);
                    s = fmaf(ct, ht, s);
                    lam[n] = fmaf(ds, ct, lam[n]);
                    if (dC) atomicAdd(dC + r, ds * ht);
                    if (dB) atomicAdd(dB + r, lam[n] * q * ut);
                    dut = fmaf(lam[n] * q, bt, dut);
                    ddt = fmaf(lam[n], fmaf(a[n], ht, bt * ut), ddt);
                    dacc[n] = fmaf(lam[n] * dt, fmaf(-dt * bt * ut, psi_ref(x), ht), dacc[n]);
                    lam[n] *= ab;
                }
            }
            const float dd = ddt / (1.0f + expf(-v));
            du[i] = from_f32<T>(dut);
            ddelta[i] = from_f32<T>(dd);
            if (z && dz) dz[i] = from_f32<T>(dyt * s * sg * (1.0f + zt * (1.0f - sg)));
            dsk_acc = fmaf(ds, ut, dsk_acc);
            dtb_acc += dd;
        }
    }
#pragma unroll
    for (int n = 0; n < NMAX; ++n)
        if (n < N) atomicAdd(dA + d * N + n, dacc[n]);
    if (dDskip) atomicAdd(dDskip + d, dsk_acc);
    if (ddt_bias) atomicAdd(ddt_bias + d, dtb_acc);
}

// Scratch floats the generic backward needs: checkpoints and one chunk of history.
inline size_t bwd_generic_scratch_floats(int64_t batch, int64_t L, int64_t D, int64_t N) {
    const int64_t nck = (L + KC - 1) / KC;
    return (size_t)(nck + KC) * (size_t)(batch * D) * (size_t)N;
}

template <typename T>
static cudaError_t launch_scan_bwd_generic(const T* u, const T* delta, const float* dt_bias,
                                           const float* A, const T* Bm, const T* Cm,
                                           const float* Dskip, const T* z, const T* dy,
                                           const float* dh_last, T* du, T* ddelta,
                                           float* ddt_bias, float* dA, float* dB, float* dC,
                                           float* dDskip, T* dz, float* scratch, int64_t batch,
                                           int64_t L, int64_t D, int N, cudaStream_t s) {
    const int64_t nch = batch * D;
    const int64_t nck = (L + KC - 1) / KC;
    float* ck = scratch;
    float* hist = scratch + (size_t)nck * nch * N;
    const unsigned blocks = (unsigned)((nch + 127) / 128);
#define SSM_BWDG(NM)                                                                          \
    scan_bwd_generic_kernel<T, NM><<<blocks, 128, 0, s>>>(u, delta, dt_bias, A, Bm, Cm, Dskip, z, \
                                                          dy, dh_last, du, ddelta, ddt_bias, dA,  \
                                                          dB, dC, dDskip, dz, ck, hist, batch, L, \
                                                          D, N)
    if (fault::launch_refused()) return cudaErrorLaunchFailure;
    if (N <= 16) SSM_BWDG(16);
    else if (N <= 32) SSM_BWDG(32);
    else if (N <= 64) SSM_BWDG(64);
    else SSM_BWDG(256);
#undef SSM_BWDG
    return cudaGetLastError();
}

}  // namespace bwdg
}  // namespace ssm
