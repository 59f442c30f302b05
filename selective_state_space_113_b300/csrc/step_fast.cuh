// step_fast.cuh -- the decode-step kernel for N == 16: one token's state
// update applied in place to the stored float32 state (ta-paperlens page, S4
// section: the recurrent form runs at constant cost per token; the update and
// readout are those of one scan step).
//
// The step is a stream over the [batch, D, 16] float32 state, read once and
// written once, so the layout of the accesses is what matters: four threads
// share a channel and each owns four consecutive states (one float4), so the
// 32 lanes of a warp read and write 512 contiguous bytes.  The four lanes of
// a channel add their partial readouts with two shuffles; the first of them
// applies the D skip and the SiLU gate and stores y.
#pragma once

#include <cstdlib>

#include "common.cuh"
#include "faults.cuh"
#include "ptx.cuh"

namespace ssm {
namespace stepk {

constexpr int NS = 16;
constexpr int THREADS = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// exp(x) - 1 for x <= 0 given 2^(x log2 e) = exp(x): a degree-4 Taylor
// polynomial where |x| < 1/32 (truncation error below 1e-9 relative), the
// difference ex2 - 1 elsewhere (where it loses no significant digits).
__device__ __forceinline__ float expm1_from(float x, float ex) {
    if (fabsf(x) < 0.03125f) {
        const float p = fmaf(x, fmaf(x, fmaf(x, 1.0f / 24.0f, 1.0f / 6.0f), 0.5f), 1.0f);
        return x * p;
    }
    return ex - 1.0f;
}

// Grid: x covers the 4*D threads of one batch entry, y is the batch entry, so
// no thread divides by D.
// J channels per group of four threads, Dh = ceil(D / J) apart in the same
// batch entry: every load of all J channels is issued before any arithmetic,
// so each thread keeps J float4 of state (and of A) in flight.
template <typename T, int J>
__global__ void __launch_bounds__(THREADS)
step16_kernel(float* __restrict__ state, const T* __restrict__ u, const T* __restrict__ delta,
              const float* __restrict__ dt_bias, const float* __restrict__ A,
              const T* __restrict__ Bm, const T* __restrict__ Cm,
              const float* __restrict__ Dskip, const T* __restrict__ z, T* __restrict__ y,
              int D, int Dh) {
    const int b = blockIdx.y;
    const int tid = blockIdx.x * THREADS + threadIdx.x;   // < 4*Dh (checked on the host)
    const int part = tid & 3;                              // states 4*part .. 4*part + 3
    // 32-bit offsets within one batch entry (4*D*16 < 2^31 is checked on the
    // host); the batch offset is applied to the base pointers once.
    const size_t row = (size_t)b * (size_t)D;
    float4* hbase = reinterpret_cast<float4*>(state + row * NS);
    bool valid[J];
    int d[J];
    float ut[J], v[J];
    float4 h4[J], a4[J];
    // Threads past the last channel stay (the shuffles below need the whole
    // warp) but work on channel 0 and store nothing.
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const int dj = (tid >> 2) + j * Dh;
        valid[j] = (tid >> 2) < Dh && dj < D;
        d[j] = valid[j] ? dj : 0;
        ut[j] = to_f32(u[row + d[j]]);
        v[j] = part == 0 ? to_f32(delta[row + d[j]]) + (dt_bias ? dt_bias[d[j]] : 0.0f) : 0.0f;
        h4[j] = hbase[d[j] * 4 + part];
        a4[j] = reinterpret_cast<const float4*>(A)[d[j] * 4 + part];
    }
    const T* Bt = Bm + (size_t)b * NS + 4 * part;
    const T* Ct = Cm + (size_t)b * NS + 4 * part;
    float bv[4], cv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        bv[i] = to_f32(Bt[i]);
        cv[i] = to_f32(Ct[i]);
    }
#pragma unroll
    for (int j = 0; j < J; ++j) {
        // softplus in the base-2 domain, dl = log2(1 + 2^(v log2 e)) = dt / ln 2,
        // computed by the first lane of the channel and shared with the others.
        float dl = 0.0f;
        if (part == 0) dl = v[j] > 20.0f ? v[j] * kLog2e : ptx::lg2(1.0f + ptx::ex2(v[j] * kLog2e));
        dl = __shfl_sync(0xffffffffu, dl, threadIdx.x & ~3);
        const float dt = dl * kLn2;
        const float a[4] = {a4[j].x, a4[j].y, a4[j].z, a4[j].w};
        const float h[4] = {h4[j].x, h4[j].y, h4[j].z, h4[j].w};
        float hn[4];
        float acc = 0.0f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float x = dt * a[i];
            const float ex = ptx::ex2(dl * a[i]);                  // exp(dt A) = A_bar
            const float em1 = expm1_from(x, ex);                   // A_bar - 1
            // B_bar / B = (A_bar - 1) / A, or dt at A == 0; the approximate
            // reciprocal (relative error ~1e-7) replaces an IEEE division.
            const float coef = (a[i] != 0.0f) ? em1 * ptx::rcp(a[i]) : dt;
            hn[i] = fmaf(ex, h[i], coef * bv[i] * ut[j]);
            acc = fmaf(cv[i], hn[i], acc);
        }
        if (valid[j]) hbase[d[j] * 4 + part] = make_float4(hn[0], hn[1], hn[2], hn[3]);
        acc += __shfl_xor_sync(0xffffffffu, acc, 1);
        acc += __shfl_xor_sync(0xffffffffu, acc, 2);
        if (valid[j] && part == 0) {
            acc = fmaf(Dskip ? Dskip[d[j]] : 0.0f, ut[j], acc);
            if (z) {
                const float zt = to_f32(z[row + d[j]]);
                acc *= zt * ptx::rcp(1.0f + ptx::ex2(-zt * kLog2e));
            }
            y[row + d[j]] = from_f32<T>(acc);
        }
    }
}

// Largest D the one-launch grid takes (64*D, the state entries of one batch
// entry, must fit an int; batch must fit the grid's y extent).
constexpr long long kMaxD = (1LL << 25);
constexpr long long kMaxBatch = 65535;

template <typename T>
static cudaError_t launch_step16(float* state, const T* u, const T* delta, const float* dt_bias,
                                 const float* A, const T* Bm, const T* Cm, const float* Dskip,
                                 const T* z, T* y, long long batch, long long D,
                                 cudaStream_t stream) {
    // Channels per thread group: 2 (measured fastest on the 256 x 5120
    // decode); SSM_STEP_J = 1 or 4 selects another (development and tests).
    const char* e = std::getenv("SSM_STEP_J");
    const int J = (e && e[0] == '1') ? 1 : (e && e[0] == '4') ? 4 : 2;
    const long long Dh = (D + J - 1) / J;
    const dim3 grid((unsigned)((4 * Dh + THREADS - 1) / THREADS), (unsigned)batch);
    if (fault::launch_refused()) return cudaErrorLaunchFailure;
    if (J == 4)
        step16_kernel<T, 4><<<grid, THREADS, 0, stream>>>(state, u, delta, dt_bias, A, Bm, Cm,
                                                          Dskip, z, y, (int)D, (int)Dh);
    else if (J == 2)
        step16_kernel<T, 2><<<grid, THREADS, 0, stream>>>(state, u, delta, dt_bias, A, Bm, Cm,
                                                          Dskip, z, y, (int)D, (int)Dh);
    else
        step16_kernel<T, 1><<<grid, THREADS, 0, stream>>>(state, u, delta, dt_bias, A, Bm, Cm,
                                                          Dskip, z, y, (int)D, (int)Dh);
    return cudaGetLastError();
}

}  // namespace stepk
}  // namespace ssm
