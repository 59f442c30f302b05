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

#include "common.cuh"
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
template <typename T>
__global__ void __launch_bounds__(THREADS)
step16_kernel(float* __restrict__ state, const T* __restrict__ u, const T* __restrict__ delta,
              const float* __restrict__ dt_bias, const float* __restrict__ A,
              const T* __restrict__ Bm, const T* __restrict__ Cm,
              const float* __restrict__ Dskip, const T* __restrict__ z, T* __restrict__ y,
              int D) {
    const int b = blockIdx.y;
    const int tid = blockIdx.x * THREADS + threadIdx.x;   // < 4*D (checked on the host)
    const int part = tid & 3;                              // states 4*part .. 4*part + 3
    // Threads past the last channel stay (the shuffles below need the whole
    // warp) but work on channel 0 and store nothing.
    const bool valid = (tid >> 2) < D;
    const int d = valid ? (tid >> 2) : 0;
    // 32-bit offsets within one batch entry (4*D*16 < 2^31 is checked on the
    // host); the batch offset is applied to the base pointers once.
    const size_t row = (size_t)b * (size_t)D;
    const T* ub = u + row;
    const float ut = to_f32(ub[d]);
    float4* hp = reinterpret_cast<float4*>(state + row * NS) + (d * 4 + part);
    const float4 h4 = *hp;
    const float4 a4 = reinterpret_cast<const float4*>(A)[d * 4 + part];
    // softplus in the base-2 domain, dl = log2(1 + 2^(v log2 e)) = dt / ln 2,
    // computed by the first lane of the channel and shared with the others.
    float dl = 0.0f;
    if (part == 0) {
        const float v = to_f32(delta[row + d]) + (dt_bias ? dt_bias[d] : 0.0f);
        dl = v > 20.0f ? v * kLog2e : ptx::lg2(1.0f + ptx::ex2(v * kLog2e));
    }
    dl = __shfl_sync(0xffffffffu, dl, threadIdx.x & ~3);
    const float dt = dl * kLn2;
    const T* Bt = Bm + (size_t)b * NS + 4 * part;
    const T* Ct = Cm + (size_t)b * NS + 4 * part;
    const float a[4] = {a4.x, a4.y, a4.z, a4.w};
    const float h[4] = {h4.x, h4.y, h4.z, h4.w};
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
        hn[i] = fmaf(ex, h[i], coef * to_f32(Bt[i]) * ut);
        acc = fmaf(to_f32(Ct[i]), hn[i], acc);
    }
    if (valid) *hp = make_float4(hn[0], hn[1], hn[2], hn[3]);
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
    if (valid && part == 0) {
        acc = fmaf(Dskip ? Dskip[d] : 0.0f, ut, acc);
        if (z) {
            const float zt = to_f32(z[row + d]);
            acc *= zt * ptx::rcp(1.0f + ptx::ex2(-zt * kLog2e));
        }
        y[row + d] = from_f32<T>(acc);
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
    const dim3 grid((unsigned)((4 * D + THREADS - 1) / THREADS), (unsigned)batch);
    step16_kernel<T><<<grid, THREADS, 0, stream>>>(state, u, delta, dt_bias, A, Bm, Cm, Dskip,
                                                   z, y, (int)D);
    return cudaGetLastError();
}

}  // namespace stepk
}  // namespace ssm
