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
#include <mutex>

#include "common.cuh"
#include "context.cuh"
#include "faults.cuh"
#include "ptx.cuh"
#include "tma_host.cuh"


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


// ---------------------------------------------------------------------------
// Tiled kernel (taken when D % 8 == 0 and every row is 16-byte aligned).  The
// step is a stream over the [batch, D, 16] state, but the kernel above holds
// in flight only what its registers carry, about half of what HBM needs to
// run at its rate.  Here each CTA is persistent and walks a contiguous range
// of tiles, a tile being TC channels x NB batch entries: NB*TC*64 bytes of
// state plus the matching u, delta and z and the NB rows of B and C.  One
// producer thread keeps STAGES tiles in flight in a shared-memory ring, each
// operand of a tile arriving by ONE tensor copy (six per tile): the copy
// engine takes a fixed time per copy whatever its size, so few large copies,
// not many small ones, are what keep HBM busy.  The state arrives 64-byte
// swizzled (the 16-byte chunk c of row r stored at chunk c ^ ((r >> 1) & 3)),
// which makes the one-thread-per-channel reads and writes of shared memory
// free of bank conflicts.
//
// G groups of TC compute threads take the ring's tiles in turn; a thread owns
// one channel, walks the tile's NB batch entries and keeps A and 1/A of its
// channel in registers (tiles are ordered channel block first, so a CTA meets
// few channel blocks).  STAGES is a multiple of G, so every stage has one
// group as its only reader.  The wait on a stage's full barrier names the
// phase by its parity, which only identifies the phase if the previous one
// has completed; the group that waits for round j of a stage is the one that
// waited for round j - 1, so that holds.  With readers alternating between
// groups, a group could meet a stage whose previous copy had not landed and
// pass its wait at once, reading the old tile and freeing the stage early.  The new state goes back into the tile in place, each
// warp re-reads its 32 rows linearly and stores them to global memory in
// 512-byte coalesced pieces; y is stored directly.  Tensor copies read
// out-of-range rows (channels past D, entries past batch) as zeros; nothing
// is stored for them.
//
// Per state the update is
//   A_bar = 2^(dl A)  (dl = dt / ln 2, the softplus taken in base 2)
//   B_bar u = coef B u,  coef = (A_bar - 1) / A, as dt p(dt A) when |dt A| < 1/32
//   (p the degree-3 Taylor polynomial of (e^x - 1) / x, truncation < 1e-9,
//   which also gives coef = dt at A == 0), else (A_bar - 1) * (1/A)
// and the readout adds C h, D u and the SiLU gate as the kernel above does.
constexpr int kTileTC = 128;   // channels per tile
constexpr int kTileNB = 4;     // batch entries per tile

// Ring depth and compute groups per element type: six bf16 stages (216 KB) or
// four float32 stages (156 KB) fit in shared memory.
template <typename T>
struct TileRing {
    static constexpr int kStages = sizeof(T) == 2 ? 6 : 4;
    static constexpr int kGroups = sizeof(T) == 2 ? 3 : 2;
};

struct StepMaps {
    CUtensorMap state, u, delta, z, B, C;
};

template <typename T, int TC, int NB>
struct TileLayout {
    static constexpr int kState = NB * TC * NS * 4;
    static constexpr int kVec = NB * TC * (int)sizeof(T);
    static constexpr int kRow = (NB * NS * (int)sizeof(T) + 127) / 128 * 128;
    static constexpr int kU = kState;
    static constexpr int kDelta = kU + kVec;
    static constexpr int kZ = kDelta + kVec;
    static constexpr int kB = kZ + kVec;
    static constexpr int kC = kB + kRow;
    static constexpr int kStage = (kC + kRow + 1023) / 1024 * 1024;   // swizzled tiles: 1 KB aligned
};

template <typename T, int TC, int NB, int STAGES>
constexpr int tile_smem_bytes() {
    return STAGES * TileLayout<T, TC, NB>::kStage + 2 * STAGES * 8 + 1024;
}

// 16 values of a B or C row in shared memory, as float32.
__device__ __forceinline__ void row16(const unsigned char* p, float (&v)[NS], const bf16*) {
    const uint4 w0 = reinterpret_cast<const uint4*>(p)[0], w1 = reinterpret_cast<const uint4*>(p)[1];
    const uint32_t w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}
__device__ __forceinline__ void row16(const unsigned char* p, float (&v)[NS], const float*) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float4 f = reinterpret_cast<const float4*>(p)[q];
        v[4 * q] = f.x; v[4 * q + 1] = f.y; v[4 * q + 2] = f.z; v[4 * q + 3] = f.w;
    }
}

template <typename T, int TC, int NB, int STAGES, int G>
__global__ void __launch_bounds__(G * TC + 32, 1)
step16_tiled_kernel(const __grid_constant__ StepMaps maps, float* __restrict__ state,
                    const float* __restrict__ dt_bias, const float* __restrict__ A,
                    const float* __restrict__ Dskip, int has_z, T* __restrict__ y, int batch,
                    int D, int tiles, unsigned long long wait_ns) {
    using L = TileLayout<T, TC, NB>;
    static_assert(STAGES % G == 0, "each stage needs a single reading group");
    constexpr int kCompute = G * TC;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024 - (ptx::smem_u32(smem_raw) & 1023)) & 1023);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * L::kStage);
    uint64_t* freed = full + STAGES;
    const int tid = threadIdx.x, lane = tid & 31;
    const int lo = (int)((long long)blockIdx.x * tiles / gridDim.x);
    const int n = (int)((long long)(blockIdx.x + 1) * tiles / gridDim.x) - lo;
    const int nbb = (batch + NB - 1) / NB;   // tiles per channel block
    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(full + s, 1);
            ptx::mbar_init(freed + s, TC / 32);
        }
        ptx::fence_mbar_init();
    }
    __syncthreads();
    const volatile unsigned* abort = &g_error_word;

    if (tid >= kCompute) {
        // ---- producer: one thread issues the six copies of each tile
        if (tid != kCompute) return;
        ptx::prefetch_tensormap(&maps.state);
        ptx::prefetch_tensormap(&maps.u);
        ptx::prefetch_tensormap(&maps.delta);
        ptx::prefetch_tensormap(&maps.B);
        ptx::prefetch_tensormap(&maps.C);
        if (has_z) ptx::prefetch_tensormap(&maps.z);
        const uint32_t bytes = (uint32_t)(L::kState + (has_z ? 3 : 2) * L::kVec +
                                          2 * NB * NS * (int)sizeof(T));
        bool ok = true;
        int k = 0;
        for (; k < n; ++k) {
            const int s = k % STAGES;
            if (k >= STAGES && !ptx::mbar_wait(freed + s, ((k / STAGES) - 1) & 1, wait_ns, abort)) {
                ok = false;
                break;
            }
            const int t = lo + k, cb = t / nbb, b0 = (t - cb * nbb) * NB, d0 = cb * TC;
            unsigned char* st = smem + s * L::kStage;
            ptx::mbar_arrive_expect_tx(full + s, bytes);
            ptx::tma_load_3d(st, &maps.state, full + s, 0, d0, b0);
            ptx::tma_load_3d(st + L::kU, &maps.u, full + s, d0, b0, 0);
            ptx::tma_load_3d(st + L::kDelta, &maps.delta, full + s, d0, b0, 0);
            if (has_z) ptx::tma_load_3d(st + L::kZ, &maps.z, full + s, d0, b0, 0);
            ptx::tma_load_3d(st + L::kB, &maps.B, full + s, 0, b0, 0);
            ptx::tma_load_3d(st + L::kC, &maps.C, full + s, 0, b0, 0);
        }
        if (!ok) atomicOr(&g_error_word, kErrTimeout);
        // every copy this thread issued lands before the CTA exits
        for (int j = k - STAGES > 0 ? k - STAGES : 0; j < k; ++j)
            if (!ptx::mbar_wait(full + j % STAGES, (j / STAGES) & 1, wait_ns, nullptr))
                atomicOr(&g_error_word, kErrTimeout);
        return;
    }

    // ---- compute: group g takes tiles g, g + G, ...; one thread per channel
    const int g = tid / TC, ch = tid % TC, wq = ch >> 5;
    int cb_held = -1;
    float a[NS], ia[NS];
    float bias = 0.0f, dsk = 0.0f;
    for (int k = g; k < n; k += G) {
        const int t = lo + k, cb = t / nbb, b0 = (t - cb * nbb) * NB, d0 = cb * TC;
        const int nch = min(TC, D - d0);
        const bool valid = ch < nch;
        if (cb != cb_held) {   // uniform across the group
            cb_held = cb;
            const int c = valid ? ch : 0;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 f = reinterpret_cast<const float4*>(A)[(size_t)(d0 + c) * 4 + q];
                a[4 * q] = f.x; a[4 * q + 1] = f.y; a[4 * q + 2] = f.z; a[4 * q + 3] = f.w;
            }
#pragma unroll
            for (int i = 0; i < NS; ++i) ia[i] = ptx::rcp(a[i]);   // unused where A == 0
            bias = dt_bias ? dt_bias[d0 + c] : 0.0f;
            dsk = Dskip ? Dskip[d0 + c] : 0.0f;
        }
        const int s = k % STAGES;
        if (!__all_sync(0xffffffffu, ptx::mbar_wait(full + s, (k / STAGES) & 1, wait_ns, abort))) {
            if (lane == 0) atomicOr(&g_error_word, kErrTimeout);
            return;
        }
        unsigned char* st = smem + s * L::kStage;
        for (int j = 0; j < NB; ++j) {
            const int b = b0 + j;
            if (b >= batch) break;
            unsigned char* sj = st + j * TC * 64;
            float4* hs[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                hs[q] = reinterpret_cast<float4*>(sj + ch * 64 + ((q ^ ((ch >> 1) & 3)) * 16));
            float h[NS];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 f = *hs[q];
                h[4 * q] = f.x; h[4 * q + 1] = f.y; h[4 * q + 2] = f.z; h[4 * q + 3] = f.w;
            }
            const float ut = to_f32(reinterpret_cast<const T*>(st + L::kU)[j * TC + ch]);
            const float v = to_f32(reinterpret_cast<const T*>(st + L::kDelta)[j * TC + ch]) + bias;
            const float zt = has_z ? to_f32(reinterpret_cast<const T*>(st + L::kZ)[j * TC + ch]) : 0.0f;
            float bv[NS], cv[NS];
            row16(st + L::kB + j * NS * (int)sizeof(T), bv, (const T*)nullptr);
            row16(st + L::kC + j * NS * (int)sizeof(T), cv, (const T*)nullptr);
            const float dl = v > 20.0f ? v * kLog2e : ptx::lg2(1.0f + ptx::ex2(v * kLog2e));
            const float dt = dl * kLn2;
            float hn[NS];
            float acc = 0.0f;
#pragma unroll
            for (int i = 0; i < NS; ++i) {
                const float x = dt * a[i];
                const float ex = ptx::ex2(dl * a[i]);
                const float p = fmaf(x, fmaf(x, fmaf(x, 1.0f / 24.0f, 1.0f / 6.0f), 0.5f), 1.0f);
                const float coef = fabsf(x) < 0.03125f ? dt * p : (ex - 1.0f) * ia[i];
                hn[i] = fmaf(ex, h[i], coef * (bv[i] * ut));
                acc = fmaf(cv[i], hn[i], acc);
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) *hs[q] = make_float4(hn[4 * q], hn[4 * q + 1], hn[4 * q + 2], hn[4 * q + 3]);
            __syncwarp();
            // the warp's 32 rows, re-read linearly: 16-byte piece q of the
            // 2 KB region is chunk (q & 3) ^ ((r >> 1) & 3) of row r = q / 4
            float4 o[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) o[m] = reinterpret_cast<const float4*>(sj + wq * 2048)[lane + 32 * m];
            __syncwarp();
            const size_t row0 = (size_t)b * (size_t)D + (size_t)d0;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int q = lane + 32 * m, r = wq * 32 + (q >> 2);
                if (r < nch)
                    reinterpret_cast<float4*>(state + (row0 + r) * NS)[(q & 3) ^ ((r >> 1) & 3)] = o[m];
            }
            if (valid) {
                acc = fmaf(dsk, ut, acc);
                if (has_z) acc *= zt * ptx::rcp(1.0f + ptx::ex2(-zt * kLog2e));
                y[row0 + ch] = from_f32<T>(acc);
            }
        }
        // every value read from the stage has been used, and the new state
        // written into it is ordered before the copy engine's next writes
        // there: hand it back
        ptx::fence_proxy_async_shared();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(freed + s);
    }
}

// Launches step16_tiled_kernel, one persistent CTA per SM.  Preconditions
// (checked by the caller): D % 8 == 0, u, delta, z, B, C, state and A 16-byte
// aligned, ceil(D / 128) * ceil(batch / 4) < 2^31.
template <typename T>
static cudaError_t launch_step16_tiled(float* state, const T* u, const T* delta,
                                       const float* dt_bias, const float* A, const T* Bm,
                                       const T* Cm, const float* Dskip, const T* z, T* y,
                                       long long batch, long long D, unsigned long long wait_ns,
                                       cudaStream_t stream) {
    constexpr int TC = kTileTC, NB = kTileNB, S = TileRing<T>::kStages, G = TileRing<T>::kGroups;
    auto kern = step16_tiled_kernel<T, TC, NB, S, G>;
    constexpr int smem = tile_smem_bytes<T, TC, NB, S>();
    static_assert(smem <= 227 * 1024, "ring exceeds a CTA's shared memory");
    const CUtensorMapDataType dt =
        sizeof(T) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    const cuuint64_t es = sizeof(T);
    StepMaps m;
    {
        const cuuint64_t dims[3] = {NS, (cuuint64_t)D, (cuuint64_t)batch};
        const cuuint64_t strides[2] = {NS * 4, (cuuint64_t)D * NS * 4};
        const cuuint32_t box[3] = {NS, TC, NB};
        if (!tma::cached_map(&m.state, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, state, dims, strides, box,
                           CU_TENSOR_MAP_SWIZZLE_64B))
            return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)batch, 1};
        const cuuint64_t strides[2] = {(cuuint64_t)D * es, (cuuint64_t)D * es * (cuuint64_t)batch};
        const cuuint32_t box[3] = {TC, NB, 1};
        if (!tma::cached_map(&m.u, dt, 3, u, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE) ||
            !tma::cached_map(&m.delta, dt, 3, delta, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE) ||
            (z && !tma::cached_map(&m.z, dt, 3, z, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE)))
            return cudaErrorInvalidValue;
        if (!z) m.z = m.u;   // not read
    }
    {
        const cuuint64_t dims[3] = {NS, (cuuint64_t)batch, 1};
        const cuuint64_t strides[2] = {NS * es, NS * es * (cuuint64_t)batch};
        const cuuint32_t box[3] = {NS, NB, 1};
        if (!tma::cached_map(&m.B, dt, 3, Bm, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE) ||
            !tma::cached_map(&m.C, dt, 3, Cm, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    }
    // per device and context, once: the kernel's shared-memory limit (an
    // attribute of the context, set again after the context was destroyed
    // and another made current) and the SM count
    constexpr int kMaxDev = 64;
    static std::mutex mu;
    struct Slot {
        unsigned long long ctx;   // context ID
        int sms;
    };
    static Slot sms_of[kMaxDev] = {};
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    unsigned long long ctx = context::current_id();
    if (ctx && dev >= 0 && dev < kMaxDev) {
        std::lock_guard<std::mutex> lock(mu);
        if (sms_of[dev].ctx == ctx) sms = sms_of[dev].sms;
    }
    if (sms == 0) {
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        ctx = context::current_id();   // current now
        if (ctx && dev >= 0 && dev < kMaxDev) {
            std::lock_guard<std::mutex> lock(mu);
            sms_of[dev] = Slot{ctx, sms};
        }
    }
    const long long tiles = ((D + TC - 1) / TC) * ((batch + NB - 1) / NB);
    const long long grid = tiles < sms ? tiles : sms;
    if (fault::launch_refused()) return cudaErrorLaunchFailure;
    kern<<<(unsigned)grid, G * TC + 32, smem, stream>>>(m, state, dt_bias, A, Dskip, z ? 1 : 0, y,
                                                        (int)batch, (int)D, (int)tiles, wait_ns);
    return cudaGetLastError();
}

}  // namespace stepk
}  // namespace ssm
