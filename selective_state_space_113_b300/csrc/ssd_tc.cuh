// ssd_tc.cuh -- the Mamba-2 form of the scan (structured state-space duality)
// on the sm_100-family tensor cores: tcgen05 MMAs with TMEM accumulators and
// TMA-staged, 128-byte-swizzled operand tiles.
//
// What it computes (news.han.ihouse.idv.tw article 1304: Mamba-2 found most of
// the SSM's computation equal to a masked matrix multiplication, reduced A to a
// scalar per head and discretises with Euler's rule), per batch entry b, head
// h, channel p < 64 of the head, step t, state n < N:
//   dt_t = softplus(dt[b,t,h] + dt_bias[h]);  h_t[n] = exp(dt_t A[h]) h_{t-1}[n]
//          + dt_t B_t[n] x_t[p];   y_t[p] = sum_n C_t[n] h_t[n] + Dskip[h] x_t[p]
// from h = 0.  In chunks of Q = 128 steps, with cum_t = A sum_{r<=t} dt_r
// inside the chunk and the N x 64 state H of the head entering the chunk:
//   S     = C B^T                                 (t x s, K = N)
//   Yx    = C H                                   (t x p, K = N)
//   Yi    = (Lmask o S) X,  Lmask[t,s] = exp(cum_t - cum_s) dt_s for s <= t
//   y     = Yi + exp(cum_t) Yx + Dskip X
//   G     = B^T (w o X),  w_s = exp(cum_end - cum_s) dt_s     (n x p, K = Q)
//   H_out = exp(cum_end) H + G
// Every product is an M = 128 tcgen05.mma (kind::f16, bf16 x bf16 -> fp32)
// issued by one thread: S (N = 128), Yx, Yi and G (N = 64), each as K = 16
// slices.  C, B and X are exact bf16 inputs; the masked scores, w o X and the
// entering state are not, so each is split into bf16 hi + lo parts
// (hi = bf16(v), lo = bf16(v - hi)) and multiplied twice, every sum in fp32.
//
// One CTA owns one (b, h) and walks its chunks in order.  Five warps:
//   warp 4      control: TMA loads of a chunk's C, B (K-major, two 64-wide
//               regions each) and X (its 128 steps x 64 channels), and the
//               MMAs, one elected thread;
//   warps 0..3  epilogue, thread i on TMEM lane i (row i of every product):
//               the step sizes and cumulative decay (a block scan), w o X, the
//               masked scores, the outputs, and the state, which it keeps in
//               registers (thread n holds row n of H) and rewrites after each
//               chunk as the next chunk's hi + lo operand.
// N = 64 runs the same code with the state padded to 128 by zeros (C and B
// regions 64..127 stay zero, so those rows of H stay zero).
// Every wait is bounded; a wait that gives up records the error, leaves the
// chunk loop, and the CTA still drains its copies and frees its TMEM.
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "faults.cuh"
#include "ptx.cuh"

namespace ssm {
namespace ssdtc {

constexpr int Q = 128;           // steps per chunk
constexpr int P = 64;            // channels per head
constexpr int NP = 128;          // state rows as the kernel holds them (N padded to 128)
constexpr int THREADS = 160;     // four epilogue warps, one control warp
constexpr int kCtl = 4;          // the control warp
constexpr float kLog2e = 1.4426950408889634f;

// Shared memory: every operand tile is 1024-byte aligned, rows of 128 bytes,
// 8-row atoms of 1 KB, 16-byte chunks swizzled by the row's index mod 8.
struct Layout {
    static constexpr int kC = 0;              // C: 2 regions [128 t][64 n], 16 KB each
    static constexpr int kB = 32768;          // B: 2 regions [128 s][64 n]
    static constexpr int kX = 65536;          // X: [128 s][64 p]
    static constexpr int kSh = 81920;         // masked scores, hi: 2 regions [128 t][64 s]
    static constexpr int kSl = 114688;        //                lo
    static constexpr int kWh = 147456;        // w o X, hi: [128 s][64 p]
    static constexpr int kWl = 163840;        //        lo
    static constexpr int kHh = 180224;        // entering state, hi: [128 n][64 p]
    static constexpr int kHl = 196608;        //                 lo
    static constexpr int kCum = 212992;       // cum_t log2(e), [Q] float
    static constexpr int kDt = kCum + 512;    // dt_t, [Q] float
    static constexpr int kWarpSum = kDt + 512;    // block scan: warp totals, [2][4] float
    static constexpr int kBar = kWarpSum + 64;    // mbarriers
    static constexpr int kNumBars = 8;
    static constexpr int kTmem = kBar + 8 * kNumBars;   // TMEM base address (written by alloc)
    static constexpr int kBytes = kTmem + 16;
    static constexpr int kSmemBytes = kBytes + 1024;    // + slack to align the base
};
static_assert(Layout::kSmemBytes <= 227 * 1024, "CTA shared memory");

// TMEM columns of the accumulators (fp32, lane = row).
constexpr uint32_t kColS = 0, kColYx = 128, kColYi = 192, kColG = 256;
constexpr uint32_t kTmemCols = 512;

// kInFull: a chunk's C, B, X landed; kInFree: the epilogue is done with them;
// kMma1 / kMma2: S and C H, then the masked product and G, completed;
// kEpReady: the masked scores and w o X are written; kHReady: the entering
// state's copy is written; kScan / kCum: the epilogue warps' block scan totals
// and cumulative decays are written (the epilogue's own rendezvous).
enum Bar : int { kInFull = 0, kInFree, kMma1, kEpReady, kMma2, kHReady, kScan, kCum };

struct Args {
    const bf16* x;
    const bf16* dt;
    const float* dt_bias;
    const float* A;
    const float* Dskip;
    bf16* y;
    float* h_last;
    long long batch, L, H;
    int N;
    unsigned long long wait_ns;
};

// Byte offset of 16-byte chunk c of row r in a 128B-swizzled region.
__device__ __forceinline__ uint32_t sw128(int r, int c) {
    return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}

// Shared-memory matrix descriptor, 128-byte swizzle.  lbo / sbo in bytes:
// K-major operands: sbo = 1024 (next 8 rows), lbo unused; MN-major: lbo = the
// next 64-wide block along M or N, sbo = 1024 (next 8 rows along K).
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = (uint64_t)((addr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;   // descriptor version of this architecture
    d |= (uint64_t)2 << 61;   // 128-byte swizzle
    return d;
}

// Instruction descriptor: fp32 accumulator, bf16 A and B, the majorness of
// each (0 K-major, 1 MN-major), N and M.
__host__ __device__ constexpr uint32_t idesc(int M, int N, int a_mn, int b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id,
                                    int accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(id), "r"(accumulate)
        : "memory");
}

// The mbarrier completes once every MMA this thread issued before has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            ptx::smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// hi = bf16(v), lo = bf16(v - hi), for a pair, packed.
__device__ __forceinline__ void split2(float a, float b, uint32_t& hi, uint32_t& lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    const __nv_bfloat162 l = __floats2bfloat162_rn(a - __low2float(h), b - __high2float(h));
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = *reinterpret_cast<const uint32_t*>(&l);
}

// Writes 32 values (one 64-byte half row, chunks c0..c0+3) as hi + lo.
__device__ __forceinline__ void store_split32(unsigned char* hi_base, unsigned char* lo_base,
                                              int row, int c0, const float (&v)[32]) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint4 h, l;
        split2(v[8 * c + 0], v[8 * c + 1], h.x, l.x);
        split2(v[8 * c + 2], v[8 * c + 3], h.y, l.y);
        split2(v[8 * c + 4], v[8 * c + 5], h.z, l.z);
        split2(v[8 * c + 6], v[8 * c + 7], h.w, l.w);
        *reinterpret_cast<uint4*>(hi_base + sw128(row, c0 + c)) = h;
        *reinterpret_cast<uint4*>(lo_base + sw128(row, c0 + c)) = l;
    }
}

// Bounded mbarrier wait (the common case, a completed phase, returns at once).
__device__ __forceinline__ bool bwait(uint64_t* bar, uint32_t parity, unsigned long long ns) {
    return ptx::mbar_wait(bar, parity, ns, nullptr);
}

// Bounded wait whose outcome every lane of the warp shares.
__device__ __forceinline__ bool wwait(uint64_t* bar, uint32_t parity, unsigned long long ns) {
    return __all_sync(0xffffffffu, bwait(bar, parity, ns));
}

// Lane 0 arrives once the whole warp's earlier writes are done.
__device__ __forceinline__ void warp_arrive(uint64_t* bar, int lane) {
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(bar);
}

__global__ void __launch_bounds__(THREADS, 1)
ssd_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmB,
              const __grid_constant__ CUtensorMap tmC, const Args a) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* sm = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + Layout::kBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + Layout::kTmem);
    float* cum = reinterpret_cast<float*>(sm + Layout::kCum);
    float* dts = reinterpret_cast<float*>(sm + Layout::kDt);
    float* wsum = reinterpret_cast<float*>(sm + Layout::kWarpSum);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const long long bh = blockIdx.x;
    const long long b = bh / a.H, hh = bh % a.H;
    const long long nchunks = (a.L + Q - 1) / Q;
    const bool two_regions = a.N > 64;

    // ---- set-up: barriers, zeroed state operand and padding regions, TMEM
    if (tid == 0) {
        ptx::mbar_init(&bar[kInFull], 1);
        ptx::mbar_init(&bar[kInFree], 4);
        ptx::mbar_init(&bar[kMma1], 1);
        ptx::mbar_init(&bar[kEpReady], 4);
        ptx::mbar_init(&bar[kMma2], 1);
        ptx::mbar_init(&bar[kHReady], 4);
        ptx::mbar_init(&bar[kScan], 4);
        ptx::mbar_init(&bar[kCum], 4);
        ptx::fence_mbar_init();
    }
    {
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
        for (int i = tid; i < 2 * 16384 / 16; i += THREADS) {
            reinterpret_cast<uint4*>(sm + Layout::kHh)[i] = z;   // kHh and kHl are adjacent
            if (!two_regions) {
                reinterpret_cast<uint4*>(sm + Layout::kC + 16384)[i % 1024] = z;
                reinterpret_cast<uint4*>(sm + Layout::kB + 16384)[i % 1024] = z;
            }
        }
    }
    if (warp == kCtl) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         ptx::smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    ptx::fence_proxy_async_shared();   // the zeroed operands, for the tensor cores
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    bool failed = false;

    if (warp == kCtl) {
        // ------------------------------------------------------------- control
        if (lane == 0) {
            ptx::prefetch_tensormap(&tmX);
            ptx::prefetch_tensormap(&tmB);
            ptx::prefetch_tensormap(&tmC);
            const uint32_t in_bytes = (two_regions ? 4 : 2) * 16384 + 16384;
            const uint32_t sC = ptx::smem_u32(sm + Layout::kC), sB = ptx::smem_u32(sm + Layout::kB);
            const uint32_t sX = ptx::smem_u32(sm + Layout::kX);
            const uint32_t sSh = ptx::smem_u32(sm + Layout::kSh), sSl = ptx::smem_u32(sm + Layout::kSl);
            const uint32_t sWh = ptx::smem_u32(sm + Layout::kWh), sWl = ptx::smem_u32(sm + Layout::kWl);
            const uint32_t sHh = ptx::smem_u32(sm + Layout::kHh), sHl = ptx::smem_u32(sm + Layout::kHl);
            constexpr uint32_t idS = idesc(128, 128, 0, 0), idY = idesc(128, 64, 0, 1),
                               idG = idesc(128, 64, 1, 1);
            for (long long c = 0; c < nchunks && !failed; ++c) {
                const uint32_t ph = (uint32_t)(c & 1);
                if (c > 0 && !bwait(&bar[kInFree], ph ^ 1u, a.wait_ns)) { failed = true; break; }
                ptx::mbar_arrive_expect_tx(&bar[kInFull], in_bytes);
                const int t0 = (int)(c * Q);
                ptx::tma_load_3d(sm + Layout::kC, &tmC, &bar[kInFull], 0, t0, (int)b);
                ptx::tma_load_3d(sm + Layout::kB, &tmB, &bar[kInFull], 0, t0, (int)b);
                if (two_regions) {
                    ptx::tma_load_3d(sm + Layout::kC + 16384, &tmC, &bar[kInFull], 64, t0, (int)b);
                    ptx::tma_load_3d(sm + Layout::kB + 16384, &tmB, &bar[kInFull], 64, t0, (int)b);
                }
                ptx::tma_load_4d(sm + Layout::kX, &tmX, &bar[kInFull], 0, (int)hh, t0, (int)b);
                if (!bwait(&bar[kInFull], ph, a.wait_ns) || !bwait(&bar[kHReady], ph, a.wait_ns)) {
                    failed = true;
                    break;
                }
                fence_after_sync();
                // S = C B^T and Yx = C H (hi, then lo)
                for (int k = 0; k < 8; ++k) {
                    const uint32_t ko = (uint32_t)((k >> 2) * 16384 + (k & 3) * 32);
                    mma(tmem + kColS, sdesc(sC + ko, 16, 1024), sdesc(sB + ko, 16, 1024), idS, k > 0);
                }
                for (int k = 0; k < 8; ++k) {
                    const uint32_t ko = (uint32_t)((k >> 2) * 16384 + (k & 3) * 32);
                    mma(tmem + kColYx, sdesc(sC + ko, 16, 1024), sdesc(sHh + k * 2048, 16384, 1024), idY, k > 0);
                }
                for (int k = 0; k < 8; ++k) {
                    const uint32_t ko = (uint32_t)((k >> 2) * 16384 + (k & 3) * 32);
                    mma(tmem + kColYx, sdesc(sC + ko, 16, 1024), sdesc(sHl + k * 2048, 16384, 1024), idY, 1);
                }
                mma_commit(&bar[kMma1]);
                if (!bwait(&bar[kEpReady], ph, a.wait_ns)) { failed = true; break; }
                fence_after_sync();
                // Yi = (masked S) X and G = B^T (w o X), each hi then lo
                for (int part = 0; part < 2; ++part) {
                    const uint32_t sS = part ? sSl : sSh, sW = part ? sWl : sWh;
                    for (int k = 0; k < 8; ++k) {
                        const uint32_t ko = (uint32_t)((k >> 2) * 16384 + (k & 3) * 32);
                        mma(tmem + kColYi, sdesc(sS + ko, 16, 1024), sdesc(sX + k * 2048, 16384, 1024), idY,
                            part > 0 || k > 0);
                        mma(tmem + kColG, sdesc(sB + k * 2048, 16384, 1024), sdesc(sW + k * 2048, 16384, 1024),
                            idG, part > 0 || k > 0);
                    }
                }
                mma_commit(&bar[kMma2]);
            }
            if (failed) atomicOr(&g_error_word, kErrTimeout);
            // Leave no copy or product in flight (bounded): the last chunk's
            // loads and MMAs have completed once its kMma2 phase has.
            if (nchunks > 0 && !failed)
                bwait(&bar[kMma2], (uint32_t)((nchunks - 1) & 1), a.wait_ns);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int row = 32 * warp + lane;   // TMEM lane; step t, or state row n
        const uint32_t lane_addr = tmem + ((uint32_t)(32 * warp) << 16);
        const float A = a.A[hh];
        const float kb2 = a.dt_bias ? a.dt_bias[hh] * kLog2e : 0.0f;
        const float dsk = a.Dskip ? a.Dskip[hh] : 0.0f;
        float Hs[P];   // row `row` of the state (zero for rows >= N)
#pragma unroll
        for (int p = 0; p < P; ++p) Hs[p] = 0.0f;
        // the zero entering state is in place
        fence_before_sync();
        warp_arrive(&bar[kHReady], lane);
        for (long long c = 0; c < nchunks && !failed; ++c) {
            const uint32_t ph = (uint32_t)(c & 1);
            const long long t0 = c * Q;
            const int nv = (int)(a.L - t0 < Q ? a.L - t0 : Q);
            // step size and the cumulative decay (inclusive block scan of A dt)
            float dtv = 0.0f;
            if (row < nv) {
                const float v2 = fmaf(__bfloat162float(a.dt[(b * a.L + t0 + row) * a.H + hh]), kLog2e, kb2);
                dtv = (v2 > 28.853901f ? v2 : ptx::lg2(1.0f + ptx::ex2(v2))) * 0.6931471805599453f;
            }
            float sc = A * dtv;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float v = __shfl_up_sync(0xffffffffu, sc, o);
                if (lane >= o) sc += v;
            }
            // warp totals (double-buffered by chunk parity), then the prefix.
            // The previous chunk's cum / dts are no longer read: every warp
            // finished its masked scores before kMma2, which this warp passed.
            if (lane == 31) wsum[4 * ph + warp] = sc;
            warp_arrive(&bar[kScan], lane);
            if (!wwait(&bar[kScan], ph, a.wait_ns)) { failed = true; break; }
            for (int w2 = 0; w2 < warp; ++w2) sc += wsum[4 * ph + w2];
            const float cend = wsum[4 * ph] + wsum[4 * ph + 1] + wsum[4 * ph + 2] + wsum[4 * ph + 3];
            const float ct = sc * kLog2e;
            cum[row] = ct;
            dts[row] = dtv;
            const float ecum = ptx::ex2(ct);                       // exp(cum_t)
            const float wt = ptx::ex2((cend - sc) * kLog2e) * dtv;  // w_t
            const float dend = ptx::ex2(cend * kLog2e);            // exp(cum_end)
            warp_arrive(&bar[kCum], lane);
            if (!wwait(&bar[kInFull], ph, a.wait_ns)) { failed = true; break; }
            // w o X, row s = row, split hi + lo
            {
                const unsigned char* X = sm + Layout::kX;
#pragma unroll
                for (int cc = 0; cc < 8; ++cc) {
                    const uint4 xv = *reinterpret_cast<const uint4*>(X + sw128(row, cc));
                    const __nv_bfloat162* x2 = reinterpret_cast<const __nv_bfloat162*>(&xv);
                    uint4 h, l;
                    uint32_t* hp = &h.x;
                    uint32_t* lp = &l.x;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float2 f = __bfloat1622float2(x2[q]);
                        split2(wt * f.x, wt * f.y, hp[q], lp[q]);
                    }
                    *reinterpret_cast<uint4*>(sm + Layout::kWh + sw128(row, cc)) = h;
                    *reinterpret_cast<uint4*>(sm + Layout::kWl + sw128(row, cc)) = l;
                }
            }
            // masked scores of row t = row: S[t,s] exp(cum_t - cum_s) dt_s, s <= t
            if (!wwait(&bar[kMma1], ph, a.wait_ns) || !wwait(&bar[kCum], ph, a.wait_ns)) {
                failed = true;
                break;
            }
            fence_after_sync();
#pragma unroll 1
            for (int piece = 0; piece < 4; ++piece) {
                float v[32];
                if (piece <= warp) {   // some s of the piece are <= t (warp-uniform)
                    tmem_ld32(lane_addr + kColS + 32 * piece, v);
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int s = 32 * piece + j;
                        v[j] = s <= row ? v[j] * ptx::ex2(ct - cum[s]) * dts[s] : 0.0f;
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = 0.0f;
                }
                // columns s = 32 piece + 0..31: region s / 64, chunks (s % 64) / 8
                const int region = piece >> 1, c0 = (piece & 1) * 4;
                store_split32(sm + Layout::kSh + region * 16384, sm + Layout::kSl + region * 16384, row,
                              c0, v);
            }
            ptx::fence_proxy_async_shared();
            fence_before_sync();
            warp_arrive(&bar[kEpReady], lane);
            // outputs of step t = row: Yi + exp(cum_t) Yx + Dskip x
            if (!wwait(&bar[kMma2], ph, a.wait_ns)) { failed = true; break; }
            fence_after_sync();
            {
                const unsigned char* X = sm + Layout::kX;
                bf16* yrow = a.y + ((b * a.L + t0 + row) * a.H + hh) * P;
#pragma unroll 1
                for (int half = 0; half < 2; ++half) {
                    float yi[32], yx[32];
                    tmem_ld32(lane_addr + kColYi + 32 * half, yi);
                    tmem_ld32(lane_addr + kColYx + 32 * half, yx);
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        const uint4 xv = *reinterpret_cast<const uint4*>(X + sw128(row, 4 * half + cc));
                        const __nv_bfloat162* x2 = reinterpret_cast<const __nv_bfloat162*>(&xv);
                        uint4 o;
                        uint32_t* op = &o.x;
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float2 f = __bfloat1622float2(x2[q]);
                            const int j = 8 * cc + 2 * q;
                            const __nv_bfloat162 r2 = __floats2bfloat162_rn(
                                fmaf(dsk, f.x, fmaf(ecum, yx[j], yi[j])),
                                fmaf(dsk, f.y, fmaf(ecum, yx[j + 1], yi[j + 1])));
                            op[q] = *reinterpret_cast<const uint32_t*>(&r2);
                        }
                        if (row < nv)
                            *reinterpret_cast<uint4*>(yrow + 32 * half + 8 * cc) = o;
                    }
                }
            }
            // X and the products' inputs are free for the next chunk
            fence_before_sync();
            warp_arrive(&bar[kInFree], lane);
            // the state: H <- exp(cum_end) H + G (row n = row), then its hi + lo
            // copy for the next chunk's C H
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float g[32];
                tmem_ld32(lane_addr + kColG + 32 * half, g);
#pragma unroll
                for (int j = 0; j < 32; ++j) Hs[32 * half + j] = fmaf(dend, Hs[32 * half + j], g[j]);
            }
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float v[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = Hs[32 * half + j];
                store_split32(sm + Layout::kHh, sm + Layout::kHl, row, 4 * half, v);
            }
            ptx::fence_proxy_async_shared();
            fence_before_sync();
            warp_arrive(&bar[kHReady], lane);
        }
        if (failed && lane == 0) atomicOr(&g_error_word, kErrTimeout);
        if (!failed && a.h_last && row < a.N) {
            float* base = a.h_last + (b * a.H + hh) * P * (long long)a.N + row;
#pragma unroll
            for (int p = 0; p < P; ++p) base[(long long)p * a.N] = Hs[p];
        }
    }
    // ---- tear-down: every TMEM read and MMA is done before the columns go
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (warp == kCtl)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
}

}  // namespace ssdtc
}  // namespace ssm

#include "tma_host.cuh"

namespace ssm {
namespace ssdtc {

// bf16, P == 64, N == 64 or 128, x, B, C, y 16-byte aligned, batch*H > 0,
// L > 0 (checked by the caller).
inline cudaError_t launch_ssd_tc(const bf16* x, const bf16* dt, const float* dt_bias,
                                 const float* A, const bf16* Bm, const bf16* Cm,
                                 const float* Dskip, bf16* y, float* h_last, long long batch,
                                 long long L, long long H, int N, unsigned long long wait_ns,
                                 cudaStream_t s) {
    CUtensorMap mX, mB, mC;
    const cuuint64_t es = 2;
    const cuuint64_t dX[4] = {(cuuint64_t)P, (cuuint64_t)H, (cuuint64_t)L, (cuuint64_t)batch};
    const cuuint64_t sX[3] = {P * es, (cuuint64_t)H * P * es, (cuuint64_t)L * H * P * es};
    const cuuint32_t bX[4] = {64u, 1u, (cuuint32_t)Q, 1u};
    const cuuint64_t dBC[3] = {(cuuint64_t)N, (cuuint64_t)L, (cuuint64_t)batch};
    const cuuint64_t sBC[2] = {(cuuint64_t)N * es, (cuuint64_t)L * N * es};
    const cuuint32_t bBC[3] = {64u, (cuuint32_t)Q, 1u};
    const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    if (!tma::make_map(&mX, bf, 4, x, dX, sX, bX, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !tma::make_map(&mB, bf, 3, Bm, dBC, sBC, bBC, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !tma::make_map(&mC, bf, 3, Cm, dBC, sBC, bBC, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    Args a;
    a.x = x;
    a.dt = dt;
    a.dt_bias = dt_bias;
    a.A = A;
    a.Dskip = Dskip;
    a.y = y;
    a.h_last = h_last;
    a.batch = batch;
    a.L = L;
    a.H = H;
    a.N = N;
    a.wait_ns = wait_ns;
    cudaError_t e = cudaFuncSetAttribute(ssd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Layout::kSmemBytes);
    if (e != cudaSuccess) return e;
    if (fault::launch_refused()) return cudaErrorLaunchFailure;
    ssd_tc_kernel<<<(unsigned)(batch * H), THREADS, Layout::kSmemBytes, s>>>(mX, mB, mC, a);
    return cudaGetLastError();
}

}  // namespace ssdtc
}  // namespace ssm
