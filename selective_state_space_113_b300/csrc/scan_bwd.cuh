// scan_bwd.cuh -- backward pass of the zero-order-hold selective scan.
//
// The fused kernel on the ta-paperlens page ("代償と、それを払う方法（並列
// スキャン）") keeps the state in on-chip memory and, in the backward pass,
// recomputes the states instead of storing them.  This file does the same:
// no [batch, L, D, N] tensor of states ever reaches HBM.
//
// Derivatives (the adjoint of the recurrence; y = s g with
// s = sum_n C_n h_n + Dskip u, g = silu(z); lam_n = dLoss/dh_t[n]):
//   ds = dy g;   dz = dy s sig(z) (1 + z (1 - sig(z)))
//   lam_n += ds C_n                       (h_t is read out at step t)
//   dC_t[n] += ds h_t[n]                  (summed over channels)
//   dB_t[n] += lam_n q_n u                (summed over channels), q = (Abar-1)/a
//   du = ds Dskip + sum_n lam_n q_n B_n
//   ddt = sum_n lam_n (a_n h_t[n] + B_n u)            (= d h_t / d dt . lam)
//   dA_n += lam_n dt (h_t[n] - dt B_n u psi(dt a_n)), psi(x) = (e^x - 1 - x)/x^2
//   ddelta = ddt sig(delta + bias);   ddt_bias += ddelta;   dDskip += ds u
//   lam_n <- Abar_n lam_n                 (h_{t-1} feeds h_t)
// starting from lam = dh_last at the last step.  The forms use h_t only
// (never h_{t-1}): Abar h_{t-1} = h_t - q B u turns d h_t/d dt and d h_t/d a
// into the two expressions above.  For a geometric A row (a_n = (n+1) a0) the
// dA term is accumulated as dt T_n - lam_n q_n B_n u with T_n the ddt term,
// which is a_n times the one above, and divided by a_n once per flush.
//
// Plan (N == 16): the sequence is cut into units of TU steps.
//   1. states entering every unit -> hin[k]: the forward pass's checkpoints
//      when the caller has them (ssm_scan_bwd_ckpt); else, when the chains
//      fill the GPU, the chained forward scan writing them as it goes; else
//      the forward kernel's unit summaries and carry (scan_tile.cuh,
//      kAggregate + carry_kernel);
//   2. adjoint summaries: each unit, walked backward from lam = 0, gives
//      Q_k = Abar_{t0} lam_{t0} and sum(dl); adj_carry_kernel combines them
//      from the last unit down into mu[k], the adjoint entering unit k at its
//      end (mu[P-1] = dh_last);
//   3. bwd_unit_kernel: per unit, the unit's inputs come into shared memory
//      by cp.async; a forward sweep from hin[k] stores the states at the
//      start of each KS-step sub-chunk in TMEM (16 columns per start, each
//      thread in its own lane); then, sub-chunk by sub-chunk from the last,
//      the states of the sub-chunk are recomputed into shared memory and
//      walked backward from mu[k].  dB and dC are summed over the warp's 32
//      channels by a butterfly of shuffles and over the CTA's 128 channels in
//      shared memory, then written as one partial per 128-channel block;
//   4. bwd_reduce_bc_kernel sums the partials over the blocks.
// Threads: one channel per thread, 128 channels (4 warps) per CTA; three
// CTAs share an SM (74 KB of shared memory and 128 TMEM columns each).
#pragma once

#include "common.cuh"
#include "ptx.cuh"
#include "tmem.cuh"

namespace ssm {
namespace bwd {

constexpr int NS = 16;
constexpr int CB = 128;       // channels per CTA, one per thread
constexpr int NW = CB / 32;   // warps per CTA
constexpr int TU = 32;        // steps per unit (the checkpoint interval)
constexpr int KS = 4;         // steps per recomputed sub-chunk
constexpr int NSUB = TU / KS;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct BwdParams {
    const void* u;
    const void* delta;
    const void* z;
    const void* dy;
    const void* Bm;
    const void* Cm;
    const float* dt_bias;
    const float* A;
    const float* Dskip;
    const float* dh_last;
    void* du;
    void* ddelta;
    void* dz;
    float* ddt_bias;
    float* dA;
    float* dDskip;
    float* part;       // [nCB][batch][L][32]: dC (0..15), (n+1) dB (16..31), per block
    const float* hin;  // [P][batch*D][NS]: the state entering unit k
    float* adj;        // [P][batch*D][NS+1]: {sum dl, Q_k} (k >= 1)
    float* mu;         // [P][batch*D][NS]: the adjoint entering unit k at its end
    long long batch, L, D, P, nCB, units;
};

__device__ __forceinline__ float ldf(const float* p) { return *p; }
__device__ __forceinline__ float ldf(const bf16* p) { return __bfloat162float(*p); }

// dl = log2(1 + 2^v2) = softplus(v) / ln 2 with v2 = v log2(e); v2 itself
// above 28.85 (v > 20), where the two agree to float32 precision.
__device__ __forceinline__ float softplus_l2(float v2) {
    return v2 > 28.853901f ? v2 : ptx::lg2(1.0f + ptx::ex2(v2));
}

// sigmoid(v) = 1 / (1 + 2^(-v2)), accurate at both tails.
__device__ __forceinline__ float sigmoid_l2(float v2) {
    return ptx::rcp(1.0f + ptx::ex2(-v2));
}

// psi(x) = (e^x - 1 - x) / x^2, given em1 = e^x - 1: a Taylor series below
// |x| = 1/4 (truncation below 1e-8 relative), the closed form above.
__device__ __forceinline__ float psi_of(float x, float em1) {
    if (fabsf(x) < 0.25f)
        return fmaf(x, fmaf(x, fmaf(x, fmaf(x, fmaf(x, 1.0f / 5040.0f, 1.0f / 720.0f),
                                               1.0f / 120.0f), 1.0f / 24.0f), 1.0f / 6.0f), 0.5f);
    return (em1 - x) / (x * x);
}

// Per-channel constants of the unit.
struct Chan {
    float a0, ia0, kb2, dsk;   // A[d,0], 1/A[d,0], dt_bias log2(e), Dskip
    bool geo;                  // the warp's rows are all (n+1) a0 with |a0| >= 1/16
};

__device__ __forceinline__ Chan load_chan(const BwdParams& p, long long d, bool valid,
                                          float (&arow)[NS]) {
    Chan c;
    const long long ds = valid ? d : 0;
    const float4* a4 = reinterpret_cast<const float4*>(p.A + ds * NS);
#pragma unroll
    for (int q = 0; q < NS / 4; ++q) {
        const float4 v = __ldg(a4 + q);
        arow[4 * q] = v.x;
        arow[4 * q + 1] = v.y;
        arow[4 * q + 2] = v.z;
        arow[4 * q + 3] = v.w;
    }
    bool g = fabsf(arow[0]) >= 0.0625f && isfinite(arow[0]);
#pragma unroll
    for (int n = 1; n < NS; ++n) g = g && (arow[n] == (float)(n + 1) * arow[0]);
    c.geo = __all_sync(0xffffffffu, g || !valid);
    if (!valid) {   // a harmless geometric row; every input of the lane is 0
#pragma unroll
        for (int n = 0; n < NS; ++n) arow[n] = -(float)(n + 1);
    }
    c.a0 = arow[0];
    c.ia0 = arow[0] != 0.0f ? 1.0f / arow[0] : 0.0f;
    c.kb2 = (p.dt_bias && valid) ? __ldg(p.dt_bias + d) * kLog2e : 0.0f;
    c.dsk = (p.Dskip && valid) ? __ldg(p.Dskip + d) : 0.0f;
    return c;
}

// Unit index -> (block, batch entry, unit within the chain); units are
// block-major so that a CTA's consecutive units share their channels.
struct Unit {
    long long cb, b, k, t0, t1;
};

__device__ __forceinline__ Unit unit_of(const BwdParams& p, long long i) {
    Unit w;
    const long long per_cb = p.batch * p.P;
    w.cb = i / per_cb;
    const long long r = i - w.cb * per_cb;
    w.b = r / p.P;
    w.k = r - w.b * p.P;
    w.t0 = w.k * TU;
    w.t1 = w.t0 + TU < p.L ? w.t0 + TU : p.L;
    return w;
}

// B and C rows of the unit's steps, widened to float32 in shared memory;
// Bs holds B, Bp holds B / (n+1).
template <typename T>
__device__ __forceinline__ void load_rows(const BwdParams& p, const Unit& w, float* Bs, float* Bp,
                                          float* Cs, bool needB) {
    const T* Bg = static_cast<const T*>(p.Bm) + (w.b * p.L + w.t0) * NS;
    const T* Cg = static_cast<const T*>(p.Cm) + (w.b * p.L + w.t0) * NS;
    const int cnt = (int)(w.t1 - w.t0) * NS;
    for (int i = threadIdx.x; i < TU * NS; i += CB) {
        const bool in = i < cnt;
        if (needB) {
            const float bv = in ? ldf(Bg + i) : 0.0f;
            Bs[i] = bv;
            Bp[i] = bv * (1.0f / (float)((i % NS) + 1));
        }
        Cs[i] = in ? ldf(Cg + i) : 0.0f;
    }
}

// ------------------------------------------------------------ phase 2
// Adjoint summary of each unit k >= 1, walked backward from lam = 0:
// adj[k] = {sum dl, Abar_{t0} lam_{t0}}.
//
// A CTA takes its units as a list of half-unit stages (the steps HS..TU-1 of
// a unit, then 0..HS-1).  While one stage computes, the next one's delta, dy
// and z rows are copied into the other shared buffer by cp.async and its C
// rows come into registers, to be widened into the other C buffer when the
// stage ends; the loads of a stage are thus in flight during a whole stage of
// arithmetic, at no cost in registers.
constexpr int HS = TU / 2;   // steps per stage

template <typename T>
struct AdjSmem {
    T dv[2][HS][CB], dy[2][HS][CB], z[2][HS][CB];
    float Cs[2][HS * NS];
};

// 16-byte global -> shared copy, zero-filled (nothing read) when !ok.
__device__ __forceinline__ void cpa16(void* dst, const void* src, bool ok) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(ptx::smem_u32(dst)),
                 "l"(src), "r"(ok ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cpa_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// every group but the newest one complete (this thread's copies)
__device__ __forceinline__ void cpa_wait_prior() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
// every group of this thread complete
__device__ __forceinline__ void cpa_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Unit of index i in the list of units with k >= 1.
__device__ __forceinline__ Unit adj_unit(const BwdParams& p, long long i) {
    const long long cbb = i / (p.P - 1);
    return unit_of(p, cbb * p.P + 1 + (i - cbb * (p.P - 1)));
}

// Issues stage (w, h) into buffer s: its rows t0 + h*HS .. min(t1, +HS) - 1,
// channels cb*CB .. +CB-1 (16-byte pieces past D or past the rows are
// zero-filled; D is a multiple of the piece), and loads its C rows into cpre.
template <typename T>
__device__ __forceinline__ void adj_issue(const BwdParams& p, const Unit& w, int h,
                                          AdjSmem<T>& sm, int s, float (&cpre)[2]) {
    constexpr int EPP = 16 / (int)sizeof(T);   // elements per 16-byte piece
    constexpr int CPR = CB / EPP;              // pieces per row
    const long long ta = w.t0 + (long long)h * HS;
    const long long rows = w.t1 - ta < HS ? w.t1 - ta : HS;
    const long long d0 = w.cb * CB;
    const long long base = (w.b * p.L + ta) * p.D + d0;
    const T* dv = static_cast<const T*>(p.delta);
    const T* dy = static_cast<const T*>(p.dy);
    const T* z = static_cast<const T*>(p.z);
    for (int q = threadIdx.x; q < HS * CPR; q += CB) {
        const int r = q / CPR, c = q - r * CPR;
        const bool ok = r < rows && d0 + c * EPP < p.D;
        const long long off = ok ? base + r * p.D + c * EPP : 0;
        cpa16(&sm.dv[s][r][c * EPP], dv + off, ok);
        cpa16(&sm.dy[s][r][c * EPP], dy + off, ok);
        if (z) cpa16(&sm.z[s][r][c * EPP], z + off, ok);
    }
    const T* Cg = static_cast<const T*>(p.Cm) + (w.b * p.L + ta) * NS;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int e = threadIdx.x + k * CB;
        cpre[k] = e < rows * NS ? ldf(Cg + e) : 0.0f;
    }
}

template <typename T>
__global__ void __launch_bounds__(CB)
adjoint_summary_kernel(const BwdParams p) {
    static_assert(HS * NS == 2 * CB, "two C values per thread and stage");
    extern __shared__ __align__(16) unsigned char adj_smem_raw[];
    AdjSmem<T>& sm = *reinterpret_cast<AdjSmem<T>*>(adj_smem_raw);
    const long long G = gridDim.x;
    const long long nsum = p.nCB * p.batch * (p.P - 1);
    const long long r0 = blockIdx.x * nsum / G, r1 = (blockIdx.x + 1) * nsum / G;
    if (r0 >= r1) return;
    const bool hasz = p.z != nullptr;
    // stage being computed: unit i (w), half h, buffer s
    long long i = r0;
    Unit w = adj_unit(p, r0);
    int h = (int)((w.t1 - w.t0 - 1) / HS);
    int s = 0;
    float cpre[2];
    adj_issue<T>(p, w, h, sm, 0, cpre);
    cpa_commit();
    sm.Cs[0][threadIdx.x] = cpre[0];
    sm.Cs[0][threadIdx.x + CB] = cpre[1];
    // a CTA's units are consecutive and mostly share their channel block: its
    // A rows and parameters are loaded again only when the block changes
    long long cur_cb = -1;
    long long d = 0;
    bool valid = false;
    float arow[NS];
    Chan c{};
    float lam[NS];
#pragma unroll
    for (int n = 0; n < NS; ++n) lam[n] = 0.0f;
    float S2 = 0.0f;
    for (;;) {
        // the next stage, issued before this one computes
        long long ni = i;
        Unit nw = w;
        int nh = h - 1;
        if (nh < 0) {
            ni = i + 1;
            if (ni < r1) {
                nw = adj_unit(p, ni);
                nh = (int)((nw.t1 - nw.t0 - 1) / HS);
            }
        }
        const bool more = ni < r1;
        if (more) adj_issue<T>(p, nw, nh, sm, s ^ 1, cpre);
        cpa_commit();
        if (w.cb != cur_cb) {
            cur_cb = w.cb;
            d = w.cb * CB + threadIdx.x;
            valid = d < p.D;
            c = load_chan(p, d, valid, arow);
        }
        cpa_wait_prior();
        __syncthreads();
        const long long ta = w.t0 + (long long)h * HS;
        const int rows = (int)(w.t1 - ta < HS ? w.t1 - ta : HS);
#pragma unroll
        for (int j = HS - 1; j >= 0; --j) {
            if (j >= rows) continue;
            float g = 1.0f;
            if (hasz) {
                const float zj = ldf(&sm.z[s][j][threadIdx.x]);
                g = zj * ptx::rcp(1.0f + ptx::ex2(-zj * kLog2e));
            }
            const float ds = ldf(&sm.dy[s][j][threadIdx.x]) * g;
            const float dl = softplus_l2(fmaf(ldf(&sm.dv[s][j][threadIdx.x]), kLog2e, c.kb2));
            S2 += dl;
            const float* Ct = sm.Cs[s] + j * NS;
            if (c.geo) {
                const float e0 = em1_near0(dl * c.a0 * kLn2, ptx::ex2(dl * c.a0));
                const float r = e0 + 1.0f;
                const float e1 = fmaf(r, e0, e0), r2 = e1 + 1.0f;
                float ea = e0, eb = e1;
#pragma unroll
                for (int n = 0; n < NS; n += 2) {
                    if (n > 0) {
                        ea = fmaf(r2, ea, e1);
                        eb = fmaf(r2, eb, e1);
                    }
                    lam[n] = fmaf(ds, Ct[n], lam[n]);
                    lam[n] = fmaf(ea, lam[n], lam[n]);
                    lam[n + 1] = fmaf(ds, Ct[n + 1], lam[n + 1]);
                    lam[n + 1] = fmaf(eb, lam[n + 1], lam[n + 1]);
                }
            } else {
#pragma unroll
                for (int n = 0; n < NS; ++n) {
                    lam[n] = fmaf(ds, Ct[n], lam[n]);
                    lam[n] *= ptx::ex2(dl * arow[n]);
                }
            }
        }
        if (h == 0) {   // the unit is done
            if (valid) {
                float* o = p.adj + (w.k * p.batch * p.D + w.b * p.D + d) * (NS + 1);
                o[0] = S2;
#pragma unroll
                for (int n = 0; n < NS; ++n) o[1 + n] = lam[n];
            }
#pragma unroll
            for (int n = 0; n < NS; ++n) lam[n] = 0.0f;
            S2 = 0.0f;
        }
        if (more) {
            sm.Cs[s ^ 1][threadIdx.x] = cpre[0];
            sm.Cs[s ^ 1][threadIdx.x + CB] = cpre[1];
        }
        __syncthreads();   // buffer s is free for the stage after next
        if (!more) break;
        i = ni;
        w = nw;
        h = nh;
        s ^= 1;
    }
}

// mu[P-1] = dh_last (or 0); mu[k-1] = Q_k + 2^(a sum dl_k) mu[k].
__global__ void adj_carry_kernel(const float* __restrict__ adj, const float* __restrict__ A,
                                 const float* __restrict__ dh_last, float* __restrict__ mu,
                                 long long batch, long long D, long long P) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long nch = batch * D;
    if (i >= nch * NS) return;
    const long long ch = i / NS, n = i % NS, d = ch % D;
    const float a = A[d * NS + n];
    float m = dh_last ? dh_last[ch * NS + n] : 0.0f;
    for (long long k = P - 1; k >= 0; --k) {
        mu[(k * nch + ch) * NS + n] = m;
        if (k > 0) {
            const float* g = adj + (k * nch + ch) * (NS + 1);
            m = fmaf(exp2f(a * g[0]), m, g[1 + n]);
        }
    }
}

// ------------------------------------------------------------ phase 3
// 32 values per lane (v[0..15] dC, v[16..31] dB) summed over the warp's 32
// lanes by a butterfly: at each stage a lane keeps one half of its values
// and adds the partner's copy of that half, so after five stages lane l holds
// the warp sum of value l.
__device__ __forceinline__ float warp_reduce32(float (&v)[32], int lane) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const bool up = lane & 16;
        const float send = up ? v[i] : v[i + 16];
        const float keep = up ? v[i + 16] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const bool up = lane & 8;
        const float send = up ? v[i] : v[i + 8];
        const float keep = up ? v[i + 8] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const bool up = lane & 4;
        const float send = up ? v[i] : v[i + 4];
        const float keep = up ? v[i + 4] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const bool up = lane & 2;
        const float send = up ? v[i] : v[i + 2];
        const float keep = up ? v[i + 2] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
    }
    {
        const bool up = lane & 1;
        const float send = up ? v[0] : v[1];
        const float keep = up ? v[1] : v[0];
        v[0] = keep + __shfl_xor_sync(0xffffffffu, send, 1);
    }
    return v[0];
}

template <typename T>
struct BwdSmem {
    T in[4][TU][CB];                   // u, delta, z, dy of the unit
    float4 hist[KS][NS / 4][CB];       // h_t of the sub-chunk walked back
    float red[KS][NW][32];             // per-warp dB/dC sums
    float Bs[TU * NS], Bp[TU * NS], Cs[TU * NS];
    uint32_t tmem;                     // TMEM base: the state at each sub-chunk start
};

// The unit's u, delta, z and dy (rows t0 .. t1 - 1, channels cb*CB .. +CB-1)
// into shared memory, 16-byte pieces by cp.async (zero-filled, nothing read,
// past D or past the unit's end; D is a multiple of the piece).
template <typename T>
__device__ __forceinline__ void bwd_issue(const BwdParams& p, const Unit& w, BwdSmem<T>& sm) {
    constexpr int EPP = 16 / (int)sizeof(T);   // elements per 16-byte piece
    constexpr int CPR = CB / EPP;              // pieces per row
    const long long rows = w.t1 - w.t0;
    const long long d0 = w.cb * CB;
    const long long base = (w.b * p.L + w.t0) * p.D + d0;
    const T* src[4] = {static_cast<const T*>(p.u), static_cast<const T*>(p.delta),
                       static_cast<const T*>(p.z), static_cast<const T*>(p.dy)};
    for (int q = threadIdx.x; q < TU * CPR; q += CB) {
        const int r = q / CPR, c = q - r * CPR;
        const bool ok = r < rows && d0 + c * EPP < p.D;
        const long long off = ok ? base + r * p.D + c * EPP : 0;
#pragma unroll
        for (int a = 0; a < 4; ++a)
            if (src[a]) cpa16(&sm.in[a][r][c * EPP], src[a] + off, ok);
    }
}

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(bf16 x) { return __bfloat162float(x); }

// One forward step (the forward kernel's arithmetic): h <- Abar h + q B u.
__device__ __forceinline__ void fwd_step(float (&h)[NS], const Chan& c, const float (&arow)[NS],
                                         float u, float dl, const float* Bt, const float* Bpt) {
    if (c.geo) {
        const float e0 = em1_near0(dl * c.a0 * kLn2, ptx::ex2(dl * c.a0));
        const float r = e0 + 1.0f;
        const float e1 = fmaf(r, e0, e0), r2 = e1 + 1.0f;
        const float up = u * c.ia0;
        float2 E = make_float2(e0, e1);
        const float2 R2 = make_float2(r2, r2), E1 = make_float2(e1, e1), UP = make_float2(up, up);
#pragma unroll
        for (int n = 0; n < NS; n += 2) {
            if (n > 0) E = __ffma2_rn(R2, E, E1);
            float2 H = make_float2(h[n], h[n + 1]);
            const float2 Bv = make_float2(Bpt[n], Bpt[n + 1]);
            H = __ffma2_rn(E, __ffma2_rn(Bv, UP, H), H);
            h[n] = H.x;
            h[n + 1] = H.y;
        }
    } else {
        const float dt = dl * kLn2;
#pragma unroll
        for (int n = 0; n < NS; ++n) {
            const float a = arow[n];
            const float e = em1_near0(dl * a * kLn2, ptx::ex2(dl * a));
            const float q = (a != 0.0f) ? e / a : dt;
            h[n] = fmaf(q * Bt[n], u, fmaf(e, h[n], h[n]));
        }
    }
}

template <typename T>
__global__ void __launch_bounds__(CB, 3)
bwd_unit_kernel(const BwdParams p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    BwdSmem<T>& sm = *reinterpret_cast<BwdSmem<T>*>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const long long G = gridDim.x;
    const long long r0 = blockIdx.x * p.units / G, r1 = (blockIdx.x + 1) * p.units / G;
    const long long nch = p.batch * p.D;

    // TMEM: 128 columns, the states at the NSUB sub-chunk starts (16 columns
    // each); warp w's threads own lanes 32 w .. 32 w + 31
    if (warp == 0) tmem::alloc(&sm.tmem, 128);
    tmem::fence_before_sync();
    __syncthreads();
    tmem::fence_after_sync();
    const uint32_t tbase = sm.tmem + ((uint32_t)(32 * warp) << 16);

    long long cur_cb = -1;
    float dacc[NS];            // dA accumulator of the channel (see the header)
    float dsk_acc = 0.0f, dtb_acc = 0.0f;
    float arow[NS];
    Chan c{};
    long long d = 0;
    bool valid = false;
#pragma unroll
    for (int n = 0; n < NS; ++n) dacc[n] = 0.0f;

    auto flush = [&]() {
        if (cur_cb >= 0 && valid) {
#pragma unroll
            for (int n = 0; n < NS; ++n) {
                const float v = c.geo ? dacc[n] / arow[n] : dacc[n];
                atomicAdd(p.dA + d * NS + n, v);
            }
            if (p.dDskip) atomicAdd(p.dDskip + d, dsk_acc);
            if (p.ddt_bias) atomicAdd(p.ddt_bias + d, dtb_acc);
        }
#pragma unroll
        for (int n = 0; n < NS; ++n) dacc[n] = 0.0f;
        dsk_acc = 0.0f;
        dtb_acc = 0.0f;
    };

    for (long long i = r0; i < r1; ++i) {
        const Unit w = unit_of(p, i);
        if (w.cb != cur_cb) {
            flush();
            cur_cb = w.cb;
            d = w.cb * CB + tid;
            valid = d < p.D;
            c = load_chan(p, d, valid, arow);
        }
        __syncthreads();   // the previous unit is done with the rows and inputs
        bwd_issue<T>(p, w, sm);
        cpa_commit();
        load_rows<T>(p, w, sm.Bs, sm.Bp, sm.Cs, true);
        cpa_wait_all();
        __syncthreads();

        const long long base = w.b * p.L * p.D + (valid ? d : 0);
        const bool zsrc = p.z != nullptr;
        const long long ch = w.b * p.D + (valid ? d : 0);
        const int nsteps = (int)(w.t1 - w.t0);
        const int s_last = (nsteps - 1) / KS;

        // sweep 1: the states at the sub-chunk starts, into TMEM
        float h[NS];
        {
            const float4* hs = reinterpret_cast<const float4*>(p.hin + (w.k * nch + ch) * NS);
#pragma unroll
            for (int q = 0; q < NS / 4; ++q) {
                const float4 v = (valid && w.k > 0) ? __ldcg(hs + q) : make_float4(0.f, 0.f, 0.f, 0.f);
                h[4 * q] = v.x;
                h[4 * q + 1] = v.y;
                h[4 * q + 2] = v.z;
                h[4 * q + 3] = v.w;
            }
        }
        for (int s = 0; s < s_last; ++s) {
            tmem::st16(tbase + (uint32_t)(NS * s), h);
#pragma unroll
            for (int j = 0; j < KS; ++j) {
                const int tt = s * KS + j;
                fwd_step(h, c, arow, to_f(sm.in[0][tt][tid]),
                         softplus_l2(fmaf(to_f(sm.in[1][tt][tid]), kLog2e, c.kb2)),
                         sm.Bs + tt * NS, sm.Bp + tt * NS);
            }
        }
        tmem::st16(tbase + (uint32_t)(NS * s_last), h);
        tmem::wait_st();

        // the adjoint entering the unit at its end
        float lam[NS];
        {
            const float4* ms = reinterpret_cast<const float4*>(p.mu + (w.k * nch + ch) * NS);
#pragma unroll
            for (int q = 0; q < NS / 4; ++q) {
                const float4 v = valid ? __ldcg(ms + q) : make_float4(0.f, 0.f, 0.f, 0.f);
                lam[4 * q] = v.x;
                lam[4 * q + 1] = v.y;
                lam[4 * q + 2] = v.z;
                lam[4 * q + 3] = v.w;
            }
        }

        // sweep 2: sub-chunks from the last, each recomputed into shared
        // memory from its start state, then walked back
        for (int s = s_last; s >= 0; --s) {
            const int tb = s * KS;
            const int cnt = nsteps - tb < KS ? nsteps - tb : KS;
            tmem::ld16(tbase + (uint32_t)(NS * s), h);
            tmem::wait_ld();
            float dlj[KS];
#pragma unroll
            for (int j = 0; j < KS; ++j)
                dlj[j] = j < cnt ? softplus_l2(fmaf(to_f(sm.in[1][tb + j][tid]), kLog2e, c.kb2))
                                 : 0.0f;
#pragma unroll
            for (int j = 0; j < KS; ++j) {
                if (j < cnt) {   // uniform over the CTA
                    fwd_step(h, c, arow, to_f(sm.in[0][tb + j][tid]), dlj[j],
                             sm.Bs + (tb + j) * NS, sm.Bp + (tb + j) * NS);
#pragma unroll
                    for (int q = 0; q < NS / 4; ++q)
                        sm.hist[j][q][tid] = make_float4(h[4 * q], h[4 * q + 1], h[4 * q + 2], h[4 * q + 3]);
                }
            }
#pragma unroll
            for (int j = KS - 1; j >= 0; --j) {
                if (j >= cnt) continue;   // uniform over the CTA
                const int tt = tb + j;
                const long long t = w.t0 + tt;
                const float* Bt = sm.Bs + tt * NS;
                const float* Bpt = sm.Bp + tt * NS;
                const float* Ct = sm.Cs + tt * NS;
                const float u = to_f(sm.in[0][tb + j][tid]), dl = dlj[j], dt = dl * kLn2;
                const float zjj = zsrc ? to_f(sm.in[2][tb + j][tid]) : 0.0f;
                const float dyjj = to_f(sm.in[3][tb + j][tid]);
                const float vjj = fmaf(to_f(sm.in[1][tb + j][tid]), kLog2e, c.kb2);
                float g = 1.0f, sg = 0.0f;
                if (zsrc) {
                    sg = ptx::rcp(1.0f + ptx::ex2(-zjj * kLog2e));
                    g = zjj * sg;
                }
                const float ds = dyjj * g;
                float hv[NS];
#pragma unroll
                for (int q = 0; q < NS / 4; ++q) {
                    const float4 v = sm.hist[j][q][tid];
                    hv[4 * q] = v.x;
                    hv[4 * q + 1] = v.y;
                    hv[4 * q + 2] = v.z;
                    hv[4 * q + 3] = v.w;
                }
                float red[32];
                float sacc = c.dsk * u, ddt = 0.0f, vsum = 0.0f;
                if (c.geo) {
                    const float e0 = em1_near0(dl * c.a0 * kLn2, ptx::ex2(dl * c.a0));
                    const float r = e0 + 1.0f;
                    const float e1 = fmaf(r, e0, e0), r2 = e1 + 1.0f;
                    const float uia = u * c.ia0;
                    float ea = e0, eb = e1;
#pragma unroll
                    for (int n = 0; n < NS; ++n) {
                        if (n >= 2) {
                            if (n & 1) eb = fmaf(r2, eb, e1);
                            else ea = fmaf(r2, ea, e1);
                        }
                        const float e = (n & 1) ? eb : ea;
                        const float hn = hv[n];
                        sacc = fmaf(Ct[n], hn, sacc);
                        const float lm = fmaf(ds, Ct[n], lam[n]);
                        red[n] = ds * hn;
                        const float tn = lm * fmaf(arow[n], hn, Bt[n] * u);
                        ddt += tn;
                        const float le = lm * e;
                        const float v = le * Bpt[n];
                        vsum += v;
                        dacc[n] = fmaf(-uia, v, fmaf(dt, tn, dacc[n]));
                        red[16 + n] = le * uia;
                        lam[n] = lm + le;
                    }
                } else {
#pragma unroll
                    for (int n = 0; n < NS; ++n) {
                        const float a = arow[n];
                        const float x = dt * a;
                        const float ab = ptx::ex2(dl * a);
                        const float e = em1_near0(x, ab);
                        const float q = (a != 0.0f) ? e / a : dt;
                        const float hn = hv[n];
                        const float bu = Bt[n] * u;
                        sacc = fmaf(Ct[n], hn, sacc);
                        const float lm = fmaf(ds, Ct[n], lam[n]);
                        red[n] = ds * hn;
                        ddt = fmaf(lm, fmaf(a, hn, bu), ddt);
                        vsum = fmaf(lm * q, Bt[n], vsum);
                        dacc[n] = fmaf(lm * dt, fmaf(-dt * bu, psi_of(x, e), hn), dacc[n]);
                        red[16 + n] = lm * q * u * (float)(n + 1);
                        lam[n] = lm * ab;
                    }
                }
                const float du = fmaf(ds, c.dsk, c.geo ? vsum * c.ia0 : vsum);
                const float dd = ddt * sigmoid_l2(vjj);
                dsk_acc = fmaf(ds, u, dsk_acc);
                dtb_acc += dd;
                if (valid) {
                    const long long o = base + t * p.D;
                    static_cast<T*>(p.du)[o] = from_f32<T>(du);
                    static_cast<T*>(p.ddelta)[o] = from_f32<T>(dd);
                    if (zsrc) {
                        const float dzv = dyjj * sacc * sg * fmaf(zjj, 1.0f - sg, 1.0f);
                        static_cast<T*>(p.dz)[o] = from_f32<T>(dzv);
                    }
                }
                sm.red[j][warp][lane] = warp_reduce32(red, lane);
            }
            __syncthreads();
            // per-block dB/dC sums of the sub-chunk's steps
            for (int e = tid; e < KS * 32; e += CB) {
                const int j = e >> 5, l = e & 31;
                if (j < cnt) {
                    float sum = 0.0f;
#pragma unroll
                    for (int ww = 0; ww < NW; ++ww) sum += sm.red[j][ww][l];
                    p.part[((w.cb * p.batch + w.b) * p.L + w.t0 + tb + j) * 32 + l] = sum;
                }
            }
            __syncthreads();
        }
    }
    flush();
    tmem::fence_before_sync();
    __syncthreads();
    tmem::fence_after_sync();
    if (warp == 0) tmem::dealloc(sm.tmem, 128);
}

// dC[b,t,n] = sum over blocks of part[..][n]; dB[b,t,n] = that of part[..][16+n] / (n+1).
__global__ void bwd_reduce_bc_kernel(const float* __restrict__ part, float* __restrict__ dB,
                                     float* __restrict__ dC, long long rows, long long nCB) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= rows * 32) return;
    const long long row = i >> 5;
    const int l = (int)(i & 31);
    float s = 0.0f;
    for (long long cb = 0; cb < nCB; ++cb) s += part[(cb * rows + row) * 32 + l];
    if (l < NS) {
        if (dC) dC[row * NS + l] = s;
    } else {
        if (dB) dB[row * NS + (l - NS)] = s * (1.0f / (float)(l - NS + 1));
    }
}

}  // namespace bwd
}  // namespace ssm
