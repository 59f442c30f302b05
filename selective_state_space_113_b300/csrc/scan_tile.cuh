// scan_tile.cuh -- the sm_103a selective-scan kernel for N == 16.
//
// What it computes is the selective scan of the pages on Mamba (ta-paperlens
// "Mamba: 状態を「選択的」にする" pseudocode; ultralytics "SSMの仕組み" zero-order
// hold; the output equation y = C h + D x of news.han.ihouse.idv.tw article
// 1304; the SiLU(z) gate of the agenticai-flow Mamba block diagram), in
// float32 with a float32 state.
//
// Work decomposition.  A chain is one 128-channel block of one batch entry
// along the whole sequence; a piece is a run of consecutive stages of one
// chain, the work of one CTA tile.  CTAs are persistent (one per SM).  A CTA
// has nine warps with fixed roles:
//   warp 8      TMA warp: walks the CTA's pieces, loads each piece's per-channel
//               parameters and carried state into shared memory, and streams
//               the unit's u, delta, z, B and C in stages of TC steps by TMA
//               (one 128-channel box per tensor and stage).
//   warps 4..7  helpers: widen a quarter of each stage's B and C rows to
//               float32, then compute, for their consumer's 32 channels, the
//               per-step values that do not depend on the state (softplus,
//               exp(dt a0), the SiLU gate) in chunks of KP steps.
//   warps 0..3  consumers: one channel per lane, all 16 states in registers;
//               the recurrence and the readout.  y goes through a shared
//               memory tile that is written back by a TMA bulk store.
// Warp w runs on SM sub-partition w % 4, so each sub-partition holds one
// consumer (FMA-bound) next to its helper (SFU-bound).
//
// Three plans and the backward's first phase use this kernel:
//   kChained   -- a static split: the chain-major space of (chain, stage) is
//                 cut into one equal contiguous range per CTA, and each CTA
//                 walks its range from the last chain to the first.  A chain
//                 cut between CTAs i-1 and i is then the first piece CTA i-1
//                 runs and the last piece CTA i runs, so the state CTA i needs
//                 (passed through global memory with release/acquire flags;
//                 bounded waits, done by the TMA warp while it prefetches) is
//                 ready long before it is wanted.  Used when the chains fill
//                 the GPU.
//   kAggregate -- phase 1 of the narrow-problem plan: chains are cut into P
//                 units of T steps taken from an atomic ticket; each runs from a
//                 zero state and records sum(log2-domain dt) and its final
//                 state (the unit's affine summary; no y is written).
//   kFromState -- phase 3: each unit starts from a state computed by the carry
//                 kernel (phase 2) from the phase-1 summaries, and writes y.
//   kCkptOnly  -- kChained's walk that writes only the states entering each
//                 32-step unit (the backward pass's checkpoints): no C or z
//                 copies, no readout, no y.
//
// Per-step arithmetic (geometric A, A[d,n] = (n+1) a0, detected per warp):
//   v2 = delta*log2(e) + dt_bias*log2(e);  x = 2^v2 = e^(delta+bias)
//   dl = log2(1 + x)                          (dt = dl * ln2 = softplus)
//   r  = 2^(dl a0) = exp(dt a0);  e_n = r^(n+1) - 1 = exp(dt A[d,n]) - 1
//        e_0 = r - 1, e_1 = r e_0 + e_0, e_(n+2) = r^2 e_n + e_1
//   (r - 1 carries the SFU's absolute error, about 2^-22, so e_0 is good to
//   about 2^-22 / |dt a0| relative; rows with |a0| < 1/16 therefore take the
//   per-state path, which forms exp(x) - 1 from its Taylor polynomial near 0)
//   h_n <- h_n + e_n (h_n + B_n u / A[d,n])  (= A_bar h + (A_bar - 1)/A B u)
//   y  = (sum_n C_n h_n + Dskip u) * z / (1 + 2^(-z log2(e)))
// B_n/(n+1) is prepared once per stage by the helpers, and u/a0 once per
// step, so B_n u / A[d,n] is one multiply-add away.  Any other A runs a
// per-state path that uses exp(dt A) - 1 directly and the dt*B limit at A = 0.
//
// Discretisation variants of the input term (template parameter DISC; the
// decay A_bar = exp(dt A) is common):
//   kZOH    (A_bar - 1)/A B_t u_t                       (above)
//   kEuler  dt B_t u_t  (ta-paperlens pseudocode):   h <- e (h) + (h + dt u B)
//   kTrap   dt/2 (B_t u_t + A_bar B_{t-1} u_{t-1})  (news.han.ihouse.idv.tw,
//           Mamba-3 "台形法則", weight 1/2):  s = h + dt/2 P_{t-1},
//           h <- A_bar s + dt/2 P_t with P_t = B_t u_t kept per state; a
//           piece's first step takes P from the step before it (header).
// For kEuler and kTrap the helpers widen B without the 1/(n+1) scale.
//
// CONV: the input is x, and u is the short causal convolution in front of the
// SSM (ta-paperlens "現場ではこう使う": d_conv; agenticai-flow: d_conv=4,
// causal-conv1d), depthwise, width 4, optional SiLU:
//     u_t = act(conv_b[d] + sum_k conv_w[d, k] x_{t-3+k}).
// Only the helpers change: they read x from the stage tile, keep x_{t-1..t-3}
// of their channel in registers, and load the weights and the three x values
// before a piece when the piece starts.
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "ptx.cuh"

namespace ssm {
namespace tile {

constexpr int NS = 16;              // state size handled here
constexpr int CW = 32;              // channels per consumer warp (one per lane)
constexpr int NCW = 4;              // consumer warps per CTA
constexpr int CB = CW * NCW;        // channels per CTA tile
#ifndef SSM_TILE_STAGES
#define SSM_TILE_STAGES 4
#endif
#ifndef SSM_TILE_KP
#define SSM_TILE_KP 8
#endif
#ifndef SSM_TILE_NPB
#define SSM_TILE_NPB 2
#endif
constexpr int S = SSM_TILE_STAGES;  // stages in the shared-memory ring
constexpr int KP = SSM_TILE_KP;     // steps per prologue chunk
constexpr int NPB = SSM_TILE_NPB;   // prologue buffers per helper/consumer pair
constexpr int NWARPS = 2 * NCW + 1; // consumers, helpers, TMA warp
constexpr int THREADS = 32 * NWARPS;
constexpr int kTmaWarp = 2 * NCW;
constexpr unsigned kSleepNs = 64;   // back-off of the TMA warp's waits

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// kCkptOnly: the chained walk that writes only the state checkpoints (no C,
// z, readout or y), the backward pass's first phase.
enum Mode : int { kChained = 0, kAggregate = 1, kFromState = 2, kCkptOnly = 3 };

// Whether a mode forms y (and so reads C and z), and whether it walks whole
// chains with its predecessor's state.
__host__ __device__ constexpr bool forms_y(int mode) { return mode == kChained || mode == kFromState; }
__host__ __device__ constexpr bool walks_chains(int mode) { return mode == kChained || mode == kCkptOnly; }

// Steps per unit of the optional state checkpoints (the backward pass's unit).
constexpr long long kCkptSteps = 32;

enum Disc : int { kZOH = 0, kEuler = 1, kTrap = 2 };

// Stage flags: first / last stage of a piece, end of work, carried state
// present in the stage header, piece ends at the end of its chain.
enum MetaFlags : int { kFirst = 1, kLast = 2, kEnd = 4, kHasState = 8, kChainEnd = 16 };

struct Meta {
    long long chain;
    long long t0;
    int nvalid;   // valid steps in the stage (< TC only at the sequence end)
    int flags;
    int geo;      // bit w: consumer warp w's 32 channels have a geometric A row
    int piece;    // index of the piece within its chain (the unit index k)
};

// Per-channel unit parameters, written by the TMA warp into the header of a
// unit's first stage.
struct ChanPar {
    float a0, ia0, kb2, dsk;   // A[d,0], 1/A[d,0], dt_bias*log2(e), Dskip[d]
};

struct Params {
    void* y;
    float* h_last;
    const void* u;          // raw u (x with CONV) and B: the steps before a piece
    const void* Bm;
    const float* conv_w;    // [D, 4] (CONV)
    const float* conv_b;    // [D] or NULL (CONV)
    int act;                // CONV: 1 = SiLU after the convolution
    const float* dt_bias;
    const float* A;
    const float* Dskip;
    int has_z;
    int test_stall;         // never publish chunk states (failure-detection tests)
    long long batch, L, D;
    long long T;            // steps per unit (narrow plan; multiple of TC)
    long long P;            // units per chain (narrow plan)
    long long nst;          // stages per chain, ceil(L / TC) (chained plan)
    long long G;            // CTAs of the chained plan's static split
    long long Wst;          // nchains * nst
    long long nchains;      // batch * nCB
    long long nCB;          // ceil(D / CB)
    long long nSB;          // ceil(D / CW): 32-channel sub-blocks per batch entry
    long long total_units;
    unsigned long long* ticket;
    unsigned* abort;
    unsigned* flags;        // [batch * nSB] completed pieces per sub-block (kChained)
    float* carry;           // [batch, D, NS] chained state (h_last or scratch)
    float* agg;             // [P][batch*D][NS+1] phase-1 summaries (kAggregate)
    const float* hin;       // [P][batch*D][NS] phase-3 initial states (kFromState)
    float* ckpt;            // NULL, or [ceil(L/32)][batch*D][NS]: the state entering each
                            // 32-step unit (entry 0, the zero state, not written)
    unsigned long long wait_ns;
};

template <typename T>
struct Cfg {
    static constexpr int es = sizeof(T);
    static constexpr int TC = es == 2 ? 32 : 16;     // steps per stage
    static constexpr int kTile = TC * CB * es;       // u / delta / z tile
    static constexpr int kRaw = TC * NS * es;        // raw B or C rows
    static constexpr int kConv = TC * NS * 4;        // widened B/(n+1) or C rows
    static constexpr int kPar = CB * (int)sizeof(ChanPar);
    static constexpr int kState = CB * NS * 4;       // carried state of the tile
    // Trapezoid: u and the B row of the step before the piece (1 KiB slot).
    static constexpr int kPrev = 1024;
    static constexpr int offU = 0;
    static constexpr int offD = offU + kTile;
    static constexpr int offZ = offD + kTile;
    static constexpr int offBr = offZ + kTile;
    static constexpr int offCr = offBr + kRaw;
    static constexpr int offBc = offCr + kRaw;
    static constexpr int offCc = offBc + kConv;
    static constexpr int offPar = offCc + kConv;
    static constexpr int offState = offPar + kPar;
    static constexpr int offPrev = offState + kState;
    static constexpr int kStage = offPrev + kPrev;
    // Prologue ring of one helper/consumer pair: NPB buffers x KP steps x
    // 32 lanes x float4.
    static constexpr int kProBuf = KP * CW * 16;
    static constexpr int kPro = NPB * kProBuf;
    static constexpr int offPro = S * kStage;
    // y tiles of one consumer: 2 buffers of [TC][32] elements.
    static constexpr int kY = TC * CW * es;
    static constexpr int offY = offPro + NCW * kPro;
    static constexpr int offMeta = offY + NCW * 2 * kY;
    static constexpr int offBar = offMeta + S * (int)sizeof(Meta);
    static constexpr int kNumBars = 3 * S + 2 * NPB * NCW;
    static constexpr int kBytes = offBar + kNumBars * 8;
    static constexpr int kSmemBytes = kBytes + 1024;   // + slack to align the base
    static constexpr int kRowsPerHelper = TC / NCW;
    static_assert(kTile % 1024 == 0 && kRaw % 128 == 0 && kConv % 128 == 0 && kPar % 128 == 0 &&
                      kState % 128 == 0 && kStage % 1024 == 0 && kY % 128 == 0,
                  "shared-memory carve-out alignment");
    static_assert(TC % KP == 0 && TC % NCW == 0 && (kRowsPerHelper * NS / 2) % 32 == 0,
                  "stage shape");
    static_assert(kSmemBytes <= 227 * 1024, "CTA shared memory");
};

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

__device__ __forceinline__ float ld_elem(const float* p) { return *p; }
__device__ __forceinline__ float ld_elem(const bf16* p) {
    const unsigned short bits = *reinterpret_cast<const unsigned short*>(p);
    return __uint_as_float(static_cast<unsigned>(bits) << 16);
}
__device__ __forceinline__ void st_elem(float* p, float v) { *p = v; }
__device__ __forceinline__ void st_elem(bf16* p, float v) { *p = __float2bfloat16_rn(v); }

// Bounded mbarrier wait shared by every role: gives up after the configured
// limit or when another warp of the grid has raised the abort word.
__device__ __forceinline__ bool bwait(uint64_t* bar, uint32_t parity, const Params& p,
                                      uint32_t sleep_ns = 0) {
    return ptx::mbar_wait(bar, parity, p.wait_ns, p.abort, sleep_ns);
}

__device__ __forceinline__ void raise_failure(const Params& p) {
    atomicOr(&g_error_word, kErrTimeout);
    atomicExch(p.abort, 1u);
}

// Widening of rows [row0, row0 + kRowsPerHelper) of a stage's B and C to
// float32, B scaled by 1/(n+1) for the zero-order hold (unscaled for the
// other variants).  Lane l handles element pairs l, l+32, ... of that row
// range; every pair a lane handles has n = 2*(l % 8) + {0, 1}.
template <typename T, int MODE, int DISC>
__device__ __forceinline__ void widen_rows(unsigned char* st, int row0, int lane) {
    using C = Cfg<T>;
    constexpr int kPairs = C::kRowsPerHelper * NS / 2;
    const int n0 = 2 * (lane % (NS / 2));
    const float s0 = DISC == kZOH ? 1.0f / (float)(n0 + 1) : 1.0f;
    const float s1 = DISC == kZOH ? 1.0f / (float)(n0 + 2) : 1.0f;
    const T* Br = reinterpret_cast<const T*>(st + C::offBr) + row0 * NS;
    const T* Cr = reinterpret_cast<const T*>(st + C::offCr) + row0 * NS;
    float2* Bc = reinterpret_cast<float2*>(st + C::offBc) + row0 * (NS / 2);
    float2* Cc = reinterpret_cast<float2*>(st + C::offCc) + row0 * (NS / 2);
    float2 bv[kPairs / 32], cv[kPairs / 32];
#pragma unroll
    for (int i = 0; i < kPairs / 32; ++i) {
        const int w = lane + 32 * i;
        bv[i] = make_float2(ld_elem(Br + 2 * w) * s0, ld_elem(Br + 2 * w + 1) * s1);
        if (forms_y(MODE)) cv[i] = make_float2(ld_elem(Cr + 2 * w), ld_elem(Cr + 2 * w + 1));
    }
#pragma unroll
    for (int i = 0; i < kPairs / 32; ++i) {
        Bc[lane + 32 * i] = bv[i];
        if (forms_y(MODE)) Cc[lane + 32 * i] = cv[i];
    }
}

// ----------------------------------------------------------------- TMA warp
// Loads the unit's per-channel parameters (and the carried state) into the
// header of its first stage; returns the geometric-A bit mask of the four
// 32-channel sub-blocks.  All 32 lanes take part; lane l handles channels
// l, l+32, l+64, l+96 of the tile.
template <typename T, int MODE, int DISC>
__device__ int fill_header(unsigned char* st, const Params& p, long long b, long long d0,
                           long long k, long long t0, bool* has_state, bool* ok_out, int lane) {
    using C = Cfg<T>;
    ChanPar* par = reinterpret_cast<ChanPar*>(st + C::offPar);
    int geo = 0;
    if (DISC == kTrap) {
        // u and the B row of the step before the piece (zero before step 0):
        // the trapezoid's first step needs B_{t0-1} u_{t0-1}.
        float* prev = reinterpret_cast<float*>(st + C::offPrev);
        const T* ur = static_cast<const T*>(p.u) + (b * p.L + (t0 > 0 ? t0 - 1 : 0)) * p.D;
        const T* br = static_cast<const T*>(p.Bm) + (b * p.L + (t0 > 0 ? t0 - 1 : 0)) * NS;
#pragma unroll
        for (int w = 0; w < NCW; ++w) {
            const long long d = d0 + CW * w + lane;
            prev[CW * w + lane] = (t0 > 0 && d < p.D) ? to_f32(ur[d]) : 0.0f;
        }
        if (lane < NS) prev[CB + lane] = t0 > 0 ? to_f32(br[lane]) : 0.0f;
    }
#pragma unroll
    for (int w = 0; w < NCW; ++w) {
        const long long d = d0 + CW * w + lane;
        const bool valid = d < p.D;
        const long long ds = valid ? d : 0;
        const float4* arow = reinterpret_cast<const float4*>(p.A + ds * NS);
        float av[NS];
#pragma unroll
        for (int q = 0; q < NS / 4; ++q) {
            const float4 v = __ldg(arow + q);
            av[4 * q] = v.x;
            av[4 * q + 1] = v.y;
            av[4 * q + 2] = v.z;
            av[4 * q + 3] = v.w;
        }
        const float bias = p.dt_bias ? __ldg(p.dt_bias + ds) : 0.0f;
        const float dsk = p.Dskip ? __ldg(p.Dskip + ds) : 0.0f;
        const float a0 = av[0];
        bool g = fabsf(a0) >= 0.0625f && isfinite(a0);
#pragma unroll
        for (int n = 1; n < NS; ++n) g = g && (av[n] == (float)(n + 1) * a0);
        if (__all_sync(0xffffffffu, g || !valid)) geo |= 1 << w;
        ChanPar cp;
        cp.a0 = a0;
        cp.ia0 = (a0 != 0.0f) ? 1.0f / a0 : 0.0f;
        cp.kb2 = bias * kLog2e;
        cp.dsk = dsk;
        par[CW * w + lane] = cp;
    }
    *has_state = false;
    *ok_out = true;
    const float* src = nullptr;
    if (walks_chains(MODE) && k > 0) {
        // Lane w polls the flag of sub-block w (bounded); the state is read
        // only once all four predecessors have published.
        bool ok = true;
        if (lane < NCW) {
            const long long sb = (d0 / CW) + lane;
            if (sb < p.nSB) {
                const unsigned* f = p.flags + b * p.nSB + sb;
                const uint64_t t0 = ptx::globaltimer();
                while (ptx::ld_acquire(f) < (unsigned)k) {
                    ptx::nanosleep(kSleepNs);
                    if (*reinterpret_cast<const volatile unsigned*>(p.abort) ||
                        ptx::globaltimer() - t0 > p.wait_ns) {
                        ok = false;
                        break;
                    }
                }
            }
        }
        ok = __all_sync(0xffffffffu, ok);
        __threadfence();
        *ok_out = ok;
        if (!ok) return geo;
        src = p.carry;
    } else if (MODE == kFromState && k > 0) {
        src = p.hin + k * p.batch * p.D * NS;
    }
    if (src) {
        float4* dst = reinterpret_cast<float4*>(st + C::offState);
#pragma unroll
        for (int w = 0; w < NCW; ++w) {
            const long long d = d0 + CW * w + lane;
            const bool valid = d < p.D;
            const float4* s4 = reinterpret_cast<const float4*>(src + (b * p.D + (valid ? d : 0)) * NS);
#pragma unroll
            for (int q = 0; q < NS / 4; ++q)
                dst[(CW * w + lane) * (NS / 4) + q] = valid ? __ldcg(s4 + q) : make_float4(0, 0, 0, 0);
        }
        *has_state = true;
    }
    return geo;
}

// ------------------------------------------------------------------ helpers
// Per-step values of KP consecutive steps of the helper's 32 channels, with
// g = z sigmoid(z) (1 without z), sug = Dskip u g, dt = dl ln 2:
//                       geometric A                  other A
//   kZOH              {r = exp(dt a0), u/a0, g, sug}  {dl, u, g, sug}
//   kEuler            {r, dt u, g, sug}               {dl, u, g, sug}
//   kTrap             {r, dt/2, u, g}                 {dl, u, g, sug}
//   kAggregate mode   the same .x/.y (kTrap: .x/.y/.z), .w = dl
// Per-lane state of the convolution (CONV): weights, bias, the last three x.
struct ConvState {
    float w0, w1, w2, w3, bias, x1, x2, x3;   // x1 = x_{t-1}, x2 = x_{t-2}, x3 = x_{t-3}
};

template <typename T, int MODE, int DISC, bool HASZ, bool CONV>
__device__ __forceinline__ void prologue_chunk(const unsigned char* st, int row0, int col,
                                               const ChanPar& cp, bool geo, float4* out,
                                               ConvState& cs, int act) {
    using C = Cfg<T>;
    const T* U = reinterpret_cast<const T*>(st + C::offU);
    const T* Dl = reinterpret_cast<const T*>(st + C::offD);
    const T* Z = reinterpret_cast<const T*>(st + C::offZ);
    // All KP results are computed before any is stored: a shared-memory store
    // between steps would keep the compiler from hoisting the next steps'
    // loads above it (it cannot prove the two do not overlap), and the KP
    // independent SFU chains would then run one after another.
    float4 o[KP];
#pragma unroll
    for (int j = 0; j < KP; ++j) {
        const int t = row0 + j;
        float u = ld_elem(U + t * CB + col);
        if (CONV) {
            const float x = u;
            float v = fmaf(cs.w0, cs.x3, cs.bias);
            v = fmaf(cs.w1, cs.x2, v);
            v = fmaf(cs.w2, cs.x1, v);
            v = fmaf(cs.w3, x, v);
            u = act ? v * ptx::rcp(1.0f + ptx::ex2(v * -kLog2e)) : v;
            cs.x3 = cs.x2;
            cs.x2 = cs.x1;
            cs.x1 = x;
        }
        const float dv = ld_elem(Dl + t * CB + col);
        const float v2 = fmaf(dv, kLog2e, cp.kb2);           // (delta + bias) log2(e)
        // softplus / ln 2; the identity above v = 20 (v2 = 28.85), where the two
        // agree to float32 and 2^v2 could overflow
        const float dl = v2 > 28.853901f ? v2 : ptx::lg2(1.0f + ptx::ex2(v2));
        float g = 1.0f;
        if (forms_y(MODE)) {
            if constexpr (HASZ) {
                const float z = ld_elem(Z + t * CB + col);
                g = z * ptx::rcp(1.0f + ptx::ex2(z * -kLog2e));
            }
        }
        const float sug = cp.dsk * u * g;
        if (geo) {
            o[j].x = ptx::ex2(dl * cp.a0);   // r
            if (DISC == kZOH) o[j].y = u * cp.ia0;
            else if (DISC == kEuler) o[j].y = dl * kLn2 * u;
            else o[j].y = dl * (0.5f * kLn2);
            if (DISC == kTrap) {
                o[j].z = u;
                o[j].w = !forms_y(MODE) ? dl : g;
            } else {
                o[j].z = !forms_y(MODE) ? 0.0f : g;
                o[j].w = !forms_y(MODE) ? dl : sug;
            }
        } else {
            o[j] = make_float4(dl, u, !forms_y(MODE) ? 0.0f : g, !forms_y(MODE) ? dl : sug);
        }
    }
#pragma unroll
    for (int j = 0; j < KP; ++j) out[j * CW] = o[j];
}

// ---------------------------------------------------------------- consumers
// Recurrence and readout of cnt (<= KP) steps, geometric A.  FULL: cnt ==
// KP, a straight-line body the compiler can schedule across steps.  The y
// values are kept in registers and stored after the last step, so that no
// shared-memory store sits between one step's loads and the next's.  P holds
// B_{t-1} u_{t-1} per state (kTrap only); dsk = Dskip[d] (kTrap only).
template <typename T, int MODE, int DISC, bool FULL>
__device__ __forceinline__ void steps_geo(const unsigned char* st, int row0, int cnt,
                                          const float4* pro, float2 (&H)[NS / 2],
                                          float2 (&P)[NS / 2], float dsk, float& S2, T* ytile,
                                          int lane) {
    using C = Cfg<T>;
    const float* Bc = reinterpret_cast<const float*>(st + C::offBc);
    const float* Cc = reinterpret_cast<const float*>(st + C::offCc);
    float yv[KP];
#pragma unroll
    for (int j = 0; j < KP; ++j) {
        yv[j] = 0.0f;
        if (!FULL && j >= cnt) break;
        const int t = row0 + j;
        const float4 pv = pro[j * CW];
        const float4* B4 = reinterpret_cast<const float4*>(Bc + t * NS);
        const float4* C4 = reinterpret_cast<const float4*>(Cc + t * NS);
        const float r = pv.x;
        const float e0 = r - 1.0f;                  // exp(dt A_0) - 1
        const float e1 = fmaf(r, e0, e0);           // exp(dt A_1) - 1
        const float r2 = e1 + 1.0f;
        const float2 R2 = make_float2(r2, r2), E1 = make_float2(e1, e1);
        // kZOH: u/a0; kEuler: dt u; kTrap: dt/2
        const float2 UP = make_float2(pv.y, pv.y);
        const float2 U2 = make_float2(pv.z, pv.z);  // kTrap: u
        float2 E = make_float2(e0, e1);
        float2 Y0 = make_float2(0.f, 0.f), Y1 = make_float2(0.f, 0.f);
#pragma unroll
        for (int q = 0; q < NS / 4; ++q) {
            const float4 b4 = B4[q];
            const int k0 = 2 * q, k1 = 2 * q + 1;
            const float2 Ba = make_float2(b4.x, b4.y), Bb = make_float2(b4.z, b4.w);
            if (k0 > 0) E = ffma2(R2, E, E1);      // (e_{n+2}, e_{n+3}) = r^2 (e_n, e_{n+1}) + e_1
            if (DISC == kZOH) {
                H[k0] = ffma2(E, ffma2(Ba, UP, H[k0]), H[k0]);   // h + e (h + B u / A)
            } else if (DISC == kEuler) {
                H[k0] = ffma2(E, H[k0], ffma2(Ba, UP, H[k0]));   // h + e h + dt u B
            } else {
                const float2 Pn = __fmul2_rn(Ba, U2);            // B_t u_t
                const float2 Sv = ffma2(UP, P[k0], H[k0]);       // h + dt/2 P_{t-1}
                H[k0] = ffma2(UP, Pn, ffma2(E, Sv, Sv));         // A_bar s + dt/2 P_t
                P[k0] = Pn;
            }
            E = ffma2(R2, E, E1);
            if (DISC == kZOH) {
                H[k1] = ffma2(E, ffma2(Bb, UP, H[k1]), H[k1]);
            } else if (DISC == kEuler) {
                H[k1] = ffma2(E, H[k1], ffma2(Bb, UP, H[k1]));
            } else {
                const float2 Pn = __fmul2_rn(Bb, U2);
                const float2 Sv = ffma2(UP, P[k1], H[k1]);
                H[k1] = ffma2(UP, Pn, ffma2(E, Sv, Sv));
                P[k1] = Pn;
            }
            if (forms_y(MODE)) {
                const float4 c4 = C4[q];
                Y0 = ffma2(make_float2(c4.x, c4.y), H[k0], Y0);
                Y1 = ffma2(make_float2(c4.z, c4.w), H[k1], Y1);
            }
        }
        if (MODE == kAggregate) {
            S2 += pv.w;
        } else if (forms_y(MODE)) {
            const float sum = (Y0.x + Y0.y) + (Y1.x + Y1.y);
            if (DISC == kTrap) yv[j] = fmaf(dsk, pv.z, sum) * pv.w;   // (sum + D u) g
            else yv[j] = fmaf(sum, pv.z, pv.w);                       // sum g + D u g
        }
    }
    if (forms_y(MODE)) {
#pragma unroll
        for (int j = 0; j < KP; ++j) {
            if (!FULL && j >= cnt) break;
            st_elem(ytile + (row0 + j) * CW + lane, yv[j]);
        }
    }
}

// Any other A (including zeros): per state, A_bar - 1 = 2^(dl A) - 1 and,
// for the zero-order hold, B_bar/B = (A_bar - 1)/A, or dt where A == 0.
// Correct, not tuned.
template <typename T, int MODE, int DISC>
__device__ __forceinline__ void steps_general(const unsigned char* st, int row0, int cnt,
                                              const float4* pro, const float* __restrict__ Arow,
                                              float2 (&H)[NS / 2], float2 (&P)[NS / 2],
                                              float& S2, T* ytile, int lane) {
    using C = Cfg<T>;
    const float* Bc = reinterpret_cast<const float*>(st + C::offBc);
    const float* Cc = reinterpret_cast<const float*>(st + C::offCc);
    float yv[KP];
#pragma unroll
    for (int j = 0; j < KP; ++j) {
        yv[j] = 0.0f;
        if (j >= cnt) break;
        const int t = row0 + j;
        const float4 pv = pro[j * CW];
        const float dl = pv.x, u = pv.y;
        const float dt = dl * kLn2;
        if (MODE == kAggregate) S2 += pv.w;
        float y = 0.0f;
#pragma unroll
        for (int n = 0; n < NS; ++n) {
            const float a = __ldg(Arow + n);
            const float e = em1_near0(dl * a * kLn2, ptx::ex2(dl * a));
            float hn = (n & 1) ? H[n / 2].y : H[n / 2].x;
            if (DISC == kZOH) {
                const float coef = (a != 0.0f) ? e / a : dt;
                const float bn = Bc[t * NS + n] * (float)(n + 1);
                hn = fmaf(coef * bn, u, fmaf(e, hn, hn));
            } else if (DISC == kEuler) {
                hn = fmaf(dt * Bc[t * NS + n], u, fmaf(e, hn, hn));
            } else {
                const float pn = Bc[t * NS + n] * u;
                float& po = (n & 1) ? P[n / 2].y : P[n / 2].x;
                const float sv = fmaf(0.5f * dt, po, hn);
                hn = fmaf(0.5f * dt, pn, fmaf(e, sv, sv));
                po = pn;
            }
            if (n & 1) H[n / 2].y = hn; else H[n / 2].x = hn;
            if (forms_y(MODE)) y = fmaf(Cc[t * NS + n], hn, y);
        }
        if (forms_y(MODE)) yv[j] = fmaf(y, pv.z, pv.w);
    }
    if (forms_y(MODE)) {
#pragma unroll
        for (int j = 0; j < KP; ++j) {
            if (j >= cnt) break;
            st_elem(ytile + (row0 + j) * CW + lane, yv[j]);
        }
    }
}

template <typename T, int MODE, int DISC, bool CONV>
__global__ void __launch_bounds__(THREADS, 1)
scan_tile_kernel(const __grid_constant__ CUtensorMap tmU, const __grid_constant__ CUtensorMap tmD,
                 const __grid_constant__ CUtensorMap tmZ, const __grid_constant__ CUtensorMap tmB,
                 const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmY,
                 const Params p) {
    using C = Cfg<T>;
    constexpr int TC = C::TC;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // Stage tiles are TMA sources and destinations: align the carve-out base
    // to 1 KiB (the launch requests kSmemBytes, which includes that slack).
    unsigned char* smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
    Meta* meta = reinterpret_cast<Meta*>(smem + C::offMeta);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::offBar);
    uint64_t* convd = full + S;
    uint64_t* empty = convd + S;
    uint64_t* pfull = empty + S;            // [NCW][NPB]
    uint64_t* pempty = pfull + NPB * NCW;   // [NCW][NPB]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&convd[s], NCW);
            ptx::mbar_init(&empty[s], NCW);
        }
        for (int i = 0; i < NPB * NCW; ++i) {
            ptx::mbar_init(&pfull[i], 1);
            ptx::mbar_init(&pempty[i], 1);
        }
        ptx::fence_mbar_init();
    }
    __syncthreads();

    if (warp == kTmaWarp) {
        // ------------------------------------------------------------ TMA warp
        if (lane == 0) {
            ptx::prefetch_tensormap(&tmU);
            ptx::prefetch_tensormap(&tmD);
            ptx::prefetch_tensormap(&tmB);
            if (forms_y(MODE)) {
                ptx::prefetch_tensormap(&tmC);
                if (p.has_z) ptx::prefetch_tensormap(&tmZ);
            }
        }
        const uint32_t stage_tx =
            !forms_y(MODE) ? 2 * C::kTile + C::kRaw
                                 : 2 * C::kTile + 2 * C::kRaw + (p.has_z ? C::kTile : 0);
        // Piece source.  kChained, kCkptOnly: the CTA's range [r0, r1) of the
        // chain-major stage space, walked from its last chain to its first.
        // Narrow-plan modes: units k * T .. (k+1) * T of a chain, from the
        // ticket counter.
        const long long r0 = (long long)blockIdx.x * p.Wst / (p.G > 0 ? p.G : 1);
        const long long r1 = ((long long)blockIdx.x + 1) * p.Wst / (p.G > 0 ? p.G : 1);
        long long next_chain = walks_chains(MODE) ? (r1 - 1) / (p.nst > 0 ? p.nst : 1) : 0;
        long long cur_chain = -1, cur_t0 = 0, cur_end = 0, cur_b = 0, cur_d0 = 0, cur_k = 0;
        bool chain_end = false;
        long long j = 0;
        bool failed = false;
        for (;; ++j) {
            const int slot = (int)(j % S);
            if (j >= S && !bwait(&empty[slot], (uint32_t)(((j / S) - 1) & 1), p, kSleepNs)) {
                failed = true;
                break;
            }
            unsigned char* st = smem + slot * C::kStage;
            int flags = 0, geo = 0;
            if (cur_chain < 0 || cur_t0 >= cur_end) {
                bool more;
                if (walks_chains(MODE)) {
                    more = r0 < r1 && next_chain >= r0 / p.nst;
                    if (more) {
                        const long long c = next_chain--;
                        const long long s0 = (r0 > c * p.nst ? r0 : c * p.nst) - c * p.nst;
                        const long long s1 =
                            (r1 < (c + 1) * p.nst ? r1 : (c + 1) * p.nst) - c * p.nst;
                        // CTA holding the chain's first stage; the pieces of a
                        // chain sit on consecutive CTAs.
                        const long long i0 = ((c * p.nst + 1) * p.G + p.Wst - 1) / p.Wst - 1;
                        cur_chain = c;
                        cur_k = (long long)blockIdx.x - i0;
                        cur_t0 = s0 * TC;
                        cur_end = s1 * TC < p.L ? s1 * TC : p.L;
                        chain_end = s1 == p.nst;
                    }
                } else {
                    unsigned long long tk = 0;
                    if (lane == 0) tk = atomicAdd(p.ticket, 1ull);
                    tk = __shfl_sync(0xffffffffu, tk, 0);
                    more = (long long)tk < p.total_units;
                    if (more) {
                        cur_k = (long long)tk / p.nchains;
                        cur_chain = (long long)tk % p.nchains;
                        cur_t0 = cur_k * p.T;
                        cur_end = cur_t0 + p.T < p.L ? cur_t0 + p.T : p.L;
                        chain_end = cur_end == p.L;
                    }
                }
                if (!more || *reinterpret_cast<const volatile unsigned*>(p.abort)) {
                    if (lane == 0) {
                        meta[slot].flags = kEnd;
                        ptx::mbar_arrive(&full[slot]);
                    }
                    ++j;
                    break;
                }
                cur_b = cur_chain / p.nCB;
                cur_d0 = (cur_chain % p.nCB) * CB;
                bool has_state = false, ok = true;
                geo = fill_header<T, MODE, DISC>(st, p, cur_b, cur_d0, cur_k, cur_t0, &has_state,
                                                 &ok, lane);
                if (!ok) {
                    if (lane == 0) raise_failure(p);
                    failed = true;
                    // Still hand the stage over (marked as the end) so that
                    // the other roles leave their loops.
                    if (lane == 0) {
                        meta[slot].flags = kEnd;
                        ptx::mbar_arrive(&full[slot]);
                    }
                    ++j;
                    break;
                }
                flags |= kFirst | (has_state ? kHasState : 0);
            }
            const int nvalid = (int)(cur_end - cur_t0 < TC ? cur_end - cur_t0 : TC);
            if (cur_t0 + TC >= cur_end) flags |= kLast | (chain_end ? kChainEnd : 0);
            __syncwarp();
            if (lane == 0) {
                meta[slot].chain = cur_chain;
                meta[slot].t0 = cur_t0;
                meta[slot].nvalid = nvalid;
                meta[slot].flags = flags;
                meta[slot].geo = geo;
                meta[slot].piece = (int)cur_k;
                ptx::mbar_arrive_expect_tx(&full[slot], stage_tx);
                const int x = (int)cur_d0, yy = (int)cur_t0, z = (int)cur_b;
                ptx::tma_load_3d(st + C::offU, &tmU, &full[slot], x, yy, z);
                ptx::tma_load_3d(st + C::offD, &tmD, &full[slot], x, yy, z);
                ptx::tma_load_3d(st + C::offBr, &tmB, &full[slot], 0, yy, z);
                if (forms_y(MODE)) {
                    if (p.has_z) ptx::tma_load_3d(st + C::offZ, &tmZ, &full[slot], x, yy, z);
                    ptx::tma_load_3d(st + C::offCr, &tmC, &full[slot], 0, yy, z);
                }
            }
            __syncwarp();
            cur_t0 += TC;
        }
        if (failed && lane == 0) raise_failure(p);
        // Never leave with bulk copies in flight: wait (bounded) for the
        // stages issued last (earlier ones were waited for by the consumers
        // before they released their slots).
        if (lane == 0)
            for (long long i = (j - S > 0 ? j - S : 0); i < j; ++i)
                ptx::mbar_wait(&full[i % S], (uint32_t)((i / S) & 1), p.wait_ns, nullptr);
        return;
    }

    if (warp >= NCW) {
        // ------------------------------------------------------------- helpers
        const int hi = warp - NCW;
        float4* pro = reinterpret_cast<float4*>(smem + C::offPro + hi * C::kPro);
        ChanPar cp{0.f, 0.f, 0.f, 0.f};
        ConvState cs{0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        bool geo = true;
        long long q = 0;   // prologue chunks produced
        bool failed = false;
        for (long long j = 0; !failed; ++j) {
            const int slot = (int)(j % S);
            if (!bwait(&full[slot], (uint32_t)((j / S) & 1), p)) {
                failed = true;
                break;
            }
            const Meta m = meta[slot];
            unsigned char* st = smem + slot * C::kStage;
            if (!(m.flags & kEnd)) widen_rows<T, MODE, DISC>(st, hi * C::kRowsPerHelper, lane);
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&convd[slot]);
            if (m.flags & kEnd) break;
            if (m.flags & kFirst) {
                cp = reinterpret_cast<const ChanPar*>(st + C::offPar)[CW * hi + lane];
                geo = (m.geo >> hi) & 1;
                if (CONV) {
                    // weights and the three x values before the piece (zero
                    // before step 0 and past the last channel)
                    const long long b = m.chain / p.nCB;
                    const long long d = (m.chain % p.nCB) * CB + CW * hi + lane;
                    const bool valid = d < p.D;
                    const float4 w4 = valid ? __ldg(reinterpret_cast<const float4*>(p.conv_w) + d)
                                            : make_float4(0.f, 0.f, 0.f, 0.f);
                    cs.w0 = w4.x;
                    cs.w1 = w4.y;
                    cs.w2 = w4.z;
                    cs.w3 = w4.w;
                    cs.bias = (valid && p.conv_b) ? __ldg(p.conv_b + d) : 0.0f;
                    const T* xs = static_cast<const T*>(p.u) + b * p.L * p.D + (valid ? d : 0);
                    const long long t0 = m.t0;
                    cs.x1 = (valid && t0 >= 1) ? to_f32(xs[(t0 - 1) * p.D]) : 0.0f;
                    cs.x2 = (valid && t0 >= 2) ? to_f32(xs[(t0 - 2) * p.D]) : 0.0f;
                    cs.x3 = (valid && t0 >= 3) ? to_f32(xs[(t0 - 3) * p.D]) : 0.0f;
                }
            }
            const int nchunks = (m.nvalid + KP - 1) / KP;
            for (int c = 0; c < nchunks; ++c, ++q) {
                const int buf = (int)(q % NPB);
                if (q >= NPB && !bwait(&pempty[NPB * hi + buf], (uint32_t)(((q / NPB) - 1) & 1), p)) {
                    failed = true;
                    break;
                }
                float4* out = pro + buf * (C::kProBuf / 16) + lane;
                if (p.has_z)
                    prologue_chunk<T, MODE, DISC, true, CONV>(st, c * KP, CW * hi + lane, cp, geo,
                                                              out, cs, p.act);
                else
                    prologue_chunk<T, MODE, DISC, false, CONV>(st, c * KP, CW * hi + lane, cp, geo,
                                                               out, cs, p.act);
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&pfull[NPB * hi + buf]);
            }
        }
        if (failed && lane == 0) raise_failure(p);
        return;
    }

    // ------------------------------------------------------------- consumers
    const int w = warp;
    const float4* pro = reinterpret_cast<const float4*>(smem + C::offPro + w * C::kPro);
    T* ytiles = reinterpret_cast<T*>(smem + C::offY + w * 2 * C::kY);
    long long k = 0, chain = 0, b = 0, d0 = 0, d = 0;
    bool valid = false, geo = true, block_live = false;
    float2 H[NS / 2];
    float2 P[NS / 2];   // B_{t-1} u_{t-1} per state (trapezoid)
    float dsk = 0.0f;
    const float* Arow = p.A;
    float S2 = 0.0f;
    long long q = 0;
    bool failed = false;
#pragma unroll
    for (int i = 0; i < NS / 2; ++i) {
        H[i] = make_float2(0.f, 0.f);
        P[i] = make_float2(0.f, 0.f);
    }
    for (long long j = 0; !failed; ++j) {
        const int slot = (int)(j % S);
        if (!bwait(&convd[slot], (uint32_t)((j / S) & 1), p)) {
            failed = true;
            break;
        }
        const Meta m = meta[slot];
        if (m.flags & kEnd) break;
        const unsigned char* st = smem + slot * C::kStage;
        if (m.flags & kFirst) {
            k = m.piece;
            chain = m.chain;
            b = chain / p.nCB;
            d0 = (chain % p.nCB) * CB + CW * w;
            d = d0 + lane;
            valid = d < p.D;
            block_live = d0 < p.D;
            geo = (m.geo >> w) & 1;
            dsk = reinterpret_cast<const ChanPar*>(st + C::offPar)[CW * w + lane].dsk;
            if (DISC == kTrap) {
                const float* prev = reinterpret_cast<const float*>(st + C::offPrev);
                const float up = prev[CW * w + lane];
#pragma unroll
                for (int i = 0; i < NS / 2; ++i)
                    P[i] = make_float2(prev[CB + 2 * i] * up, prev[CB + 2 * i + 1] * up);
            }
            S2 = 0.0f;
            if (m.flags & kHasState) {
                const float4* s4 = reinterpret_cast<const float4*>(st + C::offState) + (CW * w + lane) * (NS / 4);
#pragma unroll
                for (int i = 0; i < NS / 4; ++i) {
                    const float4 v = s4[i];
                    H[2 * i] = make_float2(v.x, v.y);
                    H[2 * i + 1] = make_float2(v.z, v.w);
                }
            } else {
#pragma unroll
                for (int i = 0; i < NS / 2; ++i) H[i] = make_float2(0.f, 0.f);
            }
            Arow = p.A + (valid ? d : 0) * NS;
        }
        T* ytile = ytiles + (int)(j & 1) * (C::kY / (int)sizeof(T));
        if (forms_y(MODE)) {
            // The store that last read this y buffer (two stages ago) must
            // have finished reading it.
            if (lane == 0) ptx::bulk_wait_group_read<1>();
            __syncwarp();
        }
        const int nchunks = (m.nvalid + KP - 1) / KP;
        for (int c = 0; c < nchunks; ++c, ++q) {
            const int buf = (int)(q % NPB);
            if (!bwait(&pfull[NPB * w + buf], (uint32_t)((q / NPB) & 1), p)) {
                failed = true;
                break;
            }
            const int cnt = m.nvalid - c * KP < KP ? m.nvalid - c * KP : KP;
            const float4* pv = pro + buf * (C::kProBuf / 16) + lane;
            if (geo) {
                if (cnt == KP)
                    steps_geo<T, MODE, DISC, true>(st, c * KP, KP, pv, H, P, dsk, S2, ytile, lane);
                else
                    steps_geo<T, MODE, DISC, false>(st, c * KP, cnt, pv, H, P, dsk, S2, ytile,
                                                    lane);
            } else {
                steps_general<T, MODE, DISC>(st, c * KP, cnt, pv, Arow, H, P, S2, ytile, lane);
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&pempty[NPB * w + buf]);
        }
        if (failed) break;
        if (forms_y(MODE) && block_live) {
            // Hand the y tile to the TMA engine (rows past L and columns past
            // D fall outside the tensor and are not written).
            ptx::fence_proxy_async_shared();
            __syncwarp();
            if (lane == 0) {
                ptx::tma_store_3d(&tmY, ytile, (int)d0, (int)m.t0, (int)b);
                ptx::bulk_commit_group();
            }
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&empty[slot]);
        // the state entering the next 32-step unit, for a later backward pass
        if (MODE != kAggregate && p.ckpt) {
            const long long tend = m.t0 + m.nvalid;
            if (tend % kCkptSteps == 0 && tend < p.L && valid) {
                float4* dst = reinterpret_cast<float4*>(
                    p.ckpt + ((tend / kCkptSteps) * p.batch * p.D + b * p.D + d) * NS);
#pragma unroll
                for (int i = 0; i < NS / 4; ++i)
                    __stcg(dst + i, make_float4(H[2 * i].x, H[2 * i].y, H[2 * i + 1].x, H[2 * i + 1].y));
            }
        }
        if (m.flags & kLast) {
            if (walks_chains(MODE)) {
                if (!(m.flags & kChainEnd)) {
                    if (valid) {
                        float4* dst = reinterpret_cast<float4*>(p.carry + (b * p.D + d) * NS);
#pragma unroll
                        for (int i = 0; i < NS / 4; ++i)
                            __stcg(dst + i, make_float4(H[2 * i].x, H[2 * i].y, H[2 * i + 1].x,
                                                        H[2 * i + 1].y));
                    }
                    __threadfence();
                    __syncwarp();
                    if (lane == 0 && block_live && !p.test_stall)
                        ptx::st_release(p.flags + b * p.nSB + d0 / CW, (unsigned)(k + 1));
                } else if (valid && p.h_last) {
                    float4* dst = reinterpret_cast<float4*>(p.h_last + (b * p.D + d) * NS);
#pragma unroll
                    for (int i = 0; i < NS / 4; ++i)
                        dst[i] = make_float4(H[2 * i].x, H[2 * i].y, H[2 * i + 1].x, H[2 * i + 1].y);
                }
            } else if (MODE == kAggregate) {
                if (valid) {
                    float* dst = p.agg + (k * p.batch * p.D + b * p.D + d) * (NS + 1);
                    dst[0] = S2;
#pragma unroll
                    for (int i = 0; i < NS / 2; ++i) {
                        dst[1 + 2 * i] = H[i].x;
                        dst[2 + 2 * i] = H[i].y;
                    }
                }
            } else {
                if (valid && p.h_last && (m.flags & kChainEnd)) {
                    float4* dst = reinterpret_cast<float4*>(p.h_last + (b * p.D + d) * NS);
#pragma unroll
                    for (int i = 0; i < NS / 4; ++i)
                        dst[i] = make_float4(H[2 * i].x, H[2 * i].y, H[2 * i + 1].x, H[2 * i + 1].y);
                }
            }
        }
    }
    if (failed && lane == 0) raise_failure(p);
    // Every y store must have completed before the CTA's shared memory goes.
    if (forms_y(MODE) && lane == 0) ptx::bulk_wait_group<0>();
    __syncwarp();
}

// Phase 2 of the narrow plan: per (channel, state), the state entering each
// chunk, from the phase-1 summaries: h_in[0] = 0,
// h_in[k+1] = 2^(A[d,n] * S2_k) h_in[k] + Q_k[n]  (2^(A S2) = exp(A sum dt)).
__global__ void carry_kernel(const float* __restrict__ agg, const float* __restrict__ A,
                             float* __restrict__ hin, long long batch, long long D, long long P) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long nch = batch * D;
    if (i >= nch * NS) return;
    const long long ch = i / NS, n = i % NS, d = ch % D;
    const float a = A[d * NS + n];
    float h = 0.0f;
    for (long long kk = 0; kk < P; ++kk) {
        hin[(kk * nch + ch) * NS + n] = h;
        if (kk + 1 < P) {
            const float* g = agg + (kk * nch + ch) * (NS + 1);
            h = fmaf(exp2f(a * g[0]), h, g[1 + n]);
        }
    }
}

}  // namespace tile
}  // namespace ssm
