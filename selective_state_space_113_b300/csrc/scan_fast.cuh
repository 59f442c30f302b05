// scan_fast.cuh -- the sm_103a selective-scan kernel for N == 16.
//
// What it computes is the selective scan of the pages on Mamba (ta-paperlens
// "Mamba: 状態を「選択的」にする" pseudocode; ultralytics "SSMの仕組み" zero-order
// hold; y = C h + D x; SiLU(z) gate), in float32 with a float32 state.
//
// Work decomposition.  A unit is 32 channels (one per lane of a consumer
// warp) of one batch entry over T consecutive steps; the T steps of a unit are
// streamed through shared memory in stages of TC steps by TMA.  Units of one
// 32-channel block form a chain along the sequence.  A CTA is one producer
// warp (TMA issue + B/C widening) and one consumer warp (the recurrence);
// several CTAs share an SM.  CTAs are persistent and take units from an
// atomic ticket counter in chunk-major order, so the units in flight at any
// time belong to different chains.
//
// Three plans use this kernel:
//   kChained   -- each unit starts from its predecessor's final state, passed
//                 through global memory with a release/acquire flag (a
//                 bounded wait).  Used when there are at least about as many
//                 chains as resident CTAs, which keeps the waits near zero.
//   kAggregate -- phase 1 of the narrow-problem plan: each unit runs from a
//                 zero state and records sum(log2-domain dt) and its final
//                 state (the unit's affine summary; no y is written).
//   kFromState -- phase 3: each unit starts from a state computed by the carry
//                 kernel (phase 2) from the phase-1 summaries, and writes y.
//
// Per-step arithmetic (geometric A, A[d,n] = (n+1) a0 -- detected per warp):
//   v2 = delta*log2(e) + dt_bias*log2(e);  x = 2^v2 = e^(delta+bias)
//   dl = log2(1 + x)                          (dt = dl * ln2 = softplus)
//   r  = 2^(dl a0) = exp(dt a0);  e_n = r^(n+1) - 1 = exp(dt A[d,n]) - 1
//        e_0 = r - 1, e_1 = r e_0 + e_0, e_(n+2) = r^2 e_n + e_1
//   h_n <- h_n + e_n (h_n + B_n u / A[d,n])  (= A_bar h + (A_bar - 1)/A B u)
//   y  = (sum_n C_n h_n + Dskip u) * z / (1 + 2^(-z log2(e)))
// B_n/(n+1) is prepared once per stage by the producer warp, and u/a0 once
// per step, so B_n u / A[d,n] is one multiply-add away.  Any other A runs a
// per-state path that uses exp(dt A) - 1 directly and the dt*B limit at A = 0.
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "ptx.cuh"

namespace ssm {
namespace fast {

constexpr int TC = 32;   // steps per pipeline stage
constexpr int S = 4;     // stages in the shared-memory ring
constexpr int LA = 2;    // stages the TMA issue runs ahead of the B/C widening
constexpr int CH = 32;   // channels per unit (one per consumer lane)
constexpr int NS = 16;   // state size handled here
constexpr unsigned kProducerSleepNs = 128;  // producer back-off between mbarrier polls

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

enum Mode : int { kChained = 0, kAggregate = 1, kFromState = 2 };

enum MetaFlags : int { kFirst = 1, kLast = 2, kEnd = 4 };

struct Meta {
    long long unit;
    long long t0;
    int nvalid;
    int flags;
    int pad[2];
};

struct Params {
    void* y;
    float* h_last;
    const float* dt_bias;
    const float* A;
    const float* Dskip;
    int has_z;
    int test_stall;        // never publish chunk states (failure-detection tests)
    long long batch, L, D;
    long long T;           // steps per unit (multiple of TC)
    long long P;           // units per chain
    long long nchains;     // batch * nCB
    long long nCB;         // ceil(D / CH)
    long long total_units;
    unsigned long long* ticket;
    unsigned* abort;
    unsigned* flags;       // [nchains] completed chunks (kChained)
    float* carry;          // [batch, D, NS] chained state (h_last or scratch)
    float* agg;            // [P][batch*D][NS+1] phase-1 summaries (kAggregate)
    const float* hin;      // [P][batch*D][NS] phase-3 initial states (kFromState)
    unsigned long long wait_ns;
};

template <typename T>
struct Layout {
    static constexpr int es = sizeof(T);
    static constexpr int kTile = TC * CH * es;       // u / delta / z tile
    static constexpr int kRaw = TC * NS * es;        // raw B or C rows
    static constexpr int kConv = TC * NS * 4;        // widened B/(n+1) or C rows
    static constexpr int offU = 0;
    static constexpr int offD = offU + kTile;
    static constexpr int offZ = offD + kTile;
    static constexpr int offBr = offZ + kTile;
    static constexpr int offCr = offBr + kRaw;
    static constexpr int offBc = offCr + kRaw;
    static constexpr int offCc = offBc + kConv;
    static constexpr int kStage = offCc + kConv;
    static constexpr int offMeta = S * kStage;
    static constexpr int offBar = offMeta + S * (int)sizeof(Meta);
    static constexpr int kBytes = offBar + 3 * S * 8;
    static_assert(kTile % 128 == 0 && kRaw % 128 == 0 && kConv % 128 == 0, "TMA alignment");
    // One pair's carve-out, rounded to 1 KiB so every pair's tiles stay aligned.
    static constexpr int kPairBytes = (kBytes + 1023) & ~1023;
    // Worker pairs (consumer + producer warp) per CTA: four for 2-byte
    // elements (one consumer per SM sub-partition), two for float32, whose
    // stages are twice as large.
    static constexpr int kPairs = es == 2 ? 4 : 2;
    static constexpr int kThreads = 64 * kPairs;
    // Dynamic shared memory a CTA requests (+1 KiB for aligning the base).
    static constexpr int kSmemBytes = kPairs * kPairBytes + 1024;
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

// Per-lane (per-channel) unit state.
struct Chan {
    long long b, d, k, chain, ch;   // ch = b*D + d
    bool valid;
    float kb2, a0, ia0, dsk;        // dt_bias*log2(e), A[d,0], 1/A[d,0], Dskip[d]
};

constexpr int K = 8;  // steps per software-pipelined sub-block

// Per-step values that do not depend on the state, for K consecutive steps:
// r = exp(dt a0), up = u/a0, and the output affine map y = sum*g + sug with
// g the SiLU gate factor z*sigmoid(z) and sug = Dskip*u*g.  In kAggregate
// mode g holds the log2-domain dt of the step instead.
struct Pre {
    float r[K], up[K], g[K], sug[K];
};

// Stage-row index of step tt; steps past the tile wrap onto valid rows whose
// values are computed and then discarded.
__device__ __forceinline__ int row(int tt) { return tt & (TC - 1); }

template <typename T, int MODE, bool HASZ>
__device__ __forceinline__ void prologue(const unsigned char* st, int tt0, int lane, const Chan& c,
                                         Pre& pr) {
    using Lt = Layout<T>;
    const T* U = reinterpret_cast<const T*>(st + Lt::offU);
    const T* Dl = reinterpret_cast<const T*>(st + Lt::offD);
    const T* Z = reinterpret_cast<const T*>(st + Lt::offZ);
#pragma unroll
    for (int j = 0; j < K; ++j) {
        const int tt = row(tt0 + j);
        const float u = ld_elem(U + tt * CH + lane);
        const float dv = ld_elem(Dl + tt * CH + lane);
        const float v2 = fmaf(dv, kLog2e, c.kb2);            // (delta + bias) log2(e)
        const float dl = ptx::lg2(1.0f + ptx::ex2(v2));      // softplus / ln 2
        pr.r[j] = ptx::ex2(dl * c.a0);                       // exp(dt a0)
        pr.up[j] = u * c.ia0;
        if (MODE == kAggregate) {
            pr.g[j] = dl;
        } else {
            const float su = c.dsk * u;
            if constexpr (HASZ) {
                const float z = ld_elem(Z + tt * CH + lane);
                const float g = z * ptx::rcp(1.0f + ptx::ex2(z * -kLog2e));
                pr.g[j] = g;
                pr.sug[j] = su * g;
            } else {
                pr.g[j] = 1.0f;
                pr.sug[j] = su;
            }
        }
    }
}

// The state recurrence and readout of up to K steps (all K unless PARTIAL).
template <typename T, int MODE, bool PARTIAL>
__device__ __forceinline__ void recur(const unsigned char* st, int tt0, int cnt, const Pre& pr,
                                      float2 (&H)[NS / 2], float& S2, T* __restrict__ yptr,
                                      long long ystride, bool valid) {
    using Lt = Layout<T>;
    const float* Bc = reinterpret_cast<const float*>(st + Lt::offBc);
    const float* Cc = reinterpret_cast<const float*>(st + Lt::offCc);
#pragma unroll
    for (int j = 0; j < K; ++j) {
        if (PARTIAL && j >= cnt) break;
        const int tt = tt0 + j;
        const float4* B4 = reinterpret_cast<const float4*>(Bc + tt * NS);
        const float4* C4 = reinterpret_cast<const float4*>(Cc + tt * NS);
        const float r = pr.r[j];
        const float e0 = r - 1.0f;                  // exp(dt A_0) - 1
        const float e1 = fmaf(r, e0, e0);           // exp(dt A_1) - 1
        const float r2 = e1 + 1.0f;
        const float2 R2 = make_float2(r2, r2), E1 = make_float2(e1, e1);
        const float2 UP = make_float2(pr.up[j], pr.up[j]);
        float2 E = make_float2(e0, e1);
        float2 Y0 = make_float2(0.f, 0.f), Y1 = make_float2(0.f, 0.f);
#pragma unroll
        for (int q = 0; q < NS / 4; ++q) {
            const float4 b4 = B4[q];
            const int k0 = 2 * q, k1 = 2 * q + 1;
            if (k0 > 0) E = ffma2(R2, E, E1);      // (e_{n+2}, e_{n+3}) = r^2 (e_n, e_{n+1}) + e_1
            const float2 Sa = ffma2(make_float2(b4.x, b4.y), UP, H[k0]);
            H[k0] = ffma2(E, Sa, H[k0]);
            E = ffma2(R2, E, E1);
            const float2 Sb = ffma2(make_float2(b4.z, b4.w), UP, H[k1]);
            H[k1] = ffma2(E, Sb, H[k1]);
            if (MODE != kAggregate) {
                const float4 c4 = C4[q];
                Y0 = ffma2(make_float2(c4.x, c4.y), H[k0], Y0);
                Y1 = ffma2(make_float2(c4.z, c4.w), H[k1], Y1);
            }
        }
        if (MODE == kAggregate) {
            S2 += pr.g[j];
        } else {
            const float y = fmaf((Y0.x + Y0.y) + (Y1.x + Y1.y), pr.g[j], pr.sug[j]);
            if (valid) st_elem(yptr + tt * ystride, y);
        }
    }
}

// Geometric-A stage: software-pipelined over sub-blocks of K steps (the
// state-independent prologue of sub-block i+1 is issued alongside the
// recurrence of sub-block i).
template <typename T, int MODE, bool HASZ>
__device__ __forceinline__ void run_stage_geo(const unsigned char* st, int nvalid, int lane,
                                              const Chan& c, float2 (&H)[NS / 2], float& S2,
                                              T* __restrict__ yptr, long long ystride) {
    const int nsb = nvalid / K;
    Pre cur, nxt;
    prologue<T, MODE, HASZ>(st, 0, lane, c, cur);
    for (int sb = 0; sb < nsb; ++sb) {
        prologue<T, MODE, HASZ>(st, (sb + 1) * K, lane, c, nxt);
        recur<T, MODE, false>(st, sb * K, K, cur, H, S2, yptr, ystride, c.valid);
        cur = nxt;
    }
    const int rem = nvalid - nsb * K;
    if (rem > 0) recur<T, MODE, true>(st, nsb * K, rem, cur, H, S2, yptr, ystride, c.valid);
}

// Any other A (including zeros): per state, A_bar - 1 = 2^(dl A) - 1 and
// B_bar/B = (A_bar - 1)/A, or dt where A == 0.  Correct, not tuned.
template <typename T, int MODE, bool HASZ>
__device__ __forceinline__ void run_stage_general(const unsigned char* st, int nvalid, int lane,
                                                  const Chan& c, const float* __restrict__ Arow,
                                                  float2 (&H)[NS / 2], float& S2,
                                                  T* __restrict__ yptr, long long ystride) {
    using Lt = Layout<T>;
    const T* U = reinterpret_cast<const T*>(st + Lt::offU);
    const T* Dl = reinterpret_cast<const T*>(st + Lt::offD);
    const T* Z = reinterpret_cast<const T*>(st + Lt::offZ);
    const float* Bc = reinterpret_cast<const float*>(st + Lt::offBc);
    const float* Cc = reinterpret_cast<const float*>(st + Lt::offCc);
    for (int tt = 0; tt < nvalid; ++tt) {
        const float u = ld_elem(U + tt * CH + lane);
        const float dv = ld_elem(Dl + tt * CH + lane);
        const float dl = ptx::lg2(1.0f + ptx::ex2(fmaf(dv, kLog2e, c.kb2)));
        const float dt = dl * kLn2;
        if (MODE == kAggregate) S2 += dl;
        float y = 0.0f;
#pragma unroll
        for (int n = 0; n < NS; ++n) {
            const float a = __ldg(Arow + n);
            const float e = ptx::ex2(dl * a) - 1.0f;
            const float coef = (a != 0.0f) ? e / a : dt;
            const float bn = Bc[tt * NS + n] * (float)(n + 1);
            float hn = (n & 1) ? H[n / 2].y : H[n / 2].x;
            hn = fmaf(coef * bn, u, fmaf(e, hn, hn));
            if (n & 1) H[n / 2].y = hn; else H[n / 2].x = hn;
            if (MODE != kAggregate) y = fmaf(Cc[tt * NS + n], hn, y);
        }
        if (MODE != kAggregate) {
            y = fmaf(c.dsk, u, y);
            if constexpr (HASZ) {
                const float z = ld_elem(Z + tt * CH + lane);
                y *= z * ptx::rcp(1.0f + ptx::ex2(z * -kLog2e));
            }
            if (c.valid) st_elem(yptr + tt * ystride, y);
        }
    }
}

// Producer-side widening of one stage's B and C rows (TC x NS each) to
// float32, B scaled by 1/(n+1).  Lane l handles element pairs l, l+32, ...:
// consecutive lanes touch consecutive words, and every pair a lane handles
// has n = 2*(l % 8) + {0, 1}.
template <typename T, int MODE>
__device__ __forceinline__ void widen_rows(unsigned char* st, int lane) {
    using Lt = Layout<T>;
    constexpr int kElemPairs = TC * NS / 2;
    const int n0 = 2 * (lane % (NS / 2));
    const float s0 = 1.0f / (float)(n0 + 1), s1 = 1.0f / (float)(n0 + 2);
    const T* Br = reinterpret_cast<const T*>(st + Lt::offBr);
    const T* Cr = reinterpret_cast<const T*>(st + Lt::offCr);
    float2* Bc = reinterpret_cast<float2*>(st + Lt::offBc);
    float2* Cc = reinterpret_cast<float2*>(st + Lt::offCc);
#pragma unroll
    for (int i = 0; i < kElemPairs / 32; ++i) {
        const int w = lane + 32 * i;
        Bc[w] = make_float2(ld_elem(Br + 2 * w) * s0, ld_elem(Br + 2 * w + 1) * s1);
        if (MODE != kAggregate) Cc[w] = make_float2(ld_elem(Cr + 2 * w), ld_elem(Cr + 2 * w + 1));
    }
}

template <typename T, int MODE>
__global__ void __launch_bounds__(Layout<T>::kThreads, 1)
scan_fast_kernel(const __grid_constant__ CUtensorMap tmU, const __grid_constant__ CUtensorMap tmD,
                 const __grid_constant__ CUtensorMap tmZ, const __grid_constant__ CUtensorMap tmB,
                 const __grid_constant__ CUtensorMap tmC, const Params p) {
    using Lt = Layout<T>;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // A CTA is kPairs independent workers; worker i is consumer warp i and
    // producer warp kPairs + i.  When the CTA is alone on its SM, warp w runs
    // on SM sub-partition w % 4, so with four pairs every sub-partition gets
    // one consumer (the recurrence) and one mostly sleeping producer.
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int pair = warp % Lt::kPairs;
    const bool producer = warp >= Lt::kPairs;
    // Stage tiles are TMA destinations: align the carve-out base to 1 KiB
    // (the launch requests kSmemBytes, which includes that slack).
    unsigned char* smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u) +
                          pair * Lt::kPairBytes;
    Meta* meta = reinterpret_cast<Meta*>(smem + Lt::offMeta);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Lt::offBar);
    uint64_t* convd = full + S;
    uint64_t* empty = convd + S;
    const volatile unsigned* vabort = p.abort;

    if (!producer && lane == 0) {
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&convd[s], 32);
            ptx::mbar_init(&empty[s], 1);
        }
        ptx::fence_mbar_init();
    }
    __syncthreads();

    if (producer) {
        // ---------------- producer warp: TMA issue (lane 0) + B/C widening
        if (lane == 0) {
            ptx::prefetch_tensormap(&tmU);
            ptx::prefetch_tensormap(&tmD);
            ptx::prefetch_tensormap(&tmB);
            if (MODE != kAggregate) {
                ptx::prefetch_tensormap(&tmC);
                if (p.has_z) ptx::prefetch_tensormap(&tmZ);
            }
        }
        long long cur_unit = -1, cur_t0 = 0, cur_end = 0, cur_b = 0, cur_d0 = 0;
        long long issued = 0;
        bool issue_done = false, failed = false;
        const uint32_t tile_bytes = Lt::kTile, raw_bytes = Lt::kRaw;
        const uint32_t stage_tx = (MODE == kAggregate)
                                      ? 2 * tile_bytes + raw_bytes
                                      : 2 * tile_bytes + 2 * raw_bytes + (p.has_z ? tile_bytes : 0);
        for (long long j = 0;; ++j) {
            while (!issue_done && !failed && issued <= j + LA) {
                const int slot = (int)(issued % S);
                if (issued >= S &&
                    !ptx::mbar_wait(&empty[slot], (uint32_t)(((issued / S) - 1) & 1), p.wait_ns,
                                    vabort, kProducerSleepNs)) {
                    failed = true;
                    break;
                }
                unsigned char* st = smem + slot * Lt::kStage;
                int flags = 0;
                if (cur_unit < 0 || cur_t0 >= cur_end) {
                    unsigned long long tk = 0;
                    if (lane == 0) tk = atomicAdd(p.ticket, 1ull);
                    tk = __shfl_sync(0xffffffffu, tk, 0);
                    if ((long long)tk >= p.total_units || *vabort) {
                        if (lane == 0) {
                            meta[slot].flags = kEnd;
                            ptx::mbar_arrive(&full[slot]);
                        }
                        issue_done = true;
                        ++issued;
                        break;
                    }
                    cur_unit = (long long)tk;
                    const long long k = cur_unit / p.nchains, chain = cur_unit % p.nchains;
                    cur_b = chain / p.nCB;
                    cur_d0 = (chain % p.nCB) * CH;
                    cur_t0 = k * p.T;
                    cur_end = cur_t0 + p.T < p.L ? cur_t0 + p.T : p.L;
                    flags |= kFirst;
                }
                const int nvalid = (int)(cur_end - cur_t0 < TC ? cur_end - cur_t0 : TC);
                if (cur_t0 + TC >= cur_end) flags |= kLast;
                if (lane == 0) {
                    meta[slot].unit = cur_unit;
                    meta[slot].t0 = cur_t0;
                    meta[slot].nvalid = nvalid;
                    meta[slot].flags = flags;
                    ptx::mbar_arrive_expect_tx(&full[slot], stage_tx);
                    const int x = (int)cur_d0, yy = (int)cur_t0, z = (int)cur_b;
                    ptx::tma_load_3d(st + Lt::offU, &tmU, &full[slot], x, yy, z);
                    ptx::tma_load_3d(st + Lt::offD, &tmD, &full[slot], x, yy, z);
                    ptx::tma_load_3d(st + Lt::offBr, &tmB, &full[slot], 0, yy, z);
                    if (MODE != kAggregate) {
                        if (p.has_z) ptx::tma_load_3d(st + Lt::offZ, &tmZ, &full[slot], x, yy, z);
                        ptx::tma_load_3d(st + Lt::offCr, &tmC, &full[slot], 0, yy, z);
                    }
                }
                __syncwarp();
                cur_t0 += TC;
                ++issued;
            }
            if (failed || j >= issued) break;
            const int slot = (int)(j % S);
            if (!ptx::mbar_wait(&full[slot], (uint32_t)((j / S) & 1), p.wait_ns, vabort,
                                kProducerSleepNs)) {
                failed = true;
                break;
            }
            const int fl = meta[slot].flags;
            if (!(fl & kEnd)) widen_rows<T, MODE>(smem + slot * Lt::kStage, lane);
            ptx::mbar_arrive(&convd[slot]);
            if (fl & kEnd) break;
        }
        if (failed) {
            if (lane == 0) {
                atomicOr(&g_error_word, kErrTimeout);
                atomicExch(p.abort, 1u);
            }
        }
        // Never leave with bulk copies in flight: wait (bounded) for every
        // issued stage that was not already waited for above.
        for (long long j = issued - S > 0 ? issued - S : 0; j < issued; ++j)
            ptx::mbar_wait(&full[j % S], (uint32_t)((j / S) & 1), p.wait_ns, nullptr);
        return;
    }

    // ---------------- consumer warp: the recurrence, one channel per lane
    Chan c;
    float2 H[NS / 2];
    float S2 = 0.0f;
    bool geo = true;
    for (long long j = 0;; ++j) {
        const int slot = (int)(j % S);
        if (!ptx::mbar_wait(&convd[slot], (uint32_t)((j / S) & 1), p.wait_ns, vabort)) {
            if (lane == 0) {
                atomicOr(&g_error_word, kErrTimeout);
                atomicExch(p.abort, 1u);
            }
            break;
        }
        const Meta m = meta[slot];
        if (m.flags & kEnd) break;
        if (m.flags & kFirst) {
            c.k = m.unit / p.nchains;
            c.chain = m.unit % p.nchains;
            c.b = c.chain / p.nCB;
            c.d = (c.chain % p.nCB) * CH + lane;
            c.valid = c.d < p.D;
            c.ch = c.b * p.D + c.d;
            const long long dsafe = c.valid ? c.d : 0;
            bool g = true;
            const float a0 = p.A[dsafe * NS];
#pragma unroll
            for (int n = 1; n < NS; ++n) g = g && (p.A[dsafe * NS + n] == (float)(n + 1) * a0);
            g = g && (a0 != 0.0f) && isfinite(a0);
            geo = __all_sync(0xffffffffu, g || !c.valid);
            c.a0 = a0;
            c.ia0 = (a0 != 0.0f) ? 1.0f / a0 : 0.0f;
            c.kb2 = (p.dt_bias ? p.dt_bias[dsafe] : 0.0f) * kLog2e;
            c.dsk = p.Dskip ? p.Dskip[dsafe] : 0.0f;
            S2 = 0.0f;
#pragma unroll
            for (int q = 0; q < NS / 2; ++q) H[q] = make_float2(0.f, 0.f);
            if (MODE == kChained && c.k > 0) {
                bool ok = true;
                if (lane == 0) {
                    const uint64_t t0 = ptx::globaltimer();
                    while (ptx::ld_acquire(p.flags + c.chain) < (unsigned)c.k) {
                        ptx::nanosleep(64);
                        if (*vabort || ptx::globaltimer() - t0 > p.wait_ns) {
                            ok = false;
                            break;
                        }
                    }
                    if (!ok) {
                        atomicOr(&g_error_word, kErrTimeout);
                        atomicExch(p.abort, 1u);
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                __threadfence();
                if (ok && c.valid) {
                    const float4* src = reinterpret_cast<const float4*>(p.carry + c.ch * NS);
#pragma unroll
                    for (int q = 0; q < NS / 4; ++q) {
                        const float4 v = __ldcg(src + q);
                        H[2 * q] = make_float2(v.x, v.y);
                        H[2 * q + 1] = make_float2(v.z, v.w);
                    }
                }
            }
            if (MODE == kFromState && c.valid) {
                const float4* src =
                    reinterpret_cast<const float4*>(p.hin + (c.k * p.batch * p.D + c.ch) * NS);
#pragma unroll
                for (int q = 0; q < NS / 4; ++q) {
                    const float4 v = __ldcg(src + q);
                    H[2 * q] = make_float2(v.x, v.y);
                    H[2 * q + 1] = make_float2(v.z, v.w);
                }
            }
        }
        const unsigned char* st = smem + slot * Lt::kStage;
        T* yptr = static_cast<T*>(p.y) + ((c.b * p.L + m.t0) * p.D + (c.valid ? c.d : 0));
        if (geo) {
            if (p.has_z) run_stage_geo<T, MODE, true>(st, m.nvalid, lane, c, H, S2, yptr, p.D);
            else run_stage_geo<T, MODE, false>(st, m.nvalid, lane, c, H, S2, yptr, p.D);
        } else {
            const float* Arow = p.A + (c.valid ? c.d : 0) * NS;
            if (p.has_z)
                run_stage_general<T, MODE, true>(st, m.nvalid, lane, c, Arow, H, S2, yptr, p.D);
            else
                run_stage_general<T, MODE, false>(st, m.nvalid, lane, c, Arow, H, S2, yptr, p.D);
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&empty[slot]);
        if (m.flags & kLast) {
            if (MODE == kChained) {
                if (c.valid) {
                    float4* dst = reinterpret_cast<float4*>(p.carry + c.ch * NS);
#pragma unroll
                    for (int q = 0; q < NS / 4; ++q)
                        __stcg(dst + q, make_float4(H[2 * q].x, H[2 * q].y, H[2 * q + 1].x,
                                                    H[2 * q + 1].y));
                }
                __threadfence();
                __syncwarp();
                if (lane == 0 && !p.test_stall)
                    ptx::st_release(p.flags + c.chain, (unsigned)(c.k + 1));
            } else if (MODE == kAggregate) {
                if (c.valid) {
                    float* dst = p.agg + (c.k * p.batch * p.D + c.ch) * (NS + 1);
                    dst[0] = S2;
#pragma unroll
                    for (int q = 0; q < NS / 2; ++q) {
                        dst[1 + 2 * q] = H[q].x;
                        dst[2 + 2 * q] = H[q].y;
                    }
                }
            } else {
                if (c.valid && p.h_last && c.k == p.P - 1) {
                    float4* dst = reinterpret_cast<float4*>(p.h_last + c.ch * NS);
#pragma unroll
                    for (int q = 0; q < NS / 4; ++q)
                        dst[q] = make_float4(H[2 * q].x, H[2 * q].y, H[2 * q + 1].x,
                                             H[2 * q + 1].y);
                }
            }
        }
    }
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
    for (long long k = 0; k < P; ++k) {
        hin[(k * nch + ch) * NS + n] = h;
        if (k + 1 < P) {
            const float* g = agg + (k * nch + ch) * (NS + 1);
            h = fmaf(exp2f(a * g[0]), h, g[1 + n]);
        }
    }
}

}  // namespace fast
}  // namespace ssm
