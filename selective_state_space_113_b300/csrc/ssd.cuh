// ssd.cuh -- the Mamba-2 form of the scan (structured state-space duality):
// one scalar A per head, the input term dt B x, head dimension P, a state of
// N per channel shared across the head's P channels through B and C.
//
// What it computes (news.han.ihouse.idv.tw article 1304: Mamba-2 found most
// of the SSM's computation equal to a masked matrix multiplication, reduced A
// to a scalar and supports a larger state; Mamba-2 discretises with Euler's
// rule; ta-paperlens and ultralytics pages: Mamba-2's state-space duality),
// per batch b, head h, channel p of the head, step t, state n:
//   dt_t = softplus(dt[b,t,h] + dt_bias[h]);  h_t[n] = exp(dt_t A[h]) h_{t-1}[n]
//          + dt_t B_t[n] x_t[p];   y_t[p] = sum_n C_t[n] h_t[n] + Dskip[h] x_t[p]
// from h = 0.  The tensor-core kernel evaluates it in the chunked matrix form
// (chunks of Q = 64 steps, cum_t = A sum_{r<=t in chunk} dt_r):
//   y_chunk = (Lmask o C B^T) X + diag(exp(cum)) C H_in + Dskip X,
//     Lmask[t, s] = exp(cum_t - cum_s) dt_s  for s <= t, 0 above the diagonal
//   H_out = exp(cum_end) H_in + B^T (w o X),   w_s = exp(cum_end - cum_s) dt_s
// with H the N x P state of the head.  One CTA (4 warps) owns one (b, h) and
// walks its chunks in order, the fp32 state in registers (warp w holds state
// rows (N/4)w .. (N/4)(w+1)-1 as mma accumulators).  The four products run on the
// tensor cores as bf16 x bf16 -> fp32 m16n8k16 mma: C B^T (K = N), the masked
// scores times X (K = Q, causal: warp w, which owns steps 16w..16w+15, needs
// only the first w+1 key tiles), C H_in (K = N) and B^T (w o X) (K = Q; the
// B^T fragments come straight from the B tile by transposing ldmatrix).  The
// masked scores, w o X and H_in are rounded to bf16 for their products
// (relative 2^-9); every sum is fp32.  The scores are formed two key tiles at
// a time, so that a CTA needs few enough registers (and, with no transposed
// copy of B, little enough shared memory) for three CTAs to share an SM.
#pragma once

#include "common.cuh"
#include "faults.cuh"
#include "ptx.cuh"

namespace ssm {
namespace ssd {

constexpr int Q = 64;      // steps per chunk
constexpr int P = 64;      // head dimension
constexpr int THREADS = 128;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t ld32(const bf16* p) {
    return *reinterpret_cast<const uint32_t*>(p);
}

// Four 8x8 bf16 tiles from shared memory, transposed: lane i gives the
// address of row i % 8 of tile i / 8 (16 contiguous bytes, 16-byte aligned);
// lane l receives (row 2(l%4), column l/4) and (row 2(l%4)+1, column l/4) of
// each tile.  Read from a [k][m] array this is the A fragment of a
// [m][k] = [k][m]^T operand.
__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], const bf16* row_addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(ptx::smem_u32(row_addr)));
}

// Splits a, b into bf16 pairs hi + lo (hi = bf16(v), lo = bf16(v - hi)), so
// that hi + lo carries about 16 significant bits: a product with an exact
// bf16 operand taken as hi x + lo x keeps that accuracy.
__device__ __forceinline__ void split_pack(float a, float b, uint32_t& hi, uint32_t& lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    const __nv_bfloat162 l = __floats2bfloat162_rn(a - __low2float(h), b - __high2float(h));
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = *reinterpret_cast<const uint32_t*>(&l);
}

constexpr int PH = 32;   // channels of the head per CTA (two CTAs per head)

// 16-byte asynchronous copy global -> shared; with valid false it reads
// nothing and writes zeros (src-size 0).
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(ptx::smem_u32(smem_dst)),
                 "l"(gsrc), "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Shared-memory layout; every row is padded by 8 elements so that the eight
// rows a fragment load touches fall in different banks.
template <int N>
struct Smem {
    static constexpr int NP = N + 8, QP = Q + 8;
    bf16 Xt[PH][QP];                // x of the chunk, transposed: [p][s]
    bf16 Xwh[PH][QP], Xwl[PH][QP];  // w o x, transposed, as hi + lo bf16 parts
    bf16 Cs[Q][NP];                 // C rows: [t][n]
    // Two buffers that take turns: one holds the chunk's B rows [s][n], the
    // other the state entering it, [p][n] hi in rows 0..PH-1 and lo in rows
    // PH..2PH-1.  While the state is updated, the next chunk's B rows stream
    // into the (spent) state buffer; the new state then goes into the B one.
    bf16 Pb[2][Q][NP];
    float dts[Q], cum[Q], w[Q], ecum[Q];
};

template <int N>
__global__ void __launch_bounds__(THREADS, 3)
ssd_chunk_kernel(const bf16* __restrict__ x, const bf16* __restrict__ dtr,
                 const float* __restrict__ dt_bias, const float* __restrict__ A,
                 const bf16* __restrict__ Bm, const bf16* __restrict__ Cm,
                 const float* __restrict__ Dskip, bf16* __restrict__ y, float* __restrict__ h_last,
                 long long batch, long long L, long long H) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Smem<N>& sm = *reinterpret_cast<Smem<N>*>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, tq = lane & 3;
    const long long hb = blockIdx.x / (P / PH);
    const int pbase = (int)(blockIdx.x % (P / PH)) * PH;   // this CTA's channels of the head
    const long long b = hb / H, hh = hb % H;
    const float a = A[hh];
    const float kb2 = dt_bias ? dt_bias[hh] * kLog2e : 0.0f;
    const float dsk = Dskip ? Dskip[hh] : 0.0f;
    static_assert(N == 64 || N == 128, "state size");
    constexpr int NT = PH / 8;     // n-tiles over the CTA's channels
    constexpr int RW = N / 4;      // state rows per warp
    constexpr int MTW = RW / 16;   // state m-tiles per warp
    float Hs[MTW][NT][4];          // state rows RW*warp + 16*mt + {g, g+8}, cols 8*nt + 2tq + {0,1}
#pragma unroll
    for (int mt = 0; mt < MTW; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) Hs[mt][nt][i] = 0.0f;
    static_assert(Q == 2 * PH, "a state buffer (hi + lo) has the shape of a B tile");
    int cb = 0;   // the buffer holding the current chunk's B rows; 1 - cb holds its state
    for (int i = tid; i < Q * (N + 8); i += THREADS) (&sm.Pb[1][0][0])[i] = __float2bfloat16_rn(0.0f);

    const long long nchunks = (L + Q - 1) / Q;
    // Staging of a chunk: x transposed into Xt, B and C rows, dt after the
    // softplus; rows past the sequence are zero.  Chunk 0 is staged here; a
    // later chunk's C rows (by cp.async), x and dt (in registers) are fetched
    // while the chunk before it updates its state, and its B rows after.
    auto x_item = [&](int i, int& s, int& p8) {
        s = i / (PH / 8);
        p8 = (i % (PH / 8)) * 8;
    };
    auto load_x = [&](long long tc, int nvc, int i) {
        int s, p8;
        x_item(i, s, p8);
        return s < nvc ? *reinterpret_cast<const uint4*>(x + ((b * L + tc + s) * H + hh) * P + pbase + p8)
                       : make_uint4(0, 0, 0, 0);
    };
    auto store_x = [&](int i, const uint4& v) {
        int s, p8;
        x_item(i, s, p8);
        const bf16* e = reinterpret_cast<const bf16*>(&v);
#pragma unroll
        for (int k = 0; k < 8; ++k) sm.Xt[p8 + k][s] = e[k];
    };
    auto load_dt = [&](long long tc, int nvc) {
        float d = 0.0f;
        if (tid < nvc) {
            const float v2 = fmaf(__bfloat162float(dtr[(b * L + tc + tid) * H + hh]), kLog2e, kb2);
            d = (v2 > 28.853901f ? v2 : ptx::lg2(1.0f + ptx::ex2(v2))) * 0.6931471805599453f;
        }
        return d;
    };
    auto load_rows = [&](const bf16* src, bf16 (*dst)[N + 8], long long tc, int nvc) {
        for (int i = tid; i < Q * (N / 8); i += THREADS) {
            const int s = i / (N / 8), n8 = (i % (N / 8)) * 8;
            *reinterpret_cast<uint4*>(&dst[s][n8]) =
                s < nvc ? *reinterpret_cast<const uint4*>(src + (b * L + tc + s) * N + n8)
                        : make_uint4(0, 0, 0, 0);
        }
    };
    constexpr int XPT = Q * (PH / 8) / THREADS;   // x items per thread
    static_assert(Q * (PH / 8) % THREADS == 0, "x staging");
    {
        const int nv0 = (int)(L < Q ? L : Q);
#pragma unroll
        for (int k = 0; k < XPT; ++k) store_x(tid + THREADS * k, load_x(0, nv0, tid + THREADS * k));
        load_rows(Bm, sm.Pb[0], 0, nv0);
        load_rows(Cm, sm.Cs, 0, nv0);
        if (tid < Q) sm.dts[tid] = load_dt(0, nv0);
    }
    for (long long c = 0; c < nchunks; ++c) {
        const long long t0 = c * Q;
        const int nv = (int)(L - t0 < Q ? L - t0 : Q);
        __syncthreads();
        // ---- cumulative decay (warp 0: a scan over 64 steps, two per lane)
        if (warp == 0) {
            const float d0 = sm.dts[2 * lane] * a, d1 = sm.dts[2 * lane + 1] * a;
            float sc = d0 + d1;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float v = __shfl_up_sync(0xffffffffu, sc, o);
                if (lane >= o) sc += v;
            }
            const float c1 = sc, c0 = sc - d1;   // inclusive sums at steps 2*lane, 2*lane+1
            const float cend = __shfl_sync(0xffffffffu, sc, 31);
            sm.cum[2 * lane] = c0;
            sm.cum[2 * lane + 1] = c1;
            sm.ecum[2 * lane] = ptx::ex2(c0 * kLog2e);
            sm.ecum[2 * lane + 1] = ptx::ex2(c1 * kLog2e);
            sm.w[2 * lane] = ptx::ex2((cend - c0) * kLog2e) * sm.dts[2 * lane];
            sm.w[2 * lane + 1] = ptx::ex2((cend - c1) * kLog2e) * sm.dts[2 * lane + 1];
        }
        __syncthreads();
        // ---- w o x, transposed, hi + lo
        for (int i = tid; i < Q * PH; i += THREADS) {
            const int pp = i / Q, s = i % Q;
            const float v = __bfloat162float(sm.Xt[pp][s]) * sm.w[s];
            const bf16 hi = __float2bfloat16_rn(v);
            sm.Xwh[pp][s] = hi;
            sm.Xwl[pp][s] = __float2bfloat16_rn(v - __bfloat162float(hi));
        }
        // ---- outputs of this warp's 16 steps: exp(cum_t) C_t H_in + masked scores X + D x
        {
            const int r0 = 16 * warp;
            float Y[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) Y[nt][i] = 0.0f;
            // C H_in (K = N), H_in as hi + lo
#pragma unroll
            for (int k0 = 0; k0 < N; k0 += 16) {
                const uint32_t a0 = ld32(&sm.Cs[r0 + g][k0 + 2 * tq]);
                const uint32_t a1 = ld32(&sm.Cs[r0 + g + 8][k0 + 2 * tq]);
                const uint32_t a2 = ld32(&sm.Cs[r0 + g][k0 + 2 * tq + 8]);
                const uint32_t a3 = ld32(&sm.Cs[r0 + g + 8][k0 + 2 * tq + 8]);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const bf16 (*Hb)[N + 8] = sm.Pb[1 - cb];
                    mma16816(Y[nt], a0, a1, a2, a3, ld32(&Hb[8 * nt + g][k0 + 2 * tq]),
                             ld32(&Hb[8 * nt + g][k0 + 2 * tq + 8]));
                    mma16816(Y[nt], a0, a1, a2, a3, ld32(&Hb[PH + 8 * nt + g][k0 + 2 * tq]),
                             ld32(&Hb[PH + 8 * nt + g][k0 + 2 * tq + 8]));
                }
            }
            const float e_lo = sm.ecum[r0 + g], e_hi = sm.ecum[r0 + g + 8];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                Y[nt][0] *= e_lo;
                Y[nt][1] *= e_lo;
                Y[nt][2] *= e_hi;
                Y[nt][3] *= e_hi;
            }
            // scores S = C B^T, two key tiles (16 keys) at a time up to the
            // diagonal; masked, decayed, split hi + lo and multiplied into X
            const int tlo = r0 + g, thi = r0 + g + 8;
            const float clo = sm.cum[tlo], chi = sm.cum[thi];
#pragma unroll
            for (int kt = 0; kt < 4; ++kt) {
                if (kt <= warp) {
                    float S[2][4];
#pragma unroll
                    for (int jj = 0; jj < 2; ++jj)
#pragma unroll
                        for (int i = 0; i < 4; ++i) S[jj][i] = 0.0f;
#pragma unroll
                    for (int k0 = 0; k0 < N; k0 += 16) {
                        const uint32_t a0 = ld32(&sm.Cs[r0 + g][k0 + 2 * tq]);
                        const uint32_t a1 = ld32(&sm.Cs[r0 + g + 8][k0 + 2 * tq]);
                        const uint32_t a2 = ld32(&sm.Cs[r0 + g][k0 + 2 * tq + 8]);
                        const uint32_t a3 = ld32(&sm.Cs[r0 + g + 8][k0 + 2 * tq + 8]);
#pragma unroll
                        for (int jj = 0; jj < 2; ++jj) {
                            const int j = 2 * kt + jj;
                            mma16816(S[jj], a0, a1, a2, a3, ld32(&sm.Pb[cb][8 * j + g][k0 + 2 * tq]),
                                     ld32(&sm.Pb[cb][8 * j + g][k0 + 2 * tq + 8]));
                        }
                    }
                    // S[t][s] *= exp(cum_t - cum_s) dt_s for s <= t, else 0
#pragma unroll
                    for (int jj = 0; jj < 2; ++jj) {
                        const int s0 = 16 * kt + 8 * jj + 2 * tq, s1 = s0 + 1;
                        const float cs0 = sm.cum[s0], cs1 = sm.cum[s1];
                        const float d0 = sm.dts[s0], d1 = sm.dts[s1];
                        S[jj][0] = s0 <= tlo ? S[jj][0] * ptx::ex2((clo - cs0) * kLog2e) * d0 : 0.0f;
                        S[jj][1] = s1 <= tlo ? S[jj][1] * ptx::ex2((clo - cs1) * kLog2e) * d1 : 0.0f;
                        S[jj][2] = s0 <= thi ? S[jj][2] * ptx::ex2((chi - cs0) * kLog2e) * d0 : 0.0f;
                        S[jj][3] = s1 <= thi ? S[jj][3] * ptx::ex2((chi - cs1) * kLog2e) * d1 : 0.0f;
                    }
                    uint32_t h0, l0, h1, l1, h2, l2, h3, l3;
                    split_pack(S[0][0], S[0][1], h0, l0);
                    split_pack(S[0][2], S[0][3], h1, l1);
                    split_pack(S[1][0], S[1][1], h2, l2);
                    split_pack(S[1][2], S[1][3], h3, l3);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        const uint32_t b0 = ld32(&sm.Xt[8 * nt + g][16 * kt + 2 * tq]);
                        const uint32_t b1 = ld32(&sm.Xt[8 * nt + g][16 * kt + 2 * tq + 8]);
                        mma16816(Y[nt], h0, h1, h2, h3, b0, b1);
                        mma16816(Y[nt], l0, l1, l2, l3, b0, b1);
                    }
                }
            }
            // + D x, store
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int p0 = 8 * nt + 2 * tq;
                bf16* yrow = y + pbase + p0;
                if (tlo < nv) {
                    const float x0 = __bfloat162float(sm.Xt[p0][tlo]), x1 = __bfloat162float(sm.Xt[p0 + 1][tlo]);
                    *reinterpret_cast<__nv_bfloat162*>(yrow + ((b * L + t0 + tlo) * H + hh) * P) =
                        __floats2bfloat162_rn(fmaf(dsk, x0, Y[nt][0]), fmaf(dsk, x1, Y[nt][1]));
                }
                if (thi < nv) {
                    const float x0 = __bfloat162float(sm.Xt[p0][thi]), x1 = __bfloat162float(sm.Xt[p0 + 1][thi]);
                    *reinterpret_cast<__nv_bfloat162*>(yrow + ((b * L + t0 + thi) * H + hh) * P) =
                        __floats2bfloat162_rn(fmaf(dsk, x0, Y[nt][2]), fmaf(dsk, x1, Y[nt][3]));
                }
            }
        }
        __syncthreads();   // the state buffer and the C tile: all readers done; Xwh/Xwl written
        // ---- the next chunk's B and C rows (asynchronously), x and dt (in registers)
        const bool more = c + 1 < nchunks;
        const long long tn = t0 + Q;
        const int nvn = more ? (int)(L - tn < Q ? L - tn : Q) : 0;
        uint4 xr[XPT];
        float dr = 0.0f;
        if (more) {
            for (int i = tid; i < Q * (N / 8); i += THREADS) {
                const int s2 = i / (N / 8), n8 = (i % (N / 8)) * 8;
                const bool ok = s2 < nvn;
                const long long row = (b * L + (ok ? tn + s2 : 0)) * N + n8;
                cp_async16(&sm.Cs[s2][n8], Cm + row, ok);
                cp_async16(&sm.Pb[1 - cb][s2][n8], Bm + row, ok);
            }
            cp_async_commit();
#pragma unroll
            for (int k = 0; k < XPT; ++k) xr[k] = load_x(tn, nvn, tid + THREADS * k);
            if (tid < Q) dr = load_dt(tn, nvn);
        }
        // ---- the state: H <- exp(cum_end) H + B^T (w o X)   (K = Q), w o X as hi + lo
        {
            const float dec = sm.ecum[Q - 1];
            const int tile = lane >> 3, row = lane & 7;
#pragma unroll
            for (int mt = 0; mt < MTW; ++mt) {
                const int m0 = RW * warp + 16 * mt;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) Hs[mt][nt][i] *= dec;
#pragma unroll
                for (int k0 = 0; k0 < Q; k0 += 16) {
                    // A = B^T rows m0.., keys k0..: tiles Bs[k0 + 8 (i/16) ..][m0 + 8 ((i/8)&1)]
                    uint32_t af[4];
                    ldsm_x4_trans(af, &sm.Pb[cb][k0 + 8 * (tile >> 1) + row][m0 + 8 * (tile & 1)]);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        mma16816(Hs[mt][nt], af[0], af[1], af[2], af[3],
                                 ld32(&sm.Xwh[8 * nt + g][k0 + 2 * tq]),
                                 ld32(&sm.Xwh[8 * nt + g][k0 + 2 * tq + 8]));
                        mma16816(Hs[mt][nt], af[0], af[1], af[2], af[3],
                                 ld32(&sm.Xwl[8 * nt + g][k0 + 2 * tq]),
                                 ld32(&sm.Xwl[8 * nt + g][k0 + 2 * tq + 8]));
                    }
                }
            }
        }
        __syncthreads();   // every read of this chunk's B rows is done
        // ---- the copy of the state the next chunk reads, [p][n] hi + lo, into the B buffer
        {
#pragma unroll
            for (int mt = 0; mt < MTW; ++mt) {
                const int m0 = RW * warp + 16 * mt;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int p0 = 8 * nt + 2 * tq;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int pp = p0 + (i & 1), mm = m0 + g + 8 * (i >> 1);
                        const float v = Hs[mt][nt][i];
                        const bf16 hi = __float2bfloat16_rn(v);
                        sm.Pb[cb][pp][mm] = hi;
                        sm.Pb[cb][PH + pp][mm] = __float2bfloat16_rn(v - __bfloat162float(hi));
                    }
                }
            }
        }
        if (more) {
#pragma unroll
            for (int k = 0; k < XPT; ++k) store_x(tid + THREADS * k, xr[k]);
            if (tid < Q) sm.dts[tid] = dr;
            cp_async_wait_all();
        }
        cb = 1 - cb;
    }
    if (h_last) {
#pragma unroll
        for (int mt = 0; mt < MTW; ++mt) {
            const int m0 = RW * warp + 16 * mt;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int p0 = pbase + 8 * nt + 2 * tq;
                float* base = h_last + ((b * H + hh) * P) * N;
                base[(long long)p0 * N + m0 + g] = Hs[mt][nt][0];
                base[(long long)(p0 + 1) * N + m0 + g] = Hs[mt][nt][1];
                base[(long long)p0 * N + m0 + g + 8] = Hs[mt][nt][2];
                base[(long long)(p0 + 1) * N + m0 + g + 8] = Hs[mt][nt][3];
            }
        }
    }
}

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

template <int N>
inline cudaError_t launch_ssd_chunk(const bf16* x, const bf16* dt, const float* dt_bias,
                                   const float* A, const bf16* Bm, const bf16* Cm,
                                   const float* Dskip, bf16* y, float* h_last, long long batch,
                                   long long L, long long H, cudaStream_t s) {
    const int smem = (int)sizeof(Smem<N>);
    cudaError_t e = cudaFuncSetAttribute(ssd_chunk_kernel<N>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (fault::launch_refused()) return cudaErrorLaunchFailure;
    ssd_chunk_kernel<N><<<(unsigned)(batch * H * (P / PH)), THREADS, smem, s>>>(
        x, dt, dt_bias, A, Bm, Cm, Dskip, y, h_last, batch, L, H);
    return cudaGetLastError();
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
