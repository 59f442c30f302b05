// scan_tile_host.cuh -- plan choice, TMA descriptors, stream-ordered workspace
// and launches for the N == 16 selective-scan kernel (scan_tile.cuh).
#pragma once

#include <cuda.h>

#include <cstdlib>
#include <cstring>
#include <mutex>

#include "../../include/ssmscan.h"
#include "context.cuh"
#include "faults.cuh"
#include "scan_tile.cuh"
#include "tma_host.cuh"

namespace ssm {
namespace tile {

// Rank-3 map over a row-major [batch, L, inner] tensor, box {box_inner, box_t, 1}
// (through the encode cache: a caller that reuses its buffers encodes once).
template <typename T>
inline bool make_map(CUtensorMap* m, const void* base, long long inner, long long L,
                     long long batch, unsigned box_inner, unsigned box_t) {
    const cuuint64_t es = sizeof(T);
    const cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)L, (cuuint64_t)batch};
    const cuuint64_t strides[2] = {(cuuint64_t)inner * es, (cuuint64_t)inner * (cuuint64_t)L * es};
    const cuuint32_t box[3] = {box_inner, box_t, 1u};
    const CUtensorMapDataType dt = sizeof(T) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                  : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    return tma::cached_map(m, dt, 3, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

inline long long env_ll(const char* name, long long dflt) {
    const char* v = std::getenv(name);
    if (!v || !*v) return dflt;
    return std::strtoll(v, nullptr, 10);
}

// Plan names accepted by SSM_FORCE_PLAN (development and tests).
enum Plan { kPlanAuto = 0, kPlanGeneric = 1, kPlanChained = 2, kPlanNarrow = 3 };

inline int forced_plan() {
    const char* v = std::getenv("SSM_FORCE_PLAN");
    if (!v) return kPlanAuto;
    if (!std::strcmp(v, "generic")) return kPlanGeneric;
    if (!std::strcmp(v, "chained")) return kPlanChained;
    if (!std::strcmp(v, "narrow")) return kPlanNarrow;
    return kPlanAuto;
}

inline long long cdiv(long long a, long long b) { return (a + b - 1) / b; }

// Sets the kernel's shared-memory limit and returns in *workers the number of
// CTAs that can be resident at once.  Done once per device, context and
// kernel (a kernel's attributes belong to its context: in a context made
// after the last one was destroyed, the limit is set again); later calls
// read the cached count.
template <typename T, int MODE, int DISC, bool CONV = false>
inline cudaError_t prepare(int sms, long long* workers) {
    constexpr int kMaxDev = 64;
    static std::mutex mu;
    struct Slot {
        unsigned long long ctx;   // context ID
        long long workers;
    };
    static Slot cached[kMaxDev] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    unsigned long long ctx = context::current_id();
    if (ctx && dev >= 0 && dev < kMaxDev) {
        std::lock_guard<std::mutex> lock(mu);
        if (cached[dev].ctx == ctx && cached[dev].workers > 0) {
            *workers = cached[dev].workers;
            return cudaSuccess;
        }
    }
    auto kern = scan_tile_kernel<T, MODE, DISC, CONV>;
    const int smem = Cfg<T>::kSmemBytes;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, THREADS, smem);
    if (e != cudaSuccess) return e;
    *workers = (long long)sms * occ;
    ctx = context::current_id();   // current now
    if (ctx && dev >= 0 && dev < kMaxDev && *workers > 0) {
        std::lock_guard<std::mutex> lock(mu);
        cached[dev] = Slot{ctx, *workers};
    }
    return cudaSuccess;
}

// CTAs of the chained plan's static split.  With no more chains than
// resident CTAs each CTA takes one whole chain; otherwise every resident CTA
// takes an equal share of the chain-major stage space (at least one chain
// each, so a cut chain's first piece is always run first by its holder).
// `piece_steps` > 0 (development and tests) asks for pieces of about that many
// steps instead, which cuts chains into consecutive pieces.
template <typename T>
inline long long chained_grid(long long nchains, long long workers, long long L,
                              long long piece_steps) {
    constexpr long long TC = Cfg<T>::TC;
    const long long nst = cdiv(L, TC);
    long long g = nchains <= workers ? nchains : workers;
    if (piece_steps > 0) {
        const long long want = cdiv(nchains * nst * TC, piece_steps);
        g = want < workers ? want : workers;
    }
    if (g > nchains * nst) g = nchains * nst;
    return g < 1 ? 1 : g;
}

// Bytes of the workspace header: two tickets, the abort word, then one flag
// per 32-channel sub-block, rounded to 256.
inline size_t header_bytes(long long batch, long long D) {
    return ((256 + (size_t)(batch * cdiv(D, CW)) * 4) + 255) & ~(size_t)255;
}

template <typename T, int MODE, int DISC, bool CONV = false>
inline cudaError_t launch_mode(long long grid, const CUtensorMap* maps, const Params& p,
                               cudaStream_t s) {
    if (fault::launch_refused()) return cudaErrorLaunchFailure;
    scan_tile_kernel<T, MODE, DISC, CONV><<<(unsigned)grid, THREADS, Cfg<T>::kSmemBytes, s>>>(
        maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], p);
    return cudaGetLastError();
}

// Fills the tensor maps and the fields of Params shared by every plan.
template <typename T>
inline bool setup(CUtensorMap* maps, Params* p, const T* u, const T* delta, const float* dt_bias,
                  const float* A, const T* Bm, const T* Cm, const float* Dskip, const T* z,
                  T* y, float* h_last, long long batch, long long L, long long D) {
    constexpr unsigned TC = Cfg<T>::TC;
    if (!make_map<T>(&maps[0], u, D, L, batch, CB, TC) ||
        !make_map<T>(&maps[1], delta, D, L, batch, CB, TC) ||
        !make_map<T>(&maps[2], z ? z : u, D, L, batch, CB, TC) ||
        !make_map<T>(&maps[3], Bm, NS, L, batch, NS, TC) ||
        !make_map<T>(&maps[4], Cm, NS, L, batch, NS, TC) ||
        !make_map<T>(&maps[5], y, D, L, batch, CW, TC))
        return false;
    *p = Params{};
    p->y = y;
    p->u = u;
    p->Bm = Bm;
    p->h_last = h_last;
    p->dt_bias = dt_bias;
    p->A = A;
    p->Dskip = Dskip;
    p->has_z = z != nullptr;
    p->test_stall = env_ll("SSM_TEST_STALL_CHAIN", 0) != 0;
    p->batch = batch;
    p->L = L;
    p->D = D;
    p->nCB = cdiv(D, CB);
    p->nSB = cdiv(D, CW);
    p->nchains = batch * p->nCB;
    p->nst = cdiv(L, Cfg<T>::TC);
    p->Wst = p->nchains * p->nst;
    p->wait_ns = (unsigned long long)env_ll("SSM_WAIT_LIMIT_NS", 2000000000LL);
    return true;
}

// Returns an ssm_status_t.  Preconditions (checked by the caller): N == 16,
// u, delta, z, B, C, y, A and h_last 16-byte aligned, D * sizeof(T) % 16 == 0,
// batch*D > 0, L > 0.
// CONV: u is x, convolved with conv_w/conv_b (act: SiLU) before the scan.
// ckpt_only (zero-order hold without the convolution, the chained plan, ckpt
// given): only the checkpoints are written (kCkptOnly; y and h_last are not).
template <typename T, int DISC, bool CONV = false>
int launch_scan_tile(const T* u, const T* delta, const float* dt_bias, const float* A,
                     const T* Bm, const T* Cm, const float* Dskip, const T* z, T* y,
                     float* h_last, long long batch, long long L, long long D, int plan,
                     cudaStream_t stream, const float* conv_w = nullptr,
                     const float* conv_b = nullptr, int act = 0, float* ckpt = nullptr,
                     bool ckpt_only = false) {
    constexpr long long TC = Cfg<T>::TC;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return SSM_ERR_CUDA;
    long long wc = 0, wa = 0, wf = 0;
    if (ckpt_only) h_last = nullptr;   // not written; nor used to hand states over
    if constexpr (DISC == kZOH && !CONV) {
        if (ckpt_only) {
            if (!ckpt || plan != kPlanChained) return SSM_ERR_UNSUPPORTED;
            if (prepare<T, (int)kCkptOnly, DISC, CONV>(sms, &wc) != cudaSuccess || wc < 1)
                return SSM_ERR_CUDA;
        }
    } else {
        if (ckpt_only) return SSM_ERR_UNSUPPORTED;
    }
    if (prepare<T, (int)kChained, DISC, CONV>(sms, &wc) != cudaSuccess ||
        prepare<T, (int)kAggregate, DISC, CONV>(sms, &wa) != cudaSuccess ||
        prepare<T, (int)kFromState, DISC, CONV>(sms, &wf) != cudaSuccess || wc < 1 || wa < 1 ||
        wf < 1)
        return SSM_ERR_CUDA;

    CUtensorMap maps[6];
    Params p;
    if (!setup<T>(maps, &p, u, delta, dt_bias, A, Bm, Cm, Dskip, z, y, h_last, batch, L, D))
        return SSM_ERR_CUDA;
    p.conv_w = conv_w;
    p.conv_b = conv_b;
    p.act = act;
    p.ckpt = ckpt;

    bool narrow = false;
    if (plan == kPlanNarrow) narrow = true;
    else if (plan == kPlanAuto) narrow = p.nchains * 100 < wc * 55;
    const long long forced_steps = env_ll("SSM_CHUNK_T", 0);
    if (narrow) {
        // About four units per resident CTA of the output pass, and no more:
        // the units are of equal length and taken from a ticket, so a count
        // just past a multiple of the CTAs leaves a last round with most of
        // them idle (12 chains x 50 units on 148 CTAs ran as 5 rounds of
        // work for 4.05 rounds' worth; 12 x 49 fits in 4).
        const long long P0 = (4 * (wf < wa ? wf : wa)) / p.nchains;
        long long steps = cdiv(cdiv(L, P0 < 2 ? 2 : P0), TC) * TC;
        if (forced_steps > 0) steps = cdiv(forced_steps, TC) * TC;
        if (steps < TC) steps = TC;
        p.T = steps;
        p.P = cdiv(L, steps);
        if (p.P < 2) narrow = false;
    }
    if (!narrow) p.G = chained_grid<T>(p.nchains, wc, L, forced_steps);

    // Workspace: [0,8) phase-A ticket, [16,24) phase-B ticket, [32,36) abort,
    // [256, 256 + 4*batch*nSB) sub-block flags, then the state buffers.
    const long long nch = batch * D;
    const size_t head = header_bytes(batch, D);
    size_t bytes = head;
    size_t off_carry = 0, off_agg = 0, off_hin = 0;
    if (!narrow) {
        if (!h_last) {
            off_carry = bytes;
            bytes += (size_t)nch * NS * 4;
        }
    } else {
        off_agg = bytes;
        bytes += (size_t)(p.P - 1) * nch * (NS + 1) * 4;
        bytes = (bytes + 255) & ~(size_t)255;
        off_hin = bytes;
        bytes += (size_t)p.P * nch * NS * 4;
    }
    unsigned char* ws = nullptr;
    if (fault::malloc_async(reinterpret_cast<void**>(&ws), bytes, stream) != cudaSuccess) {
        cudaGetLastError();
        return SSM_ERR_NOMEM;
    }
    int status = SSM_OK;
    do {
        if (cudaMemsetAsync(ws, 0, head, stream) != cudaSuccess) {
            status = SSM_ERR_CUDA;
            break;
        }
        p.abort = reinterpret_cast<unsigned*>(ws + 32);
        p.flags = reinterpret_cast<unsigned*>(ws + 256);
        if (!narrow) {
            p.ticket = reinterpret_cast<unsigned long long*>(ws);
            p.carry = h_last ? h_last : reinterpret_cast<float*>(ws + off_carry);
            cudaError_t le = cudaSuccess;
            if constexpr (DISC == kZOH && !CONV) {
                if (ckpt_only) {
                    le = launch_mode<T, (int)kCkptOnly, DISC, CONV>(p.G, maps, p, stream);
                } else {
                    le = launch_mode<T, (int)kChained, DISC, CONV>(p.G, maps, p, stream);
                }
            } else {
                le = launch_mode<T, (int)kChained, DISC, CONV>(p.G, maps, p, stream);
            }
            if (le != cudaSuccess) status = SSM_ERR_CUDA;
        } else {
            p.agg = reinterpret_cast<float*>(ws + off_agg);
            p.hin = reinterpret_cast<float*>(ws + off_hin);
            p.ticket = reinterpret_cast<unsigned long long*>(ws);
            p.total_units = p.nchains * (p.P - 1);
            if (launch_mode<T, (int)kAggregate, DISC, CONV>(
                    p.total_units < wa ? p.total_units : wa, maps, p, stream) != cudaSuccess) {
                status = SSM_ERR_CUDA;
                break;
            }
            const long long threads = nch * NS;
            if (fault::launch_refused()) {
                status = SSM_ERR_CUDA;
                break;
            }
            carry_kernel<<<(unsigned)cdiv(threads, 256), 256, 0, stream>>>(
                p.agg, A, reinterpret_cast<float*>(ws + off_hin), batch, D, p.P);
            if (cudaGetLastError() != cudaSuccess) {
                status = SSM_ERR_CUDA;
                break;
            }
            p.ticket = reinterpret_cast<unsigned long long*>(ws + 16);
            p.total_units = p.nchains * p.P;
            if (launch_mode<T, (int)kFromState, DISC, CONV>(
                    p.total_units < wf ? p.total_units : wf, maps, p, stream) != cudaSuccess)
                status = SSM_ERR_CUDA;
        }
    } while (0);
    if (cudaFreeAsync(ws, stream) != cudaSuccess && status == SSM_OK) status = SSM_ERR_CUDA;
    return status;
}

}  // namespace tile
}  // namespace ssm
