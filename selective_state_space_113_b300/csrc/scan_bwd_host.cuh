// scan_bwd_host.cuh -- workspace and launches of the N == 16 backward pass
// (scan_bwd.cuh): the states entering every unit (the caller's checkpoints,
// the chained forward scan, or the forward unit summaries and carry), the
// adjoint summaries and their carry, the unit kernel and the dB/dC
// reduction, all on one stream.
#pragma once

#include "scan_bwd.cuh"
#include "scan_tile_host.cuh"

namespace ssm {
namespace bwd {

inline size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

// CTAs of a kernel resident per SM, set up once per device (shared-memory
// limit raised first where the kernel needs more than 48 KiB).
template <typename K>
inline cudaError_t resident(K kern, int threads, int smem, int* per_sm) {
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
    }
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, kern, threads, smem);
}

// CTAs of a kernel that fit on one SM by its registers, shared memory and
// threads, and by `tmem_cols` columns of the SM's 512 TMEM columns per CTA.
// For kernels that allocate TMEM the occupancy query answers 1 (it cannot
// know how many columns a CTA takes); the allocation itself waits for free
// columns, so this count is what the SM actually holds.
template <typename K>
inline cudaError_t resident_tmem(K kern, int threads, int smem, int tmem_cols, int* per_sm) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaFuncAttributes fa;
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, kern);
    int dev = 0, regs_sm = 0, smem_sm = 0, resv = 0, thr_sm = 0;
    if (e == cudaSuccess) e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&resv, cudaDevAttrReservedSharedMemoryPerBlock, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&thr_sm, cudaDevAttrMaxThreadsPerMultiProcessor, dev);
    if (e != cudaSuccess) return e;
    const int warps = (threads + 31) / 32;
    const int regs_warp = ((fa.numRegs * 32 + 255) / 256) * 256;   // allocated per warp in units of 256
    const int by_regs = regs_sm / (regs_warp * warps);
    const int by_smem = smem_sm / (smem + (int)fa.sharedSizeBytes + resv);
    const int by_thr = thr_sm / (warps * 32);
    const int by_tmem = 512 / tmem_cols;
    int n = by_regs < by_smem ? by_regs : by_smem;
    n = n < by_thr ? n : by_thr;
    n = n < by_tmem ? n : by_tmem;
    *per_sm = n;
    return cudaSuccess;
}

// Returns an ssm_status_t.  Preconditions (checked by the caller): N == 16;
// u, delta, z, dy, B, C, A and du 16-byte aligned; D * sizeof(T) % 16 == 0;
// batch*D > 0; L > 0; dz given when z is.  `plan` is the forward's plan
// choice (kPlanAuto unless forced).
template <typename T>
int launch_scan_bwd16(const T* u, const T* delta, const float* dt_bias, const float* A,
                      const T* Bm, const T* Cm, const float* Dskip, const T* z, const T* dy,
                      const float* dh_last, T* du, T* ddelta, float* ddt_bias, float* dA,
                      float* dB, float* dC, float* dDskip, T* dz, long long batch, long long L,
                      long long D, cudaStream_t stream, const float* ckpt = nullptr,
                      int plan = tile::kPlanAuto) {
    using namespace tile;
    static_assert(TU == kCkptSteps, "checkpoint interval");
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return SSM_ERR_CUDA;
    long long wa = 0, wc = 0;
    if (prepare<T, (int)kAggregate, (int)kZOH>(sms, &wa) != cudaSuccess || wa < 1 ||
        prepare<T, (int)kChained, (int)kZOH>(sms, &wc) != cudaSuccess || wc < 1)
        return SSM_ERR_CUDA;
    // Without the forward pass's checkpoints, the states entering the units
    // come from the forward scan itself when it would run its chained plan
    // (the chains fill the GPU): one pass of its chained walk that writes
    // every unit boundary's state and nothing else (no C, z, readout or y;
    // du only lends its tensor map).
    // That is cheaper than the unit summaries and their carry below, which
    // remain for problems with too few chains, where the forward itself
    // would run them and an output pass besides.
    float* own_ckpt = nullptr;
    if (!ckpt && L > TU && plan != kPlanNarrow &&
        (plan == kPlanChained || batch * cdiv(D, tile::CB) * 100 >= wc * 55)) {
        const size_t bytes = (size_t)cdiv(L, TU) * (size_t)(batch * D) * NS * 4;
        if (fault::malloc_async(reinterpret_cast<void**>(&own_ckpt), bytes, stream) != cudaSuccess) {
            cudaGetLastError();
            return SSM_ERR_NOMEM;
        }
        const int st = launch_scan_tile<T, (int)kZOH>(u, delta, dt_bias, A, Bm, Cm, Dskip, z, du,
                                                      nullptr, batch, L, D, kPlanChained, stream,
                                                      nullptr, nullptr, 0, own_ckpt, true);
        if (st != SSM_OK) {
            cudaFreeAsync(own_ckpt, stream);
            return st;
        }
        ckpt = own_ckpt;
    }
    int occ_sum = 0, occ_unit = 0;
    if (resident(adjoint_summary_kernel<T>, CB, (int)sizeof(AdjSmem<T>), &occ_sum) != cudaSuccess ||
        resident_tmem(bwd_unit_kernel<T>, CB, (int)sizeof(BwdSmem<T>), 128, &occ_unit) != cudaSuccess ||
        occ_sum < 1 || occ_unit < 1)
        return SSM_ERR_CUDA;

    const long long P = cdiv(L, TU);
    const long long nch = batch * D;
    const long long nCB = cdiv(D, CB);
    const size_t head = header_bytes(batch, D);
    size_t off = head;
    // with checkpoints from the forward pass, no unit summaries and no
    // states of our own
    const size_t off_agg = off;
    if (!ckpt) off = round256(off + (size_t)(P > 1 ? P - 1 : 0) * nch * (NS + 1) * 4);
    const size_t off_hin = off;
    if (!ckpt) off = round256(off + (size_t)P * nch * NS * 4);
    const size_t off_adj = off;
    off = round256(off + (size_t)P * nch * (NS + 1) * 4);
    const size_t off_mu = off;
    off = round256(off + (size_t)P * nch * NS * 4);
    const size_t off_part = off;
    off = round256(off + (size_t)nCB * batch * L * 32 * 4);

    unsigned char* ws = nullptr;
    if (fault::malloc_async(reinterpret_cast<void**>(&ws), off, stream) != cudaSuccess) {
        cudaGetLastError();
        if (own_ckpt) cudaFreeAsync(own_ckpt, stream);
        return SSM_ERR_NOMEM;
    }
    int status = SSM_OK;
    do {
        if (cudaMemsetAsync(ws, 0, head, stream) != cudaSuccess ||
            cudaMemsetAsync(dA, 0, (size_t)D * NS * 4, stream) != cudaSuccess ||
            (dDskip && cudaMemsetAsync(dDskip, 0, (size_t)D * 4, stream) != cudaSuccess) ||
            (ddt_bias && cudaMemsetAsync(ddt_bias, 0, (size_t)D * 4, stream) != cudaSuccess)) {
            status = SSM_ERR_CUDA;
            break;
        }
        const float* hin = ckpt ? ckpt : reinterpret_cast<const float*>(ws + off_hin);
        // 1. the states entering every unit (unit 0 starts from zero), unless
        // the forward pass left them
        if (P > 1 && !ckpt) {
            CUtensorMap maps[6];
            Params p;
            if (!setup<T>(maps, &p, u, delta, dt_bias, A, Bm, Cm, Dskip, z, du, nullptr, batch,
                          L, D)) {
                status = SSM_ERR_CUDA;
                break;
            }
            p.T = TU;
            p.P = P;
            p.agg = reinterpret_cast<float*>(ws + off_agg);
            p.ticket = reinterpret_cast<unsigned long long*>(ws);
            p.abort = reinterpret_cast<unsigned*>(ws + 32);
            p.flags = reinterpret_cast<unsigned*>(ws + 256);
            p.total_units = p.nchains * (P - 1);
            if (launch_mode<T, (int)kAggregate, (int)kZOH>(p.total_units < wa ? p.total_units : wa,
                                                          maps, p, stream) != cudaSuccess) {
                status = SSM_ERR_CUDA;
                break;
            }
            if (fault::launch_refused()) {
                status = SSM_ERR_CUDA;
                break;
            }
            carry_kernel<<<(unsigned)cdiv(nch * NS, 256), 256, 0, stream>>>(
                p.agg, A, reinterpret_cast<float*>(ws + off_hin), batch, D, P);
            if (cudaGetLastError() != cudaSuccess) {
                status = SSM_ERR_CUDA;
                break;
            }
        }
        BwdParams bp{};
        bp.u = u;
        bp.delta = delta;
        bp.z = z;
        bp.dy = dy;
        bp.Bm = Bm;
        bp.Cm = Cm;
        bp.dt_bias = dt_bias;
        bp.A = A;
        bp.Dskip = Dskip;
        bp.dh_last = dh_last;
        bp.du = du;
        bp.ddelta = ddelta;
        bp.dz = dz;
        bp.ddt_bias = ddt_bias;
        bp.dA = dA;
        bp.dDskip = dDskip;
        bp.part = reinterpret_cast<float*>(ws + off_part);
        bp.hin = hin;
        bp.adj = reinterpret_cast<float*>(ws + off_adj);
        bp.mu = reinterpret_cast<float*>(ws + off_mu);
        bp.batch = batch;
        bp.L = L;
        bp.D = D;
        bp.P = P;
        bp.nCB = nCB;
        bp.units = nCB * batch * P;
        if (fault::launch_refused()) {
            status = SSM_ERR_CUDA;
            break;
        }
        // 2. adjoint summaries of units 1..P-1, then the adjoint entering each unit
        if (P > 1) {
            const long long nsum = nCB * batch * (P - 1);
            const long long g = (long long)sms * occ_sum;
            adjoint_summary_kernel<T><<<(unsigned)(nsum < g ? nsum : g), CB, sizeof(AdjSmem<T>),
                                        stream>>>(bp);
            if (cudaGetLastError() != cudaSuccess) {
                status = SSM_ERR_CUDA;
                break;
            }
        }
        adj_carry_kernel<<<(unsigned)cdiv(nch * NS, 256), 256, 0, stream>>>(bp.adj, A, dh_last,
                                                                           bp.mu, batch, D, P);
        // 3. the unit kernel
        {
            const long long g = (long long)sms * occ_unit;
            bwd_unit_kernel<T><<<(unsigned)(bp.units < g ? bp.units : g), CB, sizeof(BwdSmem<T>),
                                 stream>>>(bp);
        }
        // 4. dB and dC
        bwd_reduce_bc_kernel<<<(unsigned)cdiv(batch * L * 32, 256), 256, 0, stream>>>(
            bp.part, dB, dC, batch * L, nCB);
        if (cudaGetLastError() != cudaSuccess) status = SSM_ERR_CUDA;
    } while (0);
    if (cudaFreeAsync(ws, stream) != cudaSuccess && status == SSM_OK) status = SSM_ERR_CUDA;
    if (own_ckpt && cudaFreeAsync(own_ckpt, stream) != cudaSuccess && status == SSM_OK)
        status = SSM_ERR_CUDA;
    return status;
}

}  // namespace bwd
}  // namespace ssm
