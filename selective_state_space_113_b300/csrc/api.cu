// api.cu -- the extern "C" boundary of libssmscan (declared in
// include/ssmscan.h): argument validation, plan choice and kernel launch.
//
// The whole library is this one translation unit; every kernel file is
// included here.
#include "../../include/ssmscan.h"

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "ceilings.cuh"
#include "common.cuh"
#include "faults.cuh"
#include "scan_tile_host.cuh"
#include "scan_bwd_generic.cuh"
#include "scan_bwd_host.cuh"
#include "scan_generic.cuh"
#include "ssd.cuh"
#include "ssd_tc.cuh"
#include "step_fast.cuh"
#include "step_generic.cuh"

namespace {

using ssm::bf16;

bool aligned_to(const void* p, size_t a) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool all_aligned16(std::initializer_list<const void*> ps) {
    for (const void* p : ps)
        if (!aligned_to(p, 16)) return false;
    return true;
}

// a*b without signed overflow for non-negative a, b; false if it would overflow.
bool mul_ok(int64_t a, int64_t b, int64_t* out) {
    if (a == 0 || b == 0) { *out = 0; return true; }
    if (a > INT64_MAX / b) return false;
    *out = a * b;
    return true;
}

size_t elem_size(int dtype) { return dtype == SSM_BF16 ? 2 : 4; }

// Element-alignment check of every tensor argument.
bool elems_aligned(int dtype, std::initializer_list<const void*> typed,
                   std::initializer_list<const void*> f32) {
    for (const void* p : typed)
        if (!aligned_to(p, elem_size(dtype))) return false;
    for (const void* p : f32)
        if (!aligned_to(p, 4)) return false;
    return true;
}

int from_cuda(cudaError_t e) { return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA; }

}  // namespace

namespace {

// The convolution in front of the scan (ssm_conv_scan_fwd): conv_w NULL = none.
struct ConvArgs {
    const float* w;
    const float* b;
    int act;
};

// The scan with a discretisation variant (ssm_disc_t) and an optional
// convolution of u; ssm_scan_fwd is variant 0 without a convolution.
int scan_impl(const void* u, const void* delta, const float* dt_bias, const float* A,
              const void* B, const void* C, const float* Dskip, const void* z, void* y,
              float* h_last, int64_t batch, int64_t L, int64_t D, int64_t N, int dtype,
              int disc, void* stream_, ConvArgs conv = {nullptr, nullptr, 0},
              float* ckpt = nullptr, bool want_ckpt = false) {
    if (batch < 0 || L < 0 || D < 0 || N < 1) return SSM_ERR_SIZE;
    if (N > SSM_MAX_N) return SSM_ERR_UNSUPPORTED;
    if (dtype != SSM_F32 && dtype != SSM_BF16) return SSM_ERR_DTYPE;
    if (disc != SSM_DISC_ZOH && disc != SSM_DISC_EULER && disc != SSM_DISC_TRAPEZOID)
        return SSM_ERR_UNSUPPORTED;
    if (conv.act != 0 && conv.act != 1) return SSM_ERR_UNSUPPORTED;
    int64_t bl, bld, bln, bd, bdn, dn;
    if (!mul_ok(batch, L, &bl) || !mul_ok(bl, D, &bld) || !mul_ok(bl, N, &bln) ||
        !mul_ok(batch, D, &bd) || !mul_ok(bd, N, &bdn) || !mul_ok(D, N, &dn) ||
        bld > (INT64_MAX >> 4) || bln > (INT64_MAX >> 4) || bdn > (INT64_MAX >> 4))
        return SSM_ERR_SIZE;
    // A pointer may be NULL only when its tensor has no elements.
    if ((bld && (!u || !delta || !y)) || (bln && (!B || !C)) || (dn && !A))
        return SSM_ERR_NULL;
    if (!elems_aligned(dtype, {u, delta, B, C, z, y},
                       {dt_bias, A, Dskip, h_last, conv.w, conv.b}))
        return SSM_ERR_ALIGN;
    const int plan = ssm::tile::forced_plan();
    const bool fast = N == ssm::tile::NS && plan != ssm::tile::kPlanGeneric &&
                      all_aligned16({u, delta, z, B, C, y, h_last, A, conv.w}) &&
                      (D * (int64_t)elem_size(dtype)) % 16 == 0;
    if (want_ckpt) {
        // checkpoints come from the N == 16 kernel only (the backward's fast path)
        if (bd && L > 32 && !ckpt) return SSM_ERR_NULL;
        if (!all_aligned16({ckpt})) return SSM_ERR_ALIGN;
        if (bd && L > 0 && !fast) return SSM_ERR_UNSUPPORTED;
    }
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    if (bd == 0) return SSM_OK;
    if (L == 0) {
        // The state after zero steps is the initial state, 0.
        if (h_last) return from_cuda(cudaMemsetAsync(h_last, 0, sizeof(float) * bdn, stream));
        return SSM_OK;
    }
    // Fast path: N == 16, 16-byte-aligned tensors and rows (TMA tiles).
    if (fast) {
        using namespace ssm::tile;
        if (conv.w) {
            if (dtype == SSM_F32)
                return launch_scan_tile<float, kZOH, true>(
                    static_cast<const float*>(u), static_cast<const float*>(delta), dt_bias, A,
                    static_cast<const float*>(B), static_cast<const float*>(C), Dskip,
                    static_cast<const float*>(z), static_cast<float*>(y), h_last, batch, L, D,
                    plan, stream, conv.w, conv.b, conv.act);
            return launch_scan_tile<bf16, kZOH, true>(
                static_cast<const bf16*>(u), static_cast<const bf16*>(delta), dt_bias, A,
                static_cast<const bf16*>(B), static_cast<const bf16*>(C), Dskip,
                static_cast<const bf16*>(z), static_cast<bf16*>(y), h_last, batch, L, D, plan,
                stream, conv.w, conv.b, conv.act);
        }
#define SSM_TILE_CALL(TT, DISC)                                                              \
    launch_scan_tile<TT, DISC>(static_cast<const TT*>(u), static_cast<const TT*>(delta), dt_bias, \
                               A, static_cast<const TT*>(B), static_cast<const TT*>(C), Dskip,   \
                               static_cast<const TT*>(z), static_cast<TT*>(y), h_last, batch, L, \
                               D, plan, stream, nullptr, nullptr, 0, ckpt)
        if (dtype == SSM_F32) {
            if (disc == SSM_DISC_EULER) return SSM_TILE_CALL(float, kEuler);
            if (disc == SSM_DISC_TRAPEZOID) return SSM_TILE_CALL(float, kTrap);
            return SSM_TILE_CALL(float, kZOH);
        }
        if (disc == SSM_DISC_EULER) return SSM_TILE_CALL(bf16, kEuler);
        if (disc == SSM_DISC_TRAPEZOID) return SSM_TILE_CALL(bf16, kTrap);
        return SSM_TILE_CALL(bf16, kZOH);
#undef SSM_TILE_CALL
    }
    cudaError_t e;
    if (dtype == SSM_F32)
        e = ssm::launch_scan_generic<float>(
            static_cast<const float*>(u), static_cast<const float*>(delta), dt_bias, A,
            static_cast<const float*>(B), static_cast<const float*>(C), Dskip,
            static_cast<const float*>(z), static_cast<float*>(y), h_last, batch, L, D, (int)N,
            stream, disc, conv.w, conv.b, conv.act);
    else
        e = ssm::launch_scan_generic<bf16>(
            static_cast<const bf16*>(u), static_cast<const bf16*>(delta), dt_bias, A,
            static_cast<const bf16*>(B), static_cast<const bf16*>(C), Dskip,
            static_cast<const bf16*>(z), static_cast<bf16*>(y), h_last, batch, L, D, (int)N,
            stream, disc, conv.w, conv.b, conv.act);
    return from_cuda(e);
}

}  // namespace

extern "C" int ssm_scan_fwd(const void* u, const void* delta, const float* dt_bias,
                            const float* A, const void* B, const void* C,
                            const float* Dskip, const void* z, void* y, float* h_last,
                            int64_t batch, int64_t L, int64_t D, int64_t N, int dtype,
                            void* stream_) {
    const ssm::fault::Range nvtx_range("ssm_scan_fwd");
    return scan_impl(u, delta, dt_bias, A, B, C, Dskip, z, y, h_last, batch, L, D, N, dtype,
                     SSM_DISC_ZOH, stream_);
}

extern "C" int ssm_scan_fwd_ckpt(const void* u, const void* delta, const float* dt_bias,
                                 const float* A, const void* B, const void* C,
                                 const float* Dskip, const void* z, void* y, float* h_last,
                                 float* ckpt, int64_t batch, int64_t L, int64_t D, int64_t N,
                                 int dtype, void* stream_) {
    const ssm::fault::Range nvtx_range("ssm_scan_fwd_ckpt");
    return scan_impl(u, delta, dt_bias, A, B, C, Dskip, z, y, h_last, batch, L, D, N, dtype,
                     SSM_DISC_ZOH, stream_, {nullptr, nullptr, 0}, ckpt, true);
}

extern "C" int ssm_scan_fwd_disc(const void* u, const void* delta, const float* dt_bias,
                                 const float* A, const void* B, const void* C,
                                 const float* Dskip, const void* z, void* y, float* h_last,
                                 int64_t batch, int64_t L, int64_t D, int64_t N, int dtype,
                                 int disc, void* stream_) {
    const ssm::fault::Range nvtx_range("ssm_scan_fwd_disc");
    return scan_impl(u, delta, dt_bias, A, B, C, Dskip, z, y, h_last, batch, L, D, N, dtype,
                     disc, stream_);
}

extern "C" int ssm_conv_scan_fwd(const void* x, const float* conv_w, const float* conv_b,
                                 int act, const void* delta, const float* dt_bias,
                                 const float* A, const void* B, const void* C,
                                 const float* Dskip, const void* z, void* y, float* h_last,
                                 int64_t batch, int64_t L, int64_t D, int64_t N, int dtype,
                                 void* stream_) {
    const ssm::fault::Range nvtx_range("ssm_conv_scan_fwd");
    if (D > 0 && !conv_w) return SSM_ERR_NULL;
    return scan_impl(x, delta, dt_bias, A, B, C, Dskip, z, y, h_last, batch, L, D, N, dtype,
                     SSM_DISC_ZOH, stream_, ConvArgs{D > 0 ? conv_w : nullptr, conv_b, act});
}

namespace {
int bwd_impl(const void* u, const void* delta, const float* dt_bias, const float* A, const void* B,
             const void* C, const float* Dskip, const void* z, const void* dy,
             const float* dh_last, const float* ckpt, bool want_ckpt, void* du, void* ddelta,
             float* ddt_bias, float* dA, float* dB, float* dC, float* dDskip, void* dz,
             int64_t batch, int64_t L, int64_t D, int64_t N, int dtype, void* stream_) {
    if (batch < 0 || L < 0 || D < 0 || N < 1) return SSM_ERR_SIZE;
    if (N > SSM_MAX_N) return SSM_ERR_UNSUPPORTED;
    if (dtype != SSM_F32 && dtype != SSM_BF16) return SSM_ERR_DTYPE;
    int64_t bl, bld, bln, bd, bdn, dn;
    if (!mul_ok(batch, L, &bl) || !mul_ok(bl, D, &bld) || !mul_ok(bl, N, &bln) ||
        !mul_ok(batch, D, &bd) || !mul_ok(bd, N, &bdn) || !mul_ok(D, N, &dn) ||
        bld > (INT64_MAX >> 5) || bln > (INT64_MAX >> 5) || bdn > (INT64_MAX >> 5))
        return SSM_ERR_SIZE;
    if ((bld && (!u || !delta || !dy || !du || !ddelta || (z && !dz))) || (bln && (!B || !C)) ||
        (dn && (!A || !dA)))
        return SSM_ERR_NULL;
    if (!elems_aligned(dtype, {u, delta, B, C, z, dy, du, ddelta, dz},
                       {dt_bias, A, Dskip, dh_last, ddt_bias, dA, dB, dC, dDskip}))
        return SSM_ERR_ALIGN;
    const int plan = ssm::tile::forced_plan();
    const bool fast = N == ssm::bwd::NS && plan != ssm::tile::kPlanGeneric &&
                      all_aligned16({u, delta, z, dy, B, C, A, du}) &&
                      (D * (int64_t)elem_size(dtype)) % 16 == 0;
    if (want_ckpt) {
        // the forward pass's checkpoints serve the N == 16 kernels only
        if (bd && L > 32 && !ckpt) return SSM_ERR_NULL;
        if (!all_aligned16({ckpt})) return SSM_ERR_ALIGN;
        if (bd && L > 0 && !fast) return SSM_ERR_UNSUPPORTED;
    }
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    // Sums start from zero: with no step or no channel they stay zero.
    if (dn && cudaMemsetAsync(dA, 0, sizeof(float) * dn, stream) != cudaSuccess) return SSM_ERR_CUDA;
    if (D && dDskip && cudaMemsetAsync(dDskip, 0, sizeof(float) * D, stream) != cudaSuccess)
        return SSM_ERR_CUDA;
    if (D && ddt_bias && cudaMemsetAsync(ddt_bias, 0, sizeof(float) * D, stream) != cudaSuccess)
        return SSM_ERR_CUDA;
    if (bln && dB && cudaMemsetAsync(dB, 0, sizeof(float) * bln, stream) != cudaSuccess)
        return SSM_ERR_CUDA;
    if (bln && dC && cudaMemsetAsync(dC, 0, sizeof(float) * bln, stream) != cudaSuccess)
        return SSM_ERR_CUDA;
    if (bd == 0 || L == 0) return SSM_OK;
    if (fast) {
        if (dtype == SSM_F32)
            return ssm::bwd::launch_scan_bwd16<float>(
                static_cast<const float*>(u), static_cast<const float*>(delta), dt_bias, A,
                static_cast<const float*>(B), static_cast<const float*>(C), Dskip,
                static_cast<const float*>(z), static_cast<const float*>(dy), dh_last,
                static_cast<float*>(du), static_cast<float*>(ddelta), ddt_bias, dA, dB, dC,
                dDskip, static_cast<float*>(dz), batch, L, D, stream, ckpt, plan);
        return ssm::bwd::launch_scan_bwd16<bf16>(
            static_cast<const bf16*>(u), static_cast<const bf16*>(delta), dt_bias, A,
            static_cast<const bf16*>(B), static_cast<const bf16*>(C), Dskip,
            static_cast<const bf16*>(z), static_cast<const bf16*>(dy), dh_last,
            static_cast<bf16*>(du), static_cast<bf16*>(ddelta), ddt_bias, dA, dB, dC, dDskip,
            static_cast<bf16*>(dz), batch, L, D, stream, ckpt, plan);
    }
    float* scratch = nullptr;
    const size_t bytes = sizeof(float) * ssm::bwdg::bwd_generic_scratch_floats(batch, L, D, N);
    if (ssm::fault::malloc_async(reinterpret_cast<void**>(&scratch), bytes, stream) != cudaSuccess) {
        cudaGetLastError();
        return SSM_ERR_NOMEM;
    }
    cudaError_t e;
    if (dtype == SSM_F32)
        e = ssm::bwdg::launch_scan_bwd_generic<float>(
            static_cast<const float*>(u), static_cast<const float*>(delta), dt_bias, A,
            static_cast<const float*>(B), static_cast<const float*>(C), Dskip,
            static_cast<const float*>(z), static_cast<const float*>(dy), dh_last,
            static_cast<float*>(du), static_cast<float*>(ddelta), ddt_bias, dA, dB, dC, dDskip,
            static_cast<float*>(dz), scratch, batch, L, D, (int)N, stream);
    else
        e = ssm::bwdg::launch_scan_bwd_generic<bf16>(
            static_cast<const bf16*>(u), static_cast<const bf16*>(delta), dt_bias, A,
            static_cast<const bf16*>(B), static_cast<const bf16*>(C), Dskip,
            static_cast<const bf16*>(z), static_cast<const bf16*>(dy), dh_last,
            static_cast<bf16*>(du), static_cast<bf16*>(ddelta), ddt_bias, dA, dB, dC, dDskip,
            static_cast<bf16*>(dz), scratch, batch, L, D, (int)N, stream);
    const cudaError_t ef = cudaFreeAsync(scratch, stream);
    return from_cuda(e != cudaSuccess ? e : ef);
}
}  // namespace

extern "C" int ssm_scan_bwd(const void* u, const void* delta, const float* dt_bias,
                            const float* A, const void* B, const void* C, const float* Dskip,
                            const void* z, const void* dy, const float* dh_last, void* du,
                            void* ddelta, float* ddt_bias, float* dA, float* dB, float* dC,
                            float* dDskip, void* dz, int64_t batch, int64_t L, int64_t D,
                            int64_t N, int dtype, void* stream_) {
    const ssm::fault::Range nvtx_range("ssm_scan_bwd");
    return bwd_impl(u, delta, dt_bias, A, B, C, Dskip, z, dy, dh_last, nullptr, false, du, ddelta,
                    ddt_bias, dA, dB, dC, dDskip, dz, batch, L, D, N, dtype, stream_);
}

extern "C" int ssm_scan_bwd_ckpt(const void* u, const void* delta, const float* dt_bias,
                                 const float* A, const void* B, const void* C,
                                 const float* Dskip, const void* z, const void* dy,
                                 const float* dh_last, const float* ckpt, void* du, void* ddelta,
                                 float* ddt_bias, float* dA, float* dB, float* dC, float* dDskip,
                                 void* dz, int64_t batch, int64_t L, int64_t D, int64_t N,
                                 int dtype, void* stream_) {
    const ssm::fault::Range nvtx_range("ssm_scan_bwd_ckpt");
    return bwd_impl(u, delta, dt_bias, A, B, C, Dskip, z, dy, dh_last, ckpt, true, du, ddelta,
                    ddt_bias, dA, dB, dC, dDskip, dz, batch, L, D, N, dtype, stream_);
}

extern "C" int ssm_ssd_fwd(const void* x, const void* dt, const float* dt_bias, const float* A,
                           const void* B, const void* C, const float* Dskip, void* y,
                           float* h_last, int64_t batch, int64_t L, int64_t H, int64_t P,
                           int64_t N, int dtype, void* stream_) {
    const ssm::fault::Range nvtx_range("ssm_ssd_fwd");
    if (batch < 0 || L < 0 || H < 0 || P < 1 || N < 1) return SSM_ERR_SIZE;
    if (N > SSM_MAX_N) return SSM_ERR_UNSUPPORTED;
    if (dtype != SSM_F32 && dtype != SSM_BF16) return SSM_ERR_DTYPE;
    int64_t bl, blh, blhp, bln, bh, bhp, bhpn;
    if (!mul_ok(batch, L, &bl) || !mul_ok(bl, H, &blh) || !mul_ok(blh, P, &blhp) ||
        !mul_ok(bl, N, &bln) || !mul_ok(batch, H, &bh) || !mul_ok(bh, P, &bhp) ||
        !mul_ok(bhp, N, &bhpn) || blhp > (INT64_MAX >> 4) || bhpn > (INT64_MAX >> 4))
        return SSM_ERR_SIZE;
    if ((blhp && (!x || !y)) || (blh && !dt) || (bln && (!B || !C)) || (H && !A))
        return SSM_ERR_NULL;
    if (!elems_aligned(dtype, {x, dt, B, C, y}, {dt_bias, A, Dskip, h_last})) return SSM_ERR_ALIGN;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    if (bhp == 0) return SSM_OK;
    if (L == 0) {
        if (h_last) return from_cuda(cudaMemsetAsync(h_last, 0, sizeof(float) * bhpn, stream));
        return SSM_OK;
    }
    const bool tc = dtype == SSM_BF16 && P == ssm::ssdtc::P && (N == 64 || N == 128) &&
                    all_aligned16({x, B, C, y}) && ssm::tile::forced_plan() != ssm::tile::kPlanGeneric;
    cudaError_t e;
    if (tc) {
        e = ssm::ssdtc::launch_ssd_tc(
            static_cast<const bf16*>(x), static_cast<const bf16*>(dt), dt_bias, A,
            static_cast<const bf16*>(B), static_cast<const bf16*>(C), Dskip, static_cast<bf16*>(y),
            h_last, batch, L, H, (int)N,
            (unsigned long long)ssm::tile::env_ll("SSM_WAIT_LIMIT_NS", 2000000000LL), stream,
            ssm::tile::env_ll("SSM_SSD_SEG", 0), ssm::tile::env_ll("SSM_SSD_CTAS", 0));
        if (e == cudaErrorMemoryAllocation) return SSM_ERR_NOMEM;
    } else if (dtype == SSM_F32) {
        e = ssm::ssd::launch_ssd_generic<float>(
            static_cast<const float*>(x), static_cast<const float*>(dt), dt_bias, A,
            static_cast<const float*>(B), static_cast<const float*>(C), Dskip,
            static_cast<float*>(y), h_last, batch, L, H, P, (int)N, stream);
    } else {
        e = ssm::ssd::launch_ssd_generic<bf16>(
            static_cast<const bf16*>(x), static_cast<const bf16*>(dt), dt_bias, A,
            static_cast<const bf16*>(B), static_cast<const bf16*>(C), Dskip,
            static_cast<bf16*>(y), h_last, batch, L, H, P, (int)N, stream);
    }
    return from_cuda(e);
}

extern "C" int ssm_step(float* state, const void* u, const void* delta, const float* dt_bias,
                        const float* A, const void* B, const void* C, const float* Dskip,
                        const void* z, void* y, int64_t batch, int64_t D, int64_t N, int dtype,
                        void* stream_) {
    const ssm::fault::Range nvtx_range("ssm_step");
    if (batch < 0 || D < 0 || N < 1) return SSM_ERR_SIZE;
    if (N > SSM_MAX_N) return SSM_ERR_UNSUPPORTED;
    if (dtype != SSM_F32 && dtype != SSM_BF16) return SSM_ERR_DTYPE;
    int64_t bd, bdn, bn, dn;
    if (!mul_ok(batch, D, &bd) || !mul_ok(bd, N, &bdn) || !mul_ok(batch, N, &bn) ||
        !mul_ok(D, N, &dn) || bdn > (INT64_MAX >> 4))
        return SSM_ERR_SIZE;
    if ((bd && (!state || !u || !delta || !y)) || (bn && (!B || !C)) || (dn && !A))
        return SSM_ERR_NULL;
    if (!elems_aligned(dtype, {u, delta, B, C, z, y}, {state, dt_bias, A, Dskip}))
        return SSM_ERR_ALIGN;
    if (bd == 0) return SSM_OK;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    cudaError_t e;
    if (N == ssm::stepk::NS && all_aligned16({state, A}) && D <= ssm::stepk::kMaxD &&
        batch <= ssm::stepk::kMaxBatch && !std::getenv("SSM_FORCE_GENERIC_STEP")) {
        // Tiled path: persistent CTAs, tensor copies of 128-channel x 4-entry
        // tiles (needs D % 8 == 0 and 16-byte aligned rows).
        // SSM_STEP_KERNEL=threads selects the one-pass kernel below instead.
        const char* kname = std::getenv("SSM_STEP_KERNEL");
        if (D % 8 == 0 && all_aligned16({u, delta, z, B, C}) &&
            ((D + ssm::stepk::kTileTC - 1) / ssm::stepk::kTileTC) *
                    ((batch + ssm::stepk::kTileNB - 1) / ssm::stepk::kTileNB) < INT32_MAX &&
            !(kname && std::strcmp(kname, "threads") == 0)) {
            const unsigned long long wait_ns =
                (unsigned long long)ssm::tile::env_ll("SSM_WAIT_LIMIT_NS", 2000000000LL);
            if (dtype == SSM_F32)
                e = ssm::stepk::launch_step16_tiled<float>(
                    state, static_cast<const float*>(u), static_cast<const float*>(delta), dt_bias,
                    A, static_cast<const float*>(B), static_cast<const float*>(C), Dskip,
                    static_cast<const float*>(z), static_cast<float*>(y), batch, D, wait_ns,
                    stream);
            else
                e = ssm::stepk::launch_step16_tiled<bf16>(
                    state, static_cast<const bf16*>(u), static_cast<const bf16*>(delta), dt_bias,
                    A, static_cast<const bf16*>(B), static_cast<const bf16*>(C), Dskip,
                    static_cast<const bf16*>(z), static_cast<bf16*>(y), batch, D, wait_ns, stream);
            return from_cuda(e);
        }
        // One-pass path: four threads per channel, one float4 of state each.
        if (dtype == SSM_F32)
            e = ssm::stepk::launch_step16<float>(
                state, static_cast<const float*>(u), static_cast<const float*>(delta), dt_bias, A,
                static_cast<const float*>(B), static_cast<const float*>(C), Dskip,
                static_cast<const float*>(z), static_cast<float*>(y), batch, D, stream);
        else
            e = ssm::stepk::launch_step16<bf16>(
                state, static_cast<const bf16*>(u), static_cast<const bf16*>(delta), dt_bias, A,
                static_cast<const bf16*>(B), static_cast<const bf16*>(C), Dskip,
                static_cast<const bf16*>(z), static_cast<bf16*>(y), batch, D, stream);
        return from_cuda(e);
    }
    if (dtype == SSM_F32)
        e = ssm::launch_step_generic<float>(
            state, static_cast<const float*>(u), static_cast<const float*>(delta), dt_bias, A,
            static_cast<const float*>(B), static_cast<const float*>(C), Dskip,
            static_cast<const float*>(z), static_cast<float*>(y), batch, D, (int)N, stream);
    else
        e = ssm::launch_step_generic<bf16>(
            state, static_cast<const bf16*>(u), static_cast<const bf16*>(delta), dt_bias, A,
            static_cast<const bf16*>(B), static_cast<const bf16*>(C), Dskip,
            static_cast<const bf16*>(z), static_cast<bf16*>(y), batch, D, (int)N, stream);
    return from_cuda(e);
}

extern "C" int ssm_device_status(void* stream_) {
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    if (cudaStreamSynchronize(stream) != cudaSuccess) return SSM_ERR_CUDA;
    unsigned int word = 0;
    if (cudaMemcpyFromSymbol(&word, ssm::g_error_word, sizeof word) != cudaSuccess)
        return SSM_ERR_CUDA;
    if (word != 0) {
        const unsigned int zero = 0;
        if (cudaMemcpyToSymbol(ssm::g_error_word, &zero, sizeof zero) != cudaSuccess)
            return SSM_ERR_CUDA;
        if (word & ssm::kErrTimeout) return SSM_ERR_TIMEOUT;
    }
    return SSM_OK;
}

extern "C" const char* ssm_status_string(int status) {
    switch (status) {
        case SSM_OK: return "ok";
        case SSM_ERR_NULL: return "a required pointer is NULL";
        case SSM_ERR_SIZE: return "invalid or overflowing size";
        case SSM_ERR_DTYPE: return "unknown dtype";
        case SSM_ERR_ALIGN: return "pointer not aligned to its element size";
        case SSM_ERR_UNSUPPORTED: return "unsupported state size N";
        case SSM_ERR_CUDA: return "CUDA runtime error";
        case SSM_ERR_NOMEM: return "workspace allocation failed";
        case SSM_ERR_TIMEOUT: return "device-side bounded wait gave up";
        case SSM_ERR_SCRATCH: return "problem needs more scratch than the fixed no-allocation buffer";
        default: return "unknown status";
    }
}

extern "C" int ssm_abi_version(void) { return 1; }

extern "C" int ssm_unit_ceilings(double* out, int reps, void* stream_) {
    const ssm::fault::Range nvtx_range("ssm_unit_ceilings");
    if (!out) return SSM_ERR_NULL;
    if (reps < 1) return SSM_ERR_SIZE;
    if (ssm::fault::launch_refused()) return SSM_ERR_CUDA;
    double r[3] = {0.0, 0.0, 0.0};
    if (ssm::ceil::measure(r, reps, static_cast<cudaStream_t>(stream_)) != cudaSuccess) {
        cudaGetLastError();
        return SSM_ERR_CUDA;
    }
    for (int i = 0; i < 3; ++i) out[i] = r[i];
    return SSM_OK;
}

// ---------------------------------------------------------------------------
// ssm_scan_fwd_noalloc: the selective scan for callers that must not allocate
// device memory while they run (for example a serving loop whose memory is
// all reserved up front by its own pool, or code in a context where a
// cudaMalloc/cudaMallocAsync would synchronise, fail or be forbidden).  It is
// the chained variant of the N == 16 fast kernel, whose scratch (unit ticket,
// abort word, per-sub-block progress flags and, when h_last is NULL, the
// carried chunk state) lives in the fixed device array below instead of a
// stream-ordered workspace.  Inputs the fast kernel does not take (other N,
// unaligned tensors) run the generic kernel, which needs no scratch at all.
namespace {

// Scratch of the allocation-free entry point.  Every device that loads this
// library holds these bytes until the process exits.  In host code the name
// is only a host-side stand-in: kernels get the device address looked up by
// noalloc_scratch_ptr().
constexpr size_t kNoallocScratchBytes = SSM_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 128;
std::mutex g_noalloc_mu;
// Per device: the ID of the context the address was looked up in, and the
// address.
struct NoallocSlot {
    unsigned long long ctx;
    void* ptr;
};
NoallocSlot g_noalloc_slot[kMaxDevices] = {};

// Device address of g_noalloc_scratch in the current device's current
// context.  It is looked up with that device current the first time a call
// runs in that context (the first call on a device, and again in a context
// made after the last one was destroyed, which may reuse its handle but not
// its ID), so an address is never reused from a context that is gone.
int noalloc_scratch_ptr(unsigned char** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SSM_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    unsigned long long ctx = ssm::context::current_id();
    NoallocSlot& slot = g_noalloc_slot[dev];
    if (!ctx || slot.ctx != ctx || !slot.ptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return SSM_ERR_CUDA;
        }
        // The lookup makes the device's primary context current if none was.
        ctx = ssm::context::current_id();
        if (!ctx) return SSM_ERR_CUDA;
        slot.ctx = ctx;
        slot.ptr = p;
    }
    *out = static_cast<unsigned char*>(slot.ptr);
    return SSM_OK;
}

// Scratch bytes the chained plan needs: header (tickets, abort), one flag per
// 32-channel sub-block, and the carried state when h_last cannot hold it.
size_t noalloc_scratch_need(int64_t batch, int64_t D, bool have_h_last) {
    size_t bytes = ssm::tile::header_bytes(batch, D);
    if (!have_h_last) bytes += (size_t)(batch * D) * ssm::tile::NS * 4;
    return bytes;
}

template <typename T>
int launch_noalloc(const T* u, const T* delta, const float* dt_bias, const float* A,
                   const T* Bm, const T* Cm, const float* Dskip, const T* z, T* y,
                   float* h_last, long long batch, long long L, long long D,
                   unsigned char* ws, cudaStream_t stream) {
    using namespace ssm::tile;
    int dev = 0, sms = 0;
    long long workers = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        prepare<T, (int)kChained, (int)kZOH>(sms, &workers) != cudaSuccess || workers < 1)
        return SSM_ERR_CUDA;
    CUtensorMap maps[6];
    Params p;
    if (!setup<T>(maps, &p, u, delta, dt_bias, A, Bm, Cm, Dskip, z, y, h_last, batch, L, D))
        return SSM_ERR_CUDA;
    // SSM_CHUNK_T (development and tests) cuts chains into pieces of about
    // that many steps, as it does for ssm_scan_fwd's chained plan.
    p.G = chained_grid<T>(p.nchains, workers, L, env_ll("SSM_CHUNK_T", 0));
    const size_t head = header_bytes(batch, D);
    // The array keeps the previous call's contents: reset the tickets, the
    // abort word and the sub-block flags, which must start at zero.
    if (cudaMemsetAsync(ws, 0, head, stream) != cudaSuccess) return SSM_ERR_CUDA;
    p.ticket = reinterpret_cast<unsigned long long*>(ws);
    p.abort = reinterpret_cast<unsigned*>(ws + 32);
    p.flags = reinterpret_cast<unsigned*>(ws + 256);
    p.carry = h_last ? h_last : reinterpret_cast<float*>(ws + head);
    return launch_mode<T, (int)kChained, (int)kZOH>(p.G, maps, p, stream) == cudaSuccess ? SSM_OK
                                                                             : SSM_ERR_CUDA;
}

}  // namespace

extern "C" int ssm_scan_fwd_noalloc(const void* u, const void* delta, const float* dt_bias,
                                    const float* A, const void* B, const void* C,
                                    const float* Dskip, const void* z, void* y, float* h_last,
                                    int64_t batch, int64_t L, int64_t D, int64_t N, int dtype,
                                    void* stream_) {
    const ssm::fault::Range nvtx_range("ssm_scan_fwd_noalloc");
    if (batch < 0 || L < 0 || D < 0 || N < 1) return SSM_ERR_SIZE;
    if (N > SSM_MAX_N) return SSM_ERR_UNSUPPORTED;
    if (dtype != SSM_F32 && dtype != SSM_BF16) return SSM_ERR_DTYPE;
    int64_t bl, bld, bln, bd, bdn, dn;
    if (!mul_ok(batch, L, &bl) || !mul_ok(bl, D, &bld) || !mul_ok(bl, N, &bln) ||
        !mul_ok(batch, D, &bd) || !mul_ok(bd, N, &bdn) || !mul_ok(D, N, &dn) ||
        bld > (INT64_MAX >> 4) || bln > (INT64_MAX >> 4) || bdn > (INT64_MAX >> 4))
        return SSM_ERR_SIZE;
    if ((bld && (!u || !delta || !y)) || (bln && (!B || !C)) || (dn && !A)) return SSM_ERR_NULL;
    if (!elems_aligned(dtype, {u, delta, B, C, z, y}, {dt_bias, A, Dskip, h_last}))
        return SSM_ERR_ALIGN;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    if (bd == 0) return SSM_OK;
    if (L == 0) {
        if (h_last) return from_cuda(cudaMemsetAsync(h_last, 0, sizeof(float) * bdn, stream));
        return SSM_OK;
    }
    const bool fast = N == ssm::tile::NS && all_aligned16({u, delta, z, B, C, y, h_last, A}) &&
                      (D * (int64_t)elem_size(dtype)) % 16 == 0;
    if (!fast) {
        cudaError_t e;
        if (dtype == SSM_F32)
            e = ssm::launch_scan_generic<float>(
                static_cast<const float*>(u), static_cast<const float*>(delta), dt_bias, A,
                static_cast<const float*>(B), static_cast<const float*>(C), Dskip,
                static_cast<const float*>(z), static_cast<float*>(y), h_last, batch, L, D,
                (int)N, stream);
        else
            e = ssm::launch_scan_generic<bf16>(
                static_cast<const bf16*>(u), static_cast<const bf16*>(delta), dt_bias, A,
                static_cast<const bf16*>(B), static_cast<const bf16*>(C), Dskip,
                static_cast<const bf16*>(z), static_cast<bf16*>(y), h_last, batch, L, D,
                (int)N, stream);
        return from_cuda(e);
    }
    if (noalloc_scratch_need(batch, D, h_last != nullptr) > kNoallocScratchBytes)
        return SSM_ERR_SCRATCH;
    unsigned char* ws = nullptr;
    const int st = noalloc_scratch_ptr(&ws);
    if (st != SSM_OK) return st;
    if (dtype == SSM_F32)
        return launch_noalloc<float>(
            static_cast<const float*>(u), static_cast<const float*>(delta), dt_bias, A,
            static_cast<const float*>(B), static_cast<const float*>(C), Dskip,
            static_cast<const float*>(z), static_cast<float*>(y), h_last, batch, L, D, ws, stream);
    return launch_noalloc<bf16>(
        static_cast<const bf16*>(u), static_cast<const bf16*>(delta), dt_bias, A,
        static_cast<const bf16*>(B), static_cast<const bf16*>(C), Dskip,
        static_cast<const bf16*>(z), static_cast<bf16*>(y), h_last, batch, L, D, ws, stream);
}
