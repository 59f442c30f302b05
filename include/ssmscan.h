/*
 * ssmscan.h -- C ABI of libssmscan, the B300 (sm_103a) selective state-space
 * scan (the S6 core of Mamba) and its single-token decode step.
 *
 * The operation, from the pages on Mamba / selective SSMs:
 *   - "Mamba と状態空間モデル(SSM)" (ta-paperlens), section "Mamba: 状態を
 *     「選択的」にする", pseudocode: Delta, B and C are per-token, A is a
 *     learned parameter, dt = softplus(x W_d + bias), the state update and
 *     the readout y_t = C_t h;
 *   - "State Space Models (SSM)" (ultralytics glossary), section "SSMの仕組み":
 *     zero-order hold A_bar = exp(Delta A), B_bar = (A_bar - 1)/A * B, the
 *     recurrence h_t = A_bar h_{t-1} + B_bar x_t from h = 0, y_t = C h_t;
 *   - news.han.ihouse.idv.tw article 1304: the output equation y = C h + D x;
 *   - agenticai-flow Mamba guide, block diagram: the S6 output is multiplied
 *     element-wise by SiLU(z).
 *
 * For every batch entry b, channel d, step t and state n:
 *   dt         = softplus(delta[b,t,d] + dt_bias[d])
 *   A_bar      = exp(dt * A[d,n])
 *   B_bar      = (A_bar - 1) / A[d,n] * B[b,t,n]   (dt * B[b,t,n] if A[d,n] == 0)
 *   h[b,d,n]   = A_bar * h[b,d,n] + B_bar * u[b,t,d]          (h starts at 0)
 *   y[b,t,d]   = (sum_n C[b,t,n] * h[b,d,n] + Dskip[d] * u[b,t,d]) * silu(z[b,t,d])
 * with silu(z) = z / (1 + exp(-z)).  All arithmetic is float32 with the
 * state kept in float32; bf16 inputs are widened exactly and y is rounded to
 * bf16 (round-to-nearest-even) only when stored.
 *
 * Conventions shared by every entry point:
 *   - Every tensor pointer is DEVICE memory on the current CUDA device,
 *     allocated, owned and freed by the caller; the library never frees or
 *     retains a caller pointer after the call returns.  Tensors are dense and
 *     row-major with the shapes given below.
 *   - `dtype` (ssm_dtype_t) is the element type of u, delta, z, B, C and y.
 *     dt_bias, A, Dskip, h_last and state are always float32.
 *   - `stream` is a cudaStream_t (NULL: the legacy default stream).  Work is
 *     enqueued on it and the call returns without synchronising; results are
 *     valid once the stream has reached that point.
 *   - Argument errors are returned synchronously, before anything is
 *     enqueued.  A failed launch returns SSM_ERR_CUDA.  A device-side bounded
 *     wait that gives up is recorded on the device and reported by
 *     ssm_device_status().
 *   - A tensor pointer may be NULL only when that tensor has no elements
 *     (or when the entry point documents it as optional).
 *   - Any element-aligned pointer is accepted.  16-byte-aligned tensors with
 *     D * sizeof(dtype) a multiple of 16 and N == 16 take the fast kernels;
 *     everything else runs a generic GPU kernel (never the CPU).
 */
#ifndef SSMSCAN_H
#define SSMSCAN_H

#include <stdint.h>

#if defined(__GNUC__)
#define SSM_API __attribute__((visibility("default")))
#else
#define SSM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { SSM_F32 = 0, SSM_BF16 = 1 } ssm_dtype_t;

/* Discretisation of the input term for ssm_scan_fwd_disc (the decay
 * A_bar = exp(dt A) is the same in all three). */
typedef enum {
    SSM_DISC_ZOH = 0,       /* (A_bar - 1)/A B_t u_t: zero-order hold (ssm_scan_fwd) */
    SSM_DISC_EULER = 1,     /* dt B_t u_t */
    SSM_DISC_TRAPEZOID = 2  /* dt/2 (B_t u_t + A_bar B_{t-1} u_{t-1}), B_{-1} u_{-1} = 0 */
} ssm_disc_t;

typedef enum {
    SSM_OK = 0,
    SSM_ERR_NULL = -1,        /* a required pointer is NULL */
    SSM_ERR_SIZE = -2,        /* negative size, N < 1, or a size that overflows */
    SSM_ERR_DTYPE = -3,       /* dtype is not an ssm_dtype_t value */
    SSM_ERR_ALIGN = -4,       /* a pointer is not aligned to its element size */
    SSM_ERR_UNSUPPORTED = -5, /* N > SSM_MAX_N, an unknown discretisation or act */
    SSM_ERR_CUDA = -6,        /* a CUDA runtime call or launch failed */
    SSM_ERR_NOMEM = -7,       /* the stream-ordered workspace could not be allocated */
    SSM_ERR_TIMEOUT = -8,     /* a device-side bounded wait gave up (see ssm_device_status) */
    SSM_ERR_SCRATCH = -9      /* ssm_scan_fwd_noalloc: problem exceeds its fixed scratch */
} ssm_status_t;

/* Largest supported state size N. */
#define SSM_MAX_N 256

/*
 * ssm_scan_fwd -- selective scan over a whole sequence, from h = 0.
 *
 *   u, delta, z : [batch, L, D]  dtype      (z may be NULL: no gate)
 *   B, C        : [batch, L, N]  dtype
 *   dt_bias     : [D] float32               (NULL means 0)
 *   A           : [D, N] float32
 *   Dskip       : [D] float32               (NULL means 0)
 *   y           : [batch, L, D] dtype, written
 *   h_last      : [batch, D, N] float32, written with the state after the
 *                 last step (h_last == NULL: not written).  It has the layout
 *                 of ssm_step's `state`, so a prefill continues into decode.
 * Sizes: batch, L, D >= 0; 1 <= N <= SSM_MAX_N.  L == 0 writes h_last = 0.
 * The fast path may take a small stream-ordered workspace (allocated and
 * freed on `stream`); SSM_ERR_NOMEM if that fails.  Workspaces of every entry
 * point come from a memory pool the library makes on each device, which
 * keeps up to 1 GiB reserved between calls so that a call after a
 * synchronisation does not map its workspace again; that memory is held
 * until the process exits.
 * Returns an ssm_status_t.
 */
SSM_API int ssm_scan_fwd(const void *u, const void *delta, const float *dt_bias,
                 const float *A, const void *B, const void *C,
                 const float *Dskip, const void *z, void *y, float *h_last,
                 int64_t batch, int64_t L, int64_t D, int64_t N, int dtype,
                 void *stream);

/*
 * ssm_scan_fwd_disc -- ssm_scan_fwd with another discretisation of the input
 * term (ssm_disc_t; SSM_DISC_ZOH gives ssm_scan_fwd itself):
 *   SSM_DISC_EULER      h_t = A_bar h_{t-1} + dt B_t u_t, the update of the
 *                       selective-state pseudocode on the ta-paperlens page
 *                       ("Mamba: 状態を「選択的」にする");
 *   SSM_DISC_TRAPEZOID  h_t = A_bar h_{t-1} + dt/2 (B_t u_t + A_bar B_{t-1}
 *                       u_{t-1}), from h = 0 and B_{-1} u_{-1} = 0: the
 *                       trapezoidal rule Mamba-3 uses (news.han.ihouse.idv.tw
 *                       article 1304, "より正確な離散化：台形法則"; its
 *                       data-dependent weight is taken as 1/2).
 * Arguments, layouts, ownership and errors are those of ssm_scan_fwd; an
 * unknown `disc` returns SSM_ERR_UNSUPPORTED.  h_last is the state only (a
 * trapezoidal prefill does not carry B_{L-1} u_{L-1} into ssm_step, whose
 * update is the zero-order hold).
 */
SSM_API int ssm_scan_fwd_disc(const void *u, const void *delta, const float *dt_bias,
                              const float *A, const void *B, const void *C,
                              const float *Dskip, const void *z, void *y, float *h_last,
                              int64_t batch, int64_t L, int64_t D, int64_t N, int dtype,
                              int disc, void *stream);

/*
 * ssm_conv_scan_fwd -- the short causal convolution in front of the SSM,
 * then ssm_scan_fwd on its output (ta-paperlens page, "現場ではこう使う":
 * d_conv, a short convolution before the SSM; agenticai-flow page: d_conv=4
 * with causal-conv1d).  Read as depthwise (one width-4 filter per channel),
 * causal, zero input before step 0, with an optional SiLU after it (the
 * pages name no activation; act selects one):
 *     v_t[d] = conv_b[d] + sum_{k=0}^{3} conv_w[d, k] x_{t-3+k}[d]
 *     u_t[d] = act ? v_t[d] sigmoid(v_t[d]) : v_t[d]
 * and u feeds the zero-order-hold scan, also in the D skip term.
 *
 *   x           : [batch, L, D] dtype (in place of ssm_scan_fwd's u)
 *   conv_w      : [D, 4] float32, conv_w[d, 3] multiplies the current x;
 *                 required when D > 0 (else SSM_ERR_NULL)
 *   conv_b      : [D] float32 (NULL means 0)
 *   act         : 0 (none) or 1 (SiLU); another value is SSM_ERR_UNSUPPORTED
 * The other arguments, layouts, ownership and errors are those of
 * ssm_scan_fwd.  The fast path (N == 16) also wants conv_w 16-byte aligned.
 */
SSM_API int ssm_conv_scan_fwd(const void *x, const float *conv_w, const float *conv_b, int act,
                              const void *delta, const float *dt_bias, const float *A,
                              const void *B, const void *C, const float *Dskip, const void *z,
                              void *y, float *h_last, int64_t batch, int64_t L, int64_t D,
                              int64_t N, int dtype, void *stream);

/*
 * ssm_scan_bwd -- backward pass of ssm_scan_fwd (zero-order hold): the
 * derivatives of a loss with respect to every input, given its derivatives
 * dy with respect to y and dh_last with respect to h_last.  The states are
 * recomputed from the inputs, never stored (ta-paperlens page, "代償と、
 * それを払う方法（並列スキャン）": the fused kernel recomputes instead of
 * keeping the intermediate states for the backward pass).
 *
 *   inputs      : u, delta, dt_bias, A, B, C, Dskip, z exactly as given to
 *                 ssm_scan_fwd (same layouts, same NULL meanings)
 *   dy          : [batch, L, D] dtype
 *   dh_last     : [batch, D, N] float32, NULL means 0
 *   du, ddelta  : [batch, L, D] dtype, written
 *   dz          : [batch, L, D] dtype, written; required when z is given,
 *                 ignored when z is NULL
 *   dB, dC      : [batch, L, N] float32, written (sums over channels);
 *                 NULL: not computed
 *   dA          : [D, N] float32, written (sum over batch and steps)
 *   ddt_bias, dDskip : [D] float32, written (sums over batch and steps);
 *                 NULL: not computed
 * Sizes as for ssm_scan_fwd.  With L == 0 or batch == 0 the sums are zero.
 * N == 16 with u, delta, z, dy, B, C, A and du 16-byte aligned and
 * D * sizeof(dtype) a multiple of 16 runs the unit kernels; anything else
 * runs a one-thread-per-channel kernel.  Takes a stream-ordered workspace (SSM_ERR_NOMEM if that fails): about
 * 3.2 * batch * L * D * N bytes / 16 for N == 16 (the states entering every
 * 32-step unit, the adjoints leaving it and their summaries), plus
 * 128 * ceil(D / 128) * batch * L bytes of per-block dB/dC sums.  The sums
 * over channels, batch and steps are formed in float32 (dA, dDskip and
 * ddt_bias with atomic adds, so their last bits can vary between calls).
 * Returns an ssm_status_t.
 */
SSM_API int ssm_scan_bwd(const void *u, const void *delta, const float *dt_bias, const float *A,
                         const void *B, const void *C, const float *Dskip, const void *z,
                         const void *dy, const float *dh_last, void *du, void *ddelta,
                         float *ddt_bias, float *dA, float *dB, float *dC, float *dDskip,
                         void *dz, int64_t batch, int64_t L, int64_t D, int64_t N, int dtype,
                         void *stream);

/*
 * ssm_scan_fwd_ckpt / ssm_scan_bwd_ckpt -- the forward and backward passes of
 * a training step, sharing the states at the 32-step unit boundaries: the
 * forward pass writes them as it walks the sequence, and the backward pass
 * reads them instead of recomputing them in a pass of its own (the
 * backward's other phases, and its arithmetic, are those of ssm_scan_bwd).
 * This pairing is the library's; the pages say only that the fused kernel
 * recomputes the states rather than storing them all.
 *
 *   ckpt : [ceil(L / 32), batch, D, 16] float32, 16-byte aligned.  Entry k
 *          (k >= 1) is the state entering step 32 k; entry 0 (the zero state)
 *          is neither written nor read.  May be NULL when L <= 32.
 * ssm_scan_fwd_ckpt takes ssm_scan_fwd's arguments (zero-order hold, y and
 * h_last as there) and writes ckpt.  ssm_scan_bwd_ckpt takes ssm_scan_bwd's
 * arguments and ckpt, which must come from ssm_scan_fwd_ckpt with the same
 * inputs (nothing checks that); it needs no workspace for the states.  Both
 * run the N == 16 kernels only: N != 16, or a tensor or row that those
 * kernels cannot take (see ssm_scan_fwd and ssm_scan_bwd), returns
 * SSM_ERR_UNSUPPORTED before anything is enqueued.  Returns an ssm_status_t.
 */
SSM_API int ssm_scan_fwd_ckpt(const void *u, const void *delta, const float *dt_bias,
                              const float *A, const void *B, const void *C, const float *Dskip,
                              const void *z, void *y, float *h_last, float *ckpt, int64_t batch,
                              int64_t L, int64_t D, int64_t N, int dtype, void *stream);
SSM_API int ssm_scan_bwd_ckpt(const void *u, const void *delta, const float *dt_bias,
                              const float *A, const void *B, const void *C, const float *Dskip,
                              const void *z, const void *dy, const float *dh_last,
                              const float *ckpt, void *du, void *ddelta, float *ddt_bias,
                              float *dA, float *dB, float *dC, float *dDskip, void *dz,
                              int64_t batch, int64_t L, int64_t D, int64_t N, int dtype,
                              void *stream);

/*
 * ssm_ssd_fwd -- the Mamba-2 form of the scan (structured state-space
 * duality; news.han.ihouse.idv.tw article 1304: most of the SSM computation is
 * a masked matrix multiplication, A is a scalar, Euler discretisation):
 * per batch b, head h, channel p < P of the head, state n < N,
 *   dt_t   = softplus(dt[b,t,h] + dt_bias[h])
 *   h_t[n] = exp(dt_t A[h]) h_{t-1}[n] + dt_t B[b,t,n] x[b,t,h,p],   from 0
 *   y[b,t,h,p] = sum_n C[b,t,n] h_t[n] + Dskip[h] x[b,t,h,p]
 *
 *   x, y        : [batch, L, H, P] dtype
 *   dt          : [batch, L, H] dtype (before the softplus)
 *   B, C        : [batch, L, N] dtype (one group shared by all heads)
 *   dt_bias     : [H] float32 (NULL means 0);  A : [H] float32
 *   Dskip       : [H] float32 (NULL means 0)
 *   h_last      : [batch, H, P, N] float32, written (NULL: not written); the
 *                 layout of ssm_step's state with D = H * P channels
 * bf16 with P == 64, N == 64 or 128 and x, B, C, y 16-byte aligned runs the
 * tensor-core chunked kernel (the products in bf16, every sum in fp32);
 * anything else runs a one-thread-per-channel kernel.  The tensor-core kernel
 * takes one head per CTA, and allocates nothing, unless that would leave its
 * last wave of CTAs mostly empty (batch * H above the SM count, and the waves
 * rounded up more than 15% above the heads' share of the SMs).  Then
 * persistent CTAs take segments of heads from a ticket counter and pass each
 * head's state between segments through a stream-ordered workspace of about
 * batch * H * 32 KB (SSM_ERR_NOMEM if that allocation fails); the results are
 * the same bits either way.
 * Returns an ssm_status_t.
 */
SSM_API int ssm_ssd_fwd(const void *x, const void *dt, const float *dt_bias, const float *A,
                        const void *B, const void *C, const float *Dskip, void *y, float *h_last,
                        int64_t batch, int64_t L, int64_t H, int64_t P, int64_t N, int dtype,
                        void *stream);

/*
 * ssm_step -- one decode token: the same per-token update as one step of
 * ssm_scan_fwd, applied in place to a stored state (the recurrent,
 * constant-cost inference form; ta-paperlens page, S4 section).
 *
 *   state       : [batch, D, N] float32, read and overwritten in place
 *   u, delta, z : [batch, D] dtype           (z may be NULL: no gate)
 *   B, C        : [batch, N] dtype
 *   dt_bias     : [D] float32 (NULL means 0);  A : [D, N] float32
 *   Dskip       : [D] float32 (NULL means 0)
 *   y           : [batch, D] dtype, written
 * Sizes: batch, D >= 0; 1 <= N <= SSM_MAX_N.  Allocates nothing.
 * Returns an ssm_status_t.
 */
SSM_API int ssm_step(float *state, const void *u, const void *delta,
             const float *dt_bias, const float *A, const void *B,
             const void *C, const float *Dskip, const void *z, void *y,
             int64_t batch, int64_t D, int64_t N, int dtype, void *stream);

/*
 * ssm_scan_fwd_noalloc -- ssm_scan_fwd for callers that cannot allocate.
 *
 * The pages describe no such call; it exists for library users whose code
 * must not allocate device memory while it runs: a server that reserves all
 * of its memory up front in its own pool, or code running where a
 * cudaMalloc/cudaMallocAsync would synchronise the device, fail, or is not
 * allowed.  Arguments, layouts, results and errors are those of ssm_scan_fwd.
 * The difference is where the N == 16 fast kernel keeps its scratch (its unit
 * counter, per-chain progress flags and, when h_last is NULL, the state
 * carried between chunks): in one fixed device array of
 * SSM_NOALLOC_SCRATCH_BYTES inside this library, which every GPU that loads
 * the library holds until the process exits.  It always runs the chained
 * plan of that kernel; inputs that kernel does not take (N != 16, tensors not
 * 16-byte aligned, D * sizeof(dtype) not a multiple of 16) run the generic
 * kernel, which needs no scratch.  Nothing here calls cudaMalloc, cudaFree
 * or any allocating routine.
 *
 * The chained plan keeps one 128-channel block of one batch entry on one CTA
 * at a time, so a problem with fewer such blocks (batch * ceil(D/128)) than
 * resident CTAs (one per SM) runs on that fraction of the GPU: the 1 x 1M x
 * 1536 long sequence, 12 blocks, uses 12 SMs here, where ssm_scan_fwd splits
 * the sequence over the whole GPU with a stream-ordered workspace of about
 * (P-1)*batch*D*68 + P*batch*D*64 bytes for P sequence pieces.
 *
 *   - Limit: 256 + 4 * batch * ceil(D/32) bytes (rounded up to 256), plus
 *     64 * batch * D bytes when h_last is NULL, must fit in
 *     SSM_NOALLOC_SCRATCH_BYTES; otherwise SSM_ERR_SCRATCH is returned before
 *     anything is enqueued.  (batch 4, D 5120 needs 2.8 KB with h_last and
 *     1.3 MB without.)
 *   - The first call in each context of a device looks up the array's
 *     device address with that device current, sets the kernel's
 *     shared-memory attribute and queries its occupancy (a context made
 *     after cudaDeviceReset counts as new).  Make that first call before
 *     any stream capture.
 *   - All calls share the one array, and it keeps the last call's contents
 *     (each call clears the parts that must start at zero).  Calls whose
 *     work overlaps on the GPU -- on different streams, or from different
 *     host threads -- race on it and must be serialised by the caller.
 */
#define SSM_NOALLOC_SCRATCH_BYTES (4u << 20)
SSM_API int ssm_scan_fwd_noalloc(const void *u, const void *delta, const float *dt_bias,
                                 const float *A, const void *B, const void *C,
                                 const float *Dskip, const void *z, void *y, float *h_last,
                                 int64_t batch, int64_t L, int64_t D, int64_t N, int dtype,
                                 void *stream);

/*
 * ssm_device_status -- synchronises `stream`, then reads and clears this
 * device's error word, which the kernels set when a bounded device-side
 * wait gives up.  Returns SSM_OK, SSM_ERR_TIMEOUT, or SSM_ERR_CUDA if the
 * synchronisation itself failed.
 */
SSM_API int ssm_device_status(void *stream);

/* Static, human-readable text for a status code (never NULL). */
SSM_API const char *ssm_status_string(int status);

/* Library ABI version (this header describes version 1). */
SSM_API int ssm_abi_version(void);

/*
 * ssm_unit_ceilings -- measures, on the current device, the rates of the
 * three execution units that bound the scan kernels, so that a benchmark can
 * set its throughput beside ceilings measured on the same GPU in the same
 * process.  The pages have no counterpart; this is measurement support.
 *   out[0]  fp32 multiply-adds per second (packed f32x2 stream, all SMs)
 *   out[1]  2^x results of the special-function unit per second (all SMs)
 *   out[2]  warp instructions issued per second (scalar multiply-add
 *           stream, all SMs)
 * Each rate is the best of `reps` (>= 1) launches timed with CUDA events on
 * `stream`; the call synchronises `stream` and allocates nothing.  Returns
 * SSM_ERR_NULL for out == NULL, SSM_ERR_SIZE for reps < 1, SSM_ERR_CUDA if a
 * launch or event failed.
 */
SSM_API int ssm_unit_ceilings(double *out, int reps, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SSMSCAN_H */
