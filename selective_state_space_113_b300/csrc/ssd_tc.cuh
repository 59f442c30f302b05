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
// The masked scores go back into TMEM (packed bf16 pairs, the A operand of
// Yi); C, B and X are double-buffered, so a chunk's loads and its S overlap
// the previous chunk's epilogue, and so is C H in TMEM, so that C H of a chunk
// can go as soon as its entering state is written.
//
// ssd_tc_kernel: one CTA owns one (b, h) and walks its chunks in order.
// ssd_tc_dyn_kernel, the same roles and products on a ticket walk: head j =
// b H + h is cut into segments of U chunks, and each (head, segment) is a
// unit.  Persistent CTAs, one per SM, take units from a ticket counter,
// segment-major (ticket t is segment t / heads of head t % heads), and walk
// each in chunk order.  A unit's predecessor in its head went out `heads`
// tickets earlier and has long finished when the unit needs its state, which
// comes fp32 through global memory behind a counter the eight epilogue warps
// release.  Tickets go only to CTAs that are running, and a unit waits only
// on a smaller ticket, taken by a CTA that walks its units in order: the walk
// cannot deadlock, even with some CTAs not yet resident (another stream's
// kernel on some SMs).  It is the launch's choice where one head per CTA
// would leave the last wave mostly empty (see launch_ssd_tc).  Ten warps in
// both:
//   warp 8      products: one elected thread issues the MMAs, each as soon as
//               what it reads is written and its accumulator has been read,
//               in the order the epilogue produces them: C H of chunk c (the
//               state after c - 1), G (w o X of c, signalled apart from the
//               scores), Yi (the masked scores of c), then S of c + 1;
//   warp 9      copies and decays: TMA loads of a chunk's C, B (K-major, two
//               64-wide regions each) and X (its 128 steps x 64 channels) into
//               one of two buffers once the epilogue is done with the buffer,
//               and, for the whole warp, each chunk's step sizes and
//               cumulative decay (from dt values loaded a chunk ahead) once the
//               previous chunk's scores have read the shared copy.  Kept apart
//               from warp 8 because an MMA issue can stall until the tensor
//               cores take it;
//   warps 0..7  epilogue, two warps per TMEM lane quadrant (warp e serves
//               lanes 32 (e % 4) .. +31, i.e. rows of every product, and one
//               half of its columns): w o X, the masked scores, the outputs,
//               and the state, which it keeps in registers (thread n holds
//               half of row n of H) and rewrites after each chunk as the next
//               chunk's hi + lo operand.
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
constexpr int kEpWarps = 8;      // two per TMEM lane quadrant, each half the columns
constexpr int THREADS = 32 * (kEpWarps + 2);
constexpr int kCtl = kEpWarps;       // the warp that issues the products
constexpr int kLdr = kEpWarps + 1;   // the warp that issues the copies and forms the decays
constexpr float kLog2e = 1.4426950408889634f;

// Shared memory: every operand tile is 1024-byte aligned, rows of 128 bytes,
// 8-row atoms of 1 KB, 16-byte chunks swizzled by the row's index mod 8.
struct Layout {
    // input buffer i at kIn + i * kInBytes: C (2 regions [128 t][64 n], 16 KB
    // each), B (2 regions [128 s][64 n]), X ([128 s][64 p])
    static constexpr int kInBytes = 81920;
    static constexpr int kC = 0, kB = 32768, kX = 65536;   // offsets inside a buffer
    static constexpr int kWh = 2 * kInBytes;  // w o X, hi: [128 s][64 p]
    static constexpr int kWl = kWh + 16384;   //        lo
    static constexpr int kHh = kWl + 16384;   // entering state, hi: [128 n][64 p]
    static constexpr int kHl = kHh + 16384;   //                 lo
    static constexpr int kCum = kHl + 16384;  // cum_t log2(e), [Q] float
    static constexpr int kDt = kCum + 512;    // dt_t, [Q] float
    static constexpr int kBar = kDt + 512;    // mbarriers
    static constexpr int kNumBars = 12;
    static constexpr int kTmem = kBar + 8 * kNumBars;   // TMEM base address (written by alloc)
    static constexpr int kBytes = kTmem + 16;
    static constexpr int kSmemBytes = kBytes + 1024;    // + slack to align the base
};
static_assert(Layout::kSmemBytes <= 227 * 1024, "CTA shared memory");

// TMEM columns: the fp32 accumulators (lane = row; C H in two buffers, by
// chunk parity), then the masked scores as the A operand of Yi (packed bf16
// pairs, s = 2c and 2c+1 in column c).
constexpr uint32_t kColS = 0, kColYx0 = 128, kColYi = 192, kColG = 256;
constexpr uint32_t kColSh = 320, kColSl = 384, kColYx1 = 448;
constexpr uint32_t kTmemCols = 512;

// kInFull[2] / kInFree[2]: a buffer's C, B, X landed / the epilogue is done
// with them; kMmaS, kMmaYx, kMmaYi, kMmaG: S, C H, the masked product, G
// completed; kWxReady: w o X is written (by the four warps that form it);
// kEpReady: the masked scores are written; kHReady: the entering state's copy
// is written; kCum: the cumulative decays are written.
enum Bar : int { kInFull = 0, kInFree = 2, kMmaS = 4, kMmaYx, kEpReady, kMmaYi, kMmaG, kHReady,
                 kCum, kWxReady };
static_assert(kWxReady + 1 <= Layout::kNumBars, "barrier count");
constexpr int kWxWarps = 4;   // the epilogue warps of lane quadrants 0 and 1

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

// The ticket walk's arguments: those of the one-head walk, and its own, in a
// struct of its own.  The one-head kernel, given these fields after its own
// (its parameters at 520 bytes instead of 480), ran 13% slower, registers and
// shared memory unchanged; the ticket kernel ran the same with 504 or 488
// bytes of parameters (measured; the cause was not isolated).  The parameters
// are kept within 512 bytes.
struct ArgsDyn {
    const bf16* x;
    const bf16* dt;
    const float* dt_bias;
    const float* A;
    const float* Dskip;
    bf16* y;
    float* h_last;
    unsigned long long* ticket;   // units handed out (NULL: one unit per CTA, its index)
    float* carry;                 // [heads][NP][P]: the state after a head's last segment done
    unsigned* done;               // [heads]: 8 x the segments of the head done
    long long batch, L, H;
    int N;
    int seg;                      // U, chunks per segment
    unsigned long long wait_ns;
};
static_assert(sizeof(ArgsDyn) == 120 && 3 * sizeof(CUtensorMap) + sizeof(ArgsDyn) <= 512,
              "ticket kernel parameters");

// The ticket walk's shared memory: the one-head layout up to the step sizes,
// then the two chunk records and the CTA's first ticket, the barriers and
// the TMEM address.
struct LayoutDyn {
    static constexpr int kRec = Layout::kDt + 512;   // ChunkRec of the k-th chunk at [k % 2]
    static constexpr int kFirst = kRec + 96;          // the CTA's first ticket
    static constexpr int kBar = kFirst + 16;          // mbarriers
    static constexpr int kTmem = kBar + 8 * Layout::kNumBars;
    static constexpr int kBytes = kTmem + 16;
    static constexpr int kSmemBytes = kBytes + 1024;
};
static_assert(LayoutDyn::kSmemBytes <= 227 * 1024, "CTA shared memory");

// The unit a CTA walks and its chunk: head j, segment sg, chunk c of the
// head, and the end hi of the segment's chunks.
struct Walk {
    int j, sg, c, hi;
    __device__ __forceinline__ void unit(long long t, long long heads, int U, int nch) {
        sg = (int)(t / heads);
        j = (int)(t - (long long)sg * heads);
        c = sg * U;
        hi = c + U < nch ? c + U : nch;
    }
};

// A load issued here, in program order with the other volatile asm (the
// waits), so that its latency passes while the warp goes on.
__device__ __forceinline__ float ld_early(const float* p) {
    float v;
    asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

// What the epilogue (and, for `next`, the product warp) needs of the k-th
// chunk a CTA walks, written by the copy warp with the chunk's decays: where
// its outputs go, how its state enters (`start`: it continues the chunk
// before, starts its head from zero, or continues the segment before, done
// by whichever CTA), whether the state after it leaves (`end`: as h_last, or
// for the head's next segment), and how the next chunk's enters (`next`,
// with that chunk's head and segment; kNone: no next chunk).
enum : int { kCont = 0, kZero = 1, kHand = 2, kNone = 3 };   // start / next
enum : int { kEndNone = 0, kEndHead = 1, kEndHand = 2 };      // end
struct ChunkRec {
    int b, h, c, nv, j, sg, start, end, next, nj, nsg;
    float dsk;
};
static_assert(sizeof(ChunkRec) == 48, "record size");

__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Bounded wait for a counter in global memory to reach `target` (acquire).
__device__ __forceinline__ bool wait_count(const unsigned* p, unsigned target,
                                           unsigned long long ns) {
    const uint64_t t0 = ptx::globaltimer();
    while (ptx::ld_acquire(p) < target) {
        if (ptx::globaltimer() - t0 > ns) return false;
        ptx::nanosleep(128);
    }
    return true;
}


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

// 16 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}

// A-from-TMEM product: [d_tmem] (+)= [a_tmem] x (shared-memory operand b).
__device__ __forceinline__ void mma_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t id,
                                       int accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(id), "r"(accumulate)
        : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane, without waiting:
// the values are valid after a later tcgen05.wait::ld.
__device__ __forceinline__ void tmem_ld32_nowait(uint32_t taddr, float (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]),
          "=f"(v[7]), "=f"(v[8]), "=f"(v[9]), "=f"(v[10]), "=f"(v[11]), "=f"(v[12]),
          "=f"(v[13]), "=f"(v[14]), "=f"(v[15]), "=f"(v[16]), "=f"(v[17]), "=f"(v[18]),
          "=f"(v[19]), "=f"(v[20]), "=f"(v[21]), "=f"(v[22]), "=f"(v[23]), "=f"(v[24]),
          "=f"(v[25]), "=f"(v[26]), "=f"(v[27]), "=f"(v[28]), "=f"(v[29]), "=f"(v[30]),
          "=f"(v[31])
        : "r"(taddr));
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
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const long long bh = blockIdx.x;
    const long long b = bh / a.H, hh = bh % a.H;
    const long long nchunks = (a.L + Q - 1) / Q;
    const bool two_regions = a.N > 64;

    // ---- set-up: barriers, zeroed state operand and padding regions, TMEM
    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(&bar[kInFull + i], 1);
            ptx::mbar_init(&bar[kInFree + i], kEpWarps);
        }
        ptx::mbar_init(&bar[kMmaS], 1);
        ptx::mbar_init(&bar[kMmaYx], 1);
        ptx::mbar_init(&bar[kEpReady], kEpWarps);
        ptx::mbar_init(&bar[kMmaYi], 1);
        ptx::mbar_init(&bar[kMmaG], 1);
        ptx::mbar_init(&bar[kHReady], kEpWarps);
        ptx::mbar_init(&bar[kCum], 1);
        ptx::mbar_init(&bar[kWxReady], kWxWarps);
        ptx::fence_mbar_init();
    }
    {
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
        for (int i = tid; i < 2 * 16384 / 16; i += THREADS) {
            reinterpret_cast<uint4*>(sm + Layout::kHh)[i] = z;   // kHh and kHl are adjacent
            if (!two_regions) {
                const int j = i % 1024, buf = i / 1024;
                unsigned char* in = sm + buf * Layout::kInBytes;
                reinterpret_cast<uint4*>(in + Layout::kC + 16384)[j] = z;
                reinterpret_cast<uint4*>(in + Layout::kB + 16384)[j] = z;
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

    if (warp >= kCtl) {
        // ------------------------------------------------------------- control
        // Two warps, so that neither holds the other back: an MMA issue can
        // stall until the tensor cores take it.  Warp kCtl: lane 0 issues
        // the products.  Warp kLdr: lane 0 issues the copies, and the whole
        // warp computes the step sizes and the cumulative decay of each
        // chunk.  Both wait as whole warps.
        const bool leader = lane == 0;
        if (leader && warp == kLdr) {
            ptx::prefetch_tensormap(&tmX);
            ptx::prefetch_tensormap(&tmB);
            ptx::prefetch_tensormap(&tmC);
        }
        const uint32_t in_bytes = (two_regions ? 4 : 2) * 16384 + 16384;
        const uint32_t s0 = ptx::smem_u32(sm);
        const uint32_t sWh = s0 + Layout::kWh, sWl = s0 + Layout::kWl;
        const uint32_t sHh = s0 + Layout::kHh, sHl = s0 + Layout::kHl;
        constexpr uint32_t idS = idesc(128, 128, 0, 0), idY = idesc(128, 64, 0, 1),
                           idG = idesc(128, 64, 1, 1);
        const float A = a.A[hh];
        const float kb2 = a.dt_bias ? a.dt_bias[hh] * kLog2e : 0.0f;
        auto load = [&](long long c) {   // chunk c into buffer c % 2
            const int i = (int)(c & 1);
            unsigned char* in = sm + i * Layout::kInBytes;
            uint64_t* full = &bar[kInFull + i];
            const int t0 = (int)(c * Q);
            ptx::mbar_arrive_expect_tx(full, in_bytes);
            ptx::tma_load_3d(in + Layout::kC, &tmC, full, 0, t0, (int)b);
            ptx::tma_load_3d(in + Layout::kB, &tmB, full, 0, t0, (int)b);
            if (two_regions) {
                ptx::tma_load_3d(in + Layout::kC + 16384, &tmC, full, 64, t0, (int)b);
                ptx::tma_load_3d(in + Layout::kB + 16384, &tmB, full, 64, t0, (int)b);
            }
            ptx::tma_load_4d(in + Layout::kX, &tmX, full, 0, (int)hh, t0, (int)b);
        };
        // The descriptors of a product are formed once and stepped per K
        // slice: the start address sits in the low 14 bits (in 16-byte
        // units; shared memory is below 256 KB), so adding a slice's offset
        // in 16-byte units moves only that field.  Each MMA is then an add
        // and the instruction; this thread shares its SM sub-partition with
        // two epilogue warps, and the tensor cores wait for what it issues.
        // K-major operands (C, and B as S's operand): slice k at
        // (k / 4) * 16384 + (k % 4) * 32 bytes; MN-major ones: k * 2048.
        auto koff = [](int k) { return (uint64_t)((k >> 2) * 1024 + (k & 3) * 2); };
        auto issue_s = [&](long long c) {   // S = C B^T
            const uint32_t in = s0 + (uint32_t)((c & 1) * Layout::kInBytes);
            const uint64_t da = sdesc(in + Layout::kC, 16, 1024), db = sdesc(in + Layout::kB, 16, 1024);
#pragma unroll
            for (int k = 0; k < 8; ++k) mma(tmem + kColS, da + koff(k), db + koff(k), idS, k > 0);
            mma_commit(&bar[kMmaS]);
        };
        auto issue_yx = [&](long long c) {   // Yx = C H into buffer c % 2, H as hi then lo
            const uint32_t in = s0 + (uint32_t)((c & 1) * Layout::kInBytes);
            const uint32_t col = tmem + ((c & 1) ? kColYx1 : kColYx0);
            const uint64_t da = sdesc(in + Layout::kC, 16, 1024);
            const uint64_t dh = sdesc(sHh, 16384, 1024), dl = sdesc(sHl, 16384, 1024);
#pragma unroll
            for (int k = 0; k < 8; ++k) mma(col, da + koff(k), dh + (uint64_t)(k * 128), idY, k > 0);
#pragma unroll
            for (int k = 0; k < 8; ++k) mma(col, da + koff(k), dl + (uint64_t)(k * 128), idY, 1);
            mma_commit(&bar[kMmaYx]);
        };
        auto issue_g = [&](long long c) {   // G = B^T (w o X)
            const uint32_t in = s0 + (uint32_t)((c & 1) * Layout::kInBytes);
            const uint64_t db = sdesc(in + Layout::kB, 16384, 1024);
            const uint64_t dh = sdesc(sWh, 16384, 1024), dl = sdesc(sWl, 16384, 1024);
#pragma unroll
            for (int k = 0; k < 8; ++k)
                mma(tmem + kColG, db + (uint64_t)(k * 128), dh + (uint64_t)(k * 128), idG, k > 0);
#pragma unroll
            for (int k = 0; k < 8; ++k) mma(tmem + kColG, db + (uint64_t)(k * 128), dl + (uint64_t)(k * 128), idG, 1);
            mma_commit(&bar[kMmaG]);
        };
        auto issue_yi = [&](long long c) {   // Yi = (masked S) X
            const uint32_t in = s0 + (uint32_t)((c & 1) * Layout::kInBytes);
            const uint64_t dx = sdesc(in + Layout::kX, 16384, 1024);
#pragma unroll
            for (int k = 0; k < 8; ++k)
                mma_ta(tmem + kColYi, tmem + kColSh + 8 * k, dx + (uint64_t)(k * 128), idY, k > 0);
#pragma unroll
            for (int k = 0; k < 8; ++k) mma_ta(tmem + kColYi, tmem + kColSl + 8 * k, dx + (uint64_t)(k * 128), idY, 1);
            mma_commit(&bar[kMmaYi]);
        };
        auto wait = [&](int which, long long k) {   // k-th completion of a barrier, whole warp
            return __all_sync(0xffffffffu, bwait(&bar[which], (uint32_t)(k & 1), a.wait_ns));
        };
        // raw dt of the steps 4 lane .. 4 lane + 3 of a chunk (a chunk ahead),
        // kept as loaded: nothing here uses the values, so the loads complete
        // while this warp goes on (steps past L read the last one, and the
        // decay masks them)
        unsigned short raw[4];
        auto load_dt = [&](long long c) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const long long t = c * Q + 4 * lane + j;
                raw[j] = reinterpret_cast<const unsigned short*>(a.dt)[(b * a.L + (t < a.L ? t : a.L - 1)) * a.H + hh];
            }
        };
        // step sizes and cumulative decay of chunk c into the shared copy (its
        // previous readers, the masked scores of chunk c - 1, are done)
        auto scan = [&](long long c) {
            const int nv = (int)(a.L - c * Q < Q ? a.L - c * Q : Q);
            float d[4], cl[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float v2 = fmaf(__bfloat162float(__ushort_as_bfloat16(raw[j])), kLog2e, kb2);
                const float sp = (v2 > 28.853901f ? v2 : ptx::lg2(1.0f + ptx::ex2(v2))) * 0.6931471805599453f;
                d[j] = 4 * lane + j < nv ? sp : 0.0f;
                cl[j] = (j ? cl[j - 1] : 0.0f) + A * d[j];
            }
            float inc = cl[3];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float v = __shfl_up_sync(0xffffffffu, inc, o);
                if (lane >= o) inc += v;
            }
            const float ex = inc - cl[3];
            *reinterpret_cast<float4*>(cum + 4 * lane) =
                make_float4((cl[0] + ex) * kLog2e, (cl[1] + ex) * kLog2e, (cl[2] + ex) * kLog2e,
                            (cl[3] + ex) * kLog2e);
            *reinterpret_cast<float4*>(dts + 4 * lane) = make_float4(d[0], d[1], d[2], d[3]);
            __syncwarp();
            if (leader) ptx::mbar_arrive(&bar[kCum]);
        };
        if (warp == kLdr) {
            // The first two chunks' copies and chunk 0's decay; then, per
            // chunk c, the copies of chunk c + 1 once the outputs of chunk
            // c - 1 are done with its buffer, and the decay of chunk c + 1
            // once the scores of chunk c have read the shared copy (the
            // order in which the epilogue's iteration for chunk c frees them).
            load_dt(0);
            scan(0);
            if (nchunks > 1) load_dt(1);
            if (leader) {
                load(0);
                if (nchunks > 1) load(1);
            }
            for (long long c = 0; c + 1 < nchunks && !failed; ++c) {
                if (c > 0) {
                    if (!wait(kInFree + (int)((c - 1) & 1), (c - 1) >> 1)) { failed = true; break; }
                    if (leader) load(c + 1);
                }
                if (!wait(kEpReady, c)) { failed = true; break; }
                scan(c + 1);
                if (c + 2 < nchunks) load_dt(c + 2);
            }
            // Every copy issued here is waited for by the product warp
            // before the products that read it.
            if (failed && leader) atomicOr(&g_error_word, kErrTimeout);
            __syncwarp();
        } else {
            // chunk 0's S and C H (of the zero state)
            if (!wait(kInFull, 0)) failed = true;
            if (!failed) {
                fence_after_sync();
                if (leader) issue_s(0);
                if (!wait(kHReady, 0)) failed = true;
            }
            if (!failed) {
                fence_after_sync();
                if (leader) issue_yx(0);
            }
            // Each product goes as soon as what it reads is written and its
            // accumulator has been read, in the order the epilogue's phases
            // produce them within its iteration for chunk c (the state after
            // chunk c - 1, w o X of chunk c, the outputs of chunk c - 1, the
            // masked scores of chunk c): this thread issues in order, so a
            // wait on a later event would hold back an earlier product.
            for (long long c = 0; c < nchunks && !failed; ++c) {
                if (c > 0) {
                    // The state entering chunk c is written, and every
                    // epilogue warp has read G of chunk c - 1.  C H of chunk
                    // c goes into buffer c % 2, last read by the outputs of
                    // chunk c - 2, which precede the scores of chunk c - 1
                    // (kEpReady, seen in the previous iteration); C of chunk
                    // c landed before its S went.
                    if (!wait(kHReady, c)) { failed = true; break; }
                    fence_after_sync();
                    if (leader) issue_yx(c);
                }
                // G(c): w o X of chunk c is written
                if (!wait(kWxReady, c)) { failed = true; break; }
                fence_after_sync();
                if (leader) issue_g(c);
                // Yi(c): the masked scores of chunk c are in TMEM; then S of
                // chunk c + 1 (S of chunk c has been read)
                if (!wait(kEpReady, c)) { failed = true; break; }
                fence_after_sync();
                if (leader) issue_yi(c);
                if (c + 1 < nchunks) {
                    if (!wait(kInFull + (int)((c + 1) & 1), (c + 1) >> 1)) { failed = true; break; }
                    fence_after_sync();
                    if (leader) issue_s(c + 1);
                }
            }
            // Leave no product in flight (bounded): the last chunk's Yi,
            // the last product issued, completes after all of them; a
            // parity wait names the last phase alone, and Yi of the chunk
            // before completed (the outputs of that chunk, which precede
            // the last chunk's scores, waited for it).
            if (nchunks > 0 && !failed && !wait(kMmaYi, nchunks - 1)) failed = true;
            if (failed && leader) atomicOr(&g_error_word, kErrTimeout);
            __syncwarp();
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int quad = warp & 3, hf = warp >> 2;   // TMEM lane quadrant; column half
        const int row = 32 * quad + lane;            // step t, or state row n
        const uint32_t lane_addr = tmem + ((uint32_t)(32 * quad) << 16);
        const float dsk = a.Dskip ? a.Dskip[hh] : 0.0f;
        float Hs[32];   // columns 32 hf .. 32 hf + 31 of row `row` of the state
#pragma unroll
        for (int j = 0; j < 32; ++j) Hs[j] = 0.0f;
        // The state after chunk c - 1: H <- exp(cum_end) H + G (row n = row,
        // this warp's 32 columns), then its hi + lo copy for chunk c's C H
        // (the previous copy was read by chunk c - 1's Yx, which completed).
        auto state_update = [&](long long c, float dend) -> bool {
            if (!wwait(&bar[kMmaG], (uint32_t)(c & 1), a.wait_ns) ||
                !wwait(&bar[kMmaYx], (uint32_t)(c & 1), a.wait_ns))
                return false;
            fence_after_sync();
            float g[32];
            tmem_ld32(lane_addr + kColG + 32 * hf, g);
#pragma unroll
            for (int j = 0; j < 32; ++j) Hs[j] = fmaf(dend, Hs[j], g[j]);
            store_split32(sm + Layout::kHh, sm + Layout::kHl, row, 4 * hf, Hs);
            ptx::fence_proxy_async_shared();
            fence_before_sync();
            warp_arrive(&bar[kHReady], lane);
            return true;
        };
        // The outputs of chunk c, step t = row, this warp's 32 columns:
        // Yi + exp(cum_t) Yx + Dskip x; then chunk c's buffer is free.
        auto outputs = [&](long long c, float ecum) -> bool {
            if (!wwait(&bar[kMmaYi], (uint32_t)(c & 1), a.wait_ns)) return false;
            fence_after_sync();
            const unsigned char* X = sm + (c & 1) * Layout::kInBytes + Layout::kX;
            const int nv = (int)(a.L - c * Q < Q ? a.L - c * Q : Q);
            float yi[32], yx[32];
            tmem_ld32_nowait(lane_addr + kColYi + 32 * hf, yi);
            tmem_ld32_nowait(lane_addr + ((c & 1) ? kColYx1 : kColYx0) + 32 * hf, yx);
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            bf16* yrow = a.y + ((b * a.L + c * Q + row) * a.H + hh) * P + 32 * hf;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                const uint4 xv = *reinterpret_cast<const uint4*>(X + sw128(row, 4 * hf + cc));
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
                if (row < nv) *reinterpret_cast<uint4*>(yrow + 8 * cc) = o;
            }
            // X (read above and by Yi) and B (read by G) are free for chunk c + 2
            fence_before_sync();
            warp_arrive(&bar[kInFree + (int)(c & 1)], lane);
            return true;
        };
        // the zero entering state is in place
        fence_before_sync();
        warp_arrive(&bar[kHReady], lane);
        float ecum_prev = 0.0f, dend_prev = 0.0f;
        for (long long c = 0; c < nchunks && !failed; ++c) {
            const uint32_t ph = (uint32_t)(c & 1);
            const unsigned char* X = sm + (c & 1) * Layout::kInBytes + Layout::kX;
            // the previous chunk's state (its G ran first) lets chunk c's C H go
            if (c > 0 && !state_update(c - 1, dend_prev)) { failed = true; break; }
            // this row's cumulative decay (log2 units) and step size, and the chunk's total
            if (!wwait(&bar[kCum], ph, a.wait_ns)) { failed = true; break; }
            const float ct = cum[row], cend2 = cum[Q - 1];
            const float ecum = ptx::ex2(ct);                 // exp(cum_t)
            const float dend = ptx::ex2(cend2);              // exp(cum_end)
            if (!wwait(&bar[kInFull + (int)(c & 1)], (uint32_t)((c >> 1) & 1), a.wait_ns)) {
                failed = true;
                break;
            }
            // w o X, split hi + lo (the previous chunk's G, which read them,
            // completed: state_update).  The causal mask gives the warps of
            // lane quadrants 2 and 3 the most score columns, so the warps of
            // quadrants 0 and 1 form all of w o X: warp e < 4 (quad 0 or 1,
            // column half hf) takes rows s = 32 (e & 1) + lane and s + 64 of
            // its column half, with the w_s of those rows from the shared copy.
            if (quad < 2) {
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    const int s_ = 32 * quad + 64 * rr + lane;
                    const float ws = ptx::ex2(cend2 - cum[s_]) * dts[s_];
#pragma unroll
                    for (int cc = 4 * hf; cc < 4 * hf + 4; ++cc) {
                        const uint4 xv = *reinterpret_cast<const uint4*>(X + sw128(s_, cc));
                        const __nv_bfloat162* x2 = reinterpret_cast<const __nv_bfloat162*>(&xv);
                        uint4 h, l;
                        uint32_t* hp = &h.x;
                        uint32_t* lp = &l.x;
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float2 f = __bfloat1622float2(x2[q]);
                            split2(ws * f.x, ws * f.y, hp[q], lp[q]);
                        }
                        *reinterpret_cast<uint4*>(sm + Layout::kWh + sw128(s_, cc)) = h;
                        *reinterpret_cast<uint4*>(sm + Layout::kWl + sw128(s_, cc)) = l;
                    }
                }
                ptx::fence_proxy_async_shared();   // w o X, for the tensor cores (G)
                warp_arrive(&bar[kWxReady], lane);
            }
            // the previous chunk's outputs (its Yi ran after G)
            if (c > 0 && !outputs(c - 1, ecum_prev)) { failed = true; break; }
            // masked scores of row t = row, pieces hf and hf + 2 (32 columns
            // each): S[t,s] exp(cum_t - cum_s) dt_s for s <= t, into TMEM as
            // packed bf16 hi and lo (the previous chunk's Yi, which read them,
            // completed: outputs)
            if (!wwait(&bar[kMmaS], ph, a.wait_ns)) {
                failed = true;
                break;
            }
            fence_after_sync();
            float sv[2][32];
            tmem_ld32_nowait(lane_addr + kColS + 32 * hf, sv[0]);
            if (hf + 2 <= quad) tmem_ld32_nowait(lane_addr + kColS + 32 * (hf + 2), sv[1]);
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int piece = hf + 2 * k;
                uint32_t hi[16], lo[16];
                if (piece <= quad) {   // some s of the piece are <= t (warp-uniform)
                    float (&v)[32] = sv[k];
                    const float4* cum4 = reinterpret_cast<const float4*>(cum + 32 * piece);
                    const float4* dt4 = reinterpret_cast<const float4*>(dts + 32 * piece);
#pragma unroll
                    for (int j4 = 0; j4 < 8; ++j4) {
                        const float4 cq = cum4[j4], dq = dt4[j4];
                        const float cs[4] = {cq.x, cq.y, cq.z, cq.w}, ds[4] = {dq.x, dq.y, dq.z, dq.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int j = 4 * j4 + e, s_ = 32 * piece + j;
                            v[j] = s_ <= row ? v[j] * ptx::ex2(ct - cs[e]) * ds[e] : 0.0f;
                        }
                    }
#pragma unroll
                    for (int j = 0; j < 16; ++j) split2(v[2 * j], v[2 * j + 1], hi[j], lo[j]);
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) hi[j] = lo[j] = 0u;
                }
                tmem_st16(lane_addr + kColSh + 16 * piece, hi);
                tmem_st16(lane_addr + kColSl + 16 * piece, lo);
            }
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            ptx::fence_proxy_async_shared();   // w o X, for the tensor cores
            fence_before_sync();
            warp_arrive(&bar[kEpReady], lane);
            ecum_prev = ecum;
            dend_prev = dend;
        }
        // the last chunk's state and outputs
        if (!failed && nchunks > 0) {
            if (!state_update(nchunks - 1, dend_prev) || !outputs(nchunks - 1, ecum_prev))
                failed = true;
        }
        if (failed && lane == 0) atomicOr(&g_error_word, kErrTimeout);
        if (!failed && a.h_last && row < a.N) {
            float* base = a.h_last + (b * a.H + hh) * P * (long long)a.N + row;
#pragma unroll
            for (int j = 0; j < 32; ++j) base[(long long)(32 * hf + j) * a.N] = Hs[j];
        }
    }
    // ---- tear-down: every TMEM access and MMA is done before the columns go
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (warp == kCtl)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
}

__global__ void __launch_bounds__(THREADS, 1)
ssd_tc_dyn_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmB,
                  const __grid_constant__ CUtensorMap tmC, const ArgsDyn a) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* sm = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + LayoutDyn::kBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + LayoutDyn::kTmem);
    float* cum = reinterpret_cast<float*>(sm + Layout::kCum);
    float* dts = reinterpret_cast<float*>(sm + Layout::kDt);
    ChunkRec* recs = reinterpret_cast<ChunkRec*>(sm + LayoutDyn::kRec);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nchunks = (int)((a.L + Q - 1) / Q);
    const long long heads = a.batch * a.H;
    const bool two_regions = a.N > 64;
    unsigned long long* first = reinterpret_cast<unsigned long long*>(sm + LayoutDyn::kFirst);

    // ---- set-up: barriers, zeroed state operand and padding regions, TMEM
    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(&bar[kInFull + i], 1);
            ptx::mbar_init(&bar[kInFree + i], kEpWarps);
        }
        ptx::mbar_init(&bar[kMmaS], 1);
        ptx::mbar_init(&bar[kMmaYx], 1);
        ptx::mbar_init(&bar[kEpReady], kEpWarps);
        ptx::mbar_init(&bar[kMmaYi], 1);
        ptx::mbar_init(&bar[kMmaG], 1);
        ptx::mbar_init(&bar[kHReady], kEpWarps);
        ptx::mbar_init(&bar[kCum], 1);
        ptx::mbar_init(&bar[kWxReady], kWxWarps);
        ptx::fence_mbar_init();
        *first = a.ticket ? atomicAdd(a.ticket, 1ull) : (unsigned long long)blockIdx.x;
    }
    {
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
        for (int i = tid; i < 2 * 16384 / 16; i += THREADS) {
            reinterpret_cast<uint4*>(sm + Layout::kHh)[i] = z;   // kHh and kHl are adjacent
            if (!two_regions) {
                const int j = i % 1024, buf = i / 1024;
                unsigned char* in = sm + buf * Layout::kInBytes;
                reinterpret_cast<uint4*>(in + Layout::kC + 16384)[j] = z;
                reinterpret_cast<uint4*>(in + Layout::kB + 16384)[j] = z;
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
    const long long units = heads * ((nchunks + a.seg - 1) / a.seg);   // heads x segments
    const bool work = (long long)*first < units;   // the CTA has a unit at all

    if (!work) {
        // no unit left for this CTA: straight to the tear-down
    } else if (warp >= kCtl) {
        // ------------------------------------------------------------- control
        // Two warps, so that neither holds the other back: an MMA issue can
        // stall until the tensor cores take it.  Warp kCtl: lane 0 issues
        // the products.  Warp kLdr: lane 0 issues the copies, and the whole
        // warp computes the step sizes and the cumulative decay of each
        // chunk.  Both wait as whole warps.
        const bool leader = lane == 0;
        if (leader && warp == kLdr) {
            ptx::prefetch_tensormap(&tmX);
            ptx::prefetch_tensormap(&tmB);
            ptx::prefetch_tensormap(&tmC);
        }
        const uint32_t in_bytes = (two_regions ? 4 : 2) * 16384 + 16384;
        const uint32_t s0 = ptx::smem_u32(sm);
        const uint32_t sWh = s0 + Layout::kWh, sWl = s0 + Layout::kWl;
        const uint32_t sHh = s0 + Layout::kHh, sHl = s0 + Layout::kHl;
        constexpr uint32_t idS = idesc(128, 128, 0, 0), idY = idesc(128, 64, 0, 1),
                           idG = idesc(128, 64, 1, 1);
        // The walk, a chunk ahead of the copies: load_dt() takes the chunk
        // `cur` and moves it on (taking a ticket at a unit's end), and leaves
        // the chunk's head and step for the copies in slot k % 2.
        Walk cur;
        cur.unit((long long)*first, heads, a.seg, nchunks);
        int qb0 = 0, qh0 = 0, qt0 = 0, qb1 = 0, qh1 = 0, qt1 = 0;   // slots 0 and 1
        long long last = -1;   // index of the walk's last chunk, once known
        auto load = [&](long long k) {   // the k-th chunk into buffer k % 2
            const int b = (k & 1) ? qb1 : qb0, hh = (k & 1) ? qh1 : qh0;
            const int i = (int)(k & 1);
            unsigned char* in = sm + i * Layout::kInBytes;
            uint64_t* full = &bar[kInFull + i];
            const int t0 = (k & 1) ? qt1 : qt0;
            ptx::mbar_arrive_expect_tx(full, in_bytes);
            ptx::tma_load_3d(in + Layout::kC, &tmC, full, 0, t0, (int)b);
            ptx::tma_load_3d(in + Layout::kB, &tmB, full, 0, t0, (int)b);
            if (two_regions) {
                ptx::tma_load_3d(in + Layout::kC + 16384, &tmC, full, 64, t0, (int)b);
                ptx::tma_load_3d(in + Layout::kB + 16384, &tmB, full, 64, t0, (int)b);
            }
            ptx::tma_load_4d(in + Layout::kX, &tmX, full, 0, (int)hh, t0, (int)b);
        };
        // The descriptors of a product are formed once and stepped per K
        // slice: the start address sits in the low 14 bits (in 16-byte
        // units; shared memory is below 256 KB), so adding a slice's offset
        // in 16-byte units moves only that field.  Each MMA is then an add
        // and the instruction; this thread shares its SM sub-partition with
        // two epilogue warps, and the tensor cores wait for what it issues.
        // K-major operands (C, and B as S's operand): slice k at
        // (k / 4) * 16384 + (k % 4) * 32 bytes; MN-major ones: k * 2048.
        auto koff = [](int k) { return (uint64_t)((k >> 2) * 1024 + (k & 3) * 2); };
        auto issue_s = [&](long long c) {   // S = C B^T
            const uint32_t in = s0 + (uint32_t)((c & 1) * Layout::kInBytes);
            const uint64_t da = sdesc(in + Layout::kC, 16, 1024), db = sdesc(in + Layout::kB, 16, 1024);
#pragma unroll
            for (int k = 0; k < 8; ++k) mma(tmem + kColS, da + koff(k), db + koff(k), idS, k > 0);
            mma_commit(&bar[kMmaS]);
        };
        auto issue_yx = [&](long long c) {   // Yx = C H into buffer c % 2, H as hi then lo
            const uint32_t in = s0 + (uint32_t)((c & 1) * Layout::kInBytes);
            const uint32_t col = tmem + ((c & 1) ? kColYx1 : kColYx0);
            const uint64_t da = sdesc(in + Layout::kC, 16, 1024);
            const uint64_t dh = sdesc(sHh, 16384, 1024), dl = sdesc(sHl, 16384, 1024);
#pragma unroll
            for (int k = 0; k < 8; ++k) mma(col, da + koff(k), dh + (uint64_t)(k * 128), idY, k > 0);
#pragma unroll
            for (int k = 0; k < 8; ++k) mma(col, da + koff(k), dl + (uint64_t)(k * 128), idY, 1);
            mma_commit(&bar[kMmaYx]);
        };
        auto issue_g = [&](long long c) {   // G = B^T (w o X)
            const uint32_t in = s0 + (uint32_t)((c & 1) * Layout::kInBytes);
            const uint64_t db = sdesc(in + Layout::kB, 16384, 1024);
            const uint64_t dh = sdesc(sWh, 16384, 1024), dl = sdesc(sWl, 16384, 1024);
#pragma unroll
            for (int k = 0; k < 8; ++k)
                mma(tmem + kColG, db + (uint64_t)(k * 128), dh + (uint64_t)(k * 128), idG, k > 0);
#pragma unroll
            for (int k = 0; k < 8; ++k) mma(tmem + kColG, db + (uint64_t)(k * 128), dl + (uint64_t)(k * 128), idG, 1);
            mma_commit(&bar[kMmaG]);
        };
        auto issue_yi = [&](long long c) {   // Yi = (masked S) X
            const uint32_t in = s0 + (uint32_t)((c & 1) * Layout::kInBytes);
            const uint64_t dx = sdesc(in + Layout::kX, 16384, 1024);
#pragma unroll
            for (int k = 0; k < 8; ++k)
                mma_ta(tmem + kColYi, tmem + kColSh + 8 * k, dx + (uint64_t)(k * 128), idY, k > 0);
#pragma unroll
            for (int k = 0; k < 8; ++k) mma_ta(tmem + kColYi, tmem + kColSl + 8 * k, dx + (uint64_t)(k * 128), idY, 1);
            mma_commit(&bar[kMmaYi]);
        };
        auto wait = [&](int which, long long k) {   // k-th completion of a barrier, whole warp
            return __all_sync(0xffffffffu, bwait(&bar[which], (uint32_t)(k & 1), a.wait_ns));
        };
        // raw dt of the steps 4 lane .. 4 lane + 3 of a chunk (a chunk ahead),
        // with its head's A, dt_bias and D, kept as loaded: nothing here uses
        // the values, so the loads complete while this warp goes on (steps
        // past L read the last one, and the decay masks them)
        unsigned short raw[4];
        float rawA = 0.0f, rawbias = 0.0f, rawdsk = 0.0f;
        ChunkRec rec;   // of the chunk whose dt is held
        long long ndt = 0, nscan = 0;   // chunks whose dt was loaded; scanned
        auto load_dt = [&]() {   // chunk cur, the ndt-th
            const Walk ch = cur;
            const int b = ch.j / (int)a.H, hh = ch.j - b * (int)a.H;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const long long t = (long long)ch.c * Q + 4 * lane + j;
                raw[j] = reinterpret_cast<const unsigned short*>(a.dt)[((long long)b * a.L + (t < a.L ? t : a.L - 1)) * a.H + hh];
            }
            rawA = ld_early(a.A + hh);
            rawbias = a.dt_bias ? ld_early(a.dt_bias + hh) : 0.0f;
            rawdsk = a.Dskip ? ld_early(a.Dskip + hh) : 0.0f;
            rec.b = b;
            rec.h = hh;
            rec.c = ch.c;
            rec.nv = (int)(a.L - (long long)ch.c * Q < Q ? a.L - (long long)ch.c * Q : Q);
            rec.j = ch.j;
            rec.sg = ch.sg;
            rec.start = ch.c != ch.sg * a.seg ? kCont : ch.sg == 0 ? kZero : kHand;
            rec.end = ch.c != ch.hi - 1 ? kEndNone : ch.hi == nchunks ? kEndHead : kEndHand;
            if (ndt & 1) {
                qb1 = b;
                qh1 = hh;
                qt1 = ch.c * Q;
            } else {
                qb0 = b;
                qh0 = hh;
                qt0 = ch.c * Q;
            }
            // the next chunk: the unit's next, or the first of the next ticket's
            if (cur.c + 1 < cur.hi) {
                ++cur.c;
                rec.next = kCont;
            } else {
                unsigned long long t = 0;
                if (lane == 0) t = a.ticket ? atomicAdd(a.ticket, 1ull) : ~0ull;
                t = __shfl_sync(0xffffffffu, t, 0);
                if ((long long)t < units && t != ~0ull) {
                    cur.unit((long long)t, heads, a.seg, nchunks);
                    rec.next = cur.sg == 0 ? kZero : kHand;
                } else {
                    rec.next = kNone;
                    last = ndt;
                }
            }
            rec.nj = cur.j;
            rec.nsg = cur.sg;
            ++ndt;
        };
        // step sizes and cumulative decay of the chunk whose dt load_dt holds
        // into the shared copy (its previous readers, the masked scores of the
        // chunk before, are done), and its record into its slot (last read
        // by the outputs of the chunk two before, which precede those scores)
        auto scan = [&]() {   // the chunk whose dt load_dt holds
            const int nv = rec.nv;
            const float A = rawA, kb2 = rawbias * kLog2e;
            float d[4], cl[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float v2 = fmaf(__bfloat162float(__ushort_as_bfloat16(raw[j])), kLog2e, kb2);
                const float sp = (v2 > 28.853901f ? v2 : ptx::lg2(1.0f + ptx::ex2(v2))) * 0.6931471805599453f;
                d[j] = 4 * lane + j < nv ? sp : 0.0f;
                cl[j] = (j ? cl[j - 1] : 0.0f) + A * d[j];
            }
            float inc = cl[3];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float v = __shfl_up_sync(0xffffffffu, inc, o);
                if (lane >= o) inc += v;
            }
            const float ex = inc - cl[3];
            *reinterpret_cast<float4*>(cum + 4 * lane) =
                make_float4((cl[0] + ex) * kLog2e, (cl[1] + ex) * kLog2e, (cl[2] + ex) * kLog2e,
                            (cl[3] + ex) * kLog2e);
            *reinterpret_cast<float4*>(dts + 4 * lane) = make_float4(d[0], d[1], d[2], d[3]);
            if (leader) {   // read by the chunk's state update and outputs
                rec.dsk = rawdsk;
                recs[nscan & 1] = rec;
            }
            ++nscan;
            __syncwarp();
            if (leader) ptx::mbar_arrive(&bar[kCum]);
        };
        if (warp == kLdr) {
            // The first two chunks' copies and chunk 0's decay; then, per
            // chunk c, the copies of chunk c + 1 once the outputs of chunk
            // c - 1 are done with its buffer, and the decay of chunk c + 1
            // once the scores of chunk c have read the shared copy (the
            // order in which the epilogue's iteration for chunk c frees them).
            // whether the walk has a k-th chunk (known once the walk has
            // passed the chunk before)
            auto more = [&](long long k) { return last < 0 || k <= last; };
            load_dt();
            scan();
            if (more(1)) load_dt();
            if (leader) {
                load(0);
                if (more(1)) load(1);
            }
            for (long long c = 0; more(c + 1) && !failed; ++c) {
                if (c > 0) {
                    if (!wait(kInFree + (int)((c - 1) & 1), (c - 1) >> 1)) { failed = true; break; }
                    if (leader) load(c + 1);
                }
                if (!wait(kEpReady, c)) { failed = true; break; }
                scan();
                if (more(c + 2)) load_dt();
            }
            // Every copy issued here is waited for by the product warp
            // before the products that read it.
            if (failed && leader) atomicOr(&g_error_word, kErrTimeout);
            __syncwarp();
        } else {
            // chunk 0's S and C H (of the zero state)
            if (!wait(kInFull, 0)) failed = true;
            if (!failed) {
                fence_after_sync();
                if (leader) issue_s(0);
                if (!wait(kHReady, 0)) failed = true;
            }
            if (!failed) {
                fence_after_sync();
                if (leader) issue_yx(0);
            }
            // Each product goes as soon as what it reads is written and its
            // accumulator has been read, in the order the epilogue's phases
            // produce them within its iteration for chunk c (the state after
            // chunk c - 1, w o X of chunk c, the outputs of chunk c - 1, the
            // masked scores of chunk c): this thread issues in order, so a
            // wait on a later event would hold back an earlier product.
            long long c = 0;
            for (;; ++c) {
                if (c > 0) {
                    // The state entering chunk c is written, and every
                    // epilogue warp has read G of chunk c - 1.  C H of chunk
                    // c goes into buffer c % 2, last read by the outputs of
                    // chunk c - 2, which precede the scores of chunk c - 1
                    // (kEpReady, seen in the previous iteration); C of chunk
                    // c landed before its S went.
                    if (!wait(kHReady, c)) { failed = true; break; }
                    fence_after_sync();
                    if (leader) issue_yx(c);
                }
                // G(c): w o X of chunk c is written
                if (!wait(kWxReady, c)) { failed = true; break; }
                fence_after_sync();
                if (leader) issue_g(c);
                // Yi(c): the masked scores of chunk c are in TMEM; then S of
                // chunk c + 1 (S of chunk c has been read)
                if (!wait(kEpReady, c)) { failed = true; break; }
                fence_after_sync();
                if (leader) issue_yi(c);
                // the chunk's record (written before its scores) says
                // whether another chunk follows
                if (recs[c & 1].next == kNone) break;
                if (!wait(kInFull + (int)((c + 1) & 1), (c + 1) >> 1)) { failed = true; break; }
                fence_after_sync();
                if (leader) issue_s(c + 1);
            }
            // Leave no product in flight (bounded): the last chunk's Yi,
            // the last product issued, completes after all of them; a
            // parity wait names the last phase alone, and Yi of the chunk
            // before completed (the outputs of that chunk, which precede
            // the last chunk's scores, waited for it).
            if (!failed && !wait(kMmaYi, c)) failed = true;
            if (failed && leader) atomicOr(&g_error_word, kErrTimeout);
            __syncwarp();
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int quad = warp & 3, hf = warp >> 2;   // TMEM lane quadrant; column half
        const int row = 32 * quad + lane;            // step t, or state row n
        const uint32_t lane_addr = tmem + ((uint32_t)(32 * quad) << 16);
        float Hs[32];   // columns 32 hf .. 32 hf + 31 of row `row` of the state
#pragma unroll
        for (int j = 0; j < 32; ++j) Hs[j] = 0.0f;
        // The state entering a chunk that starts a unit: zero at its head's
        // start, else the one left by the head's segment before (done by
        // whichever CTA took it, once all eight of its epilogue warps have
        // released their parts).
        auto enter = [&](int kind, int j, int sg) -> bool {
            if (kind == kCont || kind == kNone) return true;
            if (kind == kZero) {
#pragma unroll
                for (int i = 0; i < 32; ++i) Hs[i] = 0.0f;
                return true;
            }
            if (!__all_sync(0xffffffffu,
                            wait_count(a.done + j, (unsigned)(kEpWarps * sg), a.wait_ns)))
                return false;
            const float4* src = reinterpret_cast<const float4*>(
                a.carry + ((long long)j * NP + row) * P + 32 * hf);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float4 v = src[j];
                Hs[4 * j] = v.x;
                Hs[4 * j + 1] = v.y;
                Hs[4 * j + 2] = v.z;
                Hs[4 * j + 3] = v.w;
            }
            return true;
        };
        // The state after a chunk that ends a unit leaves: as h_last at its
        // head's end, else for the head's next segment.
        auto leave = [&](int kind, int j) {
            if (kind == kEndNone) return;
            if (kind == kEndHead) {
                if (a.h_last && row < a.N) {
                    float* base = a.h_last + (long long)j * P * a.N + row;
#pragma unroll
                    for (int j = 0; j < 32; ++j) base[(long long)(32 * hf + j) * a.N] = Hs[j];
                }
                return;
            }
            float4* dst = reinterpret_cast<float4*>(a.carry + ((long long)j * NP + row) * P + 32 * hf);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                dst[i] = make_float4(Hs[4 * i], Hs[4 * i + 1], Hs[4 * i + 2], Hs[4 * i + 3]);
            __threadfence();
            __syncwarp();
            if (lane == 0) red_release_add(a.done + j, 1u);
        };
        // The state after the c-th chunk: H <- exp(cum_end) H + G (row n =
        // row, this warp's 32 columns); it leaves if the chunk ends a unit,
        // and the next chunk's entering state, if that starts one, replaces
        // it; then its hi + lo copy for the next chunk's C H (the previous
        // copy was read by this chunk's Yx, which completed).
        auto state_update = [&](long long c, float dend) -> bool {
            if (!wwait(&bar[kMmaG], (uint32_t)(c & 1), a.wait_ns) ||
                !wwait(&bar[kMmaYx], (uint32_t)(c & 1), a.wait_ns))
                return false;
            fence_after_sync();
            float g[32];
            tmem_ld32(lane_addr + kColG + 32 * hf, g);
#pragma unroll
            for (int j = 0; j < 32; ++j) Hs[j] = fmaf(dend, Hs[j], g[j]);
            const ChunkRec& r = recs[c & 1];
            leave(r.end, r.j);
            if (!enter(r.next, r.nj, r.nsg)) return false;
            store_split32(sm + Layout::kHh, sm + Layout::kHl, row, 4 * hf, Hs);
            ptx::fence_proxy_async_shared();
            fence_before_sync();
            warp_arrive(&bar[kHReady], lane);
            return true;
        };
        // The outputs of the c-th chunk, step t = row, this warp's 32 columns:
        // Yi + exp(cum_t) Yx + Dskip x; then the chunk's buffer is free.
        auto outputs = [&](long long c, float ecum) -> bool {
            if (!wwait(&bar[kMmaYi], (uint32_t)(c & 1), a.wait_ns)) return false;
            fence_after_sync();
            const ChunkRec& r = recs[c & 1];
            const long long b = r.b, hh = r.h, cc = r.c;
            const float dsk = r.dsk;
            const unsigned char* X = sm + (c & 1) * Layout::kInBytes + Layout::kX;
            const int nv = r.nv;
            float yi[32], yx[32];
            tmem_ld32_nowait(lane_addr + kColYi + 32 * hf, yi);
            tmem_ld32_nowait(lane_addr + ((c & 1) ? kColYx1 : kColYx0) + 32 * hf, yx);
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            bf16* yrow = a.y + ((b * a.L + cc * Q + row) * a.H + hh) * P + 32 * hf;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                const uint4 xv = *reinterpret_cast<const uint4*>(X + sw128(row, 4 * hf + cc));
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
                if (row < nv) *reinterpret_cast<uint4*>(yrow + 8 * cc) = o;
            }
            // X (read above and by Yi) and B (read by G) are free for chunk c + 2
            fence_before_sync();
            warp_arrive(&bar[kInFree + (int)(c & 1)], lane);
            return true;
        };
        // the state entering the first chunk, as its record (which comes
        // with its decays) says
        if (!wwait(&bar[kCum], 0u, a.wait_ns) || !enter(recs[0].start, recs[0].j, recs[0].sg))
            failed = true;
        store_split32(sm + Layout::kHh, sm + Layout::kHl, row, 4 * hf, Hs);
        ptx::fence_proxy_async_shared();
        fence_before_sync();
        warp_arrive(&bar[kHReady], lane);
        float ecum_prev = 0.0f, dend_prev = 0.0f;
        for (long long c = 0; !failed; ++c) {
            const uint32_t ph = (uint32_t)(c & 1);
            const unsigned char* X = sm + (c & 1) * Layout::kInBytes + Layout::kX;
            // the previous chunk's state (its G ran first) lets chunk c's C H go
            if (c > 0 && !state_update(c - 1, dend_prev)) { failed = true; break; }
            // the walk ended with the previous chunk: its outputs, and done
            if (c > 0 && recs[(c - 1) & 1].next == kNone) {
                if (!outputs(c - 1, ecum_prev)) failed = true;
                break;
            }
            // this row's cumulative decay (log2 units) and step size, and the chunk's total
            if (!wwait(&bar[kCum], ph, a.wait_ns)) { failed = true; break; }
            const float ct = cum[row], cend2 = cum[Q - 1];
            const float ecum = ptx::ex2(ct);                 // exp(cum_t)
            const float dend = ptx::ex2(cend2);              // exp(cum_end)
            if (!wwait(&bar[kInFull + (int)(c & 1)], (uint32_t)((c >> 1) & 1), a.wait_ns)) {
                failed = true;
                break;
            }
            // w o X, split hi + lo (the previous chunk's G, which read them,
            // completed: state_update).  The causal mask gives the warps of
            // lane quadrants 2 and 3 the most score columns, so the warps of
            // quadrants 0 and 1 form all of w o X: warp e < 4 (quad 0 or 1,
            // column half hf) takes rows s = 32 (e & 1) + lane and s + 64 of
            // its column half, with the w_s of those rows from the shared copy.
            if (quad < 2) {
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    const int s_ = 32 * quad + 64 * rr + lane;
                    const float ws = ptx::ex2(cend2 - cum[s_]) * dts[s_];
#pragma unroll
                    for (int cc = 4 * hf; cc < 4 * hf + 4; ++cc) {
                        const uint4 xv = *reinterpret_cast<const uint4*>(X + sw128(s_, cc));
                        const __nv_bfloat162* x2 = reinterpret_cast<const __nv_bfloat162*>(&xv);
                        uint4 h, l;
                        uint32_t* hp = &h.x;
                        uint32_t* lp = &l.x;
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float2 f = __bfloat1622float2(x2[q]);
                            split2(ws * f.x, ws * f.y, hp[q], lp[q]);
                        }
                        *reinterpret_cast<uint4*>(sm + Layout::kWh + sw128(s_, cc)) = h;
                        *reinterpret_cast<uint4*>(sm + Layout::kWl + sw128(s_, cc)) = l;
                    }
                }
                ptx::fence_proxy_async_shared();   // w o X, for the tensor cores (G)
                warp_arrive(&bar[kWxReady], lane);
            }
            // the previous chunk's outputs (its Yi ran after G)
            if (c > 0 && !outputs(c - 1, ecum_prev)) { failed = true; break; }
            // masked scores of row t = row, pieces hf and hf + 2 (32 columns
            // each): S[t,s] exp(cum_t - cum_s) dt_s for s <= t, into TMEM as
            // packed bf16 hi and lo (the previous chunk's Yi, which read them,
            // completed: outputs)
            if (!wwait(&bar[kMmaS], ph, a.wait_ns)) {
                failed = true;
                break;
            }
            fence_after_sync();
            float sv[2][32];
            tmem_ld32_nowait(lane_addr + kColS + 32 * hf, sv[0]);
            if (hf + 2 <= quad) tmem_ld32_nowait(lane_addr + kColS + 32 * (hf + 2), sv[1]);
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int piece = hf + 2 * k;
                uint32_t hi[16], lo[16];
                if (piece <= quad) {   // some s of the piece are <= t (warp-uniform)
                    float (&v)[32] = sv[k];
                    const float4* cum4 = reinterpret_cast<const float4*>(cum + 32 * piece);
                    const float4* dt4 = reinterpret_cast<const float4*>(dts + 32 * piece);
#pragma unroll
                    for (int j4 = 0; j4 < 8; ++j4) {
                        const float4 cq = cum4[j4], dq = dt4[j4];
                        const float cs[4] = {cq.x, cq.y, cq.z, cq.w}, ds[4] = {dq.x, dq.y, dq.z, dq.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int j = 4 * j4 + e, s_ = 32 * piece + j;
                            v[j] = s_ <= row ? v[j] * ptx::ex2(ct - cs[e]) * ds[e] : 0.0f;
                        }
                    }
#pragma unroll
                    for (int j = 0; j < 16; ++j) split2(v[2 * j], v[2 * j + 1], hi[j], lo[j]);
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) hi[j] = lo[j] = 0u;
                }
                tmem_st16(lane_addr + kColSh + 16 * piece, hi);
                tmem_st16(lane_addr + kColSl + 16 * piece, lo);
            }
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            ptx::fence_proxy_async_shared();   // w o X, for the tensor cores
            fence_before_sync();
            warp_arrive(&bar[kEpReady], lane);
            ecum_prev = ecum;
            dend_prev = dend;
        }
        if (failed && lane == 0) atomicOr(&g_error_word, kErrTimeout);
    }
    // ---- tear-down: every TMEM access and MMA is done before the columns go
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

#include "ssd_plan.h"
#include "tma_host.cuh"

namespace ssm {
namespace ssdtc {

// bf16, P == 64, N == 64 or 128, x, B, C, y 16-byte aligned, batch*H > 0,
// L > 0 (checked by the caller).
//
// Which walk, and the ticket walk's segments: plan() (ssd_plan.h).  The
// ticket walk's ticket, per-head counters and the states handed between
// segments live in a stream-ordered workspace of about heads x 32 KB, freed
// on the stream after the launch; a failed allocation returns
// cudaErrorMemoryAllocation.
// `want_seg` > 0 or `want_ctas` > 0 (development and tests) ask for the
// ticket walk with segments of that many chunks and at most that many CTAs.
// The one-head walk's arguments, from the ticket walk's.
inline Args one_head(const ArgsDyn& d) {
    Args a;
    a.x = d.x;
    a.dt = d.dt;
    a.dt_bias = d.dt_bias;
    a.A = d.A;
    a.Dskip = d.Dskip;
    a.y = d.y;
    a.h_last = d.h_last;
    a.batch = d.batch;
    a.L = d.L;
    a.H = d.H;
    a.N = d.N;
    a.wait_ns = d.wait_ns;
    return a;
}

inline cudaError_t launch_ssd_tc(const bf16* x, const bf16* dt, const float* dt_bias,
                                 const float* A, const bf16* Bm, const bf16* Cm,
                                 const float* Dskip, bf16* y, float* h_last, long long batch,
                                 long long L, long long H, int N, unsigned long long wait_ns,
                                 cudaStream_t s, long long want_seg = 0,
                                 long long want_ctas = 0) {
    CUtensorMap mX, mB, mC;
    const cuuint64_t es = 2;
    const cuuint64_t dX[4] = {(cuuint64_t)P, (cuuint64_t)H, (cuuint64_t)L, (cuuint64_t)batch};
    const cuuint64_t sX[3] = {P * es, (cuuint64_t)H * P * es, (cuuint64_t)L * H * P * es};
    const cuuint32_t bX[4] = {64u, 1u, (cuuint32_t)Q, 1u};
    const cuuint64_t dBC[3] = {(cuuint64_t)N, (cuuint64_t)L, (cuuint64_t)batch};
    const cuuint64_t sBC[2] = {(cuuint64_t)N * es, (cuuint64_t)L * N * es};
    const cuuint32_t bBC[3] = {64u, (cuuint32_t)Q, 1u};
    const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    if (!tma::cached_map(&mX, bf, 4, x, dX, sX, bX, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !tma::cached_map(&mB, bf, 3, Bm, dBC, sBC, bBC, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !tma::cached_map(&mC, bf, 3, Cm, dBC, sBC, bBC, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const long long heads = batch * H, nch = (L + Q - 1) / Q;
    if (nch >= (1ll << 30)) return cudaErrorInvalidValue;   // chunk indices are int
    const Plan pl = plan(heads, nch, sms, want_seg, want_ctas);
    const bool dyn = pl.dyn;
    const long long U = pl.seg, nseg = pl.nseg, units = pl.units, G = pl.ctas;
    ArgsDyn a;
    a.ticket = nullptr;
    a.carry = nullptr;
    a.done = nullptr;
    a.seg = (int)U;
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
    const int smem = dyn ? LayoutDyn::kSmemBytes : Layout::kSmemBytes;
    e = dyn ? cudaFuncSetAttribute(ssd_tc_dyn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)
            : cudaFuncSetAttribute(ssd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    unsigned char* ws = nullptr;
    if (dyn && (G < units || nseg > 1)) {   // tickets (more units than CTAs); hand-offs (heads cut)
        const size_t head_bytes = (8 + (size_t)heads * 4 + 255) & ~(size_t)255;
        const size_t bytes = head_bytes + (nseg > 1 ? (size_t)heads * NP * P * sizeof(float) : 0);
        if (fault::malloc_async(reinterpret_cast<void**>(&ws), bytes, s) != cudaSuccess) {
            cudaGetLastError();
            return cudaErrorMemoryAllocation;
        }
        if (G < units) a.ticket = reinterpret_cast<unsigned long long*>(ws);
        a.done = reinterpret_cast<unsigned*>(ws + 8);
        if (nseg > 1) a.carry = reinterpret_cast<float*>(ws + head_bytes);
        e = cudaMemsetAsync(ws, 0, head_bytes, s);
    }
    if (e == cudaSuccess) {
        if (fault::launch_refused()) {
            e = cudaErrorLaunchFailure;
        } else {
            if (dyn)
                ssd_tc_dyn_kernel<<<(unsigned)G, THREADS, smem, s>>>(mX, mB, mC, a);
            else
                ssd_tc_kernel<<<(unsigned)G, THREADS, smem, s>>>(mX, mB, mC, one_head(a));
            e = cudaGetLastError();
        }
    }
    if (ws) {
        const cudaError_t f = cudaFreeAsync(ws, s);
        if (e == cudaSuccess) e = f;
    }
    return e;
}

}  // namespace ssdtc
}  // namespace ssm
