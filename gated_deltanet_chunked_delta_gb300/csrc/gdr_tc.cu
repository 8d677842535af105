// gdr_tc.cu -- tcgen05 tensor-core path of the GDN chunked prefill (bf16
// operands, fp32 accumulation, K = V = 128, 64-token chunks).
//
// The inter-chunk state scan (FlashQLA pages, page 1 "efficiency problem":
// the scan kernel can only launch batch x heads blocks; page 1 "two fused
// kernels and automatic CP": a chunk-parallel kernel, then the scan, with the
// context-parallel step between them) runs one CTA per (segment, v-head) and
// keeps the fp32 state in tensor memory, transposed: TMEM lane v holds row v
// of S^T (column v of S), 128 columns of k.  Per chunk:
//
//   MMA1  D1 = S^T [W ; Q]^T          (M=128 lanes v, N=64 or 128, K=128)
//         -> (W S)^T and (Q S)^T
//   epi   Ut^T = U^T - (W S)^T   (bf16 into shared memory, the next A operand)
//   MMA2  D2 = Ut^T P^T               (M=128, N=64, K=64)  -> (P Ut)^T
//   MMA3  S^T += Ut^T Kt              (M=128, N=128, K=64), after the epilogue
//         scaled S^T by e^{gamma_n} in place
//   epi   O = scale e^{gamma} o (Q S) + P Ut   (row r of O from column r of D)
//
// Roles: warps 0-3 are the epilogue (thread t <-> TMEM lane t), warp 4 issues
// TMA loads of the chunk tiles into a two-stage ring, warp 5 allocates tensor
// memory and issues the MMAs from one thread.  Every wait is a bounded poll;
// a wait that runs out sets the device status word, raises a shared abort
// flag that every role polls, and the CTA drains and frees its tensor memory.
//
// Modes: kFwd emits o (and h, final_state); kStates only stores the state
// before every chunk (the backward's recompute); kSummary runs the
// context-parallel segment summary, carrying two states: S from 0 with
// pseudo-values U, and M from I with zero pseudo-values (the columns of
// X = [S | M] evolve independently), and writes H = S_end and M = M_end.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "gdr_internal.h"

namespace gdr {
namespace {

__device__ unsigned g_tc_status;

constexpr int kFwd = 0, kStates = 1, kSummary = 2;

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t su32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *b, uint32_t n) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(n) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ uint32_t mbar_try(uint64_t *b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(su32(b)), "r"(parity)
        : "memory");
    return ok;
}

// Bounded wait.  Returns false when the CTA is aborting (someone else ran out
// of polls) or when this wait itself ran out (then it raises the abort).
__device__ __forceinline__ bool bwait(uint64_t *b, uint32_t parity, long long cap, volatile int *abort) {
    for (long long i = 0;; ++i) {
        if (mbar_try(b, parity)) return true;
        if (*abort) return false;
        if (i >= cap) {
            *abort = 1;
            atomicOr(&g_tc_status, 1u);
            return false;
        }
    }
}
// Bounded wait that ignores the abort flag (used while draining).
__device__ __forceinline__ void drain_wait(uint64_t *b, uint32_t parity, long long cap) {
    for (long long i = 0; i < cap; ++i)
        if (mbar_try(b, parity)) return;
}

__device__ __forceinline__ void tma2d(void *dst, const CUtensorMap *m, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            su32(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(su32(bar))
        : "memory");
}
__device__ __forceinline__ void tma3d(void *dst, const CUtensorMap *m, int x, int y, int z, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(su32(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(z), "r"(su32(bar))
        : "memory");
}
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     su32(dst)),
                 "l"(src), "r"(bytes), "r"(su32(bar))
                 : "memory");
}

__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (tile bases are 1024-byte aligned).
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;             // leading byte offset (unused for this layout)
    d |= (uint64_t)(1024 >> 4) << 32;   // stride byte offset
    d |= (uint64_t)1 << 46;             // descriptor version
    d |= (uint64_t)2 << 61;             // 128-byte swizzle
    return d;
}
// Instruction descriptor: bf16 x bf16 -> fp32, both operands K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(bar))
                 : "memory");
}

#define R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), "=r"(r[i + 4]), "=r"(r[i + 5]), \
              "=r"(r[i + 6]), "=r"(r[i + 7])
#define W8(i) "+r"(r[i]), "+r"(r[i + 1]), "+r"(r[i + 2]), "+r"(r[i + 3]), "+r"(r[i + 4]), "+r"(r[i + 5]), \
              "+r"(r[i + 6]), "+r"(r[i + 7])
#define S8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), "r"(r[i + 4]), "r"(r[i + 5]), \
              "r"(r[i + 6]), "r"(r[i + 7])

// 32 consecutive TMEM columns of this warp's 32 lanes; waits for the data.
__device__ __forceinline__ void tmem_ld32(uint32_t ta, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : R8(0), R8(8), R8(16), R8(24)
        : "r"(ta));
    asm volatile("tcgen05.wait::ld.sync.aligned;" : W8(0), W8(8), W8(16), W8(24)::"memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t ta, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(ta),
        S8(0), S8(8), S8(16), S8(24)
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Row `row` of a K-major, 128-byte-swizzled bf16 tile of `rows` rows: writes
// 32 consecutive elements starting at column `col0` (a multiple of 32).
__device__ __forceinline__ void st_row32(char *tile, int rows, int row, int col0, const float *x) {
    const int atom = col0 >> 6;
    char *base = tile + atom * rows * 128 + row * 128;
    const int c0 = (col0 & 63) >> 3;  // first 16-byte chunk
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint4 v;
        v.x = pack_bf16(x[8 * j + 0], x[8 * j + 1]);
        v.y = pack_bf16(x[8 * j + 2], x[8 * j + 3]);
        v.z = pack_bf16(x[8 * j + 4], x[8 * j + 5]);
        v.w = pack_bf16(x[8 * j + 6], x[8 * j + 7]);
        *reinterpret_cast<uint4 *>(base + (((c0 + j) ^ (row & 7)) << 4)) = v;
    }
}

__device__ __forceinline__ float ldbf(const __nv_bfloat16 *p) { return __bfloat162float(*p); }

// ---------------------------------------------------------------------------
// the scan kernel
// ---------------------------------------------------------------------------
struct TcMaps {
    CUtensorMap W, U, P, KT, Q;
};

// One pipeline stage (all offsets 1024-byte aligned):
//   B1  [2 atoms][rows][128 B] swizzled: W rows 0-63 (+ Q rows 64-127 in kFwd)
//   U   [64][128] bf16 plain row-major
//   P   [64 rows][128 B] swizzled (kFwd only)
//   KT  [128 rows][128 B] swizzled
//   gamma, 64 fp32
template <int MODE>
struct Stage {
    static constexpr int kAtom = MODE == kFwd ? 16384 : 8192;  // bytes per 64-column atom of B1
    static constexpr int kB1 = 0;
    static constexpr int kU = 2 * kAtom;
    static constexpr int kP = kU + 16384;
    static constexpr int kKT = kP + (MODE == kFwd ? 8192 : 0);
    static constexpr int kGam = kKT + 16384;
    static constexpr int kBytes = kGam + 1024;
    static constexpr uint32_t kTx = 2 * 8192 * (MODE == kFwd ? 2 : 1) + 16384 + (MODE == kFwd ? 8192 : 0) + 16384 + 256;
};
constexpr int kSB = 32768;       // S^T in bf16: [2 atoms][128][128 B]
constexpr int kUT = 16384;       // Ut^T in bf16: [128][128 B]

template <int MODE>
__host__ __device__ constexpr int scan_smem() {
    return 1024 /* alignment slack */ + 2 * Stage<MODE>::kBytes + (MODE == kSummary ? 2 : 1) * (kSB + kUT) + 256;
}

template <int MODE, typename TO>
__global__ void __launch_bounds__(192, 1) k_scan_tc(Params p, const __grid_constant__ TcMaps maps) {
    extern __shared__ __align__(1024) char smraw[];
    char *sm = reinterpret_cast<char *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
    constexpr int NX = MODE == kSummary ? 2 : 1;  // number of carried states
    using SL = Stage<MODE>;
    static_assert(scan_smem<MODE>() <= 227 * 1024, "shared memory budget");
    char *stage0 = sm;
    char *SB = sm + 2 * SL::kBytes;               // NX x kSB
    char *UT = SB + NX * kSB;                     // NX x kUT
    uint64_t *bars = reinterpret_cast<uint64_t *>(UT + NX * kUT);
    uint64_t *full = bars;        // [2]
    uint64_t *empty = bars + 2;   // [2]
    uint64_t *bar_sb = bars + 4;
    uint64_t *bar_m1 = bars + 5;
    uint64_t *bar_ut = bars + 6;
    uint64_t *bar_m2 = bars + 7;
    uint64_t *bar_drain = bars + 8;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 9);
    volatile int *abort = reinterpret_cast<volatile int *>(bars + 10);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int sidx = blockIdx.x, h = blockIdx.y;
    const SegInfo sg = p.seg[sidx];
    const SeqInfo sq = p.seq[sg.seq];
    const int hq = h / (p.Hv / p.Hq);
    const int nch = sg.nch;
    const long long cap = p.timeout_spins;

    if (tid == 0) {
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        mbar_init(&empty[0], 129);
        mbar_init(&empty[1], 129);
        mbar_init(bar_sb, 128);
        mbar_init(bar_m1, 1);
        mbar_init(bar_ut, 128);
        mbar_init(bar_m2, 1);
        mbar_init(bar_drain, 1);
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 5) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_slot)),
                     "r"(512));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // TMEM columns
    const uint32_t tS = tmem;                                   // S^T (and M^T at +128 in summary mode)
    const uint32_t tD1 = tmem + (MODE == kSummary ? 256 : 128); // 128 (fwd) or 64 per state
    const uint32_t tD2 = tmem + 256;                            // fwd: (P Ut)^T, 64 columns

    if (warp == 4) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            int issued = 0;
            for (int cc = 0; cc < nch; ++cc) {
                const int s = cc & 1;
                if (cc >= 2 && !bwait(&empty[s], ((cc >> 1) & 1) ^ 1, cap, abort)) break;
                const int c = sg.chunk0 + cc;
                const ChunkInfo ci = p.chunk[c];
                const int row = (c * p.Hv + h) * 64;
                char *st = stage0 + s * SL::kBytes;
                mbar_expect_tx(&full[s], SL::kTx);
                tma2d(st + SL::kB1, &maps.W, 0, row, &full[s]);
                tma2d(st + SL::kB1 + SL::kAtom, &maps.W, 64, row, &full[s]);
                if (MODE == kFwd) {
                    tma3d(st + SL::kB1 + 8192, &maps.Q, 0, hq, ci.tok0, &full[s]);
                    tma3d(st + SL::kB1 + SL::kAtom + 8192, &maps.Q, 64, hq, ci.tok0, &full[s]);
                    tma2d(st + SL::kP, &maps.P, 0, row, &full[s]);
                }
                tma2d(st + SL::kU, &maps.U, 0, row, &full[s]);
                tma2d(st + SL::kKT, &maps.KT, 0, (c * p.Hv + h) * 128, &full[s]);
                bulk_g2s(st + SL::kGam, p.gam + (size_t)(c * p.Hv + h) * 64, 256, &full[s]);
                issued = cc + 1;
            }
            // never leave with copies in flight: wait for the last stages that were issued
            for (int cc = issued - 2 < 0 ? 0 : issued - 2; cc < issued; ++cc)
                drain_wait(&full[cc & 1], (cc >> 1) & 1, cap);
        }
    } else if (warp == 5) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            const uint32_t id1 = idesc_bf16(128, MODE == kFwd ? 128 : 64);
            const uint32_t id2 = idesc_bf16(128, 64);
            const uint32_t id3 = idesc_bf16(128, 128);
            for (int cc = 0; cc < nch; ++cc) {
                const int s = cc & 1;
                char *st = stage0 + s * SL::kBytes;
                if (!bwait(&full[s], (cc >> 1) & 1, cap, abort)) break;
                if (!bwait(bar_sb, cc & 1, cap, abort)) break;
                tc_fence_after();
                for (int x = 0; x < NX; ++x) {
                    const uint32_t a0 = su32(SB + x * kSB), b0 = su32(st + SL::kB1);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t ko = (kk & 3) * 32;
                        mma(tD1 + x * 64, sdesc(a0 + (kk >> 2) * 16384 + ko), sdesc(b0 + (kk >> 2) * SL::kAtom + ko),
                            id1, kk > 0);
                    }
                }
                mma_commit(bar_m1);
                if (!bwait(bar_ut, cc & 1, cap, abort)) break;
                tc_fence_after();
                if (MODE == kFwd) {
                    const uint32_t a0 = su32(UT), b0 = su32(st + SL::kP);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) mma(tD2, sdesc(a0 + kk * 32), sdesc(b0 + kk * 32), id2, kk > 0);
                }
                for (int x = 0; x < NX; ++x) {
                    const uint32_t a0 = su32(UT + x * kUT), b0 = su32(st + SL::kKT);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) mma(tS + x * 128, sdesc(a0 + kk * 32), sdesc(b0 + kk * 32), id3, 1);
                }
                mma_commit(bar_m2);
                mma_commit(&empty[s]);
            }
            // every MMA issued above has completed before the CTA tears down
            mma_commit(bar_drain);
            drain_wait(bar_drain, 0, cap);
        }
    } else {
        // ---------------- epilogue: warps 0-3, thread t <-> TMEM lane t ----------------
        const int t = tid;
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        uint32_t r[32];
        // initial state(s)
        for (int x = 0; x < NX; ++x) {
            for (int j = 0; j < 4; ++j) {
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int k = 32 * j + i;
                    float v0;
                    if (MODE == kSummary)
                        v0 = (x == 1 && k == t) ? 1.f : 0.f;
                    else if (sg.idx == 0)
                        v0 = p.h0 ? p.h0[(((size_t)sg.seq * p.Hv + h) * 128 + k) * 128 + t] : 0.f;
                    else
                        v0 = p.Sstart[(((size_t)sidx * p.Hv + h) * 128 + k) * 128 + t];
                    r[i] = __float_as_uint(v0);
                }
                tmem_st32(tS + x * 128 + 32 * j + lane_off, r);
            }
        }
        tmem_wait_st();
        float *hdst = MODE == kFwd ? p.h_out : (MODE == kStates ? p.hbuf : nullptr);
        for (int cc = 0; cc < nch; ++cc) {
            const int s = cc & 1;
            char *st = stage0 + s * SL::kBytes;
            const float *gam = reinterpret_cast<const float *>(st + SL::kGam);
            const int c = sg.chunk0 + cc;
            if (cc > 0 && !bwait(bar_m2, (cc - 1) & 1, cap, abort)) break;
            tc_fence_after();
            if (!bwait(&full[s], (cc >> 1) & 1, cap, abort)) break;
            const float dec = __expf(gam[63]);
            // (a) S^T row t -> bf16 A operand; S^T *= e^{gamma_n} in place; h = S
            for (int x = 0; x < NX; ++x) {
                for (int j = 0; j < 4; ++j) {
                    tmem_ld32(tS + x * 128 + 32 * j + lane_off, r);
                    float f[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(r[i]);
                    st_row32(SB + x * kSB, 128, t, 32 * j, f);
                    if (hdst)
#pragma unroll 8
                        for (int i = 0; i < 32; ++i)
                            hdst[(((size_t)c * p.Hv + h) * 128 + 32 * j + i) * 128 + t] = f[i];
#pragma unroll
                    for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(f[i] * dec);
                    tmem_st32(tS + x * 128 + 32 * j + lane_off, r);
                }
            }
            tmem_wait_st();
            fence_async_smem();
            tc_fence_before();
            mbar_arrive(bar_sb);
            // (c) Ut^T = U^T - (W S)^T
            if (!bwait(bar_m1, cc & 1, cap, abort)) break;
            tc_fence_after();
            const __nv_bfloat16 *Us = reinterpret_cast<const __nv_bfloat16 *>(st + SL::kU);
            for (int x = 0; x < NX; ++x) {
                for (int j = 0; j < 2; ++j) {
                    tmem_ld32(tD1 + x * 64 + 32 * j + lane_off, r);
                    float f[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float u = x == 0 ? ldbf(Us + (32 * j + i) * 128 + t) : 0.f;
                        f[i] = u - __uint_as_float(r[i]);
                    }
                    st_row32(UT + x * kUT, 128, t, 32 * j, f);
                }
            }
            fence_async_smem();
            tc_fence_before();
            mbar_arrive(bar_ut);
            // (e) output
            if (MODE == kFwd) {
                if (!bwait(bar_m2, cc & 1, cap, abort)) break;
                tc_fence_after();
                const ChunkInfo ci = p.chunk[c];
                TO *o = reinterpret_cast<TO *>(p.o);
                for (int j = 0; j < 2; ++j) {
                    uint32_t r2[32];
                    tmem_ld32(tD1 + 64 + 32 * j + lane_off, r);
                    tmem_ld32(tD2 + 32 * j + lane_off, r2);
#pragma unroll 8
                    for (int i = 0; i < 32; ++i) {
                        const int rr = 32 * j + i;
                        const float val = p.scale * __expf(gam[rr]) * __uint_as_float(r[i]) + __uint_as_float(r2[i]);
                        if (rr < ci.len) {
                            const size_t off = ((size_t)(ci.tok0 + rr) * p.Hv + h) * 128 + t;
                            if constexpr (sizeof(TO) == 4)
                                o[off] = val;
                            else
                                o[off] = __float2bfloat16_rn(val);
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&empty[s]);
        }
        // final state(s)
        if (!*abort) {
            if (nch > 0 && MODE != kFwd) bwait(bar_m2, (nch - 1) & 1, cap, abort);
            tc_fence_after();
        }
        if (!*abort) {
            const bool last = sg.idx == sq.nseg - 1;
            for (int x = 0; x < NX; ++x) {
                float *dst = nullptr;
                size_t base = 0;
                if (MODE == kSummary) {
                    dst = x == 0 ? p.Hseg : p.Mseg;
                    base = ((size_t)sidx * p.Hv + h) * 128 * 128;
                } else if (last && p.final_state) {
                    dst = p.final_state;
                    base = ((size_t)sg.seq * p.Hv + h) * 128 * 128;
                }
                if (!dst) continue;
                for (int j = 0; j < 4; ++j) {
                    tmem_ld32(tS + x * 128 + 32 * j + lane_off, r);
#pragma unroll 8
                    for (int i = 0; i < 32; ++i) dst[base + (size_t)(32 * j + i) * 128 + t] = __uint_as_float(r[i]);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512));
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                              const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encoder() {
    static EncodeFn fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeFn>(ptr);
    }
    return fn;
}

bool make_map(CUtensorMap *m, const void *base, int rank, const cuuint64_t *dims, const cuuint64_t *strides_bytes,
              const cuuint32_t *box, bool swizzle) {
    EncodeFn fn = encoder();
    if (!fn) return false;
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void *>(base), dims, strides_bytes, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool build_maps(const Params &p, TcMaps *m) {
    const cuuint64_t rows = (cuuint64_t)p.NT * p.Hv * 64;
    {
        cuuint64_t d[2] = {128, rows}, s[1] = {256};
        cuuint32_t b[2] = {64, 64};
        if (!make_map(&m->W, p.Wb, 2, d, s, b, true)) return false;
    }
    {
        cuuint64_t d[2] = {128, rows}, s[1] = {256};
        cuuint32_t b[2] = {128, 64};
        if (!make_map(&m->U, p.Ub, 2, d, s, b, false)) return false;
    }
    {
        cuuint64_t d[2] = {64, rows}, s[1] = {128};
        cuuint32_t b[2] = {64, 64};
        if (!make_map(&m->P, p.Pb, 2, d, s, b, true)) return false;
    }
    {
        cuuint64_t d[2] = {64, (cuuint64_t)p.NT * p.Hv * 128}, s[1] = {128};
        cuuint32_t b[2] = {64, 128};
        if (!make_map(&m->KT, p.KTb, 2, d, s, b, true)) return false;
    }
    {
        cuuint64_t d[3] = {128, (cuuint64_t)p.Hq, (cuuint64_t)p.Ttot};
        cuuint64_t s[2] = {256, (cuuint64_t)p.Hq * 256};
        cuuint32_t b[3] = {64, 1, 64};
        if (!make_map(&m->Q, p.q, 3, d, s, b, true)) return false;
    }
    return true;
}

template <int MODE, typename TO>
int launch_scan(const char *name, const Params &p, const TcMaps &maps, cudaStream_t st) {
    if (p.NSEG == 0) return 0;
    auto kern = k_scan_tc<MODE, TO>;
    const int smem = scan_smem<MODE>();
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return 1;
    tm_begin(p.tm, name, st);
    kern<<<dim3(p.NSEG, p.Hv), 192, smem, st>>>(p, maps);
    tm_end(p.tm, st);
    return cudaGetLastError() != cudaSuccess;
}

}  // namespace

int tc_supported(int K, int V) { return K == 128 && V == 128; }

int tc_fwd(const Params &p, int o_f32, int use_cp, cudaStream_t st) {
    if (simt_wy_tc(p, 0, st)) return 1;
    TcMaps maps;
    if (!build_maps(p, &maps)) return 1;
    if (use_cp) {
        if (launch_scan<kSummary, float>("tc_cp_summary", p, maps, st)) return 1;
        if (simt_cp_combine(p, st)) return 1;
    }
    return o_f32 ? launch_scan<kFwd, float>("tc_scan", p, maps, st)
                 : launch_scan<kFwd, __nv_bfloat16>("tc_scan", p, maps, st);
}

int tc_bwd(const Params &p, int use_cp, cudaStream_t st) { return simt_bwd(p, 0, use_cp, st); }

unsigned tc_take_status(cudaStream_t st) {
    unsigned v = 0, z = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_tc_status, sizeof(v), 0, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return 0x80000000u;
    cudaMemcpyToSymbolAsync(g_tc_status, &z, sizeof(z), 0, cudaMemcpyHostToDevice, st);
    if (cudaStreamSynchronize(st) != cudaSuccess) return 0x80000000u;
    return v;
}

}  // namespace gdr
