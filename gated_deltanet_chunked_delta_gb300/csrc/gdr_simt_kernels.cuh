// gdr_simt_kernels.cuh -- the CUDA-core (fp32 FFMA) path of the GDN chunked
// prefill: the kernels, templated on the head sizes, and the per-size launch
// sequence.  Each translation unit that includes this file instantiates the
// head sizes it dispatches (gdr_simt.cu: K, V in {64, 128}; gdr_simt_wide_k.cu:
// K = 192; gdr_simt_wide_v.cu: V in {192, 256}), so that they compile in
// parallel, and keeps its own device status word.
//
// This path computes every step in fp32 on the CUDA cores.  It serves fp32
// inputs (where bf16 tensor-core operands would not meet an fp32 tolerance),
// every head size other than K = V = 128 (K up to 192, V up to 256: the scans
// keep K x 33 and 64 x (K + 1) fp32 tiles in shared memory, and V is taken in
// 32-column blocks), and is the cross-check of the tensor-core path.
//
// Chunk algebra (one chunk of n <= 64 rows; FlashQLA pages: the forward of
// chunk i reads K and V and passes W, U and the state S between steps, page 1
// "efficiency problem"; the split into a chunk-parallel kernel and a scan with
// a context-parallel step between them, page 1 "two fused kernels and
// automatic CP"):
//   gamma_r = sum_{s<=r} g_s,  D_rs = exp(gamma_r - gamma_s)
//   L = strict_tril(diag(b)(K K^T o D)),  A = (I + L)^-1
//   W = A diag(b e^gamma) K,   U = A diag(b) V
//   Ut = U - W S0
//   O  = Qt S0 + P Ut,  Qt = scale diag(e^gamma) Q,  P = scale (Q K^T o D o tril_incl)
//   S1 = e^{gamma_n} S0 + Kt^T Ut,  Kt = diag(e^{gamma_n - gamma}) K
// Partial chunks are zero-padded (k = q = v = 0, b = 0, g = 0), which makes the
// padded rows inert in every product.  The columns of S evolve independently,
// so every scan kernel owns a 32-column block of the state.
//
// Backward (reverse mode of the chunk algebra; R = diag(b)V - diag(b e^gamma) K S0,
// so Ut = A R):
//   dUt = P^T dO + Kt dS1  (reverse state scan),  dS0 = e^{gamma_n} dS1 + Qt^T dO - W^T dUt
//   dQt = dO S0^T,  dP = dO Ut^T,  dKt = Ut dS1^T,  dBv = A^T dUt,  dBk = -dBv S0^T,
//   dA = dUt R^T,   dL = -strict_tril(A^T dA A^T)
// and the per-entry chain rule through Qt, P, Kt, B_k = diag(b e^gamma)K,
// B_v = diag(b)V and L into dq, dk, dv, dbeta and dgamma; dg is the reverse
// cumulative sum of dgamma inside the chunk.
#pragma once

#include <cuda_bf16.h>

#include "gdr_internal.h"

namespace gdr {
namespace {

__device__ unsigned g_simt_status;

__device__ __forceinline__ float ldf(const float *p, size_t i) { return p[i]; }
__device__ __forceinline__ float ldf(const __nv_bfloat16 *p, size_t i) {
    return __bfloat162float(p[i]);
}
__device__ __forceinline__ void stf(float *p, size_t i, float x) { p[i] = x; }
__device__ __forceinline__ void stf(__nv_bfloat16 *p, size_t i, float x) {
    p[i] = __float2bfloat16_rn(x);
}

// Debug-mode index check: records the failure and tells the caller to skip.
__device__ __forceinline__ bool bad(const Params &p, bool cond) {
    if (p.debug && cond) {
        atomicOr(&g_simt_status, 2u);
        return true;
    }
    return false;
}

// ---------------------------------------------------------------------------
// K1: per (chunk, v-head): gamma, A (inverted, or read back in the backward),
// P, W, U.  256 threads.
// ---------------------------------------------------------------------------
template <typename TI, int KD, int VD>
__global__ void __launch_bounds__(256) k_wy(Params p, int from_A) {
    constexpr int DM = KD > VD ? KD : VD;
    constexpr int LD = DM + 1;
    extern __shared__ float sm[];
    float *Ks = sm;              // [64][LD]  k, then B_k = diag(b e^gamma) k
    float *Xs = Ks + 64 * LD;    // [64][LD]  q, then B_v = diag(b) v
    float *Lm = Xs + 64 * LD;    // [64][65]
    float *Am = Lm + 64 * 65;    // [64][65]
    float *gam = Am + 64 * 65;   // [64]
    float *bet = gam + 64;       // [64]
    const int c = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
    const ChunkInfo ci = p.chunk[c];
    const int len = ci.len, tok0 = ci.tok0;
    if (bad(p, len < 1 || len > 64 || tok0 < 0 || tok0 + len > p.Ttot)) return;
    const int hq = h / (p.Hv / p.Hq);
    const TI *k = (const TI *)p.k;
    const TI *q = (const TI *)p.q;
    const TI *v = (const TI *)p.v;
    for (int idx = tid; idx < 64 * KD; idx += 256) {
        const int r = idx / KD, i = idx % KD;
        const size_t off = ((size_t)(tok0 + r) * p.Hq + hq) * KD + i;
        Ks[r * LD + i] = r < len ? ldf(k, off) : 0.f;
        Xs[r * LD + i] = r < len ? ldf(q, off) : 0.f;
    }
    if (tid < 64) {
        gam[tid] = tid < len ? p.g[(size_t)(tok0 + tid) * p.Hv + h] : 0.f;
        bet[tid] = tid < len ? p.beta[(size_t)(tok0 + tid) * p.Hv + h] : 0.f;
    }
    __syncthreads();
    if (tid == 0) {
        float a = 0.f;
        for (int r = 0; r < 64; ++r) { a += gam[r]; gam[r] = a; }
    }
    __syncthreads();
    if (!from_A) {
        for (int idx = tid; idx < 64 * 64; idx += 256) {
            const int r = idx >> 6, s = idx & 63;
            float val = 0.f;
            if (s < r) {
                float d = 0.f;
                for (int i = 0; i < KD; ++i) d += Ks[r * LD + i] * Ks[s * LD + i];
                val = bet[r] * __expf(gam[r] - gam[s]) * d;
            }
            Lm[r * 65 + s] = val;
        }
        __syncthreads();
        // (I + L)^-1 by forward substitution; four lanes share one column.
        const int j = tid >> 2, part = tid & 3;
        for (int r = 0; r < 64; ++r) {
            float acc = 0.f;
            for (int s = j + part; s < r; s += 4) acc += Lm[r * 65 + s] * Am[s * 65 + j];
            acc += __shfl_xor_sync(0xffffffffu, acc, 1);
            acc += __shfl_xor_sync(0xffffffffu, acc, 2);
            if (part == 0) Am[r * 65 + j] = (r < j) ? 0.f : ((r == j) ? 1.f : -acc);
            __syncwarp();
        }
    } else {
        for (int idx = tid; idx < 64 * 64; idx += 256) {
            const int r = idx >> 6, s = idx & 63;
            Am[r * 65 + s] = r < len ? p.A_in[((size_t)(tok0 + r) * p.Hv + h) * 64 + s]
                                     : (r == s ? 1.f : 0.f);
        }
    }
    __syncthreads();
    if (p.A_out && !from_A)
        for (int idx = tid; idx < len * 64; idx += 256) {
            const int r = idx >> 6, s = idx & 63;
            p.A_out[((size_t)(tok0 + r) * p.Hv + h) * 64 + s] = Am[r * 65 + s];
        }
    const size_t ch = (size_t)c * p.Hv + h;
    for (int idx = tid; idx < 64 * 64; idx += 256) {
        const int r = idx >> 6, s = idx & 63;
        float val = 0.f;
        if (s <= r) {
            float d = 0.f;
            for (int i = 0; i < KD; ++i) d += Xs[r * LD + i] * Ks[s * LD + i];
            val = p.scale * __expf(gam[r] - gam[s]) * d;
        }
        p.P[ch * 64 * 64 + idx] = val;
    }
    __syncthreads();
    for (int idx = tid; idx < 64 * KD; idx += 256) {
        const int r = idx / KD, i = idx % KD;
        Ks[r * LD + i] *= bet[r] * __expf(gam[r]);
    }
    for (int idx = tid; idx < 64 * VD; idx += 256) {
        const int r = idx / VD, jj = idx % VD;
        Xs[r * LD + jj] = r < len ? bet[r] * ldf(v, ((size_t)(tok0 + r) * p.Hv + h) * VD + jj) : 0.f;
    }
    __syncthreads();
    for (int idx = tid; idx < 64 * KD; idx += 256) {
        const int r = idx / KD, i = idx % KD;
        float acc = 0.f;
        for (int s = 0; s <= r; ++s) acc += Am[r * 65 + s] * Ks[s * LD + i];
        p.W[ch * 64 * KD + idx] = acc;
    }
    for (int idx = tid; idx < 64 * VD; idx += 256) {
        const int r = idx / VD, jj = idx % VD;
        float acc = 0.f;
        for (int s = 0; s <= r; ++s) acc += Am[r * 65 + s] * Xs[s * LD + jj];
        p.U[ch * 64 * VD + idx] = acc;
    }
    if (tid < 64) p.gam[((size_t)c * p.Hv + h) * 64 + tid] = gam[tid];
}

// ---------------------------------------------------------------------------
// K2 (context parallel, step 1): per (segment, v-head, 32 columns of [S | M]):
// run the segment from X = [0 | I] with pseudo-values [U | 0].  The columns of
// X evolve independently.  The last segment of a sequence needs no summary.
// ---------------------------------------------------------------------------
template <typename TI, int KD, int VD>
__global__ void __launch_bounds__(256) k_cp_summary(Params p) {
    constexpr int LD = KD + 1;
    extern __shared__ float sm[];
    float *X = sm;              // [KD][33]
    float *Ws = X + KD * 33;    // [64][LD]
    float *Kt = Ws + 64 * LD;   // [64][LD]
    float *R = Kt + 64 * LD;    // [64][33]
    float *gam = R + 64 * 33;   // [64]
    const int sidx = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
    const SegInfo sg = p.seg[sidx];
    const SeqInfo sq = p.seq[sg.seq];
    if (sg.idx >= sq.nseg - 1) return;
    const int x0 = blockIdx.z * 32;
    const bool isS = x0 < VD;
    const int hq = h / (p.Hv / p.Hq);
    for (int idx = tid; idx < KD * 32; idx += 256) {
        const int i = idx >> 5, j = idx & 31;
        X[i * 33 + j] = isS ? 0.f : ((i == x0 - VD + j) ? 1.f : 0.f);
    }
    for (int cc = 0; cc < sg.nch; ++cc) {
        const int c = sg.chunk0 + cc;
        const ChunkInfo ci = p.chunk[c];
        __syncthreads();
        if (tid < 64) gam[tid] = p.gam[((size_t)c * p.Hv + h) * 64 + tid];
        const float *Wg = p.W + ((size_t)c * p.Hv + h) * 64 * KD;
        for (int idx = tid; idx < 64 * KD; idx += 256) Ws[(idx / KD) * LD + idx % KD] = Wg[idx];
        for (int idx = tid; idx < 64 * 32; idx += 256) {
            const int r = idx >> 5, j = idx & 31;
            R[r * 33 + j] = isS ? p.U[(((size_t)c * p.Hv + h) * 64 + r) * VD + x0 + j] : 0.f;
        }
        __syncthreads();
        const float gl = gam[63];
        for (int idx = tid; idx < 64 * KD; idx += 256) {
            const int r = idx / KD, i = idx % KD;
            Kt[r * LD + i] = r < ci.len ? __expf(gl - gam[r]) *
                                              ldf((const TI *)p.k, ((size_t)(ci.tok0 + r) * p.Hq + hq) * KD + i)
                                        : 0.f;
        }
        for (int idx = tid; idx < 64 * 32; idx += 256) {
            const int r = idx >> 5, j = idx & 31;
            float acc = 0.f;
            for (int i = 0; i < KD; ++i) acc += Ws[r * LD + i] * X[i * 33 + j];
            R[r * 33 + j] -= acc;
        }
        __syncthreads();
        const float dec = __expf(gl);
        for (int idx = tid; idx < KD * 32; idx += 256) {
            const int i = idx >> 5, j = idx & 31;
            float acc = dec * X[i * 33 + j];
            for (int r = 0; r < 64; ++r) acc += Kt[r * LD + i] * R[r * 33 + j];
            X[i * 33 + j] = acc;
        }
    }
    __syncthreads();
    for (int idx = tid; idx < KD * 32; idx += 256) {
        const int i = idx >> 5, j = idx & 31;
        if (isS)
            p.Hseg[(((size_t)sidx * p.Hv + h) * KD + i) * VD + x0 + j] = X[i * 33 + j];
        else
            p.Mseg[(((size_t)sidx * p.Hv + h) * KD + i) * KD + x0 - VD + j] = X[i * 33 + j];
    }
}

// ---------------------------------------------------------------------------
// K3 (context parallel, step 2): per (sequence, v-head, 8 state columns), in
// segment order: S_start(j+1) = M_j S_start(j) + H_j from S_start(0) = h0.
// The reverse form serves the segmented backward scan: dS_end(last) = dht,
// dS_end(j) = N_{j+1} dS_end(j+1) + G_{j+1} (N in Mseg, G in Hseg), written
// to Sstart[j].  Each step's matrix is staged in shared memory; the next
// step's matrix and offsets are loaded into registers while this step
// computes.  Two threads share a row.
// ---------------------------------------------------------------------------
constexpr int kCombCols = 8;

template <int KD, int VD, bool kRev>
__global__ void __launch_bounds__(256) k_cp_combine(Params p) {
    extern __shared__ float sm[];
    float *Ms = sm;                  // [KD][KD+1]
    float *S = Ms + KD * (KD + 1);   // [KD][8]
    const int n = blockIdx.x, h = blockIdx.y, v0 = blockIdx.z * kCombCols, tid = threadIdx.x;
    const SeqInfo sq = p.seq[n];
    if (sq.nseg <= 1) return;
    const float *init = kRev ? p.dht : p.h0;
    for (int idx = tid; idx < KD * kCombCols; idx += 256) {
        const int i = idx >> 3, j = idx & 7;
        S[idx] = init ? init[(((size_t)n * p.Hv + h) * KD + i) * VD + v0 + j] : 0.f;
    }
    const int nsteps = sq.nseg - 1;
    constexpr int NL = KD * KD / 4 / 256;
    int rows[2], j0s[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int o = tid + 256 * u;
        rows[u] = o < KD * 2 ? (o >> 1) : -1;
        j0s[u] = (o & 1) * 4;
    }
    float4 mv[NL];
    float hv[2][4];
    // step -> the segment whose summary it applies
    auto seg_of = [&](int step) -> size_t { return (size_t)sq.seg0 + (kRev ? (sq.nseg - 1 - step) : step); };
    auto load = [&](int step) {
        const size_t sgi = seg_of(step);
        const float4 *M4 = reinterpret_cast<const float4 *>(p.Mseg + (sgi * p.Hv + h) * KD * KD);
        const float *Hs = p.Hseg + (sgi * p.Hv + h) * KD * VD;
#pragma unroll
        for (int u = 0; u < NL; ++u) mv[u] = M4[tid + 256 * u];
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int e = 0; e < 4; ++e) hv[u][e] = rows[u] >= 0 ? Hs[rows[u] * VD + v0 + j0s[u] + e] : 0.f;
    };
    load(0);
    for (int step = 0; step < nsteps; ++step) {
        const size_t sgi = seg_of(step);
        float *dst = p.Sstart + ((kRev ? sgi - 1 : sgi + 1) * p.Hv + h) * KD * VD;
        __syncthreads();
#pragma unroll
        for (int u = 0; u < NL; ++u) {
            const int idx = tid + 256 * u, row = idx / (KD / 4), c = 4 * (idx % (KD / 4));
            float *d = Ms + row * (KD + 1) + c;
            d[0] = mv[u].x; d[1] = mv[u].y; d[2] = mv[u].z; d[3] = mv[u].w;
        }
        float acc[2][4];
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[u][e] = hv[u][e];
        __syncthreads();
        if (step + 1 < nsteps) load(step + 1);  // in flight during this step's products
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            if (rows[u] < 0) continue;
#pragma unroll 16
            for (int l = 0; l < KD; ++l) {
                const float m = Ms[rows[u] * (KD + 1) + l];
                const float4 sv = *reinterpret_cast<const float4 *>(S + l * kCombCols + j0s[u]);
                acc[u][0] += m * sv.x;
                acc[u][1] += m * sv.y;
                acc[u][2] += m * sv.z;
                acc[u][3] += m * sv.w;
            }
        }
        __syncthreads();
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            if (rows[u] < 0) continue;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                S[rows[u] * kCombCols + j0s[u] + e] = acc[u][e];
                dst[rows[u] * VD + v0 + j0s[u] + e] = acc[u][e];
            }
        }
    }
}

template <int KD>
constexpr size_t smem_combine() {
    return sizeof(float) * (KD * (KD + 1) + KD * kCombCols);
}

// ---------------------------------------------------------------------------
// K4 (step 3): per (segment, v-head, 32 state columns): the sequential scan
// over the segment's chunks from its true start state.  kOut: emit o and h;
// otherwise only store the states before every chunk (backward recompute).
// ---------------------------------------------------------------------------
template <typename TI, typename TO, int KD, int VD, bool kOut>
__global__ void __launch_bounds__(256) k_scan(Params p) {
    constexpr int LD = KD + 1;
    extern __shared__ float sm[];
    float *S = sm;               // [KD][33]
    float *Ws = S + KD * 33;     // [64][LD]
    float *Qt = Ws + 64 * LD;    // [64][LD]
    float *Kt = Qt + 64 * LD;    // [64][LD]
    float *Pm = Kt + 64 * LD;    // [64][65]
    float *Ub = Pm + 64 * 65;    // [64][33]
    float *gam = Ub + 64 * 33;   // [64]
    const int sidx = blockIdx.x, h = blockIdx.y, v0 = blockIdx.z * 32, tid = threadIdx.x;
    const SegInfo sg = p.seg[sidx];
    const SeqInfo sq = p.seq[sg.seq];
    const int hq = h / (p.Hv / p.Hq);
    for (int idx = tid; idx < KD * 32; idx += 256) {
        const int i = idx >> 5, j = idx & 31;
        float s0;
        if (sg.idx == 0)
            s0 = p.h0 ? p.h0[(((size_t)sg.seq * p.Hv + h) * KD + i) * VD + v0 + j] : 0.f;
        else
            s0 = p.Sstart[(((size_t)sidx * p.Hv + h) * KD + i) * VD + v0 + j];
        S[i * 33 + j] = s0;
    }
    float *hdst = kOut ? p.h_out : p.hbuf;
    for (int cc = 0; cc < sg.nch; ++cc) {
        const int c = sg.chunk0 + cc;
        const ChunkInfo ci = p.chunk[c];
        if (bad(p, ci.len < 1 || ci.len > 64 || ci.tok0 + ci.len > p.Ttot)) return;
        __syncthreads();
        if (hdst)
            for (int idx = tid; idx < KD * 32; idx += 256) {
                const int i = idx >> 5, j = idx & 31;
                hdst[(((size_t)c * p.Hv + h) * KD + i) * VD + v0 + j] = S[i * 33 + j];
            }
        if (tid < 64) gam[tid] = p.gam[((size_t)c * p.Hv + h) * 64 + tid];
        const float *Wg = p.W + ((size_t)c * p.Hv + h) * 64 * KD;
        for (int idx = tid; idx < 64 * KD; idx += 256) Ws[(idx / KD) * LD + idx % KD] = Wg[idx];
        if (kOut) {
            const float *Pg = p.P + ((size_t)c * p.Hv + h) * 64 * 64;
            for (int idx = tid; idx < 64 * 64; idx += 256) Pm[(idx >> 6) * 65 + (idx & 63)] = Pg[idx];
        }
        for (int idx = tid; idx < 64 * 32; idx += 256) {
            const int r = idx >> 5, j = idx & 31;
            Ub[r * 33 + j] = p.U[(((size_t)c * p.Hv + h) * 64 + r) * VD + v0 + j];
        }
        __syncthreads();
        const float gl = gam[63];
        for (int idx = tid; idx < 64 * KD; idx += 256) {
            const int r = idx / KD, i = idx % KD;
            const size_t off = ((size_t)(ci.tok0 + r) * p.Hq + hq) * KD + i;
            const bool in = r < ci.len;
            if (kOut) Qt[r * LD + i] = in ? p.scale * __expf(gam[r]) * ldf((const TI *)p.q, off) : 0.f;
            Kt[r * LD + i] = in ? __expf(gl - gam[r]) * ldf((const TI *)p.k, off) : 0.f;
        }
        for (int idx = tid; idx < 64 * 32; idx += 256) {
            const int r = idx >> 5, j = idx & 31;
            float acc = 0.f;
            for (int i = 0; i < KD; ++i) acc += Ws[r * LD + i] * S[i * 33 + j];
            Ub[r * 33 + j] -= acc;
        }
        __syncthreads();
        if (kOut) {
            TO *o = (TO *)p.o;
            for (int idx = tid; idx < 64 * 32; idx += 256) {
                const int r = idx >> 5, j = idx & 31;
                float acc = 0.f;
                for (int i = 0; i < KD; ++i) acc += Qt[r * LD + i] * S[i * 33 + j];
                for (int s = 0; s <= r; ++s) acc += Pm[r * 65 + s] * Ub[s * 33 + j];
                if (r < ci.len) stf(o, ((size_t)(ci.tok0 + r) * p.Hv + h) * VD + v0 + j, acc);
            }
            __syncthreads();
        }
        const float dec = __expf(gl);
        for (int idx = tid; idx < KD * 32; idx += 256) {
            const int i = idx >> 5, j = idx & 31;
            float acc = dec * S[i * 33 + j];
            for (int r = 0; r < 64; ++r) acc += Kt[r * LD + i] * Ub[r * 33 + j];
            S[i * 33 + j] = acc;
        }
    }
    __syncthreads();
    if (sg.idx == sq.nseg - 1 && p.final_state)
        for (int idx = tid; idx < KD * 32; idx += 256) {
            const int i = idx >> 5, j = idx & 31;
            p.final_state[(((size_t)sg.seq * p.Hv + h) * KD + i) * VD + v0 + j] = S[i * 33 + j];
        }
}

// ---------------------------------------------------------------------------
// B2: reverse state scan per (sequence, v-head, 32 columns):
// stores dS1 of every chunk and dUt = P^T dO + Kt dS1; ends with dh0.
// ---------------------------------------------------------------------------
template <typename TI, int KD, int VD>
__global__ void __launch_bounds__(256) k_dh(Params p) {
    constexpr int LD = KD + 1;
    extern __shared__ float sm[];
    float *dS = sm;              // [KD][33]
    float *Ws = dS + KD * 33;    // [64][LD]
    float *Qt = Ws + 64 * LD;    // [64][LD]
    float *Kt = Qt + 64 * LD;    // [64][LD]
    float *Pm = Kt + 64 * LD;    // [64][65]
    float *dOb = Pm + 64 * 65;   // [64][33]
    float *dUb = dOb + 64 * 33;  // [64][33]
    float *gam = dUb + 64 * 33;  // [64]
    const int n = blockIdx.x, h = blockIdx.y, v0 = blockIdx.z * 32, tid = threadIdx.x;
    const SeqInfo sq = p.seq[n];
    const int hq = h / (p.Hv / p.Hq);
    for (int idx = tid; idx < KD * 32; idx += 256) {
        const int i = idx >> 5, j = idx & 31;
        dS[i * 33 + j] = p.dht ? p.dht[(((size_t)n * p.Hv + h) * KD + i) * VD + v0 + j] : 0.f;
    }
    for (int cc = sq.nch - 1; cc >= 0; --cc) {
        const int c = sq.chunk0 + cc;
        const ChunkInfo ci = p.chunk[c];
        __syncthreads();
        for (int idx = tid; idx < KD * 32; idx += 256) {
            const int i = idx >> 5, j = idx & 31;
            p.dhbuf[(((size_t)c * p.Hv + h) * KD + i) * VD + v0 + j] = dS[i * 33 + j];
        }
        if (tid < 64) gam[tid] = p.gam[((size_t)c * p.Hv + h) * 64 + tid];
        const float *Wg = p.W + ((size_t)c * p.Hv + h) * 64 * KD;
        for (int idx = tid; idx < 64 * KD; idx += 256) Ws[(idx / KD) * LD + idx % KD] = Wg[idx];
        const float *Pg = p.P + ((size_t)c * p.Hv + h) * 64 * 64;
        for (int idx = tid; idx < 64 * 64; idx += 256) Pm[(idx >> 6) * 65 + (idx & 63)] = Pg[idx];
        for (int idx = tid; idx < 64 * 32; idx += 256) {
            const int r = idx >> 5, j = idx & 31;
            dOb[r * 33 + j] = r < ci.len
                                  ? ldf((const TI *)p.dout, ((size_t)(ci.tok0 + r) * p.Hv + h) * VD + v0 + j)
                                  : 0.f;
        }
        __syncthreads();
        const float gl = gam[63];
        for (int idx = tid; idx < 64 * KD; idx += 256) {
            const int r = idx / KD, i = idx % KD;
            const size_t off = ((size_t)(ci.tok0 + r) * p.Hq + hq) * KD + i;
            const bool in = r < ci.len;
            Qt[r * LD + i] = in ? p.scale * __expf(gam[r]) * ldf((const TI *)p.q, off) : 0.f;
            Kt[r * LD + i] = in ? __expf(gl - gam[r]) * ldf((const TI *)p.k, off) : 0.f;
        }
        __syncthreads();
        for (int idx = tid; idx < 64 * 32; idx += 256) {
            const int r = idx >> 5, j = idx & 31;
            float acc = 0.f;
            for (int s = r; s < 64; ++s) acc += Pm[s * 65 + r] * dOb[s * 33 + j];
            for (int i = 0; i < KD; ++i) acc += Kt[r * LD + i] * dS[i * 33 + j];
            dUb[r * 33 + j] = acc;
            p.dubuf[(((size_t)c * p.Hv + h) * 64 + r) * VD + v0 + j] = acc;
        }
        __syncthreads();
        const float dec = __expf(gl);
        for (int idx = tid; idx < KD * 32; idx += 256) {
            const int i = idx >> 5, j = idx & 31;
            float acc = dec * dS[i * 33 + j];
            for (int r = 0; r < 64; ++r) acc += Qt[r * LD + i] * dOb[r * 33 + j] - Ws[r * LD + i] * dUb[r * 33 + j];
            dS[i * 33 + j] = acc;
        }
    }
    __syncthreads();
    if (p.dh0)
        for (int idx = tid; idx < KD * 32; idx += 256) {
            const int i = idx >> 5, j = idx & 31;
            p.dh0[(((size_t)n * p.Hv + h) * KD + i) * VD + v0 + j] = dS[i * 33 + j];
        }
}

// ---------------------------------------------------------------------------
// B3: per (chunk, v-head): every chunk-local gradient.  dq, dk go to per-v-head
// fp32 partials (summed over the group afterwards); dv, dbeta, dg are final.
// ---------------------------------------------------------------------------
template <typename TI, int KD, int VD>
__global__ void __launch_bounds__(256) k_bwd_chunk(Params p) {
    constexpr int LD = KD + 1;
    constexpr int VB = 16, LB = VB + 1;
    constexpr int NI = KD / 4;
    extern __shared__ float sm[];
    float *Ks = sm;               // [64][LD]
    float *Qs = Ks + 64 * LD;     // [64][LD]
    float *Am = Qs + 64 * LD;     // [64][65]
    float *dP = Am + 64 * 65;     // [64][65]
    float *dA = dP + 64 * 65;     // [64][65]  later dL
    float *S0b = dA + 64 * 65;    // [KD][LB]
    float *dS1b = S0b + KD * LB;  // [KD][LB]
    float *dOb = dS1b + KD * LB;  // [64][LB]
    float *dUb = dOb + 64 * LB;
    float *Vb = dUb + 64 * LB;
    float *Rb = Vb + 64 * LB;
    float *Ub = Rb + 64 * LB;
    float *dBv = Ub + 64 * LB;
    float *gam = dBv + 64 * LB;   // [64]
    float *bet = gam + 64;        // [64]
    float *dbv = bet + 64;        // [64]
    float *rowQ = dbv + 64;       // [64]
    float *rowK = rowQ + 64;      // [64]
    float *rowB = rowK + 64;      // [64]
    float *dgs = rowB + 64;       // [64]
    float *red = dgs + 64;        // [8]
    float *X = S0b;               // [64][65] after the column loop
    float *QK = S0b + 64 * 65;    // [64][65] after the column loop
    const int c = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
    const ChunkInfo ci = p.chunk[c];
    const int len = ci.len, tok0 = ci.tok0;
    if (bad(p, len < 1 || len > 64 || tok0 + len > p.Ttot)) return;
    const int hq = h / (p.Hv / p.Hq);
    const TI *kin = (const TI *)p.k;
    const TI *qin = (const TI *)p.q;
    const TI *vin = (const TI *)p.v;
    const TI *din = (const TI *)p.dout;
    for (int idx = tid; idx < 64 * KD; idx += 256) {
        const int r = idx / KD, i = idx % KD;
        const size_t off = ((size_t)(tok0 + r) * p.Hq + hq) * KD + i;
        Ks[r * LD + i] = r < len ? ldf(kin, off) : 0.f;
        Qs[r * LD + i] = r < len ? ldf(qin, off) : 0.f;
    }
    for (int idx = tid; idx < 64 * 64; idx += 256) {
        const int r = idx >> 6, s = idx & 63;
        Am[r * 65 + s] = r < len ? p.A_in[((size_t)(tok0 + r) * p.Hv + h) * 64 + s] : (r == s ? 1.f : 0.f);
        dP[r * 65 + s] = 0.f;
        dA[r * 65 + s] = 0.f;
    }
    if (tid < 64) {
        gam[tid] = tid < len ? p.g[(size_t)(tok0 + tid) * p.Hv + h] : 0.f;
        bet[tid] = tid < len ? p.beta[(size_t)(tok0 + tid) * p.Hv + h] : 0.f;
        dbv[tid] = 0.f;
    }
    if (tid < 8) red[tid] = 0.f;
    __syncthreads();
    if (tid == 0) {
        float a = 0.f;
        for (int r = 0; r < 64; ++r) { a += gam[r]; gam[r] = a; }
    }
    __syncthreads();
    const int ro = tid >> 2, io = tid & 3;
    float aQ[NI], aK[NI], aB[NI];
#pragma unroll
    for (int m = 0; m < NI; ++m) { aQ[m] = 0.f; aK[m] = 0.f; aB[m] = 0.f; }
    float s0ds1 = 0.f;
    const float *S0g = p.hbuf + ((size_t)c * p.Hv + h) * KD * VD;
    const float *dS1g = p.dhbuf + ((size_t)c * p.Hv + h) * KD * VD;
    const float *dUg = p.dubuf + ((size_t)c * p.Hv + h) * 64 * VD;
    for (int v0 = 0; v0 < VD; v0 += VB) {
        for (int idx = tid; idx < KD * VB; idx += 256) {
            const int i = idx / VB, j = idx % VB;
            S0b[i * LB + j] = S0g[i * VD + v0 + j];
            dS1b[i * LB + j] = dS1g[i * VD + v0 + j];
        }
        for (int idx = tid; idx < 64 * VB; idx += 256) {
            const int r = idx / VB, j = idx % VB;
            const size_t off = ((size_t)(tok0 + r) * p.Hv + h) * VD + v0 + j;
            dOb[r * LB + j] = r < len ? ldf(din, off) : 0.f;
            Vb[r * LB + j] = r < len ? ldf(vin, off) : 0.f;
            dUb[r * LB + j] = dUg[r * VD + v0 + j];
        }
        __syncthreads();
        for (int idx = tid; idx < 64 * VB; idx += 256) {
            const int r = idx / VB, j = idx % VB;
            float acc = 0.f;
            for (int i = 0; i < KD; ++i) acc += Ks[r * LD + i] * S0b[i * LB + j];
            Rb[r * LB + j] = bet[r] * (Vb[r * LB + j] - __expf(gam[r]) * acc);
        }
        for (int idx = tid; idx < KD * VB; idx += 256) {
            const int i = idx / VB, j = idx % VB;
            s0ds1 += S0b[i * LB + j] * dS1b[i * LB + j];
        }
        __syncthreads();
        for (int idx = tid; idx < 64 * VB; idx += 256) {
            const int r = idx / VB, j = idx % VB;
            float u = 0.f, d = 0.f;
            for (int s = 0; s <= r; ++s) u += Am[r * 65 + s] * Rb[s * LB + j];
            for (int s = r; s < 64; ++s) d += Am[s * 65 + r] * dUb[s * LB + j];
            Ub[r * LB + j] = u;
            dBv[r * LB + j] = d;
        }
        __syncthreads();
        for (int j = 0; j < VB; ++j) {
            const float o_ = dOb[ro * LB + j], u_ = Ub[ro * LB + j], b_ = dBv[ro * LB + j];
#pragma unroll
            for (int m = 0; m < NI; ++m) {
                const int i = io + 4 * m;
                const float s0 = S0b[i * LB + j];
                aQ[m] += o_ * s0;
                aK[m] += u_ * dS1b[i * LB + j];
                aB[m] -= b_ * s0;
            }
        }
        for (int e = 0; e < 16; ++e) {
            const int idx = tid + 256 * e;
            const int r = idx >> 6, s = idx & 63;
            float a1 = 0.f, a2 = 0.f;
            for (int j = 0; j < VB; ++j) {
                a1 += dOb[r * LB + j] * Ub[s * LB + j];
                a2 += dUb[r * LB + j] * Rb[s * LB + j];
            }
            if (s <= r) dP[r * 65 + s] += a1;
            dA[r * 65 + s] += a2;
        }
        for (int idx = tid; idx < 64 * VB; idx += 256) {
            const int r = idx / VB, j = idx % VB;
            if (r < len) {
                stf((TI *)p.dv, ((size_t)(tok0 + r) * p.Hv + h) * VD + v0 + j, bet[r] * dBv[r * LB + j]);
                atomicAdd(&dbv[r], dBv[r * LB + j] * Vb[r * LB + j]);
            }
        }
        __syncthreads();
    }
    // <dS1, S0>
    for (int o = 16; o > 0; o >>= 1) s0ds1 += __shfl_xor_sync(0xffffffffu, s0ds1, o);
    if ((tid & 31) == 0) atomicAdd(&red[0], s0ds1);
    {
        float pq = 0.f, pk = 0.f, pb = 0.f;
#pragma unroll
        for (int m = 0; m < NI; ++m) {
            const int i = io + 4 * m;
            pq += aQ[m] * Qs[ro * LD + i];
            pk += aK[m] * Ks[ro * LD + i];
            pb += aB[m] * Ks[ro * LD + i];
        }
        for (int o = 1; o < 4; o <<= 1) {
            pq += __shfl_xor_sync(0xffffffffu, pq, o);
            pk += __shfl_xor_sync(0xffffffffu, pk, o);
            pb += __shfl_xor_sync(0xffffffffu, pb, o);
        }
        if (io == 0) { rowQ[ro] = pq; rowK[ro] = pk; rowB[ro] = pb; }
    }
    // X = A^T dA
    for (int idx = tid; idx < 64 * 64; idx += 256) {
        const int r = idx >> 6, m = idx & 63;
        float acc = 0.f;
        for (int q2 = r; q2 < 64; ++q2) acc += Am[q2 * 65 + r] * dA[q2 * 65 + m];
        X[r * 65 + m] = acc;
    }
    __syncthreads();
    // dL = -strict_tril(X A^T), written over dA
    for (int idx = tid; idx < 64 * 64; idx += 256) {
        const int r = idx >> 6, s = idx & 63;
        float acc = 0.f;
        if (s < r)
            for (int m = 0; m <= s; ++m) acc -= X[r * 65 + m] * Am[s * 65 + m];
        dA[r * 65 + s] = acc;
    }
    __syncthreads();
    float *KK = X;
    for (int idx = tid; idx < 64 * 64; idx += 256) {
        const int r = idx >> 6, s = idx & 63;
        float a1 = 0.f, a2 = 0.f;
        for (int i = 0; i < KD; ++i) {
            a1 += Ks[r * LD + i] * Ks[s * LD + i];
            a2 += Qs[r * LD + i] * Ks[s * LD + i];
        }
        KK[r * 65 + s] = a1;
        QK[r * 65 + s] = a2;
    }
    __syncthreads();
    const float *dL = dA;
    const float gl = gam[63];
    {
        // dq for (ro, io + 4m)
        const float egr = __expf(gam[ro]);
#pragma unroll
        for (int m = 0; m < NI; ++m) aQ[m] *= p.scale * egr;
        for (int s = 0; s <= ro; ++s) {
            const float f = dP[ro * 65 + s] * p.scale * __expf(gam[ro] - gam[s]);
#pragma unroll
            for (int m = 0; m < NI; ++m) aQ[m] += f * Ks[s * LD + io + 4 * m];
        }
        // dk
        const float eL = __expf(gl - gam[ro]);
        const float fb = bet[ro] * egr;
#pragma unroll
        for (int m = 0; m < NI; ++m) aK[m] = eL * aK[m] + fb * aB[m];
        for (int r2 = ro; r2 < 64; ++r2) {
            const float f = dP[r2 * 65 + ro] * p.scale * __expf(gam[r2] - gam[ro]);
#pragma unroll
            for (int m = 0; m < NI; ++m) aK[m] += f * Qs[r2 * LD + io + 4 * m];
        }
        for (int s = 0; s < ro; ++s) {
            const float f = dL[ro * 65 + s] * bet[ro] * __expf(gam[ro] - gam[s]);
#pragma unroll
            for (int m = 0; m < NI; ++m) aK[m] += f * Ks[s * LD + io + 4 * m];
        }
        for (int r2 = ro + 1; r2 < 64; ++r2) {
            const float f = dL[r2 * 65 + ro] * bet[r2] * __expf(gam[r2] - gam[ro]);
#pragma unroll
            for (int m = 0; m < NI; ++m) aK[m] += f * Ks[r2 * LD + io + 4 * m];
        }
        if (ro < len) {
#pragma unroll
            for (int m = 0; m < NI; ++m) {
                const size_t off = ((size_t)(tok0 + ro) * p.Hv + h) * KD + io + 4 * m;
                p.dqp[off] = aQ[m];
                p.dkp[off] = aK[m];
            }
        }
    }
    if (tid < 64) {
        const int r = tid;
        const float egr = __expf(gam[r]);
        float dgam = p.scale * egr * rowQ[r] - __expf(gl - gam[r]) * rowK[r] + bet[r] * egr * rowB[r];
        float db = dbv[r] + egr * rowB[r];
        for (int s = 0; s <= r; ++s)
            dgam += dP[r * 65 + s] * p.scale * QK[r * 65 + s] * __expf(gam[r] - gam[s]);
        for (int r2 = r; r2 < 64; ++r2)
            dgam -= dP[r2 * 65 + r] * p.scale * QK[r2 * 65 + r] * __expf(gam[r2] - gam[r]);
        for (int s = 0; s < r; ++s) {
            const float e = __expf(gam[r] - gam[s]) * KK[r * 65 + s];
            dgam += dL[r * 65 + s] * bet[r] * e;
            db += dL[r * 65 + s] * e;
        }
        for (int r2 = r + 1; r2 < 64; ++r2)
            dgam -= dL[r2 * 65 + r] * bet[r2] * __expf(gam[r2] - gam[r]) * KK[r2 * 65 + r];
        dgs[r] = dgam;
        if (r < len) p.dbeta[(size_t)(tok0 + r) * p.Hv + h] = db;
    }
    __syncthreads();
    if (tid == 0) {
        float tot = __expf(gl) * red[0];
        for (int r = 0; r < 64; ++r) tot += __expf(gl - gam[r]) * rowK[r];
        dgs[len - 1] += tot;
        float acc = 0.f;
        for (int r = len - 1; r >= 0; --r) {
            acc += dgs[r];
            p.dg[(size_t)(tok0 + r) * p.Hv + h] = acc;
        }
    }
}

// dq[t, hq] = sum of the per-v-head partials of its group.
template <typename TI>
__global__ void k_group_sum(const float *part, TI *out, long long n, int Hq, int G, int KD) {
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < n;
         idx += (long long)gridDim.x * blockDim.x) {
        const int i = (int)(idx % KD);
        const long long th = idx / KD;  // t * Hq + hq
        const long long t = th / Hq;
        const int hq = (int)(th % Hq);
        float acc = 0.f;
        for (int j = 0; j < G; ++j) acc += part[((t * Hq + hq) * G + j) * KD + i];
        stf(out, (size_t)idx, acc);
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
template <typename KernelT, typename... Args>
cudaError_t launch(const char *name, KernelT kern, dim3 grid, size_t smem, cudaStream_t st, const Params &p,
                   Args... args) {
    if (grid.x == 0 || grid.y == 0 || grid.z == 0) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    tm_begin(p.tm, name, st);
    kern<<<grid, 256, smem, st>>>(p, args...);
    tm_end(p.tm, st);
    return cudaGetLastError();
}

template <int KD, int VD>
constexpr size_t smem_wy() {
    return sizeof(float) * (2 * 64 * ((KD > VD ? KD : VD) + 1) + 2 * 64 * 65 + 128);
}
template <int KD, int VD>
constexpr size_t smem_summary() {
    return sizeof(float) * (KD * 33 + 2 * 64 * (KD + 1) + 64 * 33 + 64);
}
template <int KD, int VD>
constexpr size_t smem_scan() {
    return sizeof(float) * (KD * 33 + 3 * 64 * (KD + 1) + 64 * 65 + 64 * 33 + 64);
}
template <int KD, int VD>
constexpr size_t smem_dh() {
    return sizeof(float) * (KD * 33 + 3 * 64 * (KD + 1) + 64 * 65 + 2 * 64 * 33 + 64);
}
template <int KD, int VD>
constexpr size_t smem_bwd_chunk() {
    return sizeof(float) * (2 * 64 * (KD + 1) + 3 * 64 * 65 + 2 * KD * 17 + 6 * 64 * 17 + 7 * 64 + 8);
}

template <typename TI, typename TO, int KD, int VD>
int fwd_impl(const Params &p, int use_cp, cudaStream_t st) {
    cudaError_t e;
    e = launch("simt_wy", k_wy<TI, KD, VD>, dim3(p.NT, p.Hv), smem_wy<KD, VD>(), st, p, 0);
    if (e != cudaSuccess) return 1;
    if (use_cp) {
        e = launch("simt_cp_summary", k_cp_summary<TI, KD, VD>, dim3(p.NSEG, p.Hv, (VD + KD) / 32),
                   smem_summary<KD, VD>(), st, p);
        if (e != cudaSuccess) return 1;
        e = launch("simt_cp_combine", k_cp_combine<KD, VD, false>, dim3(p.N, p.Hv, VD / kCombCols), smem_combine<KD>(),
                   st, p);
        if (e != cudaSuccess) return 1;
    }
    e = launch("simt_scan", k_scan<TI, TO, KD, VD, true>, dim3(p.NSEG, p.Hv, VD / 32), smem_scan<KD, VD>(), st, p);
    return e != cudaSuccess;
}

template <typename TI, int KD, int VD>
int bwd_impl(const Params &p0, int use_cp, cudaStream_t st) {
    cudaError_t e;
    Params p = p0;
    p.A_out = nullptr;
    e = launch("simt_wy_from_A", k_wy<TI, KD, VD>, dim3(p.NT, p.Hv), smem_wy<KD, VD>(), st, p, 1);
    if (e != cudaSuccess) return 1;
    if (use_cp) {
        e = launch("simt_cp_summary", k_cp_summary<TI, KD, VD>, dim3(p.NSEG, p.Hv, (VD + KD) / 32),
                   smem_summary<KD, VD>(), st, p);
        if (e != cudaSuccess) return 1;
        e = launch("simt_cp_combine", k_cp_combine<KD, VD, false>, dim3(p.N, p.Hv, VD / kCombCols), smem_combine<KD>(),
                   st, p);
        if (e != cudaSuccess) return 1;
    }
    Params ps = p;
    ps.final_state = nullptr;
    e = launch("simt_scan_states", k_scan<TI, float, KD, VD, false>, dim3(p.NSEG, p.Hv, VD / 32),
               smem_scan<KD, VD>(), st, ps);
    if (e != cudaSuccess) return 1;
    e = launch("simt_dh", k_dh<TI, KD, VD>, dim3(p.N, p.Hv, VD / 32), smem_dh<KD, VD>(), st, p);
    if (e != cudaSuccess) return 1;
    e = launch("simt_bwd_chunk", k_bwd_chunk<TI, KD, VD>, dim3(p.NT, p.Hv), smem_bwd_chunk<KD, VD>(), st, p);
    if (e != cudaSuccess) return 1;
    const long long n = (long long)p.Ttot * p.Hq * KD;
    const int G = p.Hv / p.Hq;
    if (n > 0) {
        const int blocks = (int)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
        tm_begin(p.tm, "group_sum_dq", st);
        k_group_sum<TI><<<blocks, 256, 0, st>>>(p.dqp, (TI *)p.dq, n, p.Hq, G, KD);
        tm_end(p.tm, st);
        tm_begin(p.tm, "group_sum_dk", st);
        k_group_sum<TI><<<blocks, 256, 0, st>>>(p.dkp, (TI *)p.dk, n, p.Hq, G, KD);
        tm_end(p.tm, st);
        if (cudaGetLastError() != cudaSuccess) return 1;
    }
    return 0;
}

// Forward and backward for every input / output dtype at one head size.
template <int KD, int VD>
int fwd_sized(const Params &p, int in_f32, int o_f32, int use_cp, cudaStream_t st) {
    if (in_f32)
        return o_f32 ? fwd_impl<float, float, KD, VD>(p, use_cp, st)
                     : fwd_impl<float, __nv_bfloat16, KD, VD>(p, use_cp, st);
    return o_f32 ? fwd_impl<__nv_bfloat16, float, KD, VD>(p, use_cp, st)
                 : fwd_impl<__nv_bfloat16, __nv_bfloat16, KD, VD>(p, use_cp, st);
}
template <int KD, int VD>
int bwd_sized(const Params &p, int in_f32, int use_cp, cudaStream_t st) {
    return in_f32 ? bwd_impl<float, KD, VD>(p, use_cp, st) : bwd_impl<__nv_bfloat16, KD, VD>(p, use_cp, st);
}

unsigned take_status(cudaStream_t st) {
    unsigned v = 0, z = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_simt_status, sizeof(v), 0, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return 0x80000000u;
    cudaMemcpyToSymbolAsync(g_simt_status, &z, sizeof(z), 0, cudaMemcpyHostToDevice, st);
    if (cudaStreamSynchronize(st) != cudaSuccess) return 0x80000000u;
    return v;
}

}  // namespace
}  // namespace gdr
