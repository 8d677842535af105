// gdr_api.cu -- the C ABI of libgdr: argument checks, the context-parallel
// plan, the workspace layout and the dispatch to the kernel paths.
//
// Context parallelism inside one card (FlashQLA pages, page 1 "two fused
// kernels and automatic CP"; page 3 "AutoCP"): a sequence of N chunks is cut
// into segments of L chunks; every segment is summarised from a zero state
// together with its composed transition, the summaries are combined in order,
// and every segment is then re-run from its true start state.  The pages'
// trigger (batch x heads <= 40, or <= 56 with seq_len >= 8192) was fitted to
// a 132-SM Hopper part; here the trigger is the condition it stands for -- the
// scan would otherwise leave SMs idle -- evaluated against this device's SM
// count.  The pages' cost model (steps 2.1 and 3 cost ~L, step 2.2 ~N/L) is
// garbled where it names the optimum; minimising a*L + b*N/L gives
// L* = sqrt(b N / a).  The plan below minimises that cost directly, with the
// per-step costs measured on GB300 and the waves of one-CTA-per-SM scans.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "gdr.h"
#include "gdr_internal.h"

namespace gdr {
int tc_fwd(const Params &p, int o_f32, int use_cp, cudaStream_t st);
int tc_bwd(const Params &p, int use_cp, cudaStream_t st);
int tc_supported(int K, int V);
unsigned tc_take_status(cudaStream_t st);
}  // namespace gdr

namespace {

using namespace gdr;

thread_local char g_err[512];

int fail(int code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

struct Plan {
    int N = 0, NT = 0, NSEG = 0, seg_len = 0, max_nch = 0, use_cp = 0, path = 0;
    long long Ttot = 0;
};

int device_sms() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) {
        cudaGetLastError();
        return 152;
    }
    return sms;
}

int check_shape(const gdr_shape *s) {
    if (!s) return fail(GDR_ERR_ARG, "shape is null");
    if (s->B < 1 || s->T < 1 || s->Hq < 1 || s->Hv < 1)
        return fail(GDR_ERR_SHAPE, "B, T, Hq, Hv must be >= 1 (got %d, %d, %d, %d)", s->B, s->T, s->Hq, s->Hv);
    if (s->Hv % s->Hq) return fail(GDR_ERR_SHAPE, "Hv (%d) must be a multiple of Hq (%d)", s->Hv, s->Hq);
    if ((s->K != 64 && s->K != 128 && s->K != 192) || (s->V != 64 && s->V != 128 && s->V != 192 && s->V != 256))
        return fail(GDR_ERR_SHAPE, "K must be 64, 128 or 192 and V 64, 128, 192 or 256 (got %d, %d)", s->K, s->V);
    if ((long long)s->B * s->T * s->Hv * (long long)std::max(s->K, s->V) >= (1LL << 40))
        return fail(GDR_ERR_SHAPE, "problem too large");
    if (s->n_seqs < 0) return fail(GDR_ERR_SHAPE, "n_seqs must be >= 0");
    if (s->n_seqs > 0) {
        if (s->B != 1) return fail(GDR_ERR_SHAPE, "varlen (n_seqs > 0) needs B == 1 (got %d)", s->B);
        if (!s->cu_seqlens || !s->cu_seqlens_host)
            return fail(GDR_ERR_ARG, "varlen needs both cu_seqlens (device) and cu_seqlens_host");
        const int32_t *cu = s->cu_seqlens_host;
        if (cu[0] != 0) return fail(GDR_ERR_SHAPE, "cu_seqlens[0] must be 0");
        for (int n = 0; n < s->n_seqs; ++n)
            if (cu[n + 1] < cu[n]) return fail(GDR_ERR_SHAPE, "cu_seqlens must be non-decreasing");
        if (cu[s->n_seqs] != s->T) return fail(GDR_ERR_SHAPE, "cu_seqlens[n_seqs] must equal T");
    }
    return GDR_OK;
}

int chunks_of(int len) { return (len + kChunk - 1) / kChunk; }

int make_plan(const gdr_shape *s, const gdr_opts *o, int want_path, int in_f32, Plan *pl) {
    int rc = check_shape(s);
    if (rc) return rc;
    const bool varlen = s->n_seqs > 0;
    pl->N = varlen ? s->n_seqs : s->B;
    pl->Ttot = (long long)s->B * s->T;
    long long nt = 0;
    int maxc = 0;
    for (int n = 0; n < pl->N; ++n) {
        const int len = varlen ? s->cu_seqlens_host[n + 1] - s->cu_seqlens_host[n] : s->T;
        nt += chunks_of(len);
        maxc = std::max(maxc, chunks_of(len));
    }
    if (nt >= (1LL << 31)) return fail(GDR_ERR_SHAPE, "too many chunks");
    pl->NT = (int)nt;
    pl->max_nch = maxc;
    // path
    int path = o ? o->path : GDR_PATH_AUTO;
    if (path == GDR_PATH_AUTO) path = (!in_f32 && tc_supported(s->K, s->V)) ? GDR_PATH_TC : GDR_PATH_SIMT;
    if (path == GDR_PATH_TC && (in_f32 || !tc_supported(s->K, s->V)))
        return fail(GDR_ERR_DTYPE, "the tensor-core path needs bf16 inputs and K = V = 128");
    if (path != GDR_PATH_SIMT && path != GDR_PATH_TC) return fail(GDR_ERR_ARG, "unknown path %d", path);
    (void)want_path;
    pl->path = path;
    // context-parallel plan
    const int forced = o ? o->cp_segments : 0;
    if (forced < 0) return fail(GDR_ERR_ARG, "cp_segments must be >= 0");
    int seg_len = std::max(1, maxc);
    if (forced > 1) {
        seg_len = std::max(1, (maxc + forced - 1) / forced);
    } else if (forced == 0 && maxc > 1 && path == GDR_PATH_TC) {
        // One scan CTA per (segment, v-head), one CTA per SM.  Estimated time in
        // chunk steps of the longest segment: the scan's waves times the segment
        // length (and its warm-up chunks), plus (when split) the summary's waves
        // (two states, each ~0.8 of a scan step) and the sequential combine (~0.7
        // of a step per segment).  With warm-up starts (the rule of
        // warmup_chunks) only the heads whose gates barely decay run the summary:
        // taken as 0.3 of them, since 60-80 % of the heads have a gate that is not
        // identically one (FlashQLA pages, page 1 "two fused kernels and automatic
        // CP", the gate-decay paragraph; a wrong guess costs a few percent either
        // way).
        const long long B = (long long)pl->N * s->Hv, S = device_sms();
        const int req = o ? o->cp_warmup : 0;
        double best = 1e300;
        for (int nseg = 1; nseg <= 64 && nseg <= maxc; ++nseg) {
            const int L = (maxc + nseg - 1) / nseg;
            if (nseg > 1 && L < 4) break;
            const int Wc = nseg == 1 || req < 0 ? 0 : (req > 0 ? req : (L >= 4 * 8 ? 8 : 0));
            const double f = Wc > 0 ? 0.3 : 1.0;
            const double waves = (double)((B * nseg + S - 1) / S);
            double t = waves * (L + Wc);
            if (nseg > 1)
                t += std::ceil(2.0 * f * (double)(B * nseg) / (double)S) * L * 0.8 + 0.7 * nseg;
            if (t < best - 1e-9) {
                best = t;
                seg_len = L;
            }
        }
    } else if (forced == 0 && maxc > 1) {
        // CUDA-core path: 32-column CTAs, two per SM
        const long long base = (long long)pl->N * s->Hv * (s->V / 32);
        const long long target = (long long)device_sms() * 2;
        if (base < target) {
            const long long want = (target + base - 1) / base;
            seg_len = std::max<int>(4, (int)((maxc + want - 1) / want));
            seg_len = std::min(seg_len, maxc);
        }
    }
    long long nseg = 0;
    for (int n = 0; n < pl->N; ++n) {
        const int len = varlen ? s->cu_seqlens_host[n + 1] - s->cu_seqlens_host[n] : s->T;
        nseg += std::max(1, (chunks_of(len) + seg_len - 1) / seg_len);
    }
    pl->seg_len = seg_len;
    pl->NSEG = (int)nseg;
    pl->use_cp = nseg > pl->N;
    return GDR_OK;
}

// Warm-up starts of CP segments (tensor-core path with a split only): option
// 0 -> 8 chunks when segments are at least four windows long (shorter ones
// would scan a large share of extra chunks), -1 -> off, n -> n.
int warmup_chunks(const Plan &pl, const gdr_opts *o) {
    if (!pl.use_cp || pl.path != GDR_PATH_TC) return 0;
    const int req = !o ? 0 : o->cp_warmup;
    return req < 0 ? 0 : req > 0 ? req : (pl.seg_len >= 4 * 8 ? 8 : 0);
}

size_t al(size_t x) { return (x + 255) & ~size_t(255); }

struct Layout {
    size_t seq, chunk, seg, gam, W, U, P, Hseg, Mseg, Nseg, Sstart, hbuf, dhbuf, dubuf, dqp, dkp, warm;
    size_t Aimg, Pimg, Aux, gT, bT;
    bool f32_tiles, bf16_tiles;
    size_t total;
};

Layout layout(const gdr_shape *s, const Plan &pl, bool bwd) {
    Layout L;
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t r = off; off += al(bytes); return r; };
    const size_t NT = pl.NT, Hv = s->Hv, K = s->K, V = s->V, NS = pl.NSEG;
    L.seq = take(sizeof(SeqInfo) * pl.N);
    L.chunk = take(sizeof(ChunkInfo) * NT);
    L.seg = take(sizeof(SegInfo) * NS);
    L.gam = take(4 * NT * Hv * 64);
    // fp32 chunk tiles serve the CUDA-core path; bf16 tile images feed the
    // tensor-core kernels.
    L.f32_tiles = pl.path == GDR_PATH_SIMT;
    L.bf16_tiles = pl.path == GDR_PATH_TC;
    L.W = L.f32_tiles ? take(4 * NT * Hv * 64 * K) : 0;
    L.U = L.f32_tiles ? take(4 * NT * Hv * 64 * V) : 0;
    L.P = L.f32_tiles ? take(4 * NT * Hv * 64 * 64) : 0;
    L.Aimg = L.bf16_tiles ? take((size_t)kTileImgBytes * NT * Hv) : 0;
    L.Pimg = L.bf16_tiles ? take((size_t)kTileImgBytes * NT * Hv) : 0;
    L.Aux = L.bf16_tiles ? take((size_t)kAuxBytes * NT * Hv) : 0;
    L.gT = L.bf16_tiles ? take(4 * NT * Hv * 64) : 0;
    L.bT = L.bf16_tiles ? take(4 * NT * Hv * 64) : 0;
    if (pl.use_cp) {
        L.Hseg = take(4 * NS * Hv * K * V);
        L.Mseg = take(4 * NS * Hv * K * K);
        L.Sstart = take(4 * NS * Hv * K * V);
        L.warm = L.bf16_tiles ? take(4 * (size_t)NS * Hv) : 0;
        L.Nseg = (bwd && L.bf16_tiles) ? take(4 * NS * Hv * K * K) : 0;
    } else {
        L.Hseg = L.Mseg = L.Nseg = L.Sstart = L.warm = 0;
    }
    if (bwd) {
        L.hbuf = take(4 * NT * Hv * K * V);
        L.dhbuf = take(4 * NT * Hv * K * V);
        L.dubuf = take(4 * NT * Hv * 64 * V);
        L.dqp = take(4 * (size_t)pl.Ttot * Hv * K);
        L.dkp = take(4 * (size_t)pl.Ttot * Hv * K);
    } else {
        L.hbuf = L.dhbuf = L.dubuf = L.dqp = L.dkp = 0;
    }
    L.total = off;
    return L;
}

bool misaligned(const void *p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u); }

int check_buf(const char *name, gdr_buf b, bool required) {
    if (!b.ptr) return required ? fail(GDR_ERR_ARG, "%s is null", name) : GDR_OK;
    if (b.dtype != GDR_BF16 && b.dtype != GDR_F32) return fail(GDR_ERR_DTYPE, "%s: unknown dtype %d", name, b.dtype);
    if (misaligned(b.ptr)) return fail(GDR_ERR_ALIGN, "%s is not 16-byte aligned", name);
    return GDR_OK;
}

int check_ptr(const char *name, const void *p, bool required) {
    if (!p) return required ? fail(GDR_ERR_ARG, "%s is null", name) : GDR_OK;
    if (misaligned(p)) return fail(GDR_ERR_ALIGN, "%s is not 16-byte aligned", name);
    return GDR_OK;
}

// --- device tables ---------------------------------------------------------

__global__ void k_prep(const int32_t *cu, int N, int T_fixed, int seg_len, SeqInfo *seq, ChunkInfo *chunk,
                       SegInfo *seg) {
    if (threadIdx.x == 0) {
        int c0 = 0, s0 = 0;
        for (int n = 0; n < N; ++n) {
            const int t0 = cu ? cu[n] : n * T_fixed;
            const int len = cu ? cu[n + 1] - cu[n] : T_fixed;
            const int nch = (len + kChunk - 1) / kChunk;
            const int nseg = max(1, (nch + seg_len - 1) / seg_len);
            SeqInfo si;
            si.tok0 = t0; si.len = len; si.chunk0 = c0; si.nch = nch;
            si.seg0 = s0; si.nseg = nseg; si.pad0 = 0; si.pad1 = 0;
            seq[n] = si;
            c0 += nch;
            s0 += nseg;
        }
    }
    __syncthreads();
    for (int n = 0; n < N; ++n) {
        const SeqInfo si = seq[n];
        for (int l = threadIdx.x; l < si.nch; l += blockDim.x) {
            ChunkInfo ci;
            ci.seq = n; ci.tok0 = si.tok0 + l * kChunk; ci.len = min(kChunk, si.len - l * kChunk); ci.local = l;
            chunk[si.chunk0 + l] = ci;
        }
        for (int j = threadIdx.x; j < si.nseg; j += blockDim.x) {
            SegInfo sg;
            sg.seq = n; sg.chunk0 = si.chunk0 + j * seg_len;
            sg.nch = max(0, min(seg_len, si.nch - j * seg_len)); sg.idx = j;
            seg[si.seg0 + j] = sg;
        }
    }
}

int fill_params(const gdr_shape *s, const Plan &pl, const Layout &L, void *ws, Params *p, const gdr_opts *o) {
    std::memset(p, 0, sizeof(*p));
    char *w = static_cast<char *>(ws);
    p->Ttot = (int)pl.Ttot;
    p->Hq = s->Hq; p->Hv = s->Hv; p->K = s->K; p->V = s->V;
    p->N = pl.N; p->NT = pl.NT; p->NSEG = pl.NSEG;
    p->seq = reinterpret_cast<SeqInfo *>(w + L.seq);
    p->chunk = reinterpret_cast<ChunkInfo *>(w + L.chunk);
    p->seg = reinterpret_cast<SegInfo *>(w + L.seg);
    auto F = [&](size_t off, bool on) { return on ? reinterpret_cast<float *>(w + off) : nullptr; };
    p->gam = F(L.gam, true);
    p->W = F(L.W, L.f32_tiles);
    p->U = F(L.U, L.f32_tiles);
    p->P = F(L.P, L.f32_tiles);
    p->Aimg = F(L.Aimg, L.bf16_tiles);
    p->Pimg = F(L.Pimg, L.bf16_tiles);
    p->Aux = F(L.Aux, L.bf16_tiles);
    p->gT = F(L.gT, L.bf16_tiles);
    p->bT = F(L.bT, L.bf16_tiles);
    p->Hseg = F(L.Hseg, pl.use_cp);
    p->Mseg = F(L.Mseg, pl.use_cp);
    p->Nseg = F(L.Nseg, L.Nseg != 0);
    p->Sstart = F(L.Sstart, pl.use_cp);
    p->hbuf = F(L.hbuf, L.hbuf != 0);
    p->dhbuf = F(L.dhbuf, L.dhbuf != 0);
    p->dubuf = F(L.dubuf, L.dubuf != 0);
    p->dqp = F(L.dqp, L.dqp != 0);
    p->dkp = F(L.dkp, L.dkp != 0);
    p->warm = L.warm ? reinterpret_cast<int *>(w + L.warm) : nullptr;
    p->cp_warmup = p->warm ? warmup_chunks(pl, o) : 0;
    p->debug = o ? o->debug_checks : 0;
    p->timeout_spins = (o && o->timeout_spins > 0) ? o->timeout_spins : (1LL << 22);
    return GDR_OK;
}

int launch_prep(const gdr_shape *s, const Plan &pl, const Params &p, cudaStream_t st) {
    const int32_t *cu = s->n_seqs > 0 ? s->cu_seqlens : nullptr;
    tm_begin(p.tm, "tables", st);
    k_prep<<<1, 256, 0, st>>>(cu, pl.N, s->T, pl.seg_len, const_cast<SeqInfo *>(p.seq),
                             const_cast<ChunkInfo *>(p.chunk), const_cast<SegInfo *>(p.seg));
    tm_end(p.tm, st);
    return cudaGetLastError() == cudaSuccess ? GDR_OK : fail(GDR_ERR_CUDA, "table launch failed");
}

}  // namespace

namespace gdr {
// Records a message for gdr_last_error() on behalf of another translation unit.
int set_last_error(int code, const char *msg) { return fail(code, "%s", msg); }

// The argument checks of gdr_fwd and the workspace that call would need, for
// the plan of the given inputs' own dtype (the path, and so the layout,
// follows the dtype).  Returns gdr_fwd's error code for arguments it would
// reject, with the same message.
int fwd_check_and_size(const gdr_shape *shape, gdr_buf q, gdr_buf k, gdr_buf v, const float *g, const float *beta,
                       const float *h0, gdr_buf o, const float *final_state, const float *A, const float *h,
                       const gdr_opts *opts, size_t *need) {
    g_err[0] = 0;
    int rc;
    if ((rc = check_buf("q", q, true)) || (rc = check_buf("k", k, true)) || (rc = check_buf("v", v, true)) ||
        (rc = check_buf("o", o, true)) || (rc = check_ptr("g", g, true)) || (rc = check_ptr("beta", beta, true)) ||
        (rc = check_ptr("h0", h0, false)) || (rc = check_ptr("final_state", final_state, false)) ||
        (rc = check_ptr("A", A, false)) || (rc = check_ptr("h", h, false)))
        return rc;
    if (q.dtype != k.dtype || q.dtype != v.dtype) return fail(GDR_ERR_DTYPE, "q, k, v must share one dtype");
    Plan pl;
    if ((rc = make_plan(shape, opts, 0, q.dtype == GDR_F32, &pl))) return rc;
    *need = layout(shape, pl, false).total;
    return GDR_OK;
}
}  // namespace gdr

extern "C" {

long long gdr_num_chunks(const gdr_shape *shape) {
    if (check_shape(shape)) return -1;
    long long nt = 0;
    const int N = shape->n_seqs > 0 ? shape->n_seqs : shape->B;
    for (int n = 0; n < N; ++n)
        nt += chunks_of(shape->n_seqs > 0 ? shape->cu_seqlens_host[n + 1] - shape->cu_seqlens_host[n] : shape->T);
    return nt;
}

// The input dtype selects the path under GDR_PATH_AUTO and the path shapes the
// plan, so the size covers both dtypes.
static size_t ws_size(const gdr_shape *shape, const gdr_opts *opts, bool bwd) {
    size_t best = 0;
    bool any = false;
    for (int in_f32 = 0; in_f32 < 2; ++in_f32) {
        Plan pl;
        if (make_plan(shape, opts, 0, in_f32, &pl)) continue;
        best = std::max(best, layout(shape, pl, bwd).total);
        any = true;
    }
    if (any) g_err[0] = 0;
    return best;
}

int gdr_get_plan(const gdr_shape *shape, int in_dtype, const gdr_opts *opts, gdr_plan *out) {
    g_err[0] = 0;
    if (!out) return fail(GDR_ERR_ARG, "out is null");
    if (in_dtype != GDR_BF16 && in_dtype != GDR_F32) return fail(GDR_ERR_DTYPE, "unknown dtype %d", in_dtype);
    Plan pl;
    const int rc = make_plan(shape, opts, 0, in_dtype == GDR_F32, &pl);
    if (rc) return rc;
    out->path = pl.path;
    out->n_chunks = pl.NT;
    out->n_segments = pl.NSEG;
    out->seg_len = pl.seg_len;
    out->cp_warmup = warmup_chunks(pl, opts);
    return GDR_OK;
}

size_t gdr_fwd_workspace_size(const gdr_shape *shape, const gdr_opts *opts) { return ws_size(shape, opts, false); }

size_t gdr_bwd_workspace_size(const gdr_shape *shape, const gdr_opts *opts) { return ws_size(shape, opts, true); }

int gdr_fwd(const gdr_shape *shape, gdr_buf q, gdr_buf k, gdr_buf v, const float *g, const float *beta,
            float scale, const float *h0, gdr_buf o, float *final_state, float *A, float *h, void *workspace,
            size_t workspace_bytes, const gdr_opts *opts, void *stream) {
    g_err[0] = 0;
    int rc;
    if ((rc = check_buf("q", q, true)) || (rc = check_buf("k", k, true)) || (rc = check_buf("v", v, true)) ||
        (rc = check_buf("o", o, true)) || (rc = check_ptr("g", g, true)) || (rc = check_ptr("beta", beta, true)) ||
        (rc = check_ptr("h0", h0, false)) || (rc = check_ptr("final_state", final_state, false)) ||
        (rc = check_ptr("A", A, false)) || (rc = check_ptr("h", h, false)))
        return rc;
    if (q.dtype != k.dtype || q.dtype != v.dtype) return fail(GDR_ERR_DTYPE, "q, k, v must share one dtype");
    const int in_f32 = q.dtype == GDR_F32;
    Plan pl;
    if ((rc = make_plan(shape, opts, 0, in_f32, &pl))) return rc;
    if (!workspace) return fail(GDR_ERR_WORKSPACE, "workspace is null");
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return fail(GDR_ERR_ALIGN, "workspace must be 256-byte aligned");
    const Layout L = layout(shape, pl, false);
    if (workspace_bytes < L.total)
        return fail(GDR_ERR_WORKSPACE, "workspace too small: %zu < %zu bytes", workspace_bytes, L.total);
    Params p;
    fill_params(shape, pl, L, workspace, &p, opts);
    p.q = q.ptr; p.k = k.ptr; p.v = v.ptr; p.g = g; p.beta = beta; p.h0 = h0; p.scale = scale;
    p.o = o.ptr; p.final_state = final_state; p.A_out = A; p.h_out = h;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    Timing tm{opts ? opts->events : nullptr, opts ? opts->names : nullptr, opts ? opts->max_events : 0, 0};
    p.tm = &tm;
    if ((rc = launch_prep(shape, pl, p, st))) return rc;
    const int bad = pl.path == GDR_PATH_TC ? tc_fwd(p, o.dtype == GDR_F32, pl.use_cp, st)
                                           : simt_fwd(p, in_f32, o.dtype == GDR_F32, pl.use_cp, st);
    if (opts && opts->n_launched) *opts->n_launched = tm.count;
    if (bad) return fail(GDR_ERR_CUDA, "forward launch failed: %s", cudaGetErrorString(cudaGetLastError()));
    return GDR_OK;
}

int gdr_bwd(const gdr_shape *shape, gdr_buf q, gdr_buf k, gdr_buf v, const float *g, const float *beta,
            const float *A, gdr_buf do_, const float *dht, float scale, const float *h0, gdr_buf dq, gdr_buf dk,
            gdr_buf dv, float *dbeta, float *dg, float *dh0, void *workspace, size_t workspace_bytes,
            const gdr_opts *opts, void *stream) {
    g_err[0] = 0;
    int rc;
    if ((rc = check_buf("q", q, true)) || (rc = check_buf("k", k, true)) || (rc = check_buf("v", v, true)) ||
        (rc = check_buf("do", do_, true)) || (rc = check_buf("dq", dq, true)) || (rc = check_buf("dk", dk, true)) ||
        (rc = check_buf("dv", dv, true)) || (rc = check_ptr("g", g, true)) || (rc = check_ptr("beta", beta, true)) ||
        (rc = check_ptr("A", A, true)) || (rc = check_ptr("dht", dht, false)) || (rc = check_ptr("h0", h0, false)) ||
        (rc = check_ptr("dbeta", dbeta, true)) || (rc = check_ptr("dg", dg, true)) ||
        (rc = check_ptr("dh0", dh0, false)))
        return rc;
    if (q.dtype != k.dtype || q.dtype != v.dtype || q.dtype != do_.dtype || q.dtype != dq.dtype ||
        q.dtype != dk.dtype || q.dtype != dv.dtype)
        return fail(GDR_ERR_DTYPE, "q, k, v, do, dq, dk, dv must share one dtype");
    const int in_f32 = q.dtype == GDR_F32;
    Plan pl;
    if ((rc = make_plan(shape, opts, 0, in_f32, &pl))) return rc;
    if (!workspace) return fail(GDR_ERR_WORKSPACE, "workspace is null");
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return fail(GDR_ERR_ALIGN, "workspace must be 256-byte aligned");
    const Layout L = layout(shape, pl, true);
    if (workspace_bytes < L.total)
        return fail(GDR_ERR_WORKSPACE, "workspace too small: %zu < %zu bytes", workspace_bytes, L.total);
    Params p;
    fill_params(shape, pl, L, workspace, &p, opts);
    p.q = q.ptr; p.k = k.ptr; p.v = v.ptr; p.g = g; p.beta = beta; p.h0 = h0; p.scale = scale;
    p.A_in = A; p.dout = do_.ptr; p.dht = dht;
    p.dq = dq.ptr; p.dk = dk.ptr; p.dv = dv.ptr; p.dbeta = dbeta; p.dg = dg; p.dh0 = dh0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    Timing tm{opts ? opts->events : nullptr, opts ? opts->names : nullptr, opts ? opts->max_events : 0, 0};
    p.tm = &tm;
    if ((rc = launch_prep(shape, pl, p, st))) return rc;
    const int bad = pl.path == GDR_PATH_TC ? tc_bwd(p, pl.use_cp, st) : simt_bwd(p, in_f32, pl.use_cp, st);
    if (opts && opts->n_launched) *opts->n_launched = tm.count;
    if (bad) return fail(GDR_ERR_CUDA, "backward launch failed: %s", cudaGetErrorString(cudaGetLastError()));
    return GDR_OK;
}

int gdr_check_status(void *stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess)
        return fail(GDR_ERR_CUDA, "stream error: %s", cudaGetErrorString(cudaGetLastError()));
    const unsigned s = simt_take_status(st) | tc_take_status(st);
    if (s & 0x80000000u) return fail(GDR_ERR_CUDA, "could not read the device status word");
    if (s & 1u) return fail(GDR_ERR_TIMEOUT, "a device-side wait ran out of polls");
    if (s & 2u) return fail(GDR_ERR_DEVICE, "a device-side index check failed");
    return GDR_OK;
}

const char *gdr_last_error(void) { return g_err; }

const char *gdr_version(void) { return "gdr 0.1.0 sm_103a"; }

}  // extern "C"
