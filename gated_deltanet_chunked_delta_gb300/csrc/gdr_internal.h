// gdr_internal.h -- host/device shared definitions of libgdr (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace gdr {

constexpr int kChunk = 64;  // tokens per chunk
// Tensor-core path per-(chunk, v-head) workspace records (bytes).
constexpr int kTileImgBytes = 16384;  // one bf16 hi | lo pair of 64x64 images (A, P)
constexpr int kAuxBytes = 768;        // beta, e^gamma, e^{gamma_n - gamma}: 3 x 64 fp32

// Per sequence: token range, chunk range and segment range (context-parallel split).
struct SeqInfo {
    int tok0, len, chunk0, nch;
    int seg0, nseg, pad0, pad1;
};
// Per chunk: owning sequence, first token (flattened), number of tokens, index in sequence.
struct ChunkInfo {
    int seq, tok0, len, local;
};
// Per segment: owning sequence, first global chunk, number of chunks, index in sequence.
struct SegInfo {
    int seq, chunk0, nch, idx;
};

// Caller-owned event brackets around every kernel launch of one call.
struct Timing {
    void **events;
    const char **names;
    int max_events;
    int count;
};

// Records the opening event of a launch named `name` (no-op without timing).
inline void tm_begin(Timing *t, const char *name, cudaStream_t st) {
    if (!t) return;
    const int i = t->count;
    if (t->events && 2 * i + 1 < t->max_events) {
        cudaEventRecord(static_cast<cudaEvent_t>(t->events[2 * i]), st);
        if (t->names) t->names[i] = name;
    }
}
inline void tm_end(Timing *t, cudaStream_t st) {
    if (!t) return;
    const int i = t->count++;
    if (t->events && 2 * i + 1 < t->max_events) cudaEventRecord(static_cast<cudaEvent_t>(t->events[2 * i + 1]), st);
}

// Everything a kernel may need.  Pointers that a launch does not use are null.
struct Params {
    // inputs
    const void *q, *k, *v;  // [Ttot,Hq,K], [Ttot,Hq,K], [Ttot,Hv,V]
    const float *g, *beta;  // [Ttot,Hv]
    const float *h0;        // [N,Hv,K,V] or null
    const float *A_in;      // [Ttot,Hv,64] (backward)
    const void *dout;       // [Ttot,Hv,V] (backward)
    const float *dht;       // [N,Hv,K,V] or null (backward)
    float scale;
    // outputs
    void *o;                // [Ttot,Hv,V]
    float *final_state;     // [N,Hv,K,V] or null
    float *A_out;           // [Ttot,Hv,64] or null
    float *h_out;           // [NT,Hv,K,V] or null
    void *dq, *dk, *dv;     // backward
    float *dbeta, *dg, *dh0;
    // sizes
    int Ttot, Hq, Hv, K, V;
    int N, NT, NSEG;
    // tables (workspace)
    const SeqInfo *seq;
    const ChunkInfo *chunk;
    const SegInfo *seg;
    // workspace arrays
    float *gam;     // [NT,Hv,64]
    float *W;       // [NT,Hv,64,K]
    float *U;       // [NT,Hv,64,V]
    float *P;       // [NT,Hv,64,64]
    float *Hseg;    // [NSEG,Hv,K,V]
    float *Mseg;    // [NSEG,Hv,K,K]
    float *Nseg;    // [NSEG,Hv,K,K] (tensor-core backward): each segment's composed
                    // transition untransposed, i.e. the reverse scan's transposed one
    float *Sstart;  // [NSEG,Hv,K,V]
    float *hbuf;    // [NT,Hv,K,V]   (backward: states before each chunk)
    float *dhbuf;   // [NT,Hv,K,V]   (backward: gradient of the state after each chunk)
    float *dubuf;   // [NT,Hv,64,V]  (backward: gradient of the chunk pseudo-values)
    float *dqp, *dkp;  // [Ttot,Hv,K] per-v-head partial dq, dk
    int cp_warmup;     // warm-up chunks of a segment start (0: the exact split only)
    int *warm;         // [NSEG,Hv] 1: the segment's warm-up start passes its bound (set on the device)
    // tensor-core path chunk tiles (bf16 shared-memory images, hi and lo terms, 16 KiB each)
    void *Aimg;     // [NT,Hv] x A
    void *Pimg;     // [NT,Hv] x P = scale (Q K^T o D o tril_incl), D_rs = e^{gamma_r - gamma_s}
    void *Aux;      // [NT,Hv] x (beta[64], e^gamma[64], e^{gamma_n - gamma}[64]) fp32
    float *gT, *bT; // [NT,Hv,64] the gates and beta as one row of 64 per (chunk, v-head),
                    // zero past the chunk's end (tensor-core path; written first by each call)
    int debug;
    long long timeout_spins;
    Timing *tm;  // host-side only: launch timing (may be null)
};

}  // namespace gdr

// Host-side entry points of each translation unit (called from gdr_api.cu).
namespace gdr {
int simt_fwd(const Params &p, int in_f32, int o_f32, int use_cp, cudaStream_t st);
int simt_bwd(const Params &p, int in_f32, int use_cp, cudaStream_t st);
unsigned simt_take_status(cudaStream_t st);  // every CUDA-core translation unit's status word
int simt_fwd_wide_k(const Params &p, int in_f32, int o_f32, int use_cp, cudaStream_t st);  // K = 192
int simt_bwd_wide_k(const Params &p, int in_f32, int use_cp, cudaStream_t st);
unsigned simt_wide_k_take_status(cudaStream_t st);
int simt_fwd_wide_v(const Params &p, int in_f32, int o_f32, int use_cp, cudaStream_t st);  // V in {192, 256}
int simt_bwd_wide_v(const Params &p, int in_f32, int use_cp, cudaStream_t st);
unsigned simt_wide_v_take_status(cudaStream_t st);
}  // namespace gdr
