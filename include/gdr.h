/*
 * gdr.h -- C ABI of libgdr: Gated DeltaNet (GDN) chunked prefill, forward and
 * backward, on one NVIDIA GB300 (sm_103a).
 *
 * The operation (FlashQLA pages; problem statement of the GDN chunked-prefill
 * kernels): for every sequence n and value head h, with qk-head
 * hq = h / (Hv / Hq) (grouped heads, page 1 high-level API shapes),
 *
 *     S_t = a_t (I - b_t k_t k_t^T) S_{t-1} + b_t k_t v_t^T,   a_t = exp(g_t),
 *     o_t = scale * S_t^T q_t,          S_0 = h0[n, h] (zeros when absent),
 *
 * evaluated chunk by chunk with 64-token chunks.  The calls mirror the
 * low-level entry points of page 1 ("usage and requirements"):
 *     forward  (q, k, v, g, beta, scale, h0, cu_seqlens) -> (o, final_state, A, h)
 *     backward (q, k, v, g, beta, A, do, dht, scale, h0, cu_seqlens)
 *                                                   -> (dq, dk, dv, dbeta, dg, dh0)
 * The cumulated gate g that the Python forward of the pages also returns is
 * not exported; the backward recomputes it from the raw g.
 *
 * Conventions shared by every call
 * --------------------------------
 * Layouts: row-major, innermost dimension last, contiguous, no padding:
 *   q, k, dq, dk        [B, T, Hq, K]
 *   v, o, do, dv        [B, T, Hv, V]
 *   g, beta, dg, dbeta  [B, T, Hv]          (fp32)
 *   A                   [B, T, Hv, 64]      (fp32; row r of its chunk's A at token r)
 *   h                   [NT, Hv, K, V]      (fp32; h[i] = state before chunk i)
 *   h0, final_state, dht, dh0   [N, Hv, K, V]   (fp32)
 * N = B for a fixed-length batch; for varlen (n_seqs > 0) B must be 1, the
 * sequences are packed along T and N = n_seqs.  Chunks restart at every
 * sequence start; NT (gdr_num_chunks) counts chunks over all sequences in order.
 * g is the per-token log-gate (<= 0 in the intended use: a_t in (0, 1]);
 * beta is the write strength as passed (already squashed by the caller).
 *
 * Sizes: K in {64, 128, 192}, V in {64, 128, 192, 256}; Hq >= 1; Hv a
 * multiple of Hq; T >= 1.  The tensor-core path takes bf16 inputs with
 * K = V = 128; every other size and fp32 inputs run on the CUDA cores.
 * Varlen sequences may have length 0 (their final state is h0).
 *
 * Ownership: the caller allocates every buffer, including the workspace
 * (sized by gdr_*_workspace_size).  The library allocates nothing, keeps no
 * state between calls and never writes its inputs.
 *
 * Execution: every call only enqueues work on `stream` (a cudaStream_t; NULL
 * is the legacy default stream) and returns; nothing synchronises.  Buffers
 * must stay valid until that work completes.  Calls on one workspace must not
 * overlap in time.
 *
 * Errors: every call returns GDR_OK (0) or one of the codes below; on an
 * argument error nothing is launched.  gdr_last_error() gives a message for
 * the calling thread's last failure.  Device-side problems (a bounded wait
 * that ran out, a violated index check in debug mode) are recorded in a device
 * status word and reported by gdr_check_status().
 */
#ifndef GDR_H
#define GDR_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define GDR_API __attribute__((visibility("default")))
#else
#define GDR_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* element types of gdr_buf */
#define GDR_BF16 0
#define GDR_F32 1

/* return codes */
#define GDR_OK 0
#define GDR_ERR_ARG 1       /* null or invalid argument */
#define GDR_ERR_SHAPE 2     /* unsupported sizes: K, V outside the sets above, Hv % Hq != 0, ... */
#define GDR_ERR_DTYPE 3     /* unsupported or mismatched element type */
#define GDR_ERR_ALIGN 4     /* a pointer not 16-byte aligned */
#define GDR_ERR_WORKSPACE 5 /* workspace missing or too small */
#define GDR_ERR_CUDA 6      /* a CUDA runtime call or launch failed */
#define GDR_ERR_TIMEOUT 7   /* a device-side bounded wait ran out (from gdr_check_status) */
#define GDR_ERR_DEVICE 8    /* a device-side index check failed (debug_checks) */

/* paths (gdr_opts.path) */
#define GDR_PATH_AUTO 0     /* tensor-core path where supported, else the CUDA-core path */
#define GDR_PATH_SIMT 1     /* fp32 CUDA-core kernels (any dtype, K,V in {64,128}) */
#define GDR_PATH_TC 2       /* tcgen05 tensor-core kernels (bf16, K = V = 128) */

/* A device buffer and its element type (GDR_BF16 or GDR_F32). */
typedef struct {
    void *ptr;
    int dtype;
} gdr_buf;

/* Problem sizes. */
typedef struct {
    int B, T, Hq, Hv, K, V;
    int n_seqs;                      /* 0: fixed-length batch; > 0: varlen, B must be 1 */
    const int32_t *cu_seqlens;       /* varlen: device array [n_seqs + 1], 0 .. T */
    const int32_t *cu_seqlens_host;  /* varlen: host copy of the same values */
} gdr_shape;

/* Options.  A zeroed struct (or NULL) selects every default. */
typedef struct {
    int cp_segments;        /* intra-card context parallelism: 0 auto, 1 off,
                               n > 1 = split the longest sequence into n segments */
    int path;               /* GDR_PATH_* */
    int debug_checks;       /* 1: kernels check every index against its extent */
    long long timeout_spins;/* cap on device-side barrier polls (0: default) */
    /* Optional per-kernel timing with caller-owned CUDA events (cudaEvent_t,
     * created by the caller).  When `events` is not NULL the call records
     * events[2i] on `stream` just before its i-th kernel launch and
     * events[2i+1] just after it, for i < max_events / 2, and stores a static
     * name of that kernel in names[i] (names may be NULL).  n_launched (may be
     * NULL) receives the number of kernels the call launched. */
    void **events;
    const char **names;
    int max_events;
    int *n_launched;
    /* Warm-up starts of context-parallel segments (FlashQLA pages: page 1,
     * "balanced solution", and page 3, "sliding-window warmup": a segment's
     * start state is approximated by scanning the few chunks before it from
     * zero).  Here it replaces the exact summary and combine for a v-head only
     * when, for every segment of every sequence, the bound on the start
     * state's error, prod_t a_t max(1, |1 - b_t |k_t|^2|) over the warm-up
     * window, is below 1e-6 (or the window reaches the sequence start, where
     * the warm-up is exact).  0 (default): 8 warm-up chunks where the plan's
     * segments are at least 32 chunks long, else the exact split; -1: always
     * the exact split; n > 0: n warm-up chunks.  Tensor-core path, forward and
     * the backward's state recompute; the reverse scan is always exact. */
    int cp_warmup;
} gdr_opts;

/* Number of 64-token chunks over all sequences (the NT of h).  -1 on bad shape. */
GDR_API long long gdr_num_chunks(const gdr_shape *shape);

/* How a call with these sizes, input dtype and options would run.  The
 * intra-card context-parallel split follows the pages' cost reasoning (page 1,
 * "two fused kernels and automatic CP": the per-segment steps cost about the
 * segment length, the combine about the number of segments), re-fitted to the
 * SM count of the current device (152 when no device is visible). */
typedef struct {
    int path;             /* GDR_PATH_SIMT or GDR_PATH_TC */
    long long n_chunks;   /* as gdr_num_chunks */
    int n_segments;       /* segments over all sequences; equal to the number of
                             sequences when no sequence is split */
    int seg_len;          /* chunks per segment (a sequence's last may be shorter) */
    int cp_warmup;        /* warm-up chunks at segment starts (0: exact split only) */
} gdr_plan;

/* Fills *out for a forward or backward call with inputs of element type
 * `in_dtype` (GDR_BF16 or GDR_F32).  Host-side only: touches no device memory
 * and launches nothing.  Returns GDR_OK or the error gdr_fwd would return for
 * these sizes, dtype and options. */
GDR_API int gdr_get_plan(const gdr_shape *shape, int in_dtype, const gdr_opts *opts, gdr_plan *out);

/* Workspace bytes needed by gdr_fwd / gdr_bwd for this shape and options.
 * Returns 0 and sets the last error on an invalid shape. */
GDR_API size_t gdr_fwd_workspace_size(const gdr_shape *shape, const gdr_opts *opts);
GDR_API size_t gdr_bwd_workspace_size(const gdr_shape *shape, const gdr_opts *opts);

/*
 * Forward.  Inputs: q, k, v (same dtype, GDR_BF16 or GDR_F32), g, beta (fp32),
 * scale, h0 (nullable: zero initial state).  Outputs: o (GDR_BF16 or GDR_F32,
 * independent of the input dtype), final_state (nullable), A (nullable; needed
 * later by gdr_bwd), h (nullable).  `workspace` must be 256-byte aligned and
 * hold gdr_fwd_workspace_size() bytes.
 */
GDR_API int gdr_fwd(const gdr_shape *shape, gdr_buf q, gdr_buf k, gdr_buf v, const float *g,
            const float *beta, float scale, const float *h0, gdr_buf o, float *final_state,
            float *A, float *h, void *workspace, size_t workspace_bytes, const gdr_opts *opts,
            void *stream);

/*
 * Backward of gdr_fwd's (o, final_state) with respect to (q, k, v, beta, g, h0).
 * Inputs: the forward's inputs, A as written by gdr_fwd, do (dtype of q),
 * dht (nullable: zero gradient of final_state), h0 (nullable).  Outputs:
 * dq, dk, dv (dtype of q), dbeta, dg (fp32), dh0 (nullable).
 * dbeta is the gradient with respect to beta as passed; dg with respect to
 * the raw per-token log-gate g.
 */
GDR_API int gdr_bwd(const gdr_shape *shape, gdr_buf q, gdr_buf k, gdr_buf v, const float *g,
            const float *beta, const float *A, gdr_buf do_, const float *dht, float scale,
            const float *h0, gdr_buf dq, gdr_buf dk, gdr_buf dv, float *dbeta, float *dg,
            float *dh0, void *workspace, size_t workspace_bytes, const gdr_opts *opts,
            void *stream);

/*
 * gdr_fwd without a workspace, for callers that cannot allocate device memory
 * (a plugin inside a host program that owns all device memory and offers no
 * allocator, or a path that must not call cudaMalloc because it may
 * synchronise the device).  The pages have no counterpart; this is a library
 * convenience.  Arguments and results are those of gdr_fwd, minus the
 * workspace: the call uses a fixed 64 MiB array compiled into the library,
 * which every GPU that loads the library keeps until the process exits.
 * Problems whose forward workspace, for the plan of the inputs' own dtype,
 * exceeds 64 MiB are rejected with GDR_ERR_WORKSPACE before anything is
 * launched; invalid arguments get gdr_fwd's error codes.  The first call on
 * each device looks the array's device address up (cudaGetSymbolAddress) and
 * keeps it for the life of the process; make that first call before any
 * stream capture, and make no call on a device after a cudaDeviceReset() of
 * it (the kept address is then stale).  All calls share the one array: calls
 * whose work overlaps on the GPU (different streams, or another thread) race
 * and corrupt each other's results, so serialise them.  Nothing carried over
 * from an earlier call is read.  The call itself allocates nothing.
 */
GDR_API int gdr_fwd_noalloc(const gdr_shape *shape, gdr_buf q, gdr_buf k, gdr_buf v, const float *g,
                            const float *beta, float scale, const float *h0, gdr_buf o, float *final_state,
                            float *A, float *h, const gdr_opts *opts, void *stream);

/* Synchronises `stream`, then reads and clears the device status word:
 * GDR_OK, GDR_ERR_TIMEOUT, GDR_ERR_DEVICE, or GDR_ERR_CUDA. */
GDR_API int gdr_check_status(void *stream);

/* Message of the calling thread's last failure ("" if none). */
GDR_API const char *gdr_last_error(void);

/* Library version, e.g. "gdr 0.1.0 sm_103a". */
GDR_API const char *gdr_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDR_H */
