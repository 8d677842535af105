/*
 * gdr_oracle.c -- plain fp64 CPU oracle for the Gated DeltaNet (GDN) recurrence.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library and
 * its Python binding) links, loads or calls this file; only the tests, the
 * smoke check and the CPU-baseline leg of the benchmark do.  It shares no code,
 * header, table or helper with the CUDA path.
 *
 * What it follows (FlashQLA pages, "GDN Chunked Prefill" problem statement):
 *   - the gated delta rule, token by token:
 *         S_t = a_t (I - b_t k_t k_t^T) S_{t-1} + b_t k_t v_t^T,   a_t = exp(g_t)
 *         o_t = scale * S_t^T q_t          (the state AFTER token t is used)
 *     The pages describe GDN as linear attention whose history is carried by an
 *     exponentially decaying gate (page 2, "what it solves"; page 1, "balanced
 *     solution" paragraph on the gate's sliding-window property).  The formula
 *     itself is the problem statement of the low-level forward entry point.
 *   - the low-level API of page 1 ("usage and requirements"): forward returns
 *     (g, A, o, h, final_state); backward returns (dq, dk, dv, db, dg, dh0).
 *   - varlen packing through cu_seqlens (page 1 usage; page 3 "main features").
 *
 * Readings taken where the pages are silent:
 *   - GQA mapping: v-head h reads qk-head h / (Hv/Hq).
 *   - A is the unit-lower-triangular inverse (I + L)^-1 with
 *     L_rs = b_r exp(gamma_r - gamma_s) (k_r . k_s) for s < r inside one chunk,
 *     gamma the chunk-local inclusive cumsum of g.  Strictly lower: a chunk of
 *     one token gives A = I.
 *   - h[i] is the state before the first token of chunk i; chunks restart at
 *     each sequence start; i counts chunks over all sequences in order.
 *
 * Layouts (all row-major, innermost last), over a flattened token axis of
 * length Ttot = cu[n_seqs]:
 *   q, k [Ttot, Hq, K];  v, o [Ttot, Hv, V];  g, beta [Ttot, Hv];
 *   h0, final [n_seqs, Hv, K, V];  hchunks [NTtot, Hv, K, V];  A [Ttot, Hv, C].
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* Planted-mistake switch for the oracle's own self-test: the tests rebuild this
 * file with -DGDR_ORACLE_MUTATION=n to check that the pins catch a dropped
 * term, a wrong index or a stale state.  0 (the default) is the oracle. */
#ifndef GDR_ORACLE_MUTATION
#define GDR_ORACLE_MUTATION 0
#endif
#define MUT(n) (GDR_ORACLE_MUTATION == (n))

typedef struct {
    int n_seqs;
    const int *cu;
    int Hq, Hv, K, V, C;
    const double *q, *k, *v, *g, *beta;
    double scale;
    const double *h0;
    const double *dout, *dht;
    double *o, *final_state, *hchunks, *A;
    double *dq_part, *dk_part, *dv, *dbeta, *dg, *dh0;
    int *chunk_off; /* [n_seqs + 1] */
} problem;

static int n_chunks(int len, int C) { return (len + C - 1) / C; }

static void fill_chunk_off(problem *p) {
    p->chunk_off[0] = 0;
    for (int n = 0; n < p->n_seqs; ++n)
        p->chunk_off[n + 1] = p->chunk_off[n] + n_chunks(p->cu[n + 1] - p->cu[n], p->C);
}

/* ------------------------------------------------------------------------- */
/* Work distribution: a shared counter over independent jobs.                 */
/* ------------------------------------------------------------------------- */
typedef struct {
    problem *p;
    int n_jobs;
    int next;
    int vblock;
    pthread_mutex_t mu;
    void (*run)(problem *, int job, int vblock);
} pool;

static void *pool_worker(void *arg) {
    pool *w = (pool *)arg;
    for (;;) {
        pthread_mutex_lock(&w->mu);
        int j = w->next++;
        pthread_mutex_unlock(&w->mu);
        if (j >= w->n_jobs) break;
        w->run(w->p, j, w->vblock);
    }
    return NULL;
}

static void run_pool(problem *p, int n_jobs, int vblock, int nthreads,
                     void (*run)(problem *, int, int)) {
    pool w;
    w.p = p; w.n_jobs = n_jobs; w.next = 0; w.vblock = vblock; w.run = run;
    pthread_mutex_init(&w.mu, NULL);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > n_jobs) nthreads = n_jobs > 0 ? n_jobs : 1;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    for (int i = 0; i < nthreads; ++i) pthread_create(&th[i], NULL, pool_worker, &w);
    for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&w.mu);
}

/* ------------------------------------------------------------------------- */
/* Forward: the token recurrence.  The V columns of S evolve independently    */
/* (every step acts on S from the left or adds a rank-1 term whose column     */
/* factor is that column's own d_t), so one job owns columns [c0, c1) of one  */
/* (sequence, v-head).                                                        */
/* ------------------------------------------------------------------------- */
static void fwd_job(problem *p, int job, int vblock) {
    const int nvb = (p->V + vblock - 1) / vblock;
    const int vb = job % nvb;
    const int h = (job / nvb) % p->Hv;
    const int n = job / (nvb * p->Hv);
    const int c0 = vb * vblock;
    const int c1 = c0 + vblock < p->V ? c0 + vblock : p->V;
    const int nc = c1 - c0;
    const int K = p->K, V = p->V, Hv = p->Hv, Hq = p->Hq;
    const int hq = MUT(4) ? h % Hq : h / (Hv / Hq);
    double *S = (double *)calloc((size_t)K * nc, sizeof(double));
    double *d = (double *)malloc(sizeof(double) * (size_t)nc);
    if (p->h0)
        for (int i = 0; i < K; ++i)
            for (int j = 0; j < nc; ++j)
                S[i * nc + j] = p->h0[(((size_t)n * Hv + h) * K + i) * V + c0 + j];
    const int t0 = p->cu[n], t1 = p->cu[n + 1];
    for (int t = t0; t < t1; ++t) {
        const int r = t - t0;
        if (p->hchunks && r % p->C == 0) {
            const size_t ci = (size_t)p->chunk_off[n] + r / p->C;
            for (int i = 0; i < K; ++i)
                for (int j = 0; j < nc; ++j)
                    p->hchunks[((ci * Hv + h) * K + i) * V + c0 + j] = S[i * nc + j];
        }
        const double a = exp(p->g[(size_t)t * Hv + h]);
        const double b = p->beta[(size_t)t * Hv + h];
        const double *kt = p->k + ((size_t)t * Hq + hq) * K;
        const double *qt = p->q + ((size_t)t * Hq + hq) * K;
        const double *vt = p->v + ((size_t)t * Hv + h) * V + c0;
        /* d = v - (a S)^T k */
        for (int j = 0; j < nc; ++j) {
            double pk = 0.0;
            for (int i = 0; i < K; ++i) pk += S[i * nc + j] * kt[i];
            d[j] = vt[j] - (MUT(1) ? 1.0 : a) * pk;
        }
        if (MUT(2)) {
            double *ot2 = p->o + ((size_t)t * Hv + h) * V + c0;
            for (int j = 0; j < nc; ++j) {
                double acc = 0.0;
                for (int i = 0; i < K; ++i) acc += S[i * nc + j] * qt[i];
                ot2[j] = p->scale * acc;
            }
        }
        /* S = a S + b k d^T */
        for (int i = 0; i < K; ++i)
            for (int j = 0; j < nc; ++j)
                S[i * nc + j] = a * S[i * nc + j] + b * kt[i] * d[j];
        /* o = scale S^T q */
        double *ot = p->o + ((size_t)t * Hv + h) * V + c0;
        for (int j = 0; j < nc && !MUT(2); ++j) {
            double acc = 0.0;
            for (int i = 0; i < K; ++i) acc += S[i * nc + j] * qt[i];
            ot[j] = p->scale * acc;
        }
    }
    if (p->final_state)
        for (int i = 0; i < K; ++i)
            for (int j = 0; j < nc; ++j)
                p->final_state[(((size_t)n * Hv + h) * K + i) * V + c0 + j] = S[i * nc + j];
    free(S);
    free(d);
}

/* ------------------------------------------------------------------------- */
/* A by its definition, one (sequence, v-head) per job.                       */
/*   gamma_r = sum_{s<=r} g_s inside the chunk,                               */
/*   L_rs    = b_r exp(gamma_r - gamma_s) (k_r . k_s)   for s < r,            */
/*   A       = (I + L)^-1 by forward substitution on the columns of I:        */
/*             A_rc = [r==c] - sum_{c<=s<r} L_rs A_sc.                        */
/* Entries of a partial chunk outside its n x n block are zero.              */
/* ------------------------------------------------------------------------- */
static void a_job(problem *p, int job, int unused) {
    (void)unused;
    const int h = job % p->Hv, n = job / p->Hv;
    const int C = p->C, K = p->K, Hv = p->Hv, Hq = p->Hq;
    const int hq = h / (Hv / Hq);
    double *gam = (double *)malloc(sizeof(double) * (size_t)C);
    double *L = (double *)malloc(sizeof(double) * (size_t)C * C);
    double *X = (double *)malloc(sizeof(double) * (size_t)C * C);
    const int t0 = p->cu[n], t1 = p->cu[n + 1];
    for (int cs = t0; cs < t1; cs += C) {
        const int len = (t1 - cs) < C ? (t1 - cs) : C;
        double acc = 0.0;
        for (int r = 0; r < len; ++r) {
            acc += p->g[(size_t)(cs + r) * Hv + h];
            gam[r] = acc;
        }
        for (int r = 0; r < len; ++r) {
            const double br = p->beta[(size_t)(cs + r) * Hv + h];
            const double *kr = p->k + ((size_t)(cs + r) * Hq + hq) * K;
            for (int s = 0; s < len; ++s) {
                double val = 0.0;
                if (s < r || (MUT(5) && s == r)) {
                    const double *ks = p->k + ((size_t)(cs + s) * Hq + hq) * K;
                    double dot = 0.0;
                    for (int i = 0; i < K; ++i) dot += kr[i] * ks[i];
                    val = br * exp(gam[r] - gam[s]) * dot;
                }
                L[r * C + s] = val;
            }
        }
        for (int c = 0; c < len; ++c) {
            for (int r = 0; r < len; ++r) {
                if (r < c) { X[r * C + c] = 0.0; continue; }
                double val = (r == c) ? 1.0 : 0.0;
                for (int s = c; s < r; ++s) val -= L[r * C + s] * X[s * C + c];
                X[r * C + c] = MUT(5) ? val / (1.0 + L[r * C + r]) : val;
            }
        }
        for (int r = 0; r < len; ++r)
            for (int c = 0; c < C; ++c)
                p->A[((size_t)(cs + r) * Hv + h) * C + c] = (c < len) ? X[r * C + c] : 0.0;
    }
    free(gam);
    free(L);
    free(X);
}

/* ------------------------------------------------------------------------- */
/* Backward: reverse mode of the token recurrence, one (sequence, v-head) per */
/* job.  For each token, in reverse:                                          */
/*   dS += scale q do^T ;   dq += scale S_t do                                */
/*   P = a S_{t-1};  d = v - P^T k                                            */
/*   dbeta = k^T dS d ;  dk += b dS d ;  dd = b dS^T k                        */
/*   dv = dd ;  dP = dS - k dd^T ;  dk -= P dd                                */
/*   dg = a <dP, S_{t-1}>_F ;  dS = a dP                                      */
/* States S_{t-1} come from fp64 checkpoints at every chunk start and are     */
/* recomputed forward inside each chunk.  dq, dk are written per v-head and   */
/* summed over the group afterwards.                                          */
/* ------------------------------------------------------------------------- */
static void forward_step(const problem *p, int t, int h, int hq, const double *Sin, double *Sout,
                         double *d) {
    const int K = p->K, V = p->V, Hv = p->Hv, Hq = p->Hq;
    const double a = exp(p->g[(size_t)t * Hv + h]);
    const double b = p->beta[(size_t)t * Hv + h];
    const double *kt = p->k + ((size_t)t * Hq + hq) * K;
    const double *vt = p->v + ((size_t)t * Hv + h) * V;
    for (int j = 0; j < V; ++j) {
        double pk = 0.0;
        for (int i = 0; i < K; ++i) pk += Sin[i * V + j] * kt[i];
        d[j] = vt[j] - a * pk;
    }
    for (int i = 0; i < K; ++i)
        for (int j = 0; j < V; ++j) Sout[i * V + j] = a * Sin[i * V + j] + b * kt[i] * d[j];
}

static void bwd_job(problem *p, int job, int unused) {
    (void)unused;
    const int h = job % p->Hv, n = job / p->Hv;
    const int C = p->C, K = p->K, V = p->V, Hv = p->Hv, Hq = p->Hq;
    const int hq = MUT(4) ? h % Hq : h / (Hv / Hq);
    const size_t KV = (size_t)K * V;
    const int t0 = p->cu[n], t1 = p->cu[n + 1];
    const int nch = n_chunks(t1 - t0, C);
    double *ckpt = (double *)malloc(sizeof(double) * KV * (size_t)(nch > 0 ? nch : 1));
    double *states = (double *)malloc(sizeof(double) * KV * (size_t)(C + 1));
    double *dS = (double *)malloc(sizeof(double) * KV);
    double *dP = (double *)malloc(sizeof(double) * KV);
    double *d = (double *)malloc(sizeof(double) * (size_t)V);
    double *dd = (double *)malloc(sizeof(double) * (size_t)V);
    double *dSd = (double *)malloc(sizeof(double) * (size_t)K);
    double *Pdd = (double *)malloc(sizeof(double) * (size_t)K);

    /* forward pass: checkpoints at chunk starts */
    double *S = states, *S2 = states + KV;
    for (size_t e = 0; e < KV; ++e)
        S[e] = p->h0 ? p->h0[((size_t)n * Hv + h) * KV + e] : 0.0;
    for (int c = 0; c < nch; ++c) {
        memcpy(ckpt + (size_t)c * KV, S, sizeof(double) * KV);
        const int te = (t0 + (c + 1) * C) < t1 ? (t0 + (c + 1) * C) : t1;
        for (int t = t0 + c * C; t < te; ++t) {
            forward_step(p, t, h, hq, S, S2, d);
            memcpy(S, S2, sizeof(double) * KV);
        }
    }

    for (size_t e = 0; e < KV; ++e)
        dS[e] = p->dht ? p->dht[((size_t)n * Hv + h) * KV + e] : 0.0;

    for (int c = nch - 1; c >= 0; --c) {
        const int ts = t0 + c * C;
        const int te = (ts + C) < t1 ? (ts + C) : t1;
        const int len = te - ts;
        memcpy(states, ckpt + (size_t)c * KV, sizeof(double) * KV);
        for (int r = 0; r < len; ++r)
            forward_step(p, ts + r, h, hq, states + (size_t)r * KV, states + (size_t)(r + 1) * KV, d);
        for (int r = len - 1; r >= 0; --r) {
            const int t = ts + r;
            const double *Sprev = states + (size_t)r * KV;
            const double *St = states + (size_t)(r + 1) * KV;
            const double a = exp(p->g[(size_t)t * Hv + h]);
            const double b = p->beta[(size_t)t * Hv + h];
            const double *kt = p->k + ((size_t)t * Hq + hq) * K;
            const double *qt = p->q + ((size_t)t * Hq + hq) * K;
            const double *vt = p->v + ((size_t)t * Hv + h) * V;
            const double *dot = p->dout + ((size_t)t * Hv + h) * V;
            double *dqt = p->dq_part + ((size_t)t * Hv + h) * K;
            double *dkt = p->dk_part + ((size_t)t * Hv + h) * K;
            double *dvt = p->dv + ((size_t)t * Hv + h) * V;
            /* o = scale S_t^T q */
            for (int i = 0; i < K; ++i) {
                double acc = 0.0;
                for (int j = 0; j < V; ++j) {
                    dS[i * V + j] += p->scale * qt[i] * dot[j];
                    acc += St[i * V + j] * dot[j];
                }
                dqt[i] = p->scale * acc;
            }
            /* recompute d = v - a S_{t-1}^T k */
            for (int j = 0; j < V; ++j) {
                double pk = 0.0;
                for (int i = 0; i < K; ++i) pk += Sprev[i * V + j] * kt[i];
                d[j] = vt[j] - a * pk;
            }
            /* S_t = P + b k d^T */
            double dbeta = 0.0;
            for (int i = 0; i < K; ++i) {
                double acc = 0.0;
                for (int j = 0; j < V; ++j) acc += dS[i * V + j] * d[j];
                dSd[i] = acc;
                dbeta += kt[i] * acc;
            }
            for (int j = 0; j < V; ++j) {
                double acc = 0.0;
                for (int i = 0; i < K; ++i) acc += dS[i * V + j] * kt[i];
                dd[j] = b * acc;
                dvt[j] = dd[j];
            }
            /* d = v - P^T k with P = a S_{t-1} */
            for (int i = 0; i < K; ++i) {
                double acc = 0.0;
                for (int j = 0; j < V; ++j) acc += a * Sprev[i * V + j] * dd[j];
                Pdd[i] = acc;
            }
            for (int i = 0; i < K; ++i) dkt[i] = b * dSd[i] + (MUT(6) ? 1.0 : -1.0) * Pdd[i];
            double dalpha = 0.0;
            for (int i = 0; i < K; ++i)
                for (int j = 0; j < V; ++j) {
                    const double v_dP = dS[i * V + j] - kt[i] * dd[j];
                    dP[i * V + j] = v_dP;
                    dalpha += v_dP * Sprev[i * V + j];
                }
            p->dbeta[(size_t)t * Hv + h] = dbeta;
            p->dg[(size_t)t * Hv + h] = (MUT(3) ? 1.0 : a) * dalpha;
            for (size_t e = 0; e < KV; ++e) dS[e] = a * dP[e];
        }
    }
    if (p->dh0)
        for (size_t e = 0; e < KV; ++e) p->dh0[((size_t)n * Hv + h) * KV + e] = dS[e];
    free(ckpt); free(states); free(dS); free(dP); free(d); free(dd); free(dSd); free(Pdd);
}

/* ------------------------------------------------------------------------- */
/* Exported entry points (called through ctypes from oracle/__init__.py).     */
/* Return 0 on success, 1 on an argument error.                               */
/* ------------------------------------------------------------------------- */
static int check_args(int n_seqs, const int *cu, int Hq, int Hv, int K, int V, int C) {
    if (n_seqs < 1 || !cu || Hq < 1 || Hv < 1 || K < 1 || V < 1 || C < 1) return 1;
    if (Hv % Hq) return 1;
    if (cu[0] != 0) return 1;
    for (int n = 0; n < n_seqs; ++n)
        if (cu[n + 1] < cu[n]) return 1;
    return 0;
}

int gdr_oracle_fwd(int n_seqs, const int *cu, int Hq, int Hv, int K, int V, int C,
                   const double *q, const double *k, const double *v, const double *g,
                   const double *beta, double scale, const double *h0, double *o,
                   double *final_state, double *hchunks, int nthreads, int vblock) {
    if (check_args(n_seqs, cu, Hq, Hv, K, V, C) || !o) return 1;
    if (vblock < 1 || vblock > V) vblock = V;
    problem p;
    memset(&p, 0, sizeof(p));
    p.n_seqs = n_seqs; p.cu = cu; p.Hq = Hq; p.Hv = Hv; p.K = K; p.V = V; p.C = C;
    p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta; p.scale = scale; p.h0 = h0;
    p.o = o; p.final_state = final_state; p.hchunks = hchunks;
    p.chunk_off = (int *)malloc(sizeof(int) * (size_t)(n_seqs + 1));
    fill_chunk_off(&p);
    const int nvb = (V + vblock - 1) / vblock;
    run_pool(&p, n_seqs * Hv * nvb, vblock, nthreads, fwd_job);
    free(p.chunk_off);
    return 0;
}

int gdr_oracle_A(int n_seqs, const int *cu, int Hq, int Hv, int K, int C, const double *k,
                 const double *g, const double *beta, double *A, int nthreads) {
    if (check_args(n_seqs, cu, Hq, Hv, K, 1, C) || !A) return 1;
    problem p;
    memset(&p, 0, sizeof(p));
    p.n_seqs = n_seqs; p.cu = cu; p.Hq = Hq; p.Hv = Hv; p.K = K; p.V = 1; p.C = C;
    p.k = k; p.g = g; p.beta = beta; p.A = A;
    run_pool(&p, n_seqs * Hv, 1, nthreads, a_job);
    return 0;
}

int gdr_oracle_bwd(int n_seqs, const int *cu, int Hq, int Hv, int K, int V, const double *q,
                   const double *k, const double *v, const double *g, const double *beta,
                   double scale, const double *h0, const double *dout, const double *dht,
                   double *dq, double *dk, double *dv, double *dbeta, double *dg, double *dh0,
                   int nthreads, int ckpt) {
    if (ckpt < 1) ckpt = 64;
    if (check_args(n_seqs, cu, Hq, Hv, K, V, ckpt) || !dout || !dq || !dk || !dv || !dbeta || !dg)
        return 1;
    const int Ttot = cu[n_seqs];
    problem p;
    memset(&p, 0, sizeof(p));
    p.n_seqs = n_seqs; p.cu = cu; p.Hq = Hq; p.Hv = Hv; p.K = K; p.V = V; p.C = ckpt;
    p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta; p.scale = scale; p.h0 = h0;
    p.dout = dout; p.dht = dht; p.dv = dv; p.dbeta = dbeta; p.dg = dg; p.dh0 = dh0;
    p.dq_part = (double *)calloc((size_t)Ttot * Hv * K + 1, sizeof(double));
    p.dk_part = (double *)calloc((size_t)Ttot * Hv * K + 1, sizeof(double));
    run_pool(&p, n_seqs * Hv, 1, nthreads, bwd_job);
    const int G = Hv / Hq;
    for (int t = 0; t < Ttot; ++t)
        for (int hq = 0; hq < Hq; ++hq)
            for (int i = 0; i < K; ++i) {
                double sq = 0.0, sk = 0.0;
                for (int j = 0; j < G; ++j) {
                    const size_t idx = ((size_t)t * Hv + hq * G + j) * K + i;
                    sq += p.dq_part[idx];
                    sk += p.dk_part[idx];
                }
                dq[((size_t)t * Hq + hq) * K + i] = sq;
                dk[((size_t)t * Hq + hq) * K + i] = sk;
            }
    free(p.dq_part);
    free(p.dk_part);
    return 0;
}
