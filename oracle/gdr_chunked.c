/*
 * gdr_chunked.c -- a second, independent fp64 CPU form of the GDN forward:
 * the chunked (WY / UT-transform) algebra with an exact context-parallel
 * split into segments.  TEST INFRASTRUCTURE ONLY: it exists to pin the chunk
 * algebra, A and h against the token recurrence of gdr_oracle.c.  It shares
 * no code with gdr_oracle.c nor with the CUDA path.
 *
 * Pages followed (FlashQLA):
 *   - "ignoring gate preprocessing and CP, the forward for chunk i reads K and
 *     V and passes W, U, S between steps" (page 1, efficiency problem): the
 *     per-chunk quantities W, U and the inter-chunk state S;
 *   - the CP split (page 1, "two fused kernels and automatic CP"): N chunks,
 *     L chunks per segment; step 2.1 runs each segment from a zero state and
 *     also composes its transition (the "correction matrix M" of page 3,
 *     technical principles); step 2.2 combines the segments in order; step 3
 *     re-runs each segment from its true start state and emits the output.
 *
 * Chunk algebra (one chunk of n <= C rows, start state S0, all per v-head):
 *   gamma_r = sum_{s<=r} g_s,   D_rs = exp(gamma_r - gamma_s)
 *   L  = strict_tril(diag(b) (K K^T o D)),   A = (I + L)^-1
 *   W  = A diag(b exp(gamma)) K,            U = A diag(b) V
 *   Ut = U - W S0                          (pseudo-values of the chunk)
 *   O  = scale (diag(exp(gamma)) Q S0 + (Q K^T o D o tril_incl) Ut)
 *   S1 = exp(gamma_n) S0 + Kt^T Ut,         Kt = diag(exp(gamma_n - gamma)) K
 * The transition of a chunk is T = exp(gamma_n) I - Kt^T W, so a segment maps
 * its start state S to M S + H with M the product of its T and H its end
 * state from S = 0.  Carrying X = [S | M] through the same update with
 * [U | 0] in place of U gives both.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int n_seqs; const int *cu;
    int Hq, Hv, K, V, C, seg;
    const double *q, *k, *v, *g, *beta, *h0;
    double scale;
    double *o, *final_state, *hchunks, *A;
    int *choff;
    int next; pthread_mutex_t mu;
} cproblem;

typedef struct {
    int n;                  /* rows in this chunk */
    double *gam, *A, *W, *U, *Kt, *Qt, *P; /* C, CxC, CxK, CxV, CxK, CxK, CxC */
    double decay;           /* exp(gamma_{n-1}) */
} chunk_t;

static void chunk_alloc(chunk_t *c, int C, int K, int V) {
    c->gam = (double *)calloc((size_t)C, sizeof(double));
    c->A = (double *)calloc((size_t)C * C, sizeof(double));
    c->W = (double *)calloc((size_t)C * K, sizeof(double));
    c->U = (double *)calloc((size_t)C * V, sizeof(double));
    c->Kt = (double *)calloc((size_t)C * K, sizeof(double));
    c->Qt = (double *)calloc((size_t)C * K, sizeof(double));
    c->P = (double *)calloc((size_t)C * C, sizeof(double));
}

static void chunk_free(chunk_t *c) {
    free(c->gam); free(c->A); free(c->W); free(c->U); free(c->Kt); free(c->Qt); free(c->P);
}

/* Fill every per-chunk quantity for tokens [ts, ts+n) of v-head h. */
static void chunk_prepare(const cproblem *p, int h, int ts, int n, chunk_t *c) {
    const int C = p->C, K = p->K, V = p->V, Hv = p->Hv, Hq = p->Hq;
    const int hq = h / (Hv / Hq);
    c->n = n;
    double run = 0.0;
    for (int r = 0; r < n; ++r) { run += p->g[(size_t)(ts + r) * Hv + h]; c->gam[r] = run; }
    c->decay = exp(c->gam[n - 1]);
#define KROW(r) (p->k + ((size_t)(ts + (r)) * Hq + hq) * K)
#define QROW(r) (p->q + ((size_t)(ts + (r)) * Hq + hq) * K)
#define VROW(r) (p->v + ((size_t)(ts + (r)) * Hv + h) * V)
#define BETA(r) (p->beta[(size_t)(ts + (r)) * Hv + h])
    /* M = I + L (dense, n x n), then A = M^-1 by solving M A = I column by column */
    double *M = (double *)calloc((size_t)n * n, sizeof(double));
    for (int r = 0; r < n; ++r) {
        M[r * n + r] = 1.0;
        for (int s = 0; s < r; ++s) {
            double kk = 0.0;
            for (int i = 0; i < K; ++i) kk += KROW(r)[i] * KROW(s)[i];
            M[r * n + s] = BETA(r) * kk * exp(c->gam[r] - c->gam[s]);
        }
    }
    for (int col = 0; col < n; ++col)
        for (int r = 0; r < n; ++r) {
            double rhs = (r == col) ? 1.0 : 0.0;
            for (int s = 0; s < r; ++s) rhs -= M[r * n + s] * c->A[s * C + col];
            c->A[r * C + col] = rhs; /* unit diagonal */
        }
    free(M);
    /* W = A diag(b e^gamma) K,  U = A diag(b) V */
    for (int r = 0; r < n; ++r) {
        for (int i = 0; i < K; ++i) {
            double acc = 0.0;
            for (int s = 0; s < n; ++s) acc += c->A[r * C + s] * BETA(s) * exp(c->gam[s]) * KROW(s)[i];
            c->W[r * K + i] = acc;
        }
        for (int j = 0; j < V; ++j) {
            double acc = 0.0;
            for (int s = 0; s < n; ++s) acc += c->A[r * C + s] * BETA(s) * VROW(s)[j];
            c->U[r * V + j] = acc;
        }
        for (int i = 0; i < K; ++i) {
            c->Kt[r * K + i] = exp(c->gam[n - 1] - c->gam[r]) * KROW(r)[i];
            c->Qt[r * K + i] = exp(c->gam[r]) * QROW(r)[i];
        }
        for (int s = 0; s < n; ++s) {
            double val = 0.0;
            if (s <= r) {
                double qk = 0.0;
                for (int i = 0; i < K; ++i) qk += QROW(r)[i] * KROW(s)[i];
                val = qk * exp(c->gam[r] - c->gam[s]);
            }
            c->P[r * C + s] = val;
        }
    }
#undef KROW
#undef QROW
#undef VROW
#undef BETA
}

/* X (K x w) <- decay X + Kt^T (R - W X), R (n x w) the right-hand pseudo-values. */
static void chunk_update(const chunk_t *c, int K, int w, double *X, const double *R, int ldR,
                         double *tmp /* C x w */) {
    for (int r = 0; r < c->n; ++r)
        for (int j = 0; j < w; ++j) {
            double acc = R ? R[r * ldR + j] : 0.0;
            for (int i = 0; i < K; ++i) acc -= c->W[r * K + i] * X[i * w + j];
            tmp[r * w + j] = acc;
        }
    for (int i = 0; i < K; ++i)
        for (int j = 0; j < w; ++j) {
            double acc = c->decay * X[i * w + j];
            for (int r = 0; r < c->n; ++r) acc += c->Kt[r * K + i] * tmp[r * w + j];
            X[i * w + j] = acc;
        }
}

static void seq_head(cproblem *p, int n, int h) {
    const int C = p->C, K = p->K, V = p->V, Hv = p->Hv;
    const int t0 = p->cu[n], t1 = p->cu[n + 1];
    const int nch = (t1 - t0 + C - 1) / C;
    const int seg = p->seg > 0 ? p->seg : (nch > 0 ? nch : 1);
    const int nseg = (nch + seg - 1) / seg;
    const size_t KV = (size_t)K * V;
    chunk_t c;
    chunk_alloc(&c, C, K, V);
    const int w = V + K;
    double *X = (double *)malloc(sizeof(double) * (size_t)K * w);
    double *tmp = (double *)malloc(sizeof(double) * (size_t)C * w);
    double *Hs = (double *)malloc(sizeof(double) * KV * (size_t)(nseg + 1));
    double *Ms = (double *)malloc(sizeof(double) * (size_t)K * K * (size_t)(nseg + 1));
    double *Sst = (double *)malloc(sizeof(double) * KV * (size_t)(nseg + 1));
    double *S = (double *)malloc(sizeof(double) * KV);
    double *Raug = (double *)calloc((size_t)C * w, sizeof(double));

    /* step 2.1: per-segment local end state H_j (from S = 0) and transition M_j */
    for (int j = 0; j < nseg; ++j) {
        memset(X, 0, sizeof(double) * (size_t)K * w);
        for (int i = 0; i < K; ++i) X[i * w + V + i] = 1.0;
        const int ce = (j + 1) * seg < nch ? (j + 1) * seg : nch;
        for (int ci = j * seg; ci < ce; ++ci) {
            const int ts = t0 + ci * C;
            const int len = (t1 - ts) < C ? (t1 - ts) : C;
            chunk_prepare(p, h, ts, len, &c);
            for (int r = 0; r < len; ++r) {
                memcpy(Raug + (size_t)r * w, c.U + (size_t)r * V, sizeof(double) * V);
                memset(Raug + (size_t)r * w + V, 0, sizeof(double) * K);
            }
            chunk_update(&c, K, w, X, Raug, w, tmp);
        }
        for (int i = 0; i < K; ++i) {
            memcpy(Hs + KV * j + (size_t)i * V, X + (size_t)i * w, sizeof(double) * V);
            memcpy(Ms + (size_t)K * K * j + (size_t)i * K, X + (size_t)i * w + V, sizeof(double) * K);
        }
    }
    /* step 2.2: S_start(j+1) = M_j S_start(j) + H_j */
    for (size_t e = 0; e < KV; ++e) Sst[e] = p->h0 ? p->h0[((size_t)n * Hv + h) * KV + e] : 0.0;
    for (int j = 0; j < nseg; ++j)
        for (int i = 0; i < K; ++i)
            for (int col = 0; col < V; ++col) {
                double acc = Hs[KV * j + (size_t)i * V + col];
                for (int l = 0; l < K; ++l)
                    acc += Ms[(size_t)K * K * j + (size_t)i * K + l] * Sst[KV * j + (size_t)l * V + col];
                Sst[KV * (j + 1) + (size_t)i * V + col] = acc;
            }
    /* step 3: re-run every segment from its true start, emit o, h, A */
    for (int j = 0; j < nseg; ++j) {
        memcpy(S, Sst + KV * j, sizeof(double) * KV);
        const int ce = (j + 1) * seg < nch ? (j + 1) * seg : nch;
        for (int ci = j * seg; ci < ce; ++ci) {
            const int ts = t0 + ci * C;
            const int len = (t1 - ts) < C ? (t1 - ts) : C;
            chunk_prepare(p, h, ts, len, &c);
            if (p->hchunks)
                memcpy(p->hchunks + (((size_t)p->choff[n] + ci) * Hv + h) * KV, S, sizeof(double) * KV);
            if (p->A)
                for (int r = 0; r < len; ++r)
                    for (int s = 0; s < C; ++s)
                        p->A[((size_t)(ts + r) * Hv + h) * C + s] = s < len ? c.A[r * C + s] : 0.0;
            /* Ut = U - W S */
            for (int r = 0; r < len; ++r)
                for (int col = 0; col < V; ++col) {
                    double acc = c.U[r * V + col];
                    for (int i = 0; i < K; ++i) acc -= c.W[r * K + i] * S[(size_t)i * V + col];
                    tmp[r * V + col] = acc;
                }
            /* O = scale (Qt S + P Ut) */
            for (int r = 0; r < len; ++r)
                for (int col = 0; col < V; ++col) {
                    double acc = 0.0;
                    for (int i = 0; i < K; ++i) acc += c.Qt[r * K + i] * S[(size_t)i * V + col];
                    for (int s = 0; s <= r; ++s) acc += c.P[r * C + s] * tmp[s * V + col];
                    p->o[((size_t)(ts + r) * Hv + h) * V + col] = p->scale * acc;
                }
            /* S = decay S + Kt^T Ut */
            for (int i = 0; i < K; ++i)
                for (int col = 0; col < V; ++col) {
                    double acc = c.decay * S[(size_t)i * V + col];
                    for (int r = 0; r < len; ++r) acc += c.Kt[r * K + i] * tmp[r * V + col];
                    S[(size_t)i * V + col] = acc;
                }
        }
    }
    if (p->final_state) {
        /* nch == 0: the state is h0 untouched */
        const double *src = nch > 0 ? S : Sst;
        memcpy(p->final_state + ((size_t)n * Hv + h) * KV, src, sizeof(double) * KV);
    }
    chunk_free(&c);
    free(X); free(tmp); free(Hs); free(Ms); free(Sst); free(S); free(Raug);
}

static void *cworker(void *arg) {
    cproblem *p = (cproblem *)arg;
    for (;;) {
        pthread_mutex_lock(&p->mu);
        int j = p->next++;
        pthread_mutex_unlock(&p->mu);
        if (j >= p->n_seqs * p->Hv) break;
        seq_head(p, j / p->Hv, j % p->Hv);
    }
    return NULL;
}

int gdr_chunked_fwd(int n_seqs, const int *cu, int Hq, int Hv, int K, int V, int C, int seg_chunks,
                    const double *q, const double *k, const double *v, const double *g,
                    const double *beta, double scale, const double *h0, double *o,
                    double *final_state, double *hchunks, double *A, int nthreads) {
    if (n_seqs < 1 || !cu || cu[0] != 0 || Hq < 1 || Hv < 1 || Hv % Hq || K < 1 || V < 1 || C < 1 || !o)
        return 1;
    for (int n = 0; n < n_seqs; ++n)
        if (cu[n + 1] < cu[n]) return 1;
    cproblem p;
    memset(&p, 0, sizeof(p));
    p.n_seqs = n_seqs; p.cu = cu; p.Hq = Hq; p.Hv = Hv; p.K = K; p.V = V; p.C = C;
    p.seg = seg_chunks; p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta; p.h0 = h0;
    p.scale = scale; p.o = o; p.final_state = final_state; p.hchunks = hchunks; p.A = A;
    p.choff = (int *)malloc(sizeof(int) * (size_t)(n_seqs + 1));
    p.choff[0] = 0;
    for (int n = 0; n < n_seqs; ++n) p.choff[n + 1] = p.choff[n] + (cu[n + 1] - cu[n] + C - 1) / C;
    pthread_mutex_init(&p.mu, NULL);
    if (nthreads < 1) nthreads = 1;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    for (int i = 0; i < nthreads; ++i) pthread_create(&th[i], NULL, cworker, &p);
    for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&p.mu);
    free(p.choff);
    return 0;
}
