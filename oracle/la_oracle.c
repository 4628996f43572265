/*
 * la_oracle.c -- plain, slow, double-precision CPU oracle for kernelised
 * (elu+1) linear attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline / reference leg may load this library.  It shares
 * no code, header, table or helper with the CUDA library; neither includes or
 * links the other.
 *
 * Every routine is a direct transcription of a definition on the source pages
 * (cited per function), written as straight loops over heads, tokens and
 * features, with no blocking, fusion or reordering beyond what the definition
 * itself states.  Layout everywhere: row-major [BH][N][d] for sequences,
 * [BH][d][d] for states (S[a][c]: a = key-feature index, c = value index) and
 * [BH][d] for normalisers.  `BH` is batch*heads flattened; a per-head decay
 * array, when given, has one entry per flattened head.
 *
 * Feature maps (argument `fmap`):
 *   0  phi(x) = elu(x) + 1 with alpha = 1, i.e. x + 1 for x > 0 and exp(x)
 *      otherwise ("Linear Attention", feature-map table, ELU+1 row; "Story of
 *      Attention - Part 5", section 1a).
 *   1  identity -- only so that the RetNet worked example (Part 5, section 4),
 *      which has no feature map and no normaliser, can pin the decayed
 *      recurrence and the decayed masked parallel form.
 * `normalise` = 1 divides by phi(q)^T z; 0 returns the bare numerator (again
 * only for the RetNet example).
 *
 * Return value of every int routine: 0 on success, -1 on a bad argument,
 * -2 on an allocation failure.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* elu(x) + 1 with alpha = 1.  The exp branch is written as exp(x) rather
 * than (exp(x) - 1) + 1 so that no cancellation occurs near zero. */
double ora_phi(double x) { return x > 0.0 ? x + 1.0 : exp(x); }

static double feat(double x, int fmap) { return fmap == 1 ? x : ora_phi(x); }

void ora_feature_map(const double *x, double *y, long n, int fmap) {
    for (long i = 0; i < n; ++i) y[i] = feat(x[i], fmap);
}

/* ------------------------------------------------------------------------ */
/* Minimal "one task per head" thread pool.                                  */

typedef void (*head_fn)(void *ctx, long h);
typedef struct {
    head_fn fn;
    void *ctx;
    long BH;
    long first, stride;
} head_job;

static void *head_worker(void *arg) {
    head_job *j = (head_job *)arg;
    for (long h = j->first; h < j->BH; h += j->stride) j->fn(j->ctx, h);
    return NULL;
}

static void for_each_head(head_fn fn, void *ctx, long BH, int nthreads) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > BH) nthreads = (int)(BH > 0 ? BH : 1);
    if (nthreads == 1) {
        for (long h = 0; h < BH; ++h) fn(ctx, h);
        return;
    }
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    head_job *jobs = (head_job *)malloc(sizeof(head_job) * (size_t)nthreads);
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].fn = fn; jobs[t].ctx = ctx; jobs[t].BH = BH;
        jobs[t].first = t; jobs[t].stride = nthreads;
        if (pthread_create(&tid[t], NULL, head_worker, &jobs[t]) == 0) ++started;
        else { jobs[t].first = BH; }
    }
    /* heads of threads that failed to start are done here */
    for (int t = 0; t < nthreads; ++t)
        if (jobs[t].first == BH)
            for (long h = t; h < BH; h += nthreads) fn(ctx, h);
    for (int t = 0; t < nthreads; ++t)
        if (jobs[t].first != BH) pthread_join(tid[t], NULL);
    (void)started;
    free(tid);
    free(jobs);
}

/* ------------------------------------------------------------------------ */
/* Non-causal form ("Linear Attention", generalised-kernel equations;
 * "Story of Attention - Part 5", section 1a, matrix form
 * phi(Q)[phi(K)^T V] / phi(Q)[phi(K)^T 1]).
 *   S[a][c] = sum_j phi(k_j)[a] v_j[c]      z[a] = sum_j phi(k_j)[a]        */

static void state_one_head(const double *k, const double *v, double *S,
                           double *z, long N, long d, int fmap) {
    memset(S, 0, sizeof(double) * (size_t)(d * d));
    memset(z, 0, sizeof(double) * (size_t)d);
    for (long j = 0; j < N; ++j) {
        const double *kj = k + j * d, *vj = v + j * d;
        for (long a = 0; a < d; ++a) {
            double pk = feat(kj[a], fmap);
            z[a] += pk;
            for (long c = 0; c < d; ++c) S[a * d + c] += pk * vj[c];
        }
    }
}

int ora_noncausal_state(const double *k, const double *v, double *S, double *z,
                        long BH, long N, long d, int fmap) {
    if (!k || !v || !S || !z || BH < 0 || N < 0 || d <= 0) return -1;
    for (long h = 0; h < BH; ++h)
        state_one_head(k + h * N * d, v + h * N * d, S + h * d * d, z + h * d,
                       N, d, fmap);
    return 0;
}

/* Read of a given state by M queries: y_i = phi(q_i)^T S / phi(q_i)^T z
 * ("Linear Attention", causal read-out; "Story of Attention - Part 5",
 * section 5, global retrieval sigma(Q) M / sigma(Q) z). */
static void read_one(const double *S, const double *z, const double *qi,
                     double *yi, long d, int fmap, int normalise) {
    double den = 0.0;
    for (long c = 0; c < d; ++c) yi[c] = 0.0;
    for (long a = 0; a < d; ++a) {
        double pq = feat(qi[a], fmap);
        den += pq * z[a];
        for (long c = 0; c < d; ++c) yi[c] += pq * S[a * d + c];
    }
    if (normalise)
        for (long c = 0; c < d; ++c) yi[c] /= den;
}

int ora_state_read(const double *S, const double *z, const double *q,
                   double *out, long BH, long M, long d, int fmap,
                   int normalise) {
    if (!S || !z || !q || !out || BH < 0 || M < 0 || d <= 0) return -1;
    for (long h = 0; h < BH; ++h)
        for (long i = 0; i < M; ++i)
            read_one(S + h * d * d, z + h * d, q + (h * M + i) * d,
                     out + (h * M + i) * d, d, fmap, normalise);
    return 0;
}

typedef struct {
    const double *q, *k, *v;
    double *out;
    long N, d;
    int fmap, normalise, err;
} nc_ctx;

static void nc_head(void *vctx, long h) {
    nc_ctx *c = (nc_ctx *)vctx;
    long N = c->N, d = c->d;
    double *S = (double *)malloc(sizeof(double) * (size_t)(d * d));
    double *z = (double *)malloc(sizeof(double) * (size_t)d);
    if (!S || !z) { c->err = -2; free(S); free(z); return; }
    state_one_head(c->k + h * N * d, c->v + h * N * d, S, z, N, d, c->fmap);
    for (long i = 0; i < N; ++i)
        read_one(S, z, c->q + (h * N + i) * d, c->out + (h * N + i) * d, d,
                 c->fmap, c->normalise);
    free(S);
    free(z);
}

int ora_noncausal(const double *q, const double *k, const double *v,
                  double *out, long BH, long N, long d, int fmap, int normalise,
                  int nthreads) {
    if (!q || !k || !v || !out || BH < 0 || N < 0 || d <= 0) return -1;
    nc_ctx c = {q, k, v, out, N, d, fmap, normalise, 0};
    for_each_head(nc_head, &c, BH, nthreads);
    return c.err;
}

/* ------------------------------------------------------------------------ */
/* Causal recurrence ("Linear Attention", running statistics
 * S_i = S_{i-1} + phi(k_i) v_i^T, z_i = z_{i-1} + phi(k_i),
 * y_i = phi(q_i)^T S_i / phi(q_i)^T z_i; "Story of Attention - Part 5",
 * section 1a causal form), with the per-head scalar decay of the lessons'
 * forget gate and RetNet's recurrent form (section 4): the state is
 * multiplied by g before each additive update, S_t = g S_{t-1} + ...
 * The same g multiplies z.  Update first, then read. */

int ora_recurrent_step(double *S, double *z, const double *q, const double *k,
                       const double *v, double *out, long d, double g,
                       int fmap, int normalise) {
    if (!S || !z || !q || !k || !v || !out || d <= 0) return -1;
    for (long a = 0; a < d; ++a) {
        double pk = feat(k[a], fmap);
        z[a] = g * z[a] + pk;
        for (long c = 0; c < d; ++c) S[a * d + c] = g * S[a * d + c] + pk * v[c];
    }
    read_one(S, z, q, out, d, fmap, normalise);
    return 0;
}

typedef struct {
    const double *q, *k, *v, *g;
    double *out;
    long N, d;
    int fmap, normalise, err;
} causal_ctx;

static void causal_head(void *vctx, long h) {
    causal_ctx *c = (causal_ctx *)vctx;
    long N = c->N, d = c->d;
    double g = c->g ? c->g[h] : 1.0;
    double *S = (double *)calloc((size_t)(d * d), sizeof(double));
    double *z = (double *)calloc((size_t)d, sizeof(double));
    if (!S || !z) { c->err = -2; free(S); free(z); return; }
    for (long t = 0; t < N; ++t) {
        long o = (h * N + t) * d;
        ora_recurrent_step(S, z, c->q + o, c->k + o, c->v + o, c->out + o, d,
                           g, c->fmap, c->normalise);
    }
    free(S);
    free(z);
}

int ora_causal(const double *q, const double *k, const double *v, double *out,
               long BH, long N, long d, const double *g, int fmap,
               int normalise, int nthreads) {
    if (!q || !k || !v || !out || BH < 0 || N < 0 || d <= 0) return -1;
    causal_ctx c = {q, k, v, g, out, N, d, fmap, normalise, 0};
    for_each_head(causal_head, &c, BH, nthreads);
    return c.err;
}

/* Causal recurrence with a data-dependent scalar gate per token and head
 * ("Linear Attention", GLA: S_t = G_t (.) S_{t-1} + k_t v_t^T with the gate
 * produced from the input; "Story of Attention - Part 5", section 7, the
 * scalar forget gate alpha_t of Gated DeltaNet), here with G_t = alpha_t
 * and the normaliser gated like the state:
 *   S_t = alpha_t S_{t-1} + phi(k_t) v_t^T,  z_t = alpha_t z_{t-1} + phi(k_t),
 *   y_t = phi(q_t)^T S_t / phi(q_t)^T z_t   (update, then read).
 * alpha [BH][N]. */
typedef struct {
    const double *q, *k, *v, *alpha;
    double *out;
    long N, d;
    int fmap, normalise, err;
} gated_ctx;

static void gated_head(void *vctx, long h) {
    gated_ctx *c = (gated_ctx *)vctx;
    long N = c->N, d = c->d;
    double *S = (double *)calloc((size_t)(d * d), sizeof(double));
    double *z = (double *)calloc((size_t)d, sizeof(double));
    if (!S || !z) { c->err = -2; free(S); free(z); return; }
    for (long t = 0; t < N; ++t) {
        long o = (h * N + t) * d;
        ora_recurrent_step(S, z, c->q + o, c->k + o, c->v + o, c->out + o, d,
                           c->alpha[h * N + t], c->fmap, c->normalise);
    }
    free(S);
    free(z);
}

int ora_causal_gated(const double *q, const double *k, const double *v,
                     const double *alpha, double *out, long BH, long N, long d,
                     int fmap, int normalise, int nthreads) {
    if (!q || !k || !v || !alpha || !out || BH < 0 || N < 0 || d <= 0) return -1;
    gated_ctx c = {q, k, v, alpha, out, N, d, fmap, normalise, 0};
    for_each_head(gated_head, &c, BH, nthreads);
    return c.err;
}

/* Final state of the causal recurrence after all N tokens -- the state a
 * decode continues from ("Linear Attention", the running statistics S_n and
 * z_n; with the forget-gate passage's scalar g):
 *   S_0 = 0, z_0 = 0;  S_t = g S_{t-1} + phi(k_t) v_t^T,  z_t = g z_{t-1} + phi(k_t).
 * S [BH][d][d] (S[a][c]: a key feature, c value column), z [BH][d]. */
int ora_causal_state(const double *k, const double *v, double *S, double *z,
                     long BH, long N, long d, const double *g, int fmap) {
    if (!k || !v || !S || !z || BH < 0 || N < 0 || d <= 0) return -1;
    for (long h = 0; h < BH; ++h) {
        const double gh = g ? g[h] : 1.0;
        double *Sh = S + h * d * d, *zh = z + h * d;
        for (long i = 0; i < d * d; ++i) Sh[i] = 0.0;
        for (long a = 0; a < d; ++a) zh[a] = 0.0;
        for (long t = 0; t < N; ++t) {
            const double *kt = k + (h * N + t) * d, *vt = v + (h * N + t) * d;
            for (long a = 0; a < d; ++a) {
                const double pk = feat(kt[a], fmap);
                zh[a] = gh * zh[a] + pk;
                for (long c = 0; c < d; ++c) Sh[a * d + c] = gh * Sh[a * d + c] + pk * vt[c];
            }
        }
    }
    return 0;
}

/* Recurrent decode step: one new token per head on a caller-owned state
 * (S [BH][d][d], z [BH][d], updated in place), then the read.  O(d^2) work
 * and memory per token ("Linear Attention", inference cost per token). */
typedef struct {
    double *S, *z;
    const double *q, *k, *v, *g;
    double *out;
    long d;
    int err;
} dec_ctx;

static void dec_head(void *vctx, long h) {
    dec_ctx *c = (dec_ctx *)vctx;
    long d = c->d;
    ora_recurrent_step(c->S + h * d * d, c->z + h * d, c->q + h * d,
                       c->k + h * d, c->v + h * d, c->out + h * d, d,
                       c->g ? c->g[h] : 1.0, 0, 1);
}

int ora_decode_step(double *S, double *z, const double *q, const double *k,
                    const double *v, double *out, long BH, long d,
                    const double *g, int nthreads) {
    if (!S || !z || !q || !k || !v || !out || BH < 0 || d <= 0) return -1;
    dec_ctx c = {S, z, q, k, v, g, out, d, 0};
    for_each_head(dec_head, &c, BH, nthreads);
    return c.err;
}

/* Delta-rule decode step ("Story of Attention - Part 5", section 7, Gated
 * DeltaNet / Delta Attention): one step of online gradient descent on
 * 1/2 ||S_{t-1} k_t - v_t||^2, with the optional scalar forget gate alpha_t:
 *   S_t = alpha_t S_{t-1} + beta_t (v_t - alpha_t S_{t-1} k_t) k_t^T,
 *   o_t = S_t q_t
 * (alpha = 1 without the gate; no feature map and no normaliser).  In the
 * page's orientation S k is the value stored for key k; here S [BH][d][d] is
 * stored transposed, S[a][c] with a the key feature and c the value column,
 * so (S k)[c] = sum_a S[a][c] k[a].  beta [BH], alpha [BH] or NULL. */
int ora_delta_step(double *S, const double *q, const double *k,
                   const double *v, const double *beta, const double *alpha,
                   double *out, long BH, long d) {
    if (!S || !q || !k || !v || !beta || !out || BH < 0 || d <= 0) return -1;
    double *pred = (double *)malloc(sizeof(double) * (size_t)d);
    if (!pred) return -2;
    for (long h = 0; h < BH; ++h) {
        double *Sh = S + h * d * d;
        const double *qh = q + h * d, *kh = k + h * d, *vh = v + h * d;
        const double a = alpha ? alpha[h] : 1.0, b = beta[h];
        for (long c = 0; c < d; ++c) {
            double s = 0.0;
            for (long r = 0; r < d; ++r) s += Sh[r * d + c] * kh[r];
            pred[c] = s;  /* S_{t-1} k_t */
        }
        for (long r = 0; r < d; ++r)
            for (long c = 0; c < d; ++c)
                Sh[r * d + c] = a * Sh[r * d + c] + b * kh[r] * (vh[c] - a * pred[c]);
        for (long c = 0; c < d; ++c) {
            double s = 0.0;
            for (long r = 0; r < d; ++r) s += Sh[r * d + c] * qh[r];
            out[h * d + c] = s;
        }
    }
    free(pred);
    return 0;
}

/* The delta rule over whole sequences: the recurrence of ora_delta_step
 * applied token after token ("Story of Attention - Part 5", section 7: the
 * write rule S_t = alpha_t S_{t-1} + beta_t (v_t - alpha_t S_{t-1} k_t) k_t^T
 * and the read o_t = S_t q_t), with one beta and one alpha per token.
 * q, k, v, out [BH][N][d]; beta, alpha [BH][N] (alpha NULL: 1); S [BH][d][d]
 * (S[a][c], a key feature) holds the start state and receives the state
 * after the last token. */
typedef struct {
    double *S;
    const double *q, *k, *v, *beta, *alpha;
    double *out;
    long N, d;
    int err;
} dfwd_ctx;

static void dfwd_head(void *arg, long h) {
    dfwd_ctx *c = (dfwd_ctx *)arg;
    const long N = c->N, d = c->d;
    double *S = c->S + h * d * d;
    double *pred = (double *)malloc(sizeof(double) * (size_t)d);
    if (!pred) {
        c->err = -2;
        return;
    }
    for (long t = 0; t < N; ++t) {
        const double *qt = c->q + (h * N + t) * d, *kt = c->k + (h * N + t) * d,
                     *vt = c->v + (h * N + t) * d;
        const double b = c->beta[h * N + t], a = c->alpha ? c->alpha[h * N + t] : 1.0;
        for (long col = 0; col < d; ++col) {
            double s = 0.0;
            for (long r = 0; r < d; ++r) s += S[r * d + col] * kt[r];
            pred[col] = s; /* S_{t-1} k_t */
        }
        for (long r = 0; r < d; ++r)
            for (long col = 0; col < d; ++col)
                S[r * d + col] = a * S[r * d + col] + b * kt[r] * (vt[col] - a * pred[col]);
        for (long col = 0; col < d; ++col) {
            double s = 0.0;
            for (long r = 0; r < d; ++r) s += S[r * d + col] * qt[r];
            c->out[(h * N + t) * d + col] = s; /* S_t q_t */
        }
    }
    free(pred);
}

int ora_delta_forward(double *S, const double *q, const double *k, const double *v,
                      const double *beta, const double *alpha, double *out, long BH,
                      long N, long d, int nthreads) {
    if (!S || !q || !k || !v || !beta || !out || BH < 0 || N < 0 || d <= 0) return -1;
    dfwd_ctx c = {S, q, k, v, beta, alpha, out, N, d, 0};
    for_each_head(dfwd_head, &c, BH, nthreads);
    return c.err;
}

/* ------------------------------------------------------------------------ */
/* Masked parallel (quadratic) form -- the other bracketing of the same
 * product ("Linear Attention: Removing the Softmax Buys Associativity",
 * parallel mode; "Story of Attention - Part 5", section 4, parallel form
 * (Q K^T (.) D) V with D_ij = g^(i-j) for i >= j, else 0):
 *   A_ij = (phi(q_i) . phi(k_j)) g^(i-j) for j <= i, else 0
 *   y_i  = sum_j A_ij v_j / sum_j A_ij.
 * `weights`, if non-NULL, receives A as [BH][N][N]. */
int ora_quadratic(const double *q, const double *k, const double *v,
                  double *out, long BH, long N, long d, const double *g,
                  int fmap, int normalise, double *weights) {
    if (!q || !k || !v || !out || BH < 0 || N < 0 || d <= 0) return -1;
    double *A = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    if (!A) return -2;
    for (long h = 0; h < BH; ++h) {
        const double *qh = q + h * N * d, *kh = k + h * N * d,
                     *vh = v + h * N * d;
        double gh = g ? g[h] : 1.0;
        for (long i = 0; i < N; ++i) {
            double den = 0.0;
            for (long j = 0; j < N; ++j) {
                double a = 0.0;
                if (j <= i) {
                    double dot = 0.0;
                    for (long f = 0; f < d; ++f)
                        dot += feat(qh[i * d + f], fmap) *
                               feat(kh[j * d + f], fmap);
                    a = dot * pow(gh, (double)(i - j));
                }
                A[j] = a;
                den += a;
                if (weights) weights[(h * N + i) * N + j] = a;
            }
            double *yi = out + (h * N + i) * d;
            for (long c = 0; c < d; ++c) {
                double num = 0.0;
                for (long j = 0; j <= i; ++j) num += A[j] * vh[j * d + c];
                yi[c] = normalise ? num / den : num;
            }
        }
    }
    free(A);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Chunked prototype (TEST-ONLY check of the block algebra).  It follows the
 * Lightning Attention block formulas ("Story of Attention - Part 5",
 * section 6), with phi applied to Q and K and with the normaliser carried
 * the same way as the numerator:
 *   O_i   = (Q_i K_i^T (.) M) V_i + Lambda Q_i S_{i-1}
 *   den_i = (Q_i K_i^T (.) M) 1   + Lambda Q_i z_{i-1}
 *   S_i   = g^B S_{i-1} + (g^B Lambda^{-1} K_i)^T V_i      (z_i likewise)
 * with M_st = g^(s-t) for s >= t, Lambda = diag(g, g^2, ..., g^B), and
 * g^B Lambda^{-1} = diag(g^(B-1), ..., g^0) written out directly.  A short
 * last block of b < B tokens uses b in place of B.
 * On top of the blocks, the sequence is cut into P segments of whole blocks;
 * each segment's local state (from zero) is formed first, the segment start
 * states are the exclusive decayed prefix over segments, and each segment
 * then runs its blocks from its start state.  With B = 1 this is the
 * recurrence; with one block it is the masked parallel form. */
int ora_chunked(const double *q, const double *k, const double *v,
                double *out, long BH, long N, long d, const double *g,
                long B, long P) {
    if (!q || !k || !v || !out || BH < 0 || N < 0 || d <= 0 || B <= 0 ||
        P <= 0)
        return -1;
    long nblk = (N + B - 1) / B;
    long blk_per_seg = (nblk + P - 1) / P;
    if (blk_per_seg < 1) blk_per_seg = 1;
    long nseg = (nblk + blk_per_seg - 1) / blk_per_seg;
    size_t dd = (size_t)(d * d);
    double *pq = (double *)malloc(sizeof(double) * (size_t)(B * d));
    double *pk = (double *)malloc(sizeof(double) * (size_t)(B * d));
    double *Sl = (double *)malloc(sizeof(double) * dd * (size_t)(nseg + 1));
    double *zl = (double *)malloc(sizeof(double) * (size_t)d * (size_t)(nseg + 1));
    double *Ss = (double *)malloc(sizeof(double) * dd * (size_t)(nseg + 1));
    double *zs = (double *)malloc(sizeof(double) * (size_t)d * (size_t)(nseg + 1));
    double *S = (double *)malloc(sizeof(double) * dd);
    double *z = (double *)malloc(sizeof(double) * (size_t)d);
    double *Snew = (double *)malloc(sizeof(double) * dd);
    double *znew = (double *)malloc(sizeof(double) * (size_t)d);
    int rc = 0;
    if (!pq || !pk || !Sl || !zl || !Ss || !zs || !S || !z || !Snew || !znew) {
        rc = -2;
        goto done;
    }
    for (long h = 0; h < BH; ++h) {
        const double *qh = q + h * N * d, *kh = k + h * N * d,
                     *vh = v + h * N * d;
        double *oh = out + h * N * d;
        double gh = g ? g[h] : 1.0;
        /* 1. local state of every segment, from zero, decayed to the
         *    segment's last token. */
        for (long s = 0; s < nseg; ++s) {
            long t0 = s * blk_per_seg * B;
            long t1 = (s + 1) * blk_per_seg * B;
            if (t1 > N) t1 = N;
            double *Sloc = Sl + (size_t)s * dd, *zloc = zl + (size_t)s * d;
            memset(Sloc, 0, sizeof(double) * dd);
            memset(zloc, 0, sizeof(double) * (size_t)d);
            for (long t = t0; t < t1; ++t) {
                double w = pow(gh, (double)(t1 - 1 - t));
                for (long a = 0; a < d; ++a) {
                    double f = w * ora_phi(kh[t * d + a]);
                    zloc[a] += f;
                    for (long c = 0; c < d; ++c)
                        Sloc[a * d + c] += f * vh[t * d + c];
                }
            }
        }
        /* 2. exclusive decayed prefix over segments. */
        memset(Ss, 0, sizeof(double) * dd);
        memset(zs, 0, sizeof(double) * (size_t)d);
        for (long s = 0; s + 1 < nseg; ++s) {
            long t0 = s * blk_per_seg * B;
            long t1 = (s + 1) * blk_per_seg * B;
            if (t1 > N) t1 = N;
            double w = pow(gh, (double)(t1 - t0));
            for (size_t e = 0; e < dd; ++e)
                Ss[(size_t)(s + 1) * dd + e] =
                    w * Ss[(size_t)s * dd + e] + Sl[(size_t)s * dd + e];
            for (long a = 0; a < d; ++a)
                zs[(size_t)(s + 1) * d + a] =
                    w * zs[(size_t)s * d + a] + zl[(size_t)s * d + a];
        }
        /* 3. blocks of every segment from its start state. */
        for (long s = 0; s < nseg; ++s) {
            memcpy(S, Ss + (size_t)s * dd, sizeof(double) * dd);
            memcpy(z, zs + (size_t)s * d, sizeof(double) * (size_t)d);
            long t_end = (s + 1) * blk_per_seg * B;
            if (t_end > N) t_end = N;
            for (long t0 = s * blk_per_seg * B; t0 < t_end; t0 += B) {
                long b = (t_end - t0 < B) ? (t_end - t0) : B;
                for (long i = 0; i < b; ++i)
                    for (long a = 0; a < d; ++a) {
                        pq[i * d + a] = ora_phi(qh[(t0 + i) * d + a]);
                        pk[i * d + a] = ora_phi(kh[(t0 + i) * d + a]);
                    }
                for (long i = 0; i < b; ++i) {
                    double lam = pow(gh, (double)(i + 1)); /* Lambda_ii */
                    double den = 0.0;
                    double *yi = oh + (t0 + i) * d;
                    for (long c = 0; c < d; ++c) yi[c] = 0.0;
                    /* intra-block: (Q K^T (.) M) V and its row sum */
                    for (long j = 0; j <= i; ++j) {
                        double dot = 0.0;
                        for (long a = 0; a < d; ++a)
                            dot += pq[i * d + a] * pk[j * d + a];
                        double m = dot * pow(gh, (double)(i - j));
                        den += m;
                        for (long c = 0; c < d; ++c)
                            yi[c] += m * vh[(t0 + j) * d + c];
                    }
                    /* inter-block: Lambda Q S_{i-1}, Lambda Q z_{i-1} */
                    for (long a = 0; a < d; ++a) {
                        double f = lam * pq[i * d + a];
                        den += f * z[a];
                        for (long c = 0; c < d; ++c) yi[c] += f * S[a * d + c];
                    }
                    for (long c = 0; c < d; ++c) yi[c] /= den;
                }
                /* S_i = g^b S_{i-1} + (g^(b-1-t) K_t)^T V_t */
                double gb = pow(gh, (double)b);
                for (long a = 0; a < d; ++a) {
                    znew[a] = gb * z[a];
                    for (long c = 0; c < d; ++c)
                        Snew[a * d + c] = gb * S[a * d + c];
                }
                for (long t = 0; t < b; ++t) {
                    double w = pow(gh, (double)(b - 1 - t));
                    for (long a = 0; a < d; ++a) {
                        double f = w * pk[t * d + a];
                        znew[a] += f;
                        for (long c = 0; c < d; ++c)
                            Snew[a * d + c] += f * vh[(t0 + t) * d + c];
                    }
                }
                memcpy(S, Snew, sizeof(double) * dd);
                memcpy(z, znew, sizeof(double) * (size_t)d);
            }
        }
    }
done:
    free(pq); free(pk); free(Sl); free(zl); free(Ss); free(zs);
    free(S); free(z); free(Snew); free(znew);
    return rc;
}
