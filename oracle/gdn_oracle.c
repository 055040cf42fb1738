/*
 * gdn_oracle.c -- fp64 CPU oracle for the Gated DeltaNet operator that CPR evaluates.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call this
 * file; only the tests, the package smoke check and the benchmark's CPU-baseline leg
 * do.  It shares no code, header, table or helper with the CUDA library.
 *
 * What it computes
 * ----------------
 * The operator is the gated delta rule (Gated DeltaNet, named on the IsoExec page
 * "IsoExec: SkyRLにおけるトレーナーと推論のミスマッチを解消する", section
 * "Chunkwise-Parallel Recurrent (CPR) Gated DeltaNet"; recurrence as defined by Yang,
 * Kautz and Hatamizadeh, "Gated Delta Networks: Improving Mamba2 with Delta Rule").
 * Per (sequence, value head), with state S in R^{dv x dk}:
 *
 *     S_t = exp(g_t) S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,    o_t = S_t q_t.
 *
 * The same page says CPR keeps this recurrence as the main computation and only
 * reorganises how it is evaluated (parallel across chunks, decode resynchronised every
 * C tokens).  Those are exact rewrites, so the oracle is the recurrence itself, token
 * by token, with no chunk size in it:
 *
 *     oracle_fwd          forward recurrence (plus, optionally, the state at every
 *                         multiple of C, which is what CPR's boundary pass produces)
 *     oracle_bwd          hand-derived reverse-mode gradient of the recurrence
 *     oracle_chunk_states the chunk (WY/UT) form of the same recurrence, used only to
 *                         pin the algebra of the boundary pass against oracle_fwd
 *
 * Conventions (readings where the pages are silent):
 *   - no scale on q; state is dv x dk row-major and o = S q;
 *   - grouped heads: value head h reads query/key head h / (Hv / Hqk);
 *   - sequences are packed along tokens by cu_seqlens; each starts from state_in
 *     (NULL = zero).
 *
 * Layouts (all double, row-major):
 *   q, k [T, Hqk, dk]   v, o [T, Hv, dv]   g, beta [T, Hv]   states [N, Hv, dv, dk].
 *
 * Every function returns 0 on success and a negative value on a bad argument.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_CKPT 64 /* backward recomputes states from a checkpoint every 64 tokens */

typedef struct {
    int n_seqs;
    const int32_t *cu;
    int hqk, hv, dk, dv;
    const double *q, *k, *v, *g, *beta, *state_in;
    double *o, *state_out;
    int chunk;
    double *bnd;           /* [sum_s ceil(L_s/C), Hv, dv, dk] start state of every chunk */
    const int64_t *chunk0; /* first global chunk index of each sequence */
    /* backward */
    const double *dout, *dstate_out;
    double *dq, *dk_, *dv_, *dg, *dbeta, *dstate_in;
} job_t;

typedef struct {
    job_t *job;
    int n_units;
    int next;
    pthread_mutex_t mu;
    void (*fn)(job_t *, int unit);
} pool_t;

static void *pool_worker(void *arg) {
    pool_t *p = (pool_t *)arg;
    for (;;) {
        pthread_mutex_lock(&p->mu);
        int u = p->next++;
        pthread_mutex_unlock(&p->mu);
        if (u >= p->n_units) return NULL;
        p->fn(p->job, u);
    }
}

static void run_pool(job_t *job, int n_units, int n_threads, void (*fn)(job_t *, int)) {
    if (n_threads < 1) n_threads = 1;
    if (n_threads > n_units) n_threads = n_units;
    pool_t p;
    p.job = job;
    p.n_units = n_units;
    p.next = 0;
    p.fn = fn;
    pthread_mutex_init(&p.mu, NULL);
    if (n_threads <= 1) {
        pool_worker(&p);
    } else {
        pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n_threads);
        for (int i = 0; i < n_threads; ++i) pthread_create(&th[i], NULL, pool_worker, &p);
        for (int i = 0; i < n_threads; ++i) pthread_join(th[i], NULL);
        free(th);
    }
    pthread_mutex_destroy(&p.mu);
}

static int check_common(int n_seqs, const int32_t *cu, int hqk, int hv, int dk, int dv) {
    if (n_seqs < 0 || !cu || hqk <= 0 || hv <= 0 || dk <= 0 || dv <= 0) return -1;
    if (hv % hqk != 0) return -1;
    if (cu[0] != 0) return -1;
    for (int s = 0; s < n_seqs; ++s)
        if (cu[s + 1] < cu[s]) return -1;
    return 0;
}

/* One recurrent step on S (dv x dk) for token t of value head h.  Writes o_t if o != NULL.
 * Order: decay, read-out of the decayed state along k, delta, rank-1 write, read-out along q. */
static void step(double *S, int dk, int dv, double a, double b, const double *kt, const double *vt,
                 const double *qt, double *ot) {
    for (int i = 0; i < dv; ++i) {
        double *row = S + (size_t)i * dk;
        double p = 0.0;
        for (int c = 0; c < dk; ++c) {
            row[c] *= a;
            p += row[c] * kt[c];
        }
        double u = b * (vt[i] - p);
        double o = 0.0;
        for (int c = 0; c < dk; ++c) {
            row[c] += u * kt[c];
            o += row[c] * qt[c];
        }
        if (ot) ot[i] = o;
    }
}

/* ------------------------------------------------------------------ forward ---- */

static void fwd_unit(job_t *J, int unit) {
    const int s = unit / J->hv, h = unit % J->hv;
    const int hq = h / (J->hv / J->hqk);
    const int dk = J->dk, dv = J->dv;
    const size_t sz = (size_t)dv * dk;
    double *S = (double *)malloc(sizeof(double) * sz);
    if (J->state_in)
        memcpy(S, J->state_in + ((size_t)s * J->hv + h) * sz, sizeof(double) * sz);
    else
        memset(S, 0, sizeof(double) * sz);
    const int t0 = J->cu[s], t1 = J->cu[s + 1];
    for (int t = t0; t < t1; ++t) {
        const int lt = t - t0;
        if (J->bnd && J->chunk > 0 && lt % J->chunk == 0) {
            const int64_t gc = J->chunk0[s] + lt / J->chunk;
            memcpy(J->bnd + ((size_t)gc * J->hv + h) * sz, S, sizeof(double) * sz);
        }
        const double *kt = J->k + ((size_t)t * J->hqk + hq) * dk;
        const double *qt = J->q + ((size_t)t * J->hqk + hq) * dk;
        const double *vt = J->v + ((size_t)t * J->hv + h) * dv;
        const double gt = J->g[(size_t)t * J->hv + h];
        const double bt = J->beta[(size_t)t * J->hv + h];
        step(S, dk, dv, exp(gt), bt, kt, vt, qt, J->o + ((size_t)t * J->hv + h) * dv);
    }
    if (J->state_out) memcpy(J->state_out + ((size_t)s * J->hv + h) * sz, S, sizeof(double) * sz);
    free(S);
}

static int64_t *chunk_offsets(int n_seqs, const int32_t *cu, int chunk) {
    int64_t *c0 = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n_seqs + 1));
    c0[0] = 0;
    for (int s = 0; s < n_seqs; ++s) {
        const int L = cu[s + 1] - cu[s];
        c0[s + 1] = c0[s] + (chunk > 0 ? (L + chunk - 1) / chunk : 0);
    }
    return c0;
}

/* Forward recurrence.  If bnd_states != NULL and chunk > 0, also writes the state before
 * token j*C of every sequence (j = 0 .. ceil(L/C)-1) into bnd_states, chunks numbered
 * globally in sequence order.  Returns the number of chunks via *n_chunks if non-NULL. */
int oracle_fwd(int n_seqs, const int32_t *cu_seqlens, int hqk, int hv, int dk, int dv,
               const double *q, const double *k, const double *v, const double *g,
               const double *beta, const double *state_in, double *o, double *state_out,
               int chunk, double *bnd_states, int n_threads) {
    if (check_common(n_seqs, cu_seqlens, hqk, hv, dk, dv)) return -1;
    if ((!q || !k || !v || !g || !beta || !o) && cu_seqlens[n_seqs] > 0) return -2;
    if (bnd_states && chunk <= 0) return -3;
    job_t J;
    memset(&J, 0, sizeof(J));
    J.n_seqs = n_seqs; J.cu = cu_seqlens; J.hqk = hqk; J.hv = hv; J.dk = dk; J.dv = dv;
    J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta; J.state_in = state_in;
    J.o = o; J.state_out = state_out; J.chunk = chunk; J.bnd = bnd_states;
    int64_t *c0 = chunk_offsets(n_seqs, cu_seqlens, chunk);
    J.chunk0 = c0;
    run_pool(&J, n_seqs * hv, n_threads, fwd_unit);
    free(c0);
    return 0;
}

/* ----------------------------------------------------------------- backward ---- */

/* Reverse-mode gradient of the recurrence.  Per token, going backwards with the incoming
 * adjoint D of S_t (derived by hand from the step above):
 *   D  += do_t q_t^T                     dq_t += S_t^T do_t
 *   du  = D k_t                          dk_t += D^T u
 *   dbeta_t = du . (v_t - p)             dv_t  = beta_t du       dp = -beta_t du
 *   D  += dp k_t^T                       dk_t += S'^T dp         (S' = exp(g_t) S_{t-1})
 *   dg_t = <D, S'>_F                     D <- exp(g_t) D
 * States are recomputed from checkpoints taken every ORACLE_CKPT tokens.  One work unit is
 * a (sequence, query/key head) pair so the grouped dq/dk sums have a single writer; value
 * heads of a group are visited in ascending order. */
static void bwd_unit(job_t *J, int unit) {
    const int s = unit / J->hqk, hq = unit % J->hqk;
    const int grp = J->hv / J->hqk;
    const int dk = J->dk, dv = J->dv;
    const size_t sz = (size_t)dv * dk;
    const int t0 = J->cu[s], t1 = J->cu[s + 1], L = t1 - t0;
    const int nck = (L + ORACLE_CKPT - 1) / ORACLE_CKPT;
    double *ck = (double *)malloc(sizeof(double) * sz * (size_t)(nck > 0 ? nck : 1));
    double *seg = (double *)malloc(sizeof(double) * sz * (ORACLE_CKPT + 1));
    double *D = (double *)malloc(sizeof(double) * sz);
    double *Sp = (double *)malloc(sizeof(double) * sz);
    double *p = (double *)malloc(sizeof(double) * (size_t)dv);
    double *u = (double *)malloc(sizeof(double) * (size_t)dv);
    double *du = (double *)malloc(sizeof(double) * (size_t)dv);

    for (int t = t0; t < t1; ++t)
        for (int c = 0; c < dk; ++c) {
            J->dq[((size_t)t * J->hqk + hq) * dk + c] = 0.0;
            J->dk_[((size_t)t * J->hqk + hq) * dk + c] = 0.0;
        }

    for (int hh = 0; hh < grp; ++hh) {
        const int h = hq * grp + hh;
        /* forward pass storing checkpoints */
        double *S = seg; /* scratch */
        if (J->state_in)
            memcpy(S, J->state_in + ((size_t)s * J->hv + h) * sz, sizeof(double) * sz);
        else
            memset(S, 0, sizeof(double) * sz);
        for (int t = t0; t < t1; ++t) {
            const int lt = t - t0;
            if (lt % ORACLE_CKPT == 0) memcpy(ck + (size_t)(lt / ORACLE_CKPT) * sz, S, sizeof(double) * sz);
            const double *kt = J->k + ((size_t)t * J->hqk + hq) * dk;
            const double *vt = J->v + ((size_t)t * J->hv + h) * dv;
            step(S, dk, dv, exp(J->g[(size_t)t * J->hv + h]), J->beta[(size_t)t * J->hv + h], kt,
                 vt, kt, NULL);
        }
        /* incoming adjoint of the final state */
        if (J->dstate_out)
            memcpy(D, J->dstate_out + ((size_t)s * J->hv + h) * sz, sizeof(double) * sz);
        else
            memset(D, 0, sizeof(double) * sz);

        for (int cb = nck - 1; cb >= 0; --cb) {
            const int ta = t0 + cb * ORACLE_CKPT;
            const int tb = (ta + ORACLE_CKPT < t1) ? ta + ORACLE_CKPT : t1;
            /* seg[i] = state before token ta+i, seg[tb-ta] = state after token tb-1 */
            memcpy(seg, ck + (size_t)cb * sz, sizeof(double) * sz);
            for (int t = ta; t < tb; ++t) {
                double *Sn = seg + (size_t)(t - ta + 1) * sz;
                memcpy(Sn, seg + (size_t)(t - ta) * sz, sizeof(double) * sz);
                const double *kt = J->k + ((size_t)t * J->hqk + hq) * dk;
                const double *vt = J->v + ((size_t)t * J->hv + h) * dv;
                step(Sn, dk, dv, exp(J->g[(size_t)t * J->hv + h]), J->beta[(size_t)t * J->hv + h],
                     kt, vt, kt, NULL);
            }
            for (int t = tb - 1; t >= ta; --t) {
                const double *Sprev = seg + (size_t)(t - ta) * sz;
                const double *St = seg + (size_t)(t - ta + 1) * sz;
                const double *kt = J->k + ((size_t)t * J->hqk + hq) * dk;
                const double *qt = J->q + ((size_t)t * J->hqk + hq) * dk;
                const double *vt = J->v + ((size_t)t * J->hv + h) * dv;
                const double *dot = J->dout + ((size_t)t * J->hv + h) * dv;
                const double a = exp(J->g[(size_t)t * J->hv + h]);
                const double b = J->beta[(size_t)t * J->hv + h];
                double *dqt = J->dq + ((size_t)t * J->hqk + hq) * dk;
                double *dkt = J->dk_ + ((size_t)t * J->hqk + hq) * dk;
                /* recompute S' = a S_{t-1}, p = S' k, u = b (v - p) */
                for (size_t e = 0; e < sz; ++e) Sp[e] = a * Sprev[e];
                for (int i = 0; i < dv; ++i) {
                    double acc = 0.0;
                    for (int c = 0; c < dk; ++c) acc += Sp[(size_t)i * dk + c] * kt[c];
                    p[i] = acc;
                    u[i] = b * (vt[i] - acc);
                }
                /* o_t = S_t q_t */
                for (int i = 0; i < dv; ++i)
                    for (int c = 0; c < dk; ++c) {
                        D[(size_t)i * dk + c] += dot[i] * qt[c];
                        dqt[c] += St[(size_t)i * dk + c] * dot[i];
                    }
                /* S_t = S' + u k^T */
                double dbeta = 0.0;
                for (int i = 0; i < dv; ++i) {
                    double acc = 0.0;
                    for (int c = 0; c < dk; ++c) acc += D[(size_t)i * dk + c] * kt[c];
                    du[i] = acc;
                    for (int c = 0; c < dk; ++c) dkt[c] += D[(size_t)i * dk + c] * u[i];
                    dbeta += acc * (vt[i] - p[i]);
                    J->dv_[((size_t)t * J->hv + h) * dv + i] = b * acc;
                }
                J->dbeta[(size_t)t * J->hv + h] = dbeta;
                /* p = S' k */
                for (int i = 0; i < dv; ++i) {
                    const double dp = -b * du[i];
                    for (int c = 0; c < dk; ++c) {
                        D[(size_t)i * dk + c] += dp * kt[c];
                        dkt[c] += Sp[(size_t)i * dk + c] * dp;
                    }
                }
                /* S' = a S_{t-1} */
                double dg = 0.0;
                for (size_t e = 0; e < sz; ++e) {
                    dg += D[e] * Sp[e];
                    D[e] *= a;
                }
                J->dg[(size_t)t * J->hv + h] = dg;
            }
        }
        if (J->dstate_in) memcpy(J->dstate_in + ((size_t)s * J->hv + h) * sz, D, sizeof(double) * sz);
    }
    free(ck); free(seg); free(D); free(Sp); free(p); free(u); free(du);
}

int oracle_bwd(int n_seqs, const int32_t *cu_seqlens, int hqk, int hv, int dk, int dv,
               const double *q, const double *k, const double *v, const double *g,
               const double *beta, const double *state_in, const double *dout,
               const double *dstate_out, double *dq, double *dk_out, double *dv_out, double *dg,
               double *dbeta, double *dstate_in, int n_threads) {
    if (check_common(n_seqs, cu_seqlens, hqk, hv, dk, dv)) return -1;
    if (cu_seqlens[n_seqs] > 0 &&
        (!q || !k || !v || !g || !beta || !dout || !dq || !dk_out || !dv_out || !dg || !dbeta))
        return -2;
    job_t J;
    memset(&J, 0, sizeof(J));
    J.n_seqs = n_seqs; J.cu = cu_seqlens; J.hqk = hqk; J.hv = hv; J.dk = dk; J.dv = dv;
    J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta; J.state_in = state_in;
    J.dout = dout; J.dstate_out = dstate_out;
    J.dq = dq; J.dk_ = dk_out; J.dv_ = dv_out; J.dg = dg; J.dbeta = dbeta; J.dstate_in = dstate_in;
    run_pool(&J, n_seqs * hqk, n_threads, bwd_unit);
    return 0;
}

/* ------------------------------------------------------------- chunk form ---- */

/* The same recurrence evaluated chunk by chunk in the WY/UT form (C tokens at a time,
 * the last chunk of a sequence may be shorter).  Within a chunk with start state S0 and
 * local tokens i = 0..n-1:
 *   G_i   = g_0 + ... + g_i
 *   A_is  = beta_i exp(G_i - G_s) (k_i . k_s)        for i > s, else 0
 *   T     = (I + A)^{-1}                              (forward substitution)
 *   Ut    = T diag(beta) V,     W = T diag(beta exp(G)) K
 *   U     = Ut - W S0^T                               (row i is the delta u_i of token i)
 *   S_end = exp(G_{n-1}) S0 + sum_s exp(G_{n-1} - G_s) u_s k_s^T
 * Writes the start state of every chunk (layout as oracle_fwd's bnd_states) and the final
 * state of every sequence.  Used only to pin the boundary algebra against oracle_fwd. */
static void chunk_unit(job_t *J, int unit) {
    const int s = unit / J->hv, h = unit % J->hv;
    const int hq = h / (J->hv / J->hqk);
    const int dk = J->dk, dv = J->dv, C = J->chunk;
    const size_t sz = (size_t)dv * dk;
    double *S = (double *)malloc(sizeof(double) * sz);
    double *G = (double *)malloc(sizeof(double) * (size_t)C);
    double *A = (double *)calloc((size_t)C * C, sizeof(double));
    double *T = (double *)calloc((size_t)C * C, sizeof(double));
    double *Ut = (double *)malloc(sizeof(double) * (size_t)C * dv);
    double *W = (double *)malloc(sizeof(double) * (size_t)C * dk);
    double *U = (double *)malloc(sizeof(double) * (size_t)C * dv);
    if (J->state_in)
        memcpy(S, J->state_in + ((size_t)s * J->hv + h) * sz, sizeof(double) * sz);
    else
        memset(S, 0, sizeof(double) * sz);
    const int t0 = J->cu[s], t1 = J->cu[s + 1];
    for (int c0 = t0, j = 0; c0 < t1; c0 += C, ++j) {
        const int n = (c0 + C <= t1) ? C : t1 - c0;
        memcpy(J->bnd + ((size_t)(J->chunk0[s] + j) * J->hv + h) * sz, S, sizeof(double) * sz);
#define KK(i) (J->k + ((size_t)(c0 + (i)) * J->hqk + hq) * dk)
#define VV(i) (J->v + ((size_t)(c0 + (i)) * J->hv + h) * dv)
#define GG(i) (J->g[(size_t)(c0 + (i)) * J->hv + h])
#define BB(i) (J->beta[(size_t)(c0 + (i)) * J->hv + h])
        double run = 0.0;
        for (int i = 0; i < n; ++i) { run += GG(i); G[i] = run; }
        for (int i = 0; i < n; ++i)
            for (int r = 0; r < n; ++r) {
                double val = 0.0;
                if (i > r) {
                    double dot = 0.0;
                    for (int c = 0; c < dk; ++c) dot += KK(i)[c] * KK(r)[c];
                    val = BB(i) * exp(G[i] - G[r]) * dot;
                }
                A[(size_t)i * C + r] = val;
            }
        /* (I + A) T = I, A strictly lower => T unit lower triangular, row by row */
        for (int i = 0; i < n; ++i)
            for (int r = 0; r < n; ++r) {
                double val = (i == r) ? 1.0 : 0.0;
                for (int m = 0; m < i; ++m) val -= A[(size_t)i * C + m] * T[(size_t)m * C + r];
                T[(size_t)i * C + r] = val;
            }
        for (int i = 0; i < n; ++i) {
            for (int e = 0; e < dv; ++e) {
                double acc = 0.0;
                for (int r = 0; r < n; ++r) acc += T[(size_t)i * C + r] * BB(r) * VV(r)[e];
                Ut[(size_t)i * dv + e] = acc;
            }
            for (int c = 0; c < dk; ++c) {
                double acc = 0.0;
                for (int r = 0; r < n; ++r) acc += T[(size_t)i * C + r] * BB(r) * exp(G[r]) * KK(r)[c];
                W[(size_t)i * dk + c] = acc;
            }
        }
        for (int i = 0; i < n; ++i)
            for (int e = 0; e < dv; ++e) {
                double acc = 0.0;
                for (int c = 0; c < dk; ++c) acc += W[(size_t)i * dk + c] * S[(size_t)e * dk + c];
                U[(size_t)i * dv + e] = Ut[(size_t)i * dv + e] - acc;
            }
        const double gl = G[n - 1];
        for (int e = 0; e < dv; ++e)
            for (int c = 0; c < dk; ++c) {
                double acc = exp(gl) * S[(size_t)e * dk + c];
                for (int r = 0; r < n; ++r) acc += exp(gl - G[r]) * U[(size_t)r * dv + e] * KK(r)[c];
                S[(size_t)e * dk + c] = acc;
            }
#undef KK
#undef VV
#undef GG
#undef BB
    }
    if (J->state_out) memcpy(J->state_out + ((size_t)s * J->hv + h) * sz, S, sizeof(double) * sz);
    free(S); free(G); free(A); free(T); free(Ut); free(W); free(U);
}

int oracle_chunk_states(int n_seqs, const int32_t *cu_seqlens, int hqk, int hv, int dk, int dv,
                        const double *k, const double *v, const double *g, const double *beta,
                        const double *state_in, int chunk, double *bnd_states, double *state_out,
                        int n_threads) {
    if (check_common(n_seqs, cu_seqlens, hqk, hv, dk, dv)) return -1;
    if (chunk <= 0 || !bnd_states) return -3;
    if (cu_seqlens[n_seqs] > 0 && (!k || !v || !g || !beta)) return -2;
    job_t J;
    memset(&J, 0, sizeof(J));
    J.n_seqs = n_seqs; J.cu = cu_seqlens; J.hqk = hqk; J.hv = hv; J.dk = dk; J.dv = dv;
    J.k = k; J.v = v; J.g = g; J.beta = beta; J.state_in = state_in;
    J.state_out = state_out; J.chunk = chunk; J.bnd = bnd_states;
    int64_t *c0 = chunk_offsets(n_seqs, cu_seqlens, chunk);
    J.chunk0 = c0;
    run_pool(&J, n_seqs * hv, n_threads, chunk_unit);
    free(c0);
    return 0;
}

/* Number of chunks (sum over sequences of ceil(L/C)). */
long long oracle_num_chunks(int n_seqs, const int32_t *cu_seqlens, int chunk) {
    if (chunk <= 0) return -1;
    long long n = 0;
    for (int s = 0; s < n_seqs; ++s) n += (cu_seqlens[s + 1] - cu_seqlens[s] + chunk - 1) / chunk;
    return n;
}
