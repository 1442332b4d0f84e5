/*
 * WKV-7 oracle: plain, slow, double-precision CPU implementation.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is compiled into liboracle.so and is
 * loaded by the tests, by the package's smoke check and by the benchmark's
 * CPU-baseline leg.  The product library (libwkv7) never links, loads or calls
 * it, and it shares no code, header or constant with the CUDA path.
 *
 * What it computes (RWKV-X Architecture, "WKV-7 Kernel (Generalized Delta
 * Rule)"): per head, a state matrix S of size N x N (N = head_size, "State is a
 * [head_size, head_size] matrix per head per RWKV-7 layer").  S[i][j] has i the
 * value index and j the key index, stored row-major (S[i*N + j]).  Per token:
 *
 *     h   = S a                      (h_i = sum_j S_ij a_j)          delta read
 *     S'  = S diag(w) + h b^T + v k^T                                 decay, delta write, kv write
 *     o   = S' r                     (o_i = sum_j S'_ij r_j)          readout after the update
 *
 * Readings taken where the page is loose (each is listed with its reason in
 * the design notes):
 *   - the delta term is h b^T with h = S a read from the state *before* the
 *     decay (S' = S (diag(w) + a b^T) + v k^T); the page's pseudo-code writes
 *     the bonus with k^T and applies the decay first, the method statement this
 *     build follows writes (S a) b^T on the old S;
 *   - the page multiplies from the left (r @ state); that is the same map on
 *     the transposed storage;
 *   - no bonus/u term, no normalisation, no gating: exactly the three lines.
 *
 * Three independent forms are provided so they can be checked against each
 * other on tiny inputs:
 *   1. sequential   -- the recurrence above, token by token;
 *   2. chunked      -- the same recurrence unrolled over a chunk of L tokens
 *                      into the WY/UT form (intra-chunk matrices, a unit
 *                      triangular inverse, one state update per chunk);
 *   3. matprod      -- S_t = S_0 A_1...A_t + sum_s v_s k_s^T A_{s+1}...A_t with
 *                      the dense transition A_t = diag(w_t) + a_t b_t^T.
 *
 * Inputs of a unit (one head of one sequence) are addressed as
 * x[base + t*tok_stride + j] for token t and channel j, the same for r, w, k,
 * v, a, b and for the output o.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_API __attribute__((visibility("default")))

/* ------------------------------------------------------------------------ */
/* Form 1: sequential recurrence.                                           */
/* ------------------------------------------------------------------------ */

/* One token of the recurrence on one head.  h is caller scratch of length N. */
static void seq_token(int N, double *S, const double *r, const double *w,
                      const double *k, const double *v, const double *a,
                      const double *b, double *o, double *h)
{
    for (int i = 0; i < N; ++i) {                 /* h = S a (old state) */
        double acc = 0.0;
        for (int j = 0; j < N; ++j) acc += S[i * N + j] * a[j];
        h[i] = acc;
    }
    for (int i = 0; i < N; ++i)                   /* S = S diag(w) + h b^T + v k^T */
        for (int j = 0; j < N; ++j)
            S[i * N + j] = S[i * N + j] * w[j] + h[i] * b[j] + v[i] * k[j];
    for (int i = 0; i < N; ++i) {                 /* o = S r (new state) */
        double acc = 0.0;
        for (int j = 0; j < N; ++j) acc += S[i * N + j] * r[j];
        o[i] = acc;
    }
}

ORACLE_API int wkv7_oracle_sequential(int N, int T, double *S, long long base,
                                      long long tok_stride, const double *r,
                                      const double *w, const double *k,
                                      const double *v, const double *a,
                                      const double *b, double *o)
{
    if (N <= 0 || T < 0) return 1;
    double *h = (double *)malloc(sizeof(double) * (size_t)N);
    if (!h) return 2;
    for (int t = 0; t < T; ++t) {
        long long off = base + (long long)t * tok_stride;
        seq_token(N, S, r + off, w + off, k + off, v + off, a + off, b + off,
                  o + off, h);
    }
    free(h);
    return 0;
}

/* The other order the pages leave open (RWKV-X Architecture, "WKV-7 Kernel
 * (Generalized Delta Rule)", whose pseudo-code decays the state first and then
 * reads a @ state): S' = S diag(w);  h = S' a;  S'' = S' + h b^T + v k^T;
 * o = S'' r.  Not the reading the build follows (that one reads h on the state
 * before the decay, above); kept only so that the difference between the two
 * readings can be measured.  One token on one head; h is caller scratch. */
static void seq_token_decay_first(int N, double *S, const double *r, const double *w,
                                  const double *k, const double *v, const double *a,
                                  const double *b, double *o, double *h)
{
    for (int i = 0; i < N; ++i)                   /* S = S diag(w) */
        for (int j = 0; j < N; ++j) S[i * N + j] *= w[j];
    for (int i = 0; i < N; ++i) {                 /* h = S a (decayed state) */
        double acc = 0.0;
        for (int j = 0; j < N; ++j) acc += S[i * N + j] * a[j];
        h[i] = acc;
    }
    for (int i = 0; i < N; ++i)                   /* S += h b^T + v k^T */
        for (int j = 0; j < N; ++j) S[i * N + j] += h[i] * b[j] + v[i] * k[j];
    for (int i = 0; i < N; ++i) {                 /* o = S r */
        double acc = 0.0;
        for (int j = 0; j < N; ++j) acc += S[i * N + j] * r[j];
        o[i] = acc;
    }
}

ORACLE_API int wkv7_oracle_sequential_decay_first(int N, int T, double *S, long long base,
                                                  long long tok_stride, const double *r,
                                                  const double *w, const double *k,
                                                  const double *v, const double *a,
                                                  const double *b, double *o)
{
    if (N <= 0 || T < 0) return 1;
    double *h = (double *)malloc(sizeof(double) * (size_t)N);
    if (!h) return 2;
    for (int t = 0; t < T; ++t) {
        long long off = base + (long long)t * tok_stride;
        seq_token_decay_first(N, S, r + off, w + off, k + off, v + off, a + off, b + off,
                              o + off, h);
    }
    free(h);
    return 0;
}

/* Many independent units (heads x sequences, or heads x batch rows), split over
 * n_threads POSIX threads.  Unit u owns S + u*N*N, starts at base[u] and runs
 * T[u] tokens.  Used for batched parity references and for CPU timing. */
typedef struct {
    int N, first, last;
    double *S;
    const long long *base;
    const int *T;
    long long tok_stride;
    const double *r, *w, *k, *v, *a, *b;
    double *o;
    int rc;
} seq_job;

static void *seq_worker(void *arg)
{
    seq_job *j = (seq_job *)arg;
    j->rc = 0;
    for (int u = j->first; u < j->last; ++u) {
        int rc = wkv7_oracle_sequential(j->N, j->T[u], j->S + (size_t)u * j->N * j->N,
                                        j->base[u], j->tok_stride, j->r, j->w, j->k,
                                        j->v, j->a, j->b, j->o);
        if (rc) j->rc = rc;
    }
    return NULL;
}

ORACLE_API int wkv7_oracle_sequential_batch(int N, int n_units, double *S,
                                            const long long *base, const int *T,
                                            long long tok_stride, const double *r,
                                            const double *w, const double *k,
                                            const double *v, const double *a,
                                            const double *b, double *o, int n_threads)
{
    if (n_units < 0 || N <= 0) return 1;
    if (n_threads < 1) n_threads = 1;
    if (n_threads > n_units) n_threads = n_units > 0 ? n_units : 1;
    seq_job *jobs = (seq_job *)calloc((size_t)n_threads, sizeof(seq_job));
    pthread_t *tid = (pthread_t *)calloc((size_t)n_threads, sizeof(pthread_t));
    if (!jobs || !tid) { free(jobs); free(tid); return 2; }
    int rc = 0;
    for (int t = 0; t < n_threads; ++t) {
        seq_job *j = &jobs[t];
        j->N = N; j->S = S; j->base = base; j->T = T; j->tok_stride = tok_stride;
        j->r = r; j->w = w; j->k = k; j->v = v; j->a = a; j->b = b; j->o = o;
        j->first = (int)((long long)n_units * t / n_threads);
        j->last = (int)((long long)n_units * (t + 1) / n_threads);
    }
    int started = 0;
    for (int t = 1; t < n_threads; ++t) {
        if (pthread_create(&tid[t], NULL, seq_worker, &jobs[t]) != 0) { rc = 3; break; }
        started = t;
    }
    seq_worker(&jobs[0]);
    for (int t = 1; t <= started; ++t) pthread_join(tid[t], NULL);
    if (rc == 3) { /* run what could not be started on this thread */
        for (int t = started + 1; t < n_threads; ++t) seq_worker(&jobs[t]);
        rc = 0;
    }
    for (int t = 0; t < n_threads; ++t) if (jobs[t].rc) rc = jobs[t].rc;
    free(jobs); free(tid);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Form 2: chunked (WY/UT) form.                                            */
/*                                                                          */
/* Unrolling the recurrence over a chunk of Lc tokens from start state S0,  */
/* with the relative decay D(s,t] = prod_{s<u<=t} w_u (per key channel,     */
/* D(t,t] = 1), gives for the in-chunk tokens t = 1..Lc:                    */
/*   h_t = S0 (D(0,t-1] . a_t) + sum_{s<t} h_s <b_s . D(s,t-1], a_t>         */
/*                             + sum_{s<t} v_s <k_s . D(s,t-1], a_t>         */
/*   o_t = S0 (D(0,t] . r_t)   + sum_{s<=t} h_s <b_s . D(s,t], r_t>          */
/*                             + sum_{s<=t} v_s <k_s . D(s,t], r_t>          */
/*   S_Lc = S0 diag(D(0,Lc]) + sum_s h_s (b_s . D(s,Lc])^T                   */
/*                          + sum_s v_s (k_s . D(s,Lc])^T                    */
/* With H = [h_1..h_Lc] this reads H (I - Mab) = S0 At + V Mak, where        */
/* Mab[s][t] = <b_s . D(s,t-1], a_t> for s < t (0 otherwise), Mak likewise   */
/* with k, and At[:,t] = D(0,t-1] . a_t.  (I - Mab) is unit upper            */
/* triangular, so T = (I - Mab)^-1 exists; W = At T, U = V Mak T, H = S0 W+U. */
/* Every decay used is a product over s < u <= t, never a quotient.          */
/* ------------------------------------------------------------------------ */

/* D(s,t][j] for 0 <= s <= t <= Lc, tokens of the chunk numbered 1..Lc and
 * the weights of token u at w + (u-1)*stride. */
static double decay(const double *w, long long stride, int s, int t, int j)
{
    double d = 1.0;
    for (int u = s + 1; u <= t; ++u) d *= w[(long long)(u - 1) * stride + j];
    return d;
}

static int chunk_step(int N, int Lc, double *S, long long base, long long ts,
                      const double *r, const double *w, const double *k,
                      const double *v, const double *a, const double *b, double *o)
{
    /* Token u (1-based) of this chunk lives at base + (u-1)*ts. */
    const double *rr = r + base, *ww = w + base, *kk = k + base, *vv = v + base;
    const double *aa = a + base, *bb = b + base;
    double *oo = o + base;
    size_t L = (size_t)Lc, NN = (size_t)N;
    double *Mab = calloc(L * L, sizeof(double));   /* [s][t], 0-based s,t */
    double *Mak = calloc(L * L, sizeof(double));
    double *Qb = calloc(L * L, sizeof(double));
    double *Qk = calloc(L * L, sizeof(double));
    double *Tm = calloc(L * L, sizeof(double));
    double *At = calloc(NN * L, sizeof(double));   /* [j][t] */
    double *Rt = calloc(NN * L, sizeof(double));   /* [j][t] */
    double *W = calloc(NN * L, sizeof(double));    /* [j][t] */
    double *VM = calloc(NN * L, sizeof(double));   /* [i][t] = (V Mak)[i][t] */
    double *U = calloc(NN * L, sizeof(double));    /* [i][t] */
    double *H = calloc(NN * L, sizeof(double));    /* [i][t] */
    double *Sn = calloc(NN * NN, sizeof(double));
    int rc = 0;
    if (!Mab || !Mak || !Qb || !Qk || !Tm || !At || !Rt || !W || !VM || !U || !H || !Sn) {
        rc = 2;
        goto done;
    }
#define X(p, u, j) ((p)[(long long)((u) - 1) * ts + (j)])
    /* Intra-chunk matrices. s, t are 1-based token numbers here. */
    for (int s = 1; s <= Lc; ++s)
        for (int t = s; t <= Lc; ++t) {
            double mab = 0, mak = 0, qb = 0, qk = 0;
            for (int j = 0; j < N; ++j) {
                double d_prev = decay(ww, ts, s, t - 1 >= s ? t - 1 : s, j); /* D(s,t-1], used when s < t */
                double d_cur = decay(ww, ts, s, t, j);                       /* D(s,t] */
                if (s < t) {
                    mab += X(bb, s, j) * d_prev * X(aa, t, j);
                    mak += X(kk, s, j) * d_prev * X(aa, t, j);
                }
                qb += X(bb, s, j) * d_cur * X(rr, t, j);
                qk += X(kk, s, j) * d_cur * X(rr, t, j);
            }
            Mab[(s - 1) * L + (t - 1)] = mab;
            Mak[(s - 1) * L + (t - 1)] = mak;
            Qb[(s - 1) * L + (t - 1)] = qb;
            Qk[(s - 1) * L + (t - 1)] = qk;
        }
    /* Decayed a and r relative to the chunk start. */
    for (int t = 1; t <= Lc; ++t)
        for (int j = 0; j < N; ++j) {
            At[j * L + (t - 1)] = decay(ww, ts, 0, t - 1, j) * X(aa, t, j);
            Rt[j * L + (t - 1)] = decay(ww, ts, 0, t, j) * X(rr, t, j);
        }
    /* UT transform: T = (I - Mab)^-1 by substitution, column by column.
     * (I - Mab) T = I  =>  T[s][t] = [s==t] + sum_{s<u<=t} Mab[s][u] T[u][t]. */
    for (int t = 0; t < Lc; ++t) {
        Tm[t * L + t] = 1.0;
        for (int s = t - 1; s >= 0; --s) {
            double acc = 0.0;
            for (int u = s + 1; u <= t; ++u) acc += Mab[s * L + u] * Tm[u * L + t];
            Tm[s * L + t] = acc;
        }
    }
    /* W = At T */
    for (int j = 0; j < N; ++j)
        for (int t = 0; t < Lc; ++t) {
            double acc = 0.0;
            for (int s = 0; s <= t; ++s) acc += At[j * L + s] * Tm[s * L + t];
            W[j * L + t] = acc;
        }
    /* U = (V Mak) T */
    for (int i = 0; i < N; ++i)
        for (int t = 0; t < Lc; ++t) {
            double acc = 0.0;
            for (int s = 0; s < t; ++s) acc += X(vv, s + 1, i) * Mak[s * L + t];
            VM[i * L + t] = acc;
        }
    for (int i = 0; i < N; ++i)
        for (int t = 0; t < Lc; ++t) {
            double acc = 0.0;
            for (int s = 0; s <= t; ++s) acc += VM[i * L + s] * Tm[s * L + t];
            U[i * L + t] = acc;
        }
    /* H = S0 W + U */
    for (int i = 0; i < N; ++i)
        for (int t = 0; t < Lc; ++t) {
            double acc = U[i * L + t];
            for (int j = 0; j < N; ++j) acc += S[i * N + j] * W[j * L + t];
            H[i * L + t] = acc;
        }
    /* O = S0 Rt + H Qb + V Qk */
    for (int i = 0; i < N; ++i)
        for (int t = 0; t < Lc; ++t) {
            double acc = 0.0;
            for (int j = 0; j < N; ++j) acc += S[i * N + j] * Rt[j * L + t];
            for (int s = 0; s <= t; ++s)
                acc += H[i * L + s] * Qb[s * L + t] + X(vv, s + 1, i) * Qk[s * L + t];
            X(oo, t + 1, i) = acc;
        }
    /* S_Lc = S0 diag(D(0,Lc]) + sum_s h_s (b_s . D(s,Lc])^T + v_s (k_s . D(s,Lc])^T */
    for (int i = 0; i < N; ++i)
        for (int j = 0; j < N; ++j) {
            double acc = S[i * N + j] * decay(ww, ts, 0, Lc, j);
            for (int s = 1; s <= Lc; ++s) {
                double d = decay(ww, ts, s, Lc, j);
                acc += H[i * L + (s - 1)] * X(bb, s, j) * d + X(vv, s, i) * X(kk, s, j) * d;
            }
            Sn[i * N + j] = acc;
        }
    memcpy(S, Sn, NN * NN * sizeof(double));
#undef X
done:
    free(Mab); free(Mak); free(Qb); free(Qk); free(Tm); free(At); free(Rt);
    free(W); free(VM); free(U); free(H); free(Sn);
    return rc;
}

/* Chunks of L tokens anchored at the first token; the last chunk holds the
 * remaining T mod L tokens (or L). */
ORACLE_API int wkv7_oracle_chunked(int N, int T, int L, double *S, long long base,
                                   long long tok_stride, const double *r,
                                   const double *w, const double *k, const double *v,
                                   const double *a, const double *b, double *o)
{
    if (N <= 0 || T < 0 || L <= 0) return 1;
    for (int t0 = 0; t0 < T; t0 += L) {
        int Lc = T - t0 < L ? T - t0 : L;
        int rc = chunk_step(N, Lc, S, base + (long long)t0 * tok_stride, tok_stride,
                            r, w, k, v, a, b, o);
        if (rc) return rc;
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Form 3: matrix products.                                                  */
/*   S_t = S_0 A_1 ... A_t + sum_{s<=t} v_s k_s^T A_{s+1} ... A_t,            */
/*   A_u = diag(w_u) + a_u b_u^T,  o_t = S_t r_t.                             */
/* Every S_t is rebuilt from scratch with dense N x N products: O(T^2 N^3),  */
/* tiny inputs only.                                                         */
/* ------------------------------------------------------------------------ */

static void matmul(int N, const double *X, const double *Y, double *Z)
{
    for (int i = 0; i < N; ++i)
        for (int j = 0; j < N; ++j) {
            double acc = 0.0;
            for (int m = 0; m < N; ++m) acc += X[i * N + m] * Y[m * N + j];
            Z[i * N + j] = acc;
        }
}

ORACLE_API int wkv7_oracle_matprod(int N, int T, double *S, long long base,
                                   long long tok_stride, const double *r,
                                   const double *w, const double *k, const double *v,
                                   const double *a, const double *b, double *o)
{
    if (N <= 0 || T < 0) return 1;
    size_t NN = (size_t)N * N;
    double *S0 = malloc(NN * sizeof(double));
    double *St = malloc(NN * sizeof(double));
    double *P = malloc(NN * sizeof(double));
    double *A = malloc(NN * sizeof(double));
    double *tmp = malloc(NN * sizeof(double));
    double *term = malloc(NN * sizeof(double));
    if (!S0 || !St || !P || !A || !tmp || !term) {
        free(S0); free(St); free(P); free(A); free(tmp); free(term);
        return 2;
    }
    memcpy(S0, S, NN * sizeof(double));
    memcpy(St, S0, NN * sizeof(double));
#define X(p, u, j) ((p)[base + (long long)((u) - 1) * tok_stride + (j)])
    for (int t = 1; t <= T; ++t) {
        /* S_0 A_1 ... A_t */
        memcpy(term, S0, NN * sizeof(double));
        for (int u = 1; u <= t; ++u) {
            for (int i = 0; i < N; ++i)
                for (int j = 0; j < N; ++j)
                    A[i * N + j] = (i == j ? X(w, u, j) : 0.0) + X(a, u, i) * X(b, u, j);
            matmul(N, term, A, tmp);
            memcpy(term, tmp, NN * sizeof(double));
        }
        memcpy(St, term, NN * sizeof(double));
        /* + sum_s v_s k_s^T A_{s+1} ... A_t */
        for (int s = 1; s <= t; ++s) {
            for (int i = 0; i < N; ++i)
                for (int j = 0; j < N; ++j) P[i * N + j] = X(v, s, i) * X(k, s, j);
            for (int u = s + 1; u <= t; ++u) {
                for (int i = 0; i < N; ++i)
                    for (int j = 0; j < N; ++j)
                        A[i * N + j] = (i == j ? X(w, u, j) : 0.0) + X(a, u, i) * X(b, u, j);
                matmul(N, P, A, tmp);
                memcpy(P, tmp, NN * sizeof(double));
            }
            for (size_t e = 0; e < NN; ++e) St[e] += P[e];
        }
        for (int i = 0; i < N; ++i) {
            double acc = 0.0;
            for (int j = 0; j < N; ++j) acc += St[i * N + j] * X(r, t, j);
            X(o, t, i) = acc;
        }
    }
#undef X
    memcpy(S, St, NN * sizeof(double));
    free(S0); free(St); free(P); free(A); free(tmp); free(term);
    return 0;
}
