/*
 * fa_oracle.c -- plain, slow, fp64 CPU oracle for exact attention and its gradients.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path links, loads or calls this
 * file; only the tests, the smoke check and the bench's CPU-baseline leg do. It shares
 * no code, header, table or helper with the CUDA path.
 *
 * What it computes is the plain definition of attention, written out with the score
 * and probability rows materialised (no tiling, no online recurrence, no log2 domain):
 *
 *   S = scale * Q K^T,  P = softmax(S) row-wise,  O = P V
 *   -- "FlashAttention: from IO-Aware Attention to GPU work partitioning"
 *      (blog.euler0525.cn), section "Attention 的性能瓶颈", the definition of S, P, O;
 *      "15. FlashAttention" (inference.shantanugoel.com), section "The score matrix is
 *      the problem".
 *   The softmax is the numerically safe one: subtract the row maximum m, sum
 *   l = sum_j exp(s_j - m), p_j = exp(s_j - m) / l  -- same blog page, section
 *   "Online Softmax", the definitions of m, l and p_j.
 *   LSE_i = m_i + ln l_i  -- same blog page, section "FlashAttention-2", the definition
 *   of L_i; "Lecture 3 -- FlashAttention-1 Algorithm" (jared-hpc.com), the LSE output.
 *
 * Backward (same blog page, section "Tiling、Fusion 与 Backward Recomputation"):
 *   dV = P^T dO,  dP = dO V^T,  D_i = sum_j P_ij dP_ij,  dS = P (.) (dP - D),
 *   dQ = scale * dS K,  dK = scale * dS^T Q.
 *   The page writes dQ = dS K and dK = dS^T Q for S = Q K^T; with S = scale * Q K^T the
 *   chain rule multiplies both by scale (dV carries none). D_i is computed as the sum
 *   over j of P_ij dP_ij, not as O_i . dO_i, so that the page's identity D_i = O_i . dO_i
 *   stays an independent check.
 *
 * Causal masking ("FlashAttention: from IO-Aware ..." section "Tile Size 与 Causal
 * Attention"): key j is visible to query i iff j <= i (equal query and key lengths).
 *
 * Precision: all arithmetic in double. bf16 inputs are widened exactly.
 * Parallelism: independent (batch, head) slices are spread over POSIX threads; each
 * slice is computed by the same sequential code, so results do not depend on the
 * thread count.
 *
 * ORACLE_MUTANT (compile-time, default 0) plants one deliberate mistake so that the
 * pin tests can show that they catch it. Never set in the real oracle build.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

/* ---- input widening ---------------------------------------------------------------- */

static double bf16_to_double(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static void widen(const uint16_t* src, double* dst, long n) {
    for (long i = 0; i < n; ++i) dst[i] = bf16_to_double(src[i]);
}

/* ---- definitions, one head ------------------------------------------------------------ */

static int visible(long i, long j, int causal) {
#if ORACLE_MUTANT == 3
    return causal ? (j <= i + 1) : 1; /* mutant: mask lets one future key through */
#else
    return causal ? (j <= i) : 1;
#endif
}

static double dot(const double* a, const double* b, long d) {
    double s = 0.0;
    for (long e = 0; e < d; ++e) s += a[e] * b[e];
    return s;
}

/* One score: s_ij = scale * q_i . k_j. */
static double score(const double* q, const double* k, long i, long j, long d, double scale) {
#if ORACLE_MUTANT == 1
    (void)scale;
    return dot(q + i * d, k + j * d, d); /* mutant: scale dropped */
#elif ORACLE_MUTANT == 4
    return scale * dot(q + j * d, k + i * d, d); /* mutant: operands transposed */
#else
    return scale * dot(q + i * d, k + j * d, d);
#endif
}

/* Materialise one probability row: prob[j] = softmax(s_i)[j] over visible j, 0 elsewhere.
 * Returns m_i and l_i through the pointers. */
static void prob_row(const double* q, const double* k, long N, long d, int causal, double scale,
                     long i, double* prob, double* m_out, double* l_out) {
    double m = -INFINITY;
    for (long j = 0; j < N; ++j) {
        if (visible(i, j, causal)) {
            prob[j] = score(q, k, i, j, d, scale);
            if (prob[j] > m) m = prob[j];
        }
    }
    double l = 0.0;
#if ORACLE_MUTANT == 2
    long first = 1; /* mutant: one term dropped from the denominator */
#else
    long first = 0;
#endif
    for (long j = first; j < N; ++j)
        if (visible(i, j, causal)) l += exp(prob[j] - m);
    for (long j = 0; j < N; ++j) prob[j] = visible(i, j, causal) ? exp(prob[j] - m) / l : 0.0;
    *m_out = m;
    *l_out = l;
}

static void forward_row(const double* q, const double* k, const double* v, long N, long d,
                        int causal, double scale, long i, double* prob, double* o_row,
                        double* lse) {
    double m, l;
    prob_row(q, k, N, d, causal, scale, i, prob, &m, &l);
    for (long e = 0; e < d; ++e) {
        double acc = 0.0;
        for (long j = 0; j < N; ++j) acc += prob[j] * v[j * d + e];
        o_row[e] = acc;
    }
#if ORACLE_MUTANT == 5
    *lse = log(l); /* mutant: max dropped from the LSE */
#else
    *lse = m + log(l);
#endif
}

/* Full backward of one head with P and dP materialised as N x N matrices. */
static void backward_head(const double* q, const double* k, const double* v, const double* dout,
                          long N, long d, int causal, double scale, double* dq, double* dk,
                          double* dv, double* P, double* dP, double* Dvec) {
    for (long i = 0; i < N; ++i) {
        double m, l;
        prob_row(q, k, N, d, causal, scale, i, P + i * N, &m, &l);
    }
    for (long i = 0; i < N; ++i)
        for (long j = 0; j < N; ++j) dP[i * N + j] = dot(dout + i * d, v + j * d, d);
    for (long i = 0; i < N; ++i) {
        double s = 0.0;
        for (long j = 0; j < N; ++j) {
#if ORACLE_MUTANT == 8
            s += dP[i * N + j]; /* mutant: D without the P weights */
#else
            s += P[i * N + j] * dP[i * N + j];
#endif
        }
        Dvec[i] = s;
    }
    /* dS overwrites dP in place. */
    for (long i = 0; i < N; ++i)
        for (long j = 0; j < N; ++j) dP[i * N + j] = P[i * N + j] * (dP[i * N + j] - Dvec[i]);
    for (long j = 0; j < N; ++j)
        for (long e = 0; e < d; ++e) {
            double a = 0.0, b = 0.0;
            for (long i = 0; i < N; ++i) {
#if ORACLE_MUTANT == 9
                a += P[j * N + i] * dout[i * d + e]; /* mutant: P not transposed */
#else
                a += P[i * N + j] * dout[i * d + e];
#endif
#if ORACLE_MUTANT == 7
                b += dP[i * N + j] * k[i * d + e]; /* mutant: wrong operand for dK */
#else
                b += dP[i * N + j] * q[i * d + e];
#endif
            }
            dv[j * d + e] = a;
            dk[j * d + e] = scale * b;
        }
    for (long i = 0; i < N; ++i)
        for (long e = 0; e < d; ++e) {
            double a = 0.0;
            for (long j = 0; j < N; ++j) a += dP[i * N + j] * k[j * d + e];
#if ORACLE_MUTANT == 6
            dq[i * d + e] = a; /* mutant: scale dropped from dQ */
#else
            dq[i * d + e] = scale * a;
#endif
        }
}

/* ---- thread pool over (batch, head) slices ------------------------------------------- */

typedef struct job job;
typedef void (*slice_fn)(const job* jb, long bh, double* scratch);

struct job {
    slice_fn fn;
    long BH, N, d;
    int causal;
    double scale;
    int in_bf16;
    const void *q, *k, *v, *dout;
    double *o, *lse, *dq, *dk, *dv;
    /* optional (grouped backward): first-order sensitivities of each gradient element to a
       relative perturbation of every P (dV) or dS (dQ, dK) entry it sums; NULL = not wanted */
    double *sq, *sk, *sv;
    const long *rows_q, *rows_k;
    long nrows_q, nrows_k;
    /* extension: grouped KV heads, query offset, sliding window */
    long Hq, Hkv, Tq, Tk, window;
    size_t scratch_doubles;
    long next;
    pthread_mutex_t mu;
    int failed;
};

/* Pointers to one head's [N, d] inputs as doubles (widening bf16 into scratch). */
static const double* head_input(const job* jb, const void* base, long bh, double* buf) {
    long nd = jb->N * jb->d;
    if (jb->in_bf16) {
        widen((const uint16_t*)base + bh * nd, buf, nd);
        return buf;
    }
    return (const double*)base + bh * nd;
}

static void* worker(void* arg) {
    job* jb = (job*)arg;
    double* scratch = (double*)malloc(jb->scratch_doubles * sizeof(double) + 64);
    if (!scratch) {
        pthread_mutex_lock(&jb->mu);
        jb->failed = 1;
        pthread_mutex_unlock(&jb->mu);
        return NULL;
    }
    for (;;) {
        pthread_mutex_lock(&jb->mu);
        long bh = jb->next++;
        pthread_mutex_unlock(&jb->mu);
        if (bh >= jb->BH) break;
        jb->fn(jb, bh, scratch);
    }
    free(scratch);
    return NULL;
}

static int run_job(job* jb, int nthreads) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > jb->BH) nthreads = (int)(jb->BH > 0 ? jb->BH : 1);
    jb->next = 0;
    jb->failed = 0;
    pthread_mutex_init(&jb->mu, NULL);
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!th) return -1;
    int started = 0;
    for (int t = 0; t < nthreads; ++t)
        if (pthread_create(&th[t], NULL, worker, jb) == 0) ++started;
    if (started == 0) worker(jb);
    for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
    free(th);
    pthread_mutex_destroy(&jb->mu);
    return jb->failed ? -1 : 0;
}

/* ---- forward ---------------------------------------------------------------------------- */

static void fwd_slice(const job* jb, long bh, double* scratch) {
    long N = jb->N, d = jb->d, nd = N * d;
    double* prob = scratch;
    double* bufq = prob + N;
    double* bufk = bufq + nd;
    double* bufv = bufk + nd;
    const double* q = head_input(jb, jb->q, bh, bufq);
    const double* k = head_input(jb, jb->k, bh, bufk);
    const double* v = head_input(jb, jb->v, bh, bufv);
    long nr = jb->rows_q ? jb->nrows_q : N;
    for (long r = 0; r < nr; ++r) {
        long i = jb->rows_q ? jb->rows_q[r] : r;
        forward_row(q, k, v, N, d, jb->causal, jb->scale, i, prob, jb->o + (bh * nr + r) * d,
                    jb->lse + bh * nr + r);
    }
}

static int forward_common(int in_bf16, const void* q, const void* k, const void* v, double* o,
                          double* lse, long B, long H, long N, long d, int causal, double scale,
                          const long* rows, long nrows, int nthreads) {
    if (B < 0 || H < 0 || N < 0 || d < 1) return -2;
    job jb;
    memset(&jb, 0, sizeof jb);
    jb.fn = fwd_slice;
    jb.BH = B * H;
    jb.N = N;
    jb.d = d;
    jb.causal = causal;
    jb.scale = scale;
    jb.in_bf16 = in_bf16;
    jb.q = q;
    jb.k = k;
    jb.v = v;
    jb.o = o;
    jb.lse = lse;
    jb.rows_q = rows;
    jb.nrows_q = nrows;
    jb.scratch_doubles = (size_t)N + (in_bf16 ? 3 * (size_t)N * (size_t)d : 0);
    if (jb.BH == 0 || N == 0) return 0;
    return run_job(&jb, nthreads);
}

/* O [B,H,N,d] and LSE [B,H,N] for every query row; inputs are bf16 bit patterns. */
int fa_oracle_forward_bf16(const uint16_t* q, const uint16_t* k, const uint16_t* v, double* o,
                           double* lse, long B, long H, long N, long d, int causal, double scale,
                           int nthreads) {
    return forward_common(1, q, k, v, o, lse, B, H, N, d, causal, scale, NULL, 0, nthreads);
}

/* Same, on the query rows listed in rows[0..nrows) of every (b,h):
 * o is [B*H, nrows, d], lse is [B*H, nrows]. */
int fa_oracle_forward_rows_bf16(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                double* o, double* lse, long B, long H, long N, long d,
                                int causal, double scale, const long* rows, long nrows,
                                int nthreads) {
    for (long r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= N) return -2;
    return forward_common(1, q, k, v, o, lse, B, H, N, d, causal, scale, rows, nrows, nthreads);
}

/* float64 inputs (used for finite differences and closed-form checks). */
int fa_oracle_forward_f64(const double* q, const double* k, const double* v, double* o,
                          double* lse, long B, long H, long N, long d, int causal, double scale,
                          int nthreads) {
    return forward_common(0, q, k, v, o, lse, B, H, N, d, causal, scale, NULL, 0, nthreads);
}

/* The materialised probability matrix P [B,H,N,N] (float64 inputs, small cases). */
static void prob_slice(const job* jb, long bh, double* scratch) {
    (void)scratch;
    long N = jb->N, d = jb->d, nd = N * d;
    const double* q = (const double*)jb->q + bh * nd;
    const double* k = (const double*)jb->k + bh * nd;
    for (long i = 0; i < N; ++i) {
        double m, l;
        prob_row(q, k, N, d, jb->causal, jb->scale, i, jb->o + (bh * N + i) * N, &m, &l);
    }
}

int fa_oracle_probs_f64(const double* q, const double* k, double* P, long B, long H, long N,
                        long d, int causal, double scale, int nthreads) {
    if (B < 0 || H < 0 || N < 0 || d < 1) return -2;
    job jb;
    memset(&jb, 0, sizeof jb);
    jb.fn = prob_slice;
    jb.BH = B * H;
    jb.N = N;
    jb.d = d;
    jb.causal = causal;
    jb.scale = scale;
    jb.q = q;
    jb.k = k;
    jb.o = P;
    jb.scratch_doubles = 1;
    if (jb.BH == 0 || N == 0) return 0;
    return run_job(&jb, nthreads);
}

/* ---- backward ------------------------------------------------------------------------- */

static void bwd_slice(const job* jb, long bh, double* scratch) {
    long N = jb->N, d = jb->d, nd = N * d, NN = N * N;
    double* P = scratch;
    double* dP = P + NN;
    double* Dv = dP + NN;
    double* bufs = Dv + N;
    const double* q = head_input(jb, jb->q, bh, bufs);
    const double* k = head_input(jb, jb->k, bh, bufs + nd);
    const double* v = head_input(jb, jb->v, bh, bufs + 2 * nd);
    const double* dout = head_input(jb, jb->dout, bh, bufs + 3 * nd);
    backward_head(q, k, v, dout, N, d, jb->causal, jb->scale, jb->dq + bh * nd, jb->dk + bh * nd,
                  jb->dv + bh * nd, P, dP, Dv);
}

static int backward_common(int in_bf16, const void* q, const void* k, const void* v,
                           const void* dout, double* dq, double* dk, double* dv, long B, long H,
                           long N, long d, int causal, double scale, int nthreads) {
    if (B < 0 || H < 0 || N < 0 || d < 1) return -2;
    job jb;
    memset(&jb, 0, sizeof jb);
    jb.fn = bwd_slice;
    jb.BH = B * H;
    jb.N = N;
    jb.d = d;
    jb.causal = causal;
    jb.scale = scale;
    jb.in_bf16 = in_bf16;
    jb.q = q;
    jb.k = k;
    jb.v = v;
    jb.dout = dout;
    jb.dq = dq;
    jb.dk = dk;
    jb.dv = dv;
    jb.scratch_doubles = 2 * (size_t)N * (size_t)N + (size_t)N + (in_bf16 ? 4 * (size_t)N * (size_t)d : 0);
    if (jb.BH == 0 || N == 0) return 0;
    return run_job(&jb, nthreads);
}

/* dQ, dK, dV [B,H,N,d] of L = sum(O (.) dO); inputs are bf16 bit patterns. */
int fa_oracle_backward_bf16(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                            const uint16_t* dout, double* dq, double* dk, double* dv, long B,
                            long H, long N, long d, int causal, double scale, int nthreads) {
    return backward_common(1, q, k, v, dout, dq, dk, dv, B, H, N, d, causal, scale, nthreads);
}

int fa_oracle_backward_f64(const double* q, const double* k, const double* v, const double* dout,
                           double* dq, double* dk, double* dv, long B, long H, long N, long d,
                           int causal, double scale, int nthreads) {
    return backward_common(0, q, k, v, dout, dq, dk, dv, B, H, N, d, causal, scale, nthreads);
}

/* Sampled backward for sizes where N x N matrices per head are too large.
 * dQ on the query rows rows_q[0..nq) -> dq [B*H, nq, d];
 * dK, dV on the key rows rows_k[0..nk) -> dk, dv [B*H, nk, d].
 * Every row statistic (m_i, l_i, D_i) is computed for all N query rows from the same
 * definitions as above, one materialised row at a time. */
static void bwd_rows_slice(const job* jb, long bh, double* scratch) {
    long N = jb->N, d = jb->d, nd = N * d;
    double* prob = scratch;
    double* dprow = prob + N;
    double* mrow = dprow + N;
    double* lrow = mrow + N;
    double* Dv = lrow + N;
    double* bufs = Dv + N;
    const double* q = head_input(jb, jb->q, bh, bufs);
    const double* k = head_input(jb, jb->k, bh, bufs + nd);
    const double* v = head_input(jb, jb->v, bh, bufs + 2 * nd);
    const double* dout = head_input(jb, jb->dout, bh, bufs + 3 * nd);
    int causal = jb->causal;
    double scale = jb->scale;
    /* Row statistics for every query row. */
    for (long i = 0; i < N; ++i) {
        prob_row(q, k, N, d, causal, scale, i, prob, &mrow[i], &lrow[i]);
        double s = 0.0;
        for (long j = 0; j < N; ++j)
            if (prob[j] != 0.0) s += prob[j] * dot(dout + i * d, v + j * d, d);
        Dv[i] = s;
    }
    /* dQ rows. */
    for (long r = 0; r < jb->nrows_q; ++r) {
        long i = jb->rows_q[r];
        double m, l;
        prob_row(q, k, N, d, causal, scale, i, prob, &m, &l);
        for (long j = 0; j < N; ++j) dprow[j] = prob[j] * (dot(dout + i * d, v + j * d, d) - Dv[i]);
        double* out = jb->dq + (bh * jb->nrows_q + r) * d;
        for (long e = 0; e < d; ++e) {
            double a = 0.0;
            for (long j = 0; j < N; ++j) a += dprow[j] * k[j * d + e];
            out[e] = scale * a;
        }
    }
    /* dK, dV rows: column j of P and dS, rebuilt from the row statistics. */
    for (long r = 0; r < jb->nrows_k; ++r) {
        long j = jb->rows_k[r];
        for (long i = 0; i < N; ++i) {
            if (!visible(i, j, causal)) {
                prob[i] = 0.0;
                dprow[i] = 0.0;
                continue;
            }
            double p = exp(score(q, k, i, j, d, scale) - mrow[i]) / lrow[i];
            prob[i] = p;
            dprow[i] = p * (dot(dout + i * d, v + j * d, d) - Dv[i]);
        }
        double* odk = jb->dk + (bh * jb->nrows_k + r) * d;
        double* odv = jb->dv + (bh * jb->nrows_k + r) * d;
        for (long e = 0; e < d; ++e) {
            double a = 0.0, b = 0.0;
            for (long i = 0; i < N; ++i) {
                a += prob[i] * dout[i * d + e];
                b += dprow[i] * q[i * d + e];
            }
            odv[e] = a;
            odk[e] = scale * b;
        }
    }
}

int fa_oracle_backward_rows_bf16(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                 const uint16_t* dout, double* dq, double* dk, double* dv, long B,
                                 long H, long N, long d, int causal, double scale,
                                 const long* rows_q, long nq, const long* rows_k, long nk,
                                 int nthreads) {
    if (B < 0 || H < 0 || N < 0 || d < 1) return -2;
    for (long r = 0; r < nq; ++r)
        if (rows_q[r] < 0 || rows_q[r] >= N) return -2;
    for (long r = 0; r < nk; ++r)
        if (rows_k[r] < 0 || rows_k[r] >= N) return -2;
    job jb;
    memset(&jb, 0, sizeof jb);
    jb.fn = bwd_rows_slice;
    jb.BH = B * H;
    jb.N = N;
    jb.d = d;
    jb.causal = causal;
    jb.scale = scale;
    jb.in_bf16 = 1;
    jb.q = q;
    jb.k = k;
    jb.v = v;
    jb.dout = dout;
    jb.dq = dq;
    jb.dk = dk;
    jb.dv = dv;
    jb.rows_q = rows_q;
    jb.nrows_q = nq;
    jb.rows_k = rows_k;
    jb.nrows_k = nk;
    jb.scratch_doubles = 5 * (size_t)N + 4 * (size_t)N * (size_t)d;
    if (jb.BH == 0 || N == 0) return 0;
    return run_job(&jb, nthreads);
}

/* ---- extension: grouped KV heads, query offset, sliding window ------------------------
 *
 * "15. FlashAttention" (inference.shantanugoel.com), section "The algorithm in plain
 * PyTorch": query head h reads KV head h / (Hq / Hkv) (grouped-query attention); query row i
 * sits at position (Tk - Tq) + i, so the last query lines up with the last key; key j is
 * visible iff j <= position (causal). Section "Stretch exercises", item 3 (sliding window):
 * tiles wholly before position - window are skipped, i.e. with a window key j is visible only
 * if j >= position - window. A row with no visible key is an error (the page raises).
 * Same definitions as above otherwise: materialised score row, safe softmax, O = P V,
 * LSE = m + ln l; dK, dV of a KV head add up the contributions of all its query heads.
 */

static int visible_ex(long pos, long j, int causal, long window) {
    if (causal && j > pos) return 0;
    if (window >= 0 && j < pos - window) return 0;
    return 1;
}

/* prob[j] for j < Tk; returns 0 if the row has no visible key. */
static int prob_row_ex(const double* qrow, const double* k, long Tk, long d, long pos, int causal,
                       long window, double scale, double* prob, double* m_out, double* l_out) {
    double m = -INFINITY;
    long nvis = 0;
    for (long j = 0; j < Tk; ++j) {
        if (visible_ex(pos, j, causal, window)) {
            prob[j] = scale * dot(qrow, k + j * d, d);
            if (prob[j] > m) m = prob[j];
            ++nvis;
        }
    }
    if (nvis == 0) return 0;
    double l = 0.0;
    for (long j = 0; j < Tk; ++j)
        if (visible_ex(pos, j, causal, window)) l += exp(prob[j] - m);
    for (long j = 0; j < Tk; ++j)
        prob[j] = visible_ex(pos, j, causal, window) ? exp(prob[j] - m) / l : 0.0;
    *m_out = m;
    *l_out = l;
    return 1;
}

static const double* slice_input(const job* jb, const void* base, long idx, long rows, double* buf) {
    long n = rows * jb->d;
    if (jb->in_bf16) {
        widen((const uint16_t*)base + idx * n, buf, n);
        return buf;
    }
    return (const double*)base + idx * n;
}

/* One (batch, KV head) slice: every query head of its group. */
static void fwd_ex_slice(const job* jb, long bkv, double* scratch) {
    long d = jb->d, Tq = jb->Tq, Tk = jb->Tk, group = jb->Hq / jb->Hkv;
    long b = bkv / jb->Hkv, hk = bkv % jb->Hkv;
    double* prob = scratch;
    double* bufk = prob + Tk;
    double* bufv = bufk + Tk * d;
    double* bufq = bufv + Tk * d;
    const double* k = slice_input(jb, jb->k, bkv, Tk, bufk);
    const double* v = slice_input(jb, jb->v, bkv, Tk, bufv);
    for (long g = 0; g < group; ++g) {
        long bhq = b * jb->Hq + hk * group + g;
        const double* q = slice_input(jb, jb->q, bhq, Tq, bufq);
        for (long i = 0; i < Tq; ++i) {
            double m, l;
            long pos = (Tk - Tq) + i;
            if (!prob_row_ex(q + i * d, k, Tk, d, pos, jb->causal, jb->window, jb->scale, prob, &m, &l)) {
                ((job*)jb)->failed = 1;
                return;
            }
            double* orow = jb->o + (bhq * Tq + i) * d;
            for (long e = 0; e < d; ++e) {
                double acc = 0.0;
                for (long j = 0; j < Tk; ++j) acc += prob[j] * v[j * d + e];
                orow[e] = acc;
            }
            jb->lse[bhq * Tq + i] = m + log(l);
        }
    }
}

static void bwd_ex_slice(const job* jb, long bkv, double* scratch) {
    long d = jb->d, Tq = jb->Tq, Tk = jb->Tk, group = jb->Hq / jb->Hkv;
    long b = bkv / jb->Hkv, hk = bkv % jb->Hkv;
    double* P = scratch;            /* Tq x Tk */
    double* dS = P + Tq * Tk;       /* Tq x Tk (dP, then dS in place) */
    double* Dv = dS + Tq * Tk;
    double* bufk = Dv + Tq;
    double* bufv = bufk + Tk * d;
    double* bufq = bufv + Tk * d;
    double* bufo = bufq + Tq * d;
    const double* k = slice_input(jb, jb->k, bkv, Tk, bufk);
    const double* v = slice_input(jb, jb->v, bkv, Tk, bufv);
    double* dk = jb->dk + bkv * Tk * d;
    double* dv = jb->dv + bkv * Tk * d;
    for (long x = 0; x < Tk * d; ++x) dk[x] = dv[x] = 0.0;
    if (jb->sv)
        for (long x = 0; x < Tk * d; ++x) jb->sk[bkv * Tk * d + x] = jb->sv[bkv * Tk * d + x] = 0.0;
    for (long g = 0; g < group; ++g) {
        long bhq = b * jb->Hq + hk * group + g;
        const double* q = slice_input(jb, jb->q, bhq, Tq, bufq);
        const double* dout = slice_input(jb, jb->dout, bhq, Tq, bufo);
        for (long i = 0; i < Tq; ++i) {
            double m, l;
            if (!prob_row_ex(q + i * d, k, Tk, d, (Tk - Tq) + i, jb->causal, jb->window, jb->scale,
                             P + i * Tk, &m, &l)) {
                ((job*)jb)->failed = 1;
                return;
            }
        }
        for (long i = 0; i < Tq; ++i)
            for (long j = 0; j < Tk; ++j) dS[i * Tk + j] = dot(dout + i * d, v + j * d, d);
        for (long i = 0; i < Tq; ++i) {
            double s = 0.0;
            for (long j = 0; j < Tk; ++j) s += P[i * Tk + j] * dS[i * Tk + j];
            Dv[i] = s;
        }
        for (long i = 0; i < Tq; ++i)
            for (long j = 0; j < Tk; ++j) dS[i * Tk + j] = P[i * Tk + j] * (dS[i * Tk + j] - Dv[i]);
        for (long j = 0; j < Tk; ++j)
            for (long e = 0; e < d; ++e) {
                double a = 0.0, c = 0.0;
                for (long i = 0; i < Tq; ++i) {
                    a += P[i * Tk + j] * dout[i * d + e];
                    c += dS[i * Tk + j] * q[i * d + e];
                }
                dv[j * d + e] += a;
                dk[j * d + e] += jb->scale * c;
            }
        double* dq = jb->dq + bhq * Tq * d;
        for (long i = 0; i < Tq; ++i)
            for (long e = 0; e < d; ++e) {
                double a = 0.0;
                for (long j = 0; j < Tk; ++j) a += dS[i * Tk + j] * k[j * d + e];
                dq[i * d + e] = jb->scale * a;
            }
        if (jb->sv) {
            /* Sensitivities: if every P_ij (resp. dS_ij) is perturbed by a relative amount of
               at most u, dV_je moves by at most u * sv_je, dK_je by u * sk_je and dQ_ie by
               u * sq_ie, where sv_je = sum_i P_ij |dO_ie|, sk_je = scale sum_i |dS_ij| |q_ie|,
               sq_ie = scale sum_j |dS_ij| |k_je| (the triangle inequality on the sums above).
               Summed over the query heads of the group like dK and dV. */
            double* sv = jb->sv + bkv * Tk * d;
            double* sk = jb->sk + bkv * Tk * d;
            double* sq = jb->sq + bhq * Tq * d;
            for (long j = 0; j < Tk; ++j)
                for (long e = 0; e < d; ++e) {
                    double a = 0.0, c = 0.0;
                    for (long i = 0; i < Tq; ++i) {
                        a += P[i * Tk + j] * fabs(dout[i * d + e]);
                        c += fabs(dS[i * Tk + j]) * fabs(q[i * d + e]);
                    }
                    sv[j * d + e] += a;
                    sk[j * d + e] += jb->scale * c;
                }
            for (long i = 0; i < Tq; ++i)
                for (long e = 0; e < d; ++e) {
                    double a = 0.0;
                    for (long j = 0; j < Tk; ++j) a += fabs(dS[i * Tk + j]) * fabs(k[j * d + e]);
                    sq[i * d + e] = jb->scale * a;
                }
        }
    }
}

static int ex_common(int in_bf16, int backward, const void* q, const void* k, const void* v,
                     const void* dout, double* o, double* lse, double* dq, double* dk, double* dv,
                     double* sq, double* sk, double* sv,
                     long B, long Hq, long Hkv, long Tq, long Tk, long d, int causal, long window,
                     double scale, int nthreads) {
    if (B < 0 || Hq < 0 || Hkv < 1 || Tq < 0 || Tk < 0 || d < 1) return -2;
    if (Hq % Hkv != 0) return -2;
    if (window >= 0 && !causal) return -2;
    job jb;
    memset(&jb, 0, sizeof jb);
    jb.fn = backward ? bwd_ex_slice : fwd_ex_slice;
    jb.BH = B * Hkv;
    jb.N = Tk;
    jb.d = d;
    jb.causal = causal;
    jb.scale = scale;
    jb.in_bf16 = in_bf16;
    jb.q = q;
    jb.k = k;
    jb.v = v;
    jb.dout = dout;
    jb.o = o;
    jb.lse = lse;
    jb.dq = dq;
    jb.dk = dk;
    jb.dv = dv;
    jb.sq = sq;
    jb.sk = sk;
    jb.sv = sv;
    jb.Hq = Hq;
    jb.Hkv = Hkv;
    jb.Tq = Tq;
    jb.Tk = Tk;
    jb.window = window;
    jb.scratch_doubles = backward ? 2 * (size_t)Tq * (size_t)Tk + (size_t)Tq + 2 * (size_t)Tk * (size_t)d + 2 * (size_t)Tq * (size_t)d
                                  : (size_t)Tk + 2 * (size_t)Tk * (size_t)d + (size_t)Tq * (size_t)d;
    if (jb.BH == 0 || Tq == 0 || Hq == 0) return 0;
    if (Tk == 0) return -3;
    int rc = run_job(&jb, nthreads);
    return rc == 0 ? 0 : -3;
}

/* O [B,Hq,Tq,d], LSE [B,Hq,Tq] from q [B,Hq,Tq,d], k/v [B,Hkv,Tk,d] (float64 inputs).
 * window < 0: none; window >= 0 needs causal. Returns -3 if a row has no visible key. */
int fa_oracle_forward_ex_f64(const double* q, const double* k, const double* v, double* o,
                             double* lse, long B, long Hq, long Hkv, long Tq, long Tk, long d,
                             int causal, long window, double scale, int nthreads) {
    return ex_common(0, 0, q, k, v, NULL, o, lse, NULL, NULL, NULL, NULL, NULL, NULL, B, Hq, Hkv, Tq, Tk, d, causal,
                     window, scale, nthreads);
}

int fa_oracle_forward_ex_bf16(const uint16_t* q, const uint16_t* k, const uint16_t* v, double* o,
                              double* lse, long B, long Hq, long Hkv, long Tq, long Tk, long d,
                              int causal, long window, double scale, int nthreads) {
    return ex_common(1, 0, q, k, v, NULL, o, lse, NULL, NULL, NULL, NULL, NULL, NULL, B, Hq, Hkv, Tq, Tk, d, causal,
                     window, scale, nthreads);
}

/* dQ [B,Hq,Tq,d], dK/dV [B,Hkv,Tk,d] of L = sum(O (.) dO). */
int fa_oracle_backward_ex_f64(const double* q, const double* k, const double* v, const double* dout,
                              double* dq, double* dk, double* dv, long B, long Hq, long Hkv, long Tq,
                              long Tk, long d, int causal, long window, double scale, int nthreads) {
    return ex_common(0, 1, q, k, v, dout, NULL, NULL, dq, dk, dv, NULL, NULL, NULL, B, Hq, Hkv, Tq, Tk, d, causal,
                     window, scale, nthreads);
}

int fa_oracle_backward_ex_bf16(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                               const uint16_t* dout, double* dq, double* dk, double* dv, long B,
                               long Hq, long Hkv, long Tq, long Tk, long d, int causal, long window,
                               double scale, int nthreads) {
    return ex_common(1, 1, q, k, v, dout, NULL, NULL, dq, dk, dv, NULL, NULL, NULL, B, Hq, Hkv, Tq, Tk, d, causal,
                     window, scale, nthreads);
}

/* backward_ex_bf16 plus the sensitivities sq [B,Hq,Tq,d], sk, sv [B,Hkv,Tk,d] (see
 * bwd_ex_slice): the bound on how far each gradient element can move when every P_ij (dV) or
 * dS_ij (dQ, dK) it sums carries a relative error of at most u is u times its sensitivity. */
int fa_oracle_backward_ex_sens_bf16(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                    const uint16_t* dout, double* dq, double* dk, double* dv,
                                    double* sq, double* sk, double* sv, long B, long Hq, long Hkv,
                                    long Tq, long Tk, long d, int causal, long window, double scale,
                                    int nthreads) {
    return ex_common(1, 1, q, k, v, dout, NULL, NULL, dq, dk, dv, sq, sk, sv, B, Hq, Hkv, Tq, Tk,
                     d, causal, window, scale, nthreads);
}

int fa_oracle_mutant_id(void) { return ORACLE_MUTANT; }
