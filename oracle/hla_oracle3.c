/*
 * hla_oracle3.c -- fp64 CPU oracle for masked third-order Higher-order Linear
 * Attention.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite and the CPU legs of
 * the benchmark load this file.  It shares no code, header, table or helper with
 * the CUDA library.
 *
 * Source: "Higher-order Linear Attention", gist.science technical summary,
 * section 3 "Derde-orde HLA" (the operator A A^T A with A = Q K^T; the masked
 * output keeps the prefix moments S^K, S^Q, P^KV and cross summaries G^(1..3))
 * and section 4, bullet "Derde-orde scans" (segment-level linear maps compose
 * third-order states exactly).  The pages print no formula; the readings below
 * are the plainest ones the section supports.
 *
 * Masked output (every factor of A A^T A causal):
 *   o_t = sum_{b<=t} sum_{a<=b} sum_{c<=b} (q_t.k_a)(k_a.q_b)(q_b.k_c) v_c,
 * i.e. O = [ (L o ((L o A)(L o A)^T)) (L o A) ] V.
 *
 * Prefix moments:  S^K_t = sum k k^T,  S^Q_t = sum q q^T,  P_t = sum k v^T.
 * Their product S^K S^Q P sums over all a, b, c <= t; the masked output keeps
 * a <= b and c <= b.  By inclusion-exclusion over the two forbidden orders,
 *   o_t = q_t^T (S^K_t S^Q_t P_t - G1_t - G2_t + G3_t),
 *   G1_t = sum_{a>b} k_a k_a^T q_b q_b^T k_c v_c^T   (key a after the query b)
 *   G2_t = sum_{c>b} ...                             (key c after the query b)
 *   G3_t = sum_{a>b, c>b} ...                        (both)
 * updated online with two auxiliary products,
 *   Z1_t = sum_{b<a<=t} k_a k_a^T q_b q_b^T  (d x d),  Z2_t = sum_{b<c<=t} q_b q_b^T k_c v_c^T  (d x dv):
 *   Z1_t = Z1 + k (k^T S^Q_{t-1}),        Z2_t = Z2 + (S^Q_{t-1} k) v^T,
 *   G1_t = G1 + (Z1_{t-1} k) v^T + k (k^T S^Q_{t-1} P_t)        (= Z1_t P_t),
 *   G2_t = G2 + k (k^T Z2_t) + (S^K_{t-1} S^Q_{t-1} k) v^T      (= S^K_t Z2_t),
 *   G3_t = G3 + k (k^T Z2_t) + (Z1_t k) v^T - (k^T S^Q_{t-1} k) k v^T.
 *
 * Segment summaries and their concatenation (segment A before B):
 *   T = S^K S^Q P - G1 - G2 + G3 = sum_{b} S^K_{<=b} q_b q_b^T P_{<=b}     (d x dv)
 *   M^QP = sum_b q_b q_b^T P_{<=b}   (d x dv),   M^KQ = sum_b S^K_{<=b} q_b q_b^T  (d x d)
 *   S^K, S^Q, P add;
 *   T    = T_A + T_B + S^K_A M^QP_B + M^KQ_B P_A + S^K_A S^Q_B P_A,
 *   M^QP = M^QP_A + M^QP_B + S^Q_B P_A,
 *   M^KQ = M^KQ_A + M^KQ_B + S^K_A S^Q_B.
 * The maps P -> M^KQ_B P and P -> S^K_A M^QP_B are the segment-level linear maps
 * the section names (M^KQP; M^KQm is the same map applied to a key mass, which
 * the unnormalised output does not need).
 *
 * Scope: no decay and no normalisation (the section states neither for the third
 * order).
 *
 * State layout per (b,h), doubles, in this order:
 *   SK d*d, SQ d*d, Z1 d*d, MKQ d*d, P d*dv, Z2 d*dv, G1 d*dv, G2 d*dv, G3 d*dv,
 *   T d*dv, MQP d*dv   (4 d^2 + 7 d dv).
 * T is derived (S^K S^Q P - G1 - G2 + G3) and ignored on input.  The chunked path
 * carries only S^K, S^Q, P, T, M^QP, M^KQ; it writes Z1, Z2, G1, G2, G3 as NaN.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int d, dv;
    double *SK, *SQ, *Z1, *MKQ, *P, *Z2, *G1, *G2, *G3, *T, *MQP;
    double *w1, *w2, *w3, *w4, *w5, *wv1, *wv2, *wd;  /* scratch */
} st3_t;

static size_t st3_size(int d, int dv) { return 4 * (size_t)d * d + 7 * (size_t)d * dv; }

static void st3_bind(st3_t *s, double *base, int d, int dv)
{
    const size_t dd = (size_t)d * d, dvv = (size_t)d * dv;
    s->d = d; s->dv = dv;
    s->SK = base; s->SQ = base + dd; s->Z1 = base + 2 * dd; s->MKQ = base + 3 * dd;
    s->P = base + 4 * dd; s->Z2 = s->P + dvv; s->G1 = s->Z2 + dvv; s->G2 = s->G1 + dvv;
    s->G3 = s->G2 + dvv; s->T = s->G3 + dvv; s->MQP = s->T + dvv;
}

static void st3_scratch(st3_t *s)
{
    const int d = s->d, dv = s->dv, w = d > dv ? d : dv;
    s->w1 = calloc((size_t)w, sizeof(double)); s->w2 = calloc((size_t)w, sizeof(double));
    s->w3 = calloc((size_t)w, sizeof(double)); s->w4 = calloc((size_t)w, sizeof(double));
    s->w5 = calloc((size_t)w, sizeof(double)); s->wv1 = calloc((size_t)w, sizeof(double));
    s->wv2 = calloc((size_t)w, sizeof(double));
    s->wd = calloc((size_t)d * (d > dv ? d : dv), sizeof(double));
}

static void st3_free_scratch(st3_t *s)
{
    free(s->w1); free(s->w2); free(s->w3); free(s->w4); free(s->w5); free(s->wv1); free(s->wv2); free(s->wd);
}

/* T = S^K S^Q P - G1 - G2 + G3 */
static void derive_T(st3_t *s)
{
    const int d = s->d, dv = s->dv;
    double *SKSQ = s->wd;  /* d x d */
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < d; ++j) {
            double acc = 0.0;
            for (int l = 0; l < d; ++l) acc += s->SK[i * d + l] * s->SQ[l * d + j];
            SKSQ[i * d + j] = acc;
        }
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int l = 0; l < d; ++l) acc += SKSQ[i * d + l] * s->P[l * dv + j];
            s->T[i * dv + j] = acc - s->G1[i * dv + j] - s->G2[i * dv + j] + s->G3[i * dv + j];
        }
}

/* one token of the serial recurrence in the moments and cross summaries; o: dv */
static void step3(st3_t *s, const double *q, const double *k, const double *v, double *o)
{
    const int d = s->d, dv = s->dv;
    double *sqk = s->w1, *ksq = s->w2, *z1k = s->w3, *sksqk = s->w4, *z1tk = s->w5;
    double *kz2 = s->wv1, *ksqp = s->wv2;
    /* values before the token: S^Q_{t-1} k, k^T S^Q_{t-1}, Z1_{t-1} k, S^K_{t-1} S^Q_{t-1} k */
    double ksqk = 0.0;
    for (int i = 0; i < d; ++i) {
        double a = 0.0, b = 0.0, c = 0.0;
        for (int j = 0; j < d; ++j) {
            a += s->SQ[i * d + j] * k[j];
            b += k[j] * s->SQ[j * d + i];
            c += s->Z1[i * d + j] * k[j];
        }
        sqk[i] = a; ksq[i] = b; z1k[i] = c;
    }
    for (int i = 0; i < d; ++i) {
        double a = 0.0;
        for (int j = 0; j < d; ++j) a += s->SK[i * d + j] * sqk[j];
        sksqk[i] = a;
        ksqk += k[i] * sqk[i];
    }
    /* P_t */
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < dv; ++j) s->P[i * dv + j] += k[i] * v[j];
    /* Z1_t, Z2_t */
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < d; ++j) s->Z1[i * d + j] += k[i] * ksq[j];
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < dv; ++j) s->Z2[i * dv + j] += sqk[i] * v[j];
    /* k^T S^Q_{t-1} P_t, k^T Z2_t, Z1_t k */
    for (int j = 0; j < dv; ++j) {
        double a = 0.0, b = 0.0;
        for (int i = 0; i < d; ++i) {
            a += ksq[i] * s->P[i * dv + j];
            b += k[i] * s->Z2[i * dv + j];
        }
        ksqp[j] = a; kz2[j] = b;
    }
    for (int i = 0; i < d; ++i) {
        double a = 0.0;
        for (int j = 0; j < d; ++j) a += s->Z1[i * d + j] * k[j];
        z1tk[i] = a;
    }
    /* cross summaries */
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < dv; ++j) {
            s->G1[i * dv + j] += z1k[i] * v[j] + k[i] * ksqp[j];
            s->G2[i * dv + j] += k[i] * kz2[j] + sksqk[i] * v[j];
            s->G3[i * dv + j] += k[i] * kz2[j] + z1tk[i] * v[j] - ksqk * k[i] * v[j];
        }
    /* S^K_t, S^Q_t */
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < d; ++j) {
            s->SK[i * d + j] += k[i] * k[j];
            s->SQ[i * d + j] += q[i] * q[j];
        }
    /* M^QP += q (q^T P_t);  M^KQ += (S^K_t q) q^T */
    for (int j = 0; j < dv; ++j) {
        double a = 0.0;
        for (int i = 0; i < d; ++i) a += q[i] * s->P[i * dv + j];
        for (int i = 0; i < d; ++i) s->MQP[i * dv + j] += q[i] * a;
    }
    for (int i = 0; i < d; ++i) {
        double a = 0.0;
        for (int j = 0; j < d; ++j) a += s->SK[i * d + j] * q[j];
        for (int j = 0; j < d; ++j) s->MKQ[i * d + j] += a * q[j];
    }
    /* o_t = ((q^T S^K) S^Q) P - q^T G1 - q^T G2 + q^T G3 */
    double *qsk = s->w1, *qsksq = s->w2;
    for (int j = 0; j < d; ++j) {
        double a = 0.0;
        for (int i = 0; i < d; ++i) a += q[i] * s->SK[i * d + j];
        qsk[j] = a;
    }
    for (int j = 0; j < d; ++j) {
        double a = 0.0;
        for (int i = 0; i < d; ++i) a += qsk[i] * s->SQ[i * d + j];
        qsksq[j] = a;
    }
    for (int j = 0; j < dv; ++j) {
        double a = 0.0;
        for (int i = 0; i < d; ++i)
            a += qsksq[i] * s->P[i * dv + j] - q[i] * (s->G1[i * dv + j] + s->G2[i * dv + j] - s->G3[i * dv + j]);
        o[j] = a;
    }
}

/* Segment summary (S^K, S^Q, P, T, M^QP, M^KQ): out = A (+) B.  out may not alias. */
static void combine3(int d, int dv, const st3_t *A, const st3_t *B, st3_t *out, double *scratch)
{
    double *SKSQ = scratch;               /* S^K_A S^Q_B, d x d */
    double *X = scratch + (size_t)d * d;  /* M^QP_B + S^Q_B P_A, d x dv */
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < d; ++j) {
            double acc = 0.0;
            for (int l = 0; l < d; ++l) acc += A->SK[i * d + l] * B->SQ[l * d + j];
            SKSQ[i * d + j] = acc;
        }
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int l = 0; l < d; ++l) acc += B->SQ[i * d + l] * A->P[l * dv + j];
            X[i * dv + j] = acc;
        }
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < dv; ++j) {
            double t = A->T[i * dv + j] + B->T[i * dv + j];
            for (int l = 0; l < d; ++l)
                t += A->SK[i * d + l] * B->MQP[l * dv + j] + B->MKQ[i * d + l] * A->P[l * dv + j] +
                     SKSQ[i * d + l] * A->P[l * dv + j];
            out->T[i * dv + j] = t;
            out->MQP[i * dv + j] = A->MQP[i * dv + j] + B->MQP[i * dv + j] + X[i * dv + j];
            out->P[i * dv + j] = A->P[i * dv + j] + B->P[i * dv + j];
        }
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < d; ++j) {
            out->MKQ[i * d + j] = A->MKQ[i * d + j] + B->MKQ[i * d + j] + SKSQ[i * d + j];
            out->SK[i * d + j] = A->SK[i * d + j] + B->SK[i * d + j];
            out->SQ[i * d + j] = A->SQ[i * d + j] + B->SQ[i * d + j];
        }
}

typedef struct {
    int B, H, n, d, dv, chunk, next;
    const double *q, *k, *v, *st_in;
    double *o, *st_out;
    pthread_mutex_t lock;
} job3_t;

static void unit_serial(job3_t *J, int u)
{
    const int d = J->d, dv = J->dv;
    const size_t sz = st3_size(d, dv);
    double *buf = calloc(sz, sizeof(double));
    st3_t s;
    st3_bind(&s, buf, d, dv);
    st3_scratch(&s);
    if (J->st_in) memcpy(buf, J->st_in + (size_t)u * sz, sz * sizeof(double));
    const double *q = J->q + (size_t)u * J->n * d, *k = J->k + (size_t)u * J->n * d;
    const double *v = J->v + (size_t)u * J->n * dv;
    for (int t = 0; t < J->n; ++t) step3(&s, q + (size_t)t * d, k + (size_t)t * d, v + (size_t)t * dv,
                                         J->o + ((size_t)u * J->n + t) * dv);
    derive_T(&s);
    if (J->st_out) memcpy(J->st_out + (size_t)u * sz, buf, sz * sizeof(double));
    st3_free_scratch(&s);
    free(buf);
}

/* Chunked: the prefix summary A (folded chunk summaries) and the running summary of
 * the current chunk B<=t from zero; o_t = q_t^T T(A (+) B<=t). */
static void unit_chunked(job3_t *J, int u)
{
    const int d = J->d, dv = J->dv, c = J->chunk;
    const size_t sz = st3_size(d, dv);
    double *bufA = calloc(sz, sizeof(double)), *bufB = calloc(sz, sizeof(double)), *bufC = calloc(sz, sizeof(double));
    double *scr = calloc((size_t)d * d + (size_t)d * dv, sizeof(double));
    st3_t A, Bs, Cs;
    st3_bind(&A, bufA, d, dv); st3_bind(&Bs, bufB, d, dv); st3_bind(&Cs, bufC, d, dv);
    st3_scratch(&A); st3_scratch(&Bs);
    if (J->st_in) {
        memcpy(bufA, J->st_in + (size_t)u * sz, sz * sizeof(double));
        derive_T(&A);
    }
    const double *q = J->q + (size_t)u * J->n * d, *k = J->k + (size_t)u * J->n * d;
    const double *v = J->v + (size_t)u * J->n * dv;
    double *scratch_o = calloc((size_t)dv, sizeof(double));
    for (int t0 = 0; t0 < J->n; t0 += c) {
        const int L = J->n - t0 < c ? J->n - t0 : c;
        memset(bufB, 0, sz * sizeof(double));
        for (int t = t0; t < t0 + L; ++t) {
            step3(&Bs, q + (size_t)t * d, k + (size_t)t * d, v + (size_t)t * dv, scratch_o);
            derive_T(&Bs);
            combine3(d, dv, &A, &Bs, &Cs, scr);
            double *o = J->o + ((size_t)u * J->n + t) * dv;
            for (int j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int i = 0; i < d; ++i) acc += q[(size_t)t * d + i] * Cs.T[i * dv + j];
                o[j] = acc;
            }
        }
        memcpy(bufA, bufC, sz * sizeof(double));
    }
    if (J->n == 0) memcpy(bufC, bufA, sz * sizeof(double));
    if (J->st_out) {
        double *out = J->st_out + (size_t)u * sz;
        st3_t O;
        st3_bind(&O, out, d, dv);
        memcpy(out, bufA, sz * sizeof(double));
        const double nan = NAN;
        for (size_t i = 0; i < (size_t)d * d; ++i) O.Z1[i] = nan;
        for (size_t i = 0; i < (size_t)d * dv; ++i) O.Z2[i] = O.G1[i] = O.G2[i] = O.G3[i] = nan;
    }
    st3_free_scratch(&A); st3_free_scratch(&Bs);
    free(bufA); free(bufB); free(bufC); free(scr); free(scratch_o);
}

static void *worker3(void *arg)
{
    job3_t *J = (job3_t *)arg;
    for (;;) {
        pthread_mutex_lock(&J->lock);
        const int u = J->next < J->B * J->H ? J->next++ : -1;
        pthread_mutex_unlock(&J->lock);
        if (u < 0) break;
        if (J->chunk > 0) unit_chunked(J, u);
        else unit_serial(J, u);
    }
    return NULL;
}

/*
 * Masked third-order forward for B*H pairs.  q, k: [B][H][n][d]; v, o: [B][H][n][dv].
 * chunk 0: serial recurrence; chunk > 0: chunked scan over segment summaries.
 * st_in: NULL (zeros) or [B*H][4d^2 + 7 d dv] in the layout above; st_out: NULL or the
 * same layout.  Returns 0, or -1 for bad arguments.
 */
int hla_oracle3_forward(int B, int H, int n, int d, int dv, int chunk, const double *q, const double *k,
                        const double *v, const double *st_in, double *o, double *st_out, int nthreads)
{
    if (B < 1 || H < 1 || n < 0 || d < 1 || dv < 1 || chunk < 0) return -1;
    job3_t J;
    J.B = B; J.H = H; J.n = n; J.d = d; J.dv = dv; J.chunk = chunk; J.next = 0;
    J.q = q; J.k = k; J.v = v; J.st_in = st_in; J.o = o; J.st_out = st_out;
    pthread_mutex_init(&J.lock, NULL);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > B * H) nthreads = B * H;
    pthread_t *th = malloc(sizeof(pthread_t) * (size_t)nthreads);
    for (int i = 0; i < nthreads; ++i) pthread_create(&th[i], NULL, worker3, &J);
    for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&J.lock);
    return 0;
}

/* Concatenation of segment summaries for `count` items (A before B), layout above;
 * only S^K, S^Q, P, T, M^QP, M^KQ are read and written (the rest of out is NaN). */
int hla_oracle3_combine(int count, int d, int dv, const double *A, const double *Bst, double *out)
{
    if (count < 0 || d < 1 || dv < 1) return -1;
    const size_t sz = st3_size(d, dv);
    double *scr = calloc((size_t)d * d + (size_t)d * dv, sizeof(double));
    for (int u = 0; u < count; ++u) {
        st3_t a, b, c;
        st3_bind(&a, (double *)(A + (size_t)u * sz), d, dv);
        st3_bind(&b, (double *)(Bst + (size_t)u * sz), d, dv);
        st3_bind(&c, out + (size_t)u * sz, d, dv);
        for (size_t i = 0; i < sz; ++i) out[(size_t)u * sz + i] = NAN;
        combine3(d, dv, &a, &b, &c, scr);
    }
    free(scr);
    return 0;
}
