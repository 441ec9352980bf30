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
 * Exponential decay (per head, factor g in [0,1]; the section states no decayed third
 * order, so this is the reading of the second order carried over): every prefix moment
 * decays by g per token, S^K_t = g S^K + k k^T, S^Q_t = g S^Q + q q^T, P_t = g P + k v^T,
 * and the masked output is the masked sum of decayed triples,
 *   o_t = sum_{b<=t} sum_{a<=b} sum_{c<=b} g^{3t-a-b-c} (q_t.k_a)(k_a.q_b)(q_b.k_c) v_c,
 * still q_t^T (S^K S^Q P - G1 - G2 + G3) with every term carrying that weight.  The
 * online updates take the factors that keep those weights (with g = 1 they are the
 * ones above):
 *   Z1_t = g^2 Z1 + g k (k^T S^Q_{t-1}),      Z2_t = g^2 Z2 + g (S^Q_{t-1} k) v^T,
 *   G1_t = g^3 G1 + g^2 (Z1_{t-1} k) v^T + g k (k^T S^Q_{t-1} P_t),
 *   G2_t = g^3 G2 + g^2 (S^K_{t-1} S^Q_{t-1} k) v^T + k (k^T Z2_t),
 *   G3_t = g^3 G3 + k (k^T Z2_t) + (Z1_t k) v^T - g (k^T S^Q_{t-1} k) k v^T,
 * so T_t = g^3 T_{t-1} + (S^K_t q)(q^T P_t).  The maps carry the weight g^{2(t-b)}:
 * M^QP_t = g^2 M^QP + q (q^T P_t), M^KQ_t = g^2 M^KQ + (S^K_t q) q^T.  Concatenation,
 * f = g^{len B}:
 *   S^K = f S^K_A + S^K_B (S^Q, P likewise),
 *   T    = f^3 T_A + T_B + f S^K_A M^QP_B + f M^KQ_B P_A + f^2 S^K_A S^Q_B P_A,
 *   M^QP = f^2 M^QP_A + M^QP_B + f S^Q_B P_A,   M^KQ = f^2 M^KQ_A + M^KQ_B + f S^K_A S^Q_B.
 *
 * Ratio normalisation (the section names h^(1..3) beside G^(1..3); the reading is that
 * of the second order, "Normalisatie" of section 1): o_t = num_t / (den_t + eps), den_t
 * the masked output of unit values,
 *   den_t = sum_{b<=t} sum_{a<=b} sum_{c<=b} g^{3t-a-b-c} (q_t.k_a)(k_a.q_b)(q_b.k_c).
 * The recurrence runs on the values with one more column that is 1 for every token: in
 * that column P is the key mass m^K = sum k, G1..G3 are h^(1..3), T gives den, and
 * M^KQ applied to it is the map M^KQm the section names.  The state then has dv + 1
 * value columns, the unit column last.
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
    double g;  /* decay per token (1: none) */
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
    const double g = s->g, g2 = g * g, g3 = g2 * g;
    /* P_t */
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < dv; ++j) s->P[i * dv + j] = g * s->P[i * dv + j] + k[i] * v[j];
    /* Z1_t, Z2_t */
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < d; ++j) s->Z1[i * d + j] = g2 * s->Z1[i * d + j] + g * k[i] * ksq[j];
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < dv; ++j) s->Z2[i * dv + j] = g2 * s->Z2[i * dv + j] + g * sqk[i] * v[j];
    /* k^T S^Q_{t-1} P_t, k^T Z2_t, Z1_t k */
    for (int j = 0; j < dv; ++j) {
        double a = 0.0, b = 0.0;
        for (int i = 0; i < d; ++i) {
            a += ksq[i] * s->P[i * dv + j];
            b += k[i] * s->Z2[i * dv + j];
        }
        ksqp[j] = a; kz2[j] = b;
    }
    for (int i = 0; i < d; ++i) {  /* Z1_t k */
        double a = 0.0;
        for (int j = 0; j < d; ++j) a += s->Z1[i * d + j] * k[j];
        z1tk[i] = a;
    }
    /* cross summaries (z1k = Z1_{t-1} k, z1tk = Z1_t k) */
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < dv; ++j) {
            s->G1[i * dv + j] = g3 * s->G1[i * dv + j] + g2 * z1k[i] * v[j] + g * k[i] * ksqp[j];
            s->G2[i * dv + j] = g3 * s->G2[i * dv + j] + g2 * sksqk[i] * v[j] + k[i] * kz2[j];
            s->G3[i * dv + j] = g3 * s->G3[i * dv + j] + k[i] * kz2[j] + z1tk[i] * v[j] - g * ksqk * k[i] * v[j];
        }
    /* S^K_t, S^Q_t */
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < d; ++j) {
            s->SK[i * d + j] = g * s->SK[i * d + j] + k[i] * k[j];
            s->SQ[i * d + j] = g * s->SQ[i * d + j] + q[i] * q[j];
        }
    /* M^QP = g^2 M^QP + q (q^T P_t);  M^KQ = g^2 M^KQ + (S^K_t q) q^T */
    for (int j = 0; j < dv; ++j) {
        double a = 0.0;
        for (int i = 0; i < d; ++i) a += q[i] * s->P[i * dv + j];
        for (int i = 0; i < d; ++i) s->MQP[i * dv + j] = g2 * s->MQP[i * dv + j] + q[i] * a;
    }
    for (int i = 0; i < d; ++i) {
        double a = 0.0;
        for (int j = 0; j < d; ++j) a += s->SK[i * d + j] * q[j];
        for (int j = 0; j < d; ++j) s->MKQ[i * d + j] = g2 * s->MKQ[i * d + j] + a * q[j];
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

/* Segment summary (S^K, S^Q, P, T, M^QP, M^KQ): out = A (+) B with f = g^{len B}.
 * out may not alias. */
static void combine3(int d, int dv, double f, const st3_t *A, const st3_t *B, st3_t *out, double *scratch)
{
    const double f2 = f * f, f3 = f2 * f;
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
            double t1 = 0.0, t2 = 0.0, t3 = 0.0;
            for (int l = 0; l < d; ++l) {
                t1 += A->SK[i * d + l] * B->MQP[l * dv + j];
                t2 += B->MKQ[i * d + l] * A->P[l * dv + j];
                t3 += SKSQ[i * d + l] * A->P[l * dv + j];
            }
            out->T[i * dv + j] = f3 * A->T[i * dv + j] + B->T[i * dv + j] + f * t1 + f * t2 + f2 * t3;
            out->MQP[i * dv + j] = f2 * A->MQP[i * dv + j] + B->MQP[i * dv + j] + f * X[i * dv + j];
            out->P[i * dv + j] = f * A->P[i * dv + j] + B->P[i * dv + j];
        }
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < d; ++j) {
            out->MKQ[i * d + j] = f2 * A->MKQ[i * d + j] + B->MKQ[i * d + j] + f * SKSQ[i * d + j];
            out->SK[i * d + j] = f * A->SK[i * d + j] + B->SK[i * d + j];
            out->SQ[i * d + j] = f * A->SQ[i * d + j] + B->SQ[i * d + j];
        }
}

typedef struct {
    int B, H, n, d, dv, chunk, next;
    int normalize;        /* the state carries one more (unit) value column */
    double eps;
    const double *gamma;  /* [H] or NULL */
    const double *q, *k, *v, *st_in;
    double *o, *st_out;
    pthread_mutex_t lock;
} job3_t;

/* The values of pair u as the recurrence sees them: [n][dve], with the unit column last
 * when normalising (dve = dv + 1). */
static double *values3(const job3_t *J, int u, int dve)
{
    double *w = malloc(sizeof(double) * ((size_t)J->n * dve + 1));
    const double *v = J->v + (size_t)u * J->n * J->dv;
    for (int t = 0; t < J->n; ++t) {
        for (int j = 0; j < J->dv; ++j) w[(size_t)t * dve + j] = v[(size_t)t * J->dv + j];
        if (dve > J->dv) w[(size_t)t * dve + J->dv] = 1.0;
    }
    return w;
}

/* Output row t of pair u from the recurrence's row r (dve columns): the numerator, or
 * numerator / (den + eps) with den in the unit column. */
static void emit3(const job3_t *J, int u, int t, const double *r)
{
    double *o = J->o + ((size_t)u * J->n + t) * J->dv;
    const double den = J->normalize ? r[J->dv] + J->eps : 1.0;
    for (int j = 0; j < J->dv; ++j) o[j] = J->normalize ? r[j] / den : r[j];
}

static void unit_serial(job3_t *J, int u)
{
    const int d = J->d, dv = J->dv + (J->normalize ? 1 : 0);
    const size_t sz = st3_size(d, dv);
    double *buf = calloc(sz, sizeof(double));
    st3_t s;
    st3_bind(&s, buf, d, dv);
    st3_scratch(&s);
    s.g = J->gamma ? J->gamma[u % J->H] : 1.0;
    if (J->st_in) memcpy(buf, J->st_in + (size_t)u * sz, sz * sizeof(double));
    const double *q = J->q + (size_t)u * J->n * d, *k = J->k + (size_t)u * J->n * d;
    double *v = values3(J, u, dv), *row = calloc((size_t)dv, sizeof(double));
    for (int t = 0; t < J->n; ++t) {
        step3(&s, q + (size_t)t * d, k + (size_t)t * d, v + (size_t)t * dv, row);
        emit3(J, u, t, row);
    }
    derive_T(&s);
    if (J->st_out) memcpy(J->st_out + (size_t)u * sz, buf, sz * sizeof(double));
    st3_free_scratch(&s);
    free(buf); free(v); free(row);
}

/* Chunked: the prefix summary A (folded chunk summaries) and the running summary of
 * the current chunk B<=t from zero; o_t = q_t^T T(A (+) B<=t). */
static void unit_chunked(job3_t *J, int u)
{
    const int d = J->d, dv = J->dv + (J->normalize ? 1 : 0), c = J->chunk;
    const double g = J->gamma ? J->gamma[u % J->H] : 1.0;
    const size_t sz = st3_size(d, dv);
    double *bufA = calloc(sz, sizeof(double)), *bufB = calloc(sz, sizeof(double)), *bufC = calloc(sz, sizeof(double));
    double *scr = calloc((size_t)d * d + (size_t)d * dv, sizeof(double));
    st3_t A, Bs, Cs;
    st3_bind(&A, bufA, d, dv); st3_bind(&Bs, bufB, d, dv); st3_bind(&Cs, bufC, d, dv);
    st3_scratch(&A); st3_scratch(&Bs);
    A.g = Bs.g = g;
    if (J->st_in) {
        memcpy(bufA, J->st_in + (size_t)u * sz, sz * sizeof(double));
        derive_T(&A);
    }
    const double *q = J->q + (size_t)u * J->n * d, *k = J->k + (size_t)u * J->n * d;
    double *v = values3(J, u, dv);
    double *scratch_o = calloc((size_t)dv, sizeof(double)), *row = calloc((size_t)dv, sizeof(double));
    for (int t0 = 0; t0 < J->n; t0 += c) {
        const int L = J->n - t0 < c ? J->n - t0 : c;
        memset(bufB, 0, sz * sizeof(double));
        for (int t = t0; t < t0 + L; ++t) {
            step3(&Bs, q + (size_t)t * d, k + (size_t)t * d, v + (size_t)t * dv, scratch_o);
            derive_T(&Bs);
            combine3(d, dv, pow(g, (double)(t - t0 + 1)), &A, &Bs, &Cs, scr);
            for (int j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int i = 0; i < d; ++i) acc += q[(size_t)t * d + i] * Cs.T[i * dv + j];
                row[j] = acc;
            }
            emit3(J, u, t, row);
        }
        memcpy(bufA, bufC, sz * sizeof(double));
    }
    free(v); free(row);
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
 * gamma: [H] decay per head, or NULL (none).  normalize: o = num / (den + eps).
 * st_in: NULL (zeros) or [B*H][4d^2 + 7 d dve] in the layout above, dve = dv (+ 1 when
 * normalising, the unit column last); st_out: NULL or the same layout.
 * Returns 0, or -1 for bad arguments.
 */
int hla_oracle3_forward_ex(int B, int H, int n, int d, int dv, int chunk, const double *gamma, int normalize,
                           double eps, const double *q, const double *k, const double *v, const double *st_in,
                           double *o, double *st_out, int nthreads)
{
    if (B < 1 || H < 1 || n < 0 || d < 1 || dv < 1 || chunk < 0) return -1;
    job3_t J;
    J.B = B; J.H = H; J.n = n; J.d = d; J.dv = dv; J.chunk = chunk; J.next = 0;
    J.normalize = normalize != 0; J.eps = eps; J.gamma = gamma;
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

int hla_oracle3_forward(int B, int H, int n, int d, int dv, int chunk, const double *q, const double *k,
                        const double *v, const double *st_in, double *o, double *st_out, int nthreads)
{
    return hla_oracle3_forward_ex(B, H, n, d, dv, chunk, NULL, 0, 0.0, q, k, v, st_in, o, st_out, nthreads);
}

/* Concatenation of segment summaries for `count` items (A before B), layout above,
 * f_i = decay_pow[i] (g^{len B}; NULL: 1); only S^K, S^Q, P, T, M^QP, M^KQ are read and
 * written (the rest of out is NaN). */
int hla_oracle3_combine_ex(int count, int d, int dv, const double *decay_pow, const double *A, const double *Bst,
                           double *out)
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
        combine3(d, dv, decay_pow ? decay_pow[u] : 1.0, &a, &b, &c, scr);
    }
    free(scr);
    return 0;
}

int hla_oracle3_combine(int count, int d, int dv, const double *A, const double *Bst, double *out)
{
    return hla_oracle3_combine_ex(count, d, dv, NULL, A, Bst, out);
}
