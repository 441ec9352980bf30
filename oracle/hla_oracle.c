/*
 * hla_oracle.c -- fp64 CPU oracle for masked second-order Higher-order Linear
 * Attention (HLA).
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke check
 * and the CPU-baseline leg of the benchmark load this file.  It shares no code,
 * header, table or helper with the CUDA library, and the CUDA library never
 * loads it.
 *
 * What it computes (sources: "Higher-order Linear Attention", gist.science
 * technical summary, section 1 "Tweede-orde HLA", bullets "Onderhoud van de
 * toestand", "Strenge causaliteit", "Outputformulering", "Normalisatie";
 * section 4 "Parallelle training via associatieve scans", bullets
 * "Associatieve operatoren" and "Scan-equivalentie"; "Belangrijkste
 * bijdragen" item 2 for the exponential-decay variant):
 *
 *   prefix summaries   S_t = sum_{i<=t} k_i k_i^T        (d x d)
 *                      C_t = sum_{i<=t} q_i v_i^T        (d x dv)
 *                      m_t = sum_{i<=t} q_i              (d)
 *   cross summaries    G_t = G_{t-1} + k_t (k_t^T C_{t-1})   (d x dv)
 *                      h_t = h_{t-1} + k_t (k_t^T m_{t-1})   (d)
 *   masked output      o_t = q_t^T (S_t C_t - G_t)
 *   ratio-normalised   o_t = q_t^T (S_t C_t - G_t) / (q_t^T (S_t m_t - h_t) + eps)
 *
 * Exponential decay (per head, factor g in [0,1]): every prefix statistic decays
 * by g per step, S_t = g S_{t-1} + k k^T, C_t = g C_{t-1} + q v^T,
 * m_t = g m_{t-1} + q, and the cross summaries take the factors that keep
 * q_t^T(S_t C_t - G_t) equal to the masked sum of decayed pairs:
 * G_t = g^2 G_{t-1} + g k_t (k_t^T C_{t-1}),  h_t = g^2 h_{t-1} + g k_t (k_t^T m_{t-1}).
 * The pages name the decayed operators without printing them; this is the
 * plainest reading that the undecayed formulas support.  With g = 1 every
 * formula above reduces to the undecayed one.
 *
 * Segment concatenation (semidirect product), segment A before segment B,
 * f = g^{len(B)}:
 *   S = f S_A + S_B,  C = f C_A + C_B,  m = f m_A + m_B,
 *   G = f^2 G_A + G_B + f S_B C_A,   h = f^2 h_A + h_B + f S_B m_A.
 * The cross term S_B C_A is the one the pages name.
 *
 * Unmasked variant (the skill card "Higher-order linear attention", section
 * "Linear-Time Higher-Order Interactions", bullet "Streaming Computation";
 * gist.science "Belangrijkste bijdragen" item 2 for its scan operators):
 *   o_t = q_t^T S_t C_t,   ratio-normalised  o_t = q_t^T S_t C_t / (q_t^T S_t m_t + eps),
 * with the same decayed S, C, m.  Only S, C, m are carried; G and h are not
 * part of this variant and are left at zero.  Its concatenation is the linear
 * part of the rule above (S, C, m).
 *
 * Asymmetric variant AHLA (gist.science summary, section 2 "Asymmetrische
 * Hogere-orde Lineaire Aandacht"): the operator Q (K^T Q)(K^T V) = A A V with
 * A = Q K^T, masked to o_t = sum_{a<=b<=t} (q_t.k_b)(q_b.k_a) v_a: the value index a
 * is routed through the intermediate key index b.  Its streaming summaries (the
 * section names P^KV, m^K, E, n):
 *   P_t = g P_{t-1} + k_t v_t^T,   m_t = g m_{t-1} + k_t,
 *   E_t = g E_{t-1} + k_t (q_t^T P_t),   n_t = g n_{t-1} + k_t (q_t . m_t),
 *   o_t = q_t^T E_t,   ratio form o_t = q_t^T E_t / (q_t^T n_t + eps),
 * so the pair weight is g^{(t-b)+(b-a)} = g^{t-a}.  Composing segment A before B
 * (f = g^{len B}) needs one more summary, R = sum_b k_b q_b^T without decay:
 *   P = f P_A + P_B,  m = f m_A + m_B,  R = R_A + R_B,
 *   E = f E_A + E_B + f R_B P_A,   n = f n_A + n_B + f R_B m_A.
 * In the five state arrays the variant keeps R in S, P in C, m^K in m, E in G
 * and n in h.
 *
 * Multi-query heads (skill card, section "Architecture Overview", bullet
 * "Multi-Head Support"): k and v may have Hkv heads with H a multiple of Hkv;
 * query head h reads key/value head h / (H / Hkv).  The summaries stay per query
 * head (C = sum q v^T depends on the query head; S is the same for every head
 * of a group).
 *
 * Layout: q [B][H][n][d], k [B][Hkv][n][d], v [B][Hkv][n][dv], o [B][H][n][dv];
 * row-major, fp64.  State, one block per (b,h): S [BH][d][d], C [BH][d][dv],
 * m [BH][d], G [BH][d][dv], h [BH][d].
 *
 * Everything is a plain loop in the order the formulas are written; no
 * blocking, no fusion.  Independent (b,h) pairs run on separate threads.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    double *S, *C, *m, *G, *h;
} ostate;

/* one (b,h) stream: the five summaries of one head, plus its decay factor */
typedef struct {
    int d, dv;
    int variant; /* 0 masked, 1 unmasked (o = q^T S C; G, h not carried), 2 asymmetric */
    double g;
    double *S, *C, *m, *G, *h; /* views into caller state for this (b,h) */
    double *kc;                /* scratch: k^T C_{t-1}, length dv        */
    double *qs;                /* scratch: q^T S_t, length d             */
} stream_t;

/* One token of the serial recurrence.  The cross summaries are updated from
 * the previous C and m first, then the prefix summaries take the new token.
 * If o != NULL the (optionally normalised) output of this token is written. */
static void step_token(stream_t *st, const double *q, const double *k,
                       const double *v, int normalize, double eps, double *o)
{
    const int d = st->d, dv = st->dv;
    const double g = st->g, g2 = g * g;
    double *S = st->S, *C = st->C, *m = st->m, *G = st->G, *h = st->h;

    if (st->variant == 2) { /* asymmetric: R in S, P in C, m^K in m, E in G, n in h */
        for (int i = 0; i < d; ++i) /* R_t = R_{t-1} + k q^T */
            for (int j = 0; j < d; ++j) S[i * d + j] += k[i] * q[j];
        for (int i = 0; i < d; ++i) { /* P_t = g P_{t-1} + k v^T, m_t = g m_{t-1} + k */
            for (int j = 0; j < dv; ++j) C[i * dv + j] = g * C[i * dv + j] + k[i] * v[j];
            m[i] = g * m[i] + k[i];
        }
        double zeta = 0.0; /* z = q^T P_t, zeta = q . m_t */
        for (int j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int i = 0; i < d; ++i) acc += q[i] * C[i * dv + j];
            st->kc[j] = acc;
        }
        for (int i = 0; i < d; ++i) zeta += q[i] * m[i];
        for (int i = 0; i < d; ++i) { /* E_t = g E_{t-1} + k z^T, n_t = g n_{t-1} + k zeta */
            for (int j = 0; j < dv; ++j) G[i * dv + j] = g * G[i * dv + j] + k[i] * st->kc[j];
            h[i] = g * h[i] + k[i] * zeta;
        }
        if (!o) return;
        double den = 0.0; /* o = q^T E_t [/ (q^T n_t + eps)] */
        if (normalize) {
            for (int i = 0; i < d; ++i) den += q[i] * h[i];
            den += eps;
        }
        for (int j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int i = 0; i < d; ++i) acc += q[i] * G[i * dv + j];
            o[j] = normalize ? acc / den : acc;
        }
        return;
    }

    if (st->variant == 0) {
        /* k^T C_{t-1} and k^T m_{t-1} */
        for (int j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int i = 0; i < d; ++i) acc += k[i] * C[i * dv + j];
            st->kc[j] = acc;
        }
        double km = 0.0;
        for (int i = 0; i < d; ++i) km += k[i] * m[i];

        /* G_t = g^2 G_{t-1} + g k (k^T C_{t-1}),  h_t = g^2 h_{t-1} + g k (k^T m_{t-1}) */
        for (int i = 0; i < d; ++i) {
            for (int j = 0; j < dv; ++j)
                G[i * dv + j] = g2 * G[i * dv + j] + g * k[i] * st->kc[j];
            h[i] = g2 * h[i] + g * k[i] * km;
        }
    }
    /* S_t = g S_{t-1} + k k^T */
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < d; ++j)
            S[i * d + j] = g * S[i * d + j] + k[i] * k[j];
    /* C_t = g C_{t-1} + q v^T,  m_t = g m_{t-1} + q */
    for (int i = 0; i < d; ++i) {
        for (int j = 0; j < dv; ++j)
            C[i * dv + j] = g * C[i * dv + j] + q[i] * v[j];
        m[i] = g * m[i] + q[i];
    }
    if (!o) return;

    /* o_t = q^T (S_t C_t - G_t), evaluated as (q^T S_t) C_t - q^T G_t so that
     * the cost per token is O(d^2 + d dv) as the pages state; the unmasked
     * variant has no G (and no h) term.  G and h are zero in that variant, so the
     * same loops serve both. */
    for (int j = 0; j < d; ++j) {
        double acc = 0.0;
        for (int i = 0; i < d; ++i) acc += q[i] * S[i * d + j];
        st->qs[j] = acc;
    }
    double den = 0.0;
    if (normalize) {
        /* q^T (S_t m_t - h_t) */
        for (int i = 0; i < d; ++i) den += st->qs[i] * m[i] - q[i] * h[i];
        den += eps;
    }
    for (int j = 0; j < dv; ++j) {
        double acc = 0.0;
        for (int i = 0; i < d; ++i) acc += st->qs[i] * C[i * dv + j] - q[i] * G[i * dv + j];
        o[j] = normalize ? acc / den : acc;
    }
}

/* R7: out = A (+) B, A earlier in time than B, f = g^{len(B)}.
 * out may alias A or B: every output is formed in a private buffer first. */
static void combine_one(int d, int dv, double f, int variant,
                        const double *SA, const double *CA, const double *mA,
                        const double *GA, const double *hA,
                        const double *SB, const double *CB, const double *mB,
                        const double *GB, const double *hB,
                        double *S, double *C, double *m, double *G, double *h)
{
    const double f2 = f * f;
    double *tG = (double *)malloc(sizeof(double) * (size_t)d * dv);
    double *th = (double *)malloc(sizeof(double) * (size_t)d);
    if (variant == 2) {
        /* asymmetric: E = f E_A + E_B + f R_B P_A, n = f n_A + n_B + f R_B m_A,
         * P = f P_A + P_B, m = f m_A + m_B, R = R_A + R_B (R in S, P in C, E in G, n in h) */
        for (int i = 0; i < d; ++i) {
            for (int j = 0; j < dv; ++j) {
                double cross = 0.0; /* (R_B P_A)[i][j] */
                for (int l = 0; l < d; ++l) cross += SB[i * d + l] * CA[l * dv + j];
                tG[i * dv + j] = f * GA[i * dv + j] + GB[i * dv + j] + f * cross;
            }
            double crossm = 0.0; /* (R_B m_A)[i] */
            for (int l = 0; l < d; ++l) crossm += SB[i * d + l] * mA[l];
            th[i] = f * hA[i] + hB[i] + f * crossm;
        }
        for (int i = 0; i < d * d; ++i) S[i] = SA[i] + SB[i];
        for (int i = 0; i < d * dv; ++i) C[i] = f * CA[i] + CB[i];
        for (int i = 0; i < d; ++i) m[i] = f * mA[i] + mB[i];
        memcpy(G, tG, sizeof(double) * (size_t)d * dv);
        memcpy(h, th, sizeof(double) * (size_t)d);
        free(tG);
        free(th);
        return;
    }
    for (int i = 0; i < d; ++i) {
        for (int j = 0; j < dv; ++j) {
            double cross = 0.0; /* (S_B C_A)[i][j] */
            for (int l = 0; l < d; ++l) cross += SB[i * d + l] * CA[l * dv + j];
            tG[i * dv + j] = f2 * GA[i * dv + j] + GB[i * dv + j] + f * cross;
        }
        double crossm = 0.0; /* (S_B m_A)[i] */
        for (int l = 0; l < d; ++l) crossm += SB[i * d + l] * mA[l];
        th[i] = f2 * hA[i] + hB[i] + f * crossm;
    }
    for (int i = 0; i < d * d; ++i) S[i] = f * SA[i] + SB[i];
    for (int i = 0; i < d * dv; ++i) C[i] = f * CA[i] + CB[i];
    for (int i = 0; i < d; ++i) m[i] = f * mA[i] + mB[i];
    memcpy(G, tG, sizeof(double) * (size_t)d * dv);
    memcpy(h, th, sizeof(double) * (size_t)d);
    free(tG);
    free(th);
}

/* ------------------------------------------------------------------------- */
/* work distribution over (b,h) pairs                                        */

typedef struct {
    int B, H, n, d, dv, chunk;
    int Hkv;      /* key/value heads; query head h reads head h / (H / Hkv) */
    int variant;  /* 0 masked, 1 unmasked, 2 asymmetric */
    const double *q, *k, *v, *gamma;
    int normalize;
    double eps;
    ostate in, out;
    double *o;
    int next; /* next unit to take, guarded by lock */
    pthread_mutex_t lock;
    int mode; /* 0 serial forward, 1 chunked-scan forward, 2 decode step */
} job_t;

static int take_unit(job_t *J, int total)
{
    pthread_mutex_lock(&J->lock);
    int u = J->next < total ? J->next++ : -1;
    pthread_mutex_unlock(&J->lock);
    return u;
}

static void load_state(stream_t *st, const ostate *in, size_t u)
{
    const int d = st->d, dv = st->dv;
    if (in && in->S) {
        memcpy(st->S, in->S + u * d * d, sizeof(double) * d * d);
        memcpy(st->C, in->C + u * d * dv, sizeof(double) * d * dv);
        memcpy(st->m, in->m + u * d, sizeof(double) * d);
        if (st->variant == 1) { /* not part of the unmasked state */
            memset(st->G, 0, sizeof(double) * d * dv);
            memset(st->h, 0, sizeof(double) * d);
        } else {
            memcpy(st->G, in->G + u * d * dv, sizeof(double) * d * dv);
            memcpy(st->h, in->h + u * d, sizeof(double) * d);
        }
    } else {
        memset(st->S, 0, sizeof(double) * d * d);
        memset(st->C, 0, sizeof(double) * d * dv);
        memset(st->m, 0, sizeof(double) * d);
        memset(st->G, 0, sizeof(double) * d * dv);
        memset(st->h, 0, sizeof(double) * d);
    }
}

static void store_state(const stream_t *st, ostate *out, size_t u)
{
    const int d = st->d, dv = st->dv;
    if (!out || !out->S) return;
    memcpy(out->S + u * d * d, st->S, sizeof(double) * d * d);
    memcpy(out->C + u * d * dv, st->C, sizeof(double) * d * dv);
    memcpy(out->m + u * d, st->m, sizeof(double) * d);
    memcpy(out->G + u * d * dv, st->G, sizeof(double) * d * dv);
    memcpy(out->h + u * d, st->h, sizeof(double) * d);
}

static stream_t stream_new(int d, int dv)
{
    stream_t st;
    st.d = d;
    st.dv = dv;
    st.variant = 0;
    st.g = 1.0;
    st.S = (double *)calloc((size_t)d * d, sizeof(double));
    st.C = (double *)calloc((size_t)d * dv, sizeof(double));
    st.m = (double *)calloc((size_t)d, sizeof(double));
    st.G = (double *)calloc((size_t)d * dv, sizeof(double));
    st.h = (double *)calloc((size_t)d, sizeof(double));
    st.kc = (double *)calloc((size_t)dv, sizeof(double));
    st.qs = (double *)calloc((size_t)d, sizeof(double));
    return st;
}

static void stream_free(stream_t *st)
{
    free(st->S); free(st->C); free(st->m); free(st->G); free(st->h);
    free(st->kc); free(st->qs);
}

/* serial recurrence over all n tokens of unit u = b*H + hh */
/* key/value head of unit u = b*H + hh */
static size_t kv_unit(const job_t *J, int u)
{
    const int b = u / J->H, hh = u % J->H;
    return (size_t)b * J->Hkv + hh / (J->H / J->Hkv);
}

static void run_serial(job_t *J, stream_t *st, int u)
{
    const int n = J->n, d = J->d, dv = J->dv;
    const size_t qo = (size_t)u * n * d, oo = (size_t)u * n * dv;
    const size_t ko = kv_unit(J, u) * n * d, vo = kv_unit(J, u) * n * dv;
    load_state(st, &J->in, u);
    for (int t = 0; t < n; ++t)
        step_token(st, J->q + qo + (size_t)t * d, J->k + ko + (size_t)t * d,
                   J->v + vo + (size_t)t * dv, J->normalize, J->eps,
                   J->o ? J->o + oo + (size_t)t * dv : NULL);
    store_state(st, &J->out, u);
}

/* Chunked scan: each chunk's own summary is built from zero by the token
 * recurrence (no outputs), the running prefix is the left fold of the
 * preceding summaries with the segment-concatenation rule, and the chunk's
 * outputs are produced by continuing the recurrence from that prefix.  Equal
 * to run_serial up to rounding whenever the concatenation rule is exact. */
static void run_chunked(job_t *J, stream_t *st, int u)
{
    const int n = J->n, d = J->d, dv = J->dv, c = J->chunk;
    const size_t qo = (size_t)u * n * d, oo = (size_t)u * n * dv;
    const size_t ko = kv_unit(J, u) * n * d, vo = kv_unit(J, u) * n * dv;
    stream_t loc = stream_new(d, dv);
    loc.g = st->g;
    loc.variant = st->variant;
    /* prefix state lives in st */
    load_state(st, &J->in, u);
    for (int t0 = 0; t0 < n; t0 += c) {
        const int len = (n - t0 < c) ? (n - t0) : c;
        /* local summary of this chunk, from zero */
        load_state(&loc, NULL, 0);
        for (int t = t0; t < t0 + len; ++t)
            step_token(&loc, J->q + qo + (size_t)t * d, J->k + ko + (size_t)t * d,
                       J->v + vo + (size_t)t * dv, 0, 0.0, NULL);
        /* outputs of this chunk: continue from the prefix in a copy */
        stream_t run = stream_new(d, dv);
        run.g = st->g;
        run.variant = st->variant;
        memcpy(run.S, st->S, sizeof(double) * d * d);
        memcpy(run.C, st->C, sizeof(double) * d * dv);
        memcpy(run.m, st->m, sizeof(double) * d);
        memcpy(run.G, st->G, sizeof(double) * d * dv);
        memcpy(run.h, st->h, sizeof(double) * d);
        for (int t = t0; t < t0 + len; ++t)
            step_token(&run, J->q + qo + (size_t)t * d, J->k + ko + (size_t)t * d,
                       J->v + vo + (size_t)t * dv, J->normalize, J->eps,
                       J->o ? J->o + oo + (size_t)t * dv : NULL);
        stream_free(&run);
        /* prefix <- prefix (+) local; the unmasked variant keeps G, h at zero */
        combine_one(d, dv, pow(st->g, (double)len), st->variant,
                    st->S, st->C, st->m, st->G, st->h,
                    loc.S, loc.C, loc.m, loc.G, loc.h,
                    st->S, st->C, st->m, st->G, st->h);
        if (st->variant == 1) {
            memset(st->G, 0, sizeof(double) * d * dv);
            memset(st->h, 0, sizeof(double) * d);
        }
    }
    store_state(st, &J->out, u);
    stream_free(&loc);
}

/* one decode step for pair u (seq*H + head): state in place, one token */
static void run_decode(job_t *J, stream_t *st, int u)
{
    const int d = J->d, dv = J->dv;
    load_state(st, &J->in, u);
    step_token(st, J->q + (size_t)u * d, J->k + kv_unit(J, u) * d, J->v + kv_unit(J, u) * dv,
               J->normalize, J->eps, J->o + (size_t)u * dv);
    store_state(st, &J->out, u);
}

static void *worker(void *arg)
{
    job_t *J = (job_t *)arg;
    stream_t st = stream_new(J->d, J->dv);
    const int total = J->B * J->H;
    for (;;) {
        int u = take_unit(J, total);
        if (u < 0) break;
        st.g = J->gamma ? J->gamma[u % J->H] : 1.0;
        st.variant = J->variant;
        if (J->mode == 0) run_serial(J, &st, u);
        else if (J->mode == 1) run_chunked(J, &st, u);
        else run_decode(J, &st, u);
    }
    stream_free(&st);
    return NULL;
}

static int run_job(job_t *J, int nthreads)
{
    const int total = J->B * J->H;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > total) nthreads = total > 0 ? total : 1;
    J->next = 0;
    pthread_mutex_init(&J->lock, NULL);
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * nthreads);
    int started = 0;
    for (int i = 1; i < nthreads; ++i)
        if (pthread_create(&th[started], NULL, worker, J) == 0) ++started;
    worker(J);
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&J->lock);
    return 0;
}

static int check_dims(int B, int H, int n, int d, int dv)
{
    return (B < 0 || H < 1 || n < 0 || d < 1 || dv < 1) ? -1 : 0;
}

static int check_heads(int H, int Hkv, int variant)
{
    return (Hkv < 1 || H % Hkv || variant < 0 || variant > 2) ? -1 : 0;
}

/* ------------------------------------------------------------------------- */
/* exported entry points (ctypes)                                            */

/* Serial recurrence over n tokens for every (b,h).  gamma: [H] or NULL (no
 * decay).  state_in / state_out: pointers may be NULL (zeros / skip).  Hkv:
 * key/value heads (H for ordinary multi-head); variant: 0 masked, 1 unmasked,
 * 2 asymmetric. */
int hla_oracle_forward(int B, int H, int Hkv, int n, int d, int dv, int variant,
                       const double *q, const double *k, const double *v,
                       const double *gamma, int normalize, double eps,
                       double *Si, double *Ci, double *mi, double *Gi, double *hi,
                       double *o,
                       double *So, double *Co, double *mo, double *Go, double *ho,
                       int nthreads)
{
    if (check_dims(B, H, n, d, dv) || check_heads(H, Hkv, variant)) return -1;
    job_t J;
    memset(&J, 0, sizeof J);
    J.B = B; J.H = H; J.n = n; J.d = d; J.dv = dv; J.chunk = 0;
    J.Hkv = Hkv; J.variant = variant;
    J.q = q; J.k = k; J.v = v; J.gamma = gamma;
    J.normalize = normalize; J.eps = eps;
    J.in = (ostate){Si, Ci, mi, Gi, hi};
    J.out = (ostate){So, Co, mo, Go, ho};
    J.o = o;
    J.mode = 0;
    return run_job(&J, nthreads);
}

/* Chunked-scan forward (chunk >= 1): see run_chunked. */
int hla_oracle_forward_chunked(int B, int H, int Hkv, int n, int d, int dv, int variant, int chunk,
                               const double *q, const double *k, const double *v,
                               const double *gamma, int normalize, double eps,
                               double *Si, double *Ci, double *mi, double *Gi, double *hi,
                               double *o,
                               double *So, double *Co, double *mo, double *Go, double *ho,
                               int nthreads)
{
    if (check_dims(B, H, n, d, dv) || check_heads(H, Hkv, variant) || chunk < 1) return -1;
    job_t J;
    memset(&J, 0, sizeof J);
    J.B = B; J.H = H; J.n = n; J.d = d; J.dv = dv; J.chunk = chunk;
    J.Hkv = Hkv; J.variant = variant;
    J.q = q; J.k = k; J.v = v; J.gamma = gamma;
    J.normalize = normalize; J.eps = eps;
    J.in = (ostate){Si, Ci, mi, Gi, hi};
    J.out = (ostate){So, Co, mo, Go, ho};
    J.o = o;
    J.mode = 1;
    return run_job(&J, nthreads);
}

/* One decode step for N independent (sequence, head) pairs, pair u using
 * gamma[u % H].  The state arrays are read and written in place.
 * q: [N][d], o: [N][dv]; k: [N/H*Hkv][d], v: [N/H*Hkv][dv]. */
int hla_oracle_decode_step(int N, int H, int Hkv, int d, int dv, int variant,
                           const double *gamma, int normalize, double eps,
                           double *S, double *C, double *m, double *G, double *h,
                           const double *q, const double *k, const double *v,
                           double *o, int nthreads)
{
    if (check_dims(1, H, 1, d, dv) || check_heads(H, Hkv, variant) || N < 0) return -1;
    if (N % H) return -1;
    job_t J;
    memset(&J, 0, sizeof J);
    J.B = N / H; J.H = H; J.n = 1; J.d = d; J.dv = dv;
    J.Hkv = Hkv; J.variant = variant;
    J.q = q; J.k = k; J.v = v; J.gamma = gamma;
    J.normalize = normalize; J.eps = eps;
    J.in = (ostate){S, C, m, G, h};
    J.out = (ostate){S, C, m, G, h};
    J.o = o;
    J.mode = 2;
    return run_job(&J, nthreads);
}

/* ------------------------------------------------------------------------- */
/* backward pass of the masked forward (zero initial state), optionally through the
 * ratio normalisation o_t = n_t / (den_t + eps), n_t = X_t^T q_t, den_t = Y_t . q_t with
 * Y_t = g^2 Y_{t-1} + u_t (the output with every value equal to one).  Reverse mode
 * with r_t = 1 / (den_t + eps), gn_t = r_t go_t, gd_t = -r_t (go_t . o_t):
 *   Lam_t = q_t gn_t^T + g^2 Lam_{t+1},  Lamy_t = gd_t q_t + g^2 Lamy_{t+1},
 *   du_t = Lam_t v_t + Lamy_t,  dv_t = Lam_t^T u_t,  dq_t = X_t gn_t + gd_t Y_t + S_t du_t,
 *   Om_t = du_t q_t^T + g Om_{t+1},  dk_t = (Om_t + Om_t^T) k_t.
 * Without normalisation gn = go and gd = 0. */
/* The state before the first token (S, C, m, G, h of one pair, or NULLs: zeros) and the
 * gradient with respect to it (NULLs: not wanted). */
typedef struct {
    const double *S, *C, *m, *G, *h;
    double *dS, *dC, *dm, *dG, *dh;
} bstate_t;

static void backward_unit(int n, int d, int dv, double g, int normalize, double eps, const double *q,
                          const double *k, const double *v, const double *go, double *dq, double *dk, double *dvo,
                          const bstate_t *st0)
{
    double *S = (double *)calloc((size_t)(n + 1) * d * d, sizeof(double));  /* S_t after token t */
    double *X = (double *)calloc((size_t)(n + 1) * d * dv, sizeof(double)); /* X_t after token t */
    double *Y = (double *)calloc((size_t)(n + 1) * d, sizeof(double));      /* Y_t after token t */
    /* the state before the first token: S_in, X_in = S_in C_in - G_in, Y_in = S_in m_in - h_in */
    if (st0 && st0->S) {
        for (int i = 0; i < d * d; ++i) S[i] = st0->S[i];
        for (int i = 0; i < d; ++i) {
            for (int j = 0; j < dv; ++j) {
                double acc = -st0->G[i * dv + j];
                for (int l = 0; l < d; ++l) acc += st0->S[i * d + l] * st0->C[l * dv + j];
                X[i * dv + j] = acc;
            }
            double acc = -st0->h[i];
            for (int l = 0; l < d; ++l) acc += st0->S[i * d + l] * st0->m[l];
            Y[i] = acc;
        }
    }
    double *U = (double *)calloc((size_t)n * d, sizeof(double));            /* u_t */
    double *gn = (double *)calloc((size_t)n * dv + 1, sizeof(double));      /* dL/dn_t */
    double *gd = (double *)calloc((size_t)n + 1, sizeof(double));           /* dL/dden_t */
    double *Lam = (double *)calloc((size_t)d * dv, sizeof(double));
    double *Lamy = (double *)calloc((size_t)d, sizeof(double));
    double *Om = (double *)calloc((size_t)d * d, sizeof(double));
    double *du = (double *)calloc((size_t)d, sizeof(double));
    for (int t = 0; t < n; ++t) { /* forward, keeping every state */
        const double *qt = q + (size_t)t * d, *kt = k + (size_t)t * d, *vt = v + (size_t)t * dv;
        const double *Sp = S + (size_t)t * d * d, *Xp = X + (size_t)t * d * dv, *Yp = Y + (size_t)t * d;
        double *St = S + (size_t)(t + 1) * d * d, *Xt = X + (size_t)(t + 1) * d * dv, *Yt = Y + (size_t)(t + 1) * d;
        double *ut = U + (size_t)t * d;
        for (int i = 0; i < d; ++i)
            for (int j = 0; j < d; ++j) St[i * d + j] = g * Sp[i * d + j] + kt[i] * kt[j];
        for (int i = 0; i < d; ++i) {
            double acc = 0.0;
            for (int j = 0; j < d; ++j) acc += St[i * d + j] * qt[j];
            ut[i] = acc;
        }
        for (int i = 0; i < d; ++i) {
            for (int j = 0; j < dv; ++j) Xt[i * dv + j] = g * g * Xp[i * dv + j] + ut[i] * vt[j];
            Yt[i] = g * g * Yp[i] + ut[i];
        }
        const double *gt = go + (size_t)t * dv;
        if (normalize) { /* n_t, den_t, then gn_t and gd_t */
            double den = eps, dot = 0.0;
            for (int i = 0; i < d; ++i) den += qt[i] * Yt[i];
            const double r = 1.0 / den;
            for (int j = 0; j < dv; ++j) {
                double nj = 0.0;
                for (int i = 0; i < d; ++i) nj += Xt[i * dv + j] * qt[i];
                gn[(size_t)t * dv + j] = r * gt[j];
                dot += gt[j] * nj * r; /* go_t . o_t */
            }
            gd[t] = -r * dot;
        } else {
            for (int j = 0; j < dv; ++j) gn[(size_t)t * dv + j] = gt[j];
            gd[t] = 0.0;
        }
    }
    for (int t = n - 1; t >= 0; --t) { /* reverse */
        const double *qt = q + (size_t)t * d, *kt = k + (size_t)t * d, *vt = v + (size_t)t * dv;
        const double *gt = gn + (size_t)t * dv, *ut = U + (size_t)t * d;
        const double *St = S + (size_t)(t + 1) * d * d, *Xt = X + (size_t)(t + 1) * d * dv;
        const double *Yt = Y + (size_t)(t + 1) * d;
        /* Lam_t = q_t gn_t^T + g^2 Lam_{t+1};  Lamy_t = gd_t q_t + g^2 Lamy_{t+1} */
        for (int i = 0; i < d; ++i) {
            for (int j = 0; j < dv; ++j) Lam[i * dv + j] = g * g * Lam[i * dv + j] + qt[i] * gt[j];
            Lamy[i] = g * g * Lamy[i] + gd[t] * qt[i];
        }
        /* du_t = Lam_t v_t + Lamy_t;  dv_t = Lam_t^T u_t */
        for (int i = 0; i < d; ++i) {
            double acc = Lamy[i];
            for (int j = 0; j < dv; ++j) acc += Lam[i * dv + j] * vt[j];
            du[i] = acc;
        }
        for (int j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int i = 0; i < d; ++i) acc += Lam[i * dv + j] * ut[i];
            dvo[(size_t)t * dv + j] = acc;
        }
        /* dq_t = X_t gn_t + gd_t Y_t + S_t du_t */
        for (int i = 0; i < d; ++i) {
            double acc = gd[t] * Yt[i];
            for (int j = 0; j < dv; ++j) acc += Xt[i * dv + j] * gt[j];
            for (int j = 0; j < d; ++j) acc += St[i * d + j] * du[j];
            dq[(size_t)t * d + i] = acc;
        }
        /* Om_t = du_t q_t^T + g Om_{t+1};  dk_t = (Om_t + Om_t^T) k_t */
        for (int i = 0; i < d; ++i)
            for (int j = 0; j < d; ++j) Om[i * d + j] = g * Om[i * d + j] + du[i] * qt[j];
        for (int i = 0; i < d; ++i) {
            double acc = 0.0;
            for (int j = 0; j < d; ++j) acc += (Om[i * d + j] + Om[j * d + i]) * kt[j];
            dk[(size_t)t * d + i] = acc;
        }
    }
    /* the initial state: S_0 = g S_in + k k^T, X_0 = g^2 X_in + ..., Y_0 = g^2 Y_in + ...
     * (n = 0: the adjoints are zero), then through X_in = S_in C_in - G_in and
     * Y_in = S_in m_in - h_in */
    if (st0 && st0->dS) {
        const double g2 = n > 0 ? g * g : 0.0, g1 = n > 0 ? g : 0.0;
        double *dX = (double *)calloc((size_t)d * dv, sizeof(double)), *dY = (double *)calloc((size_t)d, sizeof(double));
        for (int i = 0; i < d * dv; ++i) dX[i] = g2 * Lam[i];
        for (int i = 0; i < d; ++i) dY[i] = g2 * Lamy[i];
        const int have = st0->S != NULL;
        for (int i = 0; i < d; ++i)
            for (int j = 0; j < d; ++j) {
                double acc = g1 * Om[i * d + j];
                if (have) {
                    for (int c = 0; c < dv; ++c) acc += dX[i * dv + c] * st0->C[j * dv + c];
                    acc += dY[i] * st0->m[j];
                }
                st0->dS[i * d + j] = acc;
            }
        for (int j = 0; j < d; ++j) {
            for (int c = 0; c < dv; ++c) {
                double acc = 0.0;
                if (have)
                    for (int i = 0; i < d; ++i) acc += st0->S[i * d + j] * dX[i * dv + c];
                st0->dC[j * dv + c] = acc;
            }
            double acc = 0.0;
            if (have)
                for (int i = 0; i < d; ++i) acc += st0->S[i * d + j] * dY[i];
            st0->dm[j] = acc;
        }
        for (int i = 0; i < d * dv; ++i) st0->dG[i] = -dX[i];
        for (int i = 0; i < d; ++i) st0->dh[i] = -dY[i];
        free(dX); free(dY);
    }
    free(S); free(X); free(Y); free(U); free(gn); free(gd); free(Lam); free(Lamy); free(Om); free(du);
}

typedef struct {
    int B, H, Hkv, n, d, dv, next, normalize;
    double eps;
    const double *q, *k, *v, *go, *gamma;
    double *dq, *dk_pair, *dv_pair;  /* dk, dv of every query head before the group sum */
    const double *sS, *sC, *sm, *sG, *sh;  /* state before the first token [B*H][...] or NULL */
    double *dS, *dC, *dm, *dG, *dh;        /* its gradient, or NULL */
    pthread_mutex_t lock;
} bjob_t;

static void *bworker(void *arg)
{
    bjob_t *J = (bjob_t *)arg;
    for (;;) {
        pthread_mutex_lock(&J->lock);
        const int u = J->next < J->B * J->H ? J->next++ : -1;
        pthread_mutex_unlock(&J->lock);
        if (u < 0) break;
        /* query head h of batch row b reads key/value head h / (H / Hkv) */
        const size_t kvu = (size_t)(u / J->H) * J->Hkv + (u % J->H) / (J->H / J->Hkv);
        const size_t qo = (size_t)u * J->n * J->d, vo = (size_t)u * J->n * J->dv;
        const size_t ko = kvu * J->n * J->d, kvo = kvu * J->n * J->dv;
        const size_t dd = (size_t)J->d * J->d, ddv = (size_t)J->d * J->dv;
        bstate_t st0;
        st0.S = J->sS ? J->sS + u * dd : NULL;
        st0.C = J->sS ? J->sC + u * ddv : NULL;
        st0.m = J->sS ? J->sm + u * J->d : NULL;
        st0.G = J->sS ? J->sG + u * ddv : NULL;
        st0.h = J->sS ? J->sh + u * J->d : NULL;
        st0.dS = J->dS ? J->dS + u * dd : NULL;
        st0.dC = J->dS ? J->dC + u * ddv : NULL;
        st0.dm = J->dS ? J->dm + u * J->d : NULL;
        st0.dG = J->dS ? J->dG + u * ddv : NULL;
        st0.dh = J->dS ? J->dh + u * J->d : NULL;
        backward_unit(J->n, J->d, J->dv, J->gamma ? J->gamma[u % J->H] : 1.0, J->normalize, J->eps, J->q + qo,
                      J->k + ko, J->v + kvo, J->go + vo, J->dq + qo, J->dk_pair + qo, J->dv_pair + vo, &st0);
    }
    return NULL;
}

/* Gradients of sum_t go_t . o_t with respect to q, k, v for the masked forward
 * from a zero state, ratio-normalised when `normalize` (o = num / (den + eps)).
 * q, go: [B][H][n][.]; k, v, dk, dv:
 * [B][Hkv][n][.] (H a multiple of Hkv; query head h reads key/value head
 * h / (H / Hkv)).  The gradient of a shared key or value is the sum of the
 * gradients through every query head of its group (chain rule), added in head order. */
/* The same from the state (S, C, m, G, h) before the first token (sS NULL: zeros; all
 * five [B*H][...] in the layout of the forward), also returning the gradient with
 * respect to that state (dS NULL: not wanted; all five then set). */
int hla_oracle_backward_state(int B, int H, int Hkv, int n, int d, int dv, int normalize, double eps,
                              const double *q, const double *k, const double *v, const double *gamma,
                              const double *go, const double *sS, const double *sC, const double *sm,
                              const double *sG, const double *sh, double *dq, double *dk, double *dvo, double *dS,
                              double *dC, double *dm, double *dG, double *dh, int nthreads);

int hla_oracle_backward(int B, int H, int Hkv, int n, int d, int dv, int normalize, double eps, const double *q,
                        const double *k, const double *v, const double *gamma, const double *go, double *dq,
                        double *dk, double *dvo, int nthreads)
{
    return hla_oracle_backward_state(B, H, Hkv, n, d, dv, normalize, eps, q, k, v, gamma, go, NULL, NULL, NULL, NULL,
                                     NULL, dq, dk, dvo, NULL, NULL, NULL, NULL, NULL, nthreads);
}

int hla_oracle_backward_state(int B, int H, int Hkv, int n, int d, int dv, int normalize, double eps,
                              const double *q, const double *k, const double *v, const double *gamma,
                              const double *go, const double *sS, const double *sC, const double *sm,
                              const double *sG, const double *sh, double *dq, double *dk, double *dvo, double *dS,
                              double *dC, double *dm, double *dG, double *dh, int nthreads)
{
    if (check_dims(B, H, n, d, dv) || Hkv < 1 || H % Hkv) return -1;
    if (sS && (!sC || !sm || !sG || !sh)) return -1;
    if (dS && (!dC || !dm || !dG || !dh)) return -1;
    const size_t nd = (size_t)n * d, ndv = (size_t)n * dv;
    double *dkp = (double *)calloc((size_t)B * H * nd + 1, sizeof(double));
    double *dvp = (double *)calloc((size_t)B * H * ndv + 1, sizeof(double));
    bjob_t J;
    memset(&J, 0, sizeof J);
    J.B = B; J.H = H; J.Hkv = Hkv; J.n = n; J.d = d; J.dv = dv; J.normalize = normalize; J.eps = eps;
    J.q = q; J.k = k; J.v = v; J.go = go; J.gamma = gamma;
    J.dq = dq; J.dk_pair = dkp; J.dv_pair = dvp;
    J.sS = sS; J.sC = sC; J.sm = sm; J.sG = sG; J.sh = sh;
    J.dS = dS; J.dC = dC; J.dm = dm; J.dG = dG; J.dh = dh;
    pthread_mutex_init(&J.lock, NULL);
    const int total = B * H;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > total) nthreads = total > 0 ? total : 1;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * nthreads);
    int started = 0;
    for (int i = 1; i < nthreads; ++i)
        if (pthread_create(&th[started], NULL, bworker, &J) == 0) ++started;
    bworker(&J);
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&J.lock);
    /* group sums */
    const int grp = H / Hkv;
    for (int b = 0; b < B; ++b)
        for (int j = 0; j < Hkv; ++j) {
            double *dko = dk + ((size_t)b * Hkv + j) * nd, *dvo_ = dvo + ((size_t)b * Hkv + j) * ndv;
            memset(dko, 0, nd * sizeof(double));
            memset(dvo_, 0, ndv * sizeof(double));
            for (int g = 0; g < grp; ++g) {
                const size_t u = (size_t)b * H + (size_t)j * grp + g;
                for (size_t e = 0; e < nd; ++e) dko[e] += dkp[u * nd + e];
                for (size_t e = 0; e < ndv; ++e) dvo_[e] += dvp[u * ndv + e];
            }
        }
    free(dkp);
    free(dvp);
    return 0;
}

/* Segment concatenation for `count` independent items: out_i = A_i (+) B_i
 * with f_i = decay_pow[i] (NULL: f = 1), by the rule of `variant` (0 masked,
 * 2 asymmetric; the unmasked state uses the masked rule's S, C, m).  out may
 * alias A or B. */
int hla_oracle_combine(int count, int d, int dv, int variant,
                       const double *SA, const double *CA, const double *mA,
                       const double *GA, const double *hA,
                       const double *SB, const double *CB, const double *mB,
                       const double *GB, const double *hB,
                       const double *decay_pow,
                       double *S, double *C, double *m, double *G, double *h)
{
    if (count < 0 || d < 1 || dv < 1 || variant < 0 || variant > 2) return -1;
    for (int i = 0; i < count; ++i) {
        const size_t a = (size_t)i * d * d, b = (size_t)i * d * dv, c = (size_t)i * d;
        combine_one(d, dv, decay_pow ? decay_pow[i] : 1.0, variant,
                    SA + a, CA + b, mA + c, GA + b, hA + c,
                    SB + a, CB + b, mB + c, GB + b, hB + c,
                    S + a, C + b, m + c, G + b, h + c);
    }
    return 0;
}
