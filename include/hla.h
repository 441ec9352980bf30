/*
 * hla.h -- C ABI of the GB300 (sm_103a) library for the second-order
 * Higher-order Linear Attention (HLA) forward (masked, and unmasked with
 * HLA_UNMASKED), its segment concatenation and its single-token decode step.
 *
 * Definitions (gist.science technical summary of "Higher-order Linear
 * Attention"):
 *   section 1, bullet "Onderhoud van de toestand": prefix summaries
 *       S_t = sum_{i<=t} k_i k_i^T (d x d), C_t = sum_{i<=t} q_i v_i^T (d x dv),
 *       m_t = sum_{i<=t} q_i (d);
 *   section 1, bullet "Strenge causaliteit": cross summaries
 *       G_t = G_{t-1} + k_t (k_t^T C_{t-1}) (d x dv), h_t = h_{t-1} + k_t (k_t^T m_{t-1}) (d);
 *   section 1, bullet "Outputformulering": o_t = q_t^T (S_t C_t - G_t);
 *   section 1, bullet "Normalisatie": ratio-normalised output
 *       o_t = q_t^T (S_t C_t - G_t) / (q_t^T (S_t m_t - h_t) + eps);
 *   section 4, bullets "Associatieve operatoren" and "Scan-equivalentie":
 *       segments combine by a semidirect product with cross term S_B C_A, and
 *       an exclusive scan over segment summaries reproduces the serial outputs;
 *   "Belangrijkste bijdragen", item 2: the same operators with exponential
 *       decay.  Decay reading used here: every prefix statistic decays by the
 *       head's factor g per token (S_t = g S_{t-1} + k k^T, C_t = g C_{t-1} +
 *       q v^T, m_t = g m_{t-1} + q), and G_t = g^2 G_{t-1} + g k_t (k_t^T C_{t-1}),
 *       h_t = g^2 h_{t-1} + g k_t (k_t^T m_{t-1}); g = 1 is the undecayed case.
 *
 * Unmasked variant (skill card "Higher-order linear attention", section
 * "Linear-Time Higher-Order Interactions", bullet "Streaming Computation"):
 *       o_t = q_t^T S_t C_t, ratio form o_t = q_t^T S_t C_t / (q_t^T S_t m_t + eps),
 *   with the same decayed S, C, m; G and h are not part of this variant.
 * Asymmetric variant AHLA (gist.science summary, section 2): the operator
 *   Q (K^T Q)(K^T V), masked to o_t = sum_{a<=b<=t} (q_t.k_b)(q_b.k_a) v_a, with
 *   summaries P_t = g P_{t-1} + k v^T, m^K_t = g m^K_{t-1} + k,
 *   E_t = g E_{t-1} + k (q^T P_t), n_t = g n_{t-1} + k (q . m^K_t), o_t = q_t^T E_t
 *   (ratio form: / (q_t^T n_t + eps)), and R_t = R_{t-1} + k q^T (no decay), which
 *   composes segments: E = f E_A + E_B + f R_B P_A, n = f n_A + n_B + f R_B m_A,
 *   R = R_A + R_B, P = f P_A + P_B, m^K = f m^K_A + m^K_B.  The state arrays hold
 *   R in S, P in C, m^K in m, E in G and n in h.
 * Shared key/value heads (same card, section "Architecture Overview", bullet
 *   "Multi-Head Support"): k and v may carry Hkv heads, H a multiple of Hkv;
 *   query head h reads key/value head h / (H / Hkv).  The summaries stay per
 *   query head.
 *
 * Conventions shared by every call
 *   - All tensors are caller-owned device memory; the library never allocates
 *     or frees device memory.  Inputs are read-only.
 *   - Every call is asynchronous on the given CUDA stream (`stream` is a
 *     cudaStream_t passed as void*; NULL is the legacy default stream).  The
 *     returned status covers argument validation and launch errors only.  A
 *     device-side failure (a bounded wait that expired) is recorded in a sticky
 *     device flag that hla_sync_status() reports.
 *   - On any status other than HLA_OK nothing was launched, except HLA_ERR_CUDA
 *     from a failed launch; hla_last_error() gives a message.
 *   - Layout: q is [B][H][n][d], k [B][Hkv][n][d], v [B][Hkv][n][dv], o
 *     [B][H][n][dv] (Hkv = H unless key/value heads are shared); all contiguous,
 *     row-major, 16-byte aligned, element type `in_dtype` (o has the input type;
 *     accumulation is fp32, the store rounds to nearest even).
 *   - State (one block per (b,h) pair, pair index u = b*H + h, fp32, contiguous,
 *     16-byte aligned): S [BH][d][d], C [BH][d][dv], m [BH][d], G [BH][d][dv],
 *     h [BH][d].
 */
#ifndef HLA_H
#define HLA_H

#include <stddef.h>

/* Exported entry points keep default visibility in a -fvisibility=hidden build. */
#if defined(__GNUC__)
#define HLA_API __attribute__((visibility("default")))
#else
#define HLA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    HLA_OK = 0,
    HLA_ERR_ARG = 1,          /* null pointer, bad size, misalignment, short workspace */
    HLA_ERR_UNSUPPORTED = 2,  /* valid arguments outside the supported shape set      */
    HLA_ERR_CUDA = 3,         /* a CUDA runtime call failed                           */
    HLA_ERR_TIMEOUT = 4       /* a bounded device-side wait expired (sticky flag)     */
} hla_status;

typedef enum { HLA_F32 = 0, HLA_BF16 = 1 } hla_dtype;

enum {
    HLA_NORMALIZE = 1u,  /* ratio-normalised output (section 1, "Normalisatie")          */
    HLA_DECAY = 2u,      /* per-head exponential decay ("Belangrijkste bijdragen", item 2) */
    HLA_UNMASKED = 4u,   /* unmasked output o = q^T S C (skill card, "Streaming Computation");
                            state carries S, C, m; G and h are written as zeros          */
    HLA_ASYMMETRIC = 8u  /* asymmetric variant AHLA (section 2): o = q^T E, see below;
                            not combined with HLA_UNMASKED                               */
};

typedef struct {
    int B, H, n;          /* batch, heads, tokens per sequence (n >= 0)               */
    int d, dv;            /* query/key width, value width                              */
    int chunk;            /* chunk length of the chunk-parallel scheme                 */
    hla_dtype in_dtype;   /* element type of q, k, v, o                                */
    unsigned flags;       /* HLA_NORMALIZE | HLA_DECAY                                 */
    float eps;            /* added to the denominator when HLA_NORMALIZE               */
    const float *gamma;   /* [H] device fp32 decay factors in [0,1]; required with
                             HLA_DECAY, ignored otherwise                               */
    int Hkv;              /* key/value heads (H % Hkv == 0); 0 means H                  */
} hla_params;

/* The five summaries of B*H (or N) pairs; all five pointers set, or the whole
 * struct pointer passed as NULL where a call allows it. */
typedef struct {
    float *S, *C, *m, *G, *h;
} hla_state;

/*
 * Supported shapes of hla_forward_chunked
 *   in_dtype HLA_BF16, d in {64,128}, dv in {64,128}, chunk in {64,128}:
 *       tensor-core path (tcgen05 MMA, TMEM accumulators, TMA tile loads);
 *       with HLA_ASYMMETRIC only dv <= d.
 *   in_dtype HLA_F32 or HLA_BF16 with d, dv, chunk in {16,32,64,128} (d, dv in
 *       {16,32,64} for HLA_UNMASKED and HLA_ASYMMETRIC), the shapes above excepted:
 *       CUDA-core fp32 path (fp32 inputs keep full precision).  One CTA per pair
 *       holds the pair's state in shared memory; where that leaves too little room,
 *       a chunk runs as several shorter ones (64 tokens at most; 32 at d = 128 with
 *       dv = 32 or 64, 8 at d = dv = 128), which changes only the rounding.
 *   HLA_ASYMMETRIC or HLA_UNMASKED with dv = 128 and d in {16,32,64} where neither
 *       path above takes the shape: two problems over the value columns [0,64) and
 *       [64,128), each on the path above for its shape (the output's and the state's
 *       C, G columns j depend on column j of v only; S, m, h on none); the workspace
 *       then also holds the gathered halves.
 *   Anything else: HLA_ERR_UNSUPPORTED.  Any n >= 0; a final partial chunk is
 *   handled exactly (decay is applied only over the tokens present).
 */

/* Bytes of device workspace hla_forward_chunked needs for these parameters
 * (0 if none).  Returns 0 as well for unsupported parameters; the forward call
 * itself reports the error.  The workspace holds the per-segment summaries of
 * the exclusive scan and the flags that order it. */
HLA_API size_t hla_forward_workspace_size(const hla_params *p);

/* Name of the kernel hla_forward_chunked launches for these parameters on the
 * current device: "fwd_ws2_kernel" (masked, no decay, bf16, d = dv = 64),
 * "fwd_ws_kernel" (masked, bf16, d = 64, the other widths and decay),
 * "fwd_tc_kernel" (other bf16 shapes) or "fwd_simt_kernel" (fp32 inputs).  NULL
 * for invalid or unsupported parameters and for n = 0 (no launch).  The string is
 * static; nothing is launched.  For tools that attribute measured time to a kernel. */
HLA_API const char *hla_forward_kernel(const hla_params *p);

/*
 * Masked second-order forward over n tokens for every (b,h) pair, by the
 * chunk-parallel scheme of section 4: per-segment summaries are combined with
 * the semidirect-product rule in an exclusive scan, and each chunk's outputs are
 * formed from its exact prefix state.  The result equals the serial recurrence
 * of section 1 up to floating-point rounding.
 *
 *   q, k, v   inputs as described above (read only);
 *   o         output [B][H][n][dv], in_dtype;
 *   state_in  state before the first token, or NULL for zeros;
 *   state_out state after the last token (S, C, m, G, h), or NULL to skip; may
 *             not alias state_in.  With HLA_UNMASKED, G and h of state_in are
 *             ignored and those of state_out are written as zeros;
 *   workspace device scratch of at least hla_forward_workspace_size(p) bytes,
 *             256-byte aligned, set to zero before its first use; every call
 *             (also one that ends in HLA_ERR_TIMEOUT) leaves its header and flags
 *             ready for the next call (a call generation in the header, which
 *             tags the flags), so it can be reused without clearing, also by a
 *             call with other parameters.  Calls sharing one workspace must not
 *             overlap in time.
 */
HLA_API hla_status hla_forward_chunked(const hla_params *p, const void *q, const void *k,
                               const void *v, void *o, const hla_state *state_in,
                               const hla_state *state_out, void *workspace,
                               size_t workspace_bytes, void *stream);

/*
 * Segment concatenation (section 4, "Associatieve operatoren"): for each of
 * `count` items, out = A (+) B where segment A precedes segment B in time:
 *   S = f S_A + S_B,  C = f C_A + C_B,  m = f m_A + m_B,
 *   G = f^2 G_A + G_B + f S_B C_A,  h = f^2 h_A + h_B + f S_B m_A,
 * with f = decay_pow[i] (= g^{len(B)}), or f = 1 when decay_pow is NULL.
 * flags: 0 (masked), HLA_UNMASKED (S, C, m as above; G, h written as zeros) or
 * HLA_ASYMMETRIC (the AHLA rule above: S = S_A + S_B, G = f G_A + G_B + f S_B C_A,
 * h = f h_A + h_B + f S_B m_A; other flag bits are ignored).
 * A, B, out: states of `count` items with widths d, dv (any d, dv in
 * {16,32,64,128}).  out may be A or B (all five pointers equal); partial
 * aliasing between different arrays is not allowed.  The product S_B C_A is
 * formed in fp32.
 */
HLA_API hla_status hla_state_combine(int count, int d, int dv, unsigned flags, const hla_state *A,
                             const hla_state *B, const hla_state *out,
                             const float *decay_pow, void *stream);

/*
 * One decode step (section 1 recurrence applied to a single new token) for N
 * independent (sequence, head) pairs, pair u = s*H + h; pair u uses gamma[h] when
 * HLA_DECAY is set.  The fp32 state is updated in place: the cross summaries
 * from C_{t-1}, m_{t-1}, then S, C, m; the output is
 * o = q^T (S_t C_t - G_t) (divided by q^T (S_t m_t - h_t) + eps with
 * HLA_NORMALIZE).  With HLA_UNMASKED the output is o = q^T S_t C_t (divided by
 * q^T S_t m_t + eps), and G, h are neither read nor written (they may be NULL).
 * With HLA_ASYMMETRIC the state is (R, P, m^K, E, n) and the output q^T E_t.
 *   q: [N][d], o: [N][dv]; k: [N/H*Hkv][d], v: [N/H*Hkv][dv] (row s*Hkv + h/(H/Hkv)
 *   for pair u); element type `dtype` (HLA_F32 or HLA_BF16);
 *   Hkv: key/value heads per sequence, H % Hkv == 0 (0 means H);
 *   state: N pairs, read and written in place;
 *   d, dv in {16,32,64,128}; N % H == 0.
 */
HLA_API hla_status hla_decode_step(int N, int H, int Hkv, int d, int dv, hla_dtype dtype, unsigned flags,
                           float eps, const float *gamma, const hla_state *state,
                           const void *q, const void *k, const void *v, void *o,
                           void *stream);

/*
 * Backward pass (training) of the masked forward from a zero initial state (from a
 * given one: hla_backward_chunked_state below).  The pages motivate chunk-parallel training (section 4) but give no gradient; this
 * call is reverse-mode differentiation of the section 1 recurrence, evaluated
 * chunk-parallel: per-chunk local sums, a scan over chunks (the states S,
 * X = S C - G forward in time and the adjoints dL/dX, dL/dS backward in time),
 * then per-chunk gradients.  Its result equals the gradient of sum_t dout_t . o_t
 * up to floating-point rounding.
 *
 * With HLA_NORMALIZE the output is o_t = n_t / (den_t + eps), den_t = q_t^T
 * (S_t m_t - h_t) (section 1, "Normalisatie").  den is the unnormalised output of
 * unit values, so the gradient is that of the unnormalised output of the values
 * [V | 1] with upstream [r dout | -r (dout . o)], r = 1 / (den + eps).  The two
 * parts of dq and dk cancel to a large degree.  For bf16 inputs with d = dv =
 * chunk = 64 (and no given state, below) it runs on the tensor cores in nine
 * launches: the forward's local sums and scan, the outputs with r and the upstream,
 * the backward's scan and the gradients; every product over the value index, where
 * the two parts meet, is formed from bf16 hi + lo operands (about fp32 accuracy)
 * and the unit column's terms in fp32.  Otherwise it is a chain of two unnormalised
 * forwards, an elementwise kernel, two unnormalised backwards and a sum, in fp32
 * throughout (bf16 inputs are widened first) on the CUDA-core kernels.
 *
 *   p      as for hla_forward_chunked; supported: flags 0, HLA_DECAY, HLA_NORMALIZE
 *          (eps >= 0) or both (HLA_UNMASKED, HLA_ASYMMETRIC: HLA_ERR_UNSUPPORTED),
 *          Hkv dividing H (0 means H), d, dv and chunk in {16,32,64,128}, in_dtype
 *          HLA_F32 or HLA_BF16.  dv = 128 runs as two problems over the value columns [0,64) and
 *          [64,128) (the loss is a sum over value columns, each depending on its own
 *          column of v only): dq and dk are their sum, formed in fp32 and rounded once,
 *          dv their two halves; not with a given state or its gradient
 *          (HLA_ERR_UNSUPPORTED).  A 128-token chunk runs as two chunks of 64 tokens
 *          (the same gradient up to rounding).  d = 128 runs on the CUDA cores in
 *          16-token chunks (whatever chunk is given) over slices of 32 value columns
 *          when dv > 32, split as above;
 *   q      [B][H][n][d], k [B][Hkv][n][d], v [B][Hkv][n][dv], dout [B][H][n][dv],
 *          in_dtype, read only (query head h reads key/value head h / (H / Hkv));
 *   dq     [B][H][n][d], dk [B][Hkv][n][d], dv [B][Hkv][n][dv], in_dtype, written (not
 *          accumulated); with Hkv < H, dk and dv are the sums over each group;
 *   workspace device scratch of at least hla_backward_workspace_size(p) bytes,
 *          16-byte aligned (256-byte aligned with HLA_NORMALIZE or a split over value
 *          columns), no initial contents needed.
 * All tensor pointers 16-byte aligned.  Without HLA_NORMALIZE three kernel phases
 * on `stream` (plus the group sums when Hkv < H); with it, the launches above.
 */
HLA_API size_t hla_backward_workspace_size(const hla_params *p);
HLA_API hla_status hla_backward_chunked(const hla_params *p, const void *q, const void *k, const void *v,
                                        const void *dout, void *dq, void *dk, void *dv, void *workspace,
                                        size_t workspace_bytes, void *stream);

/*
 * hla_backward_chunked from a given initial state, with the gradient of that state:
 * the forward it differentiates is hla_forward_chunked with state_in, so the outputs
 * continue a stream whose state before the first token is (S, C, m, G, h); the state
 * enters the recurrence as S_in and X_in = S_in C_in - G_in.  Reverse mode gives, from
 * the adjoints at the first token (Lam = dL/dX, Om = dL/dS after it, decay g per token),
 *   dX_in = g^2 Lam,  dG = -dX_in,  dC = S_in^T dX_in,  dS = g Om + dX_in C_in^T,
 * and zero for m and h without normalisation (they enter only the denominator).  With
 * HLA_NORMALIZE the chain above runs from the state: the values' pass from (S, C, G),
 * the unit values' pass from (S, C1, G1) with m, h in column 0 of C1, G1 (Y_in =
 * S_in m_in - h_in is the unit values' X_in), and dS adds both passes' dS, while dm
 * and dh are column 0 of the unit pass's dC1, dG1.
 *   state_in    (S, C, m, G, h) fp32 [B*H][...] as for hla_forward_chunked, or NULL
 *               (zeros; the call is then hla_backward_chunked plus the state gradient);
 *   d_state_in  five fp32 arrays of the same shapes, written, or NULL (not wanted);
 *   the rest as for hla_backward_chunked (same workspace size).
 * With a state or its gradient the scan between the local sums and the gradients runs
 * on the CUDA cores (also on the tensor-core shape), plus one launch per pass for the
 * state gradient; with HLA_NORMALIZE it is the CUDA-core chain.
 */
HLA_API hla_status hla_backward_chunked_state(const hla_params *p, const void *q, const void *k, const void *v,
                                              const void *dout, const hla_state *state_in, void *dq, void *dk,
                                              void *dv, const hla_state *d_state_in, void *workspace,
                                              size_t workspace_bytes, void *stream);

/* hla_backward_chunked with per-phase tracing: phase_events is NULL (then this is
 * hla_backward_chunked) or four cudaEvent_t handles of the current device, recorded
 * on `stream` before the local-sums kernel, after it, after the scan kernel and
 * after the gradient kernel.  With HLA_NORMALIZE: at the start, after the two
 * forwards and the upstream-gradient kernel, after the first backward and at the
 * end.  The caller owns the events (created with timing enabled to read elapsed
 * times).  With n == 0 no event is recorded. */
HLA_API hla_status hla_backward_chunked_traced(const hla_params *p, const void *q, const void *k, const void *v,
                                               const void *dout, void *dq, void *dk, void *dv, void *workspace,
                                               size_t workspace_bytes, void *stream, void *const *phase_events);

/*
 * Masked third-order HLA (section 3 "Derde-orde HLA": the operator A A^T A with
 * A = Q K^T, every factor causal):
 *   o_t = sum_{b<=t} sum_{a<=b} sum_{c<=b} (q_t.k_a)(k_a.q_b)(q_b.k_c) v_c = q_t^T T_t,
 *   T_t = sum_{b<=t} S^K_b q_b q_b^T P_b   (= S^K S^Q P^KV minus the cross summaries
 *   G1 + G2 - G3 that remove a key after its query),
 * with S^K_t = sum k k^T and P_t = sum k v^T.  The streaming state of a pair is
 * (S [d][d] = S^K, P [d][dv], T [d][dv]), fp32.
 *
 * HLA_DECAY (gamma [H]): every prefix moment decays by gamma per token, so the triple
 * a, b, c <= t weighs gamma^(3t-a-b-c); the updates become S^K_t = g S^K + k k^T,
 * P_t = g P + k v^T, T_t = g^3 T + (S^K_t q)(P_t^T q)^T.  The section states no
 * decayed third order; this is the second order's reading carried over.
 * HLA_NORMALIZE (eps >= 0): o_t = num_t / (den_t + eps), den_t the masked output of
 * unit values, q_t^T h_t with the key mass m_t = g m + k (P of a unit value) and
 * h_t = g^3 h + (S^K_t q)(m_t . q) (T of a unit value; it combines the cross summaries
 * h^(1..3) the section names as T combines G^(1..3)).  m [d] and h [d] are then part of
 * the state; without HLA_NORMALIZE they are not used (may be NULL).
 *
 * Segment maps (section 4, "Derde-orde scans"): to concatenate two states with
 * hla_state3_combine, each also carries the maps of its tokens, S^Q = sum q q^T [d][d],
 * M^QP = sum_b q_b q_b^T P_b [d][dv] (the map P -> S^K_A M^QP_B), M^KQ = sum_b S^K_b q_b
 * q_b^T [d][d] (the map P -> M^KQ_B P, named M^KQP), and with normalisation mqm [d],
 * the M^QP of a unit value (so M^KQ m is the map M^KQm).  The maps are optional: the
 * forward writes them when state_out->SQ is set (then state_in, if given, must carry
 * them too), and the decode step neither reads nor writes them.
 */
typedef struct {
    float *S, *P, *T;
    float *m, *h;
    float *SQ, *MQP, *MKQ, *mqm;
} hla_state3;

/* Bytes of device workspace hla_forward3_chunked needs (0 for invalid parameters). */
HLA_API size_t hla_forward3_workspace_size(const hla_params *p);

/*
 * Masked third-order forward over n tokens for every (b,h) pair, chunk-parallel
 * (section 4, "Derde-orde scans"): chunk-local sums, a scan over chunks that composes
 * states with the segment-level linear maps M^KQ and M^QP, then per-chunk outputs.
 *   p         flags 0, HLA_DECAY (gamma [H], values in [0, 1]), HLA_NORMALIZE
 *             (eps >= 0) or both; Hkv dividing H (0 means H); d, dv and chunk in {16,32,64,128};
 *             in_dtype HLA_F32 or HLA_BF16 (fp32 arithmetic).  dv = 128 runs as two
 *             problems over the value columns [0,64) and [64,128): the output's
 *             column j and the state's P, T, M^QP columns j depend on column j of v
 *             only, while S, S^Q, M^KQ, m, h, mqm depend on no value column; each half
 *             writes its columns of o and of state_out.  A 128-token chunk runs as two
 *             of 64 tokens (the same result up to rounding).  d = 128 runs on the CUDA
 *             cores in 16-token chunks (whatever chunk is given) over slices of 32
 *             value columns when dv > 32, split as above;
 *   q         [B][H][n][d], k [B][Hkv][n][d], v [B][Hkv][n][dv], o [B][H][n][dv]; in_dtype
 *             (query head h reads key/value head h / (H / Hkv); the state is per query head);
 *   state_in  (S, P, T; with HLA_NORMALIZE also m, h) before the first token, or NULL
 *             for zeros;
 *   state_out (S, P, T; with HLA_NORMALIZE also m, h) after the last token, or NULL;
 *             may not alias state_in;
 *   workspace at least hla_forward3_workspace_size(p) bytes, 16-byte aligned (256-byte
 *             aligned with HLA_NORMALIZE or a split over value columns).
 * Three kernel launches on `stream` (tensor cores for bf16 at 64/64/64 without decay,
 * CUDA cores otherwise).  With HLA_NORMALIZE the numerator and the denominator (a
 * 16-wide unit-value tile with the same S) are two such forwards, followed by an
 * elementwise division; the denominator passes through the input element type.
 */
HLA_API hla_status hla_forward3_chunked(const hla_params *p, const void *q, const void *k, const void *v, void *o,
                                        const hla_state3 *state_in, const hla_state3 *state_out, void *workspace,
                                        size_t workspace_bytes, void *stream);

/* hla_forward3_chunked recording four caller-owned events on `stream` (NULL: none):
 * before the local-sums kernel, after it, after the scan and after the output kernel
 * (with a split over value columns: the first before the call, the other three after it). */
HLA_API hla_status hla_forward3_chunked_traced(const hla_params *p, const void *q, const void *k, const void *v,
                                               void *o, const hla_state3 *state_in, const hla_state3 *state_out,
                                               void *workspace, size_t workspace_bytes, void *stream,
                                               void *const *phase_events);

/*
 * One third-order decode step for N independent pairs, state updated in place
 * (g = gamma[i % H] with HLA_DECAY, else 1):
 *   S = g S + k k^T;  P = g P + k v^T;  T = g^3 T + (S q)(P^T q)^T;  o = T^T q;
 * with HLA_NORMALIZE also m = g m + k, h = g^3 h + (S q)(m . q) and o /= (h . q + eps).
 * q, k: [N][d], v, o: [N][dv], element type `dtype`; d, dv in {16,32,64,128}; flags
 * 0, HLA_DECAY, HLA_NORMALIZE or both; H >= 1 (only the decay rate's index uses it).
 */
HLA_API hla_status hla_decode3_step(int N, int H, int d, int dv, hla_dtype dtype, unsigned flags, float eps,
                                    const float *gamma, const hla_state3 *state, const void *q, const void *k,
                                    const void *v, void *o, void *stream);

/*
 * Concatenation of third-order states with their segment maps (section 4, "Derde-orde
 * scans"), segment A before segment B, for `count` independent items; with decay
 * f = decay_pow[i] = gamma^(tokens of B) (NULL: 1):
 *   S^K = f S^K_A + S^K_B,  S^Q = f S^Q_A + S^Q_B,  P = f P_A + P_B,
 *   T = f^3 T_A + T_B + f S^K_A M^QP_B + f M^KQ_B P_A + f^2 S^K_A S^Q_B P_A,
 *   M^QP = f^2 M^QP_A + M^QP_B + f S^Q_B P_A,   M^KQ = f^2 M^KQ_A + M^KQ_B + f S^K_A S^Q_B,
 * and with HLA_NORMALIZE the unit column likewise (m as P, h as T, mqm as M^QP).
 * A, B, out: hla_state3 with S, P, T, SQ, MQP, MKQ (and m, h, mqm with HLA_NORMALIZE),
 * fp32 [count][...]; out may alias A or B (each item is read whole before it is
 * written).  flags: 0 or HLA_NORMALIZE; d and dv in {16, 32, 64, 128}.  One launch on
 * `stream` (at d = 128 in two phases inside it: P, T, M^QP and the unit column, then
 * S, S^Q, M^KQ, each staging what it overwrites).
 */
HLA_API hla_status hla_state3_combine(int count, int d, int dv, unsigned flags, const hla_state3 *A,
                                      const hla_state3 *B, const hla_state3 *out, const float *decay_pow,
                                      void *stream);

/* Self-test of the failure path: launches one CTA that waits, with the library's
 * bounded barrier wait (a short poll limit), on a barrier that nothing completes.  The
 * wait expires, raises the sticky device flag and the kernel returns; nothing traps or
 * hangs.  The next hla_sync_status on `stream` reports HLA_ERR_TIMEOUT (once) and the
 * context stays usable. */
HLA_API hla_status hla_selftest_expired_wait(void *stream);

/* Synchronise `stream`, then report and clear the sticky device flag: HLA_OK,
 * HLA_ERR_TIMEOUT if a bounded device wait expired since the last call, or
 * HLA_ERR_CUDA if the stream reported an error. */
HLA_API hla_status hla_sync_status(void *stream);

/* Static description of a status code. */
HLA_API const char *hla_status_string(hla_status s);

/* Message describing the most recent non-OK status returned on this thread. */
HLA_API const char *hla_last_error(void);

/*
 * Forward pass for callers that cannot allocate device memory.  The paper has
 * no counterpart to this entry point; it exists for the library's users.
 *
 * Some callers cannot call cudaMalloc while they run: code executing inside a
 * host allocator hook or an allocation-free real-time loop, or a host that
 * hands out device memory only up front.  They cannot provide the workspace
 * that hla_forward_chunked needs.  This call computes exactly what
 * hla_forward_chunked computes (same arguments, same kernels) but takes its
 * scratch from one array of HLA_NOALLOC_SCRATCH_BYTES bytes that the library
 * keeps in device memory; it allocates nothing.  Every GPU that loads the
 * library holds that array until the process exits.
 *
 *   - The first call on a device looks up the array's device address while
 *     that device is current; make that first call before any stream capture.
 *     The address is kept per device together with the context it was taken
 *     in: after cudaDeviceReset (or another teardown of the primary context)
 *     the next call looks it up again, so make that call before any capture too.
 *   - Each call clears the forward's ordering header and release flags at the
 *     front of the array (one cudaMemsetAsync on `stream`) and then runs the
 *     ordinary forward on the array; the rest of the array keeps whatever the
 *     last call left there.
 *   - Every call shares the one array.  Calls that may overlap on the GPU
 *     (different streams, or different host threads on one device) race and
 *     corrupt each other's results: serialise them.
 *   - Parameters whose scratch need (hla_forward_workspace_size) exceeds
 *     HLA_NOALLOC_SCRATCH_BYTES are rejected with HLA_ERR_UNSUPPORTED before any
 *     device work.  Shapes served by the CUDA-core path need no scratch.
 */
#define HLA_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
HLA_API hla_status hla_forward_chunked_noalloc(const hla_params *p, const void *q, const void *k,
                                               const void *v, void *o, const hla_state *state_in,
                                               const hla_state *state_out, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* HLA_H */
