// hla_fwd_simt.cu -- chunked masked second-order HLA forward on CUDA cores, fp32
// arithmetic, for fp32 inputs and for widths the tensor-core kernels do not take (any
// input dtype): d, dv in {16,32,64,128} (128 for the masked variant only).
//
// One CTA per (b,h) pair walks the chunks in order, keeping the pair's state on
// chip.  Instead of G and h it carries X = S C - G (d x dv) and Y = S m - h (d),
// which obey X_t = g^2 X_{t-1} + u_t v_t^T and Y_t = g^2 Y_{t-1} + u_t with
// u_t = S_t q_t, and give o_t = q_t^T X_t, den_t = q_t^T Y_t.  (Both identities
// follow from the recurrence of the gist.science summary, section 1: expand
// S_t C_t - G_t with the updates of S, C and G.)  Per chunk of L tokens with
// local positions tau = 1..L after the prefix position p:
//   A[t,a] = g^{t-a} q_t.k_a            (a <= t)
//   u_b    = g^{tau_b} S_p q_b + sum_{a<=b} A[b,a] k_a        (= S_b q_b)
//   M[t,b] = g^{2(t-b)} q_t.u_b         (b <= t)
//   o_t    = sum_b M[t,b] v_b + g^{2 tau_t} q_t^T X_p
//   den_t  = sum_b M[t,b]     + g^{2 tau_t} q_t^T Y_p
// and the state moves to the chunk end with weights w_b = g^{L - tau_b}.
// Unmasked variant (o_t = q_t^T S_t C_t = u_t^T C_t; skill card "Higher-order
// linear attention", bullet "Streaming Computation"): with the same u,
//   M[t,b] = g^{t-b} u_t.q_b            (b <= t)
//   o_t    = sum_b M[t,b] v_b + g^{tau_t} u_t^T C_p,  den_t = sum_b M[t,b] + g^{tau_t} u_t.m_p
// and only S, C, m are carried.  Asymmetric variant AHLA (gist.science summary,
// section 2; state R, P, m^K, E, n kept in the S, C, m, X, Y buffers): with the
// same A,
//   z_b    = g^{tau_b} P_p^T q_b + sum_{a<=b} A[b,a] v_a       (= P_b^T q_b)
//   zeta_b = g^{tau_b} q_b.m_p + sum_{a<=b} A[b,a]              (= q_b . m^K_b)
//   o_t    = g^{tau_t} q_t^T E_p + sum_{b<=t} A[t,b] z_b,  den_t = g^{tau_t} q_t.n_p + sum_b A[t,b] zeta_b
// and P, m^K, E, n move to the chunk end with w_b, R = R + sum_b k_b q_b^T (no decay).
// Key/value heads may be shared: query head h reads key/value head h / (H / Hkv).
#include "hla_internal.h"
#include "hla_smem_tile.cuh"

namespace hla {
namespace {

template <typename T>
__device__ __forceinline__ float ld_in(const T *p, size_t i);
template <>
__device__ __forceinline__ float ld_in<float>(const float *p, size_t i) { return p[i]; }
template <>
__device__ __forceinline__ float ld_in<__nv_bfloat16>(const __nv_bfloat16 *p, size_t i) {
    return __bfloat162float(p[i]);
}
template <typename T>
__device__ __forceinline__ void st_out(T *p, size_t i, float x);
template <>
__device__ __forceinline__ void st_out<float>(float *p, size_t i, float x) { p[i] = x; }
template <>
__device__ __forceinline__ void st_out<__nv_bfloat16>(__nv_bfloat16 *p, size_t i, float x) {
    p[i] = __float2bfloat16_rn(x);
}

constexpr int kThreads = 256;
constexpr int kMaxChunk = 64;

template <typename T, int D, int DV>
__global__ void __launch_bounds__(kThreads) fwd_simt_kernel(FwdArgs a) {
    extern __shared__ float sm[];
    const int c = a.chunk;
    float *S = sm;                  // D*D
    float *X = S + D * D;           // D*DV
    float *Cs = X + D * DV;         // D*DV
    float *m = Cs + D * DV;         // D
    float *Y = m + D;               // D
    float *Q = Y + D;               // c*D
    float *K = Q + kMaxChunk * D;   // c*D
    float *V = K + kMaxChunk * D;   // c*DV
    constexpr int DU = D > DV ? D : DV;
    float *U = V + kMaxChunk * DV;  // c*D (u-vectors), or c*DV (z-vectors of the asymmetric variant)
    float *A = U + kMaxChunk * DU;  // c*c (A, then M)
    float *Z = A + kMaxChunk * kMaxChunk;  // c: zeta of the asymmetric variant
    float *gp = Z + kMaxChunk;      // g^x, x = 0..2c+1

    const int tid = threadIdx.x;
    const int u = blockIdx.x;  // pair index b*H + h
    const int hh = u % a.H;
    const bool decay = (a.flags & HLA_DECAY) != 0;
    const bool norm = (a.flags & HLA_NORMALIZE) != 0;
    const bool unm = (a.flags & HLA_UNMASKED) != 0;
    const bool asym = (a.flags & HLA_ASYMMETRIC) != 0;
    const float g = decay ? a.gamma[hh] : 1.f;
    const float lg = log2f(g);
    const size_t kvu = (size_t)(u / a.H) * a.Hkv + hh / (a.H / a.Hkv);  // key/value head
    const T *q = static_cast<const T *>(a.q) + (size_t)u * a.n * D;
    const T *k = static_cast<const T *>(a.k) + kvu * a.n * D;
    const T *v = static_cast<const T *>(a.v) + kvu * a.n * DV;
    T *o = static_cast<T *>(a.o) + (size_t)u * a.n * DV;

    for (int x = tid; x <= 2 * c + 1; x += kThreads) gp[x] = decay ? gpow(lg, (float)x) : 1.f;

    // ---- prefix state
    if (a.sin.S && asym) {  // R, P, m^K, E, n as stored
        const float *Si = a.sin.S + (size_t)u * D * D, *Ci = a.sin.C + (size_t)u * D * DV;
        const float *mi = a.sin.m + (size_t)u * D, *Gi = a.sin.G + (size_t)u * D * DV, *hi = a.sin.h + (size_t)u * D;
        for (int e = tid; e < D * D; e += kThreads) S[e] = Si[e];
        for (int e = tid; e < D * DV; e += kThreads) { Cs[e] = Ci[e]; X[e] = Gi[e]; }
        for (int e = tid; e < D; e += kThreads) { m[e] = mi[e]; Y[e] = hi[e]; }
    } else if (a.sin.S) {
        const float *Si = a.sin.S + (size_t)u * D * D, *Ci = a.sin.C + (size_t)u * D * DV;
        const float *mi = a.sin.m + (size_t)u * D, *Gi = a.sin.G + (size_t)u * D * DV, *hi = a.sin.h + (size_t)u * D;
        for (int e = tid; e < D * D; e += kThreads) S[e] = Si[e];
        for (int e = tid; e < D * DV; e += kThreads) Cs[e] = Ci[e];
        for (int e = tid; e < D; e += kThreads) m[e] = mi[e];
        __syncthreads();
        for (int e = tid; e < D * DV && !unm; e += kThreads) {  // X = S C - G
            const int i = e / DV, j = e % DV;
            float acc = 0.f;
            for (int l = 0; l < D; ++l) acc += S[i * D + l] * Cs[l * DV + j];
            X[e] = acc - Gi[e];
        }
        for (int i = tid; i < D && !unm; i += kThreads) {  // Y = S m - h
            float acc = 0.f;
            for (int l = 0; l < D; ++l) acc += S[i * D + l] * m[l];
            Y[i] = acc - hi[i];
        }
    } else {
        for (int e = tid; e < D * D; e += kThreads) S[e] = 0.f;
        for (int e = tid; e < D * DV; e += kThreads) X[e] = Cs[e] = 0.f;
        for (int e = tid; e < D; e += kThreads) m[e] = Y[e] = 0.f;
    }
    __syncthreads();

    for (int t0 = 0; t0 < a.n; t0 += c) {
        const int L = min(c, a.n - t0);
        for (int e = tid; e < c * D; e += kThreads) {
            const int t = e / D;
            Q[e] = t < L ? ld_in(q, (size_t)t0 * D + e) : 0.f;
            K[e] = t < L ? ld_in(k, (size_t)t0 * D + e) : 0.f;
        }
        for (int e = tid; e < c * DV; e += kThreads) {
            const int t = e / DV;
            V[e] = t < L ? ld_in(v, (size_t)t0 * DV + e) : 0.f;
        }
        __syncthreads();
        // A[t,a] = g^{t-a} q_t.k_a, a <= t
        for (int e = tid; e < c * c; e += kThreads) {
            const int t = e / c, s = e % c;
            float acc = 0.f;
            if (s <= t) {
                for (int i = 0; i < D; ++i) acc += Q[t * D + i] * K[s * D + i];
                acc *= gp[t - s];
            }
            A[e] = acc;
        }
        __syncthreads();
        if (asym) {
            // z_b = g^{b+1} (P_p^T q_b) + sum_{a<=b} A[b,a] v_a; zeta_b likewise with m_p and 1
            for (int e = tid; e < c * DV; e += kThreads) {
                const int b = e / DV, j = e % DV;
                float pz = 0.f;
                for (int i = 0; i < D; ++i) pz += Q[b * D + i] * Cs[i * DV + j];
                float acc = gp[b + 1] * pz;
                for (int s2 = 0; s2 <= b; ++s2) acc += A[b * c + s2] * V[s2 * DV + j];
                U[e] = acc;
            }
            for (int b = tid; b < c; b += kThreads) {
                float qm = 0.f;
                for (int i = 0; i < D; ++i) qm += Q[b * D + i] * m[i];
                float acc = gp[b + 1] * qm;
                for (int s2 = 0; s2 <= b; ++s2) acc += A[b * c + s2];
                Z[b] = acc;
            }
            __syncthreads();
            // o_t = g^{t+1} q_t^T E_p + sum_{b<=t} A[t,b] z_b  [/ (g^{t+1} q_t.n_p + sum_b A[t,b] zeta_b + eps)]
            for (int e = tid; e < L * DV; e += kThreads) {
                const int t = e / DV, j = e % DV;
                float num = 0.f;
                for (int b = 0; b <= t; ++b) num += A[t * c + b] * U[b * DV + j];
                float pe = 0.f;
                for (int i = 0; i < D; ++i) pe += Q[t * D + i] * X[i * DV + j];
                num += gp[t + 1] * pe;
                if (norm) {
                    float den = 0.f;
                    for (int b = 0; b <= t; ++b) den += A[t * c + b] * Z[b];
                    float pn = 0.f;
                    for (int i = 0; i < D; ++i) pn += Q[t * D + i] * Y[i];
                    den += gp[t + 1] * pn;
                    num = num / (den + a.eps);
                }
                st_out(o, (size_t)t0 * DV + e, num);
            }
            __syncthreads();
            // state to the chunk end: R += K^T Q, P, m^K, E, n with w_b = g^{L-1-b}
            const float gL = gp[L];
            for (int e = tid; e < D * D; e += kThreads) {
                const int i = e / D, j = e % D;
                float acc = 0.f;
                for (int s2 = 0; s2 < L; ++s2) acc += K[s2 * D + i] * Q[s2 * D + j];
                S[e] += acc;
            }
            for (int e = tid; e < D * DV; e += kThreads) {
                const int i = e / DV, j = e % DV;
                float ap = 0.f, ae = 0.f;
                for (int b = 0; b < L; ++b) {
                    const float wk = gp[L - 1 - b] * K[b * D + i];
                    ap += wk * V[b * DV + j];
                    ae += wk * U[b * DV + j];
                }
                Cs[e] = gL * Cs[e] + ap;
                X[e] = gL * X[e] + ae;
            }
            for (int i = tid; i < D; i += kThreads) {
                float am = 0.f, an = 0.f;
                for (int b = 0; b < L; ++b) {
                    const float wk = gp[L - 1 - b] * K[b * D + i];
                    am += wk;
                    an += wk * Z[b];
                }
                m[i] = gL * m[i] + am;
                Y[i] = gL * Y[i] + an;
            }
            __syncthreads();
            continue;
        }
        // u_b = g^{b+1} (S_p q_b) + sum_{a<=b} A[b,a] k_a   (S symmetric)
        for (int e = tid; e < c * D; e += kThreads) {
            const int b = e / D, i = e % D;
            float ps = 0.f;
            for (int j = 0; j < D; ++j) ps += S[i * D + j] * Q[b * D + j];
            float acc = gp[b + 1] * ps;
            for (int s = 0; s <= b; ++s) acc += A[b * c + s] * K[s * D + i];
            U[e] = acc;
        }
        __syncthreads();
        // M[t,b] = g^{2(t-b)} q_t.u_b (unmasked: g^{t-b} u_t.q_b), b <= t  (overwrites A)
        for (int e = tid; e < c * c; e += kThreads) {
            const int t = e / c, b = e % c;
            float acc = 0.f;
            if (b <= t) {
                if (unm) {
                    for (int i = 0; i < D; ++i) acc += U[t * D + i] * Q[b * D + i];
                    acc *= gp[t - b];
                } else {
                    for (int i = 0; i < D; ++i) acc += Q[t * D + i] * U[b * D + i];
                    acc *= gp[2 * (t - b)];
                }
            }
            A[e] = acc;
        }
        __syncthreads();
        // outputs; the prefix term is g^{2 tau} q^T X_p (masked) or g^{tau} u^T C_p (unmasked)
        for (int e = tid; e < L * DV; e += kThreads) {
            const int t = e / DV, j = e % DV;
            float num = 0.f;
            for (int b = 0; b <= t; ++b) num += A[t * c + b] * V[b * DV + j];
            const float *lhs = unm ? U + t * D : Q + t * D;
            const float *Rx = unm ? Cs : X, *Ry = unm ? m : Y;
            float px = 0.f;
            for (int i = 0; i < D; ++i) px += lhs[i] * Rx[i * DV + j];
            const float gt = unm ? gp[t + 1] : gp[2 * (t + 1)];
            num += gt * px;
            if (norm) {
                float den = 0.f;
                for (int b = 0; b <= t; ++b) den += A[t * c + b];
                float py = 0.f;
                for (int i = 0; i < D; ++i) py += lhs[i] * Ry[i];
                den += gt * py;
                num = num / (den + a.eps);
            }
            st_out(o, (size_t)t0 * DV + e, num);
        }
        __syncthreads();
        // state to the chunk end, weights w_b = g^{L-1-b}
        const float gL = gp[L], g2L = gp[2 * L];
        for (int e = tid; e < D * D; e += kThreads) {
            const int i = e / D, j = e % D;
            float acc = 0.f;
            for (int s = 0; s < L; ++s) acc += gp[L - 1 - s] * K[s * D + i] * K[s * D + j];
            S[e] = gL * S[e] + acc;
        }
        for (int e = tid; e < D * DV; e += kThreads) {
            const int i = e / DV, j = e % DV;
            float ax = 0.f, ac = 0.f;
            for (int b = 0; b < L; ++b) {
                if (!unm) ax += gp[2 * (L - 1 - b)] * U[b * D + i] * V[b * DV + j];
                ac += gp[L - 1 - b] * Q[b * D + i] * V[b * DV + j];
            }
            if (!unm) X[e] = g2L * X[e] + ax;
            Cs[e] = gL * Cs[e] + ac;
        }
        for (int i = tid; i < D; i += kThreads) {
            float am = 0.f, ay = 0.f;
            for (int b = 0; b < L; ++b) {
                am += gp[L - 1 - b] * Q[b * D + i];
                if (!unm) ay += gp[2 * (L - 1 - b)] * U[b * D + i];
            }
            m[i] = gL * m[i] + am;
            if (!unm) Y[i] = g2L * Y[i] + ay;
        }
        __syncthreads();
        // re-tabulate is unnecessary: gp depends only on g
    }

    if (a.sout.S && asym) {  // R, P, m^K, E, n as stored
        float *So = a.sout.S + (size_t)u * D * D, *Co = a.sout.C + (size_t)u * D * DV;
        float *mo = a.sout.m + (size_t)u * D, *Go = a.sout.G + (size_t)u * D * DV, *ho = a.sout.h + (size_t)u * D;
        for (int e = tid; e < D * D; e += kThreads) So[e] = S[e];
        for (int e = tid; e < D * DV; e += kThreads) { Co[e] = Cs[e]; Go[e] = X[e]; }
        for (int i = tid; i < D; i += kThreads) { mo[i] = m[i]; ho[i] = Y[i]; }
    } else if (a.sout.S) {
        float *So = a.sout.S + (size_t)u * D * D, *Co = a.sout.C + (size_t)u * D * DV;
        float *mo = a.sout.m + (size_t)u * D, *Go = a.sout.G + (size_t)u * D * DV, *ho = a.sout.h + (size_t)u * D;
        for (int e = tid; e < D * D; e += kThreads) So[e] = S[e];
        for (int e = tid; e < D * DV; e += kThreads) {
            const int i = e / DV, j = e % DV;
            float acc = 0.f;  // (S C)[i][j]
            for (int l = 0; l < D && !unm; ++l) acc += S[i * D + l] * Cs[l * DV + j];
            Co[e] = Cs[e];
            Go[e] = unm ? 0.f : acc - X[e];  // G is not part of the unmasked state
        }
        for (int i = tid; i < D; i += kThreads) {
            float acc = 0.f;
            for (int l = 0; l < D && !unm; ++l) acc += S[i * D + l] * m[l];
            mo[i] = m[i];
            ho[i] = unm ? 0.f : acc - Y[i];
        }
    }
}

// ---- masked variant with register tiles ---------------------------------------
// The same chunk algebra as above for the masked (optionally normalised, decayed)
// forward, with every product on 4x4 register tiles over padded shared-memory rows
// (leading dimensions = width + 4 floats, so that row-wise float4 reads of different
// rows fall in different banks).  Products whose right operand is read transposed
// (Q K^T, Q U^T) use column-strided tiles for the same reason.
// MC: the longest chunk the layout holds.  The pair's state (S, X, C: d x d and two
// d x dv fp32 arrays) stays in shared memory, so wide states leave room for shorter
// chunks only: a longer chunk runs as several of MC tokens (the chunk length changes
// only the rounding).
template <int D, int DV, int MC>
struct TiledLayout {
    static constexpr int LD = D + 4, LV = DV + 4, LC = MC + 4;
    static constexpr int S = 0, X = S + D * LD, Cs = X + D * LV, m = Cs + D * LV, Y = m + D;
    static constexpr int Q = Y + D, K = Q + MC * LD, U = K + MC * LD, V = U + MC * LD;
    static constexpr int A = V + MC * LV, gp = A + MC * LC;
    static constexpr int w1 = gp + 2 * MC + 4, w2 = w1 + MC, rden = w2 + MC;
    static constexpr int floats = rden + MC;
    static_assert(D % 4 == 0 && DV % 4 == 0 && X % 4 == 0 && Q % 4 == 0 && V % 4 == 0 && A % 4 == 0, "alignment");
};
constexpr int kSmemFloats = 227 * 1024 / 4;
template <int D, int DV>
constexpr int tiled_max_chunk() {
    return TiledLayout<D, DV, 64>::floats <= kSmemFloats   ? 64
           : TiledLayout<D, DV, 32>::floats <= kSmemFloats ? 32
           : TiledLayout<D, DV, 16>::floats <= kSmemFloats ? 16
                                                           : 8;
}
static_assert(TiledLayout<128, 128, tiled_max_chunk<128, 128>()>::floats <= kSmemFloats, "d = dv = 128 layout");

template <class Body>
__device__ __forceinline__ void tiles_rt(int M, int N, bool strided, Body body) {
    const int tn = N / 4, count = (M / 4) * tn;
    for (int t = threadIdx.x; t < count; t += kThreads) {
        const int m0 = (t / tn) * 4;
        const int n0 = strided ? t % tn : (t % tn) * 4, ns = strided ? tn : 1;
        float acc[4][4] = {};
        body(acc, m0, n0, ns);
    }
}

template <typename T, int D, int DV, int MC>
__global__ void __launch_bounds__(kThreads) fwd_simt_tiled_kernel(FwdArgs a) {
    using Lt = TiledLayout<D, DV, MC>;
    constexpr int LD = Lt::LD, LV = Lt::LV, LC = Lt::LC;
    extern __shared__ __align__(16) float sm[];
    float *S = sm + Lt::S, *X = sm + Lt::X, *Cs = sm + Lt::Cs, *m = sm + Lt::m, *Y = sm + Lt::Y;
    float *Q = sm + Lt::Q, *K = sm + Lt::K, *U = sm + Lt::U, *V = sm + Lt::V, *A = sm + Lt::A;
    float *gp = sm + Lt::gp, *w1 = sm + Lt::w1, *w2 = sm + Lt::w2, *rden = sm + Lt::rden;
    using tile::mac;
    using tile::each;

    const int c = a.chunk, tid = threadIdx.x;
    const int u = blockIdx.x;  // pair index b*H + h
    const int hh = u % a.H;
    const bool decay = (a.flags & HLA_DECAY) != 0, norm = (a.flags & HLA_NORMALIZE) != 0;
    const float lg = log2f(decay ? a.gamma[hh] : 1.f);
    const size_t kvu = (size_t)(u / a.H) * a.Hkv + hh / (a.H / a.Hkv);
    const T *q = static_cast<const T *>(a.q) + (size_t)u * a.n * D;
    const T *k = static_cast<const T *>(a.k) + kvu * a.n * D;
    const T *v = static_cast<const T *>(a.v) + kvu * a.n * DV;
    T *o = static_cast<T *>(a.o) + (size_t)u * a.n * DV;
    for (int x = tid; x <= 2 * c + 1; x += kThreads) gp[x] = decay ? gpow(lg, (float)x) : 1.f;

    // ---- prefix state (X = S C - G, Y = S m - h)
    if (a.sin.S) {
        const float *Si = a.sin.S + (size_t)u * D * D, *Ci = a.sin.C + (size_t)u * D * DV;
        const float *mi = a.sin.m + (size_t)u * D, *Gi = a.sin.G + (size_t)u * D * DV, *hi = a.sin.h + (size_t)u * D;
        for (int e = tid; e < D * D; e += kThreads) S[(e / D) * LD + e % D] = Si[e];
        for (int e = tid; e < D * DV; e += kThreads) Cs[(e / DV) * LV + e % DV] = Ci[e];
        for (int e = tid; e < D; e += kThreads) m[e] = mi[e];
        __syncthreads();
        tiles_rt(D, DV, false, [&](float (&acc)[4][4], int m0, int n0, int ns) {
            mac<false, false>(acc, S, LD, Cs, LV, m0, n0, ns, D);
            each(acc, m0, n0, ns, [&](int i, int j, float x) { X[i * LV + j] = x - Gi[(size_t)i * DV + j]; });
        });
        for (int i = tid; i < D; i += kThreads) {
            float acc = 0.f;
            for (int l = 0; l < D; ++l) acc = fmaf(S[i * LD + l], m[l], acc);
            Y[i] = acc - hi[i];
        }
    } else {
        for (int e = tid; e < D * D; e += kThreads) S[(e / D) * LD + e % D] = 0.f;
        for (int e = tid; e < D * DV; e += kThreads) X[(e / DV) * LV + e % DV] = Cs[(e / DV) * LV + e % DV] = 0.f;
        for (int e = tid; e < D; e += kThreads) m[e] = Y[e] = 0.f;
    }
    __syncthreads();

    for (int t0 = 0; t0 < a.n; t0 += c) {
        const int L = min(c, a.n - t0);
        for (int e = tid; e < c * D; e += kThreads) {
            const int t = e / D, i = e % D;
            Q[t * LD + i] = t < L ? ld_in(q, (size_t)t0 * D + e) : 0.f;
            K[t * LD + i] = t < L ? ld_in(k, (size_t)t0 * D + e) : 0.f;
        }
        for (int e = tid; e < c * DV; e += kThreads) {
            const int t = e / DV;
            V[t * LV + e % DV] = t < L ? ld_in(v, (size_t)t0 * DV + e) : 0.f;
        }
        for (int b = tid; b < c; b += kThreads) {
            w1[b] = b < L ? gp[L - 1 - b] : 0.f;
            w2[b] = b < L ? gp[2 * (L - 1 - b)] : 0.f;
        }
        __syncthreads();
        // A[t,s] = g^{t-s} q_t.k_s, s <= t
        tiles_rt(c, c, true, [&](float (&acc)[4][4], int m0, int n0, int ns) {
            mac<false, true>(acc, Q, LD, K, LD, m0, n0, ns, D);
            each(acc, m0, n0, ns, [&](int t, int s2, float x) { A[t * LC + s2] = s2 <= t ? gp[t - s2] * x : 0.f; });
        });
        __syncthreads();
        // U[b] = g^{b+1} S_p q_b + sum_{s<=b} A[b,s] k_s   (S symmetric)
        tiles_rt(c, D, false, [&](float (&acc)[4][4], int m0, int n0, int ns) {
            mac<false, false>(acc, Q, LD, S, LD, m0, n0, ns, D);
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] *= gp[m0 + i + 1];
            mac<false, false>(acc, A, LC, K, LD, m0, n0, ns, c);
            each(acc, m0, n0, ns, [&](int b, int i, float x) { U[b * LD + i] = x; });
        });
        __syncthreads();
        // M[t,b] = g^{2(t-b)} q_t.u_b, b <= t (overwrites A)
        tiles_rt(c, c, true, [&](float (&acc)[4][4], int m0, int n0, int ns) {
            mac<false, true>(acc, Q, LD, U, LD, m0, n0, ns, D);
            each(acc, m0, n0, ns, [&](int t, int b, float x) { A[t * LC + b] = b <= t ? gp[2 * (t - b)] * x : 0.f; });
        });
        __syncthreads();
        if (norm) {  // den_t = sum_b M[t,b] + g^{2 tau} q_t.Y_p
            for (int t = tid; t < c; t += kThreads) {
                float sm_ = 0.f, qy = 0.f;
                for (int b = 0; b < c; ++b) sm_ += A[t * LC + b];
                for (int i = 0; i < D; ++i) qy = fmaf(Q[t * LD + i], Y[i], qy);
                rden[t] = 1.f / (sm_ + gp[2 * (t + 1)] * qy + a.eps);
            }
            __syncthreads();
        }
        // o_t = sum_b M[t,b] v_b + g^{2 tau} q_t^T X_p  (/ den_t)
        tiles_rt(c, DV, false, [&](float (&acc)[4][4], int m0, int n0, int ns) {
            float px[4][4] = {};
            mac<false, false>(acc, A, LC, V, LV, m0, n0, ns, c);
            mac<false, false>(px, Q, LD, X, LV, m0, n0, ns, D);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int t = m0 + i;
                if (t >= L) continue;
                const float r = norm ? rden[t] : 1.f, gt = gp[2 * (t + 1)];
#pragma unroll
                for (int j = 0; j < 4; ++j) st_out(o, (size_t)(t0 + t) * DV + n0 + j, (acc[i][j] + gt * px[i][j]) * r);
            }
        });
        __syncthreads();
        // state to the chunk end: weights w1 = g^{L-1-b} (S, C, m), w2 = w1^2 (X, Y)
        const float gL = gp[L], g2L = gp[2 * L];
        tiles_rt(D, D, false, [&](float (&acc)[4][4], int m0, int n0, int ns) {
            mac<true, false>(acc, K, LD, K, LD, m0, n0, ns, c, w1);
            each(acc, m0, n0, ns, [&](int i, int j, float x) { S[i * LD + j] = gL * S[i * LD + j] + x; });
        });
        tiles_rt(D, DV, false, [&](float (&acc)[4][4], int m0, int n0, int ns) {
            float ax[4][4] = {};
            mac<true, false>(acc, Q, LD, V, LV, m0, n0, ns, c, w1);
            mac<true, false>(ax, U, LD, V, LV, m0, n0, ns, c, w2);
            each(acc, m0, n0, ns, [&](int i, int j, float x) { Cs[i * LV + j] = gL * Cs[i * LV + j] + x; });
            each(ax, m0, n0, ns, [&](int i, int j, float x) { X[i * LV + j] = g2L * X[i * LV + j] + x; });
        });
        for (int i = tid; i < D; i += kThreads) {
            float am = 0.f, ay = 0.f;
            for (int b = 0; b < L; ++b) {
                am = fmaf(w1[b], Q[b * LD + i], am);
                ay = fmaf(w2[b], U[b * LD + i], ay);
            }
            m[i] = gL * m[i] + am;
            Y[i] = g2L * Y[i] + ay;
        }
        __syncthreads();
    }

    if (a.sout.S) {  // G = S C - X, h = S m - Y
        float *So = a.sout.S + (size_t)u * D * D, *Co = a.sout.C + (size_t)u * D * DV;
        float *mo = a.sout.m + (size_t)u * D, *Go = a.sout.G + (size_t)u * D * DV, *ho = a.sout.h + (size_t)u * D;
        for (int e = tid; e < D * D; e += kThreads) So[e] = S[(e / D) * LD + e % D];
        tiles_rt(D, DV, false, [&](float (&acc)[4][4], int m0, int n0, int ns) {
            mac<false, false>(acc, S, LD, Cs, LV, m0, n0, ns, D);
            each(acc, m0, n0, ns, [&](int i, int j, float x) {
                Co[(size_t)i * DV + j] = Cs[i * LV + j];
                Go[(size_t)i * DV + j] = x - X[i * LV + j];
            });
        });
        for (int i = tid; i < D; i += kThreads) {
            float acc = 0.f;
            for (int l = 0; l < D; ++l) acc = fmaf(S[i * LD + l], m[l], acc);
            mo[i] = m[i];
            ho[i] = acc - Y[i];
        }
    }
}

// The unmasked and asymmetric variants (d, dv <= 64; chunks of at most kMaxChunk tokens).
template <typename T, int D, int DV>
cudaError_t launch_general(const FwdArgs &a0, cudaStream_t st) {
    constexpr int DU = D > DV ? D : DV;
    FwdArgs a = a0;
    if (a.chunk > kMaxChunk) a.chunk = kMaxChunk;
    const size_t floats = (size_t)D * D + 2 * (size_t)D * DV + 2 * D + (size_t)kMaxChunk * (2 * D + DV + DU) +
                          (size_t)kMaxChunk * kMaxChunk + kMaxChunk + 2 * kMaxChunk + 2;
    const size_t bytes = floats * sizeof(float);
    auto kern = fwd_simt_kernel<T, D, DV>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    kern<<<a.B * a.H, kThreads, bytes, st>>>(a);
    return cudaGetLastError();
}

template <typename T, int D, int DV>
cudaError_t launch_t(const FwdArgs &a0, cudaStream_t st) {
    if (!(a0.flags & (HLA_UNMASKED | HLA_ASYMMETRIC))) {
        constexpr int MC = tiled_max_chunk<D, DV>();
        FwdArgs a = a0;
        if (a.chunk > MC) a.chunk = MC;
        const size_t bytes = (size_t)TiledLayout<D, DV, MC>::floats * sizeof(float);
        auto kern = fwd_simt_tiled_kernel<T, D, DV, MC>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
        if (e != cudaSuccess) return e;
        kern<<<a.B * a.H, kThreads, bytes, st>>>(a);
        return cudaGetLastError();
    }
    if constexpr (D > 64 || DV > 64) {  // the unmasked and asymmetric kernel holds d, dv <= 64
        return cudaErrorInvalidValue;
    } else {
        return launch_general<T, D, DV>(a0, st);
    }
}

template <typename T, int D>
cudaError_t launch_dv(const FwdArgs &a, cudaStream_t st) {
    switch (a.dv) {
        case 16: return launch_t<T, D, 16>(a, st);
        case 32: return launch_t<T, D, 32>(a, st);
        case 64: return launch_t<T, D, 64>(a, st);
        case 128: return launch_t<T, D, 128>(a, st);
    }
    return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t launch_d(const FwdArgs &a, cudaStream_t st) {
    switch (a.d) {
        case 16: return launch_dv<T, 16>(a, st);
        case 32: return launch_dv<T, 32>(a, st);
        case 64: return launch_dv<T, 64>(a, st);
        case 128: return launch_dv<T, 128>(a, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

bool fwd_simt_supported(const hla_params &p) {
    auto ok = [](int x) { return x == 16 || x == 32 || x == 64; };
    auto wide = [&](int x) { return ok(x) || x == 128; };
    // the masked variant at every width; the unmasked and asymmetric ones at d, dv <= 64
    const bool general = (p.flags & (HLA_UNMASKED | HLA_ASYMMETRIC)) != 0;
    return (general ? ok(p.d) && ok(p.dv) : wide(p.d) && wide(p.dv)) && wide(p.chunk);
}

cudaError_t fwd_simt_launch(const FwdArgs &a, cudaStream_t st) {
    if (a.n == 0 && !a.sout.S) return cudaSuccess;
    return a.in_dtype == HLA_F32 ? launch_d<float>(a, st) : launch_d<__nv_bfloat16>(a, st);
}

}  // namespace hla
