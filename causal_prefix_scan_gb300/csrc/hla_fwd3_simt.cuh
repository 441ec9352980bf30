// hla_fwd3_simt.cuh -- chunk-parallel forward of masked third-order HLA on CUDA
// cores (fp32 arithmetic), for d, dv, chunk in {16,32,64} and for d = 128 with
// 16-token chunks and dv in {16,32}.
//
// "Higher-order Linear Attention", gist.science summary, section 3 "Derde-orde HLA":
// the operator A A^T A (A = Q K^T) with every factor causal,
//   o_t = sum_{b<=t} sum_{a<=b} sum_{c<=b} (q_t.k_a)(k_a.q_b)(q_b.k_c) v_c
//       = q_t^T T_t,   T_t = sum_{b<=t} S^K_b q_b q_b^T P_b,
// with the prefix moments S^K_b = sum_{a<=b} k_a k_a^T and P_b = sum_{c<=b} k_c v_c^T.
// T equals S^K S^Q P minus the cross summaries of the pages (G1 + G2 - G3).
//
// Chunk form (prefix state S^K_p, P_p, T_p before the chunk):
//   A~ = tril(Q K^T),  U = Q S^K_p + A~ K  (rows u_b = S^K_b q_b),
//   W = Q P_p + A~ V  (rows w_b = P_b^T q_b),  M = tril(Q U^T),  O = Q T_p + M W.
// Segment summaries and their concatenation (section 4, bullet "Derde-orde scans":
// segment-level linear maps compose third-order states exactly), A before B:
//   T = T_A + T_B + S^K_A M^QP_B + M^KQ_B P_A + S^K_A S^Q_B P_A,  S^K, P add,
// with the chunk-local sums (from a zero prefix, U and W without their first terms)
//   S^K = K^T K,  S^Q = Q^T Q,  P = K^T V,  T = U^T W,  M^QP = Q^T W,  M^KQ = U^T Q.
//
// Exponential decay (per head, g; every prefix moment decays by g per token, so the
// triple a, b, c <= t weighs g^(3t-a-b-c)): with G[t][s] = g^(t-s) and tau the token's
// index in its chunk,
//   A~ = G o tril(Q K^T),  U = diag(g^(tau+1)) Q S^K_p + A~ K,  W = diag(g^(tau+1)) Q P_p + A~ V,
//   M = G^3 o tril(Q U^T),  O = diag(g^(3(tau+1))) Q T_p + M W;
// the local sums weight token b by g^(e-b) (S^K, S^Q, P), g^(3(e-b)) (T) and
// g^(2(e-b)) (M^QP, M^KQ), e the chunk's last token; a chunk of L tokens composes with
// f = g^L:  S^K = f S^K_A + S^K_B (P likewise),  X = M^QP_B + f S^Q_B P_A,
//   T = f^3 T_A + T_B + f M^KQ_B P_A + f S^K_A X.
//
// Key/value heads may be shared: query head h reads key/value head h / (H / Hkv); the
// state stays per query head.
//
// Three launches: (1) one CTA per chunk writes the local sums; (2) the scan, one CTA
// per (b,h) and column block of dv, walks the chunks and writes each chunk's prefix
// state (and the final state); (3) one CTA per chunk forms the outputs.  For bf16
// inputs with d = dv = chunk = 64, (1) and (3) run on the tensor cores
// (hla_fwd3_tc.cu) and (2) as elementwise prefix sums around one tensor-core product
// stage per chunk (hla_scan_tc.cu); the kernels here are the CUDA-core versions for
// every shape.
#pragma once
#include <type_traits>

#include "hla_smem_tile.cuh"

namespace hla {
namespace fwd3tc {
cudaError_t local_tc(const Fwd3Args &a, cudaStream_t st);
cudaError_t out_tc(const Fwd3Args &a, cudaStream_t st);
}  // namespace fwd3tc
namespace scantc {
// the scan as elementwise prefix sums around one tensor-core product stage per chunk
cudaError_t fwd3_scan(const Fwd3Args &a, cudaStream_t st);
}  // namespace scantc

namespace fwd3 {
using namespace tile;
constexpr int kSplit = 4;  // column blocks of dv per (b,h) in the scan

// Workspace: the local sums of every (b,h, chunk), then the prefix states.
struct Ws3 {
    int d, dv;
    // local sums: S^K d*d, S^Q d*d, M^KQ d*d, P d*dv, T d*dv, M^QP d*dv
    __host__ __device__ size_t loc_floats() const { return 3 * (size_t)d * d + 3 * (size_t)d * dv; }
    __host__ __device__ size_t o_sk() const { return 0; }
    __host__ __device__ size_t o_sq() const { return (size_t)d * d; }
    __host__ __device__ size_t o_mkq() const { return 2 * (size_t)d * d; }
    __host__ __device__ size_t o_p() const { return 3 * (size_t)d * d; }
    __host__ __device__ size_t o_t() const { return o_p() + (size_t)d * dv; }
    __host__ __device__ size_t o_mqp() const { return o_t() + (size_t)d * dv; }
    // prefix state: S^K d*d, P d*dv, T d*dv
    __host__ __device__ size_t st_floats() const { return (size_t)d * d + 2 * (size_t)d * dv; }
    __host__ __device__ size_t s_sk() const { return 0; }
    __host__ __device__ size_t s_p() const { return (size_t)d * d; }
    __host__ __device__ size_t s_t() const { return (size_t)d * d + (size_t)d * dv; }
};

// Key/value head read by query pair u = b*H + h: b*Hkv + h / (H / Hkv).
__device__ __forceinline__ size_t kv_unit(const Fwd3Args &a, int u) {
    return (size_t)(u / a.H) * a.Hkv + (u % a.H) / (a.H / a.Hkv);
}

// ---- (1) chunk-local sums --------------------------------------------------------
// Powers g^x, x = 0 .. 3C (gp[x]); all ones without decay.
constexpr int gp_count(int C) { return 3 * C + 4; }
__device__ __forceinline__ void fill_powers(float *gp, int count, const Fwd3Args &a, int u) {
    const bool decay = a.gamma != nullptr;
    const float lg = decay ? log2f(a.gamma[u % a.H]) : 0.f;
    for (int x = threadIdx.x; x < count; x += kThreads) gp[x] = decay ? gpow(lg, (float)x) : 1.f;
}

template <int C, int D, int DV>
struct LocSmem3 {
    static constexpr int LQ = D + 4, LV = DV + 4, LT = C + 4;
    static constexpr int Q = 0, K = Q + C * LQ, V = K + C * LQ, A = V + C * LV, U = A + C * LT, W = U + C * LQ,
                         GP = W + C * LV, W1 = GP + gp_count(C), W2 = W1 + C, W3 = W2 + C, TOTAL = W3 + C;
};

template <typename T, int C, int D, int DV>
__global__ void __launch_bounds__(kThreads) fwd3_local_kernel(Fwd3Args a) {
    using Sm = LocSmem3<C, D, DV>;
    extern __shared__ __align__(16) float sm[];
    float *Q = sm + Sm::Q, *K = sm + Sm::K, *V = sm + Sm::V, *A = sm + Sm::A, *U = sm + Sm::U, *W = sm + Sm::W;
    float *gp = sm + Sm::GP, *w1 = sm + Sm::W1, *w2 = sm + Sm::W2, *w3 = sm + Sm::W3;
    const int nch = (a.n + C - 1) / C, u = blockIdx.x / nch, ch = blockIdx.x % nch;
    const int t0 = ch * C, L = min(C, a.n - t0);
    const size_t rq = ((size_t)u * a.n + t0) * D, rv = ((size_t)u * a.n + t0) * DV;
    fill_powers(gp, gp_count(C), a, u);
    load_rows<D>(static_cast<const T *>(a.q) + rq, Q, Sm::LQ, C, L);
    const size_t kvu = kv_unit(a, u), rk = (kvu * a.n + t0) * D, rkv = (kvu * a.n + t0) * DV;
    load_rows<D>(static_cast<const T *>(a.k) + rk, K, Sm::LQ, C, L);
    load_rows<DV>(static_cast<const T *>(a.v) + rkv, V, Sm::LV, C, L);
    __syncthreads();
    // token weights of the local sums, relative to the chunk's last token e = L - 1
    for (int b = threadIdx.x; b < C; b += kThreads) {
        const int x = b < L ? L - 1 - b : 0;
        w1[b] = gp[x];
        w2[b] = gp[2 * x];
        w3[b] = gp[3 * x];
    }
    tiles<true, C, C>([&](float (&acc)[4][4], int m0, int n0, int ns) {
        mac<false, true>(acc, Q, Sm::LQ, K, Sm::LQ, m0, n0, ns, D);
        each(acc, m0, n0, ns, [&](int t, int s, float x) { A[t * Sm::LT + s] = s <= t ? gp[t - s] * x : 0.f; });
    });
    __syncthreads();
    // U = A~ K, W = A~ V (no earlier state)
    tiles<false, C, D>([&](float (&acc)[4][4], int m0, int n0, int ns) {
        mac<false, false>(acc, A, Sm::LT, K, Sm::LQ, m0, n0, ns, C);
        each(acc, m0, n0, ns, [&](int t, int i, float x) { U[t * Sm::LQ + i] = x; });
    });
    tiles<false, C, DV>([&](float (&acc)[4][4], int m0, int n0, int ns) {
        mac<false, false>(acc, A, Sm::LT, V, Sm::LV, m0, n0, ns, C);
        each(acc, m0, n0, ns, [&](int t, int j, float x) { W[t * Sm::LV + j] = x; });
    });
    __syncthreads();
    const Ws3 ws{D, DV};
    float *out = a.workspace + ((size_t)u * nch + ch) * ws.loc_floats();
    auto put = [&](size_t off, int ld) {
        return [=](int i, int j, float x) { out[off + (size_t)i * ld + j] = x; };
    };
    // rows past the chunk's last token are zero in Q, K, V, U, W
    tiles<false, D, D>([&](float (&acc)[4][4], int m0, int n0, int ns) {
        mac<true, false>(acc, K, Sm::LQ, K, Sm::LQ, m0, n0, ns, C, w1);
        each(acc, m0, n0, ns, put(ws.o_sk(), D));
    });
    tiles<false, D, D>([&](float (&acc)[4][4], int m0, int n0, int ns) {
        mac<true, false>(acc, Q, Sm::LQ, Q, Sm::LQ, m0, n0, ns, C, w1);
        each(acc, m0, n0, ns, put(ws.o_sq(), D));
    });
    tiles<false, D, D>([&](float (&acc)[4][4], int m0, int n0, int ns) {
        mac<true, false>(acc, U, Sm::LQ, Q, Sm::LQ, m0, n0, ns, C, w2);
        each(acc, m0, n0, ns, put(ws.o_mkq(), D));
    });
    tiles<false, D, DV>([&](float (&acc)[4][4], int m0, int n0, int ns) {
        mac<true, false>(acc, K, Sm::LQ, V, Sm::LV, m0, n0, ns, C, w1);
        each(acc, m0, n0, ns, put(ws.o_p(), DV));
    });
    tiles<false, D, DV>([&](float (&acc)[4][4], int m0, int n0, int ns) {
        mac<true, false>(acc, U, Sm::LQ, W, Sm::LV, m0, n0, ns, C, w3);
        each(acc, m0, n0, ns, put(ws.o_t(), DV));
    });
    tiles<false, D, DV>([&](float (&acc)[4][4], int m0, int n0, int ns) {
        mac<true, false>(acc, Q, Sm::LQ, W, Sm::LV, m0, n0, ns, C, w2);
        each(acc, m0, n0, ns, put(ws.o_mqp(), DV));
    });
}

// ---- (2) scan over chunks ---------------------------------------------------------
// blockIdx.x = u * kSplit + part.  The CTA keeps S^K whole and the columns
// [part*dv/kSplit, ...) of P and T; it stores the row block `part` of S^K and its
// column blocks of P, T as each chunk's prefix state, and the same of the final state.
// The next chunk's local sums are copied into the other of two shared buffers
// (cp.async) while the current chunk is applied.
template <int C, int D, int DV>
struct ScanSmem3 {
    static constexpr int NB = DV / kSplit, LF = D + 4, LB = NB + 4;
    static constexpr int SK = 0, PB = SK + D * LF, TB = PB + D * LB, X = TB + D * LB, Y = X + D * LB,
                         RED = Y + D * LB, RSZ = kThreads * 16, BUF = RED + 2 * RSZ;
    // one buffer: S^K_B, S^Q_B, M^KQ_B (D x LF each), then the column blocks of P_B, T_B,
    // M^QP_B.  At d = 128 two buffers of three d x d sums do not fit beside the running
    // S^K: the d x d sums are then read from the workspace where they are used.
    static constexpr bool STAGE_DD = D <= 64;
    static constexpr int DD = STAGE_DD ? D * LF : 0;
    static constexpr int B_SK = 0, B_SQ = DD, B_MKQ = 2 * DD, B_P = 3 * DD, B_T = B_P + D * LB,
                         B_MQP = B_T + D * LB, BUFSZ = B_MQP + D * LB;
    static constexpr int TOTAL = BUF + 2 * BUFSZ;
};

template <int C, int D, int DV>
__global__ void __launch_bounds__(kThreads) fwd3_scan_kernel(Fwd3Args a) {
    using Sm = ScanSmem3<C, D, DV>;
    constexpr int NB = Sm::NB, LF = Sm::LF, LB = Sm::LB;
    extern __shared__ __align__(16) float sm[];
    float *SK = sm + Sm::SK, *Pb = sm + Sm::PB, *Tb = sm + Sm::TB, *X = sm + Sm::X, *Y = sm + Sm::Y;
    float *red1 = sm + Sm::RED, *red2 = red1 + Sm::RSZ;
    const int part = blockIdx.x % kSplit, u = blockIdx.x / kSplit;
    const int nch = (a.n + C - 1) / C, c0 = part * NB;
    constexpr int ROWS = D / kSplit;
    const int r0 = part * ROWS;
    const Ws3 ws{D, DV};
    const bool decay = a.gamma != nullptr;
    const float lg = decay ? log2f(a.gamma[u % a.H]) : 0.f;
    const float *loc = a.workspace + (size_t)u * nch * ws.loc_floats();
    float *st = a.workspace + (size_t)a.B * a.H * nch * ws.loc_floats() + (size_t)u * nch * ws.st_floats();
    auto issue = [&](int ch) {  // the local sums of chunk ch into buffer ch & 1
        const float *lc = loc + (size_t)ch * ws.loc_floats();
        float *b = sm + Sm::BUF + (ch & 1) * Sm::BUFSZ;
        if constexpr (Sm::STAGE_DD) {
            copy_mat_async<D>(lc + ws.o_sk(), D, b + Sm::B_SK, LF, D);
            copy_mat_async<D>(lc + ws.o_sq(), D, b + Sm::B_SQ, LF, D);
            copy_mat_async<D>(lc + ws.o_mkq(), D, b + Sm::B_MKQ, LF, D);
        }
        copy_mat_async<NB>(lc + ws.o_p() + c0, DV, b + Sm::B_P, LB, D);
        copy_mat_async<NB>(lc + ws.o_t() + c0, DV, b + Sm::B_T, LB, D);
        copy_mat_async<NB>(lc + ws.o_mqp() + c0, DV, b + Sm::B_MQP, LB, D);
    };
    if (nch > 0) issue(0);
    cp_async_commit();
    // initial state: state_in or zeros
    for (int e = threadIdx.x; e < D * D; e += kThreads)
        SK[(e / D) * LF + e % D] = a.sin_S ? a.sin_S[(size_t)u * D * D + e] : 0.f;
    for (int e = threadIdx.x; e < D * NB; e += kThreads) {
        const int r = e / NB, x = e % NB;
        const size_t g = (size_t)u * D * DV + (size_t)r * DV + c0 + x;
        Pb[r * LB + x] = a.sin_P ? a.sin_P[g] : 0.f;
        Tb[r * LB + x] = a.sin_T ? a.sin_T[g] : 0.f;
    }
    __syncthreads();
    for (int ch = 0; ch < nch; ++ch) {
        if (ch + 1 < nch) issue(ch + 1);
        cp_async_commit();
        // this chunk's prefix state
        float *so = st + (size_t)ch * ws.st_floats();
        for (int e = threadIdx.x; e < ROWS * D; e += kThreads) {
            const int r = r0 + e / D, x = e % D;
            so[ws.s_sk() + (size_t)r * D + x] = SK[r * LF + x];
        }
        for (int e = threadIdx.x; e < D * NB; e += kThreads) {
            const int r = e / NB, x = e % NB;
            so[ws.s_p() + (size_t)r * DV + c0 + x] = Pb[r * LB + x];
            so[ws.s_t() + (size_t)r * DV + c0 + x] = Tb[r * LB + x];
        }
        cp_async_wait<1>();  // chunk ch's copies (the group before the one just committed)
        __syncthreads();
        const float *b = sm + Sm::BUF + (ch & 1) * Sm::BUFSZ;
        const float *lc = loc + (size_t)ch * ws.loc_floats();
        // the d x d sums: staged (row stride LF) or in the workspace (row stride D)
        constexpr int LDD = Sm::STAGE_DD ? LF : D;
        const float *SKl = Sm::STAGE_DD ? b + Sm::B_SK : lc + ws.o_sk();
        const float *SQl = Sm::STAGE_DD ? b + Sm::B_SQ : lc + ws.o_sq();
        const float *MKQl = Sm::STAGE_DD ? b + Sm::B_MKQ : lc + ws.o_mkq();
        const float *Pl = b + Sm::B_P, *Tl = b + Sm::B_T, *MQPl = b + Sm::B_MQP;
        const int L = min(C, a.n - ch * C);
        const float f = decay ? gpow(lg, (float)L) : 1.f, f3 = f * f * f;
        // S^Q_B P_A and M^KQ_B P_A (block columns), each over all threads
        mac_ksplit<D, NB, D>(SQl, LDD, Pb, LB, red1);
        mac_ksplit<D, NB, D>(MKQl, LDD, Pb, LB, red2);
        __syncthreads();
        // X = M^QP_B + f S^Q_B P_A,  Y = M^KQ_B P_A
        for (int e = threadIdx.x; e < D * NB; e += kThreads) {
            const int o = (e / NB) * LB + e % NB;
            X[o] = MQPl[o] + f * ksplit_sum<D, NB, D>(red1, e);
            Y[o] = ksplit_sum<D, NB, D>(red2, e);
        }
        __syncthreads();
        // T <- f^3 T + T_B + f Y + f S^K_A X
        mac_ksplit<D, NB, D>(SK, LF, X, LB, red1);
        __syncthreads();
        for (int e = threadIdx.x; e < D * NB; e += kThreads) {
            const int o = (e / NB) * LB + e % NB;
            Tb[o] = f3 * Tb[o] + Tl[o] + f * (Y[o] + ksplit_sum<D, NB, D>(red1, e));
            Pb[o] = f * Pb[o] + Pl[o];  // P <- f P + P_B (read above only, before this barrier)
        }
        // S^K <- f S^K + S^K_B
        for (int e = threadIdx.x; e < D * D; e += kThreads) {
            const int r = e / D, x = e % D;
            SK[r * LF + x] = f * SK[r * LF + x] + SKl[r * LDD + x];
        }
        __syncthreads();
    }
    cp_async_wait<0>();
    // final state
    if (a.sout_S) {
        for (int e = threadIdx.x; e < ROWS * D; e += kThreads) {
            const int r = r0 + e / D, x = e % D;
            a.sout_S[(size_t)u * D * D + (size_t)r * D + x] = SK[r * LF + x];
        }
        for (int e = threadIdx.x; e < D * NB; e += kThreads) {
            const int r = e / NB, x = e % NB;
            const size_t g = (size_t)u * D * DV + (size_t)r * DV + c0 + x;
            a.sout_P[g] = Pb[r * LB + x];
            a.sout_T[g] = Tb[r * LB + x];
        }
    }
}

// ---- (3) outputs of one chunk -----------------------------------------------------
template <int C, int D, int DV>
struct OutSmem3 {
    static constexpr int LQ = D + 4, LV = DV + 4, LT = C + 4;
    static constexpr int Q = 0, K = Q + C * LQ, V = K + C * LQ, SK = V + C * LV, P = SK + D * LQ, TP = P + D * LV,
                         A = TP + D * LV, M = A + C * LT, U = M + C * LT, W = U + C * LQ, GP = W + C * LV,
                         R1 = GP + gp_count(C), R3 = R1 + C, TOTAL = R3 + C;
};

template <typename T, int C, int D, int DV>
__global__ void __launch_bounds__(kThreads) fwd3_out_kernel(Fwd3Args a) {
    using Sm = OutSmem3<C, D, DV>;
    extern __shared__ __align__(16) float sm[];
    float *Q = sm + Sm::Q, *K = sm + Sm::K, *V = sm + Sm::V, *SK = sm + Sm::SK, *P = sm + Sm::P, *Tp = sm + Sm::TP;
    float *A = sm + Sm::A, *M = sm + Sm::M, *U = sm + Sm::U, *W = sm + Sm::W;
    float *gp = sm + Sm::GP, *r1 = sm + Sm::R1, *r3 = sm + Sm::R3;
    const int nch = (a.n + C - 1) / C, u = blockIdx.x / nch, ch = blockIdx.x % nch;
    const int t0 = ch * C, L = min(C, a.n - t0);
    const size_t rq = ((size_t)u * a.n + t0) * D, rv = ((size_t)u * a.n + t0) * DV;
    const Ws3 ws{D, DV};
    fill_powers(gp, gp_count(C), a, u);
    const float *so =
        a.workspace + (size_t)a.B * a.H * nch * ws.loc_floats() + ((size_t)u * nch + ch) * ws.st_floats();
    // the prefix state arrives asynchronously while A~ is formed
    copy_mat_async<D>(so + ws.s_sk(), D, SK, Sm::LQ, D);
    copy_mat_async<DV>(so + ws.s_p(), DV, P, Sm::LV, D);
    copy_mat_async<DV>(so + ws.s_t(), DV, Tp, Sm::LV, D);
    cp_async_commit();
    load_rows<D>(static_cast<const T *>(a.q) + rq, Q, Sm::LQ, C, L);
    const size_t kvu = kv_unit(a, u), rk = (kvu * a.n + t0) * D, rkv = (kvu * a.n + t0) * DV;
    load_rows<D>(static_cast<const T *>(a.k) + rk, K, Sm::LQ, C, L);
    load_rows<DV>(static_cast<const T *>(a.v) + rkv, V, Sm::LV, C, L);
    __syncthreads();
    for (int t = threadIdx.x; t < C; t += kThreads) {  // row scales of the prefix-state terms
        r1[t] = gp[t + 1];
        r3[t] = gp[3 * (t + 1)];
    }
    tiles<true, C, C>([&](float (&acc)[4][4], int m0, int n0, int ns) {
        mac<false, true>(acc, Q, Sm::LQ, K, Sm::LQ, m0, n0, ns, D);
        each(acc, m0, n0, ns, [&](int t, int s, float x) { A[t * Sm::LT + s] = s <= t ? gp[t - s] * x : 0.f; });
    });
    cp_async_wait<0>();
    __syncthreads();
    // U = diag(g^(tau+1)) Q S^K_p + A~ K;  W = diag(g^(tau+1)) Q P_p + A~ V
    tiles<false, C, D>([&](float (&acc)[4][4], int m0, int n0, int ns) {
        mac_rs<false, false>(acc, r1, Q, Sm::LQ, SK, Sm::LQ, m0, n0, ns, D);
        mac<false, false>(acc, A, Sm::LT, K, Sm::LQ, m0, n0, ns, C);
        each(acc, m0, n0, ns, [&](int t, int i, float x) { U[t * Sm::LQ + i] = x; });
    });
    tiles<false, C, DV>([&](float (&acc)[4][4], int m0, int n0, int ns) {
        mac_rs<false, false>(acc, r1, Q, Sm::LQ, P, Sm::LV, m0, n0, ns, D);
        mac<false, false>(acc, A, Sm::LT, V, Sm::LV, m0, n0, ns, C);
        each(acc, m0, n0, ns, [&](int t, int j, float x) { W[t * Sm::LV + j] = x; });
    });
    __syncthreads();
    // M = G^3 o tril(Q U^T)
    tiles<true, C, C>([&](float (&acc)[4][4], int m0, int n0, int ns) {
        mac<false, true>(acc, Q, Sm::LQ, U, Sm::LQ, m0, n0, ns, D);
        each(acc, m0, n0, ns, [&](int t, int b, float x) { M[t * Sm::LT + b] = b <= t ? gp[3 * (t - b)] * x : 0.f; });
    });
    __syncthreads();
    // O = diag(g^(3(tau+1))) Q T_p + M W
    T *o = static_cast<T *>(a.o) + rv;
    tiles<false, C, DV>([&](float (&acc)[4][4], int m0, int n0, int ns) {
        mac_rs<false, false>(acc, r3, Q, Sm::LQ, Tp, Sm::LV, m0, n0, ns, D);
        mac<false, false>(acc, M, Sm::LT, W, Sm::LV, m0, n0, ns, C);
        each(acc, m0, n0, ns, [&](int t, int j, float x) {
            if (t < L) st_t(o, (size_t)t * DV + j, x);
        });
    });
}

template <typename Kern>
cudaError_t smem_attr(Kern kern, size_t bytes) {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <typename T, int C, int D, int DV>
cudaError_t launch_t(const Fwd3Args &a, cudaStream_t st) {
    const int nch = (a.n + C - 1) / C, units = a.B * a.H;
    const size_t b1 = LocSmem3<C, D, DV>::TOTAL * sizeof(float), b2 = ScanSmem3<C, D, DV>::TOTAL * sizeof(float),
                 b3 = OutSmem3<C, D, DV>::TOTAL * sizeof(float);
    cudaError_t e;
    // the tensor-core kernels: bf16 at 64/64/64 without decay
    constexpr bool TC_SHAPE = std::is_same<T, __nv_bfloat16>::value && C == 64 && D == 64 && DV == 64;
    const bool tc = TC_SHAPE && a.gamma == nullptr;
    if (!tc) {  // the CUDA-core kernels (the tensor-core ones set their own attributes)
        if ((e = smem_attr(fwd3_local_kernel<T, C, D, DV>, b1)) != cudaSuccess) return e;
        if ((e = smem_attr(fwd3_scan_kernel<C, D, DV>, b2)) != cudaSuccess) return e;
        if ((e = smem_attr(fwd3_out_kernel<T, C, D, DV>, b3)) != cudaSuccess) return e;
    }
    auto mark = [&](int i) { return a.events ? cudaEventRecord(a.events[i], st) : cudaSuccess; };
    if ((e = mark(0)) != cudaSuccess) return e;
    if (tc) {
        if ((e = fwd3tc::local_tc(a, st)) != cudaSuccess) return e;
    } else {
        fwd3_local_kernel<T, C, D, DV><<<units * nch, kThreads, b1, st>>>(a);
    }
    if ((e = mark(1)) != cudaSuccess) return e;
    if (tc) {
        if ((e = scantc::fwd3_scan(a, st)) != cudaSuccess) return e;
    } else {
        fwd3_scan_kernel<C, D, DV><<<units * kSplit, kThreads, b2, st>>>(a);
    }
    if ((e = mark(2)) != cudaSuccess) return e;
    if (tc) {
        if ((e = fwd3tc::out_tc(a, st)) != cudaSuccess) return e;
    } else {
        fwd3_out_kernel<T, C, D, DV><<<units * nch, kThreads, b3, st>>>(a);
    }
    if (a.sout_SQ && (e = fwd3_maps_launch(a, st)) != cudaSuccess) return e;
    if ((e = mark(3)) != cudaSuccess) return e;
    return cudaGetLastError();
}
template <typename T, int C, int D>
cudaError_t launch_dv(const Fwd3Args &a, cudaStream_t st) {
    switch (a.dv) {
        case 16: return launch_t<T, C, D, 16>(a, st);
        case 32: return launch_t<T, C, D, 32>(a, st);
        case 64: return launch_t<T, C, D, 64>(a, st);
    }
    return cudaErrorInvalidValue;
}
template <typename T, int C>
cudaError_t launch_d(const Fwd3Args &a, cudaStream_t st) {
    switch (a.d) {
        case 16: return launch_dv<T, C, 16>(a, st);
        case 32: return launch_dv<T, C, 32>(a, st);
        case 64: return launch_dv<T, C, 64>(a, st);
        case 128:
            // d = 128: the output kernel's S^K_p (128 x 128 fp32), P_p, T_p and chunk tiles
            // fit 227 KB of shared memory at 16-token chunks and dv <= 32
            if constexpr (C == 16) {
                if (a.dv == 16) return launch_t<T, C, 128, 16>(a, st);
                if (a.dv == 32) return launch_t<T, C, 128, 32>(a, st);
            }
            break;
    }
    return cudaErrorInvalidValue;
}
// One translation unit per (element type, chunk) instantiates launch_d.
}  // namespace fwd3
}  // namespace hla
