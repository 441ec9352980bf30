// hla_bwd_simt.cuh -- chunk-parallel backward pass of the masked second-order HLA
// forward on CUDA cores (fp32 arithmetic), for d, dv, chunk in {16,32,64} and for d = 128
// with 16-token chunks and dv in {16,32}, from a zero
// or a given initial state (S_in, X_in = S_in C_in - G_in; the gradient of that state
// comes from the adjoints at the first token: dX_in = g^2 Lam, dS_in = g Om +
// dX_in C_in^T, dC_in = S_in^T dX_in, dG_in = -dX_in).  The kernels compute the unnormalised gradient; the ratio-normalised
// one is composed from two such passes (hla_bwd_norm.cu).  Query heads may share key/
// value heads: dk, dv are staged per query head and summed over each group.
//
// The pages motivate chunk-parallel training ("Higher-order Linear Attention",
// gist.science summary, section 4) but print no gradient.  Forward in the working
// form of the forward kernels (section 1, with X = S C - G):
//   S_t = g S_{t-1} + k_t k_t^T,  u_t = S_t q_t,  X_t = g^2 X_{t-1} + u_t v_t^T,
//   o_t = X_t^T q_t.
// Reverse mode with the upstream gradient g_t = dL/do_t and the accumulators
//   Lam_t = dL/dX_t = q_t g_t^T + g^2 Lam_{t+1},  Om_t = dL/dS_t = du_t q_t^T + g Om_{t+1}
// gives  du_t = Lam_t v_t,  dv_t = Lam_t^T u_t,  dq_t = X_t g_t + S_t du_t,
// dk_t = (Om_t + Om_t^T) k_t.
//
// Chunk form (tau = 0..L-1 inside a chunk; S_p, X_p the states before it; Lam, Om
// the accumulators of everything after it):
//   A~[t,s] = g^{t-s} q_t.k_s,  P[s,b] = g^{2(s-b)} g_s.v_b  (lower triangles)
//   U  = diag(g^{tau+1}) Q S_p + A~ K
//   dU = P^T Q + diag(g^{2(L-tau)}) V Lam^T
//   B[t,a] = g^{t-a} du_t.k_a,  M[s,t] = g^{2(s-t)} q_s.u_t  (lower triangles)
//   dQ = P U + diag(g^{2(tau+1)}) G X_p^T + diag(g^{tau+1}) dU S_p + B K
//   dK = A~^T dU + B^T Q + diag(g^{L-tau}) K (Om + Om^T)
//   dV = M^T G + diag(g^{2(L-tau)}) U Lam
// and the chunk-to-chunk maps
//   S <- g^L S + Sloc,           X <- g^{2L} X + S_p Cq + Xloc,
//   Lam <- g^{2L} Lam + Lloc,    Om <- g^L Om + Oloc + Lam_next W,
// with the chunk-local sums (weights zero past the chunk's last token)
//   Sloc = sum_s g^{L-1-s} k_s k_s^T,  Cq = sum_s g^{2L-1-s} q_s v_s^T,
//   Xloc = sum_s g^{2(L-1-s)} (A~K)_s v_s^T,  Lloc = sum_s g^{2s} q_s g_s^T,
//   W = sum_s g^{2L-s} v_s q_s^T,  Oloc = sum_s g^s (P^T Q)_s q_s^T.
//
// Three launches: (1) one CTA per chunk writes the six local sums; (2) the scan,
// one CTA per (b,h, column block, direction), walks the chunks forward for S, X
// and backward for Lam, Om and writes the states every chunk needs; (3) one CTA
// per chunk forms dq, dk, dv.  For bf16 inputs with d = dv = chunk = 64, (1) and (3)
// run on the tensor cores (hla_bwd_tc.cu) and the scan as elementwise prefix sums
// around one tensor-core product stage per chunk (hla_scan_tc.cu); the kernels here
// are the CUDA-core versions for every shape.
#pragma once
#include <type_traits>

#include "hla_smem_tile.cuh"

namespace hla {
namespace bwdtc {
// tensor-core versions of the local-sums and gradient kernels (bf16, d = dv = chunk = 64)
cudaError_t local_tc(const BwdArgs &a, cudaStream_t st);
cudaError_t grad_tc(const BwdArgs &a, cudaStream_t st);
}  // namespace bwdtc
namespace scantc {
// the scan as elementwise prefix sums around one tensor-core product stage per chunk
cudaError_t bwd_scan(const BwdArgs &a, cudaStream_t st);
}  // namespace scantc
namespace bwd {

using namespace tile;
constexpr int kSplit = 4;  // column blocks per (b,h) and direction in the scan

// Key/value head read by query pair u = b*H + h: b*Hkv + h / (H / Hkv).
__device__ __forceinline__ size_t kv_unit(const BwdArgs &a, int u) {
    return (size_t)(u / a.H) * a.Hkv + (u % a.H) / (a.H / a.Hkv);
}

// Shared key/value heads: dk, dv of a key/value head = the sum of the per-query-head
// fp32 gradients of its group (in head order), converted to the output type.
template <typename T>
__global__ void __launch_bounds__(kThreads) bwd_group_sum_kernel(const float *pair, T *out, int B, int H, int Hkv,
                                                                  size_t per_head) {
    const size_t total = (size_t)B * Hkv * per_head;
    const int grp = H / Hkv;
    for (size_t e = (size_t)blockIdx.x * kThreads + threadIdx.x; e < total; e += (size_t)gridDim.x * kThreads) {
        const size_t j = e / per_head, x = e % per_head;  // key/value unit b*Hkv + h', element
        const size_t b = j / Hkv, hk = j % Hkv;
        const float *src = pair + ((b * H + hk * grp) * per_head + x);
        float s = 0.f;
        for (int g = 0; g < grp; ++g) s += src[(size_t)g * per_head];
        st_t(out, e, s);
    }
}

// Workspace: the six local sums of every (b,h, chunk), then the four states of
// every (b,h, chunk).
struct BwdWs {
    int d, dv;
    __host__ __device__ size_t loc_floats() const { return 2 * (size_t)d * d + 4 * (size_t)d * dv; }
    __host__ __device__ size_t st_floats() const { return 2 * (size_t)d * d + 2 * (size_t)d * dv; }
    // local sums: Sloc d*d, Cq d*dv, Xloc d*dv, Lloc d*dv, W dv*d, Oloc d*d
    __host__ __device__ size_t o_sloc() const { return 0; }
    __host__ __device__ size_t o_cq() const { return (size_t)d * d; }
    __host__ __device__ size_t o_xloc() const { return o_cq() + (size_t)d * dv; }
    __host__ __device__ size_t o_lloc() const { return o_xloc() + (size_t)d * dv; }
    __host__ __device__ size_t o_w() const { return o_lloc() + (size_t)d * dv; }
    __host__ __device__ size_t o_oloc() const { return o_w() + (size_t)d * dv; }
    // states: S_p d*d, X_p d*dv, Lam_next d*dv, Om_next d*d
    __host__ __device__ size_t o_sp() const { return 0; }
    __host__ __device__ size_t o_xp() const { return (size_t)d * d; }
    __host__ __device__ size_t o_lam() const { return o_xp() + (size_t)d * dv; }
    __host__ __device__ size_t o_om() const { return o_lam() + (size_t)d * dv; }
};

__device__ __forceinline__ void fill_gp(float *gp, int c, float lg, bool decay) {
    for (int x = threadIdx.x; x <= 2 * c; x += kThreads) gp[x] = decay ? gpow(lg, (float)x) : 1.f;
}

// ---- (1) chunk-local sums --------------------------------------------------------
template <int C, int D, int DV>
struct LocSmem {
    static constexpr int LQ = D + 4, LV = DV + 4, LT = C + 4;
    static constexpr int Q = 0, K = Q + C * LQ, V = K + C * LQ, G = V + C * LV, A = G + C * LV, P = A + C * LT,
                         U = P + C * LT, DU = U + C * LQ, GP = DU + C * LQ, WS = GP + 2 * C + 4,
                         TOTAL = WS + 6 * C;
};

template <typename T, int C, int D, int DV>
__global__ void __launch_bounds__(kThreads) bwd_local_kernel(BwdArgs a) {
    using Sm = LocSmem<C, D, DV>;
    extern __shared__ __align__(16) float sm[];
    float *Q = sm + Sm::Q, *K = sm + Sm::K, *V = sm + Sm::V, *G = sm + Sm::G, *A = sm + Sm::A, *P = sm + Sm::P;
    float *U = sm + Sm::U, *dU = sm + Sm::DU, *gp = sm + Sm::GP, *w = sm + Sm::WS;
    const int nch = (a.n + C - 1) / C, u = blockIdx.x / nch, ch = blockIdx.x % nch;
    const int t0 = ch * C, L = min(C, a.n - t0);
    const bool decay = (a.flags & HLA_DECAY) != 0;
    const float lg = log2f(decay ? a.gamma[u % a.H] : 1.f);
    const size_t rq = ((size_t)u * a.n + t0) * D, rv = ((size_t)u * a.n + t0) * DV;
    const size_t kvu = kv_unit(a, u), rk = (kvu * a.n + t0) * D, rkv = (kvu * a.n + t0) * DV;
    load_rows<D>(static_cast<const T *>(a.q) + rq, Q, Sm::LQ, C, L);
    load_rows<D>(static_cast<const T *>(a.k) + rk, K, Sm::LQ, C, L);
    load_rows<DV>(static_cast<const T *>(a.v) + rkv, V, Sm::LV, C, L);
    load_rows<DV>(static_cast<const T *>(a.go) + rv, G, Sm::LV, C, L);
    fill_gp(gp, C, lg, decay);
    __syncthreads();
    for (int s = threadIdx.x; s < C; s += kThreads) {
        const bool in = s < L;
        w[0 * C + s] = in ? gp[L - 1 - s] : 0.f;        // Sloc
        w[1 * C + s] = in ? gp[2 * L - 1 - s] : 0.f;    // Cq
        w[2 * C + s] = in ? gp[2 * (L - 1 - s)] : 0.f;  // Xloc
        w[3 * C + s] = in ? gp[2 * s] : 0.f;            // Lloc
        w[4 * C + s] = in ? gp[2 * L - s] : 0.f;        // W
        w[5 * C + s] = in ? gp[s] : 0.f;                // Oloc
    }
    // A~ = tril(g^{t-s} Q K^T), P = tril(g^{2(s-b)} G V^T)
    tiles<true, C, C>([&](float (&acc)[4][4], int m0, int n0, int ns) {
        mac<false, true>(acc, Q, Sm::LQ, K, Sm::LQ, m0, n0, ns, D);
        each(acc, m0, n0, ns, [&](int t, int s, float x) { A[t * Sm::LT + s] = s <= t ? gp[t - s] * x : 0.f; });
    });
    tiles<true, C, C>([&](float (&acc)[4][4], int m0, int n0, int ns) {
        mac<false, true>(acc, G, Sm::LV, V, Sm::LV, m0, n0, ns, DV);
        each(acc, m0, n0, ns, [&](int s, int b, float x) { P[s * Sm::LT + b] = b <= s ? gp[2 * (s - b)] * x : 0.f; });
    });
    __syncthreads();
    // U = A~ K (the part of u without the earlier state), dU = P^T Q
    tiles<false, C, D>([&](float (&acc)[4][4], int m0, int n0, int ns) {
        mac<false, false>(acc, A, Sm::LT, K, Sm::LQ, m0, n0, ns, C);
        each(acc, m0, n0, ns, [&](int t, int i, float x) { U[t * Sm::LQ + i] = x; });
    });
    tiles<false, C, D>([&](float (&acc)[4][4], int m0, int n0, int ns) {
        mac<true, false>(acc, P, Sm::LT, Q, Sm::LQ, m0, n0, ns, C);
        each(acc, m0, n0, ns, [&](int t, int i, float x) { dU[t * Sm::LQ + i] = x; });
    });
    __syncthreads();
    const BwdWs ws{D, DV};
    float *out = a.workspace + ((size_t)u * nch + ch) * ws.loc_floats();
    auto put = [&](size_t off, int ld) {
        return [=](int i, int j, float x) { out[off + (size_t)i * ld + j] = x; };
    };
    tiles<false, D, D>([&](float (&acc)[4][4], int m0, int n0, int ns) {
        mac<true, false>(acc, K, Sm::LQ, K, Sm::LQ, m0, n0, ns, C, w + 0 * C);
        each(acc, m0, n0, ns, put(ws.o_sloc(), D));
    });
    tiles<false, D, DV>([&](float (&acc)[4][4], int m0, int n0, int ns) {
        mac<true, false>(acc, Q, Sm::LQ, V, Sm::LV, m0, n0, ns, C, w + 1 * C);
        each(acc, m0, n0, ns, put(ws.o_cq(), DV));
    });
    tiles<false, D, DV>([&](float (&acc)[4][4], int m0, int n0, int ns) {
        mac<true, false>(acc, U, Sm::LQ, V, Sm::LV, m0, n0, ns, C, w + 2 * C);
        each(acc, m0, n0, ns, put(ws.o_xloc(), DV));
    });
    tiles<false, D, DV>([&](float (&acc)[4][4], int m0, int n0, int ns) {
        mac<true, false>(acc, Q, Sm::LQ, G, Sm::LV, m0, n0, ns, C, w + 3 * C);
        each(acc, m0, n0, ns, put(ws.o_lloc(), DV));
    });
    tiles<false, DV, D>([&](float (&acc)[4][4], int m0, int n0, int ns) {
        mac<true, false>(acc, V, Sm::LV, Q, Sm::LQ, m0, n0, ns, C, w + 4 * C);
        each(acc, m0, n0, ns, put(ws.o_w(), D));
    });
    tiles<false, D, D>([&](float (&acc)[4][4], int m0, int n0, int ns) {
        mac<true, false>(acc, dU, Sm::LQ, Q, Sm::LQ, m0, n0, ns, C, w + 5 * C);
        each(acc, m0, n0, ns, put(ws.o_oloc(), D));
    });
}

// ---- (2) scan over chunks ---------------------------------------------------------
// blockIdx.x = (u * kSplit + part) * 2 + dir.  dir 0: S (whole) and the columns
// [part*dv/kSplit, ...) of X, forward in time.  dir 1: Lam (whole) and the columns
// [part*d/kSplit, ...) of Om, backward in time.  Each CTA stores its column block
// of X_p / Om_next and the row block `part` of S_p / Lam_next.  The next chunk's local
// sums are copied into the other of two shared buffers (cp.async) while the current
// chunk is applied.
template <int C, int D, int DV>
struct ScanSmem {
    static constexpr int WMAX = DV > D ? DV : D;
    static constexpr int NB = WMAX / kSplit;  // widest column block
    static constexpr int FW = WMAX + 4, LB = NB + 4;
    // F: S or Lam (D x <= WMAX); BK: the column block of X or Om; then two buffers of
    // FL (the increment of F), R (the product operand block, Cq or W, <= WMAX rows)
    // and BL (the block increment).  At d = 128 two D x D increments do not fit beside
    // the rest, so FL is not staged: the update reads it from the workspace.
    static constexpr bool STAGE_FL = D <= 64;
    static constexpr int F = 0, BK = F + D * FW, RED = BK + D * LB, BUF = RED + kThreads * 16;
    static constexpr int B_FL = 0, B_R = STAGE_FL ? D * FW : 0, B_BL = B_R + WMAX * LB, BUFSZ = B_BL + D * LB;
    static constexpr int TOTAL = BUF + 2 * BUFSZ;
};

// One direction of the scan (DIR 0: S and X forward; DIR 1: Lam and Om backward).
template <int C, int D, int DV, int DIR>
__device__ __forceinline__ void scan_dir(const BwdArgs &a, float *sm, int part, int u) {
    using Sm = ScanSmem<C, D, DV>;
    // DIR 0: F = S (D x D), block of X (D x DV), R = block of Cq (D x DV)
    // DIR 1: F = Lam (D x DV), block of Om (D x D), R = block of W (DV x D)
    constexpr int FWD = DIR == 0 ? D : DV, BW = DIR == 0 ? DV : D, NBD = BW / kSplit;
    constexpr int RK = DIR == 0 ? D : DV;  // inner dimension of F R
    constexpr int ROWS = D / kSplit;
    float *F = sm + Sm::F, *Bk = sm + Sm::BK, *red = sm + Sm::RED;
    const int nch = (a.n + C - 1) / C, c0 = part * NBD, rows0 = part * ROWS;
    const bool decay = (a.flags & HLA_DECAY) != 0;
    const float lg = log2f(decay ? a.gamma[u % a.H] : 1.f);
    const BwdWs ws{D, DV};
    const float *loc = a.workspace + (size_t)u * nch * ws.loc_floats();
    float *st = a.workspace + (size_t)a.B * a.H * nch * ws.loc_floats() + (size_t)u * nch * ws.st_floats();
    auto chunk_at = [&](int it) { return DIR == 0 ? it : nch - 1 - it; };
    auto issue = [&](int it) {  // the local sums of step it into buffer it & 1
        const float *lc = loc + (size_t)chunk_at(it) * ws.loc_floats();
        float *b = sm + Sm::BUF + (it & 1) * Sm::BUFSZ;
        if constexpr (Sm::STAGE_FL)
            copy_mat_async<FWD>(lc + (DIR == 0 ? ws.o_sloc() : ws.o_lloc()), FWD, b + Sm::B_FL, Sm::FW, D);
        copy_mat_async<NBD>(lc + (DIR == 0 ? ws.o_cq() : ws.o_w()) + c0, BW, b + Sm::B_R, Sm::LB, RK);
        copy_mat_async<NBD>(lc + (DIR == 0 ? ws.o_xloc() : ws.o_oloc()) + c0, BW, b + Sm::B_BL, Sm::LB, D);
    };
    if (nch > 0) issue(0);
    cp_async_commit();
    for (int e = threadIdx.x; e < D * Sm::FW; e += kThreads) F[e] = 0.f;
    for (int e = threadIdx.x; e < D * Sm::LB; e += kThreads) Bk[e] = 0.f;
    __syncthreads();
    if (DIR == 0 && a.sin_S) {  // S = S_in; the column block of X_in = S_in C_in - G_in
        float *R1 = sm + Sm::BUF + Sm::BUFSZ + Sm::B_R;  // buffer 1 is not in use yet
        for (int e = threadIdx.x; e < D * D; e += kThreads)
            F[(e / D) * Sm::FW + e % D] = a.sin_S[(size_t)u * D * D + e];
        for (int e = threadIdx.x; e < D * NBD; e += kThreads)
            R1[(e / NBD) * Sm::LB + e % NBD] = a.sin_C[(size_t)u * D * DV + (size_t)(e / NBD) * DV + c0 + e % NBD];
        __syncthreads();
        mac_ksplit<D, NBD, D>(F, Sm::FW, R1, Sm::LB, red);
        __syncthreads();
        for (int e = threadIdx.x; e < D * NBD; e += kThreads)
            Bk[(e / NBD) * Sm::LB + e % NBD] = ksplit_sum<D, NBD, D>(red, e) -
                                               a.sin_G[(size_t)u * D * DV + (size_t)(e / NBD) * DV + c0 + e % NBD];
        __syncthreads();
    }
    for (int it = 0; it < nch; ++it) {
        if (it + 1 < nch) issue(it + 1);
        cp_async_commit();
        const int ch = chunk_at(it);
        const int L = min(C, a.n - ch * C);
        const float f1 = decay ? gpow(lg, (float)L) : 1.f, f2 = decay ? gpow(lg, (float)(2 * L)) : 1.f;
        float *so = st + (size_t)ch * ws.st_floats();
        // the states this chunk starts from (S_p, X_p) or ends into (Lam_next, Om_next)
        float *fo = so + (DIR == 0 ? ws.o_sp() : ws.o_lam()), *bo = so + (DIR == 0 ? ws.o_xp() : ws.o_om());
        for (int e = threadIdx.x; e < ROWS * FWD; e += kThreads) {
            const int r = rows0 + e / FWD, x = e % FWD;
            fo[(size_t)r * FWD + x] = F[r * Sm::FW + x];
        }
        for (int e = threadIdx.x; e < D * NBD; e += kThreads) {
            const int r = e / NBD, x = e % NBD;
            bo[(size_t)r * BW + c0 + x] = Bk[r * Sm::LB + x];
        }
        cp_async_wait<1>();  // step it's copies (the group before the one just committed)
        __syncthreads();
        const float *b = sm + Sm::BUF + (it & 1) * Sm::BUFSZ;
        const float *Fl = b + Sm::B_FL, *R = b + Sm::B_R, *Bl = b + Sm::B_BL;
        // the increment of F in the workspace (read there when it is not staged)
        const float *Flg = loc + (size_t)ch * ws.loc_floats() + (DIR == 0 ? ws.o_sloc() : ws.o_lloc());
        // block <- f_b block + Bl + F R  (F the state before this chunk's update), F R over all threads
        const float fb = DIR == 0 ? f2 : f1, ff = DIR == 0 ? f1 : f2;
        mac_ksplit<D, NBD, RK>(F, Sm::FW, R, Sm::LB, red);
        __syncthreads();
        for (int e = threadIdx.x; e < D * NBD; e += kThreads) {
            const int o = (e / NBD) * Sm::LB + e % NBD;
            Bk[o] = fb * Bk[o] + Bl[o] + ksplit_sum<D, NBD, RK>(red, e);
        }
        __syncthreads();
        for (int e = threadIdx.x; e < D * FWD; e += kThreads) {
            const int r = e / FWD, x = e % FWD;
            F[r * Sm::FW + x] = ff * F[r * Sm::FW + x] + (Sm::STAGE_FL ? Fl[r * Sm::FW + x] : Flg[e]);
        }
        __syncthreads();
    }
    cp_async_wait<0>();
    if (DIR == 1 && a.adj0) {  // Lam and Om at the first token (rows of Lam, a column block of Om)
        float *lam0 = a.adj0 + (size_t)u * (D * DV + D * D), *om0 = lam0 + D * DV;
        for (int e = threadIdx.x; e < ROWS * FWD; e += kThreads) {
            const int r = rows0 + e / FWD, x = e % FWD;
            lam0[(size_t)r * FWD + x] = F[r * Sm::FW + x];
        }
        for (int e = threadIdx.x; e < D * NBD; e += kThreads) {
            const int r = e / NBD, x = e % NBD;
            om0[(size_t)r * BW + c0 + x] = Bk[r * Sm::LB + x];
        }
    }
}

// The gradient of the initial state from the adjoints at the first token, one CTA per
// pair: dX_in = g^2 Lam, dG_in = -dX_in, dC_in = S_in^T dX_in, dS_in = g Om + dX_in C_in^T
// (without a given state: dC_in = 0, dS_in = g Om).
template <int D, int DV>
struct StateGradSmem {
    static constexpr int LS = D + 4, LX = DV + 4;
    static constexpr int S = 0, C = S + D * LS, X = C + D * LX, TOTAL = X + D * LX;
};
template <int D, int DV>
__global__ void __launch_bounds__(kThreads) bwd_state_grad_kernel(BwdArgs a) {
    using Sm = StateGradSmem<D, DV>;
    extern __shared__ __align__(16) float sm[];
    float *S = sm + Sm::S, *Cm = sm + Sm::C, *dX = sm + Sm::X;
    const int u = blockIdx.x;
    const bool decay = (a.flags & HLA_DECAY) != 0;
    const float g = decay ? a.gamma[u % a.H] : 1.f;
    const float *lam0 = a.adj0 + (size_t)u * (D * DV + D * D), *om0 = lam0 + D * DV;
    const size_t oS = (size_t)u * D * D, oC = (size_t)u * D * DV;
    const bool have = a.sin_S != nullptr;
    for (int e = threadIdx.x; e < D * DV; e += kThreads) {
        const int r = e / DV, x = e % DV;
        const float d = g * g * lam0[e];
        dX[r * Sm::LX + x] = d;
        a.dG[oC + e] = -d;
        Cm[r * Sm::LX + x] = have ? a.sin_C[oC + e] : 0.f;
    }
    for (int e = threadIdx.x; e < D * D; e += kThreads) S[(e / D) * Sm::LS + e % D] = have ? a.sin_S[oS + e] : 0.f;
    __syncthreads();
    tiles<false, D, DV>([&](float (&acc)[4][4], int m0, int n0, int ns) {
        mac<true, false>(acc, S, Sm::LS, dX, Sm::LX, m0, n0, ns, D);
        each(acc, m0, n0, ns, [&](int j, int c, float x) { a.dC[oC + (size_t)j * DV + c] = x; });
    });
    tiles<false, D, D>([&](float (&acc)[4][4], int m0, int n0, int ns) {
        mac<false, true>(acc, dX, Sm::LX, Cm, Sm::LX, m0, n0, ns, DV);
        each(acc, m0, n0, ns, [&](int i, int j, float x) { a.dS[oS + (size_t)i * D + j] = g * om0[(size_t)i * D + j] + x; });
    });
}

template <int C, int D, int DV>
__global__ void __launch_bounds__(kThreads) bwd_scan_kernel(BwdArgs a) {
    extern __shared__ __align__(16) float sm[];
    const int dir = blockIdx.x & 1, part = (blockIdx.x >> 1) % kSplit, u = (blockIdx.x >> 1) / kSplit;
    if (dir == 0) scan_dir<C, D, DV, 0>(a, sm, part, u);
    else scan_dir<C, D, DV, 1>(a, sm, part, u);
}

// ---- (3) gradients of one chunk ---------------------------------------------------
template <int C, int D, int DV>
struct GradSmem {
    static constexpr int LQ = D + 4, LV = DV + 4, LT = C + 4;
    static constexpr int Q = 0, K = Q + C * LQ, V = K + C * LQ, G = V + C * LV, SP = G + C * LV, XP = SP + D * LQ,
                         LAM = XP + D * LV, OM = LAM + D * LV, A = OM + D * LQ, P = A + C * LT, BM = P + C * LT,
                         U = BM + C * LT, DU = U + C * LQ, GP = DU + C * LQ, RS = GP + 2 * C + 4,
                         TOTAL = RS + 4 * C;
};

template <typename T, int C, int D, int DV>
__global__ void __launch_bounds__(kThreads) bwd_grad_kernel(BwdArgs a) {
    using Sm = GradSmem<C, D, DV>;
    extern __shared__ __align__(16) float sm[];
    float *Q = sm + Sm::Q, *K = sm + Sm::K, *V = sm + Sm::V, *G = sm + Sm::G, *Sp = sm + Sm::SP, *Xp = sm + Sm::XP;
    float *Lam = sm + Sm::LAM, *Om = sm + Sm::OM, *A = sm + Sm::A, *P = sm + Sm::P, *Bm = sm + Sm::BM;
    float *U = sm + Sm::U, *dU = sm + Sm::DU, *gp = sm + Sm::GP, *rs = sm + Sm::RS;
    const int nch = (a.n + C - 1) / C, u = blockIdx.x / nch, ch = blockIdx.x % nch;
    const int t0 = ch * C, L = min(C, a.n - t0);
    const bool decay = (a.flags & HLA_DECAY) != 0;
    const float lg = log2f(decay ? a.gamma[u % a.H] : 1.f);
    const size_t rq = ((size_t)u * a.n + t0) * D, rv = ((size_t)u * a.n + t0) * DV;
    const BwdWs ws{D, DV};
    const float *so =
        a.workspace + (size_t)a.B * a.H * nch * ws.loc_floats() + ((size_t)u * nch + ch) * ws.st_floats();
    // the chunk's states arrive asynchronously while A~ and P are formed
    copy_mat_async<D>(so + ws.o_sp(), D, Sp, Sm::LQ, D);
    copy_mat_async<DV>(so + ws.o_xp(), DV, Xp, Sm::LV, D);
    copy_mat_async<DV>(so + ws.o_lam(), DV, Lam, Sm::LV, D);
    copy_mat_async<D>(so + ws.o_om(), D, Om, Sm::LQ, D);
    cp_async_commit();
    const size_t kvu = kv_unit(a, u), rk = (kvu * a.n + t0) * D, rkv = (kvu * a.n + t0) * DV;
    load_rows<D>(static_cast<const T *>(a.q) + rq, Q, Sm::LQ, C, L);
    load_rows<D>(static_cast<const T *>(a.k) + rk, K, Sm::LQ, C, L);
    load_rows<DV>(static_cast<const T *>(a.v) + rkv, V, Sm::LV, C, L);
    load_rows<DV>(static_cast<const T *>(a.go) + rv, G, Sm::LV, C, L);
    fill_gp(gp, C, lg, decay);
    __syncthreads();
    float *r_u = rs, *r_x = rs + C, *r_l2 = rs + 2 * C, *r_l1 = rs + 3 * C;
    for (int t = threadIdx.x; t < C; t += kThreads) {
        const bool in = t < L;
        r_u[t] = gp[t + 1];                    // g^{tau+1}
        r_x[t] = gp[2 * (t + 1)];              // g^{2(tau+1)}
        r_l2[t] = in ? gp[2 * (L - t)] : 0.f;  // g^{2(L-tau)}
        r_l1[t] = in ? gp[L - t] : 0.f;        // g^{L-tau}
    }
    tiles<true, C, C>([&](float (&acc)[4][4], int m0, int n0, int ns) {
        mac<false, true>(acc, Q, Sm::LQ, K, Sm::LQ, m0, n0, ns, D);
        each(acc, m0, n0, ns, [&](int t, int s, float x) { A[t * Sm::LT + s] = s <= t ? gp[t - s] * x : 0.f; });
    });
    tiles<true, C, C>([&](float (&acc)[4][4], int m0, int n0, int ns) {
        mac<false, true>(acc, G, Sm::LV, V, Sm::LV, m0, n0, ns, DV);
        each(acc, m0, n0, ns, [&](int s, int b, float x) { P[s * Sm::LT + b] = b <= s ? gp[2 * (s - b)] * x : 0.f; });
    });
    cp_async_wait<0>();
    __syncthreads();
    // U = diag(g^{tau+1}) Q S_p + A~ K;  dU = P^T Q + diag(g^{2(L-tau)}) V Lam^T
    tiles<false, C, D>([&](float (&acc)[4][4], int m0, int n0, int ns) {
        mac_rs<false, false>(acc, r_u, Q, Sm::LQ, Sp, Sm::LQ, m0, n0, ns, D);
        mac<false, false>(acc, A, Sm::LT, K, Sm::LQ, m0, n0, ns, C);
        each(acc, m0, n0, ns, [&](int t, int i, float x) { U[t * Sm::LQ + i] = x; });
    });
    tiles<true, C, D>([&](float (&acc)[4][4], int m0, int n0, int ns) {
        mac<true, false>(acc, P, Sm::LT, Q, Sm::LQ, m0, n0, ns, C);
        mac_rs<false, true>(acc, r_l2, V, Sm::LV, Lam, Sm::LV, m0, n0, ns, DV);
        each(acc, m0, n0, ns, [&](int t, int i, float x) { dU[t * Sm::LQ + i] = x; });
    });
    __syncthreads();
    // B = tril(g^{t-a} dU K^T)
    tiles<true, C, C>([&](float (&acc)[4][4], int m0, int n0, int ns) {
        mac<false, true>(acc, dU, Sm::LQ, K, Sm::LQ, m0, n0, ns, D);
        each(acc, m0, n0, ns, [&](int t, int s, float x) { Bm[t * Sm::LT + s] = s <= t ? gp[t - s] * x : 0.f; });
    });
    __syncthreads();
    T *gq = static_cast<T *>(a.grad_q) + rq;
    // dk, dv: straight to the output with one query head per key/value head, else to
    // the per-query-head fp32 staging that the group sum reads
    T *gk = a.dk_pair ? nullptr : static_cast<T *>(a.grad_k) + rq;
    T *gv = a.dv_pair ? nullptr : static_cast<T *>(a.grad_v) + rv;
    float *pk = a.dk_pair ? a.dk_pair + rq : nullptr, *pv = a.dv_pair ? a.dv_pair + rv : nullptr;
    // dQ = P U + diag(g^{2(tau+1)}) G X_p^T + diag(g^{tau+1}) dU S_p + B K   (S_p symmetric)
    tiles<false, C, D>([&](float (&acc)[4][4], int m0, int n0, int ns) {
        mac<false, false>(acc, P, Sm::LT, U, Sm::LQ, m0, n0, ns, C);
        mac_rs<false, true>(acc, r_x, G, Sm::LV, Xp, Sm::LV, m0, n0, ns, DV);
        mac_rs<false, false>(acc, r_u, dU, Sm::LQ, Sp, Sm::LQ, m0, n0, ns, D);
        mac<false, false>(acc, Bm, Sm::LT, K, Sm::LQ, m0, n0, ns, C);
        each(acc, m0, n0, ns, [&](int t, int i, float x) {
            if (t < L) st_t(gq, (size_t)t * D + i, x);
        });
    });
    // dK = A~^T dU + B^T Q + diag(g^{L-tau}) K (Om + Om^T)
    tiles<false, C, D>([&](float (&acc)[4][4], int m0, int n0, int ns) {
        mac<true, false>(acc, A, Sm::LT, dU, Sm::LQ, m0, n0, ns, C);
        mac<true, false>(acc, Bm, Sm::LT, Q, Sm::LQ, m0, n0, ns, C);
        mac_rs<false, false>(acc, r_l1, K, Sm::LQ, Om, Sm::LQ, m0, n0, ns, D);
        mac_rs<false, true>(acc, r_l1, K, Sm::LQ, Om, Sm::LQ, m0, n0, ns, D);
        each(acc, m0, n0, ns, [&](int t, int i, float x) {
            if (t < L) {
                if (pk) pk[(size_t)t * D + i] = x;
                else st_t(gk, (size_t)t * D + i, x);
            }
        });
    });
    __syncthreads();
    // M = tril(g^{2(s-t)} Q U^T) into the slot of P
    tiles<true, C, C>([&](float (&acc)[4][4], int m0, int n0, int ns) {
        mac<false, true>(acc, Q, Sm::LQ, U, Sm::LQ, m0, n0, ns, D);
        each(acc, m0, n0, ns, [&](int s, int t, float x) { P[s * Sm::LT + t] = t <= s ? gp[2 * (s - t)] * x : 0.f; });
    });
    __syncthreads();
    // dV = M^T G + diag(g^{2(L-tau)}) U Lam
    tiles<false, C, DV>([&](float (&acc)[4][4], int m0, int n0, int ns) {
        mac<true, false>(acc, P, Sm::LT, G, Sm::LV, m0, n0, ns, C);
        mac_rs<false, false>(acc, r_l2, U, Sm::LQ, Lam, Sm::LV, m0, n0, ns, D);
        each(acc, m0, n0, ns, [&](int t, int j, float x) {
            if (t < L) {
                if (pv) pv[(size_t)t * DV + j] = x;
                else st_t(gv, (size_t)t * DV + j, x);
            }
        });
    });
}

template <typename Kern>
cudaError_t smem_attr(Kern kern, size_t bytes) {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <typename T, int C, int D, int DV>
cudaError_t launch_t(const BwdArgs &a, cudaStream_t st) {
    const int nch = (a.n + C - 1) / C, units = a.B * a.H;
    const size_t b1 = LocSmem<C, D, DV>::TOTAL * sizeof(float), b2 = ScanSmem<C, D, DV>::TOTAL * sizeof(float),
                 b3 = GradSmem<C, D, DV>::TOTAL * sizeof(float);
    cudaError_t e;
    constexpr bool TC = std::is_same<T, __nv_bfloat16>::value && C == 64 && D == 64 && DV == 64;
    // with a given initial state, or its gradient wanted, the scan is the CUDA-core one
    const bool tc_scan = TC && !a.sin_S && !a.adj0;
    if (!tc_scan && (e = smem_attr(bwd_scan_kernel<C, D, DV>, b2)) != cudaSuccess) return e;
    if (a.adj0 &&
        (e = smem_attr(bwd_state_grad_kernel<D, DV>, StateGradSmem<D, DV>::TOTAL * sizeof(float))) != cudaSuccess)
        return e;
    if constexpr (!TC) {  // the CUDA-core kernels (the tensor-core ones set their own attributes)
        if ((e = smem_attr(bwd_local_kernel<T, C, D, DV>, b1)) != cudaSuccess) return e;
        if ((e = smem_attr(bwd_grad_kernel<T, C, D, DV>, b3)) != cudaSuccess) return e;
    }
    auto mark = [&](int i) { return a.events ? cudaEventRecord(a.events[i], st) : cudaSuccess; };
    if ((e = mark(0)) != cudaSuccess) return e;
    if constexpr (TC) {
        if ((e = bwdtc::local_tc(a, st)) != cudaSuccess) return e;
    } else {
        bwd_local_kernel<T, C, D, DV><<<units * nch, kThreads, b1, st>>>(a);
    }
    if ((e = mark(1)) != cudaSuccess) return e;
    if (tc_scan) {
        if ((e = scantc::bwd_scan(a, st)) != cudaSuccess) return e;
    } else {
        bwd_scan_kernel<C, D, DV><<<units * kSplit * 2, kThreads, b2, st>>>(a);
    }
    if (a.adj0)
        bwd_state_grad_kernel<D, DV><<<units, kThreads, StateGradSmem<D, DV>::TOTAL * sizeof(float), st>>>(a);
    if ((e = mark(2)) != cudaSuccess) return e;
    if constexpr (TC) {
        if ((e = bwdtc::grad_tc(a, st)) != cudaSuccess) return e;
    } else {
        bwd_grad_kernel<T, C, D, DV><<<units * nch, kThreads, b3, st>>>(a);
    }
    if (a.dk_pair) {  // shared key/value heads: sum each group's gradients
        const size_t elems = (size_t)a.B * a.Hkv * a.n * (D > DV ? D : DV);
        const int blocks = (int)((elems + kThreads - 1) / kThreads < 8192 ? (elems + kThreads - 1) / kThreads : 8192);
        bwd_group_sum_kernel<T><<<blocks, kThreads, 0, st>>>(a.dk_pair, static_cast<T *>(a.grad_k), a.B, a.H, a.Hkv,
                                                            (size_t)a.n * D);
        bwd_group_sum_kernel<T><<<blocks, kThreads, 0, st>>>(a.dv_pair, static_cast<T *>(a.grad_v), a.B, a.H, a.Hkv,
                                                            (size_t)a.n * DV);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if ((e = mark(3)) != cudaSuccess) return e;
    return cudaGetLastError();
}
template <typename T, int C, int D>
cudaError_t launch_dv(const BwdArgs &a, cudaStream_t st) {
    switch (a.dv) {
        case 16: return launch_t<T, C, D, 16>(a, st);
        case 32: return launch_t<T, C, D, 32>(a, st);
        case 64: return launch_t<T, C, D, 64>(a, st);
    }
    return cudaErrorInvalidValue;
}
template <typename T, int C>
cudaError_t launch_d(const BwdArgs &a, cudaStream_t st) {
    switch (a.d) {
        case 16: return launch_dv<T, C, 16>(a, st);
        case 32: return launch_dv<T, C, 32>(a, st);
        case 64: return launch_dv<T, C, 64>(a, st);
        case 128:
            // d = 128: the gradient kernel's fp32 states (two d x d, two d x dv) and its
            // chunk tiles fit 227 KB of shared memory at 16-token chunks and dv <= 32
            if constexpr (C == 16) {
                if (a.dv == 16) return launch_t<T, C, 128, 16>(a, st);
                if (a.dv == 32) return launch_t<T, C, 128, 32>(a, st);
            }
            break;
    }
    return cudaErrorInvalidValue;
}
// One translation unit per (element type, chunk) instantiates launch_d.
}  // namespace bwd
}  // namespace hla
