// hla_fwd_tc.cu -- chunk-parallel masked second-order HLA forward on the
// sm_103a tensor cores (tcgen05 MMA, TMEM accumulators, TMA tile loads), bf16
// inputs, fp32 accumulation and fp32 state.
//
// Method (gist.science summary of "Higher-order Linear Attention", section 1 for
// the summaries and the masked output, section 4 for the segment concatenation
// and the exclusive scan).  Working form: instead of the cross summaries G, h
// the kernel carries X = S C - G and Y = S m - h, for which
//   X_t = g^2 X_{t-1} + u_t v_t^T,  Y_t = g^2 Y_{t-1} + u_t,  u_t = S_t q_t,
//   o_t = q_t^T X_t,  den_t = q_t^T Y_t
// (expand S_t C_t - G_t with the updates of S, C and G).  In this form the
// concatenation of segment A before B (f = g^{len B}) reads
//   S = f S_A + S_B, C = f C_A + C_B, m = f m_A + m_B,
//   X = f^2 X_A + X_B + f S_A C_B,  Y = f^2 Y_A + Y_B + f S_A m_B,
// which is the pages' rule with G = S C - X substituted.
//
// Per chunk of c tokens (local positions tau = 1..L after prefix position p),
// with state (S_p, X_p, Y_p) at the chunk start:
//   A   = tril(Gamma1 o Q K^T),   Gamma1[t,a] = g^{t-a}             (MMA + epilogue)
//   U   = diag(g^tau) Q S_p + A K                                     (rows u_b = S_b q_b)
//   M   = tril(Gamma2 o Q U^T),   Gamma2[t,b] = g^{2(t-b)}
//   O   = M V + diag(g^{2 tau}) Q X_p,  den = rowsum(M) + diag(g^{2 tau}) Q Y_p
//   S  <- g^L S + K^T W K,  X <- g^{2L} X + U^T W^2 V,  C <- g^L C + Q^T W V,
//   with W = diag(g^{L - tau}).
//
// Parallel structure (one launch): the (b,h) sequence is cut into `nseg`
// segments of whole chunks; one CTA per (b,h,segment), CTAs ordered by a ticket
// so that a CTA only ever waits for CTAs that started before it.
//   pass 1: the segment's own summary (S, C, X, m, Y from zero) -> workspace,
//           then a release flag;
//   scan:   the CTA folds state_in and the summaries of all earlier segments of
//           its sequence (exclusive scan by the concatenation rule);
//   pass 2: the chunk loop again from that exact prefix, writing O.
// The last segment exports state_out (S, C, m, G = S C - X, h = S m - Y).
//
// Each CTA: 128 threads (4 warps); thread 0 issues TMA and MMAs; all threads
// run the TMEM<->register epilogues.  TMEM (512 columns): work W [0,128),
// S [128,256), X [256,384), C (pass 1 / scan) or spare (pass 2) [384,512).
// Token-row accumulators use M = c rows, state accumulators M = d rows.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>

#include "hla_internal.h"

namespace hla {
namespace {

constexpr int kThreads = 128;
constexpr uint32_t TW = 0, TS = 128, TX = 256, T4 = 384, kTmemCols = 512;

__host__ __device__ constexpr int cmax(int a, int b) { return a > b ? a : b; }

struct TcParams {
    CUtensorMap tmQ, tmK, tmV;
    int B, H, n, BH;
    int nchunks, nseg, cps;
    unsigned flags;
    float eps;
    const float *gamma;
    void *o;
    StatePtrs sin, sout;
    unsigned *ticket;   // workspace header: [0] ticket counter, [1] finished CTAs
    unsigned *flagsw;   // [BH][nseg] release flags
    float *summ;        // [BH][nseg][SUM] segment summaries
    float *save;        // [BH][SAVE] prefix copy for the state export
    unsigned *err;
};

template <int C, int D, int DV>
struct Cfg {
    static constexpr int SUM = D * D + 2 * D * DV + 2 * D;  // S, X, C, m, Y
    static constexpr int SAVE = D * D + D * DV + 2 * D;     // S, X, m, Y
    // operand tiles (bytes)
    static constexpr int SZ_Q = C * D * 2, SZ_K = C * D * 2, SZ_V = C * DV * 2;
    static constexpr int SZ_TA = cmax(C * C, C * D) * 2;
    static constexpr int SZ_TU = C * D * 2;
    static constexpr int SZ_TS = cmax(cmax(D * D, C * D), C * DV) * 2;
    static constexpr int SZ_TQ = cmax(C * D, D * DV) * 2;
    static constexpr int OFF_Q = 0, OFF_K = OFF_Q + SZ_Q, OFF_V = OFF_K + SZ_K, OFF_TA = OFF_V + SZ_V,
                         OFF_TU = OFF_TA + SZ_TA, OFF_TS = OFF_TU + SZ_TU, OFF_TQ = OFF_TS + SZ_TS,
                         TILES = OFF_TQ + SZ_TQ;
    // scan / export phase operands (alias the tiles)
    static constexpr int OFF_SHI = 0, OFF_SLO = D * D * 2, OFF_CHI = 2 * D * D * 2,
                         OFF_CLO = 2 * D * D * 2 + D * DV * 2, FOLD = 2 * D * D * 2 + 2 * D * DV * 2;
    static constexpr int ARENA = cmax(TILES, FOLD);
    // fp32 vectors (m, Y, m_L, scratch) and the barriers after the arena
    static constexpr int NVEC = 4 * D;
    static constexpr int OFF_BAR = ARENA + NVEC * 4;
    static constexpr int SMEM = OFF_BAR + 64;
    static constexpr int SMEM_LAUNCH = cmax(SMEM, 120 * 1024);  // one CTA per SM
    static constexpr uint32_t TX_BYTES = SZ_Q + SZ_K + SZ_V;
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
    static_assert(C == 64 || C == 128, "chunk");
    static_assert(D == 64 || D == 128, "d");
    static_assert(DV == 64 || DV == 128, "dv");
};

// Per-CTA context.
template <int C, int D, int DV>
struct Ctx {
    using K_ = Cfg<C, D, DV>;
    const TcParams *P;
    uint8_t *sQ, *sK, *sV, *sTA, *sTU, *sTS, *sTQ;
    uint8_t *sShi, *sSlo, *sChi, *sClo;
    float *mrun, *Yrun, *mL, *tmp;  // [D] each
    uint64_t *tma_bar, *mma_bar;
    uint32_t tb;  // TMEM base
    uint32_t tph, mph;
    int tid, warp, bh;
    bool decay, norm;
    float lg;

    // g^x for the decay variant (1 without decay); 0^0 = 1
    __device__ float gp(int x) const { return decay ? gpow(lg, (float)x) : 1.f; }
    __device__ uint32_t taddr(uint32_t slot, int col) const { return tmem_warp_addr(tb + slot, warp, col); }

    // ---- synchronisation helpers; false = abort (a bounded wait expired)
    __device__ bool wait_mma() {
        bool ok = mbar_wait(mma_bar, mph, P->err);
        mph ^= 1u;
        tc_fence_after();
        return !__syncthreads_or(!ok);
    }
    __device__ bool wait_tma() {
        bool ok = mbar_wait(tma_bar, tph, P->err);
        tph ^= 1u;
        return !__syncthreads_or(!ok);
    }
    // Make this thread's shared-memory and TMEM writes visible to MMAs issued next.
    __device__ void publish() {
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }
    __device__ void commit() {
        if (tid == 0) umma_commit(mma_bar);
    }

    // ---- MMA groups (called by thread 0 only)
    // token-row product, A K-major [C x KD], B K-major [N x KD]
    __device__ void mma_kk(uint32_t slot, const uint8_t *a, const uint8_t *b, int N, int KD, bool acc) {
        const uint32_t id = make_idesc(C, N, false, false);
        for (int k = 0; k < KD; k += 16)
            umma_f16(tb + slot, desc_kmajor(a, C, k), desc_kmajor(b, N, k), id, (acc || k > 0) ? 1u : 0u);
    }
    // token-row product, A K-major [C x KD], B MN-major [KD x N]
    __device__ void mma_km(uint32_t slot, const uint8_t *a, const uint8_t *b, int N, int KD, bool acc) {
        const uint32_t id = make_idesc(C, N, false, true);
        for (int k = 0; k < KD; k += 16)
            umma_f16(tb + slot, desc_kmajor(a, C, k), desc_mnmajor(b, KD, k), id, (acc || k > 0) ? 1u : 0u);
    }
    // state product over tokens: A MN-major [C x D] (as D x C), B MN-major [C x N]
    __device__ void mma_mm(uint32_t slot, const uint8_t *a, const uint8_t *b, int N, bool acc) {
        const uint32_t id = make_idesc(D, N, true, true);
        for (int k = 0; k < C; k += 16)
            umma_f16(tb + slot, desc_mnmajor(a, C, k), desc_mnmajor(b, C, k), id, (acc || k > 0) ? 1u : 0u);
    }
    // state x state: A K-major [D x D] (rows = M), B MN-major [D x DV]
    __device__ void mma_ss(uint32_t slot, const uint8_t *a, const uint8_t *b, bool acc) {
        const uint32_t id = make_idesc(D, DV, false, true);
        for (int k = 0; k < D; k += 16)
            umma_f16(tb + slot, desc_kmajor(a, D, k), desc_mnmajor(b, D, k), id, (acc || k > 0) ? 1u : 0u);
    }

    __device__ void tma_chunk(int jj) {
        if (tid == 0) {
            fence_async_smem();  // earlier generic reads of the tiles precede the overwrite
            mbar_expect_tx(tma_bar, K_::TX_BYTES);
            const int t0 = jj * C;
            for (int kb = 0; kb < D / 64; ++kb) {
                tma_load_3d(sQ + kb * C * 128, &P->tmQ, tma_bar, kb * 64, t0, bh);
                tma_load_3d(sK + kb * C * 128, &P->tmK, tma_bar, kb * 64, t0, bh);
            }
            for (int kb = 0; kb < DV / 64; ++kb) tma_load_3d(sV + kb * C * 128, &P->tmV, tma_bar, kb * 64, t0, bh);
        }
    }

    // ---- row-wise TMEM access: this thread's row of an accumulator with MR rows
    // Calls f(col0, vals[16]) for every 16-column group of `ncols` columns of slot.
    template <int MR, typename F>
    __device__ void for_row(uint32_t slot, int ncols, F &&f) {
        float v[16];
        for (int c0 = 0; c0 < ncols; c0 += 16) {
            tmem_ld16(taddr(slot, c0), v);
            tmem_wait_ld();
            f(c0, v);
        }
    }
    // Read-modify-write: f(col0, vals) may change vals; they are stored back.
    template <int MR, typename F>
    __device__ void rmw_row(uint32_t slot, int ncols, F &&f) {
        float v[16];
        for (int c0 = 0; c0 < ncols; c0 += 16) {
            tmem_ld16(taddr(slot, c0), v);
            tmem_wait_ld();
            f(c0, v);
            tmem_st16(taddr(slot, c0), v);
        }
        tmem_wait_st();
    }
    template <int MR>
    __device__ void zero_slot(uint32_t slot, int ncols) {
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = 0.f;
        for (int c0 = 0; c0 < ncols; c0 += 16) tmem_st16(taddr(slot, c0), v);
        tmem_wait_st();
    }
};

// Row-scaled copy of a [C x W] tile: dst[r] = scale(r) * src[r].
template <int C, int W, typename F>
__device__ void scaled_tile_copy(const uint8_t *src, uint8_t *dst, int tid, F &&scale) {
    for (int r = tid; r < C; r += kThreads) {
        const float s = scale(r);
        for (int c0 = 0; c0 < W; c0 += 16) {
            float a[8], b[8], v[16];
            tile_load_row8(src, C, r, c0, a);
            tile_load_row8(src, C, r, c0 + 8, b);
#pragma unroll
            for (int i = 0; i < 8; ++i) { v[i] = s * a[i]; v[8 + i] = s * b[i]; }
            tile_store_row16(const_cast<uint8_t *>(dst), C, r, c0, v);
        }
    }
}

// Split 16 fp32 values into bf16 hi + lo parts and store both rows.
__device__ __forceinline__ void store_hilo(uint8_t *hi, uint8_t *lo, int rows, int r, int c0, const float (&v)[16]) {
    float h[16], l[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        h[i] = __bfloat162float(__float2bfloat16_rn(v[i]));
        l[i] = v[i] - h[i];
    }
    tile_store_row16(hi, rows, r, c0, h);
    tile_store_row16(lo, rows, r, c0, l);
}

// ============================================================================ pass 1
// Segment summary from zero state over chunks [jb, je).  Result: TMEM S, X, C
// slots and mrun/Yrun hold (S, X, C, m, Y) of the segment.
template <int C, int D, int DV>
__device__ bool pass1(Ctx<C, D, DV> &x, int jb, int je) {
    const TcParams &P = *x.P;
    const int rowC = owned_row<C>(x.tid);
    const int rowD = owned_row<D>(x.tid);
    for (int i = x.tid; i < D; i += kThreads) x.mrun[i] = x.Yrun[i] = 0.f;
    for (int jj = jb; jj < je; ++jj) {
        const bool first = (jj == jb);
        const int L = min(C, P.n - jj * C);
        x.tma_chunk(jj);
        // state at the chunk start -> bf16 operand copy of S; decay the state
        if (!first) {
            const float gL = x.gp(L), g2L = x.gp(2 * L);
            x.template rmw_row<D>(TS, D, [&](int c0, float (&v)[16]) {
                if (rowD >= 0) tile_store_row16(x.sTS, D, rowD, c0, v);
                if (x.decay)
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] *= gL;
            });
            if (x.decay) {
                x.template rmw_row<D>(TX, DV, [&](int, float (&v)[16]) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] *= g2L;
                });
                x.template rmw_row<D>(T4, DV, [&](int, float (&v)[16]) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] *= gL;
                });
            }
        }
        if (!x.wait_tma()) return false;
        if (x.decay && !first)  // Qg = diag(g^tau) Q
            scaled_tile_copy<C, D>(x.sQ, x.sTQ, x.tid, [&](int r) { return x.gp(r + 1); });
        x.publish();
        if (x.tid == 0) x.mma_kk(TW, x.sQ, x.sK, C, D, false);  // A = Q K^T
        x.commit();
        if (!x.wait_mma()) return false;
        // A-tilde = tril(Gamma1 o A)
        x.template for_row<C>(TW, C, [&](int c0, float (&v)[16]) {
            if (rowC < 0) return;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int a = c0 + i;
                v[i] = a <= rowC ? v[i] * x.gp(rowC - a) : 0.f;
            }
            tile_store_row16(x.sTA, C, rowC, c0, v);
        });
        x.publish();
        if (x.tid == 0) {
            if (!first) x.mma_kk(TW, x.decay ? x.sTQ : x.sQ, x.sTS, D, D, false);  // Qg S_p
            x.mma_km(TW, x.sTA, x.sK, D, C, !first);                               // + A-tilde K
        }
        x.commit();
        if (!x.wait_mma()) return false;
        // U (weighted by w^2 for the X update); K_w, V_w copies for decay
        x.template for_row<C>(TW, D, [&](int c0, float (&v)[16]) {
            if (rowC < 0) return;
            if (x.decay) {
                const float w2 = rowC < L ? x.gp(2 * (L - 1 - rowC)) : 0.f;
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] *= w2;
            }
            tile_store_row16(x.sTU, C, rowC, c0, v);
        });
        if (x.decay) {
            auto w = [&](int r) { return r < L ? x.gp(L - 1 - r) : 0.f; };
            scaled_tile_copy<C, D>(x.sK, x.sTA, x.tid, w);
            scaled_tile_copy<C, DV>(x.sV, x.sTS, x.tid, w);
        }
        x.publish();
        if (x.tid == 0) {
            x.mma_mm(TS, x.sK, x.decay ? x.sTA : x.sK, D, !first);   // S += K^T W K
            x.mma_mm(TX, x.sTU, x.sV, DV, !first);                    // X += (W^2 U)^T V
            x.mma_mm(T4, x.sQ, x.decay ? x.sTS : x.sV, DV, !first);  // C += Q^T W V
        }
        x.commit();
        // m and Y (CUDA cores, overlapping the MMAs)
        {
            const float gL = x.gp(L), g2L = x.gp(2 * L);
            for (int i = x.tid; i < D; i += kThreads) {
                float am = 0.f, ay = 0.f;
                for (int b = 0; b < L; ++b) {
                    am += x.gp(L - 1 - b) * tile_load(x.sQ, C, b, i);
                    ay += tile_load(x.sTU, C, b, i);
                }
                x.mrun[i] = gL * x.mrun[i] + am;
                x.Yrun[i] = g2L * x.Yrun[i] + ay;
            }
        }
        if (!x.wait_mma()) return false;
    }
    return true;
}

// Write the TMEM/SMEM summary (S, X, C, m, Y) of this CTA to `dst`.
template <int C, int D, int DV>
__device__ void store_summary(Ctx<C, D, DV> &x, float *dst) {
    const int rowD = owned_row<D>(x.tid);
    float *S = dst, *X = S + D * D, *Cc = X + D * DV, *m = Cc + D * DV, *Y = m + D;
    x.template for_row<D>(TS, D, [&](int c0, float (&v)[16]) {
        if (rowD >= 0)
#pragma unroll
            for (int i = 0; i < 16; i += 4)
                *reinterpret_cast<float4 *>(S + rowD * D + c0 + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
    });
    x.template for_row<D>(TX, DV, [&](int c0, float (&v)[16]) {
        if (rowD >= 0)
#pragma unroll
            for (int i = 0; i < 16; i += 4)
                *reinterpret_cast<float4 *>(X + rowD * DV + c0 + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
    });
    x.template for_row<D>(T4, DV, [&](int c0, float (&v)[16]) {
        if (rowD >= 0)
#pragma unroll
            for (int i = 0; i < 16; i += 4)
                *reinterpret_cast<float4 *>(Cc + rowD * DV + c0 + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
    });
    for (int i = x.tid; i < D; i += kThreads) { m[i] = x.mrun[i]; Y[i] = x.Yrun[i]; }
}

__device__ __forceinline__ float4 ldcg4(const float *p) { return __ldcg(reinterpret_cast<const float4 *>(p)); }

// ============================================================================ scan
// Initialise the prefix (TMEM S, X, C; mrun, Yrun) from state_in or zeros.
template <int C, int D, int DV>
__device__ bool prefix_init(Ctx<C, D, DV> &x) {
    const TcParams &P = *x.P;
    const int rowD = owned_row<D>(x.tid);
    if (!P.sin.S) {
        x.template zero_slot<D>(TS, D);
        x.template zero_slot<D>(TX, DV);
        x.template zero_slot<D>(T4, DV);
        for (int i = x.tid; i < D; i += kThreads) x.mrun[i] = x.Yrun[i] = 0.f;
        x.publish();
        return true;
    }
    const float *Si = P.sin.S + (size_t)x.bh * D * D, *Ci = P.sin.C + (size_t)x.bh * D * DV;
    const float *mi = P.sin.m + (size_t)x.bh * D, *Gi = P.sin.G + (size_t)x.bh * D * DV,
                *hi = P.sin.h + (size_t)x.bh * D;
    for (int i = x.tid; i < D; i += kThreads) x.mrun[i] = mi[i];
    __syncthreads();
    // S -> TMEM and hi/lo A operand; Y = S m - h
    float sm = 0.f;
    x.template rmw_row<D>(TS, D, [&](int c0, float (&v)[16]) {
        if (rowD < 0) return;
#pragma unroll
        for (int i = 0; i < 16; ++i) { v[i] = Si[rowD * D + c0 + i]; sm += v[i] * x.mrun[c0 + i]; }
        store_hilo(x.sShi, x.sSlo, D, rowD, c0, v);
    });
    x.template rmw_row<D>(T4, DV, [&](int c0, float (&v)[16]) {
        if (rowD < 0) return;
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = Ci[rowD * DV + c0 + i];
        store_hilo(x.sChi, x.sClo, D, rowD, c0, v);
    });
    if (rowD >= 0) x.Yrun[rowD] = sm - hi[rowD];
    x.publish();
    if (x.tid == 0) {  // X = S C (three bf16 products approximate fp32)
        x.mma_ss(TX, x.sShi, x.sChi, false);
        x.mma_ss(TX, x.sShi, x.sClo, true);
        x.mma_ss(TX, x.sSlo, x.sChi, true);
    }
    x.commit();
    if (!x.wait_mma()) return false;
    x.template rmw_row<D>(TX, DV, [&](int c0, float (&v)[16]) {
        if (rowD < 0) return;
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] -= Gi[rowD * DV + c0 + i];
    });
    x.publish();
    return true;
}

// prefix <- prefix (+) L, with L a summary (S, X, C, m, Y) and f = g^{len L}.
template <int C, int D, int DV>
__device__ bool fold(Ctx<C, D, DV> &x, const float *Lsum, float f) {
    const int rowD = owned_row<D>(x.tid);
    const float *SL = Lsum, *XL = SL + D * D, *CL = XL + D * DV, *mL = CL + D * DV, *YL = mL + D;
    const float f2 = f * f;
    for (int i = x.tid; i < D; i += kThreads) x.mL[i] = __ldcg(mL + i);
    __syncthreads();
    // S_P -> hi/lo operand; S_P m_L; S <- f S_P + S_L
    float sm = 0.f;
    x.template rmw_row<D>(TS, D, [&](int c0, float (&v)[16]) {
        if (rowD < 0) return;
        store_hilo(x.sShi, x.sSlo, D, rowD, c0, v);
#pragma unroll
        for (int i = 0; i < 16; i += 4) {
            const float4 s = ldcg4(SL + rowD * D + c0 + i);
            sm += v[i] * x.mL[c0 + i] + v[i + 1] * x.mL[c0 + i + 1] + v[i + 2] * x.mL[c0 + i + 2] +
                  v[i + 3] * x.mL[c0 + i + 3];
            v[i] = f * v[i] + s.x; v[i + 1] = f * v[i + 1] + s.y;
            v[i + 2] = f * v[i + 2] + s.z; v[i + 3] = f * v[i + 3] + s.w;
        }
    });
    // X <- f^2 X_P + X_L (the cross term is accumulated by the MMA below)
    x.template rmw_row<D>(TX, DV, [&](int c0, float (&v)[16]) {
        if (rowD < 0) return;
#pragma unroll
        for (int i = 0; i < 16; i += 4) {
            const float4 s = ldcg4(XL + rowD * DV + c0 + i);
            v[i] = f2 * v[i] + s.x; v[i + 1] = f2 * v[i + 1] + s.y;
            v[i + 2] = f2 * v[i + 2] + s.z; v[i + 3] = f2 * v[i + 3] + s.w;
        }
    });
    // C <- f C_P + C_L, and f C_L -> hi/lo operand
    x.template rmw_row<D>(T4, DV, [&](int c0, float (&v)[16]) {
        if (rowD < 0) return;
        float cl[16];
#pragma unroll
        for (int i = 0; i < 16; i += 4) {
            const float4 s = ldcg4(CL + rowD * DV + c0 + i);
            cl[i] = f * s.x; cl[i + 1] = f * s.y; cl[i + 2] = f * s.z; cl[i + 3] = f * s.w;
            v[i] = f * v[i] + s.x; v[i + 1] = f * v[i + 1] + s.y;
            v[i + 2] = f * v[i + 2] + s.z; v[i + 3] = f * v[i + 3] + s.w;
        }
        store_hilo(x.sChi, x.sClo, D, rowD, c0, cl);
    });
    if (rowD >= 0) x.tmp[rowD] = sm;
    x.publish();
    if (x.tid == 0) {  // X += S_P (f C_L)
        x.mma_ss(TX, x.sShi, x.sChi, true);
        x.mma_ss(TX, x.sShi, x.sClo, true);
        x.mma_ss(TX, x.sSlo, x.sChi, true);
    }
    x.commit();
    for (int i = x.tid; i < D; i += kThreads) {
        x.Yrun[i] = f2 * x.Yrun[i] + __ldcg(YL + i) + f * x.tmp[i];
        x.mrun[i] = f * x.mrun[i] + x.mL[i];
    }
    return x.wait_mma();
}

// Spin (bounded) until segment j of this sequence has published its summary.
template <int C, int D, int DV>
__device__ bool wait_flag(Ctx<C, D, DV> &x, int j) {
    bool ok = true;
    if (x.tid == 0) {
        const unsigned *f = x.P->flagsw + (size_t)x.bh * x.P->nseg + j;
        ok = false;
        for (uint32_t it = 0; it < kWaitLimit; ++it) {
            unsigned v;
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
            if (v) { ok = true; break; }
            __nanosleep(128);
        }
        if (!ok) atomicOr(x.P->err, DEV_TIMEOUT);
    }
    return !__syncthreads_or(!ok);
}

// ============================================================================ export
// state_out from the prefix in TMEM (S, X, C, m, Y): G = S C - X, h = S m - Y.
template <int C, int D, int DV>
__device__ bool export_state(Ctx<C, D, DV> &x) {
    const TcParams &P = *x.P;
    const int rowD = owned_row<D>(x.tid);
    float *So = P.sout.S + (size_t)x.bh * D * D, *Co = P.sout.C + (size_t)x.bh * D * DV;
    float *mo = P.sout.m + (size_t)x.bh * D, *Go = P.sout.G + (size_t)x.bh * D * DV, *ho = P.sout.h + (size_t)x.bh * D;
    float sm = 0.f;
    x.template for_row<D>(TS, D, [&](int c0, float (&v)[16]) {
        if (rowD < 0) return;
        store_hilo(x.sShi, x.sSlo, D, rowD, c0, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) { So[rowD * D + c0 + i] = v[i]; sm += v[i] * x.mrun[c0 + i]; }
    });
    x.template for_row<D>(T4, DV, [&](int c0, float (&v)[16]) {
        if (rowD < 0) return;
        store_hilo(x.sChi, x.sClo, D, rowD, c0, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) Co[rowD * DV + c0 + i] = v[i];
    });
    if (rowD >= 0) ho[rowD] = sm - x.Yrun[rowD];
    for (int i = x.tid; i < D; i += kThreads) mo[i] = x.mrun[i];
    x.publish();
    if (x.tid == 0) {  // W = S C
        x.mma_ss(TW, x.sShi, x.sChi, false);
        x.mma_ss(TW, x.sShi, x.sClo, true);
        x.mma_ss(TW, x.sSlo, x.sChi, true);
    }
    x.commit();
    if (!x.wait_mma()) return false;
    float xv[16];
    x.template for_row<D>(TW, DV, [&](int c0, float (&v)[16]) {
        tmem_ld16(x.taddr(TX, c0), xv);
        tmem_wait_ld();
        if (rowD < 0) return;
#pragma unroll
        for (int i = 0; i < 16; ++i) Go[rowD * DV + c0 + i] = v[i] - xv[i];
    });
    return true;
}

// Save / restore the parts of the prefix that pass 2 needs (S, X, m, Y).
template <int C, int D, int DV>
__device__ void save_prefix(Ctx<C, D, DV> &x, float *sv) {
    const int rowD = owned_row<D>(x.tid);
    float *S = sv, *X = S + D * D, *m = X + D * DV, *Y = m + D;
    x.template for_row<D>(TS, D, [&](int c0, float (&v)[16]) {
        if (rowD >= 0)
#pragma unroll
            for (int i = 0; i < 16; ++i) S[rowD * D + c0 + i] = v[i];
    });
    x.template for_row<D>(TX, DV, [&](int c0, float (&v)[16]) {
        if (rowD >= 0)
#pragma unroll
            for (int i = 0; i < 16; ++i) X[rowD * DV + c0 + i] = v[i];
    });
    for (int i = x.tid; i < D; i += kThreads) { m[i] = x.mrun[i]; Y[i] = x.Yrun[i]; }
}
template <int C, int D, int DV>
__device__ void restore_prefix(Ctx<C, D, DV> &x, const float *sv) {
    const int rowD = owned_row<D>(x.tid);
    const float *S = sv, *X = S + D * D, *m = X + D * DV, *Y = m + D;
    __syncthreads();
    x.template rmw_row<D>(TS, D, [&](int c0, float (&v)[16]) {
        if (rowD >= 0)
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = S[rowD * D + c0 + i];
    });
    x.template rmw_row<D>(TX, DV, [&](int c0, float (&v)[16]) {
        if (rowD >= 0)
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = X[rowD * DV + c0 + i];
    });
    for (int i = x.tid; i < D; i += kThreads) { x.mrun[i] = m[i]; x.Yrun[i] = Y[i]; }
}

// ============================================================================ pass 2
template <int C, int D, int DV>
__device__ bool pass2(Ctx<C, D, DV> &x, int jb, int je) {
    const TcParams &P = *x.P;
    const int rowC = owned_row<C>(x.tid);
    const int rowD = owned_row<D>(x.tid);
    __nv_bfloat16 *O = static_cast<__nv_bfloat16 *>(P.o) + (size_t)x.bh * P.n * DV;
    for (int jj = jb; jj < je; ++jj) {
        const int t0 = jj * C;
        const int L = min(C, P.n - t0);
        x.tma_chunk(jj);
        // state at the chunk start -> bf16 operands; then decay it to the chunk end
        {
            const float gL = x.gp(L), g2L = x.gp(2 * L);
            x.template rmw_row<D>(TS, D, [&](int c0, float (&v)[16]) {
                if (rowD >= 0) tile_store_row16(x.sTS, D, rowD, c0, v);
                if (x.decay)
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] *= gL;
            });
            x.template rmw_row<D>(TX, DV, [&](int c0, float (&v)[16]) {
                if (rowD >= 0) tile_store_row16(x.sTQ, D, rowD, c0, v);
                if (x.decay)
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] *= g2L;
            });
        }
        // den contribution q_t . Y_p, taken before Y moves on
        float qy = 0.f;
        if (!x.wait_tma()) return false;
        if (x.norm && rowC >= 0)
            for (int i = 0; i < D; ++i) qy += tile_load(x.sQ, C, rowC, i) * x.Yrun[i];
        x.publish();
        if (x.tid == 0) x.mma_kk(TW, x.sQ, x.sK, C, D, false);  // A = Q K^T
        x.commit();
        if (!x.wait_mma()) return false;
        x.template for_row<C>(TW, C, [&](int c0, float (&v)[16]) {
            if (rowC < 0) return;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int a = c0 + i;
                v[i] = a <= rowC ? v[i] * x.gp(rowC - a) : 0.f;
            }
            tile_store_row16(x.sTA, C, rowC, c0, v);
        });
        x.publish();
        if (x.tid == 0) {
            if (x.decay) {
                x.mma_kk(T4, x.sQ, x.sTS, D, D, false);  // spare = Q S_p
                x.mma_km(TW, x.sTA, x.sK, D, C, false);  // W = A-tilde K
            } else {
                x.mma_kk(TW, x.sQ, x.sTS, D, D, false);
                x.mma_km(TW, x.sTA, x.sK, D, C, true);
            }
        }
        x.commit();
        if (!x.wait_mma()) return false;
        // U = g^tau Q S_p + A-tilde K
        {
            float sp[16];
            x.template for_row<C>(TW, D, [&](int c0, float (&v)[16]) {
                if (x.decay) {
                    tmem_ld16(x.taddr(T4, c0), sp);
                    tmem_wait_ld();
                }
                if (rowC < 0) return;
                if (x.decay) {
                    const float gt = x.gp(rowC + 1);
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] += gt * sp[i];
                }
                tile_store_row16(x.sTU, C, rowC, c0, v);
                if (x.decay) {
                    const float w2 = rowC < L ? x.gp(2 * (L - 1 - rowC)) : 0.f;
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] *= w2;
                    tile_store_row16(x.sTS, C, rowC, c0, v);  // W^2 U
                }
            });
        }
        if (x.decay) scaled_tile_copy<C, D>(x.sK, x.sTA, x.tid, [&](int r) { return r < L ? x.gp(L - 1 - r) : 0.f; });
        x.publish();
        if (x.tid == 0) {
            x.mma_kk(TW, x.sQ, x.sTU, C, D, false);                 // M = Q U^T
            x.mma_mm(TX, x.decay ? x.sTS : x.sTU, x.sV, DV, true);  // X += (W^2 U)^T V
            x.mma_mm(TS, x.sK, x.decay ? x.sTA : x.sK, D, true);    // S += K^T W K
            if (x.decay) x.mma_km(T4, x.sQ, x.sTQ, DV, D, false);   // spare = Q X_p
        }
        x.commit();
        if (!x.wait_mma()) return false;
        float rs = 0.f;
        x.template for_row<C>(TW, C, [&](int c0, float (&v)[16]) {
            if (rowC < 0) return;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int b = c0 + i;
                v[i] = b <= rowC ? v[i] * x.gp(2 * (rowC - b)) : 0.f;
                rs += v[i];
            }
            tile_store_row16(x.sTA, C, rowC, c0, v);
        });
        x.publish();
        if (x.tid == 0) {
            x.mma_km(TW, x.sTA, x.sV, DV, C, false);                  // O = M V
            if (!x.decay) x.mma_km(TW, x.sQ, x.sTQ, DV, D, true);     // + Q X_p
        }
        x.commit();
        if (!x.wait_mma()) return false;
        {
            const float g2t = rowC >= 0 ? x.gp(2 * (rowC + 1)) : 0.f;
            float inv = 1.f;
            if (x.norm && rowC >= 0) inv = 1.f / (rs + g2t * qy + P.eps);
            float sp[16];
            x.template for_row<C>(TW, DV, [&](int c0, float (&v)[16]) {
                if (x.decay) {
                    tmem_ld16(x.taddr(T4, c0), sp);
                    tmem_wait_ld();
                }
                if (rowC < 0 || rowC >= L) return;
                if (x.decay)
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] += g2t * sp[i];
                if (x.norm)
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] *= inv;
                uint4 a, b;
                a.x = pack_bf16(v[0], v[1]); a.y = pack_bf16(v[2], v[3]);
                a.z = pack_bf16(v[4], v[5]); a.w = pack_bf16(v[6], v[7]);
                b.x = pack_bf16(v[8], v[9]); b.y = pack_bf16(v[10], v[11]);
                b.z = pack_bf16(v[12], v[13]); b.w = pack_bf16(v[14], v[15]);
                uint4 *dst = reinterpret_cast<uint4 *>(O + (size_t)(t0 + rowC) * DV + c0);
                dst[0] = a;
                dst[1] = b;
            });
        }
        if (x.norm) {  // Y <- g^{2L} Y + sum_b w_b^2 u_b
            __syncthreads();
            const float g2L = x.gp(2 * L);
            for (int i = x.tid; i < D; i += kThreads) {
                float ay = 0.f;
                for (int b = 0; b < L; ++b) ay += x.decay ? tile_load(x.sTS, C, b, i) : tile_load(x.sTU, C, b, i);
                x.Yrun[i] = g2L * x.Yrun[i] + ay;
            }
        }
        __syncthreads();
    }
    return true;
}

// ============================================================================ kernel
// The last CTA to finish returns the workspace header and flags to zero, so the
// next call needs no separate clearing launch.  Every CTA counts itself done
// only after its last read of a flag.  Called by one thread per CTA.
__device__ void finish_cta(const TcParams &P) {
    __threadfence();
    const unsigned done = atomicAdd(P.ticket + 1, 1u);
    if (done == gridDim.x - 1) {
        for (int i = 0; i < P.BH * P.nseg; ++i) P.flagsw[i] = 0u;
        P.ticket[0] = 0u;
        P.ticket[1] = 0u;
        __threadfence();
    }
}

template <int C, int D, int DV>
__global__ void __launch_bounds__(kThreads, 1) fwd_tc_kernel(const __grid_constant__ TcParams P) {
    using K_ = Cfg<C, D, DV>;
    // No static shared memory: the dynamic block starts at the (1024-byte
    // aligned) base of the CTA's shared window, which the swizzled tiles need.
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *base = smem_raw;
    uint64_t *bars = reinterpret_cast<uint64_t *>(base + K_::OFF_BAR);
    uint32_t *tmem_base_p = reinterpret_cast<uint32_t *>(base + K_::OFF_BAR + 16);
    int *ticket_p = reinterpret_cast<int *>(base + K_::OFF_BAR + 20);
    int *misalign_p = reinterpret_cast<int *>(base + K_::OFF_BAR + 24);

    Ctx<C, D, DV> x;
    x.P = &P;
    x.tid = threadIdx.x;
    x.warp = threadIdx.x >> 5;
    x.sQ = base + K_::OFF_Q; x.sK = base + K_::OFF_K; x.sV = base + K_::OFF_V;
    x.sTA = base + K_::OFF_TA; x.sTU = base + K_::OFF_TU; x.sTS = base + K_::OFF_TS; x.sTQ = base + K_::OFF_TQ;
    x.sShi = base + K_::OFF_SHI; x.sSlo = base + K_::OFF_SLO; x.sChi = base + K_::OFF_CHI; x.sClo = base + K_::OFF_CLO;
    float *vec = reinterpret_cast<float *>(base + K_::ARENA);
    x.mrun = vec; x.Yrun = vec + D; x.mL = vec + 2 * D; x.tmp = vec + 3 * D;
    x.tma_bar = &bars[0];
    x.mma_bar = &bars[1];
    x.tph = x.mph = 0;

    if (x.tid == 0) {
        *misalign_p = (smem_u32(base) & 1023u) != 0;
        mbar_init(x.tma_bar, 1);
        mbar_init(x.mma_bar, 1);
        fence_mbar_init();
        tma_prefetch_desc(&P.tmQ);
        tma_prefetch_desc(&P.tmK);
        tma_prefetch_desc(&P.tmV);
        *ticket_p = (int)atomicAdd(P.ticket, 1u);
    }
    __syncthreads();
    if (*misalign_p) {  // cannot happen with no static shared memory; refuse rather than corrupt
        if (x.tid == 0) {
            atomicOr(P.err, DEV_TIMEOUT);
            finish_cta(P);
        }
        return;
    }
    if (x.warp == 0) {
        tmem_alloc(tmem_base_p, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    x.tb = *tmem_base_p;
    const int ticket = *ticket_p;
    const int seg = ticket / P.BH;
    x.bh = ticket % P.BH;
    const int h = x.bh % P.H;
    x.decay = (P.flags & HLA_DECAY) != 0;
    x.norm = (P.flags & HLA_NORMALIZE) != 0;
    const float g = x.decay ? P.gamma[h] : 1.f;
    x.lg = log2f(g);

    const int jb = seg * P.cps;
    const int je = min(P.nchunks, jb + P.cps);
    const bool last = (seg == P.nseg - 1);
    const bool want_out = P.sout.S != nullptr;
    auto seg_len = [&](int s) {  // tokens in segment s
        const int b0 = s * P.cps * C;
        return min(P.n, (s + 1) * P.cps * C) - b0;
    };
    bool ok = true;
    do {
        // ---- pass 1: own summary (needed by later segments, and by the export)
        if (!last || want_out) {
            if (!(ok = pass1(x, jb, je))) break;
            store_summary(x, P.summ + ((size_t)x.bh * P.nseg + seg) * K_::SUM);
            __threadfence();
            __syncthreads();
            if (!last && x.tid == 0) {
                unsigned *f = P.flagsw + (size_t)x.bh * P.nseg + seg;
                asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(f), "r"(1u) : "memory");
            }
        }
        // ---- exclusive scan: prefix = state_in (+) L_0 (+) ... (+) L_{seg-1}
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (!(ok = prefix_init(x))) break;
        for (int j = 0; j < seg; ++j) {
            if (!(ok = wait_flag(x, j))) break;
            const float f = x.decay ? gpow(x.lg, (float)seg_len(j)) : 1.f;
            if (!(ok = fold(x, P.summ + ((size_t)x.bh * P.nseg + j) * K_::SUM, f))) break;
        }
        if (!ok) break;
        // ---- state export from prefix (+) own summary
        if (last && want_out) {
            float *sv = P.save + (size_t)x.bh * K_::SAVE;
            save_prefix(x, sv);
            __threadfence_block();
            const float f = x.decay ? gpow(x.lg, (float)seg_len(seg)) : 1.f;
            if (!(ok = fold(x, P.summ + ((size_t)x.bh * P.nseg + seg) * K_::SUM, f))) break;
            if (!(ok = export_state(x))) break;
            restore_prefix(x, sv);
            x.publish();
        }
        // ---- pass 2: outputs from the exact prefix
        if (!(ok = pass2(x, jb, je))) break;
    } while (0);

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (x.warp == 0) tmem_dealloc(x.tb, kTmemCols);
    if (x.tid == 0) finish_cta(P);
}

// ============================================================================ host side
PFN_cuTensorMapEncodeTiled_v12000 get_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

bool encode_3d(CUtensorMap *tm, const void *ptr, int width, int n, int BH, int box_rows) {
    auto enc = get_encoder();
    if (!enc) return false;
    cuuint64_t gdim[3] = {(cuuint64_t)width, (cuuint64_t)n, (cuuint64_t)BH};
    cuuint64_t gstr[2] = {(cuuint64_t)width * 2, (cuuint64_t)width * 2 * (cuuint64_t)n};
    cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), gdim, gstr, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct Plan {
    int nchunks, nseg, cps;
};
Plan make_plan(const hla_params &p, int num_sms) {
    Plan pl;
    const int BH = p.B * p.H;
    pl.nchunks = (p.n + p.chunk - 1) / p.chunk;
    int nseg = num_sms / (BH > 0 ? BH : 1);
    nseg = nseg < 1 ? 1 : nseg;
    if (nseg > pl.nchunks) nseg = pl.nchunks > 0 ? pl.nchunks : 1;
    pl.cps = (pl.nchunks + nseg - 1) / nseg;
    if (pl.cps < 1) pl.cps = 1;
    pl.nseg = (pl.nchunks + pl.cps - 1) / pl.cps;
    if (pl.nseg < 1) pl.nseg = 1;
    return pl;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct WsLayout {
    size_t off_flags, off_summ, off_save, total;
};
WsLayout ws_layout(const hla_params &p, const Plan &pl) {
    const size_t BH = (size_t)p.B * p.H;
    const size_t D = p.d, DV = p.dv;
    const size_t SUM = D * D + 2 * D * DV + 2 * D, SAVE = D * D + D * DV + 2 * D;
    WsLayout w;
    w.off_flags = 256;
    w.off_summ = align256(w.off_flags + BH * pl.nseg * 4);
    w.off_save = align256(w.off_summ + BH * pl.nseg * SUM * 4);
    w.total = align256(w.off_save + BH * SAVE * 4);
    return w;
}

template <int C, int D, int DV>
cudaError_t launch_cfg(const FwdArgs &a, cudaStream_t st, int num_sms) {
    using K_ = Cfg<C, D, DV>;
    hla_params p{a.B, a.H, a.n, a.d, a.dv, a.chunk, a.in_dtype, a.flags, a.eps, a.gamma};
    const Plan pl = make_plan(p, num_sms);
    const WsLayout wl = ws_layout(p, pl);
    TcParams P;
    memset(&P, 0, sizeof P);
    const int BH = a.B * a.H;
    if (!encode_3d(&P.tmQ, a.q, D, a.n, BH, C) || !encode_3d(&P.tmK, a.k, D, a.n, BH, C) ||
        !encode_3d(&P.tmV, a.v, DV, a.n, BH, C))
        return cudaErrorInvalidValue;
    P.B = a.B; P.H = a.H; P.n = a.n; P.BH = BH;
    P.nchunks = pl.nchunks; P.nseg = pl.nseg; P.cps = pl.cps;
    P.flags = a.flags; P.eps = a.eps; P.gamma = a.gamma;
    P.o = a.o; P.sin = a.sin; P.sout = a.sout;
    uint8_t *ws = static_cast<uint8_t *>(a.workspace);
    P.ticket = reinterpret_cast<unsigned *>(ws);
    P.flagsw = reinterpret_cast<unsigned *>(ws + wl.off_flags);
    P.summ = reinterpret_cast<float *>(ws + wl.off_summ);
    P.save = reinterpret_cast<float *>(ws + wl.off_save);
    P.err = a.err;
    auto kern = fwd_tc_kernel<C, D, DV>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, K_::SMEM_LAUNCH);
    if (e != cudaSuccess) return e;
    kern<<<BH * pl.nseg, kThreads, K_::SMEM_LAUNCH, st>>>(P);
    return cudaGetLastError();
}

template <int C, int D>
cudaError_t launch_dv(const FwdArgs &a, cudaStream_t st, int ns) {
    return a.dv == 64 ? launch_cfg<C, D, 64>(a, st, ns) : launch_cfg<C, D, 128>(a, st, ns);
}
template <int C>
cudaError_t launch_d(const FwdArgs &a, cudaStream_t st, int ns) {
    return a.d == 64 ? launch_dv<C, 64>(a, st, ns) : launch_dv<C, 128>(a, st, ns);
}

}  // namespace

bool fwd_tc_supported(const hla_params &p) {
    auto ok = [](int x) { return x == 64 || x == 128; };
    return p.in_dtype == HLA_BF16 && ok(p.d) && ok(p.dv) && ok(p.chunk);
}

size_t fwd_tc_workspace(const hla_params &p, int num_sms) {
    if (p.n == 0) return 0;
    return ws_layout(p, make_plan(p, num_sms)).total;
}

cudaError_t fwd_tc_launch(const FwdArgs &a, cudaStream_t st, int num_sms) {
    return a.chunk == 64 ? launch_d<64>(a, st, num_sms) : launch_d<128>(a, st, num_sms);
}

}  // namespace hla
