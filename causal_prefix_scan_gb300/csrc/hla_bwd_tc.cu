// hla_bwd_tc.cu -- tensor-core (tcgen05 MMA, TMEM accumulators) kernels for the
// chunk-local sums and the gradients of the backward pass, bf16 inputs,
// d = dv = chunk = 64, with or without decay.  The algebra is that of
// hla_bwd_simt.cuh (reverse mode of the masked recurrence, chunk form):
//   A~ = tril(G1 o Q K^T),  P = tril(G2 o G V^T),  U = diag(g^{tau+1}) Q S_p + A~ K,
//   dU = P^T Q + diag(g^{2(L-tau)}) V Lam^T,  B = tril(G1 o dU K^T),  M = tril(G2 o Q U^T),
//   dQ = P U + B K + diag(g^{2(tau+1)}) G X_p^T + diag(g^{tau+1}) dU S_p,
//   dK = A~^T dU + B^T Q + diag(g^{L-tau}) K (Om + Om^T),
//   dV = M^T G + diag(g^{2(L-tau)}) U Lam;
// local sums: S_loc = K^T W1 K, C_q = Q^T W2 V, X_loc = (A~K)^T W3 V, L_loc = Q^T W4 G,
// W = V^T W5 Q, O_loc = (P^T Q)^T W6 Q with the diagonal token weights W1..W6.
// Terms with different row scales go to separate accumulators and are combined in
// the epilogue; token weights of the local sums scale bf16 copies of the operands.
// The fp32 states enter as bf16 hi + lo pairs.  The scan between the two kernels
// stays on the CUDA cores (hla_bwd_simt.cuh).
#include "hla_bwd_simt.cuh"
#include "hla_chunk_tc.cuh"

namespace hla {
namespace bwdtc {
using bwd::BwdWs;
using namespace chunktc;
namespace {

constexpr int kGp = 2 * 64 + 4;  // g^x for x = 0 .. 2C

__device__ __forceinline__ void fill_gp(float *gp, const BwdArgs &a, int u) {
    const bool decay = (a.flags & HLA_DECAY) != 0;
    const float lg = log2f(decay ? a.gamma[u % a.H] : 1.f);
    for (int x = threadIdx.x; x < kGp; x += kTc) gp[x] = decay ? gpow(lg, (float)x) : 1.f;
}

// tiles of the local-sums kernel (the last four: weighted copies, with decay only)
enum { L_Q, L_K, L_V, L_G, L_A, L_P, L_UW, L_DUW, L_KW1, L_QW2, L_QW4, L_VW5, L_N };
// tiles of the gradient kernel; a tile is reused once its last reader has completed:
// V (stage 1) then dU, S_p hi (stages 1, 3) then M, S_p lo then (Om + Om^T) hi,
// X_p hi (stage 3) then B, X_p lo then (Om + Om^T) lo -- 13 tiles, two CTAs per SM
enum { G_Q, G_K, G_V, G_G, G_SH, G_SL, G_XH, G_XL, G_LH, G_LL, G_A, G_P, G_U, G_N };
constexpr int G_DU = G_V, G_M = G_SH, G_OH = G_SL, G_B = G_XH, G_OL = G_XL;

__global__ void __launch_bounds__(kTc, 2) bwd_local_tc_kernel(const __grid_constant__ BwdArgs a,
                                                                const __grid_constant__ ChunkMaps tm) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    Ctx x;
    if (!setup(x, smem_raw, L_N, a.err)) return;
    float *gp = reinterpret_cast<float *>(smem_raw + L_N * TILE + 64);
    float *w = gp + kGp;  // four token-weight vectors [64]
    const int nch = (a.n + 63) / 64, u = blockIdx.x / nch, ch = blockIdx.x % nch;
    const int t0 = ch * 64, L = min(64, a.n - t0);
    const bool decay = (a.flags & HLA_DECAY) != 0;
    {
        const CUtensorMap *m[4] = {&tm.q, &tm.k, &tm.v, &tm.g};
        const int kvu = (int)bwd::kv_unit(a, u), un[4] = {u, kvu, kvu, u};
        uint8_t *dst[4] = {x.tile(L_Q), x.tile(L_K), x.tile(L_V), x.tile(L_G)};
        tma_issue<4>(x, m, un, t0, dst);
    }
    fill_gp(gp, a, u);
    __syncthreads();
    if (decay) {  // token weights of the copies: g^{L-1-s} K, g^{2L-1-s} Q, g^{2s} Q, g^{2L-s} V
        for (int s = threadIdx.x; s < 64; s += kTc) {
            const bool in = s < L;
            w[s] = in ? gp[L - 1 - s] : 0.f;
            w[64 + s] = in ? gp[2 * L - 1 - s] : 0.f;
            w[128 + s] = in ? gp[2 * s] : 0.f;
            w[192 + s] = in ? gp[2 * L - s] : 0.f;
        }
    }
    const bool loaded = tma_wait(x);
    const uint8_t *kw1 = x.tile(L_K), *qw2 = x.tile(L_Q), *qw4 = x.tile(L_Q), *vw5 = x.tile(L_V);
    if (decay && loaded) {  // the weighted copies, from the tiles
        scale_tile(x.tile(L_K), L, w, x.tile(L_KW1));
        scale_tile(x.tile(L_Q), L, w + 64, x.tile(L_QW2));
        scale_tile(x.tile(L_Q), L, w + 128, x.tile(L_QW4));
        scale_tile(x.tile(L_V), L, w + 192, x.tile(L_VW5));
        kw1 = x.tile(L_KW1); qw2 = x.tile(L_QW2); qw4 = x.tile(L_QW4); vw5 = x.tile(L_VW5);
    }
    x.publish();
    const BwdWs ws{64, 64};
    float *out = a.workspace + ((size_t)u * nch + ch) * ws.loc_floats();
    const size_t ro = (size_t)x.row * 64 + x.c0;
    float r[16];
    do {
        if (!loaded) break;
        // A~ = Q K^T, P = G V^T
        if (x.tid == 0) {
            mma_kk(x.tb + 0, x.tile(L_Q), x.tile(L_K), false);
            mma_kk(x.tb + 64, x.tile(L_G), x.tile(L_V), false);
        }
        x.commit();
        if (!x.wait()) break;
        x.ld_row(0, r);
        store_tril_decay(x, x.tile(L_A), r, gp, 1);
        x.ld_row(64, r);
        store_tril_decay(x, x.tile(L_P), r, gp, 2);
        x.publish();
        // U = A~ K, dU = P^T Q (no earlier state or later adjoint)
        if (x.tid == 0) {
            mma_km(x.tb + 128, x.tile(L_A), x.tile(L_K), false);
            mma_mm(x.tb + 192, x.tile(L_P), x.tile(L_Q));
        }
        x.commit();
        if (!x.wait()) break;
        {  // weights of X_loc (g^{2(L-1-t)}) and O_loc (g^t) on the token rows of U and dU
            const bool in = x.row < L;
            const float w3 = in ? gp[2 * (L - 1 - x.row)] : 0.f, w6 = in ? gp[x.row] : 0.f;
            x.ld_row(128, r);
#pragma unroll
            for (int i = 0; i < 16; ++i) r[i] *= w3;
            tile_store_row16(x.tile(L_UW), 64, x.row, x.c0, r);
            x.ld_row(192, r);
#pragma unroll
            for (int i = 0; i < 16; ++i) r[i] *= w6;
            tile_store_row16(x.tile(L_DUW), 64, x.row, x.c0, r);
        }
        x.publish();
        // S_loc, C_q, X_loc, L_loc (rows = feature index)
        if (x.tid == 0) {
            mma_mm(x.tb + 0, kw1, x.tile(L_K));
            mma_mm(x.tb + 64, qw2, x.tile(L_V));
            mma_mm(x.tb + 128, x.tile(L_UW), x.tile(L_V));
            mma_mm(x.tb + 192, qw4, x.tile(L_G));
        }
        x.commit();
        if (!x.wait()) break;
        x.ld_row(0, r);
        st_row16(out + ws.o_sloc() + ro, r);
        x.ld_row(64, r);
        st_row16(out + ws.o_cq() + ro, r);
        x.ld_row(128, r);
        st_row16(out + ws.o_xloc() + ro, r);
        x.ld_row(192, r);
        st_row16(out + ws.o_lloc() + ro, r);
        x.publish();  // the reads of columns 0-127 precede their reuse
        // W (rows = value index), O_loc
        if (x.tid == 0) {
            mma_mm(x.tb + 0, vw5, x.tile(L_Q));
            mma_mm(x.tb + 64, x.tile(L_DUW), x.tile(L_Q));
        }
        x.commit();
        if (!x.wait()) break;
        x.ld_row(0, r);
        st_row16(out + ws.o_w() + ro, r);
        x.ld_row(64, r);
        st_row16(out + ws.o_oloc() + ro, r);
    } while (false);
    teardown(x);
}

// Om + Om^T (fp32, 64 x 64, row-major) into bf16 hi and lo tiles
__device__ __forceinline__ void load_sym_hilo(const float *src, uint8_t *hi, uint8_t *lo) {
    for (int e = threadIdx.x; e < 64 * 4; e += kTc) {
        const int r = e >> 2, c = (e & 3) * 16;
        float h[16], l[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float s = src[(size_t)r * 64 + c + i] + src[(size_t)(c + i) * 64 + r];
            h[i] = __bfloat162float(__float2bfloat16_rn(s));
            l[i] = s - h[i];
        }
        tile_store_row16(hi, 64, r, c, h);
        tile_store_row16(lo, 64, r, c, l);
    }
}

__global__ void __launch_bounds__(kTc, 2) bwd_grad_tc_kernel(const __grid_constant__ BwdArgs a,
                                                               const __grid_constant__ ChunkMaps tm) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    Ctx x;
    if (!setup(x, smem_raw, G_N, a.err)) return;
    float *gp = reinterpret_cast<float *>(smem_raw + G_N * TILE + 64);
    const int nch = (a.n + 63) / 64, u = blockIdx.x / nch, ch = blockIdx.x % nch;
    const int t0 = ch * 64, L = min(64, a.n - t0);
    const size_t r0 = ((size_t)u * a.n + t0) * 64;
    const BwdWs ws{64, 64};
    const float *so =
        a.workspace + (size_t)a.B * a.H * nch * ws.loc_floats() + ((size_t)u * nch + ch) * ws.st_floats();
    {  // the bf16 inputs by TMA while the threads convert the states
        const CUtensorMap *m[4] = {&tm.q, &tm.k, &tm.v, &tm.g};
        const int kvu = (int)bwd::kv_unit(a, u), un[4] = {u, kvu, kvu, u};
        uint8_t *dst[4] = {x.tile(G_Q), x.tile(G_K), x.tile(G_V), x.tile(G_G)};
        tma_issue<4>(x, m, un, t0, dst);
    }
    fill_gp(gp, a, u);
    {
        const float *ss[3] = {so + ws.o_sp(), so + ws.o_xp(), so + ws.o_lam()};
        uint8_t *hi[3] = {x.tile(G_SH), x.tile(G_XH), x.tile(G_LH)}, *lo[3] = {x.tile(G_SL), x.tile(G_XL), x.tile(G_LL)};
        load_tiles_hilo<3>(ss, hi, lo);
    }
    const bool loaded = tma_wait(x);
    x.publish();
    // row scales of this thread's token row t
    const int t = x.row;
    const bool in = t < L;
    const float r_u = gp[t + 1], r_x = gp[2 * (t + 1)];
    const float r_l2 = in ? gp[2 * (L - t)] : 0.f, r_l1 = in ? gp[L - t] : 0.f;
    const size_t ro = r0 + (size_t)t * 64 + x.c0;
    float r[16], s[16];
    do {
        if (!loaded) break;
        // stage 1: A~, P raw; Q S_p; V Lam^T
        if (x.tid == 0) {
            mma_kk(x.tb + 0, x.tile(G_Q), x.tile(G_K), false);
            mma_kk(x.tb + 64, x.tile(G_G), x.tile(G_V), false);
            mma_km(x.tb + 128, x.tile(G_Q), x.tile(G_SH), false);
            mma_km(x.tb + 128, x.tile(G_Q), x.tile(G_SL), true);
            mma_kk(x.tb + 192, x.tile(G_V), x.tile(G_LH), false);
            mma_kk(x.tb + 192, x.tile(G_V), x.tile(G_LL), true);
        }
        x.commit();
        if (!x.wait()) break;
        x.ld_row(0, r);
        store_tril_decay(x, x.tile(G_A), r, gp, 1);
        x.ld_row(64, r);
        store_tril_decay(x, x.tile(G_P), r, gp, 2);
        x.publish();
        // stage 2: A~ K, P^T Q
        if (x.tid == 0) {
            mma_km(x.tb + 0, x.tile(G_A), x.tile(G_K), false);
            mma_mm(x.tb + 64, x.tile(G_P), x.tile(G_Q));
        }
        x.commit();
        if (!x.wait()) break;
        // U = r_u (Q S_p) + A~ K;  dU = P^T Q + r_l2 (V Lam^T)
        x.ld_row(128, s);
        x.ld_row(0, r);
#pragma unroll
        for (int i = 0; i < 16; ++i) r[i] += r_u * s[i];
        tile_store_row16(x.tile(G_U), 64, t, x.c0, r);
        x.ld_row(192, s);
        x.ld_row(64, r);
#pragma unroll
        for (int i = 0; i < 16; ++i) r[i] += r_l2 * s[i];
        tile_store_row16(x.tile(G_DU), 64, t, x.c0, r);
        x.publish();
        // stage 3: B raw, M raw; G X_p^T; dU S_p
        if (x.tid == 0) {
            mma_kk(x.tb + 0, x.tile(G_DU), x.tile(G_K), false);
            mma_kk(x.tb + 64, x.tile(G_Q), x.tile(G_U), false);
            mma_kk(x.tb + 128, x.tile(G_G), x.tile(G_XH), false);
            mma_kk(x.tb + 128, x.tile(G_G), x.tile(G_XL), true);
            mma_km(x.tb + 192, x.tile(G_DU), x.tile(G_SH), false);
            mma_km(x.tb + 192, x.tile(G_DU), x.tile(G_SL), true);
        }
        x.commit();
        if (!x.wait()) break;
        x.ld_row(0, r);
        store_tril_decay(x, x.tile(G_B), r, gp, 1);
        x.ld_row(64, r);
        store_tril_decay(x, x.tile(G_M), r, gp, 2);
        x.publish();
        // stage 4: P U + B K;  A~^T dU + B^T Q; meanwhile Om + Om^T into the tiles of S_p lo
        // and X_p lo, whose readers (stage 3) are complete
        if (x.tid == 0) {
            mma_km(x.tb + 0, x.tile(G_P), x.tile(G_U), false);
            mma_km(x.tb + 0, x.tile(G_B), x.tile(G_K), true);
            mma_mm(x.tb + 64, x.tile(G_A), x.tile(G_DU));
            mma_mm(x.tb + 64, x.tile(G_B), x.tile(G_Q), true);
        }
        x.commit();
        load_sym_hilo(so + ws.o_om(), x.tile(G_OH), x.tile(G_OL));
        if (!x.wait()) break;
        // dQ = (P U + B K) + r_x (G X_p^T) + r_u (dU S_p)
        x.ld_row(0, r);
        x.ld_row(128, s);
#pragma unroll
        for (int i = 0; i < 16; ++i) r[i] += r_x * s[i];
        x.ld_row(192, s);
#pragma unroll
        for (int i = 0; i < 16; ++i) r[i] += r_u * s[i];
        if (in) st_row16_bf16(static_cast<__nv_bfloat16 *>(a.grad_q) + ro, r);
        x.publish();  // the reads of columns 0, 128, 192 precede their reuse
        // stage 5: K (Om + Om^T); M^T G; U Lam
        if (x.tid == 0) {
            mma_km(x.tb + 128, x.tile(G_K), x.tile(G_OH), false);
            mma_km(x.tb + 128, x.tile(G_K), x.tile(G_OL), true);
            mma_mm(x.tb + 0, x.tile(G_M), x.tile(G_G));
            mma_km(x.tb + 192, x.tile(G_U), x.tile(G_LH), false);
            mma_km(x.tb + 192, x.tile(G_U), x.tile(G_LL), true);
        }
        x.commit();
        if (!x.wait()) break;
        // dK = (A~^T dU + B^T Q) + r_l1 K (Om + Om^T);  dV = M^T G + r_l2 U Lam
        x.ld_row(64, r);
        x.ld_row(128, s);
#pragma unroll
        for (int i = 0; i < 16; ++i) r[i] += r_l1 * s[i];
        if (in) {  // per-query-head fp32 staging with shared key/value heads
            if (a.dk_pair) st_row16(a.dk_pair + ro, r);
            else st_row16_bf16(static_cast<__nv_bfloat16 *>(a.grad_k) + ro, r);
        }
        x.ld_row(0, r);
        x.ld_row(192, s);
#pragma unroll
        for (int i = 0; i < 16; ++i) r[i] += r_l2 * s[i];
        if (in) {
            if (a.dv_pair) st_row16(a.dv_pair + ro, r);
            else st_row16_bf16(static_cast<__nv_bfloat16 *>(a.grad_v) + ro, r);
        }
    } while (false);
    teardown(x);
}

constexpr size_t kLocalSmem = L_N * TILE + 64 + (kGp + 4 * 64) * 4;
constexpr size_t kGradSmem = G_N * TILE + 64 + kGp * 4;

}  // namespace

cudaError_t local_tc(const BwdArgs &a, cudaStream_t st) {
    cudaError_t e =
        cudaFuncSetAttribute(bwd_local_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kLocalSmem);
    if (e != cudaSuccess) return e;
    ChunkMaps m;
    if (!chunk_maps(m, a.q, a.k, a.v, a.go, a.n, a.B * a.H, a.B * a.Hkv)) return cudaErrorInvalidValue;
    bwd_local_tc_kernel<<<a.B * a.H * ((a.n + 63) / 64), kTc, kLocalSmem, st>>>(a, m);
    return cudaGetLastError();
}

cudaError_t grad_tc(const BwdArgs &a, cudaStream_t st) {
    cudaError_t e =
        cudaFuncSetAttribute(bwd_grad_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGradSmem);
    if (e != cudaSuccess) return e;
    ChunkMaps m;
    if (!chunk_maps(m, a.q, a.k, a.v, a.go, a.n, a.B * a.H, a.B * a.Hkv)) return cudaErrorInvalidValue;
    bwd_grad_tc_kernel<<<a.B * a.H * ((a.n + 63) / 64), kTc, kGradSmem, st>>>(a, m);
    return cudaGetLastError();
}

}  // namespace bwdtc
}  // namespace hla
