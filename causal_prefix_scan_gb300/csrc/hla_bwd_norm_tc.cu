// hla_bwd_norm_tc.cu -- the ratio-normalised backward pass on the tensor cores: bf16
// inputs, d = dv = chunk = 64, with or without decay, zero initial state
// ("Higher-order Linear Attention", gist.science summary, section 1, bullet
// "Normalisatie"; chunk form of hla_bwd_simt.cuh).
//
// The normalised output o_t = n_t r_t, r_t = 1 / (den_t + eps), is the unnormalised
// output of the values [V | 1] divided by its last column, so its gradient is the
// unnormalised gradient of [V | 1] under the upstream [A | -c] with A_t = r_t g_t and
// c_t = r_t (g_t . o_t).  Where the two columns meet -- every contraction over the value
// index -- the two parts cancel to a large degree (the parts of dk are several times
// their sum), so those products are formed to about fp32 accuracy:
//   P = A V^T - c 1^T          A as bf16 hi + lo (V is exact), c subtracted in fp32;
//   V Lam^T + 1 lam^T          Lam as hi + lo, the unit column's adjoint lam added in fp32;
//   A X_p^T - c Y_p^T          A and X_p as hi + lo (three products), c Y_p^T in fp32;
//   Lam W + lam w^T            (the increments of Om) Lam and W as hi + lo, lam w^T in fp32;
// and the token side of every sum over tokens that feeds both columns is rounded once
// and shared by both (C_q and m_q from one weighted Q tile, X_loc and Y_loc from one
// weighted U tile, L_loc and lam_loc from one weighted Q, W and w from another), so a
// rounding there scales the combined term and is not amplified by the cancellation.
// The unit column itself never enters an MMA: its sums (m_q, Y, lam, w) are d-vectors
// on the CUDA cores.
//
// Launches (units = B*H pairs, one CTA per chunk unless noted):
//   1. fwd_local:  A~, U_loc = A~K; S_loc, C_q, X_loc and m_q, Y_loc;
//   2. prefix:     S_p (factor g^L);
//   3. fwd_incr:   X_loc <- S_p C_q + X_loc, Y_loc <- S_p m_q + Y_loc;
//   4. prefix:     X_p, Y_p (g^{2L});
//   5. out_local:  the outputs n, den of the chunk from S_p, X_p, Y_p (U, M as in the
//                  forward), r and c per token; then P, dU_loc and the backward local
//                  sums L_loc, W, O_loc and lam_loc, w;
//   6. prefix:     Lam_n, lam_n (suffix, g^{2L});
//   7. bwd_incr:   O_loc <- O_loc + Lam_n W + lam_n w^T;
//   8. prefix:     Om_n (suffix, g^L);
//   9. grad:       dq, dk, dv (the five stages of the unnormalised gradient kernel with
//                  the mixed terms above).
#include <cstdio>

#include "hla_bwd_simt.cuh"
#include "hla_chunk_tc.cuh"

namespace hla {
namespace bwdn {
using namespace chunktc;
namespace {

constexpr int kGp = 2 * 64 + 4;  // g^x for x = 0 .. 2C

// Workspace (floats): per chunk the local sums, then per chunk the states, then r and c
// per token, then (shared key/value heads) the per-query-head fp32 dk and dv.
struct NWs {
    static constexpr size_t M = 64 * 64, V = 64;
    // local sums: S_loc, C_q, X_loc, L_loc, W (rows = value index), O_loc; m_q, Y_loc, lam_loc, w
    static constexpr size_t L_SLOC = 0, L_CQ = M, L_XLOC = 2 * M, L_LLOC = 3 * M, L_W = 4 * M, L_OLOC = 5 * M,
                            L_MQ = 6 * M, L_YLOC = L_MQ + V, L_LAM = L_YLOC + V, L_WV = L_LAM + V, LOC = L_WV + V;
    // states: S_p, X_p (before the chunk), Lam_n, Om_n (after it); Y_p, lam_n
    static constexpr size_t S_SP = 0, S_XP = M, S_LAM = 2 * M, S_OM = 3 * M, S_YP = 4 * M, S_LN = S_YP + V,
                            ST = S_LN + V;
};

struct Lay {
    size_t loc, st, r, c, dk_pair, dv_pair, total;  // float offsets
};
Lay layout(int B, int H, int Hkv, int n) {
    const size_t units = (size_t)B * H, nch = ((size_t)n + 63) / 64, toks = units * n;
    Lay l;
    l.loc = 0;
    l.st = units * nch * NWs::LOC;
    l.r = l.st + units * nch * NWs::ST;
    l.c = l.r + toks;
    l.dk_pair = l.c + toks;
    const bool shared = Hkv < H;
    l.dv_pair = l.dk_pair + (shared ? toks * 64 : 0);
    l.total = l.dv_pair + (shared ? toks * 64 : 0);
    return l;
}

struct Ptrs {  // the workspace regions of one launch
    float *loc, *st, *r, *c;
};
__device__ __forceinline__ Ptrs regions(const BwdArgs &a) {
    const size_t units = (size_t)a.B * a.H, nch = ((size_t)a.n + 63) / 64, toks = units * a.n;
    Ptrs p;
    p.loc = a.workspace;
    p.st = p.loc + units * nch * NWs::LOC;
    p.r = p.st + units * nch * NWs::ST;
    p.c = p.r + toks;
    return p;
}

__device__ __forceinline__ void fill_gp(float *gp, const BwdArgs &a, int u) {
    const bool decay = (a.flags & HLA_DECAY) != 0;
    const float lg = log2f(decay ? a.gamma[u % a.H] : 1.f);
    for (int x = threadIdx.x; x < kGp; x += kTc) gp[x] = decay ? gpow(lg, (float)x) : 1.f;
}

// D (+)= A B with A, B fp32 given as hi + lo tiles: hi.hi + hi.lo + lo.hi
__device__ __forceinline__ void mma3_km(uint32_t d, const uint8_t *ah, const uint8_t *al, const uint8_t *bh,
                                        const uint8_t *bl, bool acc) {
    mma_km(d, ah, bh, acc);
    mma_km(d, ah, bl, true);
    mma_km(d, al, bh, true);
}

// 16 fp32 values into bf16 hi and lo rows of two tiles
__device__ __forceinline__ void store_hilo16(uint8_t *hi, uint8_t *lo, int r, int c0, const float (&v)[16]) {
    float h[16], l[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        h[i] = __bfloat162float(__float2bfloat16_rn(v[i]));
        l[i] = v[i] - h[i];
    }
    tile_store_row16(hi, 64, r, c0, h);
    tile_store_row16(lo, 64, r, c0, l);
}

// A bf16 tile (rows r >= L zero) with row r scaled by s[r], in place as the hi part and
// into `lo` as the rest: each thread rewrites only the elements it read.
__device__ __forceinline__ void rowscale_hilo_inplace(uint8_t *hi, uint8_t *lo, const float *s, int L) {
    for (int e = threadIdx.x; e < 64 * 4; e += kTc) {
        const int r = e >> 2, c = (e & 3) * 16;
        const float w = r < L ? s[r] : 0.f;
        float a[8], b[8], v[16];
        tile_load_row8(hi, 64, r, c, a);
        tile_load_row8(hi, 64, r, c + 8, b);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            v[i] = w * a[i];
            v[8 + i] = w * b[i];
        }
        store_hilo16(hi, lo, r, c, v);
    }
}

// Om + Om^T (fp32, 64 x 64, row-major) into bf16 hi and lo tiles
__device__ __forceinline__ void load_sym_hilo(const float *src, uint8_t *hi, uint8_t *lo) {
    for (int e = threadIdx.x; e < 64 * 4; e += kTc) {
        const int r = e >> 2, c = (e & 3) * 16;
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = src[(size_t)r * 64 + c + i] + src[(size_t)(c + i) * 64 + r];
        store_hilo16(hi, lo, r, c, v);
    }
}

// Column sums of a bf16 tile over its 64 rows, optionally weighted per row (fp32):
// out[i] = sum_s w[s] T[s][i] for i = the calling thread's index (threads 0..63).
__device__ __forceinline__ float tile_colsum(const uint8_t *tile, int i, const float *w) {
    float acc = 0.f;
    for (int s = 0; s < 64; ++s) {
        const float x = tile_load(tile, 64, s, i);
        acc = w ? fmaf(w[s], x, acc) : acc + x;
    }
    return acc;
}

// ======================================================================= 1. fwd_local
enum { F_Q, F_K, F_V, F_A, F_UW, F_KW1, F_QW2, F_N };

__global__ void __launch_bounds__(kTc, 2) fwd_local_kernel(const __grid_constant__ BwdArgs a,
                                                             const __grid_constant__ ChunkMaps tm) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    Ctx x;
    if (!setup(x, smem_raw, F_N, a.err)) return;
    float *gp = reinterpret_cast<float *>(smem_raw + F_N * TILE + 64);
    float *w = gp + kGp;  // two token-weight vectors [64]
    const int nch = (a.n + 63) / 64, u = blockIdx.x / nch, ch = blockIdx.x % nch;
    const int t0 = ch * 64, L = min(64, a.n - t0);
    const bool decay = (a.flags & HLA_DECAY) != 0;
    {
        const CUtensorMap *m[3] = {&tm.q, &tm.k, &tm.v};
        const int kvu = (int)bwd::kv_unit(a, u), un[3] = {u, kvu, kvu};
        uint8_t *dst[3] = {x.tile(F_Q), x.tile(F_K), x.tile(F_V)};
        tma_issue<3>(x, m, un, t0, dst);
    }
    fill_gp(gp, a, u);
    __syncthreads();
    if (decay) {  // token weights of the copies: g^{L-1-s} K, g^{2L-1-s} Q
        for (int s = threadIdx.x; s < 64; s += kTc) {
            w[s] = s < L ? gp[L - 1 - s] : 0.f;
            w[64 + s] = s < L ? gp[2 * L - 1 - s] : 0.f;
        }
    }
    const bool loaded = tma_wait(x);
    const uint8_t *kw1 = x.tile(F_K), *qw2 = x.tile(F_Q);
    if (decay && loaded) {
        scale_tile(x.tile(F_K), L, w, x.tile(F_KW1));
        scale_tile(x.tile(F_Q), L, w + 64, x.tile(F_QW2));
        kw1 = x.tile(F_KW1);
        qw2 = x.tile(F_QW2);
    }
    x.publish();
    float *out = regions(a).loc + ((size_t)u * nch + ch) * NWs::LOC;
    const size_t ro = (size_t)x.row * 64 + x.c0;
    float r[16];
    do {
        if (!loaded) break;
        if (x.tid == 0) mma_kk(x.tb + 0, x.tile(F_Q), x.tile(F_K), false);  // Q K^T
        x.commit();
        if (!x.wait()) break;
        x.ld_row(0, r);
        store_tril_decay(x, x.tile(F_A), r, gp, 1);
        x.publish();
        if (x.tid == 0) mma_km(x.tb + 64, x.tile(F_A), x.tile(F_K), false);  // U_loc = A~ K
        x.commit();
        if (!x.wait()) break;
        {  // weight of X_loc and Y_loc on the token rows of U: g^{2(L-1-t)}
            const float w3 = x.row < L ? gp[2 * (L - 1 - x.row)] : 0.f;
            x.ld_row(64, r);
#pragma unroll
            for (int i = 0; i < 16; ++i) r[i] *= w3;
            tile_store_row16(x.tile(F_UW), 64, x.row, x.c0, r);
        }
        x.publish();
        if (x.tid == 0) {  // S_loc, C_q, X_loc (rows = feature index)
            mma_mm(x.tb + 0, kw1, x.tile(F_K));
            mma_mm(x.tb + 64, qw2, x.tile(F_V));
            mma_mm(x.tb + 128, x.tile(F_UW), x.tile(F_V));
        }
        x.commit();
        // the unit column's sums from the same rounded tiles: m_q = 1^T qw2, Y_loc = 1^T UW
        if (x.tid < 64) out[NWs::L_MQ + x.tid] = tile_colsum(qw2, x.tid, nullptr);
        else if (x.tid < 128) out[NWs::L_YLOC + x.tid - 64] = tile_colsum(x.tile(F_UW), x.tid - 64, nullptr);
        if (!x.wait()) break;
        x.ld_row(0, r);
        st_row16(out + NWs::L_SLOC + ro, r);
        x.ld_row(64, r);
        st_row16(out + NWs::L_CQ + ro, r);
        x.ld_row(128, r);
        st_row16(out + NWs::L_XLOC + ro, r);
    } while (false);
    teardown(x);
}

// ======================================================================= 3. fwd_incr
enum { I_AH, I_AL, I_BH, I_BL, I_N };

// MODE 0: X_loc <- S_p C_q + X_loc, Y_loc <- S_p m_q + Y_loc.
// MODE 1: O_loc <- O_loc + Lam_n W + lam_n w^T.
template <int MODE>
__global__ void __launch_bounds__(kTc, 2) incr_kernel(const __grid_constant__ BwdArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    Ctx x;
    if (!setup(x, smem_raw, I_N, a.err)) return;
    const int nch = (a.n + 63) / 64, u = blockIdx.x / nch, ch = blockIdx.x % nch;
    const Ptrs R = regions(a);
    float *lc = R.loc + ((size_t)u * nch + ch) * NWs::LOC;
    const float *so = R.st + ((size_t)u * nch + ch) * NWs::ST;
    {
        const float *ss[2] = {so + (MODE == 0 ? NWs::S_SP : NWs::S_LAM), lc + (MODE == 0 ? NWs::L_CQ : NWs::L_W)};
        uint8_t *hi[2] = {x.tile(I_AH), x.tile(I_BH)}, *lo[2] = {x.tile(I_AL), x.tile(I_BL)};
        load_tiles_hilo<2>(ss, hi, lo);
    }
    float *mq = reinterpret_cast<float *>(smem_raw + I_N * TILE + 64);  // m_q [64]
    if (MODE == 0 && x.tid < 64) mq[x.tid] = lc[NWs::L_MQ + x.tid];
    x.publish();
    const size_t ro = (size_t)x.row * 64 + x.c0;
    float *dst = lc + (MODE == 0 ? NWs::L_XLOC : NWs::L_OLOC) + ro;
    float add[16];
    ld_row16(dst, add);
    if (MODE == 1) {  // + lam_n[row] w[c]
        float wv[16];
        ld_row16(lc + NWs::L_WV + x.c0, wv);
        const float ln = so[NWs::S_LN + x.row];
#pragma unroll
        for (int i = 0; i < 16; ++i) add[i] = fmaf(ln, wv[i], add[i]);
    }
    do {
        if (x.tid == 0) mma3_km(x.tb + 0, x.tile(I_AH), x.tile(I_AL), x.tile(I_BH), x.tile(I_BL), false);
        x.commit();
        if (MODE == 0) {  // Y_loc += S_p m_q while the product runs: S_p = hi + lo from the
            // shared tiles, four threads per row, sixteen columns each
            const int i = x.tid >> 2, j0 = (x.tid & 3) * 16;
            float hv[8], lv[8], acc = 0.f;
#pragma unroll
            for (int h = 0; h < 16; h += 8) {
                tile_load_row8(x.tile(I_AH), 64, i, j0 + h, hv);
                tile_load_row8(x.tile(I_AL), 64, i, j0 + h, lv);
#pragma unroll
                for (int e = 0; e < 8; ++e) acc = fmaf(hv[e] + lv[e], mq[j0 + h + e], acc);
            }
            acc += __shfl_xor_sync(0xffffffffu, acc, 1);
            acc += __shfl_xor_sync(0xffffffffu, acc, 2);
            if ((x.tid & 3) == 0) lc[NWs::L_YLOC + i] += acc;
        }
        if (!x.wait()) break;
        float r[16];
        x.ld_row(0, r);
#pragma unroll
        for (int i = 0; i < 16; ++i) r[i] += add[i];
        st_row16(dst, r);
    } while (false);
    teardown(x);
}

// ======================================================================= 5. out_local
// Tiles are reused once their last reader has completed:
//   SA: S_p hi, then A hi;  SB: S_p lo, then A lo;  XA: X_p hi, then g^{2s} Q;
//   XB: X_p lo, then g^{2L-s} Q;  T0: A~, then M, then P;  T1: U, then the weighted dU_loc.
enum { O_Q, O_K, O_V, O_G, O_SA, O_SB, O_XA, O_XB, O_T0, O_T1, O_N };

__global__ void __launch_bounds__(kTc, 2) out_local_kernel(const __grid_constant__ BwdArgs a,
                                                             const __grid_constant__ ChunkMaps tm, float eps) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    Ctx x;
    if (!setup(x, smem_raw, O_N, a.err)) return;
    float *gp = reinterpret_cast<float *>(smem_raw + O_N * TILE + 64);
    float *yp = gp + kGp;    // Y_p [64]
    float *rr = yp + 64;     // r per token row [64]
    float *cc = rr + 64;     // c per token row [64]
    float *red = cc + 64;    // row partials of the second half of the threads [64][2]
    float *w = red + 128;    // token weights g^{2s}, g^{2L-s} [2][64]
    const int nch = (a.n + 63) / 64, u = blockIdx.x / nch, ch = blockIdx.x % nch;
    const int t0 = ch * 64, L = min(64, a.n - t0);
    const bool decay = (a.flags & HLA_DECAY) != 0;
    const Ptrs R = regions(a);
    float *lc = R.loc + ((size_t)u * nch + ch) * NWs::LOC;
    const float *so = R.st + ((size_t)u * nch + ch) * NWs::ST;
    {  // the bf16 inputs by TMA while the threads convert the states
        const CUtensorMap *m[4] = {&tm.q, &tm.k, &tm.v, &tm.g};
        const int kvu = (int)bwd::kv_unit(a, u), un[4] = {u, kvu, kvu, u};
        uint8_t *dst[4] = {x.tile(O_Q), x.tile(O_K), x.tile(O_V), x.tile(O_G)};
        tma_issue<4>(x, m, un, t0, dst);
    }
    fill_gp(gp, a, u);
    {
        const float *ss[2] = {so + NWs::S_SP, so + NWs::S_XP};
        uint8_t *hi[2] = {x.tile(O_SA), x.tile(O_XA)}, *lo[2] = {x.tile(O_SB), x.tile(O_XB)};
        load_tiles_hilo<2>(ss, hi, lo);
    }
    __syncthreads();  // gp
    for (int i = threadIdx.x; i < 64; i += kTc) {
        yp[i] = so[NWs::S_YP + i];
        w[i] = i < L ? gp[2 * i] : 0.f;
        w[64 + i] = i < L ? gp[2 * L - i] : 0.f;
    }
    const bool loaded = tma_wait(x);
    x.publish();
    const int t = x.row;
    const bool in = t < L;
    const float r_u = gp[t + 1], r_x = gp[2 * (t + 1)];
    const size_t ro = (size_t)t * 64 + x.c0;
    float r[16], s[16];
    do {
        if (!loaded) break;
        // stage 1: Q K^T; Q S_p; Q X_p
        if (x.tid == 0) {
            mma_kk(x.tb + 0, x.tile(O_Q), x.tile(O_K), false);
            mma_km(x.tb + 64, x.tile(O_Q), x.tile(O_SA), false);
            mma_km(x.tb + 64, x.tile(O_Q), x.tile(O_SB), true);
            mma_km(x.tb + 128, x.tile(O_Q), x.tile(O_XA), false);
            mma_km(x.tb + 128, x.tile(O_Q), x.tile(O_XB), true);
        }
        x.commit();
        if (!x.wait()) break;
        x.ld_row(0, r);
        store_tril_decay(x, x.tile(O_T0), r, gp, 1);
        x.publish();
        // stage 2: A~ K
        if (x.tid == 0) mma_km(x.tb + 192, x.tile(O_T0), x.tile(O_K), false);
        x.commit();
        if (!x.wait()) break;
        x.ld_row(64, s);
        x.ld_row(192, r);
#pragma unroll
        for (int i = 0; i < 16; ++i) r[i] += r_u * s[i];  // U = g^{t+1} Q S_p + A~ K
        tile_store_row16(x.tile(O_T1), 64, t, x.c0, r);
        x.publish();
        // stage 3: M = Q U^T
        if (x.tid == 0) mma_kk(x.tb + 0, x.tile(O_Q), x.tile(O_T1), false);
        x.commit();
        if (!x.wait()) break;
        x.ld_row(0, r);
        store_tril_decay(x, x.tile(O_T0), r, gp, 2);
        // this thread's part of den_t = g^{2(t+1)} q_t.Y_p + sum_s M[t][s], with M rounded
        // as the product M V sees it, so that n and den weigh the tokens alike
        float den = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) den += __bfloat162float(__float2bfloat16_rn(r[i]));
        {
            float qv[8];
#pragma unroll
            for (int h = 0; h < 16; h += 8) {
                tile_load_row8(x.tile(O_Q), 64, t, x.c0 + h, qv);
                float dq = 0.f;
#pragma unroll
                for (int i = 0; i < 8; ++i) dq = fmaf(qv[i], yp[x.c0 + h + i], dq);
                den = fmaf(r_x, dq, den);
            }
        }
        x.publish();
        // stage 4: M V
        if (x.tid == 0) mma_km(x.tb + 64, x.tile(O_T0), x.tile(O_V), false);
        x.commit();
        if (!x.wait()) break;
        // n = g^{2(t+1)} Q X_p + M V; r = 1 / (den + eps), c = r^2 (g . n); A = r g
        x.ld_row(128, s);
        x.ld_row(64, r);
        float gv[16], gn = 0.f;
        {
            float g0[8], g1[8];
            tile_load_row8(x.tile(O_G), 64, t, x.c0, g0);
            tile_load_row8(x.tile(O_G), 64, t, x.c0 + 8, g1);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                gv[i] = g0[i];
                gv[8 + i] = g1[i];
            }
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) gn = fmaf(gv[i], fmaf(r_x, s[i], r[i]), gn);
        den += __shfl_xor_sync(0xffffffffu, den, 16);
        gn += __shfl_xor_sync(0xffffffffu, gn, 16);
        if (x.half == 1 && x.lane < 16) {
            red[2 * t] = den;
            red[2 * t + 1] = gn;
        }
        __syncthreads();
        if (x.half == 0 && x.lane < 16) {
            den += red[2 * t];
            gn += red[2 * t + 1];
            const float rt = in ? 1.f / (den + eps) : 0.f, ct = rt * rt * gn;
            rr[t] = rt;
            cc[t] = ct;
            if (in) {
                R.r[(size_t)u * a.n + t0 + t] = rt;
                R.c[(size_t)u * a.n + t0 + t] = ct;
            }
        }
        __syncthreads();
        {
            const float rt = rr[t];
#pragma unroll
            for (int i = 0; i < 16; ++i) r[i] = rt * gv[i];
            store_hilo16(x.tile(O_SA), x.tile(O_SB), t, x.c0, r);
        }
        x.publish();
        // stage 5: P = A V^T (hi + lo); meanwhile the weighted copies of Q
        if (x.tid == 0) {
            mma_kk(x.tb + 0, x.tile(O_SA), x.tile(O_V), false);
            mma_kk(x.tb + 0, x.tile(O_SB), x.tile(O_V), true);
        }
        x.commit();
        const uint8_t *qw4 = x.tile(O_Q), *qw5 = x.tile(O_Q);
        if (decay) {
            scale_tile(x.tile(O_Q), L, w, x.tile(O_XA));
            scale_tile(x.tile(O_Q), L, w + 64, x.tile(O_XB));
            qw4 = x.tile(O_XA);
            qw5 = x.tile(O_XB);
        }
        if (!x.wait()) break;
        x.ld_row(0, r);
        {
            const float ct = cc[t];
#pragma unroll
            for (int i = 0; i < 16; ++i) r[i] -= ct;  // the unit column: -c_t
        }
        store_tril_decay(x, x.tile(O_T0), r, gp, 2);
        x.publish();
        // stage 6: dU_loc = P^T Q
        if (x.tid == 0) mma_mm(x.tb + 64, x.tile(O_T0), x.tile(O_Q));
        x.commit();
        if (!x.wait()) break;
        {
            const float w6 = in ? gp[t] : 0.f;
            x.ld_row(64, r);
#pragma unroll
            for (int i = 0; i < 16; ++i) r[i] *= w6;
            tile_store_row16(x.tile(O_T1), 64, t, x.c0, r);
        }
        x.publish();
        // stage 7: L_loc = qw4^T A (hi + lo), W = V^T qw5, O_loc = dUw^T Q
        if (x.tid == 0) {
            mma_mm(x.tb + 0, qw4, x.tile(O_SA));
            mma_mm(x.tb + 0, qw4, x.tile(O_SB), true);
            mma_mm(x.tb + 64, x.tile(O_V), qw5);
            mma_mm(x.tb + 128, x.tile(O_T1), x.tile(O_Q));
        }
        x.commit();
        // the unit column: lam_loc = -qw4^T c, w = 1^T qw5 (same rounded tiles)
        if (x.tid < 64) {
            const float l = tile_colsum(qw4, x.tid, cc);
            lc[NWs::L_LAM + x.tid] = -l;
        } else if (x.tid < 128) {
            lc[NWs::L_WV + x.tid - 64] = tile_colsum(qw5, x.tid - 64, nullptr);
        }
        if (!x.wait()) break;
        x.ld_row(0, r);
        st_row16(lc + NWs::L_LLOC + ro, r);
        x.ld_row(64, r);
        st_row16(lc + NWs::L_W + ro, r);
        x.ld_row(128, r);
        st_row16(lc + NWs::L_OLOC + ro, r);
    } while (false);
    teardown(x);
}

// ======================================================================= 9. grad
// A tile is reused once its last reader has completed: V (stage 1) then dU, Lam_n lo
// (stage 1) then A-tilde, S_p hi (stages 1, 3) then M, S_p lo then (Om + Om^T) hi,
// X_p hi (stage 3) then B, X_p lo then (Om + Om^T) lo -- 13 tiles, two CTAs per SM.
// U Lam_n (for dv, where nothing cancels) takes Lam_n's hi part only.
enum { G_Q, G_K, G_V, G_AH, G_AL, G_SH, G_SL, G_XH, G_XL, G_LH, G_LL, G_P, G_U, G_N };
constexpr int G_DU = G_V, G_A = G_LL, G_M = G_SH, G_OH = G_SL, G_B = G_XH, G_OL = G_XL;

__global__ void __launch_bounds__(kTc, 2) grad_kernel(const __grid_constant__ BwdArgs a,
                                                        const __grid_constant__ ChunkMaps tm) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    Ctx x;
    if (!setup(x, smem_raw, G_N, a.err)) return;
    float *gp = reinterpret_cast<float *>(smem_raw + G_N * TILE + 64);
    float *vec = gp + kGp;  // r, c, Y_p, lam_n [64] each
    float *rr = vec, *cc = vec + 64, *yp = vec + 128, *ln = vec + 192;
    const int nch = (a.n + 63) / 64, u = blockIdx.x / nch, ch = blockIdx.x % nch;
    const int t0 = ch * 64, L = min(64, a.n - t0);
    const size_t r0 = ((size_t)u * a.n + t0) * 64;
    const Ptrs R = regions(a);
    const float *so = R.st + ((size_t)u * nch + ch) * NWs::ST;
    {  // the bf16 inputs by TMA (the output gradient into A's hi tile) while the threads
       // convert the states
        const CUtensorMap *m[4] = {&tm.q, &tm.k, &tm.v, &tm.g};
        const int kvu = (int)bwd::kv_unit(a, u), un[4] = {u, kvu, kvu, u};
        uint8_t *dst[4] = {x.tile(G_Q), x.tile(G_K), x.tile(G_V), x.tile(G_AH)};
        tma_issue<4>(x, m, un, t0, dst);
    }
    fill_gp(gp, a, u);
    for (int i = threadIdx.x; i < 64; i += kTc) {
        const bool ok = i < L;
        rr[i] = ok ? R.r[(size_t)u * a.n + t0 + i] : 0.f;
        cc[i] = ok ? R.c[(size_t)u * a.n + t0 + i] : 0.f;
        yp[i] = so[NWs::S_YP + i];
        ln[i] = so[NWs::S_LN + i];
    }
    {
        const float *ss[3] = {so + NWs::S_SP, so + NWs::S_XP, so + NWs::S_LAM};
        uint8_t *hi[3] = {x.tile(G_SH), x.tile(G_XH), x.tile(G_LH)}, *lo[3] = {x.tile(G_SL), x.tile(G_XL), x.tile(G_LL)};
        load_tiles_hilo<3>(ss, hi, lo);
    }
    const bool loaded = tma_wait(x);  // also orders rr for the A tiles
    if (loaded) rowscale_hilo_inplace(x.tile(G_AH), x.tile(G_AL), rr, L);
    x.publish();
    const int t = x.row;
    const bool in = t < L;
    const float r_u = gp[t + 1], r_x = gp[2 * (t + 1)];
    const float r_l2 = in ? gp[2 * (L - t)] : 0.f, r_l1 = in ? gp[L - t] : 0.f;
    const size_t ro = r0 + (size_t)t * 64 + x.c0;
    float r[16], s[16];
    do {
        if (!loaded) break;
        // stage 1: A~ raw; P raw = A V^T (hi + lo); Q S_p; V Lam_n^T
        if (x.tid == 0) {
            mma_kk(x.tb + 0, x.tile(G_Q), x.tile(G_K), false);
            mma_kk(x.tb + 64, x.tile(G_AH), x.tile(G_V), false);
            mma_kk(x.tb + 64, x.tile(G_AL), x.tile(G_V), true);
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
        {
            const float ct = cc[t];
#pragma unroll
            for (int i = 0; i < 16; ++i) r[i] -= ct;
        }
        store_tril_decay(x, x.tile(G_P), r, gp, 2);
        x.publish();
        // stage 2: A~ K, P^T Q
        if (x.tid == 0) {
            mma_km(x.tb + 0, x.tile(G_A), x.tile(G_K), false);
            mma_mm(x.tb + 64, x.tile(G_P), x.tile(G_Q));
        }
        x.commit();
        if (!x.wait()) break;
        // U = r_u (Q S_p) + A~ K;  dU = P^T Q + r_l2 (V Lam_n^T + 1 lam_n^T)
        x.ld_row(128, s);
        x.ld_row(0, r);
#pragma unroll
        for (int i = 0; i < 16; ++i) r[i] += r_u * s[i];
        tile_store_row16(x.tile(G_U), 64, t, x.c0, r);
        x.ld_row(192, s);
        x.ld_row(64, r);
#pragma unroll
        for (int i = 0; i < 16; ++i) r[i] += r_l2 * (s[i] + ln[x.c0 + i]);
        tile_store_row16(x.tile(G_DU), 64, t, x.c0, r);
        x.publish();
        // stage 3: B raw, M raw; A X_p^T (three products); dU S_p
        if (x.tid == 0) {
            mma_kk(x.tb + 0, x.tile(G_DU), x.tile(G_K), false);
            mma_kk(x.tb + 64, x.tile(G_Q), x.tile(G_U), false);
            mma_kk(x.tb + 128, x.tile(G_AH), x.tile(G_XH), false);
            mma_kk(x.tb + 128, x.tile(G_AH), x.tile(G_XL), true);
            mma_kk(x.tb + 128, x.tile(G_AL), x.tile(G_XH), true);
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
        load_sym_hilo(so + NWs::S_OM, x.tile(G_OH), x.tile(G_OL));
        if (!x.wait()) break;
        // dQ = (P U + B K) + r_x (A X_p^T - c Y_p^T) + r_u (dU S_p)
        x.ld_row(0, r);
        x.ld_row(128, s);
        {
            const float ct = cc[t];
#pragma unroll
            for (int i = 0; i < 16; ++i) r[i] += r_x * fmaf(-ct, yp[x.c0 + i], s[i]);
        }
        x.ld_row(192, s);
#pragma unroll
        for (int i = 0; i < 16; ++i) r[i] += r_u * s[i];
        if (in) st_row16_bf16(static_cast<__nv_bfloat16 *>(a.grad_q) + ro, r);
        x.publish();  // the reads of columns 0, 128, 192 precede their reuse
        // stage 5: K (Om + Om^T); M^T A (hi + lo); U Lam_n
        if (x.tid == 0) {
            mma_km(x.tb + 128, x.tile(G_K), x.tile(G_OH), false);
            mma_km(x.tb + 128, x.tile(G_K), x.tile(G_OL), true);
            mma_mm(x.tb + 0, x.tile(G_M), x.tile(G_AH));
            mma_mm(x.tb + 0, x.tile(G_M), x.tile(G_AL), true);
            mma_km(x.tb + 192, x.tile(G_U), x.tile(G_LH), false);
        }
        x.commit();
        if (!x.wait()) break;
        // dK = (A~^T dU + B^T Q) + r_l1 K (Om + Om^T);  dV = M^T A + r_l2 U Lam_n
        x.ld_row(64, r);
        x.ld_row(128, s);
#pragma unroll
        for (int i = 0; i < 16; ++i) r[i] += r_l1 * s[i];
        if (in) {
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

constexpr size_t kFwdLocalSmem = F_N * TILE + 64 + (kGp + 2 * 64) * 4;
constexpr size_t kIncrSmem = I_N * TILE + 64 + 64 * 4;
constexpr size_t kOutSmem = O_N * TILE + 64 + (kGp + 64 * 3 + 128 + 128) * 4;
constexpr size_t kGradSmem = G_N * TILE + 64 + (kGp + 4 * 64) * 4;

template <typename K>
cudaError_t smem_attr(K kern, size_t bytes) {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace
}  // namespace bwdn

bool bwd_norm_tc_shape(const hla_params &p) {
    return p.in_dtype == HLA_BF16 && p.d == 64 && p.dv == 64 && p.chunk == 64 && (p.flags & HLA_NORMALIZE) &&
           !(p.flags & (HLA_UNMASKED | HLA_ASYMMETRIC));
}

bool bwd_norm_tc_supported(const hla_params &p, const BwdArgs &a) { return bwd_norm_tc_shape(p) && !a.sin_S && !a.dS; }

size_t bwd_norm_tc_workspace(const hla_params &p) {
    if (!bwd_norm_tc_shape(p)) return 0;
    const int hkv = p.Hkv > 0 ? p.Hkv : p.H;
    return (bwdn::layout(p.B, p.H, hkv, p.n).total * sizeof(float) + 255) & ~size_t(255);
}

hla_status bwd_norm_tc_launch(const hla_params &p, const BwdArgs &a0, cudaStream_t st) {
    using namespace bwdn;
    BwdArgs a = a0;
    const Lay l = layout(a.B, a.H, a.Hkv, a.n);
    a.dk_pair = a.Hkv < a.H ? a.workspace + l.dk_pair : nullptr;
    a.dv_pair = a.Hkv < a.H ? a.workspace + l.dv_pair : nullptr;
    const int units = a.B * a.H, nch = (a.n + 63) / 64;
    const float *gamma = (a.flags & HLA_DECAY) ? a.gamma : nullptr;
    float *loc = a.workspace + l.loc, *sta = a.workspace + l.st;
    auto fail = [](cudaError_t e, const char *where) {
        char msg[192];
        snprintf(msg, sizeof msg, "normalised backward (tensor cores), %s: %s", where, cudaGetErrorString(e));
        return report(HLA_ERR_CUDA, msg);
    };
    auto mark = [&](int i) { return a.events ? cudaEventRecord(a.events[i], st) : cudaSuccess; };
    cudaError_t e;
    if ((e = smem_attr(fwd_local_kernel, kFwdLocalSmem)) != cudaSuccess ||
        (e = smem_attr(incr_kernel<0>, kIncrSmem)) != cudaSuccess ||
        (e = smem_attr(incr_kernel<1>, kIncrSmem)) != cudaSuccess ||
        (e = smem_attr(out_local_kernel, kOutSmem)) != cudaSuccess ||
        (e = smem_attr(grad_kernel, kGradSmem)) != cudaSuccess)
        return fail(e, "kernel attributes");
    auto job = [&](size_t in_off, size_t out_off, int count, int reverse, int power) {
        return PrefixJob{loc, NWs::LOC, in_off, sta, NWs::ST, out_off, nullptr, nullptr, count, reverse, power};
    };
    PrefixArgs pa{};
    pa.units = units; pa.nch = nch; pa.n = a.n; pa.chunk = 64; pa.H = a.H; pa.gamma = gamma;
    if ((e = mark(0)) != cudaSuccess) return fail(e, "event");
    // forward: local sums, S_p, increments, X_p and Y_p, then the outputs and the backward local sums
    ChunkMaps maps;
    if (!chunk_maps(maps, a.q, a.k, a.v, a.go, a.n, units, a.B * a.Hkv)) return fail(cudaErrorInvalidValue, "tensor maps");
    fwd_local_kernel<<<units * nch, kTc, kFwdLocalSmem, st>>>(a, maps);
    pa.njobs = 1;
    pa.job[0] = job(NWs::L_SLOC, NWs::S_SP, 64 * 64, 0, 1);
    if ((e = chunk_prefix(pa, st)) != cudaSuccess) return fail(e, "S prefix");
    incr_kernel<0><<<units * nch, kTc, kIncrSmem, st>>>(a);
    pa.njobs = 2;
    pa.job[0] = job(NWs::L_XLOC, NWs::S_XP, 64 * 64, 0, 2);
    pa.job[1] = job(NWs::L_YLOC, NWs::S_YP, 64, 0, 2);
    if ((e = chunk_prefix(pa, st)) != cudaSuccess) return fail(e, "X prefix");
    out_local_kernel<<<units * nch, kTc, kOutSmem, st>>>(a, maps, p.eps);
    if ((e = cudaGetLastError()) != cudaSuccess) return fail(e, "outputs");
    if ((e = mark(1)) != cudaSuccess) return fail(e, "event");
    // backward scan: Lam_n and lam_n, the increments of Om, then Om_n
    pa.job[0] = job(NWs::L_LLOC, NWs::S_LAM, 64 * 64, 1, 2);
    pa.job[1] = job(NWs::L_LAM, NWs::S_LN, 64, 1, 2);
    if ((e = chunk_prefix(pa, st)) != cudaSuccess) return fail(e, "Lam suffix");
    incr_kernel<1><<<units * nch, kTc, kIncrSmem, st>>>(a);
    pa.njobs = 1;
    pa.job[0] = job(NWs::L_OLOC, NWs::S_OM, 64 * 64, 1, 1);
    if ((e = chunk_prefix(pa, st)) != cudaSuccess) return fail(e, "Om suffix");
    if ((e = mark(2)) != cudaSuccess) return fail(e, "event");
    grad_kernel<<<units * nch, kTc, kGradSmem, st>>>(a, maps);
    if ((e = cudaGetLastError()) != cudaSuccess) return fail(e, "gradients");
    if (a.dk_pair) {  // shared key/value heads: sum each group's gradients
        const size_t elems = (size_t)a.B * a.Hkv * a.n * 64;
        const int blocks = (int)((elems + 255) / 256 < 8192 ? (elems + 255) / 256 : 8192);
        bwd::bwd_group_sum_kernel<__nv_bfloat16><<<blocks, bwd::kThreads, 0, st>>>(
            a.dk_pair, static_cast<__nv_bfloat16 *>(a.grad_k), a.B, a.H, a.Hkv, (size_t)a.n * 64);
        bwd::bwd_group_sum_kernel<__nv_bfloat16><<<blocks, bwd::kThreads, 0, st>>>(
            a.dv_pair, static_cast<__nv_bfloat16 *>(a.grad_v), a.B, a.H, a.Hkv, (size_t)a.n * 64);
        if ((e = cudaGetLastError()) != cudaSuccess) return fail(e, "group sums");
    }
    if ((e = mark(3)) != cudaSuccess) return fail(e, "event");
    return HLA_OK;
}

}  // namespace hla
