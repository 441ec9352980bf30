// hla_fwd_tc.cuh -- chunk-parallel masked second-order HLA forward on the
// sm_103a tensor cores (tcgen05 MMA, TMEM accumulators, TMA tile loads), bf16
// inputs, fp32 accumulation and fp32 state.  Included by one translation unit
// per (decay, normalise) combination.
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
// Parallel structure (one launch): the chunks of all (b,h) sequences, laid end
// to end, are cut into equal runs, one per CTA, as many CTAs as fit on the device
// at once.  A run that crosses a sequence boundary holds a piece of each
// sequence it touches.  CTAs take runs in ticket order, so a CTA only ever waits
// for CTAs that started before it.
//   pass 1: each piece's own summary (S, C, X, m, Y from zero) -> workspace,
//           then a release flag;
//   scan:   per piece, the CTA folds state_in and the summaries of all earlier
//           pieces of its sequence (exclusive scan by the concatenation rule), in
//           one pipelined pass whose only products, f S C_B, go to the tensor cores;
//   pass 2: the chunk loop again from that exact prefix, writing O.
// The CTA holding a sequence's last piece exports state_out (S, C, m,
// G = S C - X, h = S m - Y): C, m (and Y without normalisation) before pass 2,
// the rest from the state that pass 2 leaves at the sequence end.
//
// Each CTA: 256 threads (8 warps).  Thread 0 issues TMA and MMAs.  TMEM
// epilogues: warp w reads lane quadrant w % 4 and column half w / 4 of an
// accumulator.  TMEM (512 columns): work W [0,128), S [128,256), X [256,384),
// C (pass 1 / scan) or spare (pass 2) [384,512).  Token-row accumulators use
// M = c rows, state accumulators M = d rows.  The next chunk's Q, K, V tiles
// are prefetched into a second input stage when shared memory allows.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>

#include "hla_internal.h"
#include "hla_tmap.h"

namespace hla {
namespace tc {

constexpr int kThreads = 256;

__host__ __device__ constexpr int cmax(int a, int b) { return a > b ? a : b; }
__host__ __device__ constexpr int pow2ceil(int x) { return x <= 32 ? 32 : (x <= 64 ? 64 : (x <= 128 ? 128 : (x <= 256 ? 256 : 512))); }

// TMEM columns: work W (max(c, d, dv)), S (d), X (dv), fourth slot: C in pass 1
// and the scan (dv), spare in pass 2 (d or dv).  Shapes that fit in 256 columns
// run two CTAs per SM.
__host__ __device__ constexpr int tmem_cols(int C, int D, int DV) {
    return pow2ceil(cmax(cmax(C, D), DV) + D + DV + cmax(D, DV));
}
inline int ctas_per_sm(const hla_params &p) { return tmem_cols(p.chunk, p.d, p.dv) <= 256 ? 2 : 1; }

struct TcParams {
    CUtensorMap tmQ, tmK, tmV, tmO;
    int B, H, n, BH;
    int Hkv;  // key/value heads: query head h reads key/value head h / (H / Hkv)
    // work split: the BH sequences' chunks, laid end to end, are cut into runs of
    // cpc chunks, one per CTA; a run that crosses a sequence boundary holds a
    // piece of each sequence.  A sequence has at most kmax pieces.
    int nchunks, cpc, kmax;
    // > 0 when runs align with sequences (R runs each): tickets then go out level
    // by level (piece 0 of every sequence, then piece 1, ...), so that the CTAs
    // holding the last pieces, which fold the most, are the last to be placed
    int runs_per_seq;
    float eps;
    const float *gamma;
    void *o;
    StatePtrs sin, sout;
    unsigned *ticket;   // workspace header (take_ticket, finish_call)
    unsigned *flagsw;   // [BH][kmax] release flags
    float *summ;        // [BH][kmax][SUM] piece summaries
    unsigned *err;
};

template <int C, int D, int DV>
struct Cfg {
    static constexpr int SUM = D * D + 2 * D * DV + 2 * D;  // S, X, C, m, Y
    // operand tiles (bytes)
    static constexpr int SZ_Q = C * D * 2, SZ_K = C * D * 2, SZ_V = C * DV * 2;
    static constexpr int SZ_TA = cmax(C * C, C * D) * 2;
    static constexpr int SZ_TU = C * D * 2;
    static constexpr int SZ_TS = cmax(cmax(D * D, C * D), C * DV) * 2;
    static constexpr int SZ_TQ = cmax(C * D, D * DV) * 2;
    static constexpr int SZ_IN = SZ_Q + SZ_K + SZ_V;  // one input stage
    static constexpr int WORK = SZ_TA + SZ_TU + SZ_TS + SZ_TQ;
    // scan / export phase operands: S and C as bf16 hi + lo pairs (alias the tiles)
    static constexpr int FOLD = 2 * D * D * 2 + 2 * D * DV * 2;
    // TMEM slots
    static constexpr uint32_t TW = 0, TS = cmax(cmax(C, D), DV), TX = TS + D, T4 = TX + DV;
    static constexpr int TCOLS = tmem_cols(C, D, DV);
    static constexpr int CTAS = TCOLS <= 256 ? 2 : 1;
    // row partial sums: one slot per column part of an accumulator row
    static constexpr int NP_C = C == 128 ? 2 : 4, NP_D = D == 128 ? 2 : 4;
    // fp32 vectors: m, Y [D]; pass 2's row sums [NP_C x C] and q.Y [C]; g^j and
    // g^{2j} for j < 16
    static constexpr int R1 = NP_C * C + C;
    static constexpr int NVEC = 2 * D + R1 + 32;
    static constexpr int SMALL = NVEC * 4 + 64;
    static constexpr int LIMIT = 227 * 1024;
    // two input stages (prefetch of the next chunk) when they fit
    static constexpr int NSTAGE = (2 * SZ_IN + WORK + SMALL <= LIMIT) ? 2 : 1;
    static constexpr int OFF_IN = 0;
    static constexpr int OFF_TA = NSTAGE * SZ_IN, OFF_TU = OFF_TA + SZ_TA, OFF_TS = OFF_TU + SZ_TU,
                         OFF_TQ = OFF_TS + SZ_TS, TILES = OFF_TQ + SZ_TQ;
    // two sets of scan operands when they fit in the tile arena
    static constexpr int FBUF = 2 * FOLD <= TILES ? 2 : 1;
    static constexpr int ARENA = cmax(TILES, FBUF * FOLD);
    // scan / export: two sets of row partials [NP_D x D] after the operands
    static constexpr int OFF_PART = FBUF * FOLD;
    static_assert(OFF_PART + 2 * NP_D * D * 4 <= ARENA, "scan partials");
    static constexpr int OFF_VEC = ARENA;
    static constexpr int OFF_BAR = ARENA + NVEC * 4;
    static constexpr int SMEM = OFF_BAR + 64;
    // CTAs per SM set by the shared-memory request (and TMEM / registers)
    static constexpr int SMEM_LAUNCH = CTAS == 2 ? cmax(SMEM, 78 * 1024) : cmax(SMEM, 120 * 1024);
    static_assert(CTAS == 1 || SMEM <= 112 * 1024, "two CTAs per SM need <= 112 KB each");
    static_assert(SMEM <= LIMIT, "shared memory budget");
    static_assert(C == 64 || C == 128, "chunk");
    static_assert(D == 64 || D == 128, "d");
    static_assert(DV == 64 || DV == 128, "dv");
};

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

__device__ __forceinline__ float4 ldcg4(const float *p) { return __ldcg(reinterpret_cast<const float4 *>(p)); }

__device__ __forceinline__ void st_row16(float *dst, const float (&v)[16]) {
#pragma unroll
    for (int i = 0; i < 16; i += 4)
        *reinterpret_cast<float4 *>(dst + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
}

// Row of an accumulator with MR rows held by (quadrant q, lane l), or -1.
template <int MR>
__device__ __forceinline__ int row_of(int q, int l) {
    if constexpr (MR == 128) return 32 * q + l;
    else return 16 * q + (l & 15);
}

template <int C, int D, int DV, bool DECAY, bool NORM, int VAR>
struct Kern {
    using K_ = Cfg<C, D, DV>;
    // variant: 0 masked, 1 unmasked (o = q^T S C), 2 asymmetric (AHLA)
    static constexpr bool UNM = VAR == 1, ASYM = VAR == 2;
    static constexpr uint32_t TW = K_::TW, TS = K_::TS, TX = K_::TX, T4 = K_::T4;
    const TcParams &P;
    uint8_t *base;
    // Work tiles, scan operands and small fp32 vectors, all at fixed offsets from
    // `base` (computed on use, so they occupy no registers).
    __device__ __forceinline__ uint8_t *tA() const { return base + K_::OFF_TA; }
    __device__ __forceinline__ uint8_t *tU() const { return base + K_::OFF_TU; }
    __device__ __forceinline__ uint8_t *tS() const { return base + K_::OFF_TS; }
    __device__ __forceinline__ uint8_t *tQ() const { return base + K_::OFF_TQ; }
    __device__ __forceinline__ uint8_t *fShi(int b) const { return base + b * K_::FOLD; }
    __device__ __forceinline__ uint8_t *fSlo(int b) const { return fShi(b) + D * D * 2; }
    __device__ __forceinline__ uint8_t *fChi(int b) const { return fShi(b) + 2 * D * D * 2; }
    __device__ __forceinline__ uint8_t *fClo(int b) const { return fChi(b) + D * DV * 2; }
    __device__ __forceinline__ uint8_t *tShi() const { return fShi(0); }
    __device__ __forceinline__ uint8_t *tSlo() const { return fSlo(0); }
    __device__ __forceinline__ uint8_t *tChi() const { return fChi(0); }
    __device__ __forceinline__ uint8_t *tClo() const { return fClo(0); }
    __device__ __forceinline__ float *vec() const { return reinterpret_cast<float *>(base + K_::OFF_VEC); }
    __device__ __forceinline__ float *mrun() const { return vec(); }              // [D]
    __device__ __forceinline__ float *Yrun() const { return vec() + D; }          // [D]
    __device__ __forceinline__ float *part(int b = 0) const {                     // scan: 2 x [NP_D x D]
        return reinterpret_cast<float *>(base + K_::OFF_PART) + b * K_::NP_D * D;
    }
    __device__ __forceinline__ float *rsum() const { return vec() + 2 * D; }      // pass 2: [NP_C x C]
    __device__ __forceinline__ float *den() const { return vec() + 2 * D + K_::NP_C * C; }  // pass 2: [C]
    __device__ __forceinline__ float *g16() const { return vec() + 2 * D + K_::R1; }  // g^j, g^{2j}
    uint64_t *tma_bar, *mma_bar, *mma_bar2, *mma_bar3;
    uint32_t tb, tph, mph, mph2, mph3;
    int tid, warp, lane, quad, half;
    unsigned tag;  // the value this call's release flags carry
    int rowC, rowD;  // rows this thread owns in token-row / state accumulators (-1: none)
    int bh;
    int kvh;  // key/value head (b * Hkv + h / (H / Hkv)) of pair bh
    float lg;
    bool need_mY;

    __device__ Kern(const TcParams &p, uint8_t *b) : P(p), base(b) {}

    __device__ uint8_t *sQ(int s) const { return base + K_::OFF_IN + s * K_::SZ_IN; }
    __device__ uint8_t *sK(int s) const { return sQ(s) + K_::SZ_Q; }
    __device__ uint8_t *sV(int s) const { return sK(s) + K_::SZ_K; }

    // g^x for x >= 0 (1 without decay)
    __device__ __forceinline__ float gp(int x) const {
        if constexpr (DECAY) return gpow(lg, (float)x);
        else return 1.f;
    }
    __device__ __forceinline__ uint32_t taddr(uint32_t slot, int col) const {
        return tb + slot + ((uint32_t)(32 * quad) << 16) + (uint32_t)col;
    }

    // ---- synchronisation; false = abort (a bounded wait expired)
    __device__ bool wait_mma() {
        bool ok = mbar_wait(mma_bar, mph, P.err);
        mph ^= 1u;
        tc_fence_after();
        return !__syncthreads_or(!ok);
    }
    // Second completion barrier: MMAs committed to it run on while the block
    // works on results committed to the first one.
    __device__ bool wait_mma2() {
        bool ok = mbar_wait(mma_bar2, mph2, P.err);
        mph2 ^= 1u;
        tc_fence_after();
        return !__syncthreads_or(!ok);
    }
    __device__ void commit2() {
        if (tid == 0) umma_commit(mma_bar2);
    }
    // Third barrier, three arrivals: independent products issued by the lane-0
    // threads of warps 1-3 (or 0-2), each committing its own MMAs to it, so that
    // their issue overlaps instead of queueing behind one thread.
    static constexpr uint32_t kFan = 3;
    __device__ bool wait_mma3() {
        bool ok = mbar_wait(mma_bar3, mph3, P.err);
        mph3 ^= 1u;
        tc_fence_after();
        return !__syncthreads_or(!ok);
    }
    __device__ void arrive3() {  // an arrival with no MMAs behind it
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(mma_bar3)) : "memory");
    }
    // Block barrier that also orders this thread's TMEM accesses around it.
    __device__ void tc_sync() {
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }
    __device__ bool wait_tma(int s) {
        bool ok = mbar_wait(tma_bar + s, (tph >> s) & 1u, P.err);
        tph ^= (1u << s);
        return !__syncthreads_or(!ok);
    }
    // Make shared-memory and TMEM writes of all threads visible to the MMAs issued next.
    __device__ void publish() {
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }
    __device__ void commit() {
        if (tid == 0) umma_commit(mma_bar);
    }

    // ---- MMA groups (thread 0 only).  Shapes are compile-time, the K loop is
    // unrolled, and each step adds a constant byte offset (>> 4) to descriptors
    // built once per group, so issuing costs a few instructions per MMA.
    // token-row product, A K-major [C x KD], B K-major [N x KD]
    template <int N, int KD>
    __device__ __forceinline__ void mma_kk(uint32_t slot, const uint8_t *a, const uint8_t *b, bool acc) {
        constexpr uint32_t id = make_idesc(C, N, false, false);
        const uint64_t da = make_sdesc(smem_u32(a), 16u, 1024u), db = make_sdesc(smem_u32(b), 16u, 1024u);
#pragma unroll 1
        for (int k = 0; k < KD; k += 16) {
            const uint32_t ka = ((uint32_t)(k >> 6) * C * 128u + (uint32_t)(k & 63) * 2u) >> 4;
            const uint32_t kb = ((uint32_t)(k >> 6) * N * 128u + (uint32_t)(k & 63) * 2u) >> 4;
            umma_f16(tb + slot, da + ka, db + kb, id, (acc || k > 0) ? 1u : 0u);
        }
    }
    // token-row product, A K-major [C x KD], B MN-major [KD x N]
    template <int N, int KD>
    __device__ __forceinline__ void mma_km(uint32_t slot, const uint8_t *a, const uint8_t *b, bool acc) {
        constexpr uint32_t id = make_idesc(C, N, false, true);
        const uint64_t da = make_sdesc(smem_u32(a), 16u, 1024u), db = make_sdesc(smem_u32(b), KD * 128u, 1024u);
#pragma unroll 1
        for (int k = 0; k < KD; k += 16) {
            const uint32_t ka = ((uint32_t)(k >> 6) * C * 128u + (uint32_t)(k & 63) * 2u) >> 4;
            umma_f16(tb + slot, da + ka, db + (uint32_t)(k * 8), id, (acc || k > 0) ? 1u : 0u);
        }
    }
    // state product over tokens: A MN-major [C x D] (as D x C), B MN-major [C x N]
    template <int N>
    __device__ __forceinline__ void mma_mm(uint32_t slot, const uint8_t *a, const uint8_t *b, bool acc) {
        constexpr uint32_t id = make_idesc(D, N, true, true);
        const uint64_t da = make_sdesc(smem_u32(a), C * 128u, 1024u), db = make_sdesc(smem_u32(b), C * 128u, 1024u);
#pragma unroll 1
        for (int k = 0; k < C; k += 16)
            umma_f16(tb + slot, da + (uint32_t)(k * 8), db + (uint32_t)(k * 8), id, (acc || k > 0) ? 1u : 0u);
    }
    // state x state: A K-major [D x D] (rows = M), B MN-major [D x DV]
    __device__ __forceinline__ void mma_ss(uint32_t slot, const uint8_t *a, const uint8_t *b, bool acc) {
        constexpr uint32_t id = make_idesc(D, DV, false, true);
        const uint64_t da = make_sdesc(smem_u32(a), 16u, 1024u), db = make_sdesc(smem_u32(b), D * 128u, 1024u);
#pragma unroll 1
        for (int k = 0; k < D; k += 16) {
            const uint32_t ka = ((uint32_t)(k >> 6) * D * 128u + (uint32_t)(k & 63) * 2u) >> 4;
            umma_f16(tb + slot, da + ka, db + (uint32_t)(k * 8), id, (acc || k > 0) ? 1u : 0u);
        }
    }

    __device__ void tma_chunk(int jj, int s) {
        if (tid == 0) {
            fence_async_smem();  // earlier generic reads of the stage precede the overwrite
            mbar_expect_tx(tma_bar + s, K_::SZ_IN);
            const int t0 = jj * C;
#pragma unroll
            for (int kb = 0; kb < D / 64; ++kb) {
                tma_load_3d(sQ(s) + kb * C * 128, &P.tmQ, tma_bar + s, kb * 64, t0, bh);
                tma_load_3d(sK(s) + kb * C * 128, &P.tmK, tma_bar + s, kb * 64, t0, kvh);
            }
#pragma unroll
            for (int kb = 0; kb < DV / 64; ++kb) tma_load_3d(sV(s) + kb * C * 128, &P.tmV, tma_bar + s, kb * 64, t0, kvh);
        }
    }

    // ---- TMEM row access.  An accumulator with MR = 128 rows keeps row r in lane r:
    // warp w reads lane quadrant w % 4, and the two warps of a quadrant split the
    // columns in halves.  One with MR = 64 keeps its rows in lanes 0-15 of each
    // quadrant: the 16x32bx2 shape lets both half-warps read, so the columns split
    // in quarters.  f(c0, v[16]) gets 16 consecutive columns starting at c0.
    template <int MR>
    __device__ __forceinline__ int colpart() const { return MR == 128 ? half : half * 2 + (lane >> 4); }
    template <int MR, int NC, typename F>
    __device__ __forceinline__ void for_row(uint32_t slot, F &&f) {
        float a[16], b[16];
        if constexpr (MR == 128) {
            constexpr int HALF = NC / 2;
#pragma unroll
            for (int c0 = 0; c0 < HALF; c0 += 32) {
                const int c = half * HALF + c0;
                tmem_ld16(taddr(slot, c), a);
                tmem_ld16(taddr(slot, c + 16), b);
                tmem_wait_ld();
                f(c, a);
                f(c + 16, b);
            }
        } else {
            constexpr int QC = NC / 4;
            const int cw = half * (NC / 2), cme = cw + (lane >> 4) * QC;
            if constexpr (QC == 16) {
                tmem_ld16x2<QC>(taddr(slot, cw), a);
                tmem_wait_ld();
                f(cme, a);
            } else {
                tmem_ld16x2<QC>(taddr(slot, cw), a);
                tmem_ld16x2<QC>(taddr(slot, cw + 16), b);
                tmem_wait_ld();
                f(cme, a);
                f(cme + 16, b);
            }
        }
    }
    // Read-modify-write: values changed by f are stored back.
    template <int MR, int NC, typename F>
    __device__ __forceinline__ void rmw_row(uint32_t slot, F &&f) {
        float a[16], b[16];
        if constexpr (MR == 128) {
            constexpr int HALF = NC / 2;
#pragma unroll
            for (int c0 = 0; c0 < HALF; c0 += 32) {
                const int c = half * HALF + c0;
                tmem_ld16(taddr(slot, c), a);
                tmem_ld16(taddr(slot, c + 16), b);
                tmem_wait_ld();
                f(c, a);
                f(c + 16, b);
                tmem_st16(taddr(slot, c), a);
                tmem_st16(taddr(slot, c + 16), b);
            }
        } else {
            constexpr int QC = NC / 4;
            const int cw = half * (NC / 2), cme = cw + (lane >> 4) * QC;
            if constexpr (QC == 16) {
                tmem_ld16x2<QC>(taddr(slot, cw), a);
                tmem_wait_ld();
                f(cme, a);
                tmem_st16x2<QC>(taddr(slot, cw), a);
            } else {
                tmem_ld16x2<QC>(taddr(slot, cw), a);
                tmem_ld16x2<QC>(taddr(slot, cw + 16), b);
                tmem_wait_ld();
                f(cme, a);
                f(cme + 16, b);
                tmem_st16x2<QC>(taddr(slot, cw), a);
                tmem_st16x2<QC>(taddr(slot, cw + 16), b);
            }
        }
        tmem_wait_st();
    }
    // Two accumulators with the same row layout, read together.
    template <int MR, int NC, typename F>
    __device__ __forceinline__ void for_row2(uint32_t s1, uint32_t s2, F &&f) {
        float a[16], b[16];
        if constexpr (MR == 128) {
            constexpr int HALF = NC / 2;
#pragma unroll
            for (int c0 = 0; c0 < HALF; c0 += 16) {
                const int c = half * HALF + c0;
                tmem_ld16(taddr(s1, c), a);
                tmem_ld16(taddr(s2, c), b);
                tmem_wait_ld();
                f(c, a, b);
            }
        } else {
            constexpr int QC = NC / 4;
            const int cw = half * (NC / 2), cme = cw + (lane >> 4) * QC;
#pragma unroll
            for (int c0 = 0; c0 < QC; c0 += 16) {
                tmem_ld16x2<QC>(taddr(s1, cw + c0), a);
                tmem_ld16x2<QC>(taddr(s2, cw + c0), b);
                tmem_wait_ld();
                f(cme + c0, a, b);
            }
        }
    }
    template <int MR, int NC>
    __device__ void zero_slot(uint32_t slot) {
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = 0.f;
        if constexpr (MR == 128) {
#pragma unroll
            for (int c0 = 0; c0 < NC / 2; c0 += 16) tmem_st16(taddr(slot, half * (NC / 2) + c0), v);
        } else {
            constexpr int QC = NC / 4;
#pragma unroll
            for (int c0 = 0; c0 < QC; c0 += 16) tmem_st16x2<QC>(taddr(slot, half * (NC / 2) + c0), v);
        }
        tmem_wait_st();
    }

    // Copy state accumulator `slot` (rows D, NC columns) to the bf16 tile `dst`;
    // with decay, also scale the accumulator by `scale` in place.
    template <int NC>
    __device__ __forceinline__ void extract_state(uint32_t slot, uint8_t *dst, float scale) {
        auto f = [&](int c0, float (&v)[16]) {
            tile_store_row16(dst, D, rowD, c0, v);
            if constexpr (DECAY) {
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] *= scale;
            }
        };
        if constexpr (DECAY) rmw_row<D, NC>(slot, f);
        else for_row<D, NC>(slot, f);
    }

    // Row partial sums: each column part of a row writes its own slot.
    template <int MR>
    __device__ void put_partial(float *dst, int row, float v) {
        dst[colpart<MR>() * MR + row] = v;
    }
    template <int MR>
    __device__ float sum_partials(const float *src, int row) const {
        float s = src[row] + src[MR + row];
        if constexpr (MR == 64) s += src[2 * MR + row] + src[3 * MR + row];
        return s;
    }

    // Row-scaled copy of a [C x W] tile: dst[r] = scale(r) * src[r] (all threads).
    template <int Wd, typename F>
    __device__ void scaled_tile_copy(const uint8_t *src, uint8_t *dst, F &&scale) {
        constexpr int GROUPS = Wd / 16;
        for (int e = tid; e < C * GROUPS; e += kThreads) {
            const int r = e / GROUPS, c0 = (e % GROUPS) * 16;
            const float s = scale(r);
            float a[8], b[8], v[16];
            tile_load_row8(src, C, r, c0, a);
            tile_load_row8(src, C, r, c0 + 8, b);
#pragma unroll
            for (int i = 0; i < 8; ++i) { v[i] = s * a[i]; v[8 + i] = s * b[i]; }
            tile_store_row16(dst, C, r, c0, v);
        }
    }

    // Masked, decayed row of a c x c score tile: v[i] (column c0+i of row `row`)
    // becomes 0 above the diagonal and is scaled by g^{P (row - col)} below it
    // (P = 1 for A-tilde, 2 for M).  Off-diagonal groups use one exp2 per group
    // and the factors g^{P j} held in gt.
    template <int POW>
    __device__ __forceinline__ void mask_row(int row, int c0, float (&v)[16], const float (&gt)[3]) const {
        if (c0 > row) {
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = 0.f;
        } else if (c0 + 15 <= row) {
            if constexpr (DECAY) {
                // g^{P(row-c0-i)}: start at i = 15 and multiply by g^P towards i = 0
                float f = gp(POW * (row - c0 - 15));
                const float step = gt[POW];
#pragma unroll
                for (int i = 15; i >= 0; --i) { v[i] *= f; f *= step; }
            }
        } else {  // the group holding the diagonal: factor 1 on it, times g^P per column to the left
            float f = 1.f;
            const float step = gt[POW];
#pragma unroll
            for (int i = 15; i >= 0; --i) {
                const bool keep = (c0 + i <= row);
                if constexpr (DECAY) {
                    v[i] = keep ? v[i] * f : 0.f;
                    f = keep ? f * step : f;
                } else {
                    v[i] = keep ? v[i] : 0.f;
                }
            }
        }
    }
    // g^{P j}, j < 16, into registers (only with decay)
    template <int POW>
    __device__ __forceinline__ void load_g16(float (&gt)[3]) const {
#pragma unroll
        for (int i = 0; i < 3; ++i) gt[i] = DECAY ? g16()[i] : 1.f;  // g^0, g^1, g^2
    }

    // Column sums over the rows r < L of one or two [C x D] tiles, for all threads.
    // Thread t takes an 8-column block (t % (D/8)) and every NG-th row; rows are
    // read as 16-byte vectors.  Partials combine by warp shuffles and then across
    // warps in a fixed order (deterministic), through `scr` (2 x 8 x D floats).
    //   m-sum: wlast * g^{L-1-r} * tq[r]   (weight built by multiplication from the last row)
    //   y-sum: ty[r]                       (its weights are already in the tile)
    // Results: dm[i] = sm * dm[i] + msum[i], dy[i] = sy * dy[i] + ysum[i].
    template <bool TWO>
    __device__ void tile_colsums(const uint8_t *tq, const uint8_t *ty, int L, float wlast, float *scr,
                                 float *dm, float sm, float *dy, float sy) {
        constexpr int NB = D / 8, NG = kThreads / NB;
        const int cb = tid % NB, rg = tid / NB;
        float am[8], ay[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) am[j] = ay[j] = 0.f;
        if (rg < L) {
            const int rlast = rg + ((L - 1 - rg) / NG) * NG;
            float w = wlast * gp(L - 1 - rlast);
            const float gstep = gp(NG);
            for (int r = rlast; r >= 0; r -= NG) {
                float a[8];
                tile_load_row8(tq, C, r, cb * 8, a);
#pragma unroll
                for (int j = 0; j < 8; ++j) am[j] += w * a[j];
                if constexpr (TWO) {
                    tile_load_row8(ty, C, r, cb * 8, a);
#pragma unroll
                    for (int j = 0; j < 8; ++j) ay[j] += a[j];
                }
                w *= gstep;
            }
        }
#pragma unroll
        for (int off = NB; off < 32; off <<= 1) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                am[j] += __shfl_xor_sync(0xffffffffu, am[j], off);
                if constexpr (TWO) ay[j] += __shfl_xor_sync(0xffffffffu, ay[j], off);
            }
        }
        if (lane < NB) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                scr[warp * D + cb * 8 + j] = am[j];
                if constexpr (TWO) scr[8 * D + warp * D + cb * 8 + j] = ay[j];
            }
        }
        __syncthreads();
        if (tid < D) {
            float a = 0.f, b = 0.f;
#pragma unroll
            for (int w8 = 0; w8 < kThreads / 32; ++w8) {
                a += scr[w8 * D + tid];
                if constexpr (TWO) b += scr[8 * D + w8 * D + tid];
            }
            dm[tid] = sm * dm[tid] + a;
            if constexpr (TWO) dy[tid] = sy * dy[tid] + b;
        }
        __syncthreads();
    }

    // den[t] = q_t . Y for every row t of the Q tile (all threads; partials in rsum).
    __device__ void row_dot_Y(const uint8_t *Q) { row_dot(Q, Yrun(), den()); }
    // out[r] = q_r . vec for the rows of a [C x D] tile (all threads; rsum() is
    // scratch; out is written by threads < C after an internal barrier).
    __device__ void row_dot(const uint8_t *Q, const float *vec, float *out) {
        constexpr int NPR = kThreads / C, CPT = D / NPR;
        const int r = tid % C, part = tid / C;
        float acc = 0.f;
#pragma unroll
        for (int c0 = 0; c0 < CPT; c0 += 8) {
            float q8[8];
            tile_load_row8(Q, C, r, part * CPT + c0, q8);
#pragma unroll
            for (int j = 0; j < 8; ++j) acc += q8[j] * vec[part * CPT + c0 + j];
        }
        rsum()[part * C + r] = acc;
        __syncthreads();
        if (tid < C) {
            float sacc = 0.f;
#pragma unroll
            for (int pp = 0; pp < NPR; ++pp) sacc += rsum()[pp * C + tid];
            out[tid] = sacc;
        }
    }
    // Column sums with per-row weights: dm[i] = sm * dm[i] + sum_{r < L} rw[r] t[r][i]
    // for a [C x D] tile (all threads; scr: 8 x D floats; rw in shared memory).
    __device__ void tile_colsums_rw(const uint8_t *t, int L, const float *rw, float *scr, float *dm, float sm) {
        constexpr int NB = D / 8, NG = kThreads / NB;
        const int cb = tid % NB, rg = tid / NB;
        float am[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) am[j] = 0.f;
        for (int r = rg; r < L; r += NG) {
            float a[8];
            tile_load_row8(t, C, r, cb * 8, a);
            const float w = rw[r];
#pragma unroll
            for (int j = 0; j < 8; ++j) am[j] += w * a[j];
        }
#pragma unroll
        for (int off = NB; off < 32; off <<= 1) {
#pragma unroll
            for (int j = 0; j < 8; ++j) am[j] += __shfl_xor_sync(0xffffffffu, am[j], off);
        }
        if (lane < NB) {
#pragma unroll
            for (int j = 0; j < 8; ++j) scr[warp * D + cb * 8 + j] = am[j];
        }
        __syncthreads();
        if (tid < D) {
            float a = 0.f;
#pragma unroll
            for (int w8 = 0; w8 < kThreads / 32; ++w8) a += scr[w8 * D + tid];
            dm[tid] = sm * dm[tid] + a;
        }
        __syncthreads();
    }

    // A-tilde = tril(Gamma1 o A) from TMEM W -> tA(); with ROWSUM its row partial
    // sums go to rsum() (one slot per column part).
    template <bool ROWSUM = false>
    __device__ void epi_atilde() {
        float gt[3];
        load_g16<1>(gt);
        float rs = 0.f;
        for_row<C, C>(TW, [&](int c0, float (&v)[16]) {
            if (rowC < 0) return;
            mask_row<1>(rowC, c0, v, gt);
            if constexpr (ROWSUM) {
#pragma unroll
                for (int i = 0; i < 16; ++i) rs += v[i];
            }
            tile_store_row16(tA(), C, rowC, c0, v);
        });
        if constexpr (ROWSUM) put_partial<C>(rsum(), rowC, rs);
    }

    // ======================================================================== pass 1
    // Segment summary from zero state over chunks [jb, je): TMEM S, X, C and
    // mrun() / Yrun() hold (S, X, C, m, Y) of the segment afterwards.  X, C, m, Y take
    // their decay weights relative to the segment end, g^{LB - tau} (<= 1, tau
    // the token's position in the segment), so they need no per-chunk rescaling;
    // S is rescaled per chunk because its bf16 copy feeds the next chunk.
    __device__ bool pass1(int jb, int je) {
        for (int i = tid; i < D; i += kThreads) mrun()[i] = Yrun()[i] = 0.f;
        const int LB = min(P.n, je * C) - jb * C;  // tokens in the segment
        int stage = 0;
        tma_chunk(jb, 0);
        for (int jj = jb; jj < je; ++jj) {
            const bool first = (jj == jb);
            const int L = min(C, P.n - jj * C);
            const int rest = LB - (jj - jb) * C - L;  // segment tokens after this chunk
            if (K_::NSTAGE == 1 && !first) tma_chunk(jj, 0);
            uint8_t *Q = sQ(stage), *Kt = sK(stage), *V = sV(stage);
            if (!wait_tma(stage)) return false;
            if (K_::NSTAGE == 2 && jj + 1 < je) tma_chunk(jj + 1, stage ^ 1);
            if (tid == 0) mma_kk<C, D>(TW, Q, Kt, false);  // A = Q K^T
            commit();
            // meanwhile: state at the chunk start -> bf16 copy of S, then decay S
            if (!first) {
                extract_state<D>(TS, tS(), gp(L));
                if constexpr (DECAY)  // diag(g^tau) Q
                    scaled_tile_copy<D>(Q, tQ(), [&](int r) { return gp(r + 1); });
            }
            if (!wait_mma()) return false;
            epi_atilde();
            publish();
            if (tid == 0) {
                if (!first) mma_kk<D, D>(TW, DECAY ? tQ() : Q, tS(), false);  // diag(g^tau) Q S_p
                mma_km<D, C>(TW, tA(), Kt, !first);                          // + A-tilde K
            }
            commit();
            if (!wait_mma()) return false;
            // U weighted by g^{2(LB - tau)} (the X update's left operand); K_w, V_w for decay
            {
                const float w2 = (DECAY && rowC >= 0) ? (rowC < L ? gp(2 * (rest + L - 1 - rowC)) : 0.f) : 1.f;
                for_row<C, D>(TW, [&](int c0, float (&v)[16]) {
                    if (rowC < 0) return;
                    if constexpr (DECAY) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) v[i] *= w2;
                    }
                    tile_store_row16(tU(), C, rowC, c0, v);
                });
            }
            if constexpr (DECAY) {
                scaled_tile_copy<D>(Kt, tA(), [&](int r) { return r < L ? gp(L - 1 - r) : 0.f; });
                scaled_tile_copy<DV>(V, tS(), [&](int r) { return r < L ? gp(rest + L - 1 - r) : 0.f; });
            }
            publish();
            if (tid == 0) {
                mma_mm<D>(TS, Kt, DECAY ? tA() : Kt, !first);  // S += K^T W K
                umma_commit(mma_bar3);
            } else if (tid == 32) {
                mma_mm<DV>(TX, tU(), V, !first);  // X += (W^2 U)^T V
                umma_commit(mma_bar3);
            } else if (tid == 64) {
                mma_mm<DV>(T4, Q, DECAY ? tS() : V, !first);  // C += Q^T W V
                umma_commit(mma_bar3);
            }
            if (need_mY)  // overlaps the MMAs; scratch: tQ is free once Q S_p has run
                tile_colsums<true>(Q, tU(), L, gp(rest), reinterpret_cast<float *>(tQ()), mrun(), 1.f, Yrun(), 1.f);
            if (!wait_mma3()) return false;
            stage ^= (K_::NSTAGE - 1);
        }
        return true;
    }

    // ---- accumulator shares.  A thread owns row rowD of a [D x NC] state
    // accumulator and share<NC>() consecutive columns of it, from share_col<NC>();
    // share offset c (a multiple of 16) is column share_col<NC>() + c.
    template <int NC>
    __host__ __device__ static constexpr int share() { return D == 128 ? NC / 2 : NC / 4; }
    template <int NC>
    __device__ __forceinline__ int share_col() const {
        return D == 128 ? half * (NC / 2) : half * (NC / 2) + (lane >> 4) * (NC / 4);
    }
    template <int NC>
    __device__ __forceinline__ void ld_share(uint32_t slot, int c, float (&v)[16]) {
        if constexpr (D == 128) tmem_ld16(taddr(slot, half * (NC / 2) + c), v);
        else tmem_ld16x2<NC / 4>(taddr(slot, half * (NC / 2) + c), v);
    }
    template <int NC>
    __device__ __forceinline__ void st_share(uint32_t slot, int c, const float (&v)[16]) {
        if constexpr (D == 128) tmem_st16(taddr(slot, half * (NC / 2) + c), v);
        else tmem_st16x2<NC / 4>(taddr(slot, half * (NC / 2) + c), v);
    }
    // Segment summaries keep each [D x NC] matrix in share order: the four values
    // (r, c .. c+3) sit at float offset ((c / 4) D + r) 4, so the threads of a warp,
    // which own consecutive rows, read and write consecutive 16-byte words.
    static __device__ __forceinline__ int sofs(int r, int c) { return ((c >> 2) * D + r) * 4; }
    static __device__ __forceinline__ void ld_sum16(const float *src, int r, int c, float *v) {
#pragma unroll
        for (int i = 0; i < 16; i += 4) {
            const float4 a = ldcg4(src + sofs(r, c + i));
            v[i] = a.x; v[i + 1] = a.y; v[i + 2] = a.z; v[i + 3] = a.w;
        }
    }
    template <int NC>
    __device__ void put_share(uint32_t slot, float *dst) {
        constexpr int N = share<NC>();
        float v[N];
        const int c0 = share_col<NC>();
#pragma unroll
        for (int c = 0; c < N; c += 16) ld_share<NC>(slot, c, *reinterpret_cast<float(*)[16]>(v + c));
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < N; c += 4)
            *reinterpret_cast<float4 *>(dst + sofs(rowD, c0 + c)) = make_float4(v[c], v[c + 1], v[c + 2], v[c + 3]);
    }

    // Write the summary (S, X, C, m, Y) of this CTA to `dst`.  The unmasked
    // variant keeps its running C in the X slot of TMEM and has no X, Y.
    __device__ void store_summary(float *dst) {
        float *S = dst, *X = S + D * D, *Cc = X + D * DV, *m = Cc + D * DV, *Y = m + D;
        put_share<D>(TS, S);
        if constexpr (UNM) {
            put_share<DV>(TX, Cc);
            for (int i = tid; i < D; i += kThreads) m[i] = mrun()[i];
        } else {
            put_share<DV>(TX, X);
            put_share<DV>(T4, Cc);
            for (int i = tid; i < D; i += kThreads) { m[i] = mrun()[i]; Y[i] = Yrun()[i]; }
        }
    }

    // ======================================================================== scan
    __device__ bool prefix_init() {
        if constexpr (ASYM) {  // R -> TS, P -> T4, E -> TX, m^K -> mrun(), n -> Yrun(), as stored
            if (!P.sin.S) {
                zero_slot<D, D>(TS);
                zero_slot<D, DV>(TX);
                zero_slot<D, DV>(T4);
                for (int i = tid; i < D; i += kThreads) mrun()[i] = Yrun()[i] = 0.f;
            } else {
                const float *Si = P.sin.S + (size_t)bh * D * D, *Ci = P.sin.C + (size_t)bh * D * DV;
                const float *Gi = P.sin.G + (size_t)bh * D * DV;
                auto load = [&](const float *src, int ld) {
                    return [=](int c0, float (&v)[16]) {
#pragma unroll
                        for (int i = 0; i < 16; i += 4) {
                            const float4 a = *reinterpret_cast<const float4 *>(src + rowD * ld + c0 + i);
                            v[i] = a.x; v[i + 1] = a.y; v[i + 2] = a.z; v[i + 3] = a.w;
                        }
                    };
                };
                rmw_row<D, D>(TS, load(Si, D));
                rmw_row<D, DV>(T4, load(Ci, DV));
                rmw_row<D, DV>(TX, load(Gi, DV));
                for (int i = tid; i < D; i += kThreads) {
                    mrun()[i] = P.sin.m[(size_t)bh * D + i];
                    Yrun()[i] = P.sin.h[(size_t)bh * D + i];
                }
            }
            publish();
            return true;
        }
        if constexpr (UNM) {  // S -> TS, C -> TX, m -> mrun(); G, h are not part of the state
            if (!P.sin.S) {
                zero_slot<D, D>(TS);
                zero_slot<D, DV>(TX);
                for (int i = tid; i < D; i += kThreads) mrun()[i] = 0.f;
            } else {
                const float *Si = P.sin.S + (size_t)bh * D * D, *Ci = P.sin.C + (size_t)bh * D * DV;
                const float *mi = P.sin.m + (size_t)bh * D;
                rmw_row<D, D>(TS, [&](int c0, float (&v)[16]) {
#pragma unroll
                    for (int i = 0; i < 16; i += 4) {
                        const float4 a = *reinterpret_cast<const float4 *>(Si + rowD * D + c0 + i);
                        v[i] = a.x; v[i + 1] = a.y; v[i + 2] = a.z; v[i + 3] = a.w;
                    }
                });
                rmw_row<D, DV>(TX, [&](int c0, float (&v)[16]) {
#pragma unroll
                    for (int i = 0; i < 16; i += 4) {
                        const float4 a = *reinterpret_cast<const float4 *>(Ci + rowD * DV + c0 + i);
                        v[i] = a.x; v[i + 1] = a.y; v[i + 2] = a.z; v[i + 3] = a.w;
                    }
                });
                for (int i = tid; i < D; i += kThreads) mrun()[i] = mi[i];
            }
            publish();
            return true;
        }
        if (!P.sin.S) {
            zero_slot<D, D>(TS);
            zero_slot<D, DV>(TX);
            zero_slot<D, DV>(T4);
            for (int i = tid; i < D; i += kThreads) mrun()[i] = Yrun()[i] = 0.f;
            publish();
            return true;
        }
        const float *Si = P.sin.S + (size_t)bh * D * D, *Ci = P.sin.C + (size_t)bh * D * DV;
        const float *mi = P.sin.m + (size_t)bh * D, *Gi = P.sin.G + (size_t)bh * D * DV,
                    *hi = P.sin.h + (size_t)bh * D;
        for (int i = tid; i < D; i += kThreads) mrun()[i] = mi[i];
        __syncthreads();
        float sm = 0.f;
        rmw_row<D, D>(TS, [&](int c0, float (&v)[16]) {
            if (rowD < 0) return;
#pragma unroll
            for (int i = 0; i < 16; i += 4) {
                const float4 s = *reinterpret_cast<const float4 *>(Si + rowD * D + c0 + i);
                v[i] = s.x; v[i + 1] = s.y; v[i + 2] = s.z; v[i + 3] = s.w;
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) sm += v[i] * mrun()[c0 + i];
            store_hilo(tShi(), tSlo(), D, rowD, c0, v);
        });
        rmw_row<D, DV>(T4, [&](int c0, float (&v)[16]) {
            if (rowD < 0) return;
#pragma unroll
            for (int i = 0; i < 16; i += 4) {
                const float4 s = *reinterpret_cast<const float4 *>(Ci + rowD * DV + c0 + i);
                v[i] = s.x; v[i + 1] = s.y; v[i + 2] = s.z; v[i + 3] = s.w;
            }
            store_hilo(tChi(), tClo(), D, rowD, c0, v);
        });
        put_partial<D>(part(), rowD, sm);
        publish();
        if (tid == 0) {  // X = S C (three bf16 products approximate the fp32 one)
            mma_ss(TX, tShi(), tChi(), false);
            mma_ss(TX, tShi(), tClo(), true);
            mma_ss(TX, tSlo(), tChi(), true);
        }
        commit();
        for (int i = tid; i < D; i += kThreads) Yrun()[i] = sum_partials<D>(part(), i) - hi[i];
        if (!wait_mma()) return false;
        rmw_row<D, DV>(TX, [&](int c0, float (&v)[16]) {
            if (rowD < 0) return;
#pragma unroll
            for (int i = 0; i < 16; i += 4) {
                const float4 g = *reinterpret_cast<const float4 *>(Gi + rowD * DV + c0 + i);
                v[i] -= g.x; v[i + 1] -= g.y; v[i + 2] -= g.z; v[i + 3] -= g.w;
            }
        });
        publish();
        return true;
    }

    // Spin (bounded) until pieces j0 .. j1-1 of this sequence have published their
    // summaries; the lanes of warp 0 poll the flags together.
    __device__ bool wait_flags(int j0, int j1) {
        bool ok = true;
        if (warp == 0) {
            for (int j = j0 + lane; j < j1 && ok; j += 32) {
                const unsigned *f = P.flagsw + (size_t)bh * P.kmax + j;
                ok = false;
                for (uint32_t it = 0; it < kWaitLimit; ++it) {
                    unsigned v;
                    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
                    if (v == tag) { ok = true; break; }
                    if (it > 256) __nanosleep(128);
                }
            }
            if (!ok) atomicOr(P.err, DEV_TIMEOUT);
        }
        return !__syncthreads_or(!ok);
    }

    __device__ bool wait_buf(int b) { return b == 0 ? wait_mma() : wait_mma2(); }
    __device__ void commit_buf(int b) {
        if (b == 0) commit();
        else commit2();
    }

    // prefix <- prefix (+) L_0 (+) ... (+) L_{cnt-1}, for the summaries of the first
    // `cnt` pieces of this sequence, stored one after another at Lsum; piece r
    // spans tokens [start(r), start(r+1)), with decay factor f_r = g^{len}.  One
    // fold of a summary L (factor f) into the prefix is
    //   S <- f S + S_L,  C <- f C + C_L,  m <- f m + m_L,
    //   X <- f^2 X + X_L + f S C_L,  Y <- f^2 Y + Y_L + f S m_L,
    // with S the prefix before that fold.  Unrolled over the summaries, the product
    // S C_L of step r reaches the result with weight f_r F_r^2, F_r = g^{start(cnt)
    // - start(r+1)} the decay from the end of piece r to the end of the last one.
    // The products accumulate, with that weight already on C_L, in the spare
    // accumulator, which thus needs no rescaling between steps: step r+1 runs while
    // the MMAs of step r do (two operand buffers when they fit), and its first loads
    // are issued before those MMAs.  S, C and the product-free part of X are updated
    // in place in TMEM; the sum of the products joins X at the end.  `zero_prefix`:
    // the prefix is zero and TMEM / mrun() / Yrun() are not initialised; step 0
    // sets them.
    template <typename Start>
    __device__ bool fold_all(const float *Lsum, int cnt, Start &&start, bool zero_prefix) {
        constexpr int NS = share<D>(), NV = share<DV>();
        constexpr int GW = D == 128 ? 16 : 32;  // columns per load group (register budget)
        constexpr int GS = NS < GW ? NS : GW, GV = NV < GW ? NV : GW;
        constexpr int NG = cmax(NS / GS, NV / GV);
        const int cs = share_col<D>(), cv = share_col<DV>();
        const int t_end = start(cnt);
        unsigned pend = 0u;  // bit b: MMAs committed to barrier b and not yet waited for
        bool cross = false;  // the spare accumulator holds products
        // one column group of a step: slices of S_L, m_L, C_L, X_L; m_L, Y_L entries
        float s[GS], mv[GS], cl[GV], xl[GV];
        float mLi = 0.f, YLi = 0.f;
        auto load_s = [&](int r, int g) {  // S_L, m_L slices (and the vector entries)
            const float *SL = Lsum + (size_t)r * K_::SUM, *mL = SL + D * D + 2 * D * DV;
            if (g < NS / GS) {
#pragma unroll
                for (int c = 0; c < GS; c += 16) ld_sum16(SL, rowD, cs + g * GS + c, s + c);
#pragma unroll
                for (int c = 0; c < GS; c += 4) {
                    const float4 a = ldcg4(mL + cs + g * GS + c);
                    mv[c] = a.x; mv[c + 1] = a.y; mv[c + 2] = a.z; mv[c + 3] = a.w;
                }
            }
            if (g == 0 && tid < D) {
                mLi = __ldcg(mL + tid);
                YLi = __ldcg(mL + D + tid);
            }
        };
        auto load_v = [&](int r, int g) {  // C_L, X_L slices
            const float *XL = Lsum + (size_t)r * K_::SUM + D * D, *CL = XL + D * DV;
            if (g < NV / GV) {
#pragma unroll
                for (int c = 0; c < GV; c += 16) {
                    ld_sum16(CL, rowD, cv + g * GV + c, cl + c);
                    ld_sum16(XL, rowD, cv + g * GV + c, xl + c);
                }
            }
        };
        if (cnt > 0) load_s(0, 0);
        for (int r = 0; r < cnt; ++r) {
            const int b = K_::FBUF == 2 ? (r & 1) : 0;
            const bool z = zero_prefix && r == 0;  // prefix zero: no TMEM reads, no product
            const int len = start(r + 1) - start(r);
            const float f = gp(len), f2 = f * f;
            const float coef = DECAY ? gp(len + 2 * (t_end - start(r + 1))) : 1.f;
            uint8_t *shi = fShi(b), *slo = fSlo(b), *chi = fChi(b), *clo = fClo(b);
            float sm = 0.f;
#pragma unroll
            for (int g = 0; g < NG; ++g) {
                const bool hs = g < NS / GS, hv = g < NV / GV;
                if (g > 0) load_s(r, g);
                load_v(r, g);
                // the operand buffer is free once the MMAs that read it have completed
                if (g == 0 && (pend >> b & 1u)) {
                    if (!wait_buf(b)) return false;
                    pend &= ~(1u << b);
                }
                if (hs) {  // S: old value -> operand (hi + lo), S m_L row partials, update
#pragma unroll
                    for (int c = 0; c < GS; c += 16) {
                        float v[16];
                        if (!z) {
                            ld_share<D>(TS, g * GS + c, v);
                            tmem_wait_ld();
                            store_hilo(shi, slo, D, rowD, cs + g * GS + c, v);
                        } else {
#pragma unroll
                            for (int i = 0; i < 16; ++i) v[i] = 0.f;
                        }
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            sm += v[i] * mv[c + i];
                            v[i] = f * v[i] + s[c + i];
                        }
                        st_share<D>(TS, g * GS + c, v);
                    }
                }
                if (hv) {  // C: weighted C_L -> operand, update; X without the product
#pragma unroll
                    for (int c = 0; c < GV; c += 16) {
                        float v[16], w[16];
                        if (!z) {
                            ld_share<DV>(T4, g * GV + c, v);
                            ld_share<DV>(TX, g * GV + c, w);
                            tmem_wait_ld();
                        } else {
#pragma unroll
                            for (int i = 0; i < 16; ++i) v[i] = w[i] = 0.f;
                        }
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            v[i] = f * v[i] + cl[c + i];
                            w[i] = f2 * w[i] + xl[c + i];
                            cl[c + i] *= coef;
                        }
                        if (!z) store_hilo(chi, clo, D, rowD, cv + g * GV + c, *reinterpret_cast<float(*)[16]>(cl + c));
                        st_share<DV>(T4, g * GV + c, v);
                        st_share<DV>(TX, g * GV + c, w);
                    }
                }
            }
            tmem_wait_st();
            put_partial<D>(part(b), rowD, sm);
            publish();
            const float mLc = mLi, YLc = YLi;
            if (r + 1 < cnt) load_s(r + 1, 0);  // in flight while the MMAs are issued
            if (!z) {
                if (tid == 0) {
                    mma_ss(TW, shi, chi, cross);
                    mma_ss(TW, shi, clo, true);
                    mma_ss(TW, slo, chi, true);
                }
                commit_buf(b);
                pend |= 1u << b;
                cross = true;
            }
            if (tid < D) {
                if (z) {
                    Yrun()[tid] = YLc;
                    mrun()[tid] = mLc;
                } else {
                    Yrun()[tid] = f2 * Yrun()[tid] + YLc + f * sum_partials<D>(part(b), tid);
                    mrun()[tid] = f * mrun()[tid] + mLc;
                }
            }
        }
        if ((pend & 1u) && !wait_mma()) return false;
        if ((pend & 2u) && !wait_mma2()) return false;
        if (cross) {  // X += sum of the products
            constexpr int N = share<DV>();
#pragma unroll
            for (int c = 0; c < N; c += 16) {
                float v[16], w[16];
                ld_share<DV>(TW, c, v);
                ld_share<DV>(TX, c, w);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i) w[i] += v[i];
                st_share<DV>(TX, c, w);
            }
            tmem_wait_st();
        }
        tc_sync();
        return true;
    }

    // ======================================================================== export
    // state_out = prefix (+) own summary L (f = g^{len L}).  Pass 2 carries S, X
    // (and Y with normalisation) of the prefix to the segment end, so those come
    // from TMEM afterwards; C and m, which pass 2 does not carry, and Y without
    // normalisation are combined here, before pass 2 moves the prefix on:
    // C and m go to state_out, m also to mrun() and Y to Yrun(), which pass 2 leaves alone.
    __device__ void export_pre(const float *Lown, float f) {
        const float *SL = Lown, *XL = SL + D * D, *CL = XL + D * DV, *mL = CL + D * DV, *YL = mL + D;
        (void)XL;
        float *Co = P.sout.C + (size_t)bh * D * DV, *mo = P.sout.m + (size_t)bh * D;
        constexpr int NV = share<DV>();
        const int cv = share_col<DV>();
#pragma unroll
        for (int c = 0; c < NV; c += 16) {
            float v[16], cl[16];
            ld_sum16(CL, rowD, cv + c, cl);
            ld_share<DV>(T4, c, v);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = f * v[i] + cl[i];
            st_row16(Co + rowD * DV + cv + c, v);
        }
        if constexpr (!NORM) {  // row partials of S_prefix m_L
            constexpr int NS = share<D>();
            const int cs = share_col<D>();
            float sm = 0.f;
#pragma unroll
            for (int c = 0; c < NS; c += 16) {
                float v[16];
                ld_share<D>(TS, c, v);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 16; i += 4) {
                    const float4 a = ldcg4(mL + cs + c + i);
                    sm += v[i] * a.x + v[i + 1] * a.y + v[i + 2] * a.z + v[i + 3] * a.w;
                }
            }
            put_partial<D>(part(), rowD, sm);
        }
        tc_sync();
        if (tid < D) {
            const float mLi = __ldcg(mL + tid);
            if constexpr (!NORM)
                Yrun()[tid] = f * f * Yrun()[tid] + __ldcg(YL + tid) + f * sum_partials<D>(part(), tid);
            mrun()[tid] = mo[tid] = f * mrun()[tid] + mLi;
        }
        __syncthreads();
    }

    // After pass 2: G = S C - X and h = S m - Y from the final S, X (TMEM), m, Y
    // (mrun(), Yrun()) and C (written to state_out by export_pre, read back here by
    // the threads that wrote it); S, G, h go to state_out.
    __device__ bool export_post() {
        float *So = P.sout.S + (size_t)bh * D * D, *Co = P.sout.C + (size_t)bh * D * DV;
        float *Go = P.sout.G + (size_t)bh * D * DV, *ho = P.sout.h + (size_t)bh * D;
        constexpr int NS = share<D>(), NV = share<DV>();
        const int cs = share_col<D>(), cv = share_col<DV>();
        float sm = 0.f;
#pragma unroll
        for (int c = 0; c < NS; c += 16) {
            float v[16];
            ld_share<D>(TS, c, v);
            tmem_wait_ld();
            store_hilo(tShi(), tSlo(), D, rowD, cs + c, v);
            st_row16(So + rowD * D + cs + c, v);
#pragma unroll
            for (int i = 0; i < 16; ++i) sm += v[i] * mrun()[cs + c + i];
        }
#pragma unroll
        for (int c = 0; c < NV; c += 16) {
            float v[16];
#pragma unroll
            for (int i = 0; i < 16; i += 4) {
                const float4 a = *reinterpret_cast<const float4 *>(Co + rowD * DV + cv + c + i);
                v[i] = a.x; v[i + 1] = a.y; v[i + 2] = a.z; v[i + 3] = a.w;
            }
            store_hilo(tChi(), tClo(), D, rowD, cv + c, v);
        }
        put_partial<D>(part(), rowD, sm);
        publish();
        if (tid == 0) {  // W = S C
            mma_ss(TW, tShi(), tChi(), false);
            mma_ss(TW, tShi(), tClo(), true);
            mma_ss(TW, tSlo(), tChi(), true);
        }
        commit();
        if (tid < D) ho[tid] = sum_partials<D>(part(), tid) - Yrun()[tid];
        if (!wait_mma()) return false;
#pragma unroll
        for (int c = 0; c < NV; c += 16) {
            float v[16], w[16];
            ld_share<DV>(TW, c, v);
            ld_share<DV>(TX, c, w);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] -= w[i];
            st_row16(Go + rowD * DV + cv + c, v);
        }
        return true;
    }
    // ======================================================================== pass 2
    // Outputs from the exact prefix.  Q S_p and Q X_p go to the spare columns so
    // that they overlap the epilogues; two completion barriers let the block work
    // on one group of MMA results while the next group runs.
    // With chunk >= d the next chunk's S_p fits in tU(), so S_p and X_p are extracted
    // at the end of the previous chunk; otherwise at the start of each chunk (S_p in tS()).
    static constexpr bool kTailState = C >= D;
    __device__ bool pass2(int jb, int je) {
        uint8_t *const sp_tile = kTailState ? tU() : tS();
        int stage = 0;
        tma_chunk(jb, 0);
        for (int jj = jb; jj < je; ++jj) {
            const int t0 = jj * C;
            const int L = min(C, P.n - t0);
            uint8_t *Q = sQ(stage), *Kt = sK(stage), *V = sV(stage);
            // the previous chunk's O store must have left tS() before tS() is rewritten:
            // with S_p in tS() at once, otherwise before the U epilogue (which writes
            // W^2 U there with decay), the scratch use with normalisation and the O tile
            if (!kTailState && tid == 0) bulk_wait_read();
            if (!wait_tma(stage)) return false;
            if (K_::NSTAGE == 2 && jj + 1 < je) tma_chunk(jj + 1, stage ^ 1);
            if (tid == 0) mma_kk<C, D>(TW, Q, Kt, false);  // A = Q K^T
            commit();
            if (jj == jb || !kTailState) {
                // S_p, X_p from TMEM -> bf16 operands, then S, X decay to the chunk end
                extract_state<D>(TS, sp_tile, gp(L));
                publish();
                if (tid == 0) {
                    mma_kk<D, D>(T4, Q, sp_tile, false);  // spare = Q S_p
                    umma_commit(mma_bar2);
                }
                extract_state<DV>(TX, tQ(), gp(2 * L));
            } else if (tid == 32) {  // S_p, X_p were extracted at the end of the previous chunk
                mma_kk<D, D>(T4, Q, sp_tile, false);  // spare = Q S_p, beside thread 0's issue
                umma_commit(mma_bar2);
            }
            if constexpr (NORM) row_dot_Y(Q);  // q . Y_p for the denominator
            if (!wait_mma()) return false;  // A
            epi_atilde();
            publish();
            if (tid == 0) mma_km<D, C>(TW, tA(), Kt, false);  // W = A-tilde K
            commit();
            if (kTailState && tid == 0) bulk_wait_read();  // ordered by the barriers of the waits
            if (!wait_mma2()) return false;  // Q S_p
            if (!wait_mma()) return false;   // A-tilde K
            // U = g^tau Q S_p + A-tilde K -> tU(); W^2 U -> tS() (decay)
            {
                const float gt = (DECAY && rowC >= 0) ? gp(rowC + 1) : 1.f;
                const float w2 = (rowC >= 0 && rowC < L) ? gp(2 * (L - 1 - rowC)) : 0.f;
                for_row2<C, D>(TW, T4, [&](int c0, float (&v)[16], float (&sp)[16]) {
                    if (rowC < 0) return;
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] += gt * sp[i];
                    tile_store_row16(tU(), C, rowC, c0, v);
                    if constexpr (DECAY) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) v[i] *= w2;
                        tile_store_row16(tS(), C, rowC, c0, v);
                    }
                });
            }
            if constexpr (DECAY)
                scaled_tile_copy<D>(Kt, tA(), [&](int r) { return r < L ? gp(L - 1 - r) : 0.f; });
            publish();
            // M = Q U^T and, with decay, S += K^T W K (it reads tA(), which the M
            // epilogue rewrites) on the first barrier; the other products fan out
            if (tid == 0) {
                mma_kk<C, D>(TW, Q, tU(), false);                        // M = Q U^T
                if constexpr (DECAY) mma_mm<D>(TS, Kt, tA(), true);       // S += K^T W K
                umma_commit(mma_bar);
            } else if (tid == 32) {
                if constexpr (DECAY) arrive3();
                else {
                    mma_mm<D>(TS, Kt, Kt, true);  // S += K^T K
                    umma_commit(mma_bar3);
                }
            } else if (tid == 64) {
                mma_mm<DV>(TX, DECAY ? tS() : tU(), V, true);  // X += (W^2 U)^T V
                umma_commit(mma_bar3);
            } else if (tid == 96) {
                mma_km<DV, D>(T4, Q, tQ(), false);  // spare = Q X_p
                umma_commit(mma_bar3);
            }
            // Y <- g^{2L} Y + sum_b w_b^2 u_b (weights already on the tile)
            float ay = 0.f;
            float *ysc = rsum();  // rsum is free until the M epilogue
            if constexpr (NORM && !DECAY) {
                // scratch: tS() is free here (S_p, when it is there, has been read by Q S_p)
                tile_colsums<false>(tU(), nullptr, L, 1.f, reinterpret_cast<float *>(tS()), Yrun(), gp(2 * L),
                                    nullptr, 1.f);
            } else if constexpr (NORM) {
                // with decay tS holds W^2 U, read by the X update in flight: two row groups
                const int i = tid % D, g = tid / D;
                if (g < 2)
                    for (int b = g; b < L; b += 2) ay += tile_load(tS(), C, b, i);
                if (g == 1) ysc[i] = ay;
            }
            if (!wait_mma()) return false;  // M (and the S update with decay)
            if constexpr (NORM && DECAY) {
                if (tid < D) Yrun()[tid] = gp(2 * L) * Yrun()[tid] + (ay + ysc[tid]);
                __syncthreads();  // rsum is rewritten by the M epilogue
            }
            // M = tril(Gamma2 o Q U^T) -> tA(), row sums for the denominator
            {
                float rs = 0.f;
                float gt2[3];
                load_g16<2>(gt2);
                for_row<C, C>(TW, [&](int c0, float (&v)[16]) {
                    if (rowC < 0) return;
                    mask_row<2>(rowC, c0, v, gt2);
                    if constexpr (NORM) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) rs += v[i];
                    }
                    tile_store_row16(tA(), C, rowC, c0, v);
                });
                if constexpr (NORM) put_partial<C>(rsum(), rowC, rs);
            }
            publish();
            if (tid == 0) mma_km<DV, C>(TW, tA(), V, false);  // O = M V
            commit();
            if (!wait_mma3()) return false;  // X, S updates and Q X_p
            if (!wait_mma()) return false;   // M V
            // Q, K, V of this chunk are no longer read: with one input stage, start the
            // next chunk's load now so that it overlaps the output epilogue
            if (K_::NSTAGE == 1 && jj + 1 < je) tma_chunk(jj + 1, 0);
            {
                const float g2t = (DECAY && rowC >= 0) ? gp(2 * (rowC + 1)) : 1.f;
                float inv = 1.f;
                if constexpr (NORM) {
                    if (rowC >= 0) inv = 1.f / (sum_partials<C>(rsum(), rowC) + g2t * den()[rowC] + P.eps);
                }
                // O tile -> tS() (free: its last reader, the X update, has completed),
                // then one TMA store; rows past the sequence end are not written
                for_row2<C, DV>(TW, T4, [&](int c0, float (&v)[16], float (&sp)[16]) {
                    if (rowC < 0) return;
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] = (v[i] + g2t * sp[i]) * inv;
                    tile_store_row16(tS(), C, rowC, c0, v);
                });
            }
            if (kTailState && jj + 1 < je) {
                // the next chunk's S_p, X_p -> tU(), tQ() (their last readers, M, the X
                // update and Q X_p, have completed), then S, X decay to its end
                const int Ln = min(C, P.n - (jj + 1) * C);
                extract_state<D>(TS, tU(), gp(Ln));
                extract_state<DV>(TX, tQ(), gp(2 * Ln));
            }
            publish();  // tile writes visible to the TMA and the next MMAs; TMEM reads done
            if (tid == 0) {
#pragma unroll
                for (int kb = 0; kb < DV / 64; ++kb) tma_store_3d(tS() + kb * C * 128, &P.tmO, kb * 64, t0, bh);
                bulk_commit();
            }
            stage ^= (K_::NSTAGE - 1);
        }
        if (tid == 0) bulk_wait_read();  // tS() and the arena are free again after this barrier
        __syncthreads();
        return true;
    }

    // ======================================================================== unmasked variant
    // o_t = q_t^T S_t C_t = u_t^T C_t with u_t = S_t q_t (skill card "Higher-order
    // linear attention", bullet "Streaming Computation").  Per chunk, with U as in
    // the masked path:
    //   M' = tril(Gamma1 o U Q^T),   O = M' V + diag(g^tau) U C_p,
    //   den = rowsum(M') + diag(g^tau) U m_p,
    // and S, C, m move to the chunk end.  TMEM: work W, S, C (in the X slot), spare.

    // Pass 1: the piece's S, C, m from zero; every weight is relative to the piece
    // end (g^{LB - tau}), so nothing is rescaled per chunk and no U is needed.
    __device__ bool pass1_unm(int jb, int je) {
        for (int i = tid; i < D; i += kThreads) mrun()[i] = 0.f;
        const int LB = min(P.n, je * C) - jb * C;
        int stage = 0;
        tma_chunk(jb, 0);
        for (int jj = jb; jj < je; ++jj) {
            const bool first = (jj == jb);
            const int L = min(C, P.n - jj * C);
            const int rest = LB - (jj - jb) * C - L;
            if (K_::NSTAGE == 1 && !first) tma_chunk(jj, 0);
            uint8_t *Q = sQ(stage), *Kt = sK(stage), *V = sV(stage);
            if (!wait_tma(stage)) return false;
            if (K_::NSTAGE == 2 && jj + 1 < je) tma_chunk(jj + 1, stage ^ 1);
            if constexpr (DECAY) {  // K_w, V_w: rows weighted by g^{rest + L - 1 - tau}
                scaled_tile_copy<D>(Kt, tA(), [&](int r) { return r < L ? gp(rest + L - 1 - r) : 0.f; });
                scaled_tile_copy<DV>(V, tS(), [&](int r) { return r < L ? gp(rest + L - 1 - r) : 0.f; });
            }
            publish();
            if (tid == 0) {
                mma_mm<D>(TS, Kt, DECAY ? tA() : Kt, !first);  // S += K^T W K
                mma_mm<DV>(TX, Q, DECAY ? tS() : V, !first);   // C += Q^T W V
            }
            commit();
            if (need_mY)  // m += sum_tau g^{rest + L - 1 - tau} q_tau; scratch: tQ
                tile_colsums<false>(Q, nullptr, L, gp(rest), reinterpret_cast<float *>(tQ()), mrun(), 1.f,
                                    nullptr, 1.f);
            if (!wait_mma()) return false;
            stage ^= (K_::NSTAGE - 1);
        }
        return true;
    }

    // prefix <- prefix (+) L_0 (+) ... (+) L_{cnt-1} for the unmasked state: the
    // linear part of the concatenation rule, S <- f S + S_L, C <- f C + C_L,
    // m <- f m + m_L (f = g^{len L}).  `zero_prefix`: step 0 sets the prefix.
    template <typename Start>
    __device__ bool fold_unm(const float *Lsum, int cnt, Start &&start, bool zero_prefix) {
        constexpr int NS = share<D>(), NV = share<DV>();
        const int cs = share_col<D>(), cv = share_col<DV>();
        for (int r = 0; r < cnt; ++r) {
            const float *SL = Lsum + (size_t)r * K_::SUM, *CL = SL + D * D + D * DV, *mL = CL + D * DV;
            const float f = gp(start(r + 1) - start(r));
            const bool z = zero_prefix && r == 0;
            const float mLi = tid < D ? __ldcg(mL + tid) : 0.f;
#pragma unroll
            for (int c = 0; c < NS; c += 16) {
                float s[16], v[16];
                ld_sum16(SL, rowD, cs + c, s);
                if (!z) {
                    ld_share<D>(TS, c, v);
                    tmem_wait_ld();
                }
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] = z ? s[i] : f * v[i] + s[i];
                st_share<D>(TS, c, v);
            }
#pragma unroll
            for (int c = 0; c < NV; c += 16) {
                float s[16], v[16];
                ld_sum16(CL, rowD, cv + c, s);
                if (!z) {
                    ld_share<DV>(TX, c, v);
                    tmem_wait_ld();
                }
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] = z ? s[i] : f * v[i] + s[i];
                st_share<DV>(TX, c, v);
            }
            tmem_wait_st();
            if (tid < D) mrun()[tid] = z ? mLi : f * mrun()[tid] + mLi;
        }
        tc_sync();
        return true;
    }

    // State export, part 1 (unmasked): pass 2 carries S and C (and m with
    // normalisation) to the sequence end; without normalisation m is combined
    // here: m = f m_prefix + m_L -> mrun() and state_out.
    __device__ void export_pre_unm(const float *Lown, float f) {
        if constexpr (!NORM) {
            const float *mL = Lown + D * D + 2 * D * DV;
            float *mo = P.sout.m + (size_t)bh * D;
            if (tid < D) mrun()[tid] = mo[tid] = f * mrun()[tid] + __ldcg(mL + tid);
            __syncthreads();
        }
    }

    // State export, part 2 (unmasked): S, C, m at the sequence end; G and h are
    // not part of this variant and are written as zeros.
    __device__ void export_post_unm() {
        float *So = P.sout.S + (size_t)bh * D * D, *Co = P.sout.C + (size_t)bh * D * DV;
        float *mo = P.sout.m + (size_t)bh * D, *Go = P.sout.G + (size_t)bh * D * DV, *ho = P.sout.h + (size_t)bh * D;
        constexpr int NS = share<D>(), NV = share<DV>();
        const int cs = share_col<D>(), cv = share_col<DV>();
#pragma unroll
        for (int c = 0; c < NS; c += 16) {
            float v[16];
            ld_share<D>(TS, c, v);
            tmem_wait_ld();
            st_row16(So + rowD * D + cs + c, v);
        }
#pragma unroll
        for (int c = 0; c < NV; c += 16) {
            float v[16], zero[16];
            ld_share<DV>(TX, c, v);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) zero[i] = 0.f;
            st_row16(Co + rowD * DV + cv + c, v);
            st_row16(Go + rowD * DV + cv + c, zero);
        }
        for (int i = tid; i < D; i += kThreads) { mo[i] = mrun()[i]; ho[i] = 0.f; }
    }

    // Pass 2 (unmasked): outputs from the exact prefix (S in TS, C in TX, m).
    __device__ bool pass2_unm(int jb, int je) {
        int stage = 0;
        tma_chunk(jb, 0);
        for (int jj = jb; jj < je; ++jj) {
            const int t0 = jj * C;
            const int L = min(C, P.n - t0);
            uint8_t *Q = sQ(stage), *Kt = sK(stage), *V = sV(stage);
            if (tid == 0) bulk_wait_read();  // the previous chunk's O store has left tS()
            if (!wait_tma(stage)) return false;
            if (K_::NSTAGE == 2 && jj + 1 < je) tma_chunk(jj + 1, stage ^ 1);
            if (tid == 0) mma_kk<C, D>(TW, Q, Kt, false);  // A = Q K^T
            commit();
            // meanwhile: S_p -> bf16 operand, then decay S to the chunk end
            extract_state<D>(TS, tS(), gp(L));
            publish();
            if (tid == 0) mma_kk<D, D>(T4, Q, tS(), false);  // spare = Q S_p
            commit2();
            // meanwhile: C_p -> bf16 operand (rows d, MN-major for U C_p), decay C
            extract_state<DV>(TX, tQ(), gp(L));
            if (!wait_mma()) return false;  // A
            epi_atilde();
            publish();
            if (tid == 0) mma_km<D, C>(TW, tA(), Kt, false);  // W = A-tilde K
            commit();
            if (!wait_mma2()) return false;  // Q S_p
            if (!wait_mma()) return false;   // A-tilde K
            // U = g^tau Q S_p + A-tilde K -> tU(); with normalisation, row partials of
            // u_t . m_p (into rsum(), free until the M' epilogue)
            {
                const float gt = (DECAY && rowC >= 0) ? gp(rowC + 1) : 1.f;
                float um = 0.f;
                for_row2<C, D>(TW, T4, [&](int c0, float (&v)[16], float (&sp)[16]) {
                    if (rowC < 0) return;
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        v[i] += gt * sp[i];
                        if constexpr (NORM) um += v[i] * mrun()[c0 + i];
                    }
                    tile_store_row16(tU(), C, rowC, c0, v);
                });
                if constexpr (NORM) put_partial<C>(rsum(), rowC, um);
            }
            if constexpr (DECAY) {  // K_w, V_w: rows weighted by g^{L - 1 - tau}
                scaled_tile_copy<D>(Kt, tA(), [&](int r) { return r < L ? gp(L - 1 - r) : 0.f; });
                scaled_tile_copy<DV>(V, tS(), [&](int r) { return r < L ? gp(L - 1 - r) : 0.f; });
            }
            publish();
            if (tid == 0) {
                mma_kk<C, D>(TW, tU(), Q, false);             // M' = U Q^T
                mma_mm<D>(TS, Kt, DECAY ? tA() : Kt, true);   // S += K^T W K (reads tA(): done before
            }                                                // the M' epilogue rewrites tA())
            commit();
            if (tid == 0) {
                mma_mm<DV>(TX, Q, DECAY ? tS() : V, true);    // C += Q^T W V
                mma_km<DV, D>(T4, tU(), tQ(), false);         // spare = U C_p
            }
            commit2();
            if constexpr (NORM) {  // den = u . m_p, before m moves on
                if (tid < C) den()[tid] = sum_partials<C>(rsum(), tid);
            }
            if (!wait_mma()) return false;  // M' and the S update
            // M' = tril(Gamma1 o U Q^T) -> tA(), row sums for the denominator
            {
                float rs = 0.f;
                float gt1[3];
                load_g16<1>(gt1);
                for_row<C, C>(TW, [&](int c0, float (&v)[16]) {
                    if (rowC < 0) return;
                    mask_row<1>(rowC, c0, v, gt1);
                    if constexpr (NORM) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) rs += v[i];
                    }
                    tile_store_row16(tA(), C, rowC, c0, v);
                });
                if constexpr (NORM) put_partial<C>(rsum(), rowC, rs);
            }
            publish();
            if (tid == 0) mma_km<DV, C>(TW, tA(), V, false);  // O = M' V
            commit();
            if (!wait_mma2()) return false;  // C update and U C_p
            if (!wait_mma()) return false;   // M' V
            if constexpr (NORM)  // m <- g^L m + sum_tau g^{L - 1 - tau} q_tau (scratch: tQ, read by U C_p)
                tile_colsums<false>(Q, nullptr, L, 1.f, reinterpret_cast<float *>(tQ()), mrun(), gp(L), nullptr,
                                    1.f);
            if (K_::NSTAGE == 1 && jj + 1 < je) tma_chunk(jj + 1, 0);
            {
                const float g1t = (DECAY && rowC >= 0) ? gp(rowC + 1) : 1.f;
                float inv = 1.f;
                if constexpr (NORM) {
                    if (rowC >= 0) inv = 1.f / (sum_partials<C>(rsum(), rowC) + g1t * den()[rowC] + P.eps);
                }
                for_row2<C, DV>(TW, T4, [&](int c0, float (&v)[16], float (&sp)[16]) {
                    if (rowC < 0) return;
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] = (v[i] + g1t * sp[i]) * inv;
                    tile_store_row16(tS(), C, rowC, c0, v);
                });
            }
            publish();
            if (tid == 0) {
#pragma unroll
                for (int kb = 0; kb < DV / 64; ++kb) tma_store_3d(tS() + kb * C * 128, &P.tmO, kb * 64, t0, bh);
                bulk_commit();
            }
            stage ^= (K_::NSTAGE - 1);
        }
        if (tid == 0) bulk_wait_read();
        __syncthreads();
        return true;
    }

    // ======================================================================== asymmetric variant
    // AHLA (gist.science summary, section 2): o_t = sum_{a<=b<=t} (q_t.k_b)(q_b.k_a) v_a
    // = q_t^T E_t.  Per chunk, with A-tilde as in the masked path and the state
    // (P_p, E_p, m_p, n_p) at the chunk start:
    //   Z    = A-tilde V + diag(g^tau) Q P_p          (rows z_b = P_b^T q_b)
    //   zeta = rowsum(A-tilde) + diag(g^tau) Q m_p    (zeta_b = q_b . m^K_b)
    //   O    = A-tilde Z + diag(g^tau) Q E_p,  den = A-tilde zeta + diag(g^tau) Q n_p
    //   P <- g^L P + K^T W V,  E <- g^L E + K^T W Z,  m^K <- g^L m^K + K^T w,
    //   n <- g^L n + K^T W zeta,  R <- R + K^T Q  (W = diag(g^{L - tau})).
    // TMEM: work W (A, Z, O), R in the S slot (spare in pass 2), E in the X slot,
    // P in the fourth slot; m^K in mrun(), n in Yrun().  Requires dv <= d.
    //   zeta, and n, are formed only when the normaliser or the state is wanted.

    // Pass 1: the piece's R, P, E, m^K, n from zero.  P and m^K are rescaled per
    // chunk (their values at the chunk start feed the next chunk); E and n take
    // weights relative to the piece end; R has no decay.
    __device__ bool pass1_asym(int jb, int je) {
        for (int i = tid; i < D; i += kThreads) mrun()[i] = Yrun()[i] = 0.f;
        const int LB = min(P.n, je * C) - jb * C;
        int stage = 0;
        tma_chunk(jb, 0);
        for (int jj = jb; jj < je; ++jj) {
            const bool first = (jj == jb);
            const int L = min(C, P.n - jj * C);
            const int rest = LB - (jj - jb) * C - L;
            if (K_::NSTAGE == 1 && !first) tma_chunk(jj, 0);
            uint8_t *Q = sQ(stage), *Kt = sK(stage), *V = sV(stage);
            if (!wait_tma(stage)) return false;
            if (K_::NSTAGE == 2 && jj + 1 < je) tma_chunk(jj + 1, stage ^ 1);
            if (tid == 0) mma_kk<C, D>(TW, Q, Kt, false);  // A = Q K^T
            commit();
            if (!first) {  // P_p -> bf16 operand, P decayed to the chunk end; diag(g^tau) Q
                extract_state<DV>(T4, tQ(), gp(L));
                if constexpr (DECAY) scaled_tile_copy<D>(Q, tS(), [&](int r) { return gp(r + 1); });
            }
            if (need_mY) row_dot(Q, mrun(), den());  // q_b . m_p (m local to the piece)
            if (!wait_mma()) return false;
            epi_atilde<true>();
            publish();
            if (tid == 0) {
                mma_km<DV, C>(TW, tA(), V, false);                                    // A-tilde V
                if (!first) mma_km<DV, D>(TW, DECAY ? tS() : Q, tQ(), true);         // + diag(g^tau) Q P_p
            }
            commit();
            if (need_mY && tid < C) {  // zeta_b (in den()), then the weight of k_b in n
                const float zeta = sum_partials<C>(rsum(), tid) + (first ? 0.f : gp(tid + 1) * den()[tid]);
                den()[tid] = tid < L ? gp(rest + L - 1 - tid) * zeta : 0.f;
            }
            if (!wait_mma()) return false;
            // Z -> tU() with the piece-end factor g^rest (E's weights are g^{rest} W)
            {
                const float zs = DECAY ? gp(rest) : 1.f;
                for_row<C, DV>(TW, [&](int c0, float (&v)[16]) {
                    if (rowC < 0) return;
                    if constexpr (DECAY) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) v[i] *= zs;
                    }
                    tile_store_row16(tU(), C, rowC, c0, v);
                });
            }
            if constexpr (DECAY)  // K_w = diag(g^{L-1-tau}) K
                scaled_tile_copy<D>(Kt, tA(), [&](int r) { return r < L ? gp(L - 1 - r) : 0.f; });
            publish();
            if (tid == 0) {
                mma_mm<DV>(T4, DECAY ? tA() : Kt, V, !first);    // P += K^T W V
                mma_mm<DV>(TX, DECAY ? tA() : Kt, tU(), !first); // E += g^rest K^T W Z
                mma_mm<D>(TS, Kt, Q, !first);                    // R += K^T Q
            }
            commit();
            if (need_mY) {  // n += sum_b g^{rest+L-1-b} zeta_b k_b; m^K <- g^L m^K + sum_b g^{L-1-b} k_b
                tile_colsums_rw(Kt, L, den(), reinterpret_cast<float *>(tQ()), Yrun(), 1.f);
                tile_colsums<false>(Kt, nullptr, L, 1.f, reinterpret_cast<float *>(tQ()), mrun(), gp(L), nullptr,
                                    1.f);
            }
            if (!wait_mma()) return false;
            stage ^= (K_::NSTAGE - 1);
        }
        return true;
    }

    // prefix <- prefix (+) L_0 (+) ... (+) L_{cnt-1} by the asymmetric rule
    //   R <- R + R_L,  P <- f P + P_L,  m^K <- f m^K + m_L,
    //   E <- f E + E_L + f R_L P,   n <- f n + n_L + f R_L m^K   (P, m^K before the step).
    // Unrolled, the product of step r reaches the result with weight
    // g^{start(cnt) - start(r)}; it accumulates, weighted, in the spare accumulator
    // (R_L from the summary as the A operand, the old P from TMEM as B), as in the
    // masked fold; step r+1 runs while the MMAs of step r do.
    template <typename Start>
    __device__ bool fold_asym(const float *Lsum, int cnt, Start &&start, bool zero_prefix) {
        constexpr int NS = share<D>(), NV = share<DV>();
        const int cs = share_col<D>(), cv = share_col<DV>();
        const int t_end = start(cnt);
        unsigned pend = 0u;
        bool cross = false;
        for (int r = 0; r < cnt; ++r) {
            const float *RL = Lsum + (size_t)r * K_::SUM, *EL = RL + D * D, *PL = EL + D * DV, *mL = PL + D * DV,
                        *nL = mL + D;
            const int b = K_::FBUF == 2 ? (r & 1) : 0;
            const bool z = zero_prefix && r == 0;
            const float f = gp(start(r + 1) - start(r));
            const float coef = DECAY ? gp(t_end - start(r)) : 1.f;
            uint8_t *shi = fShi(b), *slo = fSlo(b), *chi = fChi(b), *clo = fClo(b);
            const float mLi = tid < D ? __ldcg(mL + tid) : 0.f, nLi = tid < D ? __ldcg(nL + tid) : 0.f;
            if (pend >> b & 1u) {
                if (!wait_buf(b)) return false;
                pend &= ~(1u << b);
            } else if (r > 0) {
                __syncthreads();  // every thread's m^K update of the last step precedes the reads below
            }
            float rm = 0.f;  // row partial of R_L m_old
#pragma unroll
            for (int c = 0; c < NS; c += 16) {  // R: R_L -> operand (hi + lo), R += R_L
                float rl[16], v[16];
                ld_sum16(RL, rowD, cs + c, rl);
                if (!z) {
                    ld_share<D>(TS, c, v);
                    tmem_wait_ld();
                }
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    rm += rl[i] * (z ? 0.f : mrun()[cs + c + i]);
                    v[i] = z ? rl[i] : v[i] + rl[i];
                }
                if (!z) store_hilo(shi, slo, D, rowD, cs + c, rl);
                st_share<D>(TS, c, v);
            }
#pragma unroll
            for (int c = 0; c < NV; c += 16) {  // P: weighted old P -> operand, update; E without the product
                float pl[16], el[16], v[16], w[16];
                ld_sum16(PL, rowD, cv + c, pl);
                ld_sum16(EL, rowD, cv + c, el);
                if (!z) {
                    ld_share<DV>(T4, c, v);
                    ld_share<DV>(TX, c, w);
                    tmem_wait_ld();
                }
                float o[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    o[i] = z ? 0.f : coef * v[i];
                    v[i] = z ? pl[i] : f * v[i] + pl[i];
                    w[i] = z ? el[i] : f * w[i] + el[i];
                }
                if (!z) store_hilo(chi, clo, D, rowD, cv + c, o);
                st_share<DV>(T4, c, v);
                st_share<DV>(TX, c, w);
            }
            tmem_wait_st();
            put_partial<D>(part(b), rowD, rm);
            publish();
            if (!z) {
                if (tid == 0) {
                    mma_ss(TW, shi, chi, cross);
                    mma_ss(TW, shi, clo, true);
                    mma_ss(TW, slo, chi, true);
                }
                commit_buf(b);
                pend |= 1u << b;
                cross = true;
            }
            if (tid < D) {
                if (z) {
                    Yrun()[tid] = nLi;
                    mrun()[tid] = mLi;
                } else {
                    Yrun()[tid] = f * Yrun()[tid] + nLi + f * sum_partials<D>(part(b), tid);
                    mrun()[tid] = f * mrun()[tid] + mLi;
                }
            }
        }
        if ((pend & 1u) && !wait_mma()) return false;
        if ((pend & 2u) && !wait_mma2()) return false;
        if (cross) {  // E += sum of the products
            constexpr int N = share<DV>();
#pragma unroll
            for (int c = 0; c < N; c += 16) {
                float v[16], w[16];
                ld_share<DV>(TW, c, v);
                ld_share<DV>(TX, c, w);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i) w[i] += v[i];
                st_share<DV>(TX, c, w);
            }
            tmem_wait_st();
        }
        tc_sync();
        return true;
    }

    // State export, part 1 (asymmetric): R = R_prefix + R_L to state_out now (pass 2
    // uses its slot); without the normaliser also m^K = f m_p + m_L and
    // n = f n_p + n_L + f R_L m_p (pass 2 carries P, E, and m^K, n when normalising).
    __device__ void export_pre_asym(const float *Lown, float f) {
        const float *RL = Lown, *mL = Lown + D * D + 2 * D * DV, *nL = mL + D;
        float *Ro = P.sout.S + (size_t)bh * D * D;
        constexpr int NS = share<D>();
        const int cs = share_col<D>();
        float rm = 0.f;
#pragma unroll
        for (int c = 0; c < NS; c += 16) {
            float rl[16], v[16];
            ld_sum16(RL, rowD, cs + c, rl);
            ld_share<D>(TS, c, v);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                rm += rl[i] * mrun()[cs + c + i];
                v[i] += rl[i];
            }
            st_row16(Ro + rowD * D + cs + c, v);
        }
        if constexpr (!NORM) put_partial<D>(part(), rowD, rm);
        tc_sync();
        if constexpr (!NORM) {
            if (tid < D) {
                const float mp = mrun()[tid];
                Yrun()[tid] = f * Yrun()[tid] + __ldcg(nL + tid) + f * sum_partials<D>(part(), tid);
                mrun()[tid] = f * mp + __ldcg(mL + tid);
            }
            __syncthreads();
        }
    }

    // State export, part 2 (asymmetric): P, E, m^K, n at the sequence end.
    __device__ void export_post_asym() {
        float *Co = P.sout.C + (size_t)bh * D * DV, *Go = P.sout.G + (size_t)bh * D * DV;
        constexpr int NV = share<DV>();
        const int cv = share_col<DV>();
#pragma unroll
        for (int c = 0; c < NV; c += 16) {
            float v[16], w[16];
            ld_share<DV>(T4, c, v);
            ld_share<DV>(TX, c, w);
            tmem_wait_ld();
            st_row16(Co + rowD * DV + cv + c, v);
            st_row16(Go + rowD * DV + cv + c, w);
        }
        for (int i = tid; i < D; i += kThreads) {
            P.sout.m[(size_t)bh * D + i] = mrun()[i];
            P.sout.h[(size_t)bh * D + i] = Yrun()[i];
        }
    }

    // Pass 2 (asymmetric): outputs from the exact prefix (P in the fourth slot, E in
    // the X slot, m^K, n).  The S slot is the spare accumulator here.  With the
    // normaliser: den() holds q_b . m_p, then zeta_b, then the weight of k_b in the
    // n update; rsum() holds row partials, then den_t in its first C entries.
    __device__ bool pass2_asym(int jb, int je) {
        int stage = 0;
        tma_chunk(jb, 0);
        for (int jj = jb; jj < je; ++jj) {
            const int t0 = jj * C;
            const int L = min(C, P.n - t0);
            uint8_t *Q = sQ(stage), *Kt = sK(stage), *V = sV(stage);
            if (tid == 0) bulk_wait_read();  // the previous chunk's O store has left tS()
            if (!wait_tma(stage)) return false;
            if (K_::NSTAGE == 2 && jj + 1 < je) tma_chunk(jj + 1, stage ^ 1);
            if (tid == 0) mma_kk<C, D>(TW, Q, Kt, false);  // A = Q K^T
            commit();
            extract_state<DV>(T4, tQ(), gp(L));  // P_p -> bf16, P decayed to the chunk end
            publish();
            if (tid == 0) mma_km<DV, D>(TS, Q, tQ(), false);  // spare = Q P_p
            commit2();
            extract_state<DV>(TX, tS(), gp(L));  // E_p -> bf16, E decayed to the chunk end
            if constexpr (NORM) row_dot(Q, mrun(), den());  // q_b . m_p
            if (!wait_mma()) return false;  // A
            epi_atilde<NORM>();
            publish();
            if (tid == 0) mma_km<DV, C>(TW, tA(), V, false);  // A-tilde V
            commit();
            if constexpr (NORM) {  // zeta_b = rowsum(A-tilde)_b + g^tau q_b . m_p
                if (tid < C) den()[tid] = sum_partials<C>(rsum(), tid) + gp(tid + 1) * den()[tid];
            }
            if (!wait_mma2()) return false;  // Q P_p
            if (!wait_mma()) return false;   // A-tilde V
            // Z = A-tilde V + g^tau Q P_p -> tU()
            {
                const float gt = (DECAY && rowC >= 0) ? gp(rowC + 1) : 1.f;
                for_row2<C, DV>(TW, TS, [&](int c0, float (&v)[16], float (&sp)[16]) {
                    if (rowC < 0) return;
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] += gt * sp[i];
                    tile_store_row16(tU(), C, rowC, c0, v);
                });
            }
            if constexpr (DECAY)  // K_w = diag(g^{L-1-tau}) K -> tQ (P_p has been read)
                scaled_tile_copy<D>(Kt, tQ(), [&](int r) { return r < L ? gp(L - 1 - r) : 0.f; });
            publish();
            if (tid == 0) mma_km<DV, C>(TW, tA(), tU(), false);  // O = A-tilde Z
            commit();
            if (tid == 0) {
                mma_km<DV, D>(TS, Q, tS(), false);               // spare = Q E_p
                mma_mm<DV>(T4, DECAY ? tQ() : Kt, V, true);      // P += K^T W V
                mma_mm<DV>(TX, DECAY ? tQ() : Kt, tU(), true);   // E += K^T W Z
            }
            commit2();
            if constexpr (NORM) {
                // den_t = sum_b A-tilde[t,b] zeta_b + g^tau q_t . n_p: one partial per
                // (row, part) over C / NPR columns of A-tilde and D / NPR of q (tA read only)
                constexpr int NPR = kThreads / C, CA = C / NPR, CQ = D / NPR;
                const int r = tid % C, pp = tid / C;
                float acc = 0.f, accq = 0.f;
#pragma unroll
                for (int c0 = 0; c0 < CA; c0 += 8) {
                    float a8[8];
                    tile_load_row8(tA(), C, r, pp * CA + c0, a8);
#pragma unroll
                    for (int j = 0; j < 8; ++j) acc += a8[j] * den()[pp * CA + c0 + j];
                }
#pragma unroll
                for (int c0 = 0; c0 < CQ; c0 += 8) {
                    float q8[8];
                    tile_load_row8(Q, C, r, pp * CQ + c0, q8);
#pragma unroll
                    for (int j = 0; j < 8; ++j) accq += q8[j] * Yrun()[pp * CQ + c0 + j];
                }
                rsum()[pp * C + r] = acc + (DECAY ? gp(r + 1) : 1.f) * accq;
                __syncthreads();
                if (tid < C) {
                    float sacc = 0.f;
#pragma unroll
                    for (int q2 = 0; q2 < NPR; ++q2) sacc += rsum()[q2 * C + tid];
                    rsum()[tid] = sacc;
                    den()[tid] = tid < L ? gp(L - 1 - tid) * den()[tid] : 0.f;  // weight of k_b in n
                }
            }
            if (!wait_mma()) return false;   // O = A-tilde Z
            if (!wait_mma2()) return false;  // Q E_p, P and E updates
            if constexpr (NORM) {  // n, m^K to the chunk end (scratch: tA, whose readers have finished)
                tile_colsums_rw(Kt, L, den(), reinterpret_cast<float *>(tA()), Yrun(), gp(L));
                tile_colsums<false>(Kt, nullptr, L, 1.f, reinterpret_cast<float *>(tA()), mrun(), gp(L), nullptr,
                                    1.f);
            }
            if (K_::NSTAGE == 1 && jj + 1 < je) tma_chunk(jj + 1, 0);
            {
                const float g1t = (DECAY && rowC >= 0) ? gp(rowC + 1) : 1.f;
                float inv = 1.f;
                if constexpr (NORM) {
                    if (rowC >= 0) inv = 1.f / (rsum()[rowC] + P.eps);
                }
                for_row2<C, DV>(TW, TS, [&](int c0, float (&v)[16], float (&sp)[16]) {
                    if (rowC < 0) return;
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] = (v[i] + g1t * sp[i]) * inv;
                    tile_store_row16(tS(), C, rowC, c0, v);
                });
            }
            publish();
            if (tid == 0) {
#pragma unroll
                for (int kb = 0; kb < DV / 64; ++kb) tma_store_3d(tS() + kb * C * 128, &P.tmO, kb * 64, t0, bh);
                bulk_commit();
            }
            stage ^= (K_::NSTAGE - 1);
        }
        if (tid == 0) bulk_wait_read();
        __syncthreads();
        return true;
    }
};

// Every thread of the CTA, after its last read of a flag (finish_call).
__device__ __forceinline__ void finish_cta(const TcParams &P, unsigned tag, volatile unsigned *s_last) {
    finish_call(P.ticket, tag, P.flagsw, nullptr, P.BH * P.kmax, s_last);
}

template <int C, int D, int DV, bool DECAY, bool NORM, int VAR>
__global__ void __launch_bounds__(kThreads, Cfg<C, D, DV>::CTAS) fwd_tc_kernel(const __grid_constant__ TcParams P) {
    using K_ = Cfg<C, D, DV>;
    // No static shared memory: the dynamic block starts at the (1024-byte
    // aligned) base of the CTA's shared window, which the swizzled tiles need.
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *base = smem_raw;
    uint64_t *bars = reinterpret_cast<uint64_t *>(base + K_::OFF_BAR);
    uint32_t *tmem_base_p = reinterpret_cast<uint32_t *>(base + K_::OFF_BAR + 32);
    int *ticket_p = reinterpret_cast<int *>(base + K_::OFF_BAR + 36);
    int *misalign_p = reinterpret_cast<int *>(base + K_::OFF_BAR + 40);
    volatile unsigned *last_p = reinterpret_cast<volatile unsigned *>(base + K_::OFF_BAR + 44);
    unsigned *tag_p = reinterpret_cast<unsigned *>(base + K_::OFF_BAR + 56);

    Kern<C, D, DV, DECAY, NORM, VAR> x(P, base);
    x.tid = threadIdx.x;
    x.warp = threadIdx.x >> 5;
    x.lane = threadIdx.x & 31;
    x.quad = x.warp & 3;
    x.half = x.warp >> 2;
    x.rowC = row_of<C>(x.quad, x.lane);
    x.rowD = row_of<D>(x.quad, x.lane);
    x.tma_bar = &bars[0];  // [0], [1]: input stages
    x.mma_bar = &bars[2];
    x.mma_bar2 = &bars[3];
    x.mma_bar3 = reinterpret_cast<uint64_t *>(base + K_::OFF_BAR + 48);
    x.tph = x.mph = x.mph2 = x.mph3 = 0;

    if (x.tid == 0) {
        *misalign_p = (smem_u32(base) & 1023u) != 0;
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        mbar_init(&bars[2], 1);
        mbar_init(&bars[3], 1);
        mbar_init(x.mma_bar3, decltype(x)::kFan);
        fence_mbar_init();
        tma_prefetch_desc(&P.tmQ);
        tma_prefetch_desc(&P.tmK);
        tma_prefetch_desc(&P.tmV);
        tma_prefetch_desc(&P.tmO);
        const CallTicket t = take_ticket(P.ticket);
        *ticket_p = (int)t.ticket;
        *tag_p = t.tag;
    }
    __syncthreads();
    x.tag = *tag_p;
    if (*misalign_p) {  // cannot happen with no static shared memory; refuse rather than corrupt
        if (x.tid == 0) atomicOr(P.err, DEV_TIMEOUT);
        finish_cta(P, x.tag, last_p);
        return;
    }
    if (x.warp == 0) {
        tmem_alloc(tmem_base_p, K_::TCOLS);
        tmem_relinquish();
    }
    const int ticket = *ticket_p;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    x.tb = *tmem_base_p;
    const bool want_out = P.sout.S != nullptr;
    x.need_mY = NORM || want_out;

    // This CTA's run of chunks [g0, g1) in the end-to-end order of all sequences,
    // and the pieces it holds: one per sequence that the run touches.  Pieces of a
    // sequence get increasing tickets in either ticket order.
    const long long NC = P.nchunks;
    const int run = P.runs_per_seq > 0 ? (ticket % P.BH) * P.runs_per_seq + ticket / P.BH : ticket;
    const long long g0 = (long long)run * P.cpc;
    const long long g1 = min((long long)P.BH * NC, g0 + P.cpc);
    const int bh_lo = (int)(g0 / NC), bh_hi = (int)((g1 - 1) / NC);
    struct Piece {
        int jb, je, k;  // chunks [jb, je) of the sequence; piece index k within it
        long long first_run;
        bool last;      // the sequence's last piece
    };
    auto piece = [&](int bh) {
        Piece pc;
        pc.jb = (int)(max(g0, bh * NC) - bh * NC);
        pc.je = (int)(min(g1, (bh + 1) * NC) - bh * NC);
        pc.first_run = (bh * NC) / P.cpc;
        pc.k = (int)(run - pc.first_run);
        pc.last = (pc.je == P.nchunks);
        return pc;
    };
    // Select sequence bh: its decay constant and the table of g^j, g^{2j}, j < 16.
    x.bh = -1;
    auto select = [&](int bh) {
        if (bh == x.bh) return;
        __syncthreads();  // every thread is done with the previous sequence's table
        x.bh = bh;
        x.kvh = (bh / P.H) * P.Hkv + (bh % P.H) / (P.H / P.Hkv);
        float g = 1.f;
        if constexpr (DECAY) g = P.gamma[bh % P.H];
        x.lg = log2f(g);
        if (x.tid < 32) x.g16()[x.tid] = DECAY ? gpow(x.lg, (float)((x.tid & 15) * (x.tid < 16 ? 1 : 2))) : 1.f;
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    };
    bool ok = true;
    do {
        // ---- phase 1: the summary of every piece that a later piece, or the
        // export, needs; a release flag publishes it to later pieces
        for (int bh = bh_lo; bh <= bh_hi && ok; ++bh) {
            const Piece pc = piece(bh);
            if (pc.last && !want_out) continue;
            select(bh);
            if constexpr (VAR == 1) ok = x.pass1_unm(pc.jb, pc.je);
            else if constexpr (VAR == 2) ok = x.pass1_asym(pc.jb, pc.je);
            else ok = x.pass1(pc.jb, pc.je);
            if (!ok) break;
            x.store_summary(P.summ + ((size_t)bh * P.kmax + pc.k) * K_::SUM);
            // the block barrier orders every thread's summary stores before the
            // release store of the flag, which makes them visible at gpu scope
            __syncthreads();
            if (!pc.last && x.tid == 0) {
                unsigned *f = P.flagsw + (size_t)bh * P.kmax + pc.k;
                asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(f), "r"(x.tag) : "memory");
            }
        }
        if (!ok) break;
        // ---- phase 2, per piece: exclusive scan (prefix = state_in (+) the
        // summaries of the sequence's earlier pieces), then the outputs
        for (int bh = bh_lo; bh <= bh_hi && ok; ++bh) {
            const Piece pc = piece(bh);
            select(bh);
            // first token of piece r of this sequence
            auto start = [&](int r) -> int {
                return r == 0 ? 0 : (int)(((pc.first_run + r) * P.cpc - bh * NC) * C);
            };
            if (P.sin.S || pc.k == 0) {
                if (!(ok = x.prefix_init())) break;
            }
            if (pc.k > 0) {  // with a zero state_in the first fold step sets the prefix
                if (!(ok = x.wait_flags(0, pc.k))) break;
                const float *Ls = P.summ + (size_t)bh * P.kmax * K_::SUM;
                if constexpr (VAR == 1) ok = x.fold_unm(Ls, pc.k, start, !P.sin.S);
                else if constexpr (VAR == 2) ok = x.fold_asym(Ls, pc.k, start, !P.sin.S);
                else ok = x.fold_all(Ls, pc.k, start, !P.sin.S);
                if (!ok) break;
            }
            // ---- state export, part 1: what pass 2 does not carry to the sequence end
            if (pc.last && want_out) {
                const float *Lown = P.summ + ((size_t)bh * P.kmax + pc.k) * K_::SUM;
                const float fown = DECAY ? gpow(x.lg, (float)(P.n - start(pc.k))) : 1.f;
                if constexpr (VAR == 1) x.export_pre_unm(Lown, fown);
                else if constexpr (VAR == 2) x.export_pre_asym(Lown, fown);
                else x.export_pre(Lown, fown);
            }
            if constexpr (VAR == 1) ok = x.pass2_unm(pc.jb, pc.je);
            else if constexpr (VAR == 2) ok = x.pass2_asym(pc.jb, pc.je);
            else ok = x.pass2(pc.jb, pc.je);
            if (!ok) break;
            // ---- state export, part 2: the final state at the sequence end
            if (pc.last && want_out) {
                if constexpr (VAR == 1) x.export_post_unm();
                else if constexpr (VAR == 2) x.export_post_asym();
                else ok = x.export_post();
                if (!ok) break;
            }
        }
    } while (0);

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (x.warp == 0) tmem_dealloc(x.tb, K_::TCOLS);
    if (x.tid == 0) bulk_wait_all();  // the output stores are complete before the CTA ends
    finish_cta(P, x.tag, last_p);
}

// ============================================================================ host side
struct Plan {
    int nchunks;  // chunks per sequence
    int cpc;      // chunks per CTA (a run in the end-to-end order of all sequences)
    int ncta;     // CTAs: at most the number that fit on the device at once
    int kmax;     // upper bound on the pieces (runs touched) of one sequence
};
inline Plan make_plan(const hla_params &p, int num_sms) {
    Plan pl;
    const long long BH = (long long)p.B * p.H;
    pl.nchunks = (p.n + p.chunk - 1) / p.chunk;
    const long long total = BH * pl.nchunks;
    const long long slots = (long long)num_sms * ctas_per_sm(p);
    long long cpc = (total + slots - 1) / (slots > 0 ? slots : 1);
    if (cpc < 1) cpc = 1;
    pl.cpc = (int)cpc;
    pl.ncta = (int)((total + cpc - 1) / cpc);
    if (pl.ncta < 1) pl.ncta = 1;
    pl.kmax = (pl.nchunks + pl.cpc - 1) / pl.cpc + 1;
    return pl;
}

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct WsLayout {
    size_t off_flags, off_summ, total;
};
inline WsLayout ws_layout(const hla_params &p, const Plan &pl) {
    const size_t BH = (size_t)p.B * p.H;
    const size_t D = p.d, DV = p.dv;
    const size_t SUM = D * D + 2 * D * DV + 2 * D;
    WsLayout w;
    w.off_flags = 256;
    w.off_summ = align256(w.off_flags + BH * pl.kmax * 4);
    w.total = align256(w.off_summ + BH * pl.kmax * SUM * 4);
    return w;
}

template <int C, int D, int DV, bool DECAY, bool NORM, int VAR>
cudaError_t launch_cfg(const FwdArgs &a, cudaStream_t st, int num_sms) {
    using K_ = Cfg<C, D, DV>;
    hla_params p{a.B, a.H, a.n, a.d, a.dv, a.chunk, a.in_dtype, a.flags, a.eps, a.gamma};
    const Plan pl = make_plan(p, num_sms);
    const WsLayout wl = ws_layout(p, pl);
    TcParams P;
    memset(&P, 0, sizeof P);
    const int BH = a.B * a.H, BHkv = a.B * a.Hkv;
    if (!encode_3d(&P.tmQ, a.q, D, a.n, BH, C) || !encode_3d(&P.tmK, a.k, D, a.n, BHkv, C) ||
        !encode_3d(&P.tmV, a.v, DV, a.n, BHkv, C) || !encode_3d(&P.tmO, a.o, DV, a.n, BH, C))
        return cudaErrorInvalidValue;
    P.B = a.B; P.H = a.H; P.n = a.n; P.BH = BH; P.Hkv = a.Hkv;
    P.nchunks = pl.nchunks; P.cpc = pl.cpc; P.kmax = pl.kmax;
    P.runs_per_seq = pl.nchunks % pl.cpc == 0 ? pl.nchunks / pl.cpc : 0;
    P.eps = a.eps; P.gamma = a.gamma;
    P.o = a.o; P.sin = a.sin; P.sout = a.sout;
    uint8_t *ws = static_cast<uint8_t *>(a.workspace);
    P.ticket = reinterpret_cast<unsigned *>(ws);
    P.flagsw = reinterpret_cast<unsigned *>(ws + wl.off_flags);
    P.summ = reinterpret_cast<float *>(ws + wl.off_summ);
    P.err = a.err;
    auto kern = fwd_tc_kernel<C, D, DV, DECAY, NORM, VAR>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, K_::SMEM_LAUNCH);
    if (e != cudaSuccess) return e;
    kern<<<pl.ncta, kThreads, K_::SMEM_LAUNCH, st>>>(P);
    return cudaGetLastError();
}

// Launcher for one (decay, normalise) combination over all supported shapes;
// explicitly instantiated in hla_fwd_tc_f<flags>.cu.
template <bool DECAY, bool NORM, int VAR>
cudaError_t launch_flags(const FwdArgs &a, cudaStream_t st, int ns) {
    const int key = (a.chunk == 128 ? 4 : 0) | (a.d == 128 ? 2 : 0) | (a.dv == 128 ? 1 : 0);
    switch (key) {
        case 0: return launch_cfg<64, 64, 64, DECAY, NORM, VAR>(a, st, ns);
        case 2: return launch_cfg<64, 128, 64, DECAY, NORM, VAR>(a, st, ns);
        case 3: return launch_cfg<64, 128, 128, DECAY, NORM, VAR>(a, st, ns);
        case 4: return launch_cfg<128, 64, 64, DECAY, NORM, VAR>(a, st, ns);
        case 6: return launch_cfg<128, 128, 64, DECAY, NORM, VAR>(a, st, ns);
        case 7: return launch_cfg<128, 128, 128, DECAY, NORM, VAR>(a, st, ns);
        default:  // dv > d: not for the asymmetric variant, whose spare accumulator is d wide
            if constexpr (VAR == 2) return cudaErrorInvalidValue;
            else return key == 1 ? launch_cfg<64, 64, 128, DECAY, NORM, VAR>(a, st, ns)
                                 : launch_cfg<128, 64, 128, DECAY, NORM, VAR>(a, st, ns);
    }
}

}  // namespace tc
}  // namespace hla
