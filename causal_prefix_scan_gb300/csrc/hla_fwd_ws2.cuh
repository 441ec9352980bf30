// hla_fwd_ws2.cuh -- the masked second-order HLA forward for d = 64 without decay,
// on 128-token tiles (sm_103a: tcgen05 MMA, TMEM accumulators, TMA).
//
// Same method and work split as hla_fwd_ws.cuh (gist.science summary of "Higher-order
// Linear Attention", section 1 for the summaries and the masked output, section 4
// for the segment concatenation and the exclusive scan): pass 1 forms every piece's
// summary from zero, the scan forms each piece's exact prefix, pass 2 writes O.  The
// chunk length of the chunked form only changes the rounding, so this kernel always
// works on chunks of 128 tokens: every token-row MMA then has 128 rows (the full
// tensor-core rate, and twice the work per handoff of a 64-row tile).
//
// What makes 128-token tiles fit two CTAs per SM (256 TMEM columns, ~110 KB of
// shared memory each):
//   * one 128-column TMEM slot (A) carries the whole token chain of a chunk:
//       Q K^T (fp32) -> A-tilde, written back in place as packed bf16 (columns 0-63)
//       -> U = Q S_p + A-tilde K (columns 64-127; A-tilde is read from TMEM as the
//       A operand) -> Q U^T (fp32) -> M packed (0-63) -> O = Q X_p + M V (64-127);
//     with dv = 128, O has a slot of its own;
//   * pass 1 keeps S and C stacked in one 128-lane accumulator [S; C]: its state
//     products are single MMAs with M = 128 whose A operand has a zero half (a 2 KB
//     zero block reached through the leading-byte offset of an MN-major descriptor);
//   * the A-tilde / M tiles live in TMEM, not in shared memory; Q is double buffered,
//     V single buffered, K double buffered in pass 1 (its second slot is the scan
//     operand space, idle then) and single buffered in pass 2.
// The scan between the passes: summaries and X'' are stored in share order (a warp's
// 32 rows of the same four columns are 512 contiguous bytes); S_pre, which step 1
// leaves in TMEM, is not formed again by step 2 of the same pair; the A-tilde of the
// first pass-2 chunk, which needs no scan result, is packed while the scan waits.
// The kernel is dispatched for dv = 64 (two CTAs per SM); its layout also covers
// dv = 128 (O in a slot of its own, one CTA per SM).
// Roles are those of hla_fwd_ws.cuh: warp 0 TMA, warp 1 MMA (whole warp, one elected
// lane issues), warps 2-5 E (chain epilogues), warps 6-9 T (state extraction).
#pragma once

#include "hla_fwd_ws.cuh"

namespace hla {
namespace ws2 {

using tc::cmax;
using ws::kBarAH;
using ws::kBarE;
using ws::kBarT;
using ws::kThreads;
using ws::kWarpE;
using ws::kWarpT;
using ws::WsParams;
using ws::bulk_wait_read1;
using ws::mbar_arrive;

constexpr int CT = 128, D = 64;

enum : int {
    B_QF = 0,    // [2] Q slot landed
    B_KF = 2,    // [2] K slot landed
    B_VF = 4,    // V landed
    B_QE = 5,    // [2] Q slot free (MMA commit + T)
    B_KE = 7,    // [2] K slot free
    B_VE = 9,    // V free
    B_AF = 10,   // MMA -> E: Q K^T in TMEM
    B_AR = 11,   // E -> MMA: A-tilde packed in TMEM
    B_UF = 12,   // MMA -> E, T: U accumulated (Q S_p has read the S_p tile)
    B_UR = 13,   // E -> MMA: U in smem
    B_MF = 14,   // MMA -> E: Q U^T in TMEM
    B_MR = 15,   // E -> MMA: M packed in TMEM
    B_OF = 16,   // MMA -> E: O accumulated, M V has read M
    B_OFREE = 17,  // E -> MMA: O read, TMEM slot A (and O) free
    B_ST = 18,   // T -> MMA: S_p tile ready
    B_ST2 = 19,  // T -> MMA: X_p tile ready
    B_XD = 20,   // MMA -> T: the chunk's state updates and tile reads done
    B_AUX = 21,  // scan / export products
    B_FIN = 22,  // MMA warp's final drain
    NBARS = 23
};

template <int DV, bool NORM>
struct Lay {
    static_assert(DV == 64 || DV == 128, "dv");
    // ---- TMEM
    static constexpr bool OWN_O = DV > 64;  // O in its own slot (else columns 64-127 of A)
    static constexpr uint32_t TA = 0;
    static constexpr uint32_t TO = OWN_O ? 128u : 64u;
    static constexpr uint32_t TS = OWN_O ? 256u : 128u;   // S (M = 64 layout) in pass 2
    static constexpr uint32_t TX = TS + D;                  // X (M = 64 layout)
    static constexpr uint32_t TSC = OWN_O ? 128u : TS;      // pass 1: [S; C] stacked (M = 128)
    static constexpr int TUSED = TX + DV;
    static constexpr int TCOLS = TUSED <= 256 ? 256 : 512;
    static constexpr int CTAS = TCOLS == 256 ? 2 : 1;
    // ---- shared memory
    static constexpr int NQ = 2;
    static constexpr int SQ = CT * D * 2, SK = CT * D * 2, SV = CT * DV * 2;
    static constexpr int SZ = 2048;                       // zero block (16 rows of 128 B)
    static constexpr int SU = CT * DV * 2 > CT * D * 2 ? CT * DV * 2 : CT * D * 2;  // U; O staging
    static constexpr int SSX = D * cmax(D, DV) * 2;       // S_p, then X_p
    static constexpr int SAUX = SK;                       // second K slot in pass 1; scan operands
    // Both K slots lie below the zero block Z1 and V, which the stacked state product
    // reaches from K through a (positive) leading byte offset.
    static constexpr int OFF_Z0 = 0, OFF_Q = SZ, OFF_K = OFF_Q + NQ * SQ, OFF_AUX = OFF_K + SK;
    static constexpr int OFF_V = OFF_AUX + SAUX, OFF_Z1 = OFF_V + SV, OFF_U = OFF_Z1 + SZ, OFF_SX = OFF_U + SU;
    static constexpr int TILES_END = OFF_SX + SSX;
    // scan operands: S hi, lo (and with dv = 128 C hi) in the U space; C hi, lo (C lo) in AUX
    static constexpr int OFF_SHI = OFF_U, OFF_SLO = OFF_SHI + D * D * 2;
    static constexpr int OFF_CHI = DV > 64 ? OFF_SLO + D * D * 2 : OFF_AUX;
    static constexpr int OFF_CLO = DV > 64 ? OFF_AUX : OFF_CHI + D * DV * 2;
    static_assert(OFF_SLO + D * D * 2 <= OFF_U + SU && OFF_CLO + D * DV * 2 <= OFF_AUX + SAUX &&
                  (DV == 64 || OFF_CHI + D * DV * 2 <= OFF_U + SU), "scan operands");
    static constexpr int NVEC = 2 * D + 8 * D;  // m, Y running sums; reduction scratch
    static constexpr int OFF_VEC = TILES_END, OFF_BAR = OFF_VEC + NVEC * 4, OFF_MISC = OFF_BAR + NBARS * 8;
    static constexpr int SMEM = OFF_MISC + 64;
    static constexpr int LIMIT = CTAS == 2 ? 112 * 1024 : 227 * 1024;
    static_assert(SMEM <= LIMIT, "shared memory");
    static constexpr int SMEM_LAUNCH = CTAS == 2 ? cmax(SMEM, 78 * 1024) : cmax(SMEM, 120 * 1024);
    // summaries (row-major fp32): S [D][D], X [D][DV], C [D][DV], m [D], Y [D]; X'', Y''
    static constexpr int SUM = D * D + 2 * D * DV + 2 * D;
    static constexpr int XPP = D * DV + D;
};

// MMA with the A operand in TMEM (M = 128: row m in lane m, K pairs packed per
// 32-bit column, lower K index in the low half), issued by one elected lane of a warp.
HLA_DEVICE void umma_f16_tmem_a_warp(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                     uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p, e;\n elect.sync _|e, 0xffffffff;\n setp.ne.b32 p, %4, 0;\n"
        " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}


template <int DV, bool NORM>
struct Fwd2 {
    using L_ = Lay<DV, NORM>;
    static constexpr uint32_t TA = L_::TA, TO = L_::TO, TS = L_::TS, TX = L_::TX, TSC = L_::TSC;
    const WsParams &P;
    uint8_t *base;
    uint64_t *bars;
    volatile int *abort_p;
    unsigned tag;  // the value this call's release flags carry
    uint32_t tb;
    int tid, warp, lane, quad;
    int bh;
    int ah, part;
    bool need_mY;
    bool sp_early = false;  // the current piece's first pass-2 S_p tile was handed over in its setup
    int ts_bh = -1;  // the pair whose S_pre (with its hi / lo tiles) the scan left in TS

    __device__ Fwd2(const WsParams &p, uint8_t *b) : P(p), base(b) {}

    // ---------------------------------------------------------------- smem
    __device__ __forceinline__ uint8_t *sQ(int s) const { return base + L_::OFF_Q + s * L_::SQ; }
    // K: two slots in pass 1 (the second is the scan operand space, idle then), one in pass 2
    int n1;  // this CTA's pass-1 chunks (they come first in the chunk numbering)
    __device__ __forceinline__ int kslot(int it) const { return it < n1 ? (it & 1) : 0; }
    __device__ __forceinline__ uint32_t kpar(int it) const {
        return (uint32_t)((it < n1 ? (it >> 1) : ((n1 + 1) >> 1) + (it - n1)) & 1);
    }
    __device__ __forceinline__ uint8_t *sK(int it) const { return base + (kslot(it) ? L_::OFF_AUX : L_::OFF_K); }
    __device__ __forceinline__ uint8_t *sV() const { return base + L_::OFF_V; }
    __device__ __forceinline__ uint8_t *z0() const { return base + L_::OFF_Z0; }
    __device__ __forceinline__ uint8_t *z1() const { return base + L_::OFF_Z1; }
    __device__ __forceinline__ uint8_t *tU() const { return base + L_::OFF_U; }
    __device__ __forceinline__ uint8_t *tSX() const { return base + L_::OFF_SX; }
    __device__ __forceinline__ uint8_t *fShi() const { return base + L_::OFF_SHI; }
    __device__ __forceinline__ uint8_t *fSlo() const { return base + L_::OFF_SLO; }
    __device__ __forceinline__ uint8_t *fChi() const { return base + L_::OFF_CHI; }
    __device__ __forceinline__ uint8_t *fClo() const { return base + L_::OFF_CLO; }
    __device__ __forceinline__ float *mrun() const { return reinterpret_cast<float *>(base + L_::OFF_VEC); }
    __device__ __forceinline__ float *Yrun() const { return mrun() + D; }
    __device__ __forceinline__ float *scr() const { return mrun() + 2 * D; }  // [8D]
    __device__ __forceinline__ uint64_t *bar(int i) const { return bars + i; }
    __device__ __forceinline__ uint32_t taddr(uint32_t slot, int col) const {
        return tb + slot + ((uint32_t)(32 * quad) << 16) + (uint32_t)col;
    }

    // ---------------------------------------------------------------- waits
    // Bounded, warp-uniform waits: a poll sleeps in hardware until the phase completes;
    // the CTA's abort flag or the time limit end the wait (the latter raises the
    // device status word).  wait() flips bit b of the parity word ph.
    __device__ bool waitp(int b, uint32_t par) {
        bool ok = false;
        if (!*abort_p) {
            ok = mbar_try_wait(bar(b), par);
            if (!ok) ok = wait_slow(b, par);
        }
        return __all_sync(0xffffffffu, ok);
    }
    __device__ bool wait(int b, uint32_t &ph) {
        const uint32_t par = (ph >> b) & 1u;
        ph ^= 1u << b;
        return waitp(b, par);
    }
    __device__ __noinline__ bool wait_slow(int b, uint32_t par) {
        const uint64_t t0 = globaltimer_ns();
        while (!*abort_p) {
            if (mbar_try_wait(bar(b), par)) return true;
            if (globaltimer_ns() - t0 > (uint64_t)kWaitLimitUs * 1000u) {
                atomicOr(P.err, DEV_TIMEOUT);
                *abort_p = 1;
            }
        }
        return false;
    }
    // Bounded wait by one warp for the flags of pieces 0 .. k - 1 of the current pair
    // (lanes poll different flags); on expiry the CTA aborts and the status word is raised.
    __device__ bool wait_flags(const unsigned *flags, int k) {
        bool ok = true;
        for (int j = lane; j < k && ok; j += 32) {
            const unsigned *f = flags + (size_t)bh * P.kmax + j;
            ok = false;
            for (uint32_t it = 0; it < kWaitLimit; ++it) {
                unsigned v;
                asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
                if (v == tag) { ok = true; break; }
                if (*abort_p) break;
                if (it > 256) __nanosleep(128);
            }
            if (!ok && !*abort_p) {
                atomicOr(P.err, DEV_TIMEOUT);
                *abort_p = 1;
            }
        }
        return __all_sync(0xffffffffu, ok);
    }

    // ---------------------------------------------------------------- stage ring
    // Chunk number it (both passes) uses Q slot it % 2 for the (it / 2)-th time and the
    // V buffer for the it-th time (K: kslot / kpar above).
    static __device__ __forceinline__ uint32_t qpar(int it) { return (uint32_t)((it >> 1) & 1); }
    static __device__ __forceinline__ uint32_t vpar(int it) { return (uint32_t)(it & 1); }

    // ---------------------------------------------------------------- MMA groups (whole warp)
    // token-row product into TMEM columns `slot`: A K-major [CT x KD] smem, B K-major [N x KD]
    template <int N, int KD>
    __device__ __forceinline__ void mma_kk(uint32_t slot, const uint8_t *a, const uint8_t *b, bool acc) {
        constexpr uint32_t id = make_idesc(CT, N, false, false);
        const uint64_t da = make_sdesc(smem_u32(a), 16u, 1024u), db = make_sdesc(smem_u32(b), 16u, 1024u);
#pragma unroll
        for (int k = 0; k < KD; k += 16) {
            const uint32_t ka = ((uint32_t)(k >> 6) * CT * 128u + (uint32_t)(k & 63) * 2u) >> 4;
            const uint32_t kb = ((uint32_t)(k >> 6) * N * 128u + (uint32_t)(k & 63) * 2u) >> 4;
            umma_f16_warp(tb + slot, da + ka, db + kb, id, (acc || k > 0) ? 1u : 0u);
        }
    }
    // token-row product: A K-major [CT x KD] smem, B MN-major [KD x N] (rows of B = K index)
    template <int N, int KD>
    __device__ __forceinline__ void mma_km(uint32_t slot, const uint8_t *a, const uint8_t *b, int brows, bool acc) {
        constexpr uint32_t id = make_idesc(CT, N, false, true);
        const uint64_t da = make_sdesc(smem_u32(a), 16u, 1024u),
                       db = make_sdesc(smem_u32(b), (uint32_t)brows * 128u, 1024u);
#pragma unroll
        for (int k = 0; k < KD; k += 16) {
            const uint32_t ka = ((uint32_t)(k >> 6) * CT * 128u + (uint32_t)(k & 63) * 2u) >> 4;
            umma_f16_warp(tb + slot, da + ka, db + (uint32_t)(k * 8), id, (acc || k > 0) ? 1u : 0u);
        }
    }
    // token-row product with A in TMEM (packed bf16, K = CT): B MN-major [CT x N] smem
    template <int N>
    __device__ __forceinline__ void mma_tm(uint32_t slot, uint32_t aslot, const uint8_t *b, bool acc) {
        constexpr uint32_t id = make_idesc(CT, N, false, true);
        const uint64_t db = make_sdesc(smem_u32(b), CT * 128u, 1024u);
#pragma unroll
        for (int k = 0; k < CT; k += 16)
            umma_f16_tmem_a_warp(tb + slot, tb + aslot + (uint32_t)(k / 2), db + (uint32_t)(k * 8), id,
                                 (acc || k > 0) ? 1u : 0u);
    }
    // state product over tokens, M = D: A MN-major [CT x D] (as D x CT), B MN-major [CT x N]
    template <int N>
    __device__ __forceinline__ void mma_mm(uint32_t slot, const uint8_t *a, const uint8_t *b, bool acc) {
        constexpr uint32_t id = make_idesc(D, N, true, true);
        const uint64_t da = make_sdesc(smem_u32(a), CT * 128u, 1024u), db = make_sdesc(smem_u32(b), CT * 128u, 1024u);
#pragma unroll
        for (int k = 0; k < CT; k += 16)
            umma_f16_warp(tb + slot, da + (uint32_t)(k * 8), db + (uint32_t)(k * 8), id, (acc || k > 0) ? 1u : 0u);
    }
    // Stacked state product (pass 1), M = 128 rows [S; C] with N = DV columns:
    //   S rows += K^T K:  A = {features of K (M-block 0), zero block (M-block 1)}, B = K
    //   C rows += Q^T V:  A = {zero block (M-block 0), features of Q (M-block 1)}, B = V
    // The zero half is reached through the leading-byte offset (distance between the
    // two 64-wide M blocks of an MN-major operand), which must be positive: the zero
    // block before Q serves the C half, the one after K the S half.  B for the S half
    // is K in its first 64 columns; with DV = 128 its second block (V) fills columns
    // of the S rows that are never read.
    __device__ __forceinline__ void mma_stack_S(const uint8_t *K, const uint8_t *V, bool first) {
        constexpr uint32_t id = make_idesc(128, DV, true, true);
        const uint32_t bl = DV > 64 ? (uint32_t)(V - K) : (uint32_t)CT * 128u;
#pragma unroll
        for (int k = 0; k < CT; k += 16) {
            const uint32_t a0 = smem_u32(K) + (uint32_t)k * 128u;
            const uint64_t da = make_sdesc(a0, smem_u32(z1()) - a0, 1024u);
            const uint64_t db = make_sdesc(smem_u32(K) + (uint32_t)k * 128u, bl, 1024u);
            umma_f16_warp(tb + TSC, da, db, id, (first && k == 0) ? 0u : 1u);
        }
    }
    __device__ __forceinline__ void mma_stack_C(const uint8_t *Q, const uint8_t *V) {
        constexpr uint32_t id = make_idesc(128, DV, true, true);
        const uint32_t z = smem_u32(z0());
#pragma unroll
        for (int k = 0; k < CT; k += 16) {
            const uint64_t da = make_sdesc(z, smem_u32(Q) + (uint32_t)k * 128u - z, 1024u);
            const uint64_t db = make_sdesc(smem_u32(V) + (uint32_t)k * 128u, CT * 128u, 1024u);
            umma_f16_warp(tb + TSC, da, db, id, 1u);
        }
    }
    // state x state, M = D: A K-major [D x D], B MN-major [D x DV] (scan and export)
    __device__ __forceinline__ void mma_ss(uint32_t slot, const uint8_t *a, const uint8_t *b, bool acc) {
        constexpr uint32_t id = make_idesc(D, DV, false, true);
        const uint64_t da = make_sdesc(smem_u32(a), 16u, 1024u), db = make_sdesc(smem_u32(b), D * 128u, 1024u);
#pragma unroll
        for (int k = 0; k < D; k += 16) {
            const uint32_t ka = ((uint32_t)(k & 63) * 2u) >> 4;
            umma_f16_warp(tb + slot, da + ka, db + (uint32_t)(k * 8), id, (acc || k > 0) ? 1u : 0u);
        }
    }

    // ---------------------------------------------------------------- TMEM rows
    // 128-row accumulator: thread (quad, lane) owns row 32 quad + lane (four warps, one
    // per quadrant).  f(c0, v[16]) gets 16 consecutive fp32 columns from c0.
    template <int NC, typename F>
    __device__ __forceinline__ void rows128(uint32_t slot, F &&f) {
        float a[16], b[16];
#pragma unroll
        for (int c = 0; c < NC; c += 32) {
            tmem_ld16(taddr(slot, c), a);
            tmem_ld16(taddr(slot, c + 16), b);
            tmem_wait_ld();
            f(c, a);
            f(c + 16, b);
        }
    }
    // 64-row accumulator (M = 64 layout: rows in lanes 0-15 of each quadrant): thread owns
    // row 16 quad + (lane & 15) and column half (lane >> 4).
    template <int NC, typename F>
    __device__ __forceinline__ void rows64(uint32_t slot, F &&f) {
        constexpr int HW = NC / 2;
        const int cme = (lane >> 4) * HW;
        float a[16], b[16];
#pragma unroll
        for (int c = 0; c < HW; c += 32) {
            tmem_ld16x2<HW>(taddr(slot, c), a);
            if constexpr (HW >= 32) tmem_ld16x2<HW>(taddr(slot, c + 16), b);
            tmem_wait_ld();
            f(cme + c, a);
            if constexpr (HW >= 32) f(cme + c + 16, b);
        }
    }
    // Score tile epilogue: the fp32 c x c tile in slot A (columns 0-127) becomes the
    // masked tile, packed as bf16 pairs in place (columns 0-63).  The warp of quadrant q
    // holds rows 32 q .. 32 q + 31, so its group g of 32 columns is entirely masked for
    // g > q (written as zeros, never read), unmasked for g < q and masked on the
    // diagonal for g = q.  Group g is packed into columns 16 g .. 16 g + 15, which lie in
    // a group read before they are written.  ROWSUM: also the row's sum.
    // pack_group: a (columns c0 .. c0 + 15), b (c0 + 16 .. c0 + 31) -> 16 packed pairs in a
    template <bool ROWSUM>
    __device__ __forceinline__ void pack_group(float (&a)[16], const float (&b)[16], int c0, int row, bool diag,
                                               float &rs) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {  // in place: pair i reads a[2i], a[2i + 1] (not yet overwritten)
            const float x0 = (!diag || c0 + 2 * i <= row) ? a[2 * i] : 0.f;
            const float x1 = (!diag || c0 + 2 * i + 1 <= row) ? a[2 * i + 1] : 0.f;
            if constexpr (ROWSUM) rs += x0 + x1;
            a[i] = __uint_as_float(pack_bf16(x0, x1));
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float y0 = (!diag || c0 + 16 + 2 * i <= row) ? b[2 * i] : 0.f;
            const float y1 = (!diag || c0 + 17 + 2 * i <= row) ? b[2 * i + 1] : 0.f;
            if constexpr (ROWSUM) rs += y0 + y1;
            a[8 + i] = __uint_as_float(pack_bf16(y0, y1));
        }
    }
    template <bool ROWSUM>
    __device__ __forceinline__ void pack_scores(int row, float &rs) {
        float a[16], b[16];
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            if (g > quad) break;  // warp-uniform
            tmem_ld16(taddr(TA, 32 * g), a);
            tmem_ld16(taddr(TA, 32 * g + 16), b);
            tmem_wait_ld();
            pack_group<ROWSUM>(a, b, 32 * g, row, g == quad, rs);
            tmem_st16(taddr(TA, 16 * g), a);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) b[i] = 0.f;
#pragma unroll
        for (int g = 1; g < 4; ++g)  // the zero groups (packed columns inside group 0 or 1, read above)
            if (g > quad) tmem_st16(taddr(TA, 16 * g), b);
        tmem_wait_st();
    }

    // Column sums of rows r < L of a [CT x D] bf16 tile with weights w(r), by 128 threads
    // (index gt, named barrier nb): out[i] = sc * out[i] + sum (fixed order).
    template <typename Wf>
    __device__ void colsum128(int gt, int nb, const uint8_t *t, int L, Wf &&w, float *scrp, float *out, float sc) {
        constexpr int NB = D / 8, NG = 128 / NB;
        const int cb = gt % NB, rg = gt / NB, wl = gt >> 5;
        float am[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) am[j] = 0.f;
        for (int r = rg; r < L; r += NG) {
            float a[8];
            tile_load_row8(t, CT, r, cb * 8, a);
            const float wr = w(r);
#pragma unroll
            for (int j = 0; j < 8; ++j) am[j] += wr * a[j];
        }
#pragma unroll
        for (int off = NB; off < 32; off <<= 1) {
#pragma unroll
            for (int j = 0; j < 8; ++j) am[j] += __shfl_xor_sync(0xffffffffu, am[j], off);
        }
        if ((gt & 31) < NB) {
#pragma unroll
            for (int j = 0; j < 8; ++j) scrp[wl * D + cb * 8 + j] = am[j];
        }
        ws::nbar(nb, 128);
        if (gt < D) out[gt] = sc * out[gt] + ((scrp[gt] + scrp[D + gt]) + (scrp[2 * D + gt] + scrp[3 * D + gt]));
        ws::nbar(nb, 128);
    }

    // single-thread wait (TMA thread)
    __device__ bool wait1(int b, uint32_t par) {
        if (*abort_p) return false;
        return mbar_try_wait(bar(b), par) || wait_slow(b, par);
    }

    // ======================================================================== TMA producer
    // Loads of chunk it: K (free once chunk it-1's S update ran), Q into slot it % 2 (free
    // once chunk it-2 released it), V (free once chunk it-1's M V ran).
    __device__ bool tma_chunk(int it, int j, int pbh) {
        const int t0 = j * CT, qs = it & 1;
        const int pk = (pbh / P.H) * P.Hkv + (pbh % P.H) / (P.H / P.Hkv);
        const int ks = kslot(it);
        // The second chunk's loads wait until the first chunk's Q and K have landed: at the
        // start of the launch every CTA requests its inputs at once, and the first chunk's
        // tiles, which the chain needs first, then do not share DRAM with the second's.
        if (it == 1 && (!wait1(B_KF + kslot(0), kpar(0)) || !wait1(B_QF, qpar(0)))) return false;
        if (!wait1(B_KE + ks, kpar(it) ^ 1u)) return false;
        fence_async_smem();  // earlier generic reads of the buffer precede the overwrite
        mbar_expect_tx(bar(B_KF + ks), L_::SK);
        tma_load_3d(sK(it), &P.tmK, bar(B_KF + ks), 0, t0, pk);
        if (!wait1(B_QE + qs, qpar(it) ^ 1u)) return false;
        fence_async_smem();
        mbar_expect_tx(bar(B_QF + qs), L_::SQ);
        tma_load_3d(sQ(qs), &P.tmQ, bar(B_QF + qs), 0, t0, pbh);
        if (!wait1(B_VE, vpar(it) ^ 1u)) return false;
        fence_async_smem();
        mbar_expect_tx(bar(B_VF), L_::SV);
#pragma unroll
        for (int kb = 0; kb < DV / 64; ++kb) tma_load_3d(sV() + kb * CT * 128, &P.tmV, bar(B_VF), kb * 64, t0, pk);
        return true;
    }
    // Wait, bounded, for loads that may still be in flight: the last use of each full
    // barrier (an earlier phase of the same barrier has completed before it).  Only a
    // barrier's latest phase may be polled: two phases on, its parity repeats.
    __device__ void tma_drain(int it_end) {
        auto poll = [&](int b, uint32_t par) {
            for (uint32_t i = 0; i < kWaitLimit; ++i) {
                if (mbar_try_wait(bar(b), par)) break;
                if (i > 4096) __nanosleep(64);
            }
        };
        bool kdone[2] = {false, false};
        for (int it = it_end - 1; it >= 0 && it >= it_end - 2; --it) {
            if (it == it_end - 1) poll(B_VF, vpar(it));
            poll(B_QF + (it & 1), qpar(it));
            const int ks = kslot(it);
            if (!kdone[ks]) poll(B_KF + ks, kpar(it));
            kdone[ks] = true;
        }
        // K slot 1 is last used by the final odd chunk of pass 1, which may lie further back
        if (!kdone[1] && n1 >= 2) {
            const int it = (n1 - 1) & 1 ? n1 - 1 : n1 - 2;
            if (it < it_end) poll(B_KF + 1, kpar(it));
        }
    }

    // ======================================================================== MMA warp
    // Pass 1: A slot = Q K^T, then A-tilde (0-63) and U = Q S_p + A-tilde K (64-127);
    // [S; C] stacked in TSC, X in TX.
    __device__ bool mma_pass1(int it, bool first, uint32_t &ph) {
        const int qs = it & 1;
        const int ks = kslot(it);
        if (!waitp(B_KF + ks, kpar(it)) || !waitp(B_QF + qs, qpar(it))) return false;
        tc_fence_after();
        uint8_t *Q = sQ(qs), *K = sK(it), *V = sV();
        mma_kk<CT, D>(TA, Q, K, false);  // Q K^T
        umma_commit_warp(bar(B_AF));
        if (!wait(B_ST, ph) || !wait(B_AR, ph)) return false;
        tc_fence_after();
        if (!first) mma_kk<D, D>(TA + 64, Q, tSX(), false);  // Q S_p
        mma_tm<D>(TA + 64, TA, K, !first);                    // + A-tilde K
        umma_commit_warp(bar(B_UF));
        mma_stack_S(K, V, first);  // S rows of [S; C] += K^T K (the first chunk starts [S; C] at zero)
        umma_commit_warp(bar(B_KE + ks));
        if (!wait(B_UR, ph) || !waitp(B_VF, vpar(it))) return false;
        tc_fence_after();
        mma_stack_C(Q, V);                 // C rows += Q^T V
        mma_mm<DV>(TX, tU(), V, !first);   // X += U^T V
        umma_commit_warp(bar(B_XD));
        umma_commit_warp(bar(B_QE + qs));
        umma_commit_warp(bar(B_VE));
        return true;
    }
    // Pass 2: A slot = Q K^T, then A-tilde (0-63) and U (64-127), then Q U^T, then M
    // (0-63) and O = Q X_p + M V (columns 64-127, or its own slot with dv = 128).
    __device__ bool mma_pass2(int it, uint32_t &ph, bool &pend) {
        const int qs = it & 1;
        const int ks = kslot(it);
        if (!waitp(B_KF + ks, kpar(it)) || !waitp(B_QF + qs, qpar(it))) return false;
        uint8_t *Q = sQ(qs), *K = sK(it), *V = sV();
        if (pend && !wait(B_OFREE, ph)) return false;  // slot A (M) and O read by the previous chunk
        pend = false;
        tc_fence_after();
        mma_kk<CT, D>(TA, Q, K, false);  // Q K^T
        umma_commit_warp(bar(B_AF));
        if (!wait(B_ST, ph) || !wait(B_AR, ph)) return false;
        tc_fence_after();
        mma_kk<D, D>(TA + 64, Q, tSX(), false);  // Q S_p
        mma_tm<D>(TA + 64, TA, K, true);          // + A-tilde K
        umma_commit_warp(bar(B_UF));
        mma_mm<D>(TS, K, K, true);                // S += K^T K
        umma_commit_warp(bar(B_KE + ks));
        if (!wait(B_UR, ph)) return false;
        tc_fence_after();
        mma_kk<CT, D>(TA, Q, tU(), false);  // Q U^T
        umma_commit_warp(bar(B_MF));
        if (!wait(B_ST2, ph) || !waitp(B_VF, vpar(it))) return false;
        tc_fence_after();
        mma_mm<DV>(TX, tU(), V, true);  // X += U^T V
        if (!wait(B_MR, ph)) return false;
        tc_fence_after();
        mma_km<DV, D>(TO, Q, tSX(), D, false);  // Q X_p
        umma_commit_warp(bar(B_XD));
        umma_commit_warp(bar(B_QE + qs));
        mma_tm<DV>(TO, TA, V, true);  // + M V
        umma_commit_warp(bar(B_OF));
        umma_commit_warp(bar(B_VE));
        pend = true;
        return true;
    }

    // ======================================================================== E group
    // et = tid - 64; thread (quad, lane) owns token row 32 quad + lane of every tile.
    __device__ __forceinline__ int grow() const { return 32 * quad + lane; }
    __device__ __forceinline__ void e_arrive(int b) {
        fence_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(b));
    }
    __device__ __forceinline__ void e_arrive_tmem(int b) {  // after TMEM writes
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(b));
    }
    __device__ void e_atilde(uint32_t &ph) {
        wait(B_AF, ph);
        tc_fence_after();
        float rs = 0.f;
        pack_scores<false>(grow(), rs);
        e_arrive_tmem(B_AR);
    }
    __device__ void e_pass1(int it, int L, uint32_t &ph, int et) {
        e_atilde(ph);
        wait(B_UF, ph);
        tc_fence_after();
        const int row = grow();
        rows128<D>(TA + 64, [&](int c0, float (&v)[16]) { tile_store_row16(tU(), CT, row, c0, v); });
        e_arrive(B_UR);
        if (need_mY) {  // Y += sum_b u_b
            ws::nbar(kBarE, 128);
            colsum128(et, kBarE, tU(), L, [](int) { return 1.f; }, scr(), Yrun(), 1.f);
        }
    }
    // atilde_done: the chunk's A-tilde was packed ahead (the first chunk of pass 2, whose
    // Q K^T needs no scan result, is packed before the scan).
    __device__ void e_pass2(int it, int j, int L, uint32_t &ph, int et, bool atilde_done) {
        const int qs = it & 1, row = grow();
        if (!atilde_done) e_atilde(ph);
        float qy = 0.f;
        if constexpr (NORM) {  // q . Y_p for this row, before Y moves on
            waitp(B_QF + qs, qpar(it));
            const uint8_t *Qs = sQ(qs);
#pragma unroll
            for (int c = 0; c < D; c += 8) {
                float q8[8];
                tile_load_row8(Qs, CT, row, c, q8);
#pragma unroll
                for (int i = 0; i < 8; ++i) qy += q8[i] * Yrun()[c + i];
            }
        }
        wait(B_UF, ph);
        tc_fence_after();
        if (et == 0) bulk_wait_read();  // the previous chunk's O store has read the U buffer
        ws::nbar(kBarE, 128);
        rows128<D>(TA + 64, [&](int c0, float (&v)[16]) { tile_store_row16(tU(), CT, row, c0, v); });
        e_arrive(B_UR);
        if constexpr (NORM) {  // Y += sum_b u_b
            ws::nbar(kBarE, 128);
            colsum128(et, kBarE, tU(), L, [](int) { return 1.f; }, scr(), Yrun(), 1.f);
        }
        wait(B_MF, ph);
        tc_fence_after();
        float rs = 0.f;
        pack_scores<NORM>(row, rs);  // M = tril(Q U^T), packed in place
        e_arrive_tmem(B_MR);
        wait(B_OF, ph);
        tc_fence_after();
        float inv = 1.f;
        if constexpr (NORM) inv = 1.f / (rs + qy + P.eps);
        // O -> the U buffer (its readers, Q U^T and the X update, completed before O did)
        rows128<DV>(TO, [&](int c0, float (&v)[16]) {
            if constexpr (NORM) {
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] *= inv;
            }
            tile_store_row16(tU(), CT, row, c0, v);
        });
        fence_async_smem();
        tc_fence_before();
        ws::nbar(kBarE, 128);
        if (et == 0) {
#pragma unroll
            for (int kb = 0; kb < DV / 64; ++kb) tma_store_3d(tU() + kb * CT * 128, &P.tmO, kb * 64, j * CT, bh);
            bulk_commit();
        }
        if (lane == 0) mbar_arrive(bar(B_OFREE));
    }

    // ======================================================================== T group
    // tt = tid - 192.
    __device__ __forceinline__ void t_arrive(int b) {
        fence_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(b));
    }
    __device__ __forceinline__ void arrive_empties(int qs, int ks) {
        mbar_arrive(bar(B_QE + qs));
        mbar_arrive(bar(B_KE + ks));
        mbar_arrive(bar(B_VE));
    }
    __device__ void t_pass1(int it, int L, bool first, uint32_t &ph, int tt) {
        const int qs = it & 1, ks = kslot(it);
        waitp(B_KF + ks, kpar(it));
        waitp(B_QF + qs, qpar(it));
        ph ^= 1u << B_UF;  // E's U barrier completes every chunk; T waits for it in pass 2 only
        if (!first) {  // S_p from the S rows of [S; C] (lanes 0-63, quadrants 0 and 1)
            wait(B_XD, ph);
            tc_fence_after();
            if (quad < 2) {
                const int r = 32 * quad + lane;
                rows128<D>(TSC, [&](int c0, float (&v)[16]) { tile_store_row16(tSX(), D, r, c0, v); });
            }
        }
        t_arrive(B_ST);
        if (need_mY)  // m += sum_r q_r
            colsum128(tt, kBarT, sQ(qs), L, [](int) { return 1.f; }, scr() + 4 * D, mrun(), 1.f);
        else
            ws::nbar(kBarT, 128);
        waitp(B_VF, vpar(it));
        if (tt == 0) arrive_empties(qs, ks);
    }
    // S_p (TS) into the operand tile for Q S_p, then the MMA warp may go on (T warps)
    __device__ void t_sp_tile() {
        const int r = 16 * quad + (lane & 15);
        rows64<D>(TS, [&](int c0, float (&v)[16]) { tile_store_row16(tSX(), D, r, c0, v); });
        t_arrive(B_ST);
    }
    __device__ void t_pass2(int it, bool first, uint32_t &ph, int tt) {
        const int qs = it & 1, ks = kslot(it);
        waitp(B_KF + ks, kpar(it));
        if (!first) {
            wait(B_XD, ph);
            tc_fence_after();
        }
        const int r = 16 * quad + (lane & 15);
        if (!(first && sp_early)) t_sp_tile();
        wait(B_UF, ph);  // Q S_p has read the S_p tile
        tc_fence_after();
        rows64<DV>(TX, [&](int c0, float (&v)[16]) { tile_store_row16(tSX(), D, r, c0, v); });  // X_p
        t_arrive(B_ST2);
        waitp(B_QF + qs, qpar(it));
        waitp(B_VF, vpar(it));
        ws::nbar(kBarT, 128);
        if (tt == 0) arrive_empties(qs, ks);
    }

    // ======================================================================== all hands
    // Warps 2-9 (ah = tid - 64; part = 0 for E warps, 1 for T warps).  The pass-2 states
    // S (TS) and X (TX) use the 64-row TMEM layout: thread (quad, part, lane) owns row
    // 16 quad + (lane & 15) and shr<NC>() columns from shc<NC>().  Summaries in the
    // workspace are row-major fp32.
    static constexpr int NPR = 4;  // threads per row of a 64-row state
    __device__ __forceinline__ int srow() const { return 16 * quad + (lane & 15); }
    __device__ __forceinline__ int rpart() const { return part * 2 + (lane >> 4); }
    template <int NC>
    __host__ __device__ static constexpr int shr() { return NC / 4; }
    template <int NC>
    __device__ __forceinline__ int shc() const { return part * (NC / 2) + (lane >> 4) * (NC / 4); }
    template <int NC>
    __device__ __forceinline__ void ld_sh(uint32_t slot, int c, float (&v)[16]) {
        tmem_ld16x2<NC / 4>(taddr(slot, part * (NC / 2) + c), v);
    }
    template <int NC>
    __device__ __forceinline__ void st_sh(uint32_t slot, int c, const float (&v)[16]) {
        tmem_st16x2<NC / 4>(taddr(slot, part * (NC / 2) + c), v);
    }
    static __device__ __forceinline__ void ld16g(const float *src, float (&v)[16]) {  // 16 floats, L2
#pragma unroll
        for (int i = 0; i < 16; i += 4) {
            const float4 a = tc::ldcg4(src + i);
            v[i] = a.x; v[i + 1] = a.y; v[i + 2] = a.z; v[i + 3] = a.w;
        }
    }
    static __device__ __forceinline__ void st16g(float *dst, const float (&v)[16]) { tc::st_row16(dst, v); }
    // Summaries and X'' in the workspace are in share order: element (r, c) of a
    // D-row matrix at ((c / 4) * D + r) * 4 + c % 4, so that the lanes of a warp (32
    // consecutive rows, the same columns) read or write 512 contiguous bytes.
    static __device__ __forceinline__ int sofs(int r, int c) { return ((c >> 2) * D + r) * 4; }
    static __device__ __forceinline__ void ld16s(const float *src, int r, int c, float (&v)[16]) {
#pragma unroll
        for (int i = 0; i < 16; i += 4) {
            const float4 a = tc::ldcg4(src + sofs(r, c + i));
            v[i] = a.x; v[i + 1] = a.y; v[i + 2] = a.z; v[i + 3] = a.w;
        }
    }
    static __device__ __forceinline__ void st16s(float *dst, int r, int c, const float (&v)[16]) {
#pragma unroll
        for (int i = 0; i < 16; i += 4)
            *reinterpret_cast<float4 *>(dst + sofs(r, c + i)) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
    }
    __device__ __forceinline__ void ah_sync() {
        tc_fence_before();
        ws::nbar(kBarAH, 256);
        tc_fence_after();
    }
    __device__ __forceinline__ const float *summ_of(int r) const {
        return P.summ + ((size_t)bh * P.kmax + r) * L_::SUM;
    }
    __device__ __forceinline__ float *xpp_of(int r) const { return P.xpp + ((size_t)bh * P.kmax + r) * L_::XPP; }
    // v += sum_{r<k} src(r)[row][c..c+15] (share order), four pieces per round trip
    template <typename Src>
    __device__ __forceinline__ void acc_rows(float (&v)[16], int k, int row, int c, Src &&src) {
        for (int r = 0; r < k; r += 4) {
            float a[4][16], wr[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                ld16s(src(min(r + u, k - 1)), row, c, a[u]);
                wr[u] = (r + u < k) ? 1.f : 0.f;
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] += (wr[0] * a[0][i] + wr[1] * a[1][i]) + (wr[2] * a[2][i] + wr[3] * a[3][i]);
        }
    }
    __device__ void ah_wait_flags(const unsigned *flags, int k) {
        if (warp == kWarpE) wait_flags(flags, k);
        ah_sync();
    }
    template <typename Src>
    __device__ __forceinline__ float acc_elems(int k, int i, Src &&src) {
        float y = 0.f;
        for (int r = 0; r < k; r += 8) {
            float a[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) a[u] = __ldcg(src(min(r + u, k - 1)) + i);
#pragma unroll
            for (int u = 0; u < 8; ++u) y += (r + u < k) ? a[u] : 0.f;
        }
        return y;
    }
    // TX += S C with S from the fold tiles (hi, lo) and C from (hi, lo): three bf16
    // products approximate the fp32 one.  Issued by one warp.
    __device__ void ah_product() {
        fence_async_smem();
        ah_sync();
        if (warp == kWarpE) {
            mma_ss(TX, fShi(), fChi(), true);
            mma_ss(TX, fShi(), fClo(), true);
            mma_ss(TX, fSlo(), fChi(), true);
            umma_commit_warp(bar(B_AUX));
        }
    }
    __device__ void ah_product_wait(uint32_t &aux_ph) {
        wait(B_AUX, aux_ph);
        tc_fence_after();
    }
    __device__ float ah_rowdot_S(const float *vec) {  // this thread's share of (S in TS) . vec
        float acc = 0.f;
        float v[16];
        ld_sh<D>(TS, 0, v);
        tmem_wait_ld();
        const int c0 = shc<D>();
#pragma unroll
        for (int i = 0; i < 16; ++i) acc += v[i] * vec[c0 + i];
        return acc;
    }
    template <int NC>
    __device__ void st_tmem_zero(uint32_t slot) {
        float z[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) z[i] = 0.f;
#pragma unroll
        for (int c = 0; c < shr<NC>(); c += 16) st_sh<NC>(slot, c, z);
        tmem_wait_st();
    }

    // Pass-1 summary -> dst (share order).  S, C from the stacked [S; C] accumulator
    // (quadrants 0, 1: S rows; 2, 3: C rows), X from TX, m, Y from the running sums.
    __device__ void ah_store_summary(float *dst) {
        float *S = dst, *X = S + D * D, *Cc = X + D * DV, *m = Cc + D * DV, *Y = m + D;
        const int r = 32 * (quad & 1) + lane;
        if (quad < 2) {
#pragma unroll
            for (int c = 0; c < D / 2; c += 16) {
                float v[16];
                tmem_ld16(taddr(TSC, part * (D / 2) + c), v);
                tmem_wait_ld();
                st16s(S, r, part * (D / 2) + c, v);
            }
        } else {
#pragma unroll
            for (int c = 0; c < DV / 2; c += 16) {
                float v[16];
                tmem_ld16(taddr(TSC, part * (DV / 2) + c), v);
                tmem_wait_ld();
                st16s(Cc, r, part * (DV / 2) + c, v);
            }
        }
        const int sr = srow(), cv = shc<DV>();
#pragma unroll
        for (int c = 0; c < shr<DV>(); c += 16) {
            float v[16];
            ld_sh<DV>(TX, c, v);
            tmem_wait_ld();
            st16s(X, sr, cv + c, v);
        }
        for (int i = ah; i < D; i += 256) {
            m[i] = mrun()[i];
            Y[i] = Yrun()[i];
        }
    }

    // S_pre(k) = S_in + sum_{r<k} S_r -> TS (and the hi / lo tiles when `tiles`), after
    // the flags A of pieces r < k.
    __device__ void ah_prefix_S(int k, bool tiles) {
        if (k > 0) ah_wait_flags(P.flagA, k);
        const int row = srow(), c0 = shc<D>();
        float v[16];
        if (P.sin.S) {
            ld16g(P.sin.S + ((size_t)bh * D + row) * D + c0, v);
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = 0.f;
        }
        acc_rows(v, k, row, c0, [&](int r) { return summ_of(r); });
        st_sh<D>(TS, 0, v);
        if (tiles) tc::store_hilo(fShi(), fSlo(), D, row, c0, v);
        tmem_wait_st();
    }

    // Scan, step 1 (a piece with a later piece): X''_k = X_k + S_pre(k) B,
    // Y''_k = Y_k + S_pre(k) b with B = C_k, b = m_k; the first piece with a state_in
    // also folds it in: B += C_in, b += m_in, minus G_in, h_in.  The product
    // accumulates into TX, which holds X_k (reloaded unless pass 1 just left it there).
    __device__ void ah_xpp(int k, bool tx_has_xk, uint32_t &aux_ph) {
        const bool sin = P.sin.S != nullptr;
        const bool fold_in = (k == 0 && sin);
        if (k == 0 && !sin) {  // X''_0 = X_0, Y''_0 = Y_0: readers take them from the summary
            ah_sync();
            if (ah == 0) {
                unsigned *f = P.flagB + (size_t)bh * P.kmax;
                asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(f), "r"(tag) : "memory");
            }
            return;
        }
        const float *Lk = summ_of(k), *Xk = Lk + D * D, *Ck = Xk + D * DV, *mk = Ck + D * DV, *Yk = mk + D;
        const int row = srow(), cv = shc<DV>();
        constexpr int NV = shr<DV>();
        float *bvec = scr(), *pscr = scr() + D;
        // B tiles and b: independent of the other pieces, built before their flags are awaited
#pragma unroll
        for (int c = 0; c < NV; c += 16) {
            float a[16];
            ld16s(Ck, row, cv + c, a);
            if (fold_in) {
                float b[16];
                ld16g(P.sin.C + ((size_t)bh * D + row) * DV + cv + c, b);
#pragma unroll
                for (int i = 0; i < 16; ++i) a[i] += b[i];
            }
            tc::store_hilo(fChi(), fClo(), D, row, cv + c, a);
        }
        for (int i = ah; i < D; i += 256) bvec[i] = __ldcg(mk + i) + (fold_in ? P.sin.m[(size_t)bh * D + i] : 0.f);
        if (!tx_has_xk || fold_in) {  // TX = X_k (- G_in)
#pragma unroll
            for (int c = 0; c < NV; c += 16) {
                float x[16];
                ld16s(Xk, row, cv + c, x);
                if (fold_in) {
                    float g[16];
                    ld16g(P.sin.G + ((size_t)bh * D + row) * DV + cv + c, g);
#pragma unroll
                    for (int i = 0; i < 16; ++i) x[i] -= g[i];
                }
                st_sh<DV>(TX, c, x);
            }
            tmem_wait_st();
        }
        ah_prefix_S(k, true);
        ts_bh = bh;
        ah_product();
        pscr[rpart() * D + row] = ah_rowdot_S(bvec);  // Y'' partials while the products run
        ah_product_wait(aux_ph);
        float *Xo = xpp_of(k), *Yo = Xo + D * DV;
#pragma unroll
        for (int c = 0; c < NV; c += 16) {
            float x[16];
            ld_sh<DV>(TX, c, x);
            tmem_wait_ld();
            st16s(Xo, row, cv + c, x);
        }
        ah_sync();
        for (int i = ah; i < D; i += 256) {
            float y = __ldcg(Yk + i);
#pragma unroll
            for (int q = 0; q < NPR; ++q) y += pscr[q * D + i];
            if (fold_in) y -= P.sin.h[(size_t)bh * D + i];
            Yo[i] = y;
        }
        ah_sync();  // every store of X'', Y'' precedes the release
        if (ah == 0) {
            unsigned *fl = P.flagB + (size_t)bh * P.kmax + k;
            asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(fl), "r"(tag) : "memory");
        }
    }

    // X_pre = sum_{r<k} X''_r -> TX and Y_pre -> Yrun (X''_0, Y''_0 are the summary's X_0,
    // Y_0 when there is no state_in), after the flags B of pieces r < k; four pieces per
    // round trip, X and Y of a round read together.
    __device__ void ah_prefix_X(int k, bool sin) {
        ah_wait_flags(P.flagB, k);
        const int row = srow(), cv = shc<DV>();
        constexpr int NV = shr<DV>();
        auto xsrc = [&](int r) -> const float * { return (r == 0 && !sin) ? summ_of(0) + D * D : xpp_of(r); };
        auto ysrc = [&](int r) -> const float * {
            return (r == 0 && !sin) ? summ_of(0) + D * D + 2 * D * DV + D : xpp_of(r) + D * DV;
        };
        float v[NV];
#pragma unroll
        for (int i = 0; i < NV; ++i) v[i] = 0.f;
        float y = 0.f;
        for (int r = 0; r < k; r += 4) {
            float yv[4], wr[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                wr[u] = (r + u < k) ? 1.f : 0.f;
                yv[u] = ah < D ? __ldcg(ysrc(min(r + u, k - 1)) + ah) : 0.f;
            }
#pragma unroll
            for (int cb = 0; cb < NV; cb += 16) {
                float a[4][16];
#pragma unroll
                for (int u = 0; u < 4; ++u) ld16s(xsrc(min(r + u, k - 1)), row, cv + cb, a[u]);
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    v[cb + i] += (wr[0] * a[0][i] + wr[1] * a[1][i]) + (wr[2] * a[2][i] + wr[3] * a[3][i]);
            }
            y += (wr[0] * yv[0] + wr[1] * yv[1]) + (wr[2] * yv[2] + wr[3] * yv[3]);
        }
#pragma unroll
        for (int cb = 0; cb < NV; cb += 16) {
            float t[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) t[i] = v[cb + i];
            st_sh<DV>(TX, cb, t);
        }
        tmem_wait_st();
        if (ah < D) Yrun()[ah] = y;
    }

    // Scan, step 2 (ts_bh is cleared: pass 2 moves TS on): the pass-2 start state TS = S_pre(k), TX = X_pre(k), Yrun = Y_pre(k);
    // for a sequence's last piece with state_out also Y_end = Y_pre + Y_k + S_pre m_k
    // (in state_out.h until the export replaces it by h).
    __device__ void ah_setup_pass2(int k, bool last, bool want_out, uint32_t &aux_ph, bool atilde, uint32_t &ph) {
        const bool sin = P.sin.S != nullptr;
        const int row = srow(), cv = shc<DV>();
        constexpr int NV = shr<DV>();
        float *bvec = scr(), *pscr = scr() + D;
        if (k > 0 || sin) {
            if (ts_bh != bh) ah_prefix_S(k, k == 0);  // else still in TS (and the tiles) from step 1
        } else {
            st_tmem_zero<D>(TS);
        }
        // TS = S_pre is final: the T warps hand the first pass-2 chunk its S_p operand now,
        // so that U = Q S_p + A-tilde K runs while the X_pre rounds below are in flight.  The
        // MMA warp then moves TS on (S += K^T K), so every later read of S_pre comes first:
        // the last piece's S_pre m_k for Y_end.  (Folding state_in into piece 0 reads TS
        // after its product; there the tile is handed over in pass 2 as for later chunks.)
        sp_early = !(k == 0 && sin);
        if (sp_early) {
            if (last && want_out) {
                const float *mk = summ_of(k) + D * D + 2 * D * DV;
                for (int i = ah; i < D; i += 256) bvec[i] = __ldcg(mk + i);
                ah_sync();
                pscr[rpart() * D + row] = ah_rowdot_S(bvec);
            }
            ah_sync();
            if (part == 1) t_sp_tile();
        }
        if (atilde && part == 0) e_atilde(ph);  // the first pass-2 chunk's A-tilde (E warps)
        if (last && want_out) {  // C_end = C_in + sum_{r<=k} C_r, m_end likewise -> state_out
            float *Co = P.sout.C + ((size_t)bh * D + row) * DV;
#pragma unroll
            for (int c = 0; c < NV; c += 16) {
                float v[16];
                if (sin) {
                    ld16g(P.sin.C + ((size_t)bh * D + row) * DV + cv + c, v);
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] = 0.f;
                }
                acc_rows(v, k + 1, row, cv + c, [&](int r) { return summ_of(r) + D * D + D * DV; });
                st16g(Co + cv + c, v);
            }
            for (int i = ah; i < D; i += 256)
                P.sout.m[(size_t)bh * D + i] =
                    (sin ? P.sin.m[(size_t)bh * D + i] : 0.f) +
                    acc_elems(k + 1, i, [&](int r) { return summ_of(r) + D * D + 2 * D * DV; });
        }
        if (k > 0) {  // X_pre = sum_{r<k} X''_r, Y_pre likewise
            ah_prefix_X(k, sin);
        } else if (sin) {  // X_pre = X_in = S_in C_in - G_in, Y_pre = S_in m_in - h_in
#pragma unroll
            for (int c = 0; c < NV; c += 16) {
                float a[16], g[16];
                ld16g(P.sin.C + ((size_t)bh * D + row) * DV + cv + c, a);
                tc::store_hilo(fChi(), fClo(), D, row, cv + c, a);
                ld16g(P.sin.G + ((size_t)bh * D + row) * DV + cv + c, g);
#pragma unroll
                for (int i = 0; i < 16; ++i) g[i] = -g[i];
                st_sh<DV>(TX, c, g);
            }
            tmem_wait_st();
            for (int i = ah; i < D; i += 256) bvec[i] = P.sin.m[(size_t)bh * D + i];
            ah_product();
            pscr[rpart() * D + row] = ah_rowdot_S(bvec);
            ah_product_wait(aux_ph);
            ah_sync();
            for (int i = ah; i < D; i += 256) {
                float y = -P.sin.h[(size_t)bh * D + i];
#pragma unroll
                for (int q = 0; q < NPR; ++q) y += pscr[q * D + i];
                Yrun()[i] = y;
            }
        } else {
            st_tmem_zero<DV>(TX);
            for (int i = ah; i < D; i += 256) Yrun()[i] = 0.f;
        }
        if (last && want_out) {
            const float *mk = summ_of(k) + D * D + 2 * D * DV, *Yk = mk + D;
            if (!sp_early) {
                for (int i = ah; i < D; i += 256) bvec[i] = __ldcg(mk + i);
                ah_sync();
                pscr[rpart() * D + row] = ah_rowdot_S(bvec);
            }
            ah_sync();
            for (int i = ah; i < D; i += 256) {
                float sm = 0.f;
#pragma unroll
                for (int q = 0; q < NPR; ++q) sm += pscr[q * D + i];
                P.sout.h[(size_t)bh * D + i] = __ldcg(Yk + i) + Yrun()[i] + sm;
            }
        }
        ts_bh = -1;
        ah_sync();
    }

    // After pass 2 of a sequence's last piece: S_end (TS), X_end (TX); C_end and m_end
    // (state_out, from the setup); G = S C - X as -(X + S (-C)) with the product
    // accumulated into TX; h = S m - Y (Y_end in state_out.h).
    __device__ void ah_export_post(uint32_t &aux_ph) {
        const int row = srow(), cs = shc<D>(), cv = shc<DV>();
        constexpr int NV = shr<DV>();
        float *So = P.sout.S + ((size_t)bh * D + row) * D, *Co = P.sout.C + ((size_t)bh * D + row) * DV;
        float *Go = P.sout.G + ((size_t)bh * D + row) * DV;
        float *mo = P.sout.m + (size_t)bh * D;
        float *ho = P.sout.h + (size_t)bh * D;
        float *pscr = scr() + D;
#pragma unroll
        for (int c = 0; c < NV; c += 16) {
            float v[16];
            ld16g(Co + cv + c, v);  // this thread's own C_end values from the setup
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = -v[i];
            tc::store_hilo(fChi(), fClo(), D, row, cv + c, v);
        }
        float sm = 0.f;
        {
            float v[16];
            ld_sh<D>(TS, 0, v);
            tmem_wait_ld();
            tc::store_hilo(fShi(), fSlo(), D, row, cs, v);
            st16g(So + cs, v);
#pragma unroll
            for (int i = 0; i < 16; ++i) sm += v[i] * mo[cs + i];
        }
        pscr[rpart() * D + row] = sm;
        ah_product();  // TX = X_end - S_end C_end = -G
        for (int i = ah; i < D; i += 256) {
            float h = -ho[i];
#pragma unroll
            for (int q = 0; q < NPR; ++q) h += pscr[q * D + i];
            ho[i] = h;
        }
        ah_product_wait(aux_ph);
#pragma unroll
        for (int c = 0; c < NV; c += 16) {
            float t[16];
            ld_sh<DV>(TX, c, t);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) t[i] = -t[i];
            st16g(Go + cv + c, t);
        }
    }
};

template <int DV, bool NORM>
__global__ void __launch_bounds__(kThreads, Lay<DV, NORM>::CTAS) fwd_ws2_kernel(const __grid_constant__ WsParams P) {
    using L_ = Lay<DV, NORM>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *base = smem_raw;
    Fwd2<DV, NORM> x(P, base);
    uint32_t *misc = reinterpret_cast<uint32_t *>(base + L_::OFF_MISC);  // TMEM base, ticket, abort, misaligned, last, tag
    x.bars = reinterpret_cast<uint64_t *>(base + L_::OFF_BAR);
    x.abort_p = reinterpret_cast<volatile int *>(misc + 2);
    x.tid = threadIdx.x;
    x.warp = threadIdx.x >> 5;
    x.lane = threadIdx.x & 31;
    x.quad = x.warp & 3;
    x.ah = (int)threadIdx.x - 64;
    x.part = (x.warp - kWarpE) >> 2;
    x.bh = -1;
    if (x.tid == 0) {
        misc[2] = 0u;
        misc[3] = (smem_u32(base) & 1023u) != 0;
        mbar_init(x.bar(B_QF), 1);
        mbar_init(x.bar(B_QF + 1), 1);
        mbar_init(x.bar(B_KF), 1);
        mbar_init(x.bar(B_KF + 1), 1);
        mbar_init(x.bar(B_VF), 1);
        mbar_init(x.bar(B_QE), 2);  // the MMA warp's commit and T's arrival
        mbar_init(x.bar(B_QE + 1), 2);
        mbar_init(x.bar(B_KE), 2);
        mbar_init(x.bar(B_KE + 1), 2);
        mbar_init(x.bar(B_VE), 2);
        const int one[7] = {B_AF, B_UF, B_MF, B_OF, B_XD, B_AUX, B_FIN};
        const int four[6] = {B_AR, B_UR, B_MR, B_OFREE, B_ST, B_ST2};  // one arrival per warp of a group
        for (int i = 0; i < 7; ++i) mbar_init(x.bar(one[i]), 1);
        for (int i = 0; i < 6; ++i) mbar_init(x.bar(four[i]), 4);
        fence_mbar_init();
        tma_prefetch_desc(&P.tmQ);
        tma_prefetch_desc(&P.tmK);
        tma_prefetch_desc(&P.tmV);
        tma_prefetch_desc(&P.tmO);
    }
    // the two zero blocks (read by the stacked state products)
    for (int i = threadIdx.x; i < L_::SZ / 16; i += kThreads) {
        reinterpret_cast<uint4 *>(x.z0())[i] = make_uint4(0, 0, 0, 0);
        reinterpret_cast<uint4 *>(x.z1())[i] = make_uint4(0, 0, 0, 0);
    }
    fence_async_smem();
    __syncthreads();
    if (misc[3]) {  // cannot happen with no static shared memory; refuse rather than corrupt
        if (x.tid == 0) {
            atomicOr(P.err, DEV_TIMEOUT);
            misc[5] = take_ticket(P.ticket).tag;
        }
        __syncthreads();
        ws::finish_cta(P, misc[5], misc + 4);
        return;
    }
    if (x.warp == ws::kWarpMma) {
        tmem_alloc(misc + 0, L_::TCOLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    x.tb = misc[0];
    if (x.tid == 0) {
        const CallTicket t = take_ticket(P.ticket);
        misc[1] = t.ticket;
        misc[5] = t.tag;
    }
    __syncthreads();
    const int ticket = (int)misc[1];
    x.tag = misc[5];
    const bool want_out = P.sout.S != nullptr;
    x.need_mY = NORM || want_out;

    const long long NCH = P.nchunks;
    const int run = P.runs_per_seq > 0 ? (ticket % P.BH) * P.runs_per_seq + ticket / P.BH : ticket;
    long long g0 = (long long)run * P.cpc;
    long long g1 = min((long long)P.BH * NCH, g0 + P.cpc);
    int split_k = -1;
    if (P.tail_split) {  // pieces 0 .. R-3 of cpc chunks, then two of cpc / 2 (R = runs_per_seq)
        const int level = ticket / P.BH, seq = ticket % P.BH, whole = P.runs_per_seq - 2;
        auto start = [&](int j) {
            return j <= whole ? (long long)j * P.cpc : (long long)whole * P.cpc + (long long)(j - whole) * (P.cpc / 2);
        };
        g0 = (long long)seq * NCH + start(level);
        g1 = (long long)seq * NCH + start(level + 1);
        split_k = level;
    }
    const int bh_lo = (int)(g0 / NCH), bh_hi = (int)((g1 - 1) / NCH);
    struct Piece {
        int jb, je, k;
        bool last;
    };
    auto piece = [&](int bh) {
        Piece pc;
        pc.jb = (int)(max(g0, bh * NCH) - bh * NCH);
        pc.je = (int)(min(g1, (bh + 1) * NCH) - bh * NCH);
        pc.k = split_k >= 0 ? split_k : (int)(run - (bh * NCH) / P.cpc);
        pc.last = (pc.je == P.nchunks);
        return pc;
    };
    auto select = [&](int bh) { x.bh = bh; };
    int n_phase1 = 0;  // pieces that run pass 1, and their chunks
    x.n1 = 0;
    for (int bh = bh_lo; bh <= bh_hi; ++bh) {
        const Piece pc = piece(bh);
        if (!(pc.last && !want_out)) {
            ++n_phase1;
            x.n1 += pc.je - pc.jb;
        }
    }

    if (x.warp == ws::kWarpTma) {
        if (x.lane == 0) {
            int it = 0;
            bool ok = true;
            for (int ph2 = 0; ph2 < 2 && ok; ++ph2)
                for (int bh = bh_lo; bh <= bh_hi && ok; ++bh) {
                    const Piece pc = piece(bh);
                    if (ph2 == 0 && pc.last && !want_out) continue;
                    for (int j = pc.jb; j < pc.je && ok; ++j) ok = x.tma_chunk(it++, j, bh);
                }
            x.tma_drain(it);
        }
        __syncwarp();
    } else if (x.warp == ws::kWarpMma) {
        int it = 0;
        uint32_t ph = 0;
        bool ok = true, pend = false;
        for (int bh = bh_lo; bh <= bh_hi && ok; ++bh) {
            const Piece pc = piece(bh);
            if (pc.last && !want_out) continue;
            for (int j = pc.jb; j < pc.je && ok; ++j) ok = x.mma_pass1(it++, j == pc.jb, ph);
        }
        for (int bh = bh_lo; bh <= bh_hi && ok; ++bh) {
            const Piece pc = piece(bh);
            for (int j = pc.jb; j < pc.je && ok; ++j) ok = x.mma_pass2(it++, ph, pend);
        }
        umma_commit_warp(x.bar(B_FIN));  // every MMA issued completes before TMEM is released
        mbar_wait(x.bar(B_FIN), 0u, P.err);
        __syncwarp();
    } else {
        // E (warps 2-5) and T (warps 6-9); after an expired wait these keep to the same
        // control flow (every wait then returns at once) so that named barriers stay matched.
        const bool isE = x.warp < kWarpT;
        const int gt = isE ? (int)threadIdx.x - 64 : (int)threadIdx.x - 192;
        uint32_t ph = 0, aux_ph = 0;
        int it = 0;
        int last_p1 = -1;  // the piece whose pass-1 state TMEM still holds
        for (int bh = bh_lo; bh <= bh_hi; ++bh) {
            const Piece pc = piece(bh);
            if (pc.last && !want_out) continue;
            select(bh);
            if (x.need_mY) {
                if (gt < D) (isE ? x.Yrun() : x.mrun())[gt] = 0.f;
                ws::nbar(isE ? kBarE : kBarT, 128);
            }
            for (int j = pc.jb; j < pc.je; ++j) {
                const int L = min(CT, P.n - j * CT);
                if (isE) x.e_pass1(it, L, ph, gt);
                else x.t_pass1(it, L, j == pc.jb, ph, gt);
                ++it;
            }
            if (!isE) {
                x.wait(B_XD, ph);
                tc_fence_after();
            }
            x.ah_sync();
            x.ah_store_summary(P.summ + ((size_t)bh * P.kmax + pc.k) * L_::SUM);
            x.ah_sync();
            if (x.ah == 128 && !pc.last) {  // (a T thread: the release waits for the stores to drain)
                unsigned *f = P.flagA + (size_t)bh * P.kmax + pc.k;
                asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(f), "r"(x.tag) : "memory");
            }
            last_p1 = bh;
        }
        bool atilde_done = isE;  // packed in the first setup, while T hands over S_p
        for (int bh = bh_lo; bh <= bh_hi; ++bh) {
            const Piece pc = piece(bh);
            if (pc.last) continue;
            select(bh);
            x.ah_xpp(pc.k, n_phase1 == 1 && last_p1 == bh, aux_ph);
        }
        for (int bh = bh_lo; bh <= bh_hi; ++bh) {
            const Piece pc = piece(bh);
            select(bh);
            x.ah_setup_pass2(pc.k, pc.last, want_out, aux_ph, atilde_done, ph);
            for (int j = pc.jb; j < pc.je; ++j) {
                const int L = min(CT, P.n - j * CT);
                if (isE) x.e_pass2(it, j, L, ph, gt, atilde_done);
                else x.t_pass2(it, j == pc.jb, ph, gt);
                atilde_done = false;
                ++it;
            }
            if (!isE) {
                x.wait(B_XD, ph);
                tc_fence_after();
            }
            if (isE && gt == 0) bulk_wait_read();  // the staging buffer (scan operand space) is read
            x.ah_sync();
            if (pc.last && want_out) x.ah_export_post(aux_ph);
            x.ah_sync();
        }
        if (isE && gt == 0) bulk_wait_all();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (x.warp == ws::kWarpMma) tmem_dealloc(x.tb, L_::TCOLS);
    ws::finish_cta(P, x.tag, misc + 4);
}

// ============================================================================ host side
// The plan and workspace of this kernel: chunks of 128 tokens.
inline hla_params as_ct(const hla_params &p) {
    hla_params q = p;
    q.chunk = CT;
    return q;
}
// dv = 64 only: there two CTAs share an SM (256 TMEM columns each), so one chunk's
// chain of MMAs and epilogues overlaps the other's.  With dv = 128 the slots need more
// than 256 columns, one CTA holds the SM, and the 64-token kernel is the faster one.
inline bool ws2_supported(const hla_params &p) {
    return !(p.flags & (HLA_UNMASKED | HLA_ASYMMETRIC | HLA_DECAY)) && p.in_dtype == HLA_BF16 && p.d == 64 &&
           p.dv == 64 && (p.chunk == 64 || p.chunk == 128);
}
inline int ws2_ctas_per_sm(const hla_params &p) { return p.dv == 64 ? 2 : 1; }
inline tc::Plan work_plan(const hla_params &p0, int num_sms) {
    const hla_params p = as_ct(p0);
    tc::Plan pl;
    const long long BH = (long long)p.B * p.H;
    pl.nchunks = (p.n + CT - 1) / CT;
    const long long total = BH * pl.nchunks;
    const long long slots = (long long)num_sms * ws2_ctas_per_sm(p);
    long long cpc = (total + slots - 1) / (slots > 0 ? slots : 1);
    if (cpc < 1) cpc = 1;
    pl.cpc = (int)cpc;
    pl.ncta = (int)((total + cpc - 1) / cpc);
    if (pl.ncta < 1) pl.ncta = 1;
    pl.kmax = (pl.nchunks + pl.cpc - 1) / pl.cpc + 1;
    return pl;
}
inline ws::WsLayout work_layout(const hla_params &p, const tc::Plan &pl) { return ws::work_layout(as_ct(p), pl); }

template <int DV, bool NORM>
cudaError_t launch_cfg(const FwdArgs &a, cudaStream_t st, int num_sms) {
    using L_ = Lay<DV, NORM>;
    hla_params p{a.B, a.H, a.n, a.d, a.dv, a.chunk, a.in_dtype, a.flags, a.eps, a.gamma};
    const tc::Plan pl = work_plan(p, num_sms);
    const ws::WsLayout wl = work_layout(p, pl);
    WsParams P;
    memset(&P, 0, sizeof P);
    const int BH = a.B * a.H, BHkv = a.B * a.Hkv;
    if (!tc::encode_3d(&P.tmQ, a.q, D, a.n, BH, CT) || !tc::encode_3d(&P.tmK, a.k, D, a.n, BHkv, CT) ||
        !tc::encode_3d(&P.tmV, a.v, DV, a.n, BHkv, CT) || !tc::encode_3d(&P.tmO, a.o, DV, a.n, BH, CT))
        return cudaErrorInvalidValue;
    P.B = a.B; P.H = a.H; P.n = a.n; P.BH = BH; P.Hkv = a.Hkv;
    P.nchunks = pl.nchunks; P.cpc = pl.cpc; P.kmax = pl.kmax;
    P.runs_per_seq = pl.nchunks % pl.cpc == 0 ? pl.nchunks / pl.cpc : 0;
    // The last piece of each sequence has the deepest scan and alone exports the state: split
    // in two halves when the grid still fits on the device at once, so that its pass 2 and the
    // export no longer end the launch (the piece count stays within kmax = runs + 1).
    int ncta = pl.ncta;
    if (P.runs_per_seq > 1 && pl.cpc % 2 == 0 && P.runs_per_seq + 1 <= pl.kmax &&
        (long long)BH * (P.runs_per_seq + 1) <= (long long)num_sms * ws2_ctas_per_sm(p)) {
        P.tail_split = 1;
        P.runs_per_seq += 1;
        ncta = BH * P.runs_per_seq;
    }
    P.eps = a.eps; P.gamma = a.gamma;
    P.sin = a.sin; P.sout = a.sout;
    uint8_t *wsp = static_cast<uint8_t *>(a.workspace);
    P.ticket = reinterpret_cast<unsigned *>(wsp);
    P.flagA = reinterpret_cast<unsigned *>(wsp + wl.off_flagA);
    P.flagB = reinterpret_cast<unsigned *>(wsp + wl.off_flagB);
    P.summ = reinterpret_cast<float *>(wsp + wl.off_summ);
    P.xpp = reinterpret_cast<float *>(wsp + wl.off_xpp);
    P.err = a.err;
    auto kern = fwd_ws2_kernel<DV, NORM>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L_::SMEM_LAUNCH);
    if (e != cudaSuccess) return e;
    kern<<<ncta, kThreads, L_::SMEM_LAUNCH, st>>>(P);
    return cudaGetLastError();
}
template <bool NORM>
cudaError_t launch_flags(const FwdArgs &a, cudaStream_t st, int ns) {
    return launch_cfg<64, NORM>(a, st, ns);
}
}  // namespace ws2
}  // namespace hla
