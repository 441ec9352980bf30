// hla_fwd_ws.cuh -- warp-specialised chunk-parallel masked second-order HLA
// forward on the sm_103a tensor cores (tcgen05 MMA, TMEM accumulators, TMA),
// bf16 inputs, fp32 accumulation and fp32 state.
//
// Method (gist.science summary of "Higher-order Linear Attention", section 1 for
// the summaries and the masked output, section 4 for the segment concatenation
// and the exclusive scan).  The kernel carries X = S C - G and Y = S m - h
// instead of G, h:
//   X_t = g^2 X_{t-1} + u_t v_t^T,  Y_t = g^2 Y_{t-1} + u_t,  u_t = S_t q_t,
//   o_t = q_t^T X_t,  den_t = q_t^T Y_t,
// and segment A before segment B (f = g^{len B}) concatenate as
//   S = f S_A + S_B, C = f C_A + C_B, m = f m_A + m_B,
//   X = f^2 X_A + X_B + f S_A C_B,  Y = f^2 Y_A + Y_B + f S_A m_B.
// Per chunk of L tokens (local positions tau = 1..L) with state (S_p, X_p, Y_p):
//   A   = tril(Gamma1 o Q K^T),   Gamma1[t,a] = g^{t-a}
//   U   = diag(g^tau) Q S_p + A K                   (rows u_b = S_b q_b)
//   M   = tril(Gamma2 o Q U^T),   Gamma2[t,b] = g^{2(t-b)}
//   O   = M V + diag(g^{2 tau}) Q X_p,  den = rowsum(M) + diag(g^{2 tau}) Q Y_p
//   S  <- g^L S + K^T W K,  X <- g^{2L} X + U^T W^2 V,  W = diag(g^{L - tau}).
//
// Work split: the chunks of all sequences, laid end to end, are cut into equal
// runs, one per CTA; a run holds a piece of every sequence it touches.  CTAs
// take runs in ticket order, so a CTA only waits for CTAs that started before it.
//   pass 1  each piece's summary (S, X, C, m, Y) from zero -> workspace, flag A;
//   scan    the exclusive scan by the concatenation rule without a chain of
//           products: piece k forms S_pre(k) = sum_r F S_r (elementwise), then its
//           own X''_k = X_k + f_k S_pre(k) C_k (one product) -> workspace, flag B;
//           X_pre(k) = sum_{r<k} F^2 X''_r is again elementwise.  (Unrolling the
//           rule: the cross term of piece r only involves the S prefix before r.)
//   pass 2  the chunk loop again from the exact prefix, writing O.
//   export  the CTA holding a sequence's last piece writes state_out.
//
// Roles (320 threads):
//   warp 0      TMA producer: Q, K, V tiles of every chunk into a ring of stages;
//   warp 1      one thread issues every MMA of the chunk loop, in chunk order;
//   warps 2-5   "E": the epilogues on the chain of each chunk (A-tilde, U, M, O),
//               row sums and the normalisation;
//   warps 6-9   "T": the state side: S_p, X_p (bf16 operands) from TMEM and the
//               per-chunk decay of S, X, decay-weighted operand copies, m sums.
// Handoffs are mbarriers (no block barrier inside the chunk loop), so chunk j+1's
// Q K^T and its A-tilde epilogue overlap chunk j's M and O stages, and the state
// extraction runs beside the chain.  E and T together ("all hands", 256 threads)
// run the scan and the export.
#pragma once

#include "hla_fwd_tc.cuh"

namespace hla {
namespace ws {

using tc::cmax;

constexpr int kThreads = 320;
constexpr int kWarpTma = 0, kWarpMma = 1, kWarpE = 2, kWarpT = 6;
constexpr int kBarE = 1, kBarT = 2, kBarAH = 3;  // named barriers (0 is __syncthreads)

struct WsParams {
    CUtensorMap tmQ, tmK, tmV, tmO;
    int B, H, n, BH, Hkv;
    int nchunks, cpc, kmax, runs_per_seq;
    int tail_split;  // the last piece of each sequence split into two halves (runs_per_seq counts both)
    float eps;
    const float *gamma;
    StatePtrs sin, sout;
    unsigned *ticket;  // workspace header (take_ticket, finish_call)
    unsigned *flagA;   // [BH][kmax]: piece summary published
    unsigned *flagB;   // [BH][kmax]: piece X'', Y'' published
    float *summ;       // [BH][kmax][SUM]: S, X, C, m, Y of each piece from zero
    float *xpp;        // [BH][kmax][D*DV + D]: X'', Y'' of each piece
    unsigned *err;
};

// Barrier indices.  Stage barriers come in NST-sized groups.
enum : int {
    B_QF = 0, B_KF = 2, B_VF = 4,    // TMA -> consumers: tile of stage s landed
    B_QE = 6, B_KE = 8, B_VE = 10,   // consumers -> TMA: stage s free (MMA, E, T)
    B_AF = 12,    // MMA -> E: Q K^T (A) in TMEM
    B_AR = 13,    // E -> MMA: A-tilde in smem, A's TMEM drained
    B_UF = 14,    // MMA -> E (and T with decay, pass 1): U accumulated
    B_UR = 15,    // E -> MMA: U (and W^2 U) in smem, U's TMEM drained
    B_MF = 16,    // MMA -> E: Q U^T in TMEM
    B_MR = 17,    // E -> MMA: M in smem, TMEM drained
    B_OF = 18,    // MMA -> E: O accumulated
    B_OFREE = 19, // E -> MMA: O's TMEM drained
    B_ST = 20,    // T -> MMA: S_p (and decay operand copies) ready, S decayed
    B_ST2 = 21,   // T -> MMA (decay): second operand set ready (X_p / W K, W Q)
    B_SD = 22,    // MMA -> T (decay, pass 2): S update done (its operand buffer free)
    B_XD = 23,    // MMA -> T: every MMA of the chunk that reads T's tiles, and the state updates, done
    B_AUX = 24,   // scan / export products (issued by an all-hands thread)
    B_FIN = 25,   // MMA thread's final drain
    NBARS = 26
};

template <int C, int D, int DV, bool DECAY, bool NORM>
struct Lay {
    // ---- TMEM: A slot (Q K^T, Q U^T; pass 1: U; decay pass 2: also A-tilde K and M V),
    // UO slot (pass 2: U or Q S_p, then O or Q X_p; pass 1: C), S, X.
    static constexpr int WA = cmax(cmax(C, D), DECAY ? DV : 0);
    static constexpr int WUO = cmax(D, DV);
    static constexpr uint32_t TA = 0, TUO = WA, TS = WA + WUO, TX = WA + WUO + D;
    static constexpr int TUSED = WA + WUO + D + DV;
    static constexpr int TCOLS = TUSED <= 256 ? 256 : 512;
    static constexpr int CTAS = TCOLS == 256 ? 2 : 1;
    static_assert(TUSED <= 512, "TMEM");
    // ---- shared memory (bytes)
    static constexpr int SQ = C * D * 2, SK = C * D * 2, SV = C * DV * 2, STG = SQ + SK + SV;
    static constexpr int SA = C * cmax(C, D) * 2;                 // A-tilde / M; W Q (pass 1), W^2 U (decay)
    static constexpr int SU = C * D * 2;                          // U (pass 2), W^2 U (pass 1)
    static constexpr int SSP = D * D * 2;                         // S_p
    static constexpr int SXP = cmax(D * DV, DECAY ? C * D : 0) * 2;  // X_p; decay: g^tau Q, W K
    static constexpr int SO = C * DV * 2;                         // output staging
    // fp32 vectors: m, Y running sums [D], row-sum partials [2C], reduction scratch [8D]
    static constexpr int NVEC = 2 * D + 2 * C + 8 * D;
    static constexpr int SMALL = NVEC * 4 + NBARS * 8 + 64;
    static constexpr int LIMIT = CTAS == 2 ? 112 * 1024 : 227 * 1024;
    static constexpr int TILES0 = SA + SU + SSP + SXP;
    static constexpr bool fits(int nst, int no) { return nst * STG + TILES0 + no * SO + SMALL <= LIMIT; }
    static constexpr int NST = fits(2, 1) ? 2 : 1;
    static constexpr int NO = fits(NST, 2) ? 2 : 1;
    static_assert(fits(NST, NO), "shared memory");
    static constexpr int OFF_A = NST * STG, OFF_U = OFF_A + SA, OFF_SP = OFF_U + SU, OFF_XP = OFF_SP + SSP,
                         OFF_O = OFF_XP + SXP, TILES_END = OFF_O + NO * SO;
    // scan / export operands alias the tiles: S hi, S lo [D x D], C hi, C lo [D x DV]
    static constexpr int FOLD = 2 * D * D * 2 + 2 * D * DV * 2;
    static_assert(FOLD <= TILES_END - OFF_A, "scan operands");
    static constexpr int OFF_VEC = TILES_END, OFF_BAR = OFF_VEC + NVEC * 4;
    static constexpr int OFF_MISC = OFF_BAR + NBARS * 8;  // TMEM base, ticket, abort flag
    static constexpr int SMEM = OFF_MISC + 64;
    // request enough shared memory that no more than CTAS CTAs share an SM
    static constexpr int SMEM_LAUNCH = CTAS == 2 ? cmax(SMEM, 78 * 1024) : cmax(SMEM, 120 * 1024);
    // summary layout (floats): S [D*D], X [D*DV], C [D*DV], m [D], Y [D]
    static constexpr int SUM = D * D + 2 * D * DV + 2 * D;
    static constexpr int XPP = D * DV + D;
    static_assert(C == 64 || C == 128, "chunk");
    static_assert(D == 64 || D == 128, "d");
    static_assert(DV == 64 || DV == 128, "dv");
};

// Named barrier over `count` threads.  The ids (kBarE, kBarT, kBarAH) are immediates,
// so that the kernels declare 4 of the 16 hardware barriers (0 is __syncthreads): a
// register id makes the compiler reserve all 16 for the CTA.
__device__ __forceinline__ void nbar(int id, int count) {
    if (id == kBarE) asm volatile("bar.sync 1, %0;" ::"r"(count) : "memory");
    else if (id == kBarT) asm volatile("bar.sync 2, %0;" ::"r"(count) : "memory");
    else asm volatile("bar.sync 3, %0;" ::"r"(count) : "memory");
}
// Named barrier that also ORs a predicate over the participating threads.
__device__ __forceinline__ bool nbar_or(int id, int count, bool v) {
    uint32_t r;
#define HLA_NBAR_OR(ID)                                                                                       \
    asm volatile(                                                                                             \
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, " #ID ", %2, p;\n selp.u32 %0, 1, 0, q;\n}\n" \
        : "=r"(r)                                                                                             \
        : "r"((uint32_t)v), "r"(count)                                                                        \
        : "memory")
    if (id == kBarE) HLA_NBAR_OR(1);
    else if (id == kBarT) HLA_NBAR_OR(2);
    else HLA_NBAR_OR(3);
#undef HLA_NBAR_OR
    return r != 0;
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void bulk_wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }


template <int C, int D, int DV, bool DECAY, bool NORM>
struct Fwd {
    using L_ = Lay<C, D, DV, DECAY, NORM>;
    static constexpr uint32_t TA = L_::TA, TUO = L_::TUO, TS = L_::TS, TX = L_::TX;
    static constexpr int NST = L_::NST;
    const WsParams &P;
    uint8_t *base;
    uint64_t *bars;
    volatile int *abort_p;  // CTA-wide: set once any wait of this CTA gave up
    unsigned tag;           // the value this call's release flags carry
    uint32_t tb;            // TMEM base address
    int tid, warp, lane, quad;
    float lg;               // log2 of the current sequence's decay rate
    int bh, kvh;
    bool need_mY;

    __device__ Fwd(const WsParams &p, uint8_t *b) : P(p), base(b) {}

    // ---------------------------------------------------------------- smem
    __device__ __forceinline__ uint8_t *sQ(int s) const { return base + s * L_::STG; }
    __device__ __forceinline__ uint8_t *sK(int s) const { return sQ(s) + L_::SQ; }
    __device__ __forceinline__ uint8_t *sV(int s) const { return sK(s) + L_::SK; }
    __device__ __forceinline__ uint8_t *tA() const { return base + L_::OFF_A; }
    __device__ __forceinline__ uint8_t *tU() const { return base + L_::OFF_U; }
    __device__ __forceinline__ uint8_t *tSp() const { return base + L_::OFF_SP; }
    __device__ __forceinline__ uint8_t *tXp() const { return base + L_::OFF_XP; }
    __device__ __forceinline__ uint8_t *tO(int b) const { return base + L_::OFF_O + b * L_::SO; }
    __device__ __forceinline__ uint8_t *fShi() const { return base + L_::OFF_A; }
    __device__ __forceinline__ uint8_t *fSlo() const { return fShi() + D * D * 2; }
    __device__ __forceinline__ uint8_t *fChi() const { return fShi() + 2 * D * D * 2; }
    __device__ __forceinline__ uint8_t *fClo() const { return fChi() + D * DV * 2; }
    __device__ __forceinline__ float *vec() const { return reinterpret_cast<float *>(base + L_::OFF_VEC); }
    __device__ __forceinline__ float *mrun() const { return vec(); }               // [D]
    __device__ __forceinline__ float *Yrun() const { return vec() + D; }           // [D]
    __device__ __forceinline__ float *rsum() const { return vec() + 2 * D; }       // [2C]
    __device__ __forceinline__ float *scr() const { return vec() + 2 * D + 2 * C; }  // [8D]
    __device__ __forceinline__ uint64_t *bar(int i) const { return bars + i; }

    // g^x (1 without decay)
    __device__ __forceinline__ float gp(float x) const {
        if constexpr (DECAY) return gpow(lg, x);
        else return 1.f;
    }
    __device__ __forceinline__ uint32_t taddr(uint32_t slot, int col) const {
        return tb + slot + ((uint32_t)(32 * quad) << 16) + (uint32_t)col;
    }

    // ---------------------------------------------------------------- waits
    // Bounded wait for the phase of `b` with parity bit `b` of `ph`, which flips.  A poll
    // sleeps in hardware until the phase completes (mbarrier suspend hint), so waiting
    // warps take no issue slots.  Gives up when the CTA's abort flag is raised, or after
    // the time limit (then it raises the device status word and the abort flag).
    // Uniform over the warp.
    __device__ bool wait(int b, uint32_t &ph) {
        const uint32_t par = (ph >> b) & 1u;
        ph ^= 1u << b;
        bool ok = false;
        if (!*abort_p) {
            ok = mbar_try_wait(bar(b), par);
            if (!ok) ok = wait_slow(b, par);
        }
        return __all_sync(0xffffffffu, ok);
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
    // Single-thread variant (TMA and MMA threads).
    __device__ bool wait1(int b, uint32_t par) {
        if (*abort_p) return false;
        return mbar_try_wait(bar(b), par) || wait_slow(b, par);
    }
    // Spin (bounded) until pieces 0 .. k-1 of sequence bh have set their flag in
    // `flags`; the lanes of the calling warp poll the flags together.
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

    // ---------------------------------------------------------------- MMA groups
    // Issued by a whole warp (one elected lane issues).  Shapes are compile-time; each K
    // step adds a constant (>> 4) to descriptors built once.
    // token-row product, A K-major [C x KD], B K-major [N x KD]
    template <int N, int KD>
    __device__ __forceinline__ void mma_kk(uint32_t slot, const uint8_t *a, const uint8_t *b, bool acc) {
        constexpr uint32_t id = make_idesc(C, N, false, false);
        const uint64_t da = make_sdesc(smem_u32(a), 16u, 1024u), db = make_sdesc(smem_u32(b), 16u, 1024u);
#pragma unroll
        for (int k = 0; k < KD; k += 16) {
            const uint32_t ka = ((uint32_t)(k >> 6) * C * 128u + (uint32_t)(k & 63) * 2u) >> 4;
            const uint32_t kb = ((uint32_t)(k >> 6) * N * 128u + (uint32_t)(k & 63) * 2u) >> 4;
            umma_f16_warp(tb + slot, da + ka, db + kb, id, (acc || k > 0) ? 1u : 0u);
        }
    }
    // token-row product, A K-major [C x KD], B MN-major [KD x N]
    template <int N, int KD>
    __device__ __forceinline__ void mma_km(uint32_t slot, const uint8_t *a, const uint8_t *b, bool acc) {
        constexpr uint32_t id = make_idesc(C, N, false, true);
        const uint64_t da = make_sdesc(smem_u32(a), 16u, 1024u), db = make_sdesc(smem_u32(b), KD * 128u, 1024u);
#pragma unroll
        for (int k = 0; k < KD; k += 16) {
            const uint32_t ka = ((uint32_t)(k >> 6) * C * 128u + (uint32_t)(k & 63) * 2u) >> 4;
            umma_f16_warp(tb + slot, da + ka, db + (uint32_t)(k * 8), id, (acc || k > 0) ? 1u : 0u);
        }
    }
    // state product over tokens: A MN-major [C x D] (as D x C), B MN-major [C x N]
    template <int N>
    __device__ __forceinline__ void mma_mm(uint32_t slot, const uint8_t *a, const uint8_t *b, bool acc) {
        constexpr uint32_t id = make_idesc(D, N, true, true);
        const uint64_t da = make_sdesc(smem_u32(a), C * 128u, 1024u), db = make_sdesc(smem_u32(b), C * 128u, 1024u);
#pragma unroll
        for (int k = 0; k < C; k += 16)
            umma_f16_warp(tb + slot, da + (uint32_t)(k * 8), db + (uint32_t)(k * 8), id, (acc || k > 0) ? 1u : 0u);
    }
    // state x state: A K-major [D x D], B MN-major [D x DV]
    __device__ __forceinline__ void mma_ss(uint32_t slot, const uint8_t *a, const uint8_t *b, bool acc) {
        constexpr uint32_t id = make_idesc(D, DV, false, true);
        const uint64_t da = make_sdesc(smem_u32(a), 16u, 1024u), db = make_sdesc(smem_u32(b), D * 128u, 1024u);
#pragma unroll
        for (int k = 0; k < D; k += 16) {
            const uint32_t ka = ((uint32_t)(k >> 6) * D * 128u + (uint32_t)(k & 63) * 2u) >> 4;
            umma_f16_warp(tb + slot, da + ka, db + (uint32_t)(k * 8), id, (acc || k > 0) ? 1u : 0u);
        }
    }

    // ---------------------------------------------------------------- TMEM rows
    // A group of four warps (one per lane quadrant) reads an accumulator with MR rows
    // and NC columns.  MR = 128: thread (quad, lane) owns row 32 quad + lane, all
    // columns.  MR = 64: rows sit in lanes 0-15 of each quadrant; thread (quad, lane)
    // owns row 16 quad + (lane & 15) and column half (lane >> 4).  f(c0, v[16]) gets
    // 16 consecutive columns from c0.
    template <int MR>
    __device__ __forceinline__ int grow() const {
        return MR == 128 ? 32 * quad + lane : 16 * quad + (lane & 15);
    }
    template <int MR, int NC, typename F>
    __device__ __forceinline__ void g_rows(uint32_t slot, F &&f) {
        float a[16], b[16];
        if constexpr (MR == 128) {
#pragma unroll
            for (int c = 0; c < NC; c += 32) {
                tmem_ld16(taddr(slot, c), a);
                tmem_ld16(taddr(slot, c + 16), b);
                tmem_wait_ld();
                f(c, a);
                f(c + 16, b);
            }
        } else {
            constexpr int HW = NC / 2;
            const int cme = (lane >> 4) * HW;
#pragma unroll
            for (int c = 0; c < HW; c += 32) {
                tmem_ld16x2<HW>(taddr(slot, c), a);
                tmem_ld16x2<HW>(taddr(slot, c + 16), b);
                tmem_wait_ld();
                f(cme + c, a);
                f(cme + c + 16, b);
            }
        }
    }
    // Two accumulators with the same row layout: f(c0, a[16], b[16]).
    template <int MR, int NC, typename F>
    __device__ __forceinline__ void g_rows2(uint32_t s1, uint32_t s2, F &&f) {
        float a[16], b[16];
        if constexpr (MR == 128) {
#pragma unroll
            for (int c = 0; c < NC; c += 16) {
                tmem_ld16(taddr(s1, c), a);
                tmem_ld16(taddr(s2, c), b);
                tmem_wait_ld();
                f(c, a, b);
            }
        } else {
            constexpr int HW = NC / 2;
            const int cme = (lane >> 4) * HW;
#pragma unroll
            for (int c = 0; c < HW; c += 16) {
                tmem_ld16x2<HW>(taddr(s1, c), a);
                tmem_ld16x2<HW>(taddr(s2, c), b);
                tmem_wait_ld();
                f(cme + c, a, b);
            }
        }
    }
    // Read-modify-write: f may change the values, which are stored back.
    template <int MR, int NC, typename F>
    __device__ __forceinline__ void g_rmw(uint32_t slot, F &&f) {
        float a[16];
        if constexpr (MR == 128) {
#pragma unroll
            for (int c = 0; c < NC; c += 16) {
                tmem_ld16(taddr(slot, c), a);
                tmem_wait_ld();
                f(c, a);
                tmem_st16(taddr(slot, c), a);
            }
        } else {
            constexpr int HW = NC / 2;
            const int cme = (lane >> 4) * HW;
#pragma unroll
            for (int c = 0; c < HW; c += 16) {
                tmem_ld16x2<HW>(taddr(slot, c), a);
                tmem_wait_ld();
                f(cme + c, a);
                tmem_st16x2<HW>(taddr(slot, c), a);
            }
        }
        tmem_wait_st();
    }

    // Masked, decayed row of a c x c score tile (columns c0..c0+15 of row `row`):
    // 0 above the diagonal, scaled by g^{POW (row - col)} on and below it.  gt holds
    // g^0, g^POW (one step); off-diagonal groups use one power and multiplications.
    template <int POW>
    __device__ __forceinline__ void mask_row(int row, int c0, float (&v)[16], float gstep) const {
        if (c0 > row) {
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = 0.f;
        } else if (c0 + 15 <= row) {
            if constexpr (DECAY) {
                float f = gp((float)(POW * (row - c0 - 15)));
#pragma unroll
                for (int i = 15; i >= 0; --i) { v[i] *= f; f *= gstep; }
            }
        } else {
            float f = 1.f;
#pragma unroll
            for (int i = 15; i >= 0; --i) {
                const bool keep = (c0 + i <= row);
                if constexpr (DECAY) {
                    v[i] = keep ? v[i] * f : 0.f;
                    f = keep ? f * gstep : f;
                } else {
                    v[i] = keep ? v[i] : 0.f;
                }
            }
        }
    }

    // Row-scaled copy of a [C x Wd] tile by a group of 128 threads (index gt):
    // dst[r] = scale(r) * src[r].
    template <int Wd, typename F>
    __device__ void scaled_copy(int gt, const uint8_t *src, uint8_t *dst, F &&scale) {
        constexpr int GROUPS = Wd / 16;
        for (int e = gt; e < C * GROUPS; e += 128) {
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

    // Column sums of rows r < L of a [C x D] bf16 tile with weights w(r), by a group
    // of 128 threads (index gt, named barrier `nb`): out[i] = sc * out[i] + sum.
    // Thread gt takes an 8-column block and every NG-th row; lanes with the same block
    // combine by shuffles, the four warps in a fixed order through scr (4 x D).
    template <typename Wf>
    __device__ void colsum128(int gt, int nb, const uint8_t *t, int L, Wf &&w, float *scrp, float *out, float sc) {
        constexpr int NB = D / 8, NG = 128 / NB;
        const int cb = gt % NB, rg = gt / NB, wl = gt >> 5;
        float am[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) am[j] = 0.f;
        for (int r = rg; r < L; r += NG) {
            float a[8];
            tile_load_row8(t, C, r, cb * 8, a);
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
        nbar(nb, 128);
        if (gt < D) out[gt] = sc * out[gt] + ((scrp[gt] + scrp[D + gt]) + (scrp[2 * D + gt] + scrp[3 * D + gt]));
        nbar(nb, 128);
    }

    // ======================================================================== stage ring
    // Chunk number `it` (counted over both passes) uses stage it % NST for the
    // (it / NST)-th time; its full barriers complete with that parity.
    __device__ __forceinline__ uint32_t full_par(int it) const { return (uint32_t)((it / NST) & 1); }
    // Multi-thread wait with an explicit parity (stage barriers).
    __device__ bool waitp(int b, uint32_t par) {
        uint32_t ph = par << b;
        return wait(b, ph);
    }
    // Single-thread wait with parity tracking.
    __device__ bool wt(int b, uint32_t &ph) {
        const uint32_t par = (ph >> b) & 1u;
        ph ^= 1u << b;
        return wait1(b, par);
    }

    // ======================================================================== TMA producer
    __device__ bool tma_chunk(int it, int j, int pbh) {
        const int s = it % NST;
        const uint32_t ep = full_par(it) ^ 1u;  // a fresh stage counts as free
        const int t0 = j * C;
        const int pk = (pbh / P.H) * P.Hkv + (pbh % P.H) / (P.H / P.Hkv);
        if (!wait1(B_KE + s, ep)) return false;
        fence_async_smem();  // earlier generic reads of the stage precede the overwrite
        mbar_expect_tx(bar(B_KF + s), L_::SK);
#pragma unroll
        for (int kb = 0; kb < D / 64; ++kb) tma_load_3d(sK(s) + kb * C * 128, &P.tmK, bar(B_KF + s), kb * 64, t0, pk);
        if (!wait1(B_QE + s, ep)) return false;
        fence_async_smem();
        mbar_expect_tx(bar(B_QF + s), L_::SQ);
#pragma unroll
        for (int kb = 0; kb < D / 64; ++kb) tma_load_3d(sQ(s) + kb * C * 128, &P.tmQ, bar(B_QF + s), kb * 64, t0, pbh);
        if (!wait1(B_VE + s, ep)) return false;
        fence_async_smem();
        mbar_expect_tx(bar(B_VF + s), L_::SV);
#pragma unroll
        for (int kb = 0; kb < DV / 64; ++kb) tma_load_3d(sV(s) + kb * C * 128, &P.tmV, bar(B_VF + s), kb * 64, t0, pk);
        return true;
    }
    // After the last load (or an abort): wait, bounded, for the loads that may still
    // be in flight, so that none lands after the CTA has left.
    __device__ void tma_drain(int it_end) {
        for (int it = it_end - NST; it < it_end; ++it) {
            if (it < 0) continue;
            const int s = it % NST;
            const uint32_t fp = full_par(it);
            const int fb[3] = {B_KF, B_QF, B_VF};
#pragma unroll
            for (int q = 0; q < 3; ++q) {
                for (uint32_t i = 0; i < kWaitLimit; ++i) {
                    if (mbar_try_wait(bar(fb[q] + s), fp)) break;
                    if (i > 4096) __nanosleep(64);
                }
            }
        }
    }

    // ======================================================================== MMA thread
    // The MMA warp: all 32 lanes run these programs (waits are warp-wide), one elected
    // lane issues each instruction.
    // Pass 1 (summary from zero).  TMEM: A slot = Q K^T, then U; UO slot = C.
    __device__ bool mma_pass1(int it, bool first, uint32_t &ph) {
        const int s = it % NST;
        const uint32_t fp = full_par(it);
        if (!waitp(B_KF + s, fp) || !waitp(B_QF + s, fp)) return false;
        tc_fence_after();
        uint8_t *Q = sQ(s), *K = sK(s), *V = sV(s);
        mma_kk<C, D>(TA, Q, K, false);  // A = Q K^T
        umma_commit_warp(bar(B_AF));
        if (!wait(B_ST, ph) || !wait(B_AR, ph)) return false;
        tc_fence_after();
        if (!first) mma_kk<D, D>(TA, DECAY ? tXp() : Q, tSp(), false);  // diag(g^tau) Q S_p
        mma_km<D, C>(TA, tA(), K, !first);                               // + A-tilde K
        umma_commit_warp(bar(B_UF));
        if constexpr (!DECAY) mma_mm<D>(TS, K, K, !first);  // S += K^T K
        if (!wait(B_UR, ph)) return false;
        if constexpr (DECAY) {
            if (!wait(B_ST2, ph)) return false;
        }
        if (!waitp(B_VF + s, fp)) return false;
        tc_fence_after();
        if constexpr (DECAY) {
            mma_mm<D>(TS, K, tXp(), !first);   // S += K^T (W K)
            mma_mm<DV>(TUO, tA(), V, !first);  // C += (W' Q)^T V, weights to the segment end
        } else {
            mma_mm<DV>(TUO, Q, V, !first);  // C += Q^T V
        }
        mma_mm<DV>(TX, tU(), V, !first);  // X += (W'^2 U)^T V
        umma_commit_warp(bar(B_XD));
        umma_commit_warp(bar(B_QE + s));
        umma_commit_warp(bar(B_KE + s));
        umma_commit_warp(bar(B_VE + s));
        return true;
    }
    // Pass 2 (outputs).  Without decay: UO slot = Q S_p + A-tilde K (U), then
    // Q X_p + M V (O); A slot = Q K^T, then Q U^T.  With decay the row factors
    // g^tau, g^{2 tau} are applied in the epilogues, so Q S_p and Q X_p go to the
    // UO slot and A-tilde K, M V to the A slot.
    __device__ bool mma_pass2(int it, uint32_t &ph, bool &pend_ofree) {
        const int s = it % NST;
        const uint32_t fp = full_par(it);
        if (!waitp(B_KF + s, fp) || !waitp(B_QF + s, fp)) return false;
        uint8_t *Q = sQ(s), *K = sK(s), *V = sV(s);
        if constexpr (DECAY) {  // the A slot holds the previous chunk's M V until its O epilogue
            if (pend_ofree && !wait(B_OFREE, ph)) return false;
            pend_ofree = false;
        }
        tc_fence_after();
        mma_kk<C, D>(TA, Q, K, false);  // A = Q K^T
        umma_commit_warp(bar(B_AF));
        if (!wait(B_ST, ph)) return false;
        if constexpr (!DECAY) {  // the UO slot holds the previous chunk's O until its epilogue
            if (pend_ofree && !wait(B_OFREE, ph)) return false;
            pend_ofree = false;
        }
        tc_fence_after();
        mma_kk<D, D>(TUO, Q, tSp(), false);  // Q S_p
        if constexpr (DECAY) {
            mma_mm<D>(TS, K, tXp(), true);  // S += K^T (W K)
            umma_commit_warp(bar(B_SD));
        } else {
            mma_mm<D>(TS, K, K, true);  // S += K^T K
        }
        if (!wait(B_AR, ph)) return false;
        tc_fence_after();
        mma_km<D, C>(DECAY ? TA : TUO, tA(), K, !DECAY);  // A-tilde K
        umma_commit_warp(bar(B_UF));
        umma_commit_warp(bar(B_KE + s));
        if (!wait(B_UR, ph)) return false;
        if constexpr (DECAY) {
            // the X update reads W^2 U from the A-tilde tile, which the M epilogue
            // rewrites: it is issued before Q U^T, whose commit the M epilogue waits for
            if (!wait(B_ST2, ph) || !waitp(B_VF + s, fp)) return false;
            tc_fence_after();
            mma_mm<DV>(TX, tA(), V, true);     // X += (W^2 U)^T V
            mma_kk<C, D>(TA, Q, tU(), false);  // Q U^T
            umma_commit_warp(bar(B_MF));
        } else {
            tc_fence_after();
            mma_kk<C, D>(TA, Q, tU(), false);  // Q U^T
            umma_commit_warp(bar(B_MF));
            if (!wait(B_ST2, ph) || !waitp(B_VF + s, fp)) return false;
            tc_fence_after();
        }
        mma_km<DV, D>(TUO, Q, tXp(), false);  // Q X_p
        if constexpr (!DECAY) mma_mm<DV>(TX, tU(), V, true);  // X += U^T V
        umma_commit_warp(bar(B_XD));
        umma_commit_warp(bar(B_QE + s));
        if (!wait(B_MR, ph)) return false;
        tc_fence_after();
        mma_km<DV, C>(DECAY ? TA : TUO, tA(), V, !DECAY);  // M V
        umma_commit_warp(bar(B_OF));
        umma_commit_warp(bar(B_VE + s));
        pend_ofree = true;
        return true;
    }

    // ======================================================================== E group
    // et = tid - 64 in [0, 128); one warp per lane quadrant.
    __device__ __forceinline__ void e_arrive(int b) {
        fence_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(b));
    }
    // T's release of stage s (the MMA thread's commits are the other arrival).  Its
    // reads of the stage are done, and all three tiles of this use have landed, so
    // the arrival cannot count towards the stage's previous use.
    __device__ __forceinline__ void arrive_empties(int s) {
        mbar_arrive(bar(B_QE + s));
        mbar_arrive(bar(B_KE + s));
        mbar_arrive(bar(B_VE + s));
    }
    // A-tilde = tril(Gamma1 o Q K^T) -> tA
    __device__ bool e_atilde(uint32_t &ph) {
        wait(B_AF, ph);
        tc_fence_after();
        const float g1 = gp(1.f);
        const int row = grow<C>();
        g_rows<C, C>(TA, [&](int c0, float (&v)[16]) {
            mask_row<1>(row, c0, v, g1);
            tile_store_row16(tA(), C, row, c0, v);
        });
        e_arrive(B_AR);
        return true;
    }
    // pass 1: U weighted by g^{2 (tokens to the segment end)} -> tU; Y sums
    __device__ bool e_pass1(int it, int L, int rest, uint32_t &ph, int et) {
        e_atilde(ph);
        wait(B_UF, ph);
        tc_fence_after();
        const int row = grow<C>();
        const float w2 = (row < L) ? gp(2.f * (float)(rest + L - 1 - row)) : 0.f;
        g_rows<C, D>(TA, [&](int c0, float (&v)[16]) {
            if constexpr (DECAY) {
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] *= w2;
            }
            tile_store_row16(tU(), C, row, c0, v);
        });
        e_arrive(B_UR);
        if (need_mY) {
            nbar(kBarE, 128);  // the whole tile is written
            colsum128(et, kBarE, tU(), L, [](int) { return 1.f; }, scr(), Yrun(), 1.f);
        }
        return true;
    }
    // pass 2: U, M, O epilogues of one chunk; O leaves through staging buffer ob
    __device__ bool e_pass2(int it, int j, int L, uint32_t &ph, int et, int ob) {
        const int s = it % NST;
        const int row = grow<C>();
        e_atilde(ph);
        float qy = 0.f;
        if constexpr (NORM) {  // g^{2 tau} q . Y_p for this row, before Y moves on
            waitp(B_QF + s, full_par(it));
            const uint8_t *Qs = sQ(s);
            constexpr int CW = C == 128 ? D : D / 2;
            const int cb = C == 128 ? 0 : (lane >> 4) * CW;
#pragma unroll 4
            for (int c = 0; c < CW; c += 8) {
                float q8[8];
                tile_load_row8(Qs, C, row, cb + c, q8);
#pragma unroll
                for (int i = 0; i < 8; ++i) qy += q8[i] * Yrun()[cb + c + i];
            }
            if constexpr (C == 64) qy += __shfl_xor_sync(0xffffffffu, qy, 16);
            qy *= gp(2.f * (float)(row + 1));
        }
        wait(B_UF, ph);
        tc_fence_after();
        if constexpr (DECAY) {  // U = g^tau Q S_p + A-tilde K -> tU;  W^2 U -> tA
            const float gu = gp((float)(row + 1));
            const float w2 = (row < L) ? gp(2.f * (float)(L - 1 - row)) : 0.f;
            g_rows2<C, D>(TA, TUO, [&](int c0, float (&a)[16], float (&sp)[16]) {
#pragma unroll
                for (int i = 0; i < 16; ++i) a[i] += gu * sp[i];
                tile_store_row16(tU(), C, row, c0, a);
#pragma unroll
                for (int i = 0; i < 16; ++i) a[i] *= w2;
                tile_store_row16(tA(), C, row, c0, a);
            });
        } else {
            g_rows<C, D>(TUO, [&](int c0, float (&v)[16]) { tile_store_row16(tU(), C, row, c0, v); });
        }
        e_arrive(B_UR);
        if constexpr (NORM) {  // Y <- g^{2L} Y + sum_b w_b^2 u_b
            nbar(kBarE, 128);
            colsum128(et, kBarE, DECAY ? tA() : tU(), L, [](int) { return 1.f; }, scr(), Yrun(),
                      gp(2.f * (float)L));
        }
        wait(B_MF, ph);
        tc_fence_after();
        {  // M = tril(Gamma2 o Q U^T) -> tA; row sums for the denominator
            const float g2 = gp(2.f);
            float rs = 0.f;
            g_rows<C, C>(TA, [&](int c0, float (&v)[16]) {
                mask_row<2>(row, c0, v, g2);
                if constexpr (NORM) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) rs += v[i];
                }
                tile_store_row16(tA(), C, row, c0, v);
            });
            if constexpr (NORM) rsum()[(C == 128 ? 0 : (lane >> 4) * C) + row] = rs;
        }
        e_arrive(B_MR);
        wait(B_OF, ph);
        tc_fence_after();
        float inv = 1.f;
        // the staging buffer is free once the store issued from it (NO chunks ago) has read it
        if (et == 0) {
            if constexpr (L_::NO == 2) bulk_wait_read1();
            else bulk_wait_read();
        }
        nbar(kBarE, 128);
        if constexpr (NORM) {
            const float rsr = C == 128 ? rsum()[row] : rsum()[row] + rsum()[C + row];
            inv = 1.f / (rsr + qy + P.eps);
        }
        uint8_t *O = tO(ob);
        if constexpr (DECAY) {
            const float g2t = gp(2.f * (float)(row + 1));
            g_rows2<C, DV>(TA, TUO, [&](int c0, float (&a)[16], float (&x)[16]) {
#pragma unroll
                for (int i = 0; i < 16; ++i) a[i] = (a[i] + g2t * x[i]) * inv;
                tile_store_row16(O, C, row, c0, a);
            });
        } else {
            g_rows<C, DV>(TUO, [&](int c0, float (&v)[16]) {
                if constexpr (NORM) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] *= inv;
                }
                tile_store_row16(O, C, row, c0, v);
            });
        }
        fence_async_smem();
        tc_fence_before();
        nbar(kBarE, 128);
        if (et == 0) {
#pragma unroll
            for (int kb = 0; kb < DV / 64; ++kb) tma_store_3d(O + kb * C * 128, &P.tmO, kb * 64, j * C, bh);
            bulk_commit();
        }
        if (lane == 0) mbar_arrive(bar(B_OFREE));
        return true;
    }

    // ======================================================================== T group
    // tt = tid - 192 in [0, 128); one warp per lane quadrant.
    __device__ __forceinline__ void t_arrive(int b) {
        fence_async_smem();
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(b));
    }
    // state [D x NC] in TMEM slot -> bf16 tile with D rows; with decay the slot is
    // then scaled by `dec` in place
    template <int NC>
    __device__ void t_extract(uint32_t slot, uint8_t *tile, float dec) {
        const int row = grow<D>();
        if constexpr (DECAY) {
            g_rmw<D, NC>(slot, [&](int c0, float (&v)[16]) {
                tile_store_row16(tile, D, row, c0, v);
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] *= dec;
            });
        } else {
            g_rows<D, NC>(slot, [&](int c0, float (&v)[16]) { tile_store_row16(tile, D, row, c0, v); });
        }
    }
    __device__ bool t_pass1(int it, int L, int rest, bool first, uint32_t &ph, int tt) {
        const int s = it % NST;
        const uint32_t fp = full_par(it);
        waitp(B_KF + s, fp);
        waitp(B_QF + s, fp);
        if (!first) {  // the previous chunk's MMAs are done: S_p -> tSp, S <- g^L S
            wait(B_XD, ph);
            tc_fence_after();
            t_extract<D>(TS, tSp(), gp((float)L));
        }
        if constexpr (DECAY) scaled_copy<D>(tt, sQ(s), tXp(), [&](int r) { return gp((float)(r + 1)); });
        t_arrive(B_ST);
        if constexpr (DECAY) {  // once Q S_p and A-tilde K ran: W K -> tXp, W' Q -> tA
            wait(B_UF, ph);
            scaled_copy<D>(tt, sK(s), tXp(), [&](int r) { return r < L ? gp((float)(L - 1 - r)) : 0.f; });
            scaled_copy<D>(tt, sQ(s), tA(), [&](int r) { return r < L ? gp((float)(rest + L - 1 - r)) : 0.f; });
            t_arrive(B_ST2);
        }
        if (need_mY)  // m += sum_r g^{rest + L - 1 - r} q_r (fp32 weights)
            colsum128(tt, kBarT, sQ(s), L, [&](int r) { return gp((float)(rest + L - 1 - r)); }, scr() + 4 * D,
                      mrun(), 1.f);
        else
            nbar(kBarT, 128);
        waitp(B_VF + s, fp);
        if (tt == 0) arrive_empties(s);
        return true;
    }
    __device__ bool t_pass2(int it, int L, bool first, uint32_t &ph, int tt) {
        const int s = it % NST;
        const uint32_t fp = full_par(it);
        waitp(B_KF + s, fp);
        if (!first) {  // the previous chunk's MMAs are done
            wait(B_XD, ph);
            tc_fence_after();
        }
        t_extract<D>(TS, tSp(), gp((float)L));  // S_p -> tSp, S <- g^L S
        if constexpr (DECAY)  // W K for the S update, in the X_p buffer until that update ran
            scaled_copy<D>(tt, sK(s), tXp(), [&](int r) { return r < L ? gp((float)(L - 1 - r)) : 0.f; });
        t_arrive(B_ST);
        if constexpr (DECAY) {
            wait(B_SD, ph);
            tc_fence_after();
        }
        t_extract<DV>(TX, tXp(), gp(2.f * (float)L));  // X_p -> tXp, X <- g^{2L} X
        t_arrive(B_ST2);
        waitp(B_QF + s, fp);
        waitp(B_VF + s, fp);
        nbar(kBarT, 128);
        if (tt == 0) arrive_empties(s);
        return true;
    }

    // ======================================================================== all hands
    // Warps 2-9 (256 threads, ah = tid - 64).  A [D x NC] state matrix is shared out
    // by rows: thread (quad, part, lane) owns row grow<D>() and shr<NC>() consecutive
    // columns from shc<NC>() (part = 0 for E warps, 1 for T warps).
    int ah, part;
    int first_run;  // run holding the current sequence's first chunk
    static constexpr int NPR = D == 128 ? 2 : 4;  // threads per row
    __device__ __forceinline__ int rpart() const { return D == 128 ? part : part * 2 + (lane >> 4); }
    template <int NC>
    __host__ __device__ static constexpr int shr() { return D == 128 ? NC / 2 : NC / 4; }
    template <int NC>
    __device__ __forceinline__ int shc() const {
        return D == 128 ? part * (NC / 2) : part * (NC / 2) + (lane >> 4) * (NC / 4);
    }
    template <int NC>
    __device__ __forceinline__ void ld_sh(uint32_t slot, int c, float (&v)[16]) {
        if constexpr (D == 128) tmem_ld16(taddr(slot, part * (NC / 2) + c), v);
        else tmem_ld16x2<NC / 4>(taddr(slot, part * (NC / 2) + c), v);
    }
    template <int NC>
    __device__ __forceinline__ void st_sh(uint32_t slot, int c, const float (&v)[16]) {
        if constexpr (D == 128) tmem_st16(taddr(slot, part * (NC / 2) + c), v);
        else tmem_st16x2<NC / 4>(taddr(slot, part * (NC / 2) + c), v);
    }
    // Summary matrices are stored in share order: the four values (r, c .. c+3) sit at
    // float offset ((c / 4) D + r) 4, so a warp's threads (consecutive rows) touch
    // consecutive 16-byte words.
    static __device__ __forceinline__ int sofs(int r, int c) { return ((c >> 2) * D + r) * 4; }
    static __device__ __forceinline__ void ld_sum16(const float *src, int r, int c, float (&v)[16]) {
#pragma unroll
        for (int i = 0; i < 16; i += 4) {
            const float4 a = tc::ldcg4(src + sofs(r, c + i));
            v[i] = a.x; v[i + 1] = a.y; v[i + 2] = a.z; v[i + 3] = a.w;
        }
    }
    static __device__ __forceinline__ void ld_row16(const float *src, float (&v)[16]) {
#pragma unroll
        for (int i = 0; i < 16; i += 4) {
            const float4 a = *reinterpret_cast<const float4 *>(src + i);
            v[i] = a.x; v[i + 1] = a.y; v[i + 2] = a.z; v[i + 3] = a.w;
        }
    }
    // v += sum_{r<k} w(r) share_r for one 16-column group of a summary matrix; src(r)
    // points at the matrix of piece r.  Loads go out four pieces at a time (the batch
    // past k is padded with piece k-1 at weight 0), so that a group costs ceil(k/4)
    // memory round trips instead of k.
    template <typename Src, typename Wt>
    __device__ __forceinline__ void acc_shares(float (&v)[16], int k, int row, int c, Src &&src, Wt &&w) {
        for (int r = 0; r < k; r += 4) {
            float a[4][16], wr[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int rr = min(r + u, k - 1);
                ld_sum16(src(rr), row, c, a[u]);
                wr[u] = (r + u < k) ? w(r + u) : 0.f;
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] += (wr[0] * a[0][i] + wr[1] * a[1][i]) + (wr[2] * a[2][i] + wr[3] * a[3][i]);
        }
    }
    // sum_{r<k} w(r) src(r)[i] for one vector element, eight pieces per round trip.
    template <typename Src, typename Wt>
    __device__ __forceinline__ float acc_elems(int k, int i, Src &&src, Wt &&w) {
        float y = 0.f;
        for (int r = 0; r < k; r += 8) {
            float a[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) a[u] = __ldcg(src(min(r + u, k - 1)) + i);
#pragma unroll
            for (int u = 0; u < 8; ++u) y += (r + u < k) ? w(r + u) * a[u] : 0.f;
        }
        return y;
    }
    __device__ __forceinline__ void ah_sync() {
        tc_fence_before();
        nbar(kBarAH, 256);
        tc_fence_after();
    }
    // first token of piece r of the current sequence
    __device__ __forceinline__ int tstart(int r) const {
        return r == 0 ? 0 : (int)(((long long)(first_run + r) * P.cpc - (long long)bh * P.nchunks) * C);
    }
    __device__ __forceinline__ const float *summ_of(int r) const {
        return P.summ + ((size_t)bh * P.kmax + r) * L_::SUM;
    }
    __device__ __forceinline__ float *xpp_of(int r) const { return P.xpp + ((size_t)bh * P.kmax + r) * L_::XPP; }
    // warp 2 polls the flags of pieces 0 .. k-1; the barrier carries the acquire to all
    __device__ void ah_wait_flags(const unsigned *flags, int k) {
        if (warp == kWarpE) wait_flags(flags, k);
        ah_sync();
    }
    // products of the scan and the export: UO slot <- S C (three bf16 products on the hi
    // and lo halves approximate the fp32 product), issued by one thread
    __device__ void ah_product(uint32_t &aux_ph) {
        fence_async_smem();
        ah_sync();
        if (warp == kWarpE) {  // issued by one warp, one elected lane
            mma_ss(TUO, fShi(), fChi(), false);
            mma_ss(TUO, fShi(), fClo(), true);
            mma_ss(TUO, fSlo(), fChi(), true);
            umma_commit_warp(bar(B_AUX));
        }
    }
    __device__ void ah_product_wait(uint32_t &aux_ph) {
        wait(B_AUX, aux_ph);
        tc_fence_after();
    }
    // partial dot of this thread's row share of the [D x D] accumulator TS with vec
    __device__ float ah_rowdot_S(const float *vec) {
        constexpr int N = shr<D>();
        const int c0 = shc<D>();
        float acc = 0.f;
#pragma unroll
        for (int c = 0; c < N; c += 16) {
            float v[16];
            ld_sh<D>(TS, c, v);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) acc += v[i] * vec[c0 + c + i];
        }
        return acc;
    }

    // Pass-1 summary (TS, TX, UO slot = C, m, Y) -> dst
    template <int NC>
    __device__ void put_sh(uint32_t slot, float *dst) {
        constexpr int N = shr<NC>();
        const int c0 = shc<NC>(), row = grow<D>();
#pragma unroll
        for (int c = 0; c < N; c += 16) {
            float v[16];
            ld_sh<NC>(slot, c, v);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; i += 4)
                *reinterpret_cast<float4 *>(dst + sofs(row, c0 + c + i)) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
        }
    }
    __device__ void ah_store_summary(float *dst) {
        float *S = dst, *X = S + D * D, *Cc = X + D * DV, *m = Cc + D * DV, *Y = m + D;
        put_sh<D>(TS, S);
        put_sh<DV>(TX, X);
        put_sh<DV>(TUO, Cc);
        for (int i = ah; i < D; i += 256) {
            m[i] = mrun()[i];
            Y[i] = Yrun()[i];
        }
    }

    // S_pre(k) = g^{t_k} S_in + sum_{r<k} g^{t_k - t_{r+1}} S_r -> TS (and the bf16 hi / lo
    // operand tiles when `tiles`)
    __device__ void ah_prefix_S(int k, bool tiles) {
        constexpr int N = shr<D>();
        const int row = grow<D>(), c0 = shc<D>();
        const int tk = tstart(k);
        const float *Si = P.sin.S ? P.sin.S + (size_t)bh * D * D + (size_t)row * D : nullptr;
        const float fin = gp((float)tk);
#pragma unroll
        for (int c = 0; c < N; c += 16) {
            float v[16];
            if (Si) {
                ld_row16(Si + c0 + c, v);
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] *= fin;
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] = 0.f;
            }
            acc_shares(v, k, row, c0 + c, [&](int r) { return summ_of(r); },
                       [&](int r) { return gp((float)(tk - tstart(r + 1))); });
            st_sh<D>(TS, c, v);
            if (tiles) tc::store_hilo(fShi(), fSlo(), D, row, c0 + c, v);
        }
        tmem_wait_st();
    }

    // Scan, step 1 (pieces that have a later piece): X''_k = X_k + S_pre(k) B and
    // Y''_k = Y_k + S_pre(k) b with B = f C_k, b = f m_k (f = g^{len k}); the first
    // piece with a state_in also folds that in: B += f^2 C_in, b += f^2 m_in, minus
    // f^2 G_in, f^2 h_in.  -> workspace, then flag B.
    __device__ void ah_xpp(int k, int len, uint32_t &aux_ph) {
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
        if (k > 0) ah_wait_flags(P.flagA, k);
        ah_prefix_S(k, true);
        const float f = gp((float)len), f2 = f * f;
        const float *Lk = summ_of(k), *Xk = Lk + D * D, *Ck = Xk + D * DV, *mk = Ck + D * DV, *Yk = mk + D;
        const int row = grow<D>(), cv = shc<DV>();
        constexpr int NV = shr<DV>();
        float *bvec = scr(), *pscr = scr() + D;
#pragma unroll
        for (int c = 0; c < NV; c += 16) {
            float a[16];
            ld_sum16(Ck, row, cv + c, a);
#pragma unroll
            for (int i = 0; i < 16; ++i) a[i] *= f;
            if (fold_in) {
                float b[16];
                ld_row16(P.sin.C + ((size_t)bh * D + row) * DV + cv + c, b);
#pragma unroll
                for (int i = 0; i < 16; ++i) a[i] += f2 * b[i];
            }
            tc::store_hilo(fChi(), fClo(), D, row, cv + c, a);
        }
        for (int i = ah; i < D; i += 256)
            bvec[i] = f * __ldcg(mk + i) + (fold_in ? f2 * P.sin.m[(size_t)bh * D + i] : 0.f);
        ah_product(aux_ph);
        // Y'' partials while the products run (bvec is visible after the barrier above)
        pscr[rpart() * D + row] = ah_rowdot_S(bvec);
        ah_product_wait(aux_ph);
        float *Xo = xpp_of(k), *Yo = Xo + D * DV;
#pragma unroll
        for (int c = 0; c < NV; c += 16) {
            float t[16], x[16];
            ld_sh<DV>(TUO, c, t);
            ld_sum16(Xk, row, cv + c, x);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) x[i] += t[i];
            if (fold_in) {
                float g[16];
                ld_row16(P.sin.G + ((size_t)bh * D + row) * DV + cv + c, g);
#pragma unroll
                for (int i = 0; i < 16; ++i) x[i] -= f2 * g[i];
            }
#pragma unroll
            for (int i = 0; i < 16; i += 4)
                *reinterpret_cast<float4 *>(Xo + sofs(row, cv + c + i)) = make_float4(x[i], x[i + 1], x[i + 2], x[i + 3]);
        }
        ah_sync();
        for (int i = ah; i < D; i += 256) {
            float y = __ldcg(Yk + i);
#pragma unroll
            for (int q = 0; q < NPR; ++q) y += pscr[q * D + i];
            if (fold_in) y -= f2 * P.sin.h[(size_t)bh * D + i];
            Yo[i] = y;
        }
        ah_sync();  // every store of X'', Y'' precedes the release
        if (ah == 0) {
            unsigned *fl = P.flagB + (size_t)bh * P.kmax + k;
            asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(fl), "r"(tag) : "memory");
        }
    }

    // Scan, step 2 and the pass-2 start state of piece k: TS = S_pre(k), TX = X_pre(k),
    // Yrun = Y_pre(k); for a sequence's last piece with state_out also Y_end = f^2 Y_pre +
    // Y_k + f S_pre m_k, which needs S_pre (state_out.h holds it until the export).
    __device__ void ah_setup_pass2(int k, int len, bool last, bool want_out, uint32_t &aux_ph) {
        const bool sin = P.sin.S != nullptr;
        const int row = grow<D>(), cv = shc<DV>();
        constexpr int NV = shr<DV>();
        float *bvec = scr(), *pscr = scr() + D;
        if (k > 0 || sin) {
            if (k > 0) ah_wait_flags(P.flagA, k);
            ah_prefix_S(k, k == 0);
        } else {
            float z[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) z[i] = 0.f;
#pragma unroll
            for (int c = 0; c < shr<D>(); c += 16) st_sh<D>(TS, c, z);
            tmem_wait_st();
        }
        if (k > 0) {  // X_pre = sum_{r<k} g^{2 (t_k - t_{r+1})} X''_r, Y_pre likewise
            ah_wait_flags(P.flagB, k);
            const int tk = tstart(k);
            auto wx = [&](int r) { return gp(2.f * (float)(tk - tstart(r + 1))); };
            auto xsrc = [&](int r) -> const float * { return (r == 0 && !sin) ? summ_of(0) + D * D : xpp_of(r); };
#pragma unroll
            for (int c = 0; c < NV; c += 16) {
                float v[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] = 0.f;
                acc_shares(v, k, row, cv + c, xsrc, wx);
                st_sh<DV>(TX, c, v);
            }
            tmem_wait_st();
            auto ysrc = [&](int r) -> const float * {
                return (r == 0 && !sin) ? summ_of(0) + D * D + 2 * D * DV + D : xpp_of(r) + D * DV;
            };
            for (int i = ah; i < D; i += 256) Yrun()[i] = acc_elems(k, i, ysrc, wx);
        } else if (sin) {  // X_pre = X_in = S_in C_in - G_in, Y_pre = S_in m_in - h_in
#pragma unroll
            for (int c = 0; c < NV; c += 16) {
                float a[16];
                ld_row16(P.sin.C + ((size_t)bh * D + row) * DV + cv + c, a);
                tc::store_hilo(fChi(), fClo(), D, row, cv + c, a);
            }
            for (int i = ah; i < D; i += 256) bvec[i] = P.sin.m[(size_t)bh * D + i];
            ah_product(aux_ph);
            pscr[rpart() * D + row] = ah_rowdot_S(bvec);
            ah_product_wait(aux_ph);
#pragma unroll
            for (int c = 0; c < NV; c += 16) {
                float t[16], g[16];
                ld_sh<DV>(TUO, c, t);
                ld_row16(P.sin.G + ((size_t)bh * D + row) * DV + cv + c, g);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i) t[i] -= g[i];
                st_sh<DV>(TX, c, t);
            }
            tmem_wait_st();
            ah_sync();
            for (int i = ah; i < D; i += 256) {
                float y = -P.sin.h[(size_t)bh * D + i];
#pragma unroll
                for (int q = 0; q < NPR; ++q) y += pscr[q * D + i];
                Yrun()[i] = y;
            }
        } else {
            float z[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) z[i] = 0.f;
#pragma unroll
            for (int c = 0; c < NV; c += 16) st_sh<DV>(TX, c, z);
            tmem_wait_st();
            for (int i = ah; i < D; i += 256) Yrun()[i] = 0.f;
        }
        if (last && want_out) {  // Y_end = f^2 Y_pre + Y_k + f S_pre m_k (S_pre is still in TS)
            const float f = gp((float)len);
            const float *mk = summ_of(k) + D * D + 2 * D * DV, *Yk = mk + D;
            for (int i = ah; i < D; i += 256) bvec[i] = __ldcg(mk + i);
            ah_sync();
            pscr[rpart() * D + row] = ah_rowdot_S(bvec);
            ah_sync();
            for (int i = ah; i < D; i += 256) {
                float sm = 0.f;
#pragma unroll
                for (int q = 0; q < NPR; ++q) sm += pscr[q * D + i];
                P.sout.h[(size_t)bh * D + i] = __ldcg(Yk + i) + f * f * Yrun()[i] + f * sm;  // Y_end until the export
            }
        }
        ah_sync();
    }

    // After pass 2 of a sequence's last piece k (length len): S_end, X_end in TMEM, Y_end
    // in state_out.h.  C_end = f (g^{t_k} C_in + sum_r g^{t_k - t_{r+1}} C_r) + C_k and m_end
    // likewise (f = g^{len}) -> state_out; G = S C - X (hi / lo products), h = S m - Y.
    __device__ void ah_export_post(int k, int len, uint32_t &aux_ph) {
        const bool sin = P.sin.S != nullptr;
        const int row = grow<D>(), cs = shc<D>(), cv = shc<DV>();
        constexpr int NS = shr<D>(), NV = shr<DV>();
        float *So = P.sout.S + ((size_t)bh * D + row) * D, *Co = P.sout.C + ((size_t)bh * D + row) * DV;
        float *Go = P.sout.G + ((size_t)bh * D + row) * DV;
        float *mo = P.sout.m + (size_t)bh * D;
        float *ho = P.sout.h + (size_t)bh * D;
        float *pscr = scr() + D;
        const float f = gp((float)len);
        const int tk = tstart(k);
        const float fin = gp((float)tk);
        auto wc = [&](int r) { return gp((float)(tk - tstart(r + 1))); };
        const float *Ck = summ_of(k) + D * D + D * DV, *mk = Ck + D * DV;
#pragma unroll
        for (int c = 0; c < NV; c += 16) {
            float v[16];
            if (sin) {
                ld_row16(P.sin.C + ((size_t)bh * D + row) * DV + cv + c, v);
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] *= fin;
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] = 0.f;
            }
            acc_shares(v, k, row, cv + c, [&](int r) { return summ_of(r) + D * D + D * DV; }, wc);
            float a[16];
            ld_sum16(Ck, row, cv + c, a);
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = f * v[i] + a[i];
            tc::st_row16(Co + cv + c, v);
            tc::store_hilo(fChi(), fClo(), D, row, cv + c, v);
        }
        for (int i = ah; i < D; i += 256) {
            const float mp = (sin ? fin * P.sin.m[(size_t)bh * D + i] : 0.f) +
                             acc_elems(k, i, [&](int r) { return summ_of(r) + D * D + 2 * D * DV; }, wc);
            mo[i] = f * mp + __ldcg(mk + i);
        }
        ah_sync();  // m_end complete
        float sm = 0.f;
#pragma unroll
        for (int c = 0; c < NS; c += 16) {
            float v[16];
            ld_sh<D>(TS, c, v);
            tmem_wait_ld();
            tc::store_hilo(fShi(), fSlo(), D, row, cs + c, v);
            tc::st_row16(So + cs + c, v);
#pragma unroll
            for (int i = 0; i < 16; ++i) sm += v[i] * mo[cs + c + i];
        }
        pscr[rpart() * D + row] = sm;
        ah_product(aux_ph);
        for (int i = ah; i < D; i += 256) {
            float h = -ho[i];
#pragma unroll
            for (int q = 0; q < NPR; ++q) h += pscr[q * D + i];
            ho[i] = h;
        }
        ah_product_wait(aux_ph);
#pragma unroll
        for (int c = 0; c < NV; c += 16) {
            float t[16], x[16];
            ld_sh<DV>(TUO, c, t);
            ld_sh<DV>(TX, c, x);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) t[i] -= x[i];
            tc::st_row16(Go + cv + c, t);
        }
    }
};

// Every thread of the CTA, after its last read of a flag (finish_call).
__device__ __forceinline__ void finish_cta(const WsParams &P, unsigned tag, volatile unsigned *s_last) {
    finish_call(P.ticket, tag, P.flagA, P.flagB, P.BH * P.kmax, s_last);
}

template <int C, int D, int DV, bool DECAY, bool NORM>
__global__ void __launch_bounds__(kThreads, Lay<C, D, DV, DECAY, NORM>::CTAS)
    fwd_ws_kernel(const __grid_constant__ WsParams P) {
    using L_ = Lay<C, D, DV, DECAY, NORM>;
    // No static shared memory: the dynamic block starts at the (1024-byte aligned)
    // base of the CTA's shared window, which the swizzled tiles need.
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *base = smem_raw;
    Fwd<C, D, DV, DECAY, NORM> x(P, base);
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
    x.lg = 0.f;
    if (x.tid == 0) {
        misc[2] = 0u;
        misc[3] = (smem_u32(base) & 1023u) != 0;
        for (int s = 0; s < L_::NST; ++s) {
            mbar_init(x.bar(B_QF + s), 1);
            mbar_init(x.bar(B_KF + s), 1);
            mbar_init(x.bar(B_VF + s), 1);
            mbar_init(x.bar(B_QE + s), 2);  // the MMA thread's commit and T's arrival
            mbar_init(x.bar(B_KE + s), 2);
            mbar_init(x.bar(B_VE + s), 2);
        }
        const int one[8] = {B_AF, B_UF, B_MF, B_OF, B_SD, B_XD, B_AUX, B_FIN};
        const int four[6] = {B_AR, B_UR, B_MR, B_OFREE, B_ST, B_ST2};  // one arrival per warp of a group
        for (int i = 0; i < 8; ++i) mbar_init(x.bar(one[i]), 1);
        for (int i = 0; i < 6; ++i) mbar_init(x.bar(four[i]), 4);
        fence_mbar_init();
        tma_prefetch_desc(&P.tmQ);
        tma_prefetch_desc(&P.tmK);
        tma_prefetch_desc(&P.tmV);
        tma_prefetch_desc(&P.tmO);
    }
    __syncthreads();
    if (misc[3]) {  // cannot happen with no static shared memory; refuse rather than corrupt
        if (x.tid == 0) {
            atomicOr(P.err, DEV_TIMEOUT);
            misc[5] = take_ticket(P.ticket).tag;
        }
        __syncthreads();
        finish_cta(P, misc[5], misc + 4);
        return;
    }
    // TMEM first, then the ticket: a CTA that waits for TMEM holds no ticket that
    // other CTAs could be waiting for.
    if (x.warp == kWarpMma) {
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

    // This CTA's run of chunks [g0, g1) in the end-to-end order of all sequences, and
    // the pieces it holds: one per sequence the run touches.
    const long long NCH = P.nchunks;
    const int run = P.runs_per_seq > 0 ? (ticket % P.BH) * P.runs_per_seq + ticket / P.BH : ticket;
    const long long g0 = (long long)run * P.cpc;
    const long long g1 = min((long long)P.BH * NCH, g0 + P.cpc);
    const int bh_lo = (int)(g0 / NCH), bh_hi = (int)((g1 - 1) / NCH);
    struct Piece {
        int jb, je, k, len;
        bool last;
    };
    auto piece = [&](int bh) {
        Piece pc;
        pc.jb = (int)(max(g0, bh * NCH) - bh * NCH);
        pc.je = (int)(min(g1, (bh + 1) * NCH) - bh * NCH);
        pc.k = (int)(run - (bh * NCH) / P.cpc);
        pc.last = (pc.je == P.nchunks);
        pc.len = min(P.n, pc.je * C) - pc.jb * C;
        return pc;
    };
    auto select = [&](int bh) {
        x.bh = bh;
        x.kvh = (bh / P.H) * P.Hkv + (bh % P.H) / (P.H / P.Hkv);
        x.first_run = (int)((bh * NCH) / P.cpc);
        float g = 1.f;
        if constexpr (DECAY) g = P.gamma[bh % P.H];
        x.lg = log2f(g);
    };

    if (x.warp == kWarpTma) {
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
    } else if (x.warp == kWarpMma) {
        int it = 0;
        uint32_t ph = 0;
        bool ok = true, pend_ofree = false;
        for (int bh = bh_lo; bh <= bh_hi && ok; ++bh) {
            const Piece pc = piece(bh);
            if (pc.last && !want_out) continue;
            for (int j = pc.jb; j < pc.je && ok; ++j) ok = x.mma_pass1(it++, j == pc.jb, ph);
        }
        for (int bh = bh_lo; bh <= bh_hi && ok; ++bh) {
            const Piece pc = piece(bh);
            for (int j = pc.jb; j < pc.je && ok; ++j) ok = x.mma_pass2(it++, ph, pend_ofree);
        }
        // every MMA issued has completed before TMEM is released
        umma_commit_warp(x.bar(B_FIN));
        mbar_wait(x.bar(B_FIN), 0u, P.err);
        __syncwarp();
    } else {
        // E (warps 2-5) and T (warps 6-9).  After an expired wait these keep running
        // the same control flow (every wait then returns at once), so that their named
        // barriers stay matched.
        const bool isE = x.warp < kWarpT;
        const int gt = isE ? (int)threadIdx.x - 64 : (int)threadIdx.x - 192;
        uint32_t ph = 0, aux_ph = 0;
        int it = 0, ob = 0;
        // ---- phase 1: the summary of every piece that a later piece or the export needs
        for (int bh = bh_lo; bh <= bh_hi; ++bh) {
            const Piece pc = piece(bh);
            if (pc.last && !want_out) continue;
            select(bh);
            if (x.need_mY) {
                if (gt < D) (isE ? x.Yrun() : x.mrun())[gt] = 0.f;
                nbar(isE ? kBarE : kBarT, 128);
            }
            for (int j = pc.jb; j < pc.je; ++j) {
                const int L = min(C, P.n - j * C);
                const int rest = pc.len - (j - pc.jb) * C - L;
                if (isE) x.e_pass1(it, L, rest, ph, gt);
                else x.t_pass1(it, L, rest, j == pc.jb, ph, gt);
                ++it;
            }
            if (!isE) {  // the piece's last state updates are done
                x.wait(B_XD, ph);
                tc_fence_after();
            }
            x.ah_sync();
            x.ah_store_summary(P.summ + ((size_t)bh * P.kmax + pc.k) * L_::SUM);
            x.ah_sync();
            if (x.ah == 0 && !pc.last) {
                unsigned *f = P.flagA + (size_t)bh * P.kmax + pc.k;
                asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(f), "r"(x.tag) : "memory");
            }
        }
        // ---- scan, step 1: X'', Y'' of every piece that has a later piece
        for (int bh = bh_lo; bh <= bh_hi; ++bh) {
            const Piece pc = piece(bh);
            if (pc.last) continue;
            select(bh);
            x.ah_xpp(pc.k, pc.len, aux_ph);
        }
        // ---- scan, step 2, then pass 2 (and the export) per piece
        for (int bh = bh_lo; bh <= bh_hi; ++bh) {
            const Piece pc = piece(bh);
            select(bh);
            x.ah_setup_pass2(pc.k, pc.len, pc.last, want_out, aux_ph);
            for (int j = pc.jb; j < pc.je; ++j) {
                const int L = min(C, P.n - j * C);
                if (isE) x.e_pass2(it, j, L, ph, gt, ob);
                else x.t_pass2(it, L, j == pc.jb, ph, gt);
                ++it;
                ob ^= (L_::NO - 1);
            }
            if (!isE) {
                x.wait(B_XD, ph);
                tc_fence_after();
            }
            if (isE && gt == 0) bulk_wait_read();  // the staging buffers (scan operand space) are read
            x.ah_sync();
            if (pc.last && want_out) x.ah_export_post(pc.k, pc.len, aux_ph);
            x.ah_sync();
        }
        if (isE && gt == 0) bulk_wait_all();  // the output stores are complete before the CTA counts itself done
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (x.warp == kWarpMma) tmem_dealloc(x.tb, L_::TCOLS);
    finish_cta(P, x.tag, misc + 4);
}

// ============================================================================ host side
struct WsLayout {
    size_t off_flagA, off_flagB, off_summ, off_xpp, total;
};
inline int ws_ctas_per_sm(const hla_params &p) {
    const bool decay = (p.flags & HLA_DECAY) != 0;
    const int WA = cmax(cmax(p.chunk, p.d), decay ? p.dv : 0), WUO = cmax(p.d, p.dv);
    return WA + WUO + p.d + p.dv <= 256 ? 2 : 1;
}
inline tc::Plan work_plan(const hla_params &p, int num_sms) {
    tc::Plan pl;
    const long long BH = (long long)p.B * p.H;
    pl.nchunks = (p.n + p.chunk - 1) / p.chunk;
    const long long total = BH * pl.nchunks;
    const long long slots = (long long)num_sms * ws_ctas_per_sm(p);
    long long cpc = (total + slots - 1) / (slots > 0 ? slots : 1);
    if (cpc < 1) cpc = 1;
    pl.cpc = (int)cpc;
    pl.ncta = (int)((total + cpc - 1) / cpc);
    if (pl.ncta < 1) pl.ncta = 1;
    pl.kmax = (pl.nchunks + pl.cpc - 1) / pl.cpc + 1;
    return pl;
}
inline WsLayout work_layout(const hla_params &p, const tc::Plan &pl) {
    const size_t BH = (size_t)p.B * p.H, D = p.d, DV = p.dv;
    const size_t SUM = D * D + 2 * D * DV + 2 * D, XPP = D * DV + D;
    WsLayout w;
    w.off_flagA = 256;
    w.off_flagB = w.off_flagA + BH * pl.kmax * 4;
    w.off_summ = tc::align256(w.off_flagB + BH * pl.kmax * 4);
    w.off_xpp = tc::align256(w.off_summ + BH * pl.kmax * SUM * 4);
    w.total = tc::align256(w.off_xpp + BH * pl.kmax * XPP * 4);
    return w;
}

template <int C, int D, int DV, bool DECAY, bool NORM>
cudaError_t ws_launch_cfg(const FwdArgs &a, cudaStream_t st, int num_sms) {
    using L_ = Lay<C, D, DV, DECAY, NORM>;
    hla_params p{a.B, a.H, a.n, a.d, a.dv, a.chunk, a.in_dtype, a.flags, a.eps, a.gamma};
    const tc::Plan pl = work_plan(p, num_sms);
    const WsLayout wl = work_layout(p, pl);
    WsParams P;
    memset(&P, 0, sizeof P);
    const int BH = a.B * a.H, BHkv = a.B * a.Hkv;
    if (!tc::encode_3d(&P.tmQ, a.q, D, a.n, BH, C) || !tc::encode_3d(&P.tmK, a.k, D, a.n, BHkv, C) ||
        !tc::encode_3d(&P.tmV, a.v, DV, a.n, BHkv, C) || !tc::encode_3d(&P.tmO, a.o, DV, a.n, BH, C))
        return cudaErrorInvalidValue;
    P.B = a.B; P.H = a.H; P.n = a.n; P.BH = BH; P.Hkv = a.Hkv;
    P.nchunks = pl.nchunks; P.cpc = pl.cpc; P.kmax = pl.kmax;
    P.runs_per_seq = pl.nchunks % pl.cpc == 0 ? pl.nchunks / pl.cpc : 0;
    P.eps = a.eps; P.gamma = a.gamma;
    P.sin = a.sin; P.sout = a.sout;
    uint8_t *ws = static_cast<uint8_t *>(a.workspace);
    P.ticket = reinterpret_cast<unsigned *>(ws);
    P.flagA = reinterpret_cast<unsigned *>(ws + wl.off_flagA);
    P.flagB = reinterpret_cast<unsigned *>(ws + wl.off_flagB);
    P.summ = reinterpret_cast<float *>(ws + wl.off_summ);
    P.xpp = reinterpret_cast<float *>(ws + wl.off_xpp);
    P.err = a.err;
    auto kern = fwd_ws_kernel<C, D, DV, DECAY, NORM>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L_::SMEM_LAUNCH);
    if (e != cudaSuccess) return e;
    kern<<<pl.ncta, kThreads, L_::SMEM_LAUNCH, st>>>(P);
    return cudaGetLastError();
}

// Shapes served by this kernel: the masked variant with d = 64.
inline bool ws_supported(const hla_params &p) {
    return !(p.flags & (HLA_UNMASKED | HLA_ASYMMETRIC)) && p.in_dtype == HLA_BF16 && p.d == 64 &&
           (p.dv == 64 || p.dv == 128) && (p.chunk == 64 || p.chunk == 128);
}
template <bool DECAY, bool NORM>
cudaError_t ws_launch_flags(const FwdArgs &a, cudaStream_t st, int ns) {
    const int key = (a.chunk == 128 ? 2 : 0) | (a.dv == 128 ? 1 : 0);
    switch (key) {
        case 0: return ws_launch_cfg<64, 64, 64, DECAY, NORM>(a, st, ns);
        case 1: return ws_launch_cfg<64, 64, 128, DECAY, NORM>(a, st, ns);
        case 2: return ws_launch_cfg<128, 64, 64, DECAY, NORM>(a, st, ns);
        default: return ws_launch_cfg<128, 64, 128, DECAY, NORM>(a, st, ns);
    }
}
}  // namespace ws
}  // namespace hla
