// hla_fwd3_maps.cu -- the segment maps of masked third-order HLA and the concatenation
// of third-order states ("Higher-order Linear Attention", gist.science summary,
// section 4, bullet "Derde-orde scans": segment-level linear maps compose third-order
// states exactly).  Segment A before segment B, f = g^(tokens of B) (1 without decay):
//   S^K = f S^K_A + S^K_B,  S^Q = f S^Q_A + S^Q_B,  P = f P_A + P_B,
//   T    = f^3 T_A + T_B + f S^K_A M^QP_B + f M^KQ_B P_A + f^2 S^K_A S^Q_B P_A,
//   M^QP = f^2 M^QP_A + M^QP_B + f S^Q_B P_A,
//   M^KQ = f^2 M^KQ_A + M^KQ_B + f S^K_A S^Q_B,
// and, normalised, the unit column (m as P, h as T, mqm as M^QP).
//
// The maps of a whole forward: folding the chunks' local sums with the rule above,
// the contribution of chunk c to the sequence's maps is independent of the other
// chunks once its prefix state (S^K_p, P_p, which the scan writes anyway) is known:
//   S^Q  += F_c S^Q_c,
//   M^QP += F_c^2 (M^QP_c + f_c S^Q_c P_p(c)),
//   M^KQ += F_c^2 (M^KQ_c + f_c S^K_p(c) S^Q_c),
// F_c = g^(tokens after chunk c), f_c = g^(tokens of chunk c), on top of the state_in
// maps scaled by g^(n) (S^Q) and g^(2n) (M^QP, M^KQ).  One CTA per chunk adds its part.
#include "hla_fwd3_simt.cuh"

namespace hla {
namespace fwd3 {
namespace {

__device__ __forceinline__ float powg(const float *gamma, int H, int u, int x) {
    return gamma ? gpow(log2f(gamma[u % H]), (float)x) : 1.f;
}

// out maps = state_in maps (scaled to the segment end) or zeros
__global__ void __launch_bounds__(kThreads) maps_init_kernel(Fwd3Args a) {
    const int u = blockIdx.x, D = a.d, DV = a.dv;
    const float F = powg(a.gamma, a.H, u, a.n), F2 = F * F;
    const size_t oD = (size_t)u * D * D, oV = (size_t)u * D * DV;
    for (int e = threadIdx.x; e < D * D; e += kThreads) {
        a.sout_SQ[oD + e] = a.sin_SQ ? F * a.sin_SQ[oD + e] : 0.f;
        a.sout_MKQ[oD + e] = a.sin_MKQ ? F2 * a.sin_MKQ[oD + e] : 0.f;
    }
    for (int e = threadIdx.x; e < D * DV; e += kThreads) a.sout_MQP[oV + e] = a.sin_MQP ? F2 * a.sin_MQP[oV + e] : 0.f;
}

template <int D, int DV>
struct MapsSmem {
    static constexpr int LD = D + 4, LV = DV + 4;
    static constexpr int SQ = 0, SK = SQ + D * LD, PP = SK + D * LD, TOTAL = PP + D * LV;
};

template <int D, int DV>
__global__ void __launch_bounds__(kThreads) maps_chunk_kernel(Fwd3Args a) {
    using Sm = MapsSmem<D, DV>;
    extern __shared__ __align__(16) float sm[];
    float *SQ = sm + Sm::SQ, *SK = sm + Sm::SK, *PP = sm + Sm::PP;
    const int C = a.chunk, nch = (a.n + C - 1) / C, u = blockIdx.x / nch, ch = blockIdx.x % nch;
    const int L = min(C, a.n - ch * C), after = a.n - min(a.n, (ch + 1) * C);
    const float f = powg(a.gamma, a.H, u, L), F = powg(a.gamma, a.H, u, after), F2 = F * F;
    const Ws3 ws{D, DV};
    const float *lc = a.workspace + ((size_t)u * nch + ch) * ws.loc_floats();
    const float *so =
        a.workspace + (size_t)a.B * a.H * nch * ws.loc_floats() + ((size_t)u * nch + ch) * ws.st_floats();
    for (int e = threadIdx.x; e < D * D; e += kThreads) {
        SQ[(e / D) * Sm::LD + e % D] = lc[ws.o_sq() + e];
        SK[(e / D) * Sm::LD + e % D] = so[ws.s_sk() + e];
    }
    for (int e = threadIdx.x; e < D * DV; e += kThreads) PP[(e / DV) * Sm::LV + e % DV] = so[ws.s_p() + e];
    __syncthreads();
    const size_t oD = (size_t)u * D * D, oV = (size_t)u * D * DV;
    for (int e = threadIdx.x; e < D * D; e += kThreads) atomicAdd(a.sout_SQ + oD + e, F * lc[ws.o_sq() + e]);
    tiles<false, D, DV>([&](float (&acc)[4][4], int m0, int n0, int ns) {
        mac<false, false>(acc, SQ, Sm::LD, PP, Sm::LV, m0, n0, ns, D);
        each(acc, m0, n0, ns, [&](int i, int j, float x) {
            atomicAdd(a.sout_MQP + oV + (size_t)i * DV + j, F2 * (lc[ws.o_mqp() + (size_t)i * DV + j] + f * x));
        });
    });
    tiles<false, D, D>([&](float (&acc)[4][4], int m0, int n0, int ns) {
        mac<false, false>(acc, SK, Sm::LD, SQ, Sm::LD, m0, n0, ns, D);
        each(acc, m0, n0, ns, [&](int i, int j, float x) {
            atomicAdd(a.sout_MKQ + oD + (size_t)i * D + j, F2 * (lc[ws.o_mkq() + (size_t)i * D + j] + f * x));
        });
    });
}

template <int D, int DV>
cudaError_t maps_t(const Fwd3Args &a, cudaStream_t st) {
    const int nch = (a.n + a.chunk - 1) / a.chunk, units = a.B * a.H;
    maps_init_kernel<<<units, kThreads, 0, st>>>(a);
    constexpr size_t bytes = MapsSmem<D, DV>::TOTAL * sizeof(float);
    cudaError_t e = smem_attr(maps_chunk_kernel<D, DV>, bytes);
    if (e != cudaSuccess) return e;
    if (nch > 0) maps_chunk_kernel<D, DV><<<units * nch, kThreads, bytes, st>>>(a);
    return cudaGetLastError();
}

// ---- concatenation of states with their maps, one CTA per item
struct Comb3 {
    int count, d, dv;
    bool norm;
    hla_state3 A, B, out;
    const float *decay_pow;
};

template <int D, int DV>
struct CombSmem {
    static constexpr int LD = D + 4, LV = DV + 4;
    static constexpr int SKA = 0, SQB = SKA + D * LD, MKQB = SQB + D * LD, W = MKQB + D * LD, PA = W + D * LD,
                         MQPB = PA + D * LV, VEC = MQPB + D * LV, TOTAL = VEC + 2 * D;
};

template <int D, int DV>
__global__ void __launch_bounds__(kThreads) combine3_kernel(Comb3 c) {
    using Sm = CombSmem<D, DV>;
    extern __shared__ __align__(16) float sm[];
    float *SKA = sm + Sm::SKA, *SQB = sm + Sm::SQB, *MKQB = sm + Sm::MKQB, *W = sm + Sm::W, *PA = sm + Sm::PA,
          *MQPB = sm + Sm::MQPB, *mA = sm + Sm::VEC, *mqmB = mA + D;
    const int i0 = blockIdx.x;
    const float f = c.decay_pow ? c.decay_pow[i0] : 1.f, f2 = f * f, f3 = f2 * f;
    const size_t oD = (size_t)i0 * D * D, oV = (size_t)i0 * D * DV, od = (size_t)i0 * D;
    for (int e = threadIdx.x; e < D * D; e += kThreads) {
        const int o = (e / D) * Sm::LD + e % D;
        SKA[o] = c.A.S[oD + e];
        SQB[o] = c.B.SQ[oD + e];
        MKQB[o] = c.B.MKQ[oD + e];
    }
    for (int e = threadIdx.x; e < D * DV; e += kThreads) {
        const int o = (e / DV) * Sm::LV + e % DV;
        PA[o] = c.A.P[oV + e];
        MQPB[o] = c.B.MQP[oV + e];
    }
    if (c.norm)
        for (int e = threadIdx.x; e < D; e += kThreads) {
            mA[e] = c.A.m[od + e];
            mqmB[e] = c.B.mqm[od + e];
        }
    __syncthreads();
    // W = S^K_A S^Q_B
    tiles<false, D, D>([&](float (&acc)[4][4], int m0, int n0, int ns) {
        mac<false, false>(acc, SKA, Sm::LD, SQB, Sm::LD, m0, n0, ns, D);
        each(acc, m0, n0, ns, [&](int i, int j, float x) { W[i * Sm::LD + j] = x; });
    });
    __syncthreads();
    // T, M^QP (elementwise parts of A and B read by the thread that writes the element)
    tiles<false, D, DV>([&](float (&acc)[4][4], int m0, int n0, int ns) {
        float sq_p[4][4] = {}, t[4][4] = {};
        mac<false, false>(t, SKA, Sm::LD, MQPB, Sm::LV, m0, n0, ns, D);  // S^K_A M^QP_B
        mac<false, false>(t, MKQB, Sm::LD, PA, Sm::LV, m0, n0, ns, D);   // + M^KQ_B P_A
        mac<false, false>(acc, W, Sm::LD, PA, Sm::LV, m0, n0, ns, D);    // S^K_A S^Q_B P_A
        mac<false, false>(sq_p, SQB, Sm::LD, PA, Sm::LV, m0, n0, ns, D); // S^Q_B P_A
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const size_t g = oV + (size_t)(m0 + i) * DV + n0 + j * ns;
                const float tA = c.A.T[g], tB = c.B.T[g], qA = c.A.MQP[g], qB = c.B.MQP[g];
                const float pA = c.A.P[g], pB = c.B.P[g];
                c.out.T[g] = f3 * tA + tB + f * t[i][j] + f2 * acc[i][j];
                c.out.MQP[g] = f2 * qA + qB + f * sq_p[i][j];
                c.out.P[g] = f * pA + pB;
            }
    });
    for (int e = threadIdx.x; e < D * D; e += kThreads) {
        const int r = e / D, x = e % D;
        const float sA = c.A.S[oD + e], sB = c.B.S[oD + e], qA = c.A.SQ[oD + e], qB = c.B.SQ[oD + e];
        const float kA = c.A.MKQ[oD + e], kB = c.B.MKQ[oD + e];
        c.out.S[oD + e] = f * sA + sB;
        c.out.SQ[oD + e] = f * qA + qB;
        c.out.MKQ[oD + e] = f2 * kA + kB + f * W[r * Sm::LD + x];
    }
    if (c.norm) {  // the unit column: m as P, h as T, mqm as M^QP
        for (int i = threadIdx.x; i < D; i += kThreads) {
            float skq = 0.f, mkm = 0.f, wmm = 0.f, sqm = 0.f;
            for (int l = 0; l < D; ++l) {
                skq = fmaf(SKA[i * Sm::LD + l], mqmB[l], skq);
                mkm = fmaf(MKQB[i * Sm::LD + l], mA[l], mkm);
                wmm = fmaf(W[i * Sm::LD + l], mA[l], wmm);
                sqm = fmaf(SQB[i * Sm::LD + l], mA[l], sqm);
            }
            const float hA = c.A.h[od + i], hB = c.B.h[od + i], mAi = mA[i], mB = c.B.m[od + i];
            const float qA = c.A.mqm[od + i], qB = mqmB[i];
            c.out.h[od + i] = f3 * hA + hB + f * (skq + mkm) + f2 * wmm;
            c.out.m[od + i] = f * mAi + mB;
            c.out.mqm[od + i] = f2 * qA + qB + f * sqm;
        }
    }
}

// d = 128: the four d x d operands of the kernel above (128 x 132 floats each) do not fit
// one CTA's shared memory beside P_A and M^QP_B, so the concatenation runs in two phases
// that each stage only what is overwritten while it is read (out may alias A or B).
// Phase 1 forms P, T, M^QP (and m, h, mqm) with S^Q_B P_A staged, using
// S^K_A (S^Q_B P_A) for the W P_A term and S^K_A (S^Q_B m_A) for W m_A; the d x d operands
// stay in global memory, which phase 1 does not write.  Phase 2 stages S^K_A and S^Q_B
// and writes S, S^Q and M^KQ, forming W tile by tile.
template <int DV>
struct WideSmem {
    static constexpr int D = 128, LD = D + 4, LV = DV + 4;
    static constexpr int PA = 0, MQPB = PA + D * LV, SQP = MQPB + D * LV, VEC = SQP + D * LV, P1 = VEC + 3 * D;
    static constexpr int SKA = 0, SQB = SKA + D * LD, P2 = SQB + D * LD;
    static constexpr int TOTAL = P1 > P2 ? P1 : P2;
};

template <int DV>
__global__ void __launch_bounds__(kThreads) combine3_wide_kernel(Comb3 c) {
    using Sm = WideSmem<DV>;
    constexpr int D = Sm::D;
    extern __shared__ __align__(16) float sm[];
    const int i0 = blockIdx.x;
    const float f = c.decay_pow ? c.decay_pow[i0] : 1.f, f2 = f * f, f3 = f2 * f;
    const size_t oD = (size_t)i0 * D * D, oV = (size_t)i0 * D * DV, od = (size_t)i0 * D;
    const float *SKA_g = c.A.S + oD, *SQB_g = c.B.SQ + oD, *MKQB_g = c.B.MKQ + oD;
    // ---- phase 1: P, T, M^QP and the unit column
    float *PA = sm + Sm::PA, *MQPB = sm + Sm::MQPB, *SQP = sm + Sm::SQP;
    float *mA = sm + Sm::VEC, *mqmB = mA + D, *sqm = mqmB + D;
    for (int e = threadIdx.x; e < D * DV; e += kThreads) {
        const int o = (e / DV) * Sm::LV + e % DV;
        PA[o] = c.A.P[oV + e];
        MQPB[o] = c.B.MQP[oV + e];
    }
    if (c.norm)
        for (int e = threadIdx.x; e < D; e += kThreads) {
            mA[e] = c.A.m[od + e];
            mqmB[e] = c.B.mqm[od + e];
        }
    __syncthreads();
    // S^Q_B P_A and S^Q_B m_A
    tiles<false, D, DV>([&](float (&acc)[4][4], int m0, int n0, int ns) {
        mac<false, false>(acc, SQB_g, D, PA, Sm::LV, m0, n0, ns, D);
        each(acc, m0, n0, ns, [&](int i, int j, float x) { SQP[i * Sm::LV + j] = x; });
    });
    if (c.norm)
        for (int i = threadIdx.x; i < D; i += kThreads) {
            float acc = 0.f;
            for (int l = 0; l < D; ++l) acc = fmaf(SQB_g[(size_t)i * D + l], mA[l], acc);
            sqm[i] = acc;
        }
    __syncthreads();
    tiles<false, D, DV>([&](float (&acc)[4][4], int m0, int n0, int ns) {
        float t[4][4] = {};
        mac<false, false>(t, SKA_g, D, MQPB, Sm::LV, m0, n0, ns, D);  // S^K_A M^QP_B
        mac<false, false>(t, MKQB_g, D, PA, Sm::LV, m0, n0, ns, D);   // + M^KQ_B P_A
        mac<false, false>(acc, SKA_g, D, SQP, Sm::LV, m0, n0, ns, D); // S^K_A S^Q_B P_A
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int r = m0 + i, col = n0 + j * ns;
                const size_t g = oV + (size_t)r * DV + col;
                const float tA = c.A.T[g], tB = c.B.T[g], qA = c.A.MQP[g], qB = MQPB[r * Sm::LV + col];
                const float pA = PA[r * Sm::LV + col], pB = c.B.P[g];
                c.out.T[g] = f3 * tA + tB + f * t[i][j] + f2 * acc[i][j];
                c.out.MQP[g] = f2 * qA + qB + f * SQP[r * Sm::LV + col];
                c.out.P[g] = f * pA + pB;
            }
    });
    if (c.norm) {
        for (int i = threadIdx.x; i < D; i += kThreads) {
            float skq = 0.f, mkm = 0.f, wmm = 0.f;
            for (int l = 0; l < D; ++l) {
                skq = fmaf(SKA_g[(size_t)i * D + l], mqmB[l], skq);
                mkm = fmaf(MKQB_g[(size_t)i * D + l], mA[l], mkm);
                wmm = fmaf(SKA_g[(size_t)i * D + l], sqm[l], wmm);
            }
            const float hA = c.A.h[od + i], hB = c.B.h[od + i], mAi = mA[i], mB = c.B.m[od + i];
            const float qA = c.A.mqm[od + i], qB = mqmB[i];
            c.out.h[od + i] = f3 * hA + hB + f * (skq + mkm) + f2 * wmm;
            c.out.m[od + i] = f * mAi + mB;
            c.out.mqm[od + i] = f2 * qA + qB + f * sqm[i];
        }
    }
    __syncthreads();  // every read of phase 1 is done before phase 2 writes S, S^Q, M^KQ
    // ---- phase 2: S, S^Q, M^KQ
    float *SKA = sm + Sm::SKA, *SQB = sm + Sm::SQB;
    for (int e = threadIdx.x; e < D * D; e += kThreads) {
        const int o = (e / D) * Sm::LD + e % D;
        SKA[o] = SKA_g[e];
        SQB[o] = SQB_g[e];
    }
    __syncthreads();
    tiles<false, D, D>([&](float (&acc)[4][4], int m0, int n0, int ns) {
        mac<false, false>(acc, SKA, Sm::LD, SQB, Sm::LD, m0, n0, ns, D);  // W = S^K_A S^Q_B
        each(acc, m0, n0, ns, [&](int i, int j, float x) {
            const size_t g = oD + (size_t)i * D + j;
            const float kA = c.A.MKQ[g], kB = c.B.MKQ[g], qA = c.A.SQ[g], qB = SQB[i * Sm::LD + j];
            c.out.S[g] = f * SKA[i * Sm::LD + j] + c.B.S[g];
            c.out.SQ[g] = f * qA + qB;
            c.out.MKQ[g] = f2 * kA + kB + f * x;
        });
    });
}

template <int DV>
cudaError_t combine_wide_t(const Comb3 &c, cudaStream_t st) {
    constexpr size_t bytes = WideSmem<DV>::TOTAL * sizeof(float);
    static_assert(bytes <= 227 * 1024, "shared memory");
    cudaError_t e = smem_attr(combine3_wide_kernel<DV>, bytes);
    if (e != cudaSuccess) return e;
    combine3_wide_kernel<DV><<<c.count, kThreads, bytes, st>>>(c);
    return cudaGetLastError();
}

template <int D, int DV>
cudaError_t combine_t(const Comb3 &c, cudaStream_t st) {
    constexpr size_t bytes = CombSmem<D, DV>::TOTAL * sizeof(float);
    cudaError_t e = smem_attr(combine3_kernel<D, DV>, bytes);
    if (e != cudaSuccess) return e;
    combine3_kernel<D, DV><<<c.count, kThreads, bytes, st>>>(c);
    return cudaGetLastError();
}

template <template <int, int> class Fn, typename Arg>
cudaError_t by_width(int d, int dv, const Arg &a, cudaStream_t st) {
    auto dvs = [&](auto dd) -> cudaError_t {
        constexpr int DD = decltype(dd)::value;
        switch (dv) {
            case 16: return Fn<DD, 16>::run(a, st);
            case 32: return Fn<DD, 32>::run(a, st);
            case 64: return Fn<DD, 64>::run(a, st);
        }
        return cudaErrorInvalidValue;
    };
    switch (d) {
        case 16: return dvs(std::integral_constant<int, 16>{});
        case 32: return dvs(std::integral_constant<int, 32>{});
        case 64: return dvs(std::integral_constant<int, 64>{});
    }
    return cudaErrorInvalidValue;
}
template <int D, int DV>
struct MapsFn {
    static cudaError_t run(const Fwd3Args &a, cudaStream_t st) { return maps_t<D, DV>(a, st); }
};
template <int D, int DV>
struct CombFn {
    static cudaError_t run(const Comb3 &c, cudaStream_t st) { return combine_t<D, DV>(c, st); }
};
}  // namespace
}  // namespace fwd3

cudaError_t fwd3_maps_launch(const Fwd3Args &a, cudaStream_t st) {
    if (a.d == 128) {
        if (a.dv == 16) return fwd3::maps_t<128, 16>(a, st);
        if (a.dv == 32) return fwd3::maps_t<128, 32>(a, st);
        return cudaErrorInvalidValue;
    }
    return fwd3::by_width<fwd3::MapsFn>(a.d, a.dv, a, st);
}

cudaError_t state3_combine_launch(int count, int d, int dv, bool norm, const hla_state3 &A, const hla_state3 &B,
                                  const hla_state3 &out, const float *decay_pow, cudaStream_t st) {
    if (count == 0) return cudaSuccess;
    fwd3::Comb3 c{count, d, dv, norm, A, B, out, decay_pow};
    if (d == 128) {
        switch (dv) {
            case 16: return fwd3::combine_wide_t<16>(c, st);
            case 32: return fwd3::combine_wide_t<32>(c, st);
            case 64: return fwd3::combine_wide_t<64>(c, st);
            case 128: return fwd3::combine_wide_t<128>(c, st);
        }
        return cudaErrorInvalidValue;
    }
    if (dv == 128) {  // the concatenation at dv = 128 (the forward reaches it through value halves)
        switch (d) {
            case 16: return fwd3::combine_t<16, 128>(c, st);
            case 32: return fwd3::combine_t<32, 128>(c, st);
            case 64: return fwd3::combine_t<64, 128>(c, st);
        }
        return cudaErrorInvalidValue;
    }
    return fwd3::by_width<fwd3::CombFn>(d, dv, c, st);
}

}  // namespace hla
