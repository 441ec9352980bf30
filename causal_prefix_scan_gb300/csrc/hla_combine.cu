// hla_combine.cu -- segment concatenation of HLA states (gist.science summary,
// section 4, "Associatieve operatoren"): out = A (+) B, A before B in time,
// f = g^{len(B)}:
//   S = f S_A + S_B,  C = f C_A + C_B,  m = f m_A + m_B,
//   G = f^2 G_A + G_B + f S_B C_A,   h = f^2 h_A + h_B + f S_B m_A.
// The unmasked state (S, C, m) uses the linear terms and writes G, h as zeros.
// The asymmetric variant AHLA (R, P, m^K, E, n in the same arrays) combines by
//   S = S_A + S_B,  C = f C_A + C_B,  m = f m_A + m_B,
//   G = f G_A + G_B + f S_B C_A,   h = f h_A + h_B + f S_B m_A
// (the same cross product, E decays like P).
// Two launches on one stream: the cross terms (G, h), which read S_B, C_A and
// m_A, run first; the linear terms (S, C, m) second.  Each output element is
// read and written by one thread only, so out may be A or B.
#include "hla_internal.h"

namespace hla {
namespace {

constexpr int kRows = 16;     // rows of S_B C_A per CTA
constexpr int kThreads = 256; // 16 rows x 16 column lanes
constexpr int kKt = 32;       // contraction tile

template <int D, int DV>
__global__ void __launch_bounds__(kThreads) cross_kernel(CombineArgs a) {
    __shared__ float sb[kRows][D + 1];
    __shared__ float ca[kKt][DV];
    __shared__ float ma[D];
    const int item = blockIdx.x;
    const int r0 = blockIdx.y * kRows;
    const int tid = threadIdx.x;
    const int lr = tid / 16, lc = tid % 16;  // row in slab, column lane
    constexpr int NCOL = DV / 16 > 0 ? DV / 16 : 1;
    const float f = a.decay_pow ? a.decay_pow[item] : 1.f;
    const bool asym = (a.flags & HLA_ASYMMETRIC) != 0, unm = (a.flags & HLA_UNMASKED) != 0;
    const float f2 = asym ? f : f * f;  // decay of G (E for the asymmetric variant)
    const float fx = unm ? 0.f : 1.f;   // the unmasked state has no G, h
    const float *SB = a.B.S + (size_t)item * D * D;
    const float *CA = a.A.C + (size_t)item * D * DV;
    for (int e = tid; e < kRows * D; e += kThreads) {
        const int r = e / D, c = e % D;
        sb[r][c] = (r0 + r < D) ? SB[(size_t)(r0 + r) * D + c] : 0.f;
    }
    for (int i = tid; i < D; i += kThreads) ma[i] = a.A.m[(size_t)item * D + i];
    float acc[NCOL];
#pragma unroll
    for (int j = 0; j < NCOL; ++j) acc[j] = 0.f;
    for (int k0 = 0; k0 < D; k0 += kKt) {
        __syncthreads();
        for (int e = tid; e < kKt * DV; e += kThreads) {
            const int r = e / DV, c = e % DV;
            ca[r][c] = (k0 + r < D) ? CA[(size_t)(k0 + r) * DV + c] : 0.f;
        }
        __syncthreads();
        for (int kk = 0; kk < kKt && k0 + kk < D; ++kk) {
            const float s = sb[lr][k0 + kk];
#pragma unroll
            for (int j = 0; j < NCOL; ++j) {
                const int c = lc + 16 * j;
                if (c < DV) acc[j] += s * ca[kk][c];
            }
        }
    }
    const int row = r0 + lr;
    if (row < D) {
        const size_t gb = (size_t)item * D * DV + (size_t)row * DV;
#pragma unroll
        for (int j = 0; j < NCOL; ++j) {
            const int c = lc + 16 * j;
            if (c < DV) a.out.G[gb + c] = fx * (f2 * a.A.G[gb + c] + a.B.G[gb + c] + f * acc[j]);
        }
        if (lc == 0) {
            float s = 0.f;
            for (int l = 0; l < D; ++l) s += sb[lr][l] * ma[l];
            const size_t hb = (size_t)item * D + row;
            a.out.h[hb] = fx * (f2 * a.A.h[hb] + a.B.h[hb] + f * s);
        }
    }
}

__global__ void linear_kernel(CombineArgs a) {
    const size_t nS = (size_t)a.d * a.d, nC = (size_t)a.d * a.dv, nm = (size_t)a.d;
    const size_t per = nS + nC + nm;
    const size_t total = per * (size_t)a.count;
    for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < total; e += (size_t)gridDim.x * blockDim.x) {
        const size_t item = e / per, r = e % per;
        const float f = a.decay_pow ? a.decay_pow[item] : 1.f;
        if (r < nS) {  // S (R of the asymmetric variant, which does not decay)
            const size_t i = item * nS + r;
            a.out.S[i] = ((a.flags & HLA_ASYMMETRIC) ? 1.f : f) * a.A.S[i] + a.B.S[i];
        } else if (r < nS + nC) {
            const size_t i = item * nC + (r - nS);
            a.out.C[i] = f * a.A.C[i] + a.B.C[i];
        } else {
            const size_t i = item * nm + (r - nS - nC);
            a.out.m[i] = f * a.A.m[i] + a.B.m[i];
        }
    }
}

template <int D, int DV>
cudaError_t launch_t(const CombineArgs &a, cudaStream_t st) {
    dim3 grid(a.count, (D + kRows - 1) / kRows);
    cross_kernel<D, DV><<<grid, kThreads, 0, st>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const size_t total = ((size_t)a.d * a.d + (size_t)a.d * a.dv + a.d) * (size_t)a.count;
    const int blocks = (int)std::min<size_t>((total + 255) / 256, 152 * 16);
    linear_kernel<<<blocks, 256, 0, st>>>(a);
    return cudaGetLastError();
}
template <int D>
cudaError_t launch_dv(const CombineArgs &a, cudaStream_t st) {
    switch (a.dv) {
        case 16: return launch_t<D, 16>(a, st);
        case 32: return launch_t<D, 32>(a, st);
        case 64: return launch_t<D, 64>(a, st);
        case 128: return launch_t<D, 128>(a, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t combine_launch(const CombineArgs &a, cudaStream_t st) {
    if (a.count == 0) return cudaSuccess;
    switch (a.d) {
        case 16: return launch_dv<16>(a, st);
        case 32: return launch_dv<32>(a, st);
        case 64: return launch_dv<64>(a, st);
        case 128: return launch_dv<128>(a, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace hla
