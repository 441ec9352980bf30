// hla_fwd3_simt.cu -- shape checks, workspace size and dispatch of the third-order
// forward kernels in hla_fwd3_simt.cuh (instantiated per element type and chunk length
// in hla_fwd3_<type>_c<chunk>.cu), and the third-order decode step.
//
// Decode step ("Higher-order Linear Attention", gist.science summary, section 3: the
// online update of the third-order state), state (S^K, P, T) per pair:
//   S^K_t = S^K + k k^T,  P_t = P + k v^T,  u = S^K_t q,  w = P_t^T q,
//   T_t = T + u w^T,  o = T_t^T q = T^T q + (u.q) w.
// Each array is streamed once from HBM and written once.
#include "hla_fwd3_simt.cuh"

namespace hla {
namespace fwd3 {
#define HLA_FWD3_EXTERN(T, C) extern template cudaError_t launch_d<T, C>(const Fwd3Args &, cudaStream_t);
HLA_FWD3_EXTERN(float, 16)
HLA_FWD3_EXTERN(float, 32)
HLA_FWD3_EXTERN(float, 64)
HLA_FWD3_EXTERN(__nv_bfloat16, 16)
HLA_FWD3_EXTERN(__nv_bfloat16, 32)
HLA_FWD3_EXTERN(__nv_bfloat16, 64)
#undef HLA_FWD3_EXTERN

namespace {
template <typename T>
cudaError_t launch_c(const Fwd3Args &a, cudaStream_t st) {
    switch (a.chunk) {
        case 16: return launch_d<T, 16>(a, st);
        case 32: return launch_d<T, 32>(a, st);
        case 64: return launch_d<T, 64>(a, st);
    }
    return cudaErrorInvalidValue;
}

template <int width>
__device__ __forceinline__ float group_sum(float x) {
#pragma unroll
    for (int off = width / 2; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

template <typename T, int D, int DV>
__global__ void __launch_bounds__(kThreads, 3) decode3_kernel(Decode3Args a) {
    constexpr int CG = D / 4, CGV = DV / 4;
    constexpr int NS = D * D / 4, NC = D * DV / 4;
    constexpr int ITS = (NS + kThreads - 1) / kThreads;
    constexpr int ITC = (NC + kThreads - 1) / kThreads;
    static_assert(CG <= 32 && kThreads % CG == 0, "row groups must fit in a warp");
    __shared__ float qs[D], ks[D], us[D], vs[DV];
    __shared__ float4 redv[kThreads];
    __shared__ float4 wsum[CGV], ysum[CGV];
    __shared__ float red[kThreads / 32];
    const int tid = threadIdx.x;
    const size_t u = blockIdx.x;
    const T *q = static_cast<const T *>(a.q) + u * D;
    const T *k = static_cast<const T *>(a.k) + u * D;
    const T *v = static_cast<const T *>(a.v) + u * DV;
    for (int i = tid; i < D; i += kThreads) { qs[i] = ld_t(q, i); ks[i] = ld_t(k, i); }
    for (int j = tid; j < DV; j += kThreads) vs[j] = ld_t(v, j);
    __syncthreads();
    float4 *S = reinterpret_cast<float4 *>(a.S + u * D * D);
    float4 *P = reinterpret_cast<float4 *>(a.P + u * D * DV);
    float4 *Tm = reinterpret_cast<float4 *>(a.T + u * D * DV);
    auto colsum = [&](float4 x, float4 *dst) {
        redv[tid] = x;
        __syncthreads();
        if (tid < CGV) {
            float4 s = make_float4(0, 0, 0, 0);
            for (int t = tid; t < kThreads; t += CGV) {
                const float4 y = redv[t];
                s.x += y.x; s.y += y.y; s.z += y.z; s.w += y.w;
            }
            dst[tid] = s;
        }
        __syncthreads();
    };
    // ---- S^K_t = S^K + k k^T;  u = S^K_t q (the lanes of one row form an aligned group)
    float4 sv[ITS];
#pragma unroll
    for (int i = 0; i < ITS; ++i) {
        const int e = tid + i * kThreads;
        if (e < NS) sv[i] = S[e];
    }
#pragma unroll
    for (int i = 0; i < ITS; ++i) {
        const int e = tid + i * kThreads;
        float part = 0.f;
        int row = 0;
        if (e < NS) {
            row = e / CG;
            const int c0 = (e % CG) * 4;
            const float kr = ks[row];
            float4 s = sv[i];
            s.x += kr * ks[c0]; s.y += kr * ks[c0 + 1]; s.z += kr * ks[c0 + 2]; s.w += kr * ks[c0 + 3];
            S[e] = s;
            part = s.x * qs[c0] + s.y * qs[c0 + 1] + s.z * qs[c0 + 2] + s.w * qs[c0 + 3];
        }
        if (NS >= kThreads || i * kThreads < NS) {
            part = group_sum<CG>(part);
            if (e < NS && (e % CG) == 0) us[row] = part;
        }
    }
    // ---- P_t = P + k v^T;  w = P_t^T q
    float4 cv[ITC];
#pragma unroll
    for (int i = 0; i < ITC; ++i) {
        const int e = tid + i * kThreads;
        if (e < NC) cv[i] = P[e];
    }
    float4 wp = make_float4(0, 0, 0, 0);
#pragma unroll
    for (int i = 0; i < ITC; ++i) {
        const int e = tid + i * kThreads;
        if (e < NC) {
            const int row = e / CGV, c0 = (e % CGV) * 4;
            const float kr = ks[row], qr = qs[row];
            float4 x = cv[i];
            x.x += kr * vs[c0]; x.y += kr * vs[c0 + 1]; x.z += kr * vs[c0 + 2]; x.w += kr * vs[c0 + 3];
            P[e] = x;
            wp.x += qr * x.x; wp.y += qr * x.y; wp.z += qr * x.z; wp.w += qr * x.w;
        }
    }
    colsum(wp, wsum);  // also orders the writes of us[] before their reads
    // ---- y = T^T q from T_{t-1};  T_t = T + u w^T
#pragma unroll
    for (int i = 0; i < ITC; ++i) {
        const int e = tid + i * kThreads;
        if (e < NC) cv[i] = Tm[e];
    }
    float4 yp = make_float4(0, 0, 0, 0);
#pragma unroll
    for (int i = 0; i < ITC; ++i) {
        const int e = tid + i * kThreads;
        if (e < NC) {
            const int row = e / CGV, cg = e % CGV;
            const float qr = qs[row], ur = us[row];
            const float4 w = wsum[cg];
            float4 x = cv[i];
            yp.x += qr * x.x; yp.y += qr * x.y; yp.z += qr * x.z; yp.w += qr * x.w;
            x.x += ur * w.x; x.y += ur * w.y; x.z += ur * w.z; x.w += ur * w.w;
            Tm[e] = x;
        }
    }
    colsum(yp, ysum);
    // u.q
    float p = 0.f;
    for (int i = tid; i < D; i += kThreads) p += us[i] * qs[i];
    p = group_sum<32>(p);
    if ((tid & 31) == 0) red[tid >> 5] = p;
    __syncthreads();
    float uq = 0.f;
#pragma unroll
    for (int i = 0; i < kThreads / 32; ++i) uq += red[i];
    T *o = static_cast<T *>(a.o) + u * DV;
    for (int j = tid; j < DV; j += kThreads) {
        const float *w = reinterpret_cast<const float *>(&wsum[j >> 2]);
        const float *y = reinterpret_cast<const float *>(&ysum[j >> 2]);
        st_t(o, j, y[j & 3] + uq * w[j & 3]);
    }
}

template <typename T, int D, int DV>
cudaError_t decode3_t(const Decode3Args &a, cudaStream_t st) {
    decode3_kernel<T, D, DV><<<a.N, kThreads, 0, st>>>(a);
    return cudaGetLastError();
}
template <typename T, int D>
cudaError_t decode3_dv(const Decode3Args &a, cudaStream_t st) {
    switch (a.dv) {
        case 16: return decode3_t<T, D, 16>(a, st);
        case 32: return decode3_t<T, D, 32>(a, st);
        case 64: return decode3_t<T, D, 64>(a, st);
        case 128: return decode3_t<T, D, 128>(a, st);
    }
    return cudaErrorInvalidValue;
}
template <typename T>
cudaError_t decode3_d(const Decode3Args &a, cudaStream_t st) {
    switch (a.d) {
        case 16: return decode3_dv<T, 16>(a, st);
        case 32: return decode3_dv<T, 32>(a, st);
        case 64: return decode3_dv<T, 64>(a, st);
        case 128: return decode3_dv<T, 128>(a, st);
    }
    return cudaErrorInvalidValue;
}
}  // namespace
}  // namespace fwd3

bool fwd3_supported(const hla_params &p) {
    auto ok = [](int x) { return x == 16 || x == 32 || x == 64; };
    const int hkv = p.Hkv > 0 ? p.Hkv : p.H;
    return ok(p.d) && ok(p.dv) && ok(p.chunk) && hkv == p.H && p.flags == 0;
}

size_t fwd3_workspace(const hla_params &p) {
    const size_t nch = ((size_t)p.n + p.chunk - 1) / p.chunk;
    const fwd3::Ws3 w{p.d, p.dv};
    return (size_t)p.B * p.H * nch * (w.loc_floats() + w.st_floats()) * sizeof(float);
}

cudaError_t fwd3_launch(const Fwd3Args &a, cudaStream_t st) {
    return a.in_dtype == HLA_F32 ? fwd3::launch_c<float>(a, st) : fwd3::launch_c<__nv_bfloat16>(a, st);
}

cudaError_t decode3_launch(const Decode3Args &a, cudaStream_t st) {
    if (a.N == 0) return cudaSuccess;
    return a.dtype == HLA_F32 ? fwd3::decode3_d<float>(a, st) : fwd3::decode3_d<__nv_bfloat16>(a, st);
}

}  // namespace hla
