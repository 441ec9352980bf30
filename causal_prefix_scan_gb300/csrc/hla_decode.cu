// hla_decode.cu -- one decode step of masked second-order HLA for N independent
// (sequence, head) pairs, state updated in place.
//
// Recurrence (gist.science summary, section 1; decay factor g per head):
//   G_t = g^2 G_{t-1} + g k (k^T C_{t-1}),   h_t = g^2 h_{t-1} + g k (k^T m_{t-1})
//   S_t = g S_{t-1} + k k^T,  C_t = g C_{t-1} + q v^T,  m_t = g m_{t-1} + q
//   o   = q^T (S_t C_t - G_t)      [/ (q^T (S_t m_t - h_t) + eps)]
// The output is assembled without forming S_t C_t: with w = S_t q (S symmetric),
// r = C_{t-1}^T k, z = C_{t-1}^T w and y = G_{t-1}^T q,
//   o = g z + (w.q) v - g^2 y - g (q.k) r,
//   den = g (w.m_{t-1}) + w.q - g^2 (q.h_{t-1}) - g (q.k)(k.m_{t-1}).
// So each of S, C, G is streamed once from HBM and written once: the kernel is
// bound by HBM bandwidth (2 x 4 (d^2 + 2 d dv + 2 d) bytes per pair and step).
// Unmasked variant (o = q^T S_t C_t, skill card "Higher-order linear attention",
// bullet "Streaming Computation"): o = g z + (w.q) v, den = g (w.m_{t-1}) + w.q;
// G and h are neither read nor written.  Shared key/value heads: pair u = s*H + h
// reads key/value row s*Hkv + h/(H/Hkv).
#include "hla_internal.h"

namespace hla {
namespace {

constexpr int kThreads = 256;

template <typename T>
__device__ __forceinline__ float ldf(const T *p, size_t i);
template <>
__device__ __forceinline__ float ldf<float>(const float *p, size_t i) { return p[i]; }
template <>
__device__ __forceinline__ float ldf<__nv_bfloat16>(const __nv_bfloat16 *p, size_t i) {
    return __bfloat162float(p[i]);
}
template <typename T>
__device__ __forceinline__ void stf(T *p, size_t i, float x);
template <>
__device__ __forceinline__ void stf<float>(float *p, size_t i, float x) { p[i] = x; }
template <>
__device__ __forceinline__ void stf<__nv_bfloat16>(__nv_bfloat16 *p, size_t i, float x) {
    p[i] = __float2bfloat16_rn(x);
}

// Sum over the `width` consecutive lanes of an aligned lane group.
template <int width>
__device__ __forceinline__ float group_sum(float x) {
#pragma unroll
    for (int off = width / 2; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

__device__ __forceinline__ float block_sum(float x, float *red) {
    x = group_sum<32>(x);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) red[w] = x;
    __syncthreads();
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kThreads / 32; ++i) s += red[i];
    return s;
}

// Three CTAs per SM keep enough loads in flight; the register cap (85) is above what
// the bf16 and fp32 instantiations need.
template <typename T, int D, int DV, bool UNM>
__global__ void __launch_bounds__(kThreads, 3) decode_kernel(DecodeArgs a) {
    constexpr int CG = D / 4;           // float4 column groups of S
    constexpr int CGV = DV / 4;         // float4 column groups of C, G
    constexpr int NS = D * D / 4;       // float4 elements of S
    constexpr int NC = D * DV / 4;      // float4 elements of C or G
    constexpr int ITS = (NS + kThreads - 1) / kThreads;
    constexpr int ITC = (NC + kThreads - 1) / kThreads;

    __shared__ float qs[D], ks[D], ws[D], vs[DV];
    __shared__ float4 redv[kThreads];
    __shared__ float4 rsum[CGV], zsum[CGV], ysum[CGV];
    __shared__ float red[kThreads / 32];

    const int tid = threadIdx.x;
    const size_t u = blockIdx.x;
    const bool decay = (a.flags & HLA_DECAY) != 0;
    const bool norm = (a.flags & HLA_NORMALIZE) != 0;
    constexpr bool unm = UNM;
    const float g = decay ? a.gamma[u % a.H] : 1.f;
    const float g2 = g * g;
    const size_t kvu = (u / a.H) * a.Hkv + (u % a.H) / (a.H / a.Hkv);  // key/value row

    const T *q = static_cast<const T *>(a.q) + u * D;
    const T *k = static_cast<const T *>(a.k) + kvu * D;
    const T *v = static_cast<const T *>(a.v) + kvu * DV;
    for (int i = tid; i < D; i += kThreads) { qs[i] = ldf(q, i); ks[i] = ldf(k, i); }
    for (int j = tid; j < DV; j += kThreads) vs[j] = ldf(v, j);
    __syncthreads();

    float4 *S = reinterpret_cast<float4 *>(a.st.S + u * D * D);
    float4 *C = reinterpret_cast<float4 *>(a.st.C + u * D * DV);
    float4 *G = unm ? nullptr : reinterpret_cast<float4 *>(a.st.G + u * D * DV);
    float *m = a.st.m + u * D;
    float *h = unm ? nullptr : a.st.h + u * D;

    // ---- S: S_t = g S + k k^T, w = S_t q  (rows of one lane group share a row)
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
            s.x = g * s.x + kr * ks[c0 + 0];
            s.y = g * s.y + kr * ks[c0 + 1];
            s.z = g * s.z + kr * ks[c0 + 2];
            s.w = g * s.w + kr * ks[c0 + 3];
            S[e] = s;
            part = s.x * qs[c0] + s.y * qs[c0 + 1] + s.z * qs[c0 + 2] + s.w * qs[c0 + 3];
        }
        // lanes of one row form an aligned group of CG lanes (CG divides 32)
        if constexpr (CG <= 32 && (kThreads % CG) == 0) {
            if (NS >= kThreads || i * kThreads < NS) {
                part = group_sum<CG>(part);
                if (e < NS && (e % CG) == 0) ws[row] = part;
            }
        }
    }
    __syncthreads();

    // ---- C: r = C^T k, z = C^T w from C_{t-1}; C_t = g C + q v^T
    float4 cv[ITC];
#pragma unroll
    for (int i = 0; i < ITC; ++i) {
        const int e = tid + i * kThreads;
        if (e < NC) cv[i] = C[e];
    }
    float4 rp = make_float4(0, 0, 0, 0), zp = rp;
#pragma unroll
    for (int i = 0; i < ITC; ++i) {
        const int e = tid + i * kThreads;
        if (e < NC) {
            const int row = e / CGV, c0 = (e % CGV) * 4;
            const float kr = ks[row], wr = ws[row], qr = qs[row];
            float4 c = cv[i];
            rp.x += kr * c.x; rp.y += kr * c.y; rp.z += kr * c.z; rp.w += kr * c.w;
            zp.x += wr * c.x; zp.y += wr * c.y; zp.z += wr * c.z; zp.w += wr * c.w;
            c.x = g * c.x + qr * vs[c0 + 0];
            c.y = g * c.y + qr * vs[c0 + 1];
            c.z = g * c.z + qr * vs[c0 + 2];
            c.w = g * c.w + qr * vs[c0 + 3];
            C[e] = c;
        }
    }
    // column reduction over the threads sharing a column group (tid % CGV)
    redv[tid] = rp;
    __syncthreads();
    if (tid < CGV) {
        float4 s = make_float4(0, 0, 0, 0);
        for (int t = tid; t < kThreads; t += CGV) {
            const float4 x = redv[t];
            s.x += x.x; s.y += x.y; s.z += x.z; s.w += x.w;
        }
        rsum[tid] = s;
    }
    __syncthreads();
    redv[tid] = zp;
    __syncthreads();
    if (tid < CGV) {
        float4 s = make_float4(0, 0, 0, 0);
        for (int t = tid; t < kThreads; t += CGV) {
            const float4 x = redv[t];
            s.x += x.x; s.y += x.y; s.z += x.z; s.w += x.w;
        }
        zsum[tid] = s;
    }
    __syncthreads();

    // ---- G: y = G^T q from G_{t-1}; G_t = g^2 G + g k r^T  (masked variant only)
    float4 yp = make_float4(0, 0, 0, 0);
#pragma unroll
    for (int i = 0; i < ITC; ++i) {
        const int e = tid + i * kThreads;
        if constexpr (!UNM) {
            if (e < NC) cv[i] = G[e];
        }
    }
#pragma unroll
    for (int i = 0; i < ITC; ++i) {
        const int e = tid + i * kThreads;
        if (!UNM && e < NC) {
            const int row = e / CGV, cg = e % CGV;
            const float qr = qs[row], gk = g * ks[row];
            float4 x = cv[i];
            const float4 r = rsum[cg];
            yp.x += qr * x.x; yp.y += qr * x.y; yp.z += qr * x.z; yp.w += qr * x.w;
            x.x = g2 * x.x + gk * r.x;
            x.y = g2 * x.y + gk * r.y;
            x.z = g2 * x.z + gk * r.z;
            x.w = g2 * x.w + gk * r.w;
            G[e] = x;
        }
    }
    redv[tid] = yp;
    __syncthreads();
    if (tid < CGV) {
        float4 s = make_float4(0, 0, 0, 0);
        for (int t = tid; t < kThreads; t += CGV) {
            const float4 x = redv[t];
            s.x += x.x; s.y += x.y; s.z += x.z; s.w += x.w;
        }
        ysum[tid] = s;
    }

    // ---- scalars and the m, h vectors
    float pwq = 0.f, pqk = 0.f, pkm = 0.f, pwm = 0.f, pqh = 0.f;
    for (int i = tid; i < D; i += kThreads) {
        const float mo = m[i], ho = unm ? 0.f : h[i];
        pwq += ws[i] * qs[i];
        pqk += qs[i] * ks[i];
        pkm += ks[i] * mo;
        pwm += ws[i] * mo;
        pqh += qs[i] * ho;
    }
    const float wq = block_sum(pwq, red);
    const float qk = block_sum(pqk, red);
    const float km = block_sum(pkm, red);
    float den = 1.f;
    if (norm) {
        const float wm = block_sum(pwm, red);
        const float qh = block_sum(pqh, red);
        den = unm ? g * wm + wq + a.eps : g * wm + wq - g2 * qh - g * qk * km + a.eps;
    }
    __syncthreads();  // all reads of m, h done before they are overwritten
    for (int i = tid; i < D; i += kThreads) {
        const float mo = m[i];
        if (!unm) h[i] = g2 * h[i] + g * ks[i] * km;
        m[i] = g * mo + qs[i];
    }
    T *o = static_cast<T *>(a.o) + u * DV;
    for (int j = tid; j < DV; j += kThreads) {
        const int cg = j >> 2, c = j & 3;
        const float *r = reinterpret_cast<const float *>(&rsum[cg]);
        const float *z = reinterpret_cast<const float *>(&zsum[cg]);
        const float *y = reinterpret_cast<const float *>(&ysum[cg]);
        const float num = unm ? g * z[c] + wq * vs[j] : g * z[c] + wq * vs[j] - g2 * y[c] - g * qk * r[c];
        stf(o, j, norm ? num / den : num);
    }
}

// Asymmetric variant AHLA (gist.science summary, section 2), state (R, P, m^K,
// E, n) in the (S, C, m, G, h) arrays:
//   R += k q^T;  z = g P_{t-1}^T q + (q.k) v (= P_t^T q);  P = g P + k v^T;
//   zeta = g (q.m) + q.k (= q.m^K_t);  m^K = g m^K + k;
//   o = g E_{t-1}^T q + (q.k) z (= E_t^T q);  E = g E + k z^T;  n = g n + k zeta;
//   den = g (q.n_{t-1}) + (q.k) zeta.
// Each array is streamed once from HBM and written once.
template <typename T, int D, int DV>
__global__ void __launch_bounds__(kThreads, 3) decode_asym_kernel(DecodeArgs a) {
    constexpr int CG = D / 4, CGV = DV / 4;
    constexpr int NS = D * D / 4, NC = D * DV / 4;
    constexpr int ITS = (NS + kThreads - 1) / kThreads;
    constexpr int ITC = (NC + kThreads - 1) / kThreads;
    __shared__ float qs[D], ks[D], vs[DV], zs[DV];
    __shared__ float4 redv[kThreads];
    __shared__ float4 ysum[CGV];
    __shared__ float red[kThreads / 32];

    const int tid = threadIdx.x;
    const size_t u = blockIdx.x;
    const bool decay = (a.flags & HLA_DECAY) != 0;
    const bool norm = (a.flags & HLA_NORMALIZE) != 0;
    const float g = decay ? a.gamma[u % a.H] : 1.f;
    const size_t kvu = (u / a.H) * a.Hkv + (u % a.H) / (a.H / a.Hkv);
    const T *q = static_cast<const T *>(a.q) + u * D;
    const T *k = static_cast<const T *>(a.k) + kvu * D;
    const T *v = static_cast<const T *>(a.v) + kvu * DV;
    for (int i = tid; i < D; i += kThreads) { qs[i] = ldf(q, i); ks[i] = ldf(k, i); }
    for (int j = tid; j < DV; j += kThreads) vs[j] = ldf(v, j);
    __syncthreads();
    float4 *R = reinterpret_cast<float4 *>(a.st.S + u * D * D);
    float4 *P = reinterpret_cast<float4 *>(a.st.C + u * D * DV);
    float4 *E = reinterpret_cast<float4 *>(a.st.G + u * D * DV);
    float *m = a.st.m + u * D;
    float *n = a.st.h + u * D;

    // ---- R += k q^T
    float4 rv[ITS];
#pragma unroll
    for (int i = 0; i < ITS; ++i) {
        const int e = tid + i * kThreads;
        if (e < NS) rv[i] = R[e];
    }
#pragma unroll
    for (int i = 0; i < ITS; ++i) {
        const int e = tid + i * kThreads;
        if (e < NS) {
            const int row = e / CG, c0 = (e % CG) * 4;
            const float kr = ks[row];
            float4 x = rv[i];
            x.x += kr * qs[c0]; x.y += kr * qs[c0 + 1]; x.z += kr * qs[c0 + 2]; x.w += kr * qs[c0 + 3];
            R[e] = x;
        }
    }
    // column reduction of x over the threads sharing a column group -> dst
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
    // ---- P: y1 = P_{t-1}^T q; P = g P + k v^T
    float4 cv[ITC];
#pragma unroll
    for (int i = 0; i < ITC; ++i) {
        const int e = tid + i * kThreads;
        if (e < NC) cv[i] = P[e];
    }
    float4 yp = make_float4(0, 0, 0, 0);
#pragma unroll
    for (int i = 0; i < ITC; ++i) {
        const int e = tid + i * kThreads;
        if (e < NC) {
            const int row = e / CGV, c0 = (e % CGV) * 4;
            const float qr = qs[row], kr = ks[row];
            float4 x = cv[i];
            yp.x += qr * x.x; yp.y += qr * x.y; yp.z += qr * x.z; yp.w += qr * x.w;
            x.x = g * x.x + kr * vs[c0]; x.y = g * x.y + kr * vs[c0 + 1];
            x.z = g * x.z + kr * vs[c0 + 2]; x.w = g * x.w + kr * vs[c0 + 3];
            P[e] = x;
        }
    }
    colsum(yp, ysum);
    // scalars q.k, q.m_{t-1}, q.n_{t-1}
    float pqk = 0.f, pqm = 0.f, pqn = 0.f;
    for (int i = tid; i < D; i += kThreads) {
        pqk += qs[i] * ks[i];
        pqm += qs[i] * m[i];
        pqn += qs[i] * n[i];
    }
    const float qk = block_sum(pqk, red);
    const float qm = block_sum(pqm, red);
    const float qn = norm ? block_sum(pqn, red) : 0.f;
    const float zeta = g * qm + qk;
    for (int j = tid; j < DV; j += kThreads) {
        const float *y1 = reinterpret_cast<const float *>(&ysum[j >> 2]);
        zs[j] = g * y1[j & 3] + qk * vs[j];
    }
    __syncthreads();
    // ---- E: y2 = E_{t-1}^T q; E = g E + k z^T
#pragma unroll
    for (int i = 0; i < ITC; ++i) {
        const int e = tid + i * kThreads;
        if (e < NC) cv[i] = E[e];
    }
    yp = make_float4(0, 0, 0, 0);
#pragma unroll
    for (int i = 0; i < ITC; ++i) {
        const int e = tid + i * kThreads;
        if (e < NC) {
            const int row = e / CGV, c0 = (e % CGV) * 4;
            const float qr = qs[row], kr = ks[row];
            float4 x = cv[i];
            yp.x += qr * x.x; yp.y += qr * x.y; yp.z += qr * x.z; yp.w += qr * x.w;
            x.x = g * x.x + kr * zs[c0]; x.y = g * x.y + kr * zs[c0 + 1];
            x.z = g * x.z + kr * zs[c0 + 2]; x.w = g * x.w + kr * zs[c0 + 3];
            E[e] = x;
        }
    }
    colsum(yp, ysum);
    for (int i = tid; i < D; i += kThreads) {
        m[i] = g * m[i] + ks[i];
        n[i] = g * n[i] + ks[i] * zeta;
    }
    const float den = norm ? g * qn + qk * zeta + a.eps : 1.f;
    T *o = static_cast<T *>(a.o) + u * DV;
    for (int j = tid; j < DV; j += kThreads) {
        const float *y2 = reinterpret_cast<const float *>(&ysum[j >> 2]);
        const float num = g * y2[j & 3] + qk * zs[j];
        stf(o, j, norm ? num / den : num);
    }
}

template <typename T, int D, int DV>
cudaError_t launch_t(const DecodeArgs &a, cudaStream_t st) {
    if (a.flags & HLA_ASYMMETRIC) decode_asym_kernel<T, D, DV><<<a.N, kThreads, 0, st>>>(a);
    else if (a.flags & HLA_UNMASKED) decode_kernel<T, D, DV, true><<<a.N, kThreads, 0, st>>>(a);
    else decode_kernel<T, D, DV, false><<<a.N, kThreads, 0, st>>>(a);
    return cudaGetLastError();
}
template <typename T, int D>
cudaError_t launch_dv(const DecodeArgs &a, cudaStream_t st) {
    switch (a.dv) {
        case 16: return launch_t<T, D, 16>(a, st);
        case 32: return launch_t<T, D, 32>(a, st);
        case 64: return launch_t<T, D, 64>(a, st);
        case 128: return launch_t<T, D, 128>(a, st);
    }
    return cudaErrorInvalidValue;
}
template <typename T>
cudaError_t launch_d(const DecodeArgs &a, cudaStream_t st) {
    switch (a.d) {
        case 16: return launch_dv<T, 16>(a, st);
        case 32: return launch_dv<T, 32>(a, st);
        case 64: return launch_dv<T, 64>(a, st);
        case 128: return launch_dv<T, 128>(a, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t decode_launch(const DecodeArgs &a, cudaStream_t st) {
    if (a.N == 0) return cudaSuccess;
    return a.dtype == HLA_F32 ? launch_d<float>(a, st) : launch_d<__nv_bfloat16>(a, st);
}

}  // namespace hla
