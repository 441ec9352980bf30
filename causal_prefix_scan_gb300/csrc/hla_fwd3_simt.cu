// hla_fwd3_simt.cu -- shape checks, workspace size and dispatch of the third-order
// forward kernels in hla_fwd3_simt.cuh (instantiated per element type and chunk length
// in hla_fwd3_<type>_c<chunk>.cu), and the third-order decode step.
//
// Decode step ("Higher-order Linear Attention", gist.science summary, section 3: the
// online update of the third-order state), state (S^K, P, T) per pair, decay g per
// token (1 without decay):
//   S^K_t = g S^K + k k^T,  P_t = g P + k v^T,  u = S^K_t q,  w = P_t^T q,
//   T_t = g^3 T + u w^T,  o = T_t^T q = g^3 T^T q + (u.q) w.
// Ratio-normalised: the unit-value column of the state, the key mass m_t = g m + k and
// h_t = g^3 h + u (m_t.q), gives den = h_t.q, and o = T_t^T q / (den + eps).
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
    __shared__ float red[kThreads / 32], red2[kThreads / 32];
    const int tid = threadIdx.x;
    const size_t u = blockIdx.x;
    const float g = a.gamma ? a.gamma[u % a.H] : 1.f, g3 = g * g * g;
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
            s.x = fmaf(g, s.x, kr * ks[c0]); s.y = fmaf(g, s.y, kr * ks[c0 + 1]);
            s.z = fmaf(g, s.z, kr * ks[c0 + 2]); s.w = fmaf(g, s.w, kr * ks[c0 + 3]);
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
            x.x = fmaf(g, x.x, kr * vs[c0]); x.y = fmaf(g, x.y, kr * vs[c0 + 1]);
            x.z = fmaf(g, x.z, kr * vs[c0 + 2]); x.w = fmaf(g, x.w, kr * vs[c0 + 3]);
            P[e] = x;
            wp.x += qr * x.x; wp.y += qr * x.y; wp.z += qr * x.z; wp.w += qr * x.w;
        }
    }
    colsum(wp, wsum);  // also orders the writes of us[] before their reads
    // ---- the unit-value column (ratio normalisation): m_t = g m + k, w1 = m_t.q,
    // y1 = h.q, h_t = g^3 h + u w1
    float w1 = 0.f, y1 = 0.f;
    if (a.m) {
        float pm = 0.f, ph = 0.f, hi = 0.f;
        if (tid < D) {
            const float mi = fmaf(g, a.m[u * D + tid], ks[tid]);
            a.m[u * D + tid] = mi;
            hi = a.h[u * D + tid];
            pm = mi * qs[tid];
            ph = hi * qs[tid];
        }
        pm = group_sum<32>(pm);
        ph = group_sum<32>(ph);
        if ((tid & 31) == 0) { red[tid >> 5] = pm; red2[tid >> 5] = ph; }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < kThreads / 32; ++i) { w1 += red[i]; y1 += red2[i]; }
        if (tid < D) a.h[u * D + tid] = fmaf(g3, hi, us[tid] * w1);
        __syncthreads();  // red is reused below
    }
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
            x.x = fmaf(g3, x.x, ur * w.x); x.y = fmaf(g3, x.y, ur * w.y);
            x.z = fmaf(g3, x.z, ur * w.z); x.w = fmaf(g3, x.w, ur * w.w);
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
    const float inv = a.m ? 1.f / (fmaf(g3, y1, uq * w1) + a.eps) : 1.f;
    T *o = static_cast<T *>(a.o) + u * DV;
    for (int j = tid; j < DV; j += kThreads) {
        const float *w = reinterpret_cast<const float *>(&wsum[j >> 2]);
        const float *y = reinterpret_cast<const float *>(&ysum[j >> 2]);
        st_t(o, j, fmaf(g3, y[j & 3], uq * w[j & 3]) * inv);
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
    const bool shape = (ok(p.d) && ok(p.dv) && ok(p.chunk)) || (p.d == 128 && p.chunk == 16 && (p.dv == 16 || p.dv == 32));
    return shape && p.H % hkv == 0 && (p.flags & ~(unsigned)(HLA_DECAY | HLA_NORMALIZE)) == 0;
}

namespace fwd3 {
namespace {
size_t pass_workspace(const hla_params &p, int dv) {
    const size_t nch = ((size_t)p.n + p.chunk - 1) / p.chunk;
    const Ws3 w{p.d, dv};
    return (size_t)p.B * p.H * nch * (w.loc_floats() + w.st_floats()) * sizeof(float);
}
size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
constexpr int kUnit = 16;  // width of the unit-value tile of the denominator pass

// Workspace of the ratio-normalised forward: the passes' scratch (shared: the passes
// run one after the other), the unit-value tile E and the denominator output (element
// type of the inputs, [rows][16], a one in column 0 of E), and the denominator pass's
// states (P and T of width 16 before and after, S after).
struct NormWs {
    size_t pass, e, den, pin, tin, pout, tout, sscr, mqpin, mqpout, sqs, mkqs, total;
};
NormWs norm_ws(const hla_params &p) {
    NormWs w;
    const size_t rows = (size_t)p.B * p.H * p.n, units = (size_t)p.B * p.H, esz = p.in_dtype == HLA_F32 ? 4 : 2;
    const size_t a = pass_workspace(p, p.dv), b = pass_workspace(p, kUnit);
    size_t o = 0;
    auto take = [&](size_t bytes) { const size_t at = o; o = align256(o + bytes); return at; };
    w.pass = take(a > b ? a : b);
    w.e = take(rows * kUnit * esz);
    w.den = take(rows * kUnit * esz);
    w.pin = take(units * p.d * kUnit * 4);
    w.tin = take(units * p.d * kUnit * 4);
    w.pout = take(units * p.d * kUnit * 4);
    w.tout = take(units * p.d * kUnit * 4);
    w.sscr = take(units * (size_t)p.d * p.d * 4);
    // the unit values' segment maps: M^QP with mqm in column 0, before and after; S^Q and
    // M^KQ of that pass (equal to the values' ones) land in scratch
    w.mqpin = take(units * p.d * kUnit * 4);
    w.mqpout = take(units * p.d * kUnit * 4);
    w.sqs = take(units * (size_t)p.d * p.d * 4);
    w.mkqs = take(units * (size_t)p.d * p.d * 4);
    w.total = o;
    return w;
}

template <typename T>
__global__ void __launch_bounds__(kThreads) unit_tile_kernel(T *e, size_t rows) {
    for (size_t i = (size_t)blockIdx.x * kThreads + threadIdx.x; i < rows * kUnit; i += (size_t)gridDim.x * kThreads)
        st_t(e, i, (i % kUnit) == 0 ? 1.f : 0.f);
}
// d-vectors per pair <-> column 0 of [d][16] tiles (the other columns zero)
__global__ void __launch_bounds__(kThreads) to_column_kernel(float *dst, const float *src, size_t count) {
    for (size_t i = (size_t)blockIdx.x * kThreads + threadIdx.x; i < count * kUnit; i += (size_t)gridDim.x * kThreads)
        dst[i] = (i % kUnit) == 0 ? src[i / kUnit] : 0.f;
}
__global__ void __launch_bounds__(kThreads) from_column_kernel(float *dst, const float *src, size_t count) {
    for (size_t i = (size_t)blockIdx.x * kThreads + threadIdx.x; i < count; i += (size_t)gridDim.x * kThreads)
        dst[i] = src[i * kUnit];
}
// o = num / (den + eps), row by row (num is o itself)
template <typename T>
__global__ void __launch_bounds__(kThreads) ratio_kernel(T *o, const T *den, size_t rows, int dv, float eps) {
    for (size_t i = (size_t)blockIdx.x * kThreads + threadIdx.x; i < rows * dv; i += (size_t)gridDim.x * kThreads) {
        const size_t r = i / dv;
        st_t(o, i, ld_t(o, i) / (ld_t(den, r * kUnit) + eps));
    }
}
int grid_for(size_t work) {
    const size_t b = (work + kThreads - 1) / kThreads;
    return (int)(b < 4096 ? (b > 0 ? b : 1) : 4096);
}

template <typename T>
cudaError_t norm_t(const Fwd3Args &a0, const Norm3 &nm, cudaStream_t st) {
    hla_params p{};
    p.B = a0.B; p.H = a0.H; p.n = a0.n; p.d = a0.d; p.dv = a0.dv; p.chunk = a0.chunk; p.in_dtype = a0.in_dtype;
    const NormWs w = norm_ws(p);
    uint8_t *base = reinterpret_cast<uint8_t *>(a0.workspace);
    auto f = [&](size_t off) { return reinterpret_cast<float *>(base + off); };
    const size_t rows = (size_t)a0.B * a0.H * a0.n, pd = (size_t)a0.B * a0.H * a0.d;
    T *E = reinterpret_cast<T *>(base + w.e), *den = reinterpret_cast<T *>(base + w.den);
    cudaError_t e;
    auto mark = [&](int i) { return a0.events ? cudaEventRecord(a0.events[i], st) : cudaSuccess; };
    if ((e = mark(0)) != cudaSuccess) return e;
    unit_tile_kernel<T><<<grid_for(rows * kUnit), kThreads, 0, st>>>(E, rows);
    if (nm.m_in) {
        to_column_kernel<<<grid_for(pd * kUnit), kThreads, 0, st>>>(f(w.pin), nm.m_in, pd);
        to_column_kernel<<<grid_for(pd * kUnit), kThreads, 0, st>>>(f(w.tin), nm.h_in, pd);
    }
    if (nm.mqm_in) to_column_kernel<<<grid_for(pd * kUnit), kThreads, 0, st>>>(f(w.mqpin), nm.mqm_in, pd);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // numerator: the forward of the values, into o
    Fwd3Args a = a0;
    a.events = nullptr;
    a.workspace = f(w.pass);
    if ((e = launch_c<T>(a, st)) != cudaSuccess) return e;
    if ((e = mark(1)) != cudaSuccess) return e;
    // denominator: the forward of the unit values, same S
    Fwd3Args b = a;
    b.dv = kUnit;
    b.v = E;
    b.o = den;
    b.sin_P = nm.m_in ? f(w.pin) : nullptr;
    b.sin_T = nm.m_in ? f(w.tin) : nullptr;
    if (!a0.sin_S) b.sin_P = b.sin_T = nullptr;
    b.sout_S = nm.m_out ? f(w.sscr) : nullptr;
    b.sout_P = nm.m_out ? f(w.pout) : nullptr;
    b.sout_T = nm.m_out ? f(w.tout) : nullptr;
    b.sin_MQP = nm.mqm_in ? f(w.mqpin) : nullptr;  // S^Q, M^KQ of state_in: those of the values
    b.sout_SQ = a0.sout_SQ ? f(w.sqs) : nullptr;
    b.sout_MQP = a0.sout_SQ ? f(w.mqpout) : nullptr;
    b.sout_MKQ = a0.sout_SQ ? f(w.mkqs) : nullptr;
    if ((e = launch_c<T>(b, st)) != cudaSuccess) return e;
    if ((e = mark(2)) != cudaSuccess) return e;
    ratio_kernel<T><<<grid_for(rows * a0.dv), kThreads, 0, st>>>(static_cast<T *>(a0.o), den, rows, a0.dv, nm.eps);
    if (nm.m_out) {
        from_column_kernel<<<grid_for(pd), kThreads, 0, st>>>(nm.m_out, f(w.pout), pd);
        from_column_kernel<<<grid_for(pd), kThreads, 0, st>>>(nm.h_out, f(w.tout), pd);
    }
    if (nm.mqm_out) from_column_kernel<<<grid_for(pd), kThreads, 0, st>>>(nm.mqm_out, f(w.mqpout), pd);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    return mark(3);
}
}  // namespace
}  // namespace fwd3

size_t fwd3_workspace(const hla_params &p) {
    if (p.flags & HLA_NORMALIZE) return fwd3::norm_ws(p).total;
    return fwd3::pass_workspace(p, p.dv);
}

cudaError_t fwd3_launch(const Fwd3Args &a, cudaStream_t st) {
    return a.in_dtype == HLA_F32 ? fwd3::launch_c<float>(a, st) : fwd3::launch_c<__nv_bfloat16>(a, st);
}

cudaError_t fwd3_norm_launch(const Fwd3Args &a, const Norm3 &nm, cudaStream_t st) {
    return a.in_dtype == HLA_F32 ? fwd3::norm_t<float>(a, nm, st) : fwd3::norm_t<__nv_bfloat16>(a, nm, st);
}

cudaError_t decode3_launch(const Decode3Args &a, cudaStream_t st) {
    if (a.N == 0) return cudaSuccess;
    return a.dtype == HLA_F32 ? fwd3::decode3_d<float>(a, st) : fwd3::decode3_d<__nv_bfloat16>(a, st);
}

}  // namespace hla
