// hla_bwd_norm.cu -- backward pass through the ratio normalisation
// o_t = n_t / (den_t + eps) ("Higher-order Linear Attention", gist.science summary,
// section 1, bullet "Normalisatie"), composed from the unnormalised kernels.
//
// The denominator den_t = q_t^T (S_t m_t - h_t) is the masked output with every value
// equal to one, so the normalised output is the unnormalised one of the augmented values
// [V | 1] followed by a division.  With r_t = 1 / (den_t + eps), the gradient is that of
// the unnormalised forward of [V | 1] with upstream [r_t g_t | -r_t (g_t . o_t)]:
//   1. n = forward(q, k, V) and den = forward(q, k, E) (E: a one in column 0 of a
//      16-wide value tile), both unnormalised;
//   2. gn = r g, g1 = [-r (g . n r), 0, ...] (one elementwise kernel);
//   3. (dq, dk, dv) = backward(q, k, V, gn), (dq1, dk1, -) = backward(q, k, E, g1);
//   4. dq += dq1, dk += dk1.
// The two parts of dq and dk cancel to a large degree (with positive features and
// zero-mean values the parts of dk are several times the sum), so every intermediate
// stays in fp32: bf16 inputs are widened once and the whole chain runs on the fp32
// CUDA-core kernels; rounding n, den, the upstream gradients or the partial results to
// bf16 costs several per cent of the result.
//
// The fp32 forward walks a sequence's chunks in one CTA, so step 1 splits every
// sequence into P equal segments viewed as heads of their own: a forward from zero
// gives each segment's state, an exclusive scan over the segments of a sequence (the
// concatenation rule of section 4) gives each segment's initial state, and a second
// forward from those states gives the outputs.
//
// From a given initial state (S, C, m, G, h): both forwards start from it, the values'
// pass from (S, C, G) and the unit values' pass from (S, C1, G1) with m and h in column
// 0 of C1 and G1 (den is the output of unit values); both backward passes return their
// state gradients, and dS = dS_1 + dS_2, dC, dG from the values' pass, dm and dh from
// column 0 of the unit pass's dC1, dG1.
#include <cstdint>
#include <cstdio>

#include "hla_internal.h"

namespace hla {
namespace {

constexpr int kEwThreads = 256;

template <typename T>
__device__ __forceinline__ float ldx(const T *p, size_t i);
template <>
__device__ __forceinline__ float ldx<__nv_bfloat16>(const __nv_bfloat16 *p, size_t i) {
    return __bfloat162float(p[i]);
}
template <typename T>
__device__ __forceinline__ void stx(T *p, size_t i, float x);
template <>
__device__ __forceinline__ void stx<float>(float *p, size_t i, float x) { p[i] = x; }
template <>
__device__ __forceinline__ void stx<__nv_bfloat16>(__nv_bfloat16 *p, size_t i, float x) {
    p[i] = __float2bfloat16_rn(x);
}

// E: [rows][w1] with a one in column 0.
__global__ void __launch_bounds__(kEwThreads) unit_value_kernel(float *e, size_t rows, int w1) {
    for (size_t i = (size_t)blockIdx.x * kEwThreads + threadIdx.x; i < rows * w1; i += (size_t)gridDim.x * kEwThreads)
        e[i] = (i % w1) == 0 ? 1.f : 0.f;
}

// One token row per warp: gn = r g, g1[., 0] = -r (g . n) r, other columns 0.
__global__ void __launch_bounds__(kEwThreads) norm_upstream_kernel(const float *num, const float *den1, const float *g,
                                                                    float *gn, float *g1, size_t rows, int dv, int w1,
                                                                    float eps) {
    const int lane = threadIdx.x & 31;
    for (size_t r = ((size_t)blockIdx.x * kEwThreads + threadIdx.x) / 32; r < rows;
         r += (size_t)gridDim.x * kEwThreads / 32) {
        const float rr = 1.f / (den1[r * w1] + eps);
        float dot = 0.f;
        for (int j = lane; j < dv; j += 32) {
            const float gj = g[r * dv + j];
            dot = fmaf(gj, num[r * dv + j], dot);
            gn[r * dv + j] = rr * gj;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
        for (int j = lane; j < w1; j += 32) g1[r * w1 + j] = j == 0 ? -rr * rr * dot : 0.f;
    }
}

// Exclusive scan over the P segments of each sequence: pre_0 = 0, pre_s = pre_{s-1} (+)
// seg_{s-1} by the concatenation rule with A = pre_{s-1}, B = seg_{s-1}, f = g^{len}:
//   S = f S_A + S_B, C = f C_A + C_B, m = f m_A + m_B,
//   G = f^2 G_A + G_B + f S_B C_A, h = f^2 h_A + h_B + f S_B m_A.
// Item i = sequence * P + s.  CTA (sequence, row block) writes rows [r0, r0 + kScanRows)
// of every state; each keeps its own copy of the whole prefix C and m (the right
// factor of the cross terms) in shared memory.
// Capacity: d <= 128 and d * dv <= 4096 (d <= 64 with dv <= 64; d = 128 runs over value
// slices of at most 32 columns).
constexpr int kScanMaxD = 128, kScanMaxC = 4096, kScanRows = 16;
// init: the state before the first segment of every sequence (init.S NULL: zeros).
__global__ void __launch_bounds__(kEwThreads) segment_scan_kernel(StatePtrs seg, StatePtrs pre, StatePtrs init, int P,
                                                                   int d, int dv, int H, const float *gamma,
                                                                   int seg_len) {
    __shared__ float sb[kScanRows * kScanMaxD], ca[kScanMaxC], ma[kScanMaxD];
    const int seq = blockIdx.x, r0 = blockIdx.y * kScanRows, tid = threadIdx.x;
    const size_t nS = (size_t)d * d, nC = (size_t)d * dv;
    const float f = gamma ? exp2f(log2f(gamma[seq % H]) * (float)seg_len) : 1.f, f2 = f * f;
    {
        const size_t i0 = (size_t)seq * P;
        const bool given = init.S != nullptr;
        for (int e = tid; e < kScanRows * d; e += kEwThreads)
            pre.S[i0 * nS + (size_t)r0 * d + e] = given ? init.S[(size_t)seq * nS + (size_t)r0 * d + e] : 0.f;
        for (int e = tid; e < kScanRows * dv; e += kEwThreads) {
            const size_t g = (size_t)seq * nC + (size_t)r0 * dv + e;
            pre.C[i0 * nC + (size_t)r0 * dv + e] = given ? init.C[g] : 0.f;
            pre.G[i0 * nC + (size_t)r0 * dv + e] = given ? init.G[g] : 0.f;
        }
        for (int e = tid; e < kScanRows; e += kEwThreads) {
            pre.m[i0 * d + r0 + e] = given ? init.m[(size_t)seq * d + r0 + e] : 0.f;
            pre.h[i0 * d + r0 + e] = given ? init.h[(size_t)seq * d + r0 + e] : 0.f;
        }
        for (size_t e = tid; e < nC; e += kEwThreads) ca[e] = given ? init.C[(size_t)seq * nC + e] : 0.f;
        for (int e = tid; e < d; e += kEwThreads) ma[e] = given ? init.m[(size_t)seq * d + e] : 0.f;
    }
    __syncthreads();
    for (int s = 1; s < P; ++s) {
        const size_t a = (size_t)seq * P + s - 1;  // pre_{s-1} and seg_{s-1}; pre_s is item a + 1
        for (int e = tid; e < kScanRows * d; e += kEwThreads) sb[e] = seg.S[a * nS + (size_t)r0 * d + e];
        __syncthreads();
        for (int e = tid; e < kScanRows * dv; e += kEwThreads) {
            const int r = e / dv, c = e % dv;
            const size_t gi = a * nC + (size_t)(r0 + r) * dv + c;
            float acc = 0.f;
            for (int k = 0; k < d; ++k) acc = fmaf(sb[r * d + k], ca[k * dv + c], acc);
            pre.G[gi + nC] = f2 * pre.G[gi] + seg.G[gi] + f * acc;
            pre.C[gi + nC] = f * ca[(r0 + r) * dv + c] + seg.C[gi];
        }
        for (int r = tid; r < kScanRows; r += kEwThreads) {
            float acc = 0.f;
            for (int k = 0; k < d; ++k) acc = fmaf(sb[r * d + k], ma[k], acc);
            const size_t hi = a * d + r0 + r;
            pre.h[hi + d] = f2 * pre.h[hi] + seg.h[hi] + f * acc;
            pre.m[hi + d] = f * ma[r0 + r] + seg.m[hi];
        }
        for (int e = tid; e < kScanRows * d; e += kEwThreads) {
            const size_t si = a * nS + (size_t)r0 * d + e;
            pre.S[si + nS] = f * pre.S[si] + sb[e];
        }
        __syncthreads();  // every read of ca, ma and sb for this step is done
        for (size_t e = tid; e < nC; e += kEwThreads) ca[e] = f * ca[e] + seg.C[a * nC + e];
        for (int e = tid; e < d; e += kEwThreads) ma[e] = f * ma[e] + seg.m[a * d + e];
        __syncthreads();
    }
}

// d-vectors per pair <-> column 0 of [d][w1] tiles (the other columns zero)
__global__ void __launch_bounds__(kEwThreads) to_column_kernel(float *dst, const float *src, size_t count, int w1) {
    for (size_t i = (size_t)blockIdx.x * kEwThreads + threadIdx.x; i < count * w1; i += (size_t)gridDim.x * kEwThreads)
        dst[i] = (i % w1) == 0 ? src[i / w1] : 0.f;
}
__global__ void __launch_bounds__(kEwThreads) from_column_kernel(float *dst, const float *src, size_t count, int w1) {
    for (size_t i = (size_t)blockIdx.x * kEwThreads + threadIdx.x; i < count; i += (size_t)gridDim.x * kEwThreads)
        dst[i] = src[i * w1];
}

__global__ void __launch_bounds__(kEwThreads) repeat_kernel(float *dst, const float *src, int H, int P) {
    for (int i = threadIdx.x; i < H * P; i += kEwThreads) dst[i] = src[i / P];
}

template <typename Ti>
__global__ void __launch_bounds__(kEwThreads) widen_kernel(float *dst, const Ti *src, size_t count) {
    for (size_t i = (size_t)blockIdx.x * kEwThreads + threadIdx.x; i < count; i += (size_t)gridDim.x * kEwThreads)
        dst[i] = ldx(src, i);
}

// dst = a + b (b NULL: dst = a), rounded once to the output type; dst may alias a.
template <typename To>
__global__ void __launch_bounds__(kEwThreads) sum_kernel(To *dst, const float *a, const float *b, size_t count) {
    for (size_t i = (size_t)blockIdx.x * kEwThreads + threadIdx.x; i < count; i += (size_t)gridDim.x * kEwThreads)
        stx(dst, i, b ? a[i] + b[i] : a[i]);
}

int grid_for(size_t work) {
    const size_t b = (work + kEwThreads - 1) / kEwThreads;
    return (int)(b < 8192 ? (b > 0 ? b : 1) : 8192);
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

hla_status cuda_err(cudaError_t e, const char *where) {
    char msg[192];
    snprintf(msg, sizeof msg, "normalised backward, %s: %s", where, cudaGetErrorString(e));
    return report(HLA_ERR_CUDA, msg);
}

constexpr int kUnitWidth = 16;

// Segments per sequence for the forwards: a power of two up to 16 that divides n into
// pieces of at least one chunk, with B H P at most 4 x 152 CTAs; 1 (no split) with
// shared key/value heads, whose head mapping the segment view does not keep.
int segments(const hla_params &p) {
    const int hkv = p.Hkv > 0 ? p.Hkv : p.H;
    if (hkv != p.H) return 1;
    int P = 1;
    while (P < 16 && p.n % (2 * P) == 0 && p.n / (2 * P) >= p.chunk && (long long)p.B * p.H * 2 * P <= 4 * 152) P *= 2;
    return P;
}

size_t state_floats(int d, int dv) { return (size_t)d * d + 2 * (size_t)d * dv + 2 * (size_t)d; }

// The unnormalised fp32 problem of width dv.
hla_params unnormalised(const hla_params &p, int dv) {
    hla_params q = p;
    q.flags &= ~(unsigned)HLA_NORMALIZE;
    q.in_dtype = HLA_F32;
    q.dv = dv;
    q.eps = 0.f;
    return q;
}

}  // namespace

NormLayout bwd_norm_layout(const hla_params &p) {
    NormLayout L;
    const int hkv = p.Hkv > 0 ? p.Hkv : p.H;
    const size_t rq = (size_t)p.B * p.H * p.n, rkv = (size_t)p.B * hkv * p.n;
    const int w1 = kUnitWidth;
    const hla_params pv = unnormalised(p, p.dv), pe = unnormalised(p, w1);
    const size_t fws = hla_forward_workspace_size(&pv), fws1 = hla_forward_workspace_size(&pe);
    const size_t bws = bwd_simt_workspace(pv), bws1 = bwd_simt_workspace(pe);
    const bool wide = p.in_dtype != HLA_F32;
    size_t o = 0;
    auto take = [&](size_t floats) { const size_t at = o; o = align256(o + floats * 4); return at; };
    L.w1 = w1;
    L.fwd_ws_bytes = fws > fws1 ? fws : fws1;
    L.fwd_ws = take((L.fwd_ws_bytes + 3) / 4);
    L.num = take(rq * p.dv);
    L.den1 = take(rq * w1);
    L.unit = take(rkv * w1);
    L.gn = take(rq * p.dv);
    L.g1 = take(rq * w1);
    L.dq1 = take(rq * p.d);
    L.dk1 = take(rkv * p.d);
    L.dv1 = take(rkv * w1);
    L.bwd_ws = take(((bws > bws1 ? bws : bws1) + 3) / 4);
    // segmented forwards: the repeated decay rates and two state sets (segments, prefixes)
    L.P = segments(p);
    const size_t items = (size_t)p.B * p.H * L.P, sf = state_floats(p.d, p.dv > w1 ? p.dv : w1);
    L.grep = L.P > 1 ? take((size_t)p.H * L.P) : 0;
    L.seg = L.P > 1 ? take(items * sf) : 0;
    L.pre = L.P > 1 ? take(items * sf) : 0;
    const size_t units = (size_t)p.B * p.H;
    L.ce = take(units * p.d * w1);
    L.ge = take(units * p.d * w1);
    L.ds2 = take(units * p.d * p.d);
    L.dce = take(units * p.d * w1);
    L.dge = take(units * p.d * w1);
    L.zvec = take(units * p.d);
    // bf16 inputs: fp32 copies of q, k, v, g and fp32 results before the final rounding
    L.q32 = wide ? take(rq * p.d) : 0;
    L.k32 = wide ? take(rkv * p.d) : 0;
    L.v32 = wide ? take(rkv * p.dv) : 0;
    L.g32 = wide ? take(rq * p.dv) : 0;
    L.dq32 = wide ? take(rq * p.d) : 0;
    L.dk32 = wide ? take(rkv * p.d) : 0;
    L.dv32 = wide ? take(rkv * p.dv) : 0;
    L.total = o;
    return L;
}

hla_status bwd_norm_launch(const hla_params &p, const BwdArgs &a0, void *workspace, cudaStream_t st) {
    const NormLayout L = bwd_norm_layout(p);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    auto f = [&](size_t off) { return reinterpret_cast<float *>(ws + off); };
    const int hkv = p.Hkv > 0 ? p.Hkv : p.H;
    const size_t rq = (size_t)p.B * p.H * p.n, rkv = (size_t)p.B * hkv * p.n;
    const bool wide = p.in_dtype != HLA_F32;
    auto mark = [&](int i) { return a0.events ? cudaEventRecord(a0.events[i], st) : cudaSuccess; };
    cudaError_t e;
    if ((e = mark(0)) != cudaSuccess) return cuda_err(e, "event");
    // fp32 operands
    const float *q = static_cast<const float *>(a0.q), *k = static_cast<const float *>(a0.k);
    const float *v = static_cast<const float *>(a0.v), *g = static_cast<const float *>(a0.go);
    float *dq = static_cast<float *>(a0.grad_q), *dk = static_cast<float *>(a0.grad_k);
    float *dv = static_cast<float *>(a0.grad_v);
    if (wide) {
        const __nv_bfloat16 *src[4] = {static_cast<const __nv_bfloat16 *>(a0.q), static_cast<const __nv_bfloat16 *>(a0.k),
                                       static_cast<const __nv_bfloat16 *>(a0.v),
                                       static_cast<const __nv_bfloat16 *>(a0.go)};
        float *dst[4] = {f(L.q32), f(L.k32), f(L.v32), f(L.g32)};
        const size_t cnt[4] = {rq * p.d, rkv * p.d, rkv * p.dv, rq * p.dv};
        for (int i = 0; i < 4; ++i)
            widen_kernel<__nv_bfloat16><<<grid_for(cnt[i]), kEwThreads, 0, st>>>(dst[i], src[i], cnt[i]);
        q = dst[0]; k = dst[1]; v = dst[2]; g = dst[3];
        dq = f(L.dq32); dk = f(L.dk32); dv = f(L.dv32);
    }
    // 1. numerator and denominator (unnormalised forwards)
    if (L.fwd_ws_bytes && (e = cudaMemsetAsync(ws + L.fwd_ws, 0, L.fwd_ws_bytes, st)) != cudaSuccess)
        return cuda_err(e, "workspace clear");
    unit_value_kernel<<<grid_for(rkv * L.w1), kEwThreads, 0, st>>>(f(L.unit), rkv, L.w1);
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_err(e, "operands");
    const hla_params pv = unnormalised(p, p.dv), pe = unnormalised(p, L.w1);
    // a given initial state: (S, C, G) for the values, (S, C1, G1) with m, h in column 0
    // for the unit values; m and h of both are unused by the unnormalised passes
    const bool given = a0.sin_S != nullptr, want = a0.dS != nullptr;
    const size_t units = (size_t)p.B * p.H, pd = units * p.d;
    hla_state sv{}, se{};
    if (given || want) {
        if ((e = cudaMemsetAsync(f(L.zvec), 0, pd * 4, st)) != cudaSuccess) return cuda_err(e, "state operands");
    }
    if (given) {
        to_column_kernel<<<grid_for(pd * L.w1), kEwThreads, 0, st>>>(f(L.ce), a0.sin_m, pd, L.w1);
        to_column_kernel<<<grid_for(pd * L.w1), kEwThreads, 0, st>>>(f(L.ge), a0.sin_h, pd, L.w1);
        if ((e = cudaGetLastError()) != cudaSuccess) return cuda_err(e, "state operands");
        sv = hla_state{const_cast<float *>(a0.sin_S), const_cast<float *>(a0.sin_C), f(L.zvec),
                       const_cast<float *>(a0.sin_G), f(L.zvec)};
        se = hla_state{const_cast<float *>(a0.sin_S), f(L.ce), f(L.zvec), f(L.ge), f(L.zvec)};
    }
    const hla_state *sv_in = given ? &sv : nullptr, *se_in = given ? &se : nullptr;
    hla_status s;
    if (L.P == 1) {
        s = hla_forward_chunked(&pv, q, k, v, f(L.num), sv_in, nullptr, ws + L.fwd_ws, L.fwd_ws_bytes, st);
        if (s != HLA_OK) return s;
        s = hla_forward_chunked(&pe, q, k, f(L.unit), f(L.den1), se_in, nullptr, ws + L.fwd_ws, L.fwd_ws_bytes, st);
        if (s != HLA_OK) return s;
    } else {
        const int P = L.P;
        if (p.flags & HLA_DECAY) repeat_kernel<<<1, kEwThreads, 0, st>>>(f(L.grep), p.gamma, p.H, P);
        const size_t items = (size_t)p.B * p.H * P;
        for (int part = 0; part < 2; ++part) {
            hla_params ps = part == 0 ? pv : pe;
            const int dvp = ps.dv;
            ps.H = p.H * P;
            ps.Hkv = p.H * P;
            ps.n = p.n / P;
            ps.gamma = (p.flags & HLA_DECAY) ? f(L.grep) : nullptr;
            const size_t nS = (size_t)p.d * p.d, nC = (size_t)p.d * dvp;
            auto states = [&](size_t off) {
                hla_state t;
                t.S = f(off);
                t.C = t.S + items * nS;
                t.m = t.C + items * nC;
                t.G = t.m + items * p.d;
                t.h = t.G + items * nC;
                return t;
            };
            const hla_state sg = states(L.seg), pr = states(L.pre);
            const void *vv = part == 0 ? static_cast<const void *>(v) : f(L.unit);
            float *out = part == 0 ? f(L.num) : f(L.den1);
            s = hla_forward_chunked(&ps, q, k, vv, out, nullptr, &sg, ws + L.fwd_ws, L.fwd_ws_bytes, st);
            if (s != HLA_OK) return s;
            StatePtrs init{};
            if (given) init = to_ptrs(part == 0 ? &sv : &se);
            if (p.d > kScanMaxD || (size_t)p.d * dvp > (size_t)kScanMaxC)
                return hla::report(HLA_ERR_UNSUPPORTED, "normalised backward: state too wide for the segment scan");
            segment_scan_kernel<<<dim3(p.B * p.H, p.d / kScanRows), kEwThreads, 0, st>>>(
                to_ptrs(&sg), to_ptrs(&pr), init, P, p.d, dvp, p.H, (p.flags & HLA_DECAY) ? p.gamma : nullptr, p.n / P);
            if ((e = cudaGetLastError()) != cudaSuccess) return cuda_err(e, "segment scan");
            s = hla_forward_chunked(&ps, q, k, vv, out, &pr, nullptr, ws + L.fwd_ws, L.fwd_ws_bytes, st);
            if (s != HLA_OK) return s;
        }
    }
    // 2. upstream gradients of the augmented problem
    norm_upstream_kernel<<<grid_for(rq * 32), kEwThreads, 0, st>>>(f(L.num), f(L.den1), g, f(L.gn), f(L.g1), rq,
                                                                    p.dv, L.w1, p.eps);
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_err(e, "upstream gradients");
    if ((e = mark(1)) != cudaSuccess) return cuda_err(e, "event");
    // 3. the two unnormalised backward passes
    BwdArgs a = a0;
    a.in_dtype = HLA_F32;
    a.events = nullptr;
    a.q = q; a.k = k; a.v = v; a.go = f(L.gn);
    a.grad_q = dq; a.grad_k = dk; a.grad_v = dv;
    a.workspace = f(L.bwd_ws);
    a.dk_pair = a.Hkv < a.H ? a.workspace + bwd_pair_offset(pv) : nullptr;
    a.dv_pair = a.dk_pair ? a.dk_pair + rq * p.d : nullptr;
    a.adj0 = want ? a.workspace + bwd_adj0_offset(pv) : nullptr;  // dS, dC, dG of the values' pass: final
    if ((e = bwd_simt_launch(a, st)) != cudaSuccess) return cuda_err(e, "backward of the numerator");
    if ((e = mark(2)) != cudaSuccess) return cuda_err(e, "event");
    BwdArgs b = a;
    b.dv = L.w1;
    b.v = f(L.unit);
    b.go = f(L.g1);
    b.grad_q = f(L.dq1);
    b.grad_k = f(L.dk1);
    b.grad_v = f(L.dv1);
    b.dk_pair = b.Hkv < b.H ? b.workspace + bwd_pair_offset(pe) : nullptr;
    b.dv_pair = b.dk_pair ? b.dk_pair + rq * p.d : nullptr;
    b.sin_C = given ? f(L.ce) : nullptr;
    b.sin_G = given ? f(L.ge) : nullptr;
    b.dS = want ? f(L.ds2) : nullptr;
    b.dC = want ? f(L.dce) : nullptr;
    b.dG = want ? f(L.dge) : nullptr;
    b.adj0 = want ? b.workspace + bwd_adj0_offset(pe) : nullptr;
    if ((e = bwd_simt_launch(b, st)) != cudaSuccess) return cuda_err(e, "backward of the denominator");
    if (want) {  // dS += dS of the unit pass; dm, dh from column 0 of its dC, dG
        sum_kernel<float><<<grid_for(units * p.d * p.d), kEwThreads, 0, st>>>(a0.dS, a0.dS, f(L.ds2),
                                                                              units * p.d * p.d);
        from_column_kernel<<<grid_for(pd), kEwThreads, 0, st>>>(a0.dm, f(L.dce), pd, L.w1);
        from_column_kernel<<<grid_for(pd), kEwThreads, 0, st>>>(a0.dh, f(L.dge), pd, L.w1);
        if ((e = cudaGetLastError()) != cudaSuccess) return cuda_err(e, "state gradient");
    }
    // 4. dq = dq + dq1, dk = dk + dk1 (and dv), each rounded once to the output type
    if (wide) {
        sum_kernel<__nv_bfloat16><<<grid_for(rq * p.d), kEwThreads, 0, st>>>(
            static_cast<__nv_bfloat16 *>(a0.grad_q), dq, f(L.dq1), rq * p.d);
        sum_kernel<__nv_bfloat16><<<grid_for(rkv * p.d), kEwThreads, 0, st>>>(
            static_cast<__nv_bfloat16 *>(a0.grad_k), dk, f(L.dk1), rkv * p.d);
        sum_kernel<__nv_bfloat16><<<grid_for(rkv * p.dv), kEwThreads, 0, st>>>(
            static_cast<__nv_bfloat16 *>(a0.grad_v), dv, nullptr, rkv * p.dv);
    } else {
        sum_kernel<float><<<grid_for(rq * p.d), kEwThreads, 0, st>>>(dq, dq, f(L.dq1), rq * p.d);
        sum_kernel<float><<<grid_for(rkv * p.d), kEwThreads, 0, st>>>(dk, dk, f(L.dk1), rkv * p.d);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_err(e, "gradient sums");
    if ((e = mark(3)) != cudaSuccess) return cuda_err(e, "event");
    return HLA_OK;
}

}  // namespace hla
