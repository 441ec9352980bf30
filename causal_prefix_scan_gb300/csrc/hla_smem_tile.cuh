// hla_smem_tile.cuh -- small fp32 matrix products on shared-memory tiles for the
// CUDA-core kernels (backward, third order): each thread accumulates a 4x4 register
// tile; operands are row-major shared-memory arrays with padded rows, read as float4.
#pragma once
#include "hla_internal.h"

namespace hla {
namespace tile {

constexpr int kThreads = 256;

template <typename T>
__device__ __forceinline__ float ld_t(const T *p, size_t i);
template <>
__device__ __forceinline__ float ld_t<float>(const float *p, size_t i) { return p[i]; }
template <>
__device__ __forceinline__ float ld_t<__nv_bfloat16>(const __nv_bfloat16 *p, size_t i) {
    return __bfloat162float(p[i]);
}
template <typename T>
__device__ __forceinline__ void st_t(T *p, size_t i, float x);
template <>
__device__ __forceinline__ void st_t<float>(float *p, size_t i, float x) { p[i] = x; }
template <>
__device__ __forceinline__ void st_t<__nv_bfloat16>(__nv_bfloat16 *p, size_t i, float x) {
    p[i] = __float2bfloat16_rn(x);
}

// ---- small shared-memory products on a 4x4 register tile per thread --------------
// acc[i][j] += sum_k w_k A(m0+i, k) B(k, n0 + j*ns).  A(m,k) = TA ? A[k*lda+m] : A[m*lda+k];
// B(k,n) = TB ? B[n*ldb+k] : B[k*ldb+n].  K a multiple of 4, leading dimensions multiples
// of 4 floats, bases 16-byte aligned.  ns == 1: four adjacent columns; else strided.
template <bool TA, bool TB>
__device__ __forceinline__ void mac(float (&acc)[4][4], const float *A, int lda, const float *B, int ldb, int m0,
                                    int n0, int ns, int K, const float *kw = nullptr) {
#pragma unroll 2
    for (int k = 0; k < K; k += 4) {
        float a[4][4], b[4][4];  // [kk][i], [kk][j]
        if (TA) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const float4 x = *reinterpret_cast<const float4 *>(A + (size_t)(k + kk) * lda + m0);
                a[kk][0] = x.x; a[kk][1] = x.y; a[kk][2] = x.z; a[kk][3] = x.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float4 x = *reinterpret_cast<const float4 *>(A + (size_t)(m0 + i) * lda + k);
                a[0][i] = x.x; a[1][i] = x.y; a[2][i] = x.z; a[3][i] = x.w;
            }
        }
        if (kw) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const float w = kw[k + kk];
#pragma unroll
                for (int i = 0; i < 4; ++i) a[kk][i] *= w;
            }
        }
        if (TB) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float4 x = *reinterpret_cast<const float4 *>(B + (size_t)(n0 + j * ns) * ldb + k);
                b[0][j] = x.x; b[1][j] = x.y; b[2][j] = x.z; b[3][j] = x.w;
            }
        } else if (ns == 1) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const float4 x = *reinterpret_cast<const float4 *>(B + (size_t)(k + kk) * ldb + n0);
                b[kk][0] = x.x; b[kk][1] = x.y; b[kk][2] = x.z; b[kk][3] = x.w;
            }
        } else {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                for (int j = 0; j < 4; ++j) b[kk][j] = B[(size_t)(k + kk) * ldb + n0 + j * ns];
        }
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[kk][i], b[kk][j], acc[i][j]);
    }
}

// The same term scaled by rs[row] before it is added.
template <bool TA, bool TB>
__device__ __forceinline__ void mac_rs(float (&acc)[4][4], const float *rs, const float *A, int lda, const float *B,
                                       int ldb, int m0, int n0, int ns, int K) {
    float t[4][4] = {};
    mac<TA, TB>(t, A, lda, B, ldb, m0, n0, ns, K);
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(rs[m0 + i], t[i][j], acc[i][j]);
}

// Every 4x4 tile of an M x N result, one per thread per round.  STRIDED spreads a
// thread's four columns N/4 apart (conflict-free rows when B is read transposed).
template <bool STRIDED, class Body>
__device__ __forceinline__ void tiles(int M, int N, Body body) {
    const int tn = N / 4, count = (M / 4) * tn;
    for (int t = threadIdx.x; t < count; t += kThreads) {
        const int m0 = (t / tn) * 4;
        const int n0 = STRIDED ? t % tn : (t % tn) * 4, ns = STRIDED ? tn : 1;
        float acc[4][4] = {};
        body(acc, m0, n0, ns);
    }
}

template <class F>
__device__ __forceinline__ void each(const float (&acc)[4][4], int m0, int n0, int ns, F f) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) f(m0 + i, n0 + j * ns, acc[i][j]);
}

template <typename T>
__device__ __forceinline__ void load_rows(const T *src, float *dst, int ld, int rows, int L, int W) {
    for (int e = threadIdx.x; e < rows * W; e += kThreads) {
        const int r = e / W, x = e % W;
        dst[r * ld + x] = r < L ? ld_t(src, (size_t)r * W + x) : 0.f;
    }
}

// ---- asynchronous global -> shared copies (16-byte cp.async, L2 only) -------------
__device__ __forceinline__ void cp_async16(float *dst, const float *src) {
    const unsigned d = static_cast<unsigned>(__cvta_generic_to_shared(dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

// rows x cols floats (cols a multiple of 4; both leading dimensions multiples of 4,
// both bases 16-byte aligned) from global (ld src_ld) to shared (ld dst_ld).
__device__ __forceinline__ void copy_mat_async(const float *src, int src_ld, float *dst, int dst_ld, int rows,
                                               int cols) {
    const int q = cols / 4;
    for (int e = threadIdx.x; e < rows * q; e += kThreads) {
        const int r = e / q, c = (e % q) * 4;
        cp_async16(dst + (size_t)r * dst_ld + c, src + (size_t)r * src_ld + c);
    }
}

// acc[i][j] += sum_k A[(m0+i)*lda + k] B[k*ldb + n0+j] for a 2x2 tile (K a multiple of
// 4; lda a multiple of 4; n0 even, ldb even).
__device__ __forceinline__ void mac22(float (&acc)[2][2], const float *A, int lda, const float *B, int ldb, int m0,
                                      int n0, int K) {
#pragma unroll 4
    for (int k = 0; k < K; k += 4) {
        const float4 a0 = *reinterpret_cast<const float4 *>(A + (size_t)m0 * lda + k);
        const float4 a1 = *reinterpret_cast<const float4 *>(A + (size_t)(m0 + 1) * lda + k);
        const float av0[4] = {a0.x, a0.y, a0.z, a0.w}, av1[4] = {a1.x, a1.y, a1.z, a1.w};
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const float2 b = *reinterpret_cast<const float2 *>(B + (size_t)(k + kk) * ldb + n0);
            acc[0][0] = fmaf(av0[kk], b.x, acc[0][0]);
            acc[0][1] = fmaf(av0[kk], b.y, acc[0][1]);
            acc[1][0] = fmaf(av1[kk], b.x, acc[1][0]);
            acc[1][1] = fmaf(av1[kk], b.y, acc[1][1]);
        }
    }
}

// Every 2x2 tile of an M x N result (M, N even), one per thread per round.
template <class Body>
__device__ __forceinline__ void tiles22(int M, int N, Body body) {
    const int tn = N / 2, count = (M / 2) * tn;
    for (int t = threadIdx.x; t < count; t += kThreads) {
        float acc[2][2] = {};
        body(acc, (t / tn) * 2, (t % tn) * 2);
    }
}

}  // namespace tile
}  // namespace hla
