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
template <bool STRIDED, int M, int N, class Body>
__device__ __forceinline__ void tiles(Body body) {
    constexpr int tn = N / 4, count = (M / 4) * tn;
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

// `rows` rows of W values (row-major, ld W) into shared rows of ld `ld`; rows >= L zero.
template <int W, typename T>
__device__ __forceinline__ void load_rows(const T *src, float *dst, int ld, int rows, int L) {
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

// rows x COLS floats (COLS a multiple of 4; both leading dimensions multiples of 4,
// both bases 16-byte aligned) from global (ld src_ld) to shared (ld dst_ld).
template <int COLS>
__device__ __forceinline__ void copy_mat_async(const float *src, int src_ld, float *dst, int dst_ld, int rows) {
    constexpr int q = COLS / 4;
    for (int e = threadIdx.x; e < rows * q; e += kThreads) {
        const int r = e / q, c = (e % q) * 4;
        cp_async16(dst + (size_t)r * dst_ld + c, src + (size_t)r * src_ld + c);
    }
}

// Partial products of an M x N result (M a multiple of 4, N in {4, 8, 16}; K a power
// of two >= 4) over all threads: the (M/4)(N/4) 4x4 tiles times G contraction slices
// of K / G, G = min(kThreads / tiles, K / 4).  Thread t < tiles * G takes tile
// t % tiles and slice t / tiles and stores its 16 partial sums to
// red[slice][M][N]; ksplit_sum adds the G slices of one element.
__host__ __device__ constexpr int ksplit_slices(int M, int N, int K) {
    return (kThreads / ((M / 4) * (N / 4))) < K / 4 ? kThreads / ((M / 4) * (N / 4)) : K / 4;
}
template <int M, int N, int K>
__device__ __forceinline__ void mac_ksplit(const float *A, int lda, const float *B, int ldb, float *red) {
    constexpr int tn = N / 4, T = (M / 4) * tn, G = ksplit_slices(M, N, K), kr = K / G;
    if (threadIdx.x >= T * G) return;
    const int t = threadIdx.x % T, g = threadIdx.x / T;
    const int m0 = (t / tn) * 4, n0 = (t % tn) * 4;
    float acc[4][4] = {};
    mac<false, false>(acc, A + g * kr, lda, B + (size_t)g * kr * ldb, ldb, m0, n0, 1, kr);
#pragma unroll
    for (int i = 0; i < 4; ++i)
        *reinterpret_cast<float4 *>(red + ((size_t)g * M + m0 + i) * N + n0) =
            make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
}
template <int M, int N, int K>
__device__ __forceinline__ float ksplit_sum(const float *red, int e) {
    constexpr int G = ksplit_slices(M, N, K);
    float s = 0.f;
#pragma unroll
    for (int g = 0; g < G; ++g) s += red[(size_t)g * M * N + e];
    return s;
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
