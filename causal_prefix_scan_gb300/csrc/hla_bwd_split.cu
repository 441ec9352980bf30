// hla_bwd_split.cu -- the copies around a call split over value columns (the backward
// pass, and the third-order forward, whose output and value-width state columns split the
// same way: column j depends on the values' column j only).  The backward at d = 128 runs
// over slices of 32 value columns; otherwise a split is two halves of 64.
//
// The loss sum_t dout_t . o_t is a sum over value columns, and column j of the output
// depends on column j of the values only (o_t[j] = q_t^T X_t[:, j], X_t[:, j] built from
// v[:, j]).  So the gradient for dv = 128 is the sum of the gradients of two 64-column
// problems (same q, k; value and upstream columns [0, 64) and [64, 128)): dq and dk add,
// dv is the two halves side by side (likewise for any number of equal slices).  With ratio normalisation each half keeps the full
// denominator (it does not depend on the values), and its upstream for the unit column
// is its own share r (dout_h . o_h) of r (dout . o), so the halves add up exactly too.
// These kernels gather a half of the value columns, scatter a half back, and accumulate
// dq, dk in fp32 before the one final rounding.
#include "hla_internal.h"

namespace hla {
namespace {

constexpr int kThreads = 256;

int grid_for(size_t work) {
    const size_t b = (work + kThreads - 1) / kThreads;
    return (int)(b < 8192 ? (b > 0 ? b : 1) : 8192);
}

// Columns [part*w, part*w+w) of [rows][nparts*w] elements <-> [rows][w], in 16-byte
// pieces (per_row pieces of a narrow row: w elements of 2 or 4 bytes).
__global__ void __launch_bounds__(kThreads) cols_copy_kernel(const uint4 *src, uint4 *dst, size_t rows, int per_row,
                                                             int nparts, int part, int gather) {
    const size_t total = rows * per_row;
    for (size_t i = (size_t)blockIdx.x * kThreads + threadIdx.x; i < total; i += (size_t)gridDim.x * kThreads) {
        const size_t r = i / per_row, c = i % per_row;
        const size_t wide = r * nparts * per_row + (size_t)part * per_row + c, narrow = r * per_row + c;
        if (gather) dst[narrow] = src[wide];
        else dst[wide] = src[narrow];
    }
}

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__global__ void __launch_bounds__(kThreads) acc_add_kernel(float *acc, const T *src, size_t count, int first) {
    for (size_t i = (size_t)blockIdx.x * kThreads + threadIdx.x; i < count; i += (size_t)gridDim.x * kThreads)
        acc[i] = first ? to_f(src[i]) : acc[i] + to_f(src[i]);
}

template <typename T>
__global__ void __launch_bounds__(kThreads) acc_store_kernel(T *dst, const float *acc, size_t count);
template <>
__global__ void __launch_bounds__(kThreads) acc_store_kernel<float>(float *dst, const float *acc, size_t count) {
    for (size_t i = (size_t)blockIdx.x * kThreads + threadIdx.x; i < count; i += (size_t)gridDim.x * kThreads)
        dst[i] = acc[i];
}
template <>
__global__ void __launch_bounds__(kThreads) acc_store_kernel<__nv_bfloat16>(__nv_bfloat16 *dst, const float *acc,
                                                                            size_t count) {
    for (size_t i = (size_t)blockIdx.x * kThreads + threadIdx.x; i < count; i += (size_t)gridDim.x * kThreads)
        dst[i] = __float2bfloat16_rn(acc[i]);
}

}  // namespace

cudaError_t cols_part_copy(const void *src, void *dst, size_t rows, hla_dtype dt, int width, int part_width,
                           int part, bool gather, cudaStream_t st) {
    const int el = dt == HLA_F32 ? 4 : 2;
    if (part_width * el % 16 != 0 || width % part_width != 0 || part < 0 || part >= width / part_width)
        return cudaErrorInvalidValue;
    const int per_row = part_width * el / 16;
    cols_copy_kernel<<<grid_for(rows * per_row), kThreads, 0, st>>>(static_cast<const uint4 *>(src),
                                                                     static_cast<uint4 *>(dst), rows, per_row,
                                                                     width / part_width, part, gather ? 1 : 0);
    return cudaGetLastError();
}

cudaError_t acc_add(float *acc, const void *src, size_t count, hla_dtype dt, bool first, cudaStream_t st) {
    if (dt == HLA_F32)
        acc_add_kernel<float><<<grid_for(count), kThreads, 0, st>>>(acc, static_cast<const float *>(src), count, first);
    else
        acc_add_kernel<__nv_bfloat16><<<grid_for(count), kThreads, 0, st>>>(
            acc, static_cast<const __nv_bfloat16 *>(src), count, first);
    return cudaGetLastError();
}

cudaError_t acc_store(void *dst, const float *acc, size_t count, hla_dtype dt, cudaStream_t st) {
    if (dt == HLA_F32)
        acc_store_kernel<float><<<grid_for(count), kThreads, 0, st>>>(static_cast<float *>(dst), acc, count);
    else
        acc_store_kernel<__nv_bfloat16><<<grid_for(count), kThreads, 0, st>>>(static_cast<__nv_bfloat16 *>(dst), acc,
                                                                             count);
    return cudaGetLastError();
}

}  // namespace hla
