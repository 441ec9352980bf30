// hla_tmap.h -- host-side tensor maps for the TMA tile loads: a [units][n][width] bf16
// tensor read in boxes of 64 features x box_rows tokens of one unit, 128-byte swizzled
// (the layout the kernels' shared-memory tiles use); rows past n read as zeros.
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>

#include "hla_internal.h"

namespace hla {
namespace tc {

inline PFN_cuTensorMapEncodeTiled_v12000 get_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

inline bool encode_3d(CUtensorMap *tm, const void *ptr, int width, int n, int BH, int box_rows) {
    auto enc = get_encoder();
    if (!enc) return false;
    cuuint64_t gdim[3] = {(cuuint64_t)width, (cuuint64_t)n, (cuuint64_t)BH};
    cuuint64_t gstr[2] = {(cuuint64_t)width * 2, (cuuint64_t)width * 2 * (cuuint64_t)n};
    cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), gdim, gstr, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tc
}  // namespace hla
