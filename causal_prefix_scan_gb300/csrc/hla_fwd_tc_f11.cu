// Tensor-core forward kernels with decay=true, normalise=true, asymmetric (AHLA) output (all supported shapes).
#include "hla_fwd_tc.cuh"

template cudaError_t hla::tc::launch_flags<true, true, 2>(const hla::FwdArgs &, cudaStream_t, int);
