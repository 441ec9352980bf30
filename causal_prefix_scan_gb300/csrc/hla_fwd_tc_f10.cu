// Tensor-core forward kernels with decay=true, normalise=true, unmasked output (all supported shapes).
#include "hla_fwd_tc.cuh"

template cudaError_t hla::tc::launch_flags<true, true, 1>(const hla::FwdArgs &, cudaStream_t, int);
