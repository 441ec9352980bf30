// Tensor-core forward kernels with decay=false, normalise=true, unmasked output (all supported shapes).
#include "hla_fwd_tc.cuh"

template cudaError_t hla::tc::launch_flags<false, true, 1>(const hla::FwdArgs &, cudaStream_t, int);
