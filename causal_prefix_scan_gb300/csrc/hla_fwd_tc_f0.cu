// Tensor-core forward kernels with decay=false, normalise=false, masked output (all supported shapes).
#include "hla_fwd_tc.cuh"

template cudaError_t hla::tc::launch_flags<false, false, 0>(const hla::FwdArgs &, cudaStream_t, int);
