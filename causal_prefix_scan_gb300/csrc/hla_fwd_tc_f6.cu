// Tensor-core forward kernels with decay=true, normalise=false, masked output (all supported shapes).
#include "hla_fwd_tc.cuh"

template cudaError_t hla::tc::launch_flags<true, false, 0>(const hla::FwdArgs &, cudaStream_t, int);
