// Tensor-core forward kernels with decay=false, normalise=true, masked output (all supported shapes).
#include "hla_fwd_ws2.cuh"

template cudaError_t hla::tc::launch_flags<false, true, 0>(const hla::FwdArgs &, cudaStream_t, int);
template cudaError_t hla::ws::ws_launch_flags<false, true>(const hla::FwdArgs &, cudaStream_t, int);
template cudaError_t hla::ws2::launch_flags<true>(const hla::FwdArgs &, cudaStream_t, int);
