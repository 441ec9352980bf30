// Tensor-core forward kernels with decay=false, normalise=false, masked output (all supported shapes).
#include "hla_fwd_ws2.cuh"

template cudaError_t hla::tc::launch_flags<false, false, 0>(const hla::FwdArgs &, cudaStream_t, int);
template cudaError_t hla::ws::ws_launch_flags<false, false>(const hla::FwdArgs &, cudaStream_t, int);
template cudaError_t hla::ws2::launch_flags<false>(const hla::FwdArgs &, cudaStream_t, int);
