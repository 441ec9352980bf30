// Tensor-core forward kernels with decay=true, normalise=true, masked output (all supported shapes).
#include "hla_fwd_ws.cuh"

template cudaError_t hla::tc::launch_flags<true, true, 0>(const hla::FwdArgs &, cudaStream_t, int);
template cudaError_t hla::ws::ws_launch_flags<true, true>(const hla::FwdArgs &, cudaStream_t, int);
