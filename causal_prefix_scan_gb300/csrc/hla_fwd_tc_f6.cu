// Tensor-core forward kernels with decay=true, normalise=false, masked output (all supported shapes).
#include "hla_fwd_ws.cuh"

template cudaError_t hla::tc::launch_flags<true, false, 0>(const hla::FwdArgs &, cudaStream_t, int);
template cudaError_t hla::ws::ws_launch_flags<true, false>(const hla::FwdArgs &, cudaStream_t, int);
