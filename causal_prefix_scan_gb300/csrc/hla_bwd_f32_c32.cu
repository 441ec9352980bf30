// Backward kernels for f32 inputs and chunk length 32.
#include "hla_bwd_simt.cuh"

namespace hla {
namespace bwd {
template cudaError_t launch_d<float, 32>(const BwdArgs &, cudaStream_t);
}  // namespace bwd
}  // namespace hla
