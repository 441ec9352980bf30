// Third-order forward kernels for f32 inputs and chunk length 16.
#include "hla_fwd3_simt.cuh"

namespace hla {
namespace fwd3 {
template cudaError_t launch_d<float, 16>(const Fwd3Args &, cudaStream_t);
}  // namespace fwd3
}  // namespace hla
