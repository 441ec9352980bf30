// Third-order forward kernels for f32 inputs and chunk length 64.
#include "hla_fwd3_simt.cuh"

namespace hla {
namespace fwd3 {
template cudaError_t launch_d<float, 64>(const Fwd3Args &, cudaStream_t);
}  // namespace fwd3
}  // namespace hla
