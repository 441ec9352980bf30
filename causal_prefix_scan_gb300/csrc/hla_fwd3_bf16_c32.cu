// Third-order forward kernels for bf16 inputs and chunk length 32.
#include "hla_fwd3_simt.cuh"

namespace hla {
namespace fwd3 {
template cudaError_t launch_d<__nv_bfloat16, 32>(const Fwd3Args &, cudaStream_t);
}  // namespace fwd3
}  // namespace hla
