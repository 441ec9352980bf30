// Backward kernels for bf16 inputs and chunk length 32.
#include "hla_bwd_simt.cuh"

namespace hla {
namespace bwd {
template cudaError_t launch_d<__nv_bfloat16, 32>(const BwdArgs &, cudaStream_t);
}  // namespace bwd
}  // namespace hla
