// hla_fwd_tc.cu -- host entry of the tensor-core forward: support check,
// workspace size, and dispatch to the (decay, normalise, unmasked) launchers
// compiled in hla_fwd_tc_f0..f7.cu.
#include "hla_fwd_tc.cuh"

namespace hla {
namespace tc {
extern template cudaError_t launch_flags<false, false, false>(const FwdArgs &, cudaStream_t, int);
extern template cudaError_t launch_flags<false, false, true>(const FwdArgs &, cudaStream_t, int);
extern template cudaError_t launch_flags<false, true, false>(const FwdArgs &, cudaStream_t, int);
extern template cudaError_t launch_flags<false, true, true>(const FwdArgs &, cudaStream_t, int);
extern template cudaError_t launch_flags<true, false, false>(const FwdArgs &, cudaStream_t, int);
extern template cudaError_t launch_flags<true, false, true>(const FwdArgs &, cudaStream_t, int);
extern template cudaError_t launch_flags<true, true, false>(const FwdArgs &, cudaStream_t, int);
extern template cudaError_t launch_flags<true, true, true>(const FwdArgs &, cudaStream_t, int);
}  // namespace tc

bool fwd_tc_supported(const hla_params &p) {
    auto ok = [](int x) { return x == 64 || x == 128; };
    if (p.flags & HLA_ASYMMETRIC) return false;  // the asymmetric variant runs on the CUDA-core path
    return p.in_dtype == HLA_BF16 && ok(p.d) && ok(p.dv) && ok(p.chunk);
}

size_t fwd_tc_workspace(const hla_params &p, int num_sms) {
    if (p.n == 0) return 0;
    return tc::ws_layout(p, tc::make_plan(p, num_sms)).total;
}

cudaError_t fwd_tc_launch(const FwdArgs &a, cudaStream_t st, int num_sms) {
    const int key = ((a.flags & HLA_DECAY) ? 4 : 0) | ((a.flags & HLA_NORMALIZE) ? 2 : 0) |
                    ((a.flags & HLA_UNMASKED) ? 1 : 0);
    switch (key) {
        case 0: return tc::launch_flags<false, false, false>(a, st, num_sms);
        case 1: return tc::launch_flags<false, false, true>(a, st, num_sms);
        case 2: return tc::launch_flags<false, true, false>(a, st, num_sms);
        case 3: return tc::launch_flags<false, true, true>(a, st, num_sms);
        case 4: return tc::launch_flags<true, false, false>(a, st, num_sms);
        case 5: return tc::launch_flags<true, false, true>(a, st, num_sms);
        case 6: return tc::launch_flags<true, true, false>(a, st, num_sms);
        default: return tc::launch_flags<true, true, true>(a, st, num_sms);
    }
}

}  // namespace hla
