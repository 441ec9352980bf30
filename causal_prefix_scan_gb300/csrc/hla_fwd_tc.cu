// hla_fwd_tc.cu -- host entry of the tensor-core forward: support check,
// workspace size, and dispatch to the (decay, normalise) launchers compiled in
// hla_fwd_tc_f0..f3.cu.
#include "hla_fwd_tc.cuh"

namespace hla {
namespace tc {
extern template cudaError_t launch_flags<false, false>(const FwdArgs &, cudaStream_t, int);
extern template cudaError_t launch_flags<false, true>(const FwdArgs &, cudaStream_t, int);
extern template cudaError_t launch_flags<true, false>(const FwdArgs &, cudaStream_t, int);
extern template cudaError_t launch_flags<true, true>(const FwdArgs &, cudaStream_t, int);
}  // namespace tc

bool fwd_tc_supported(const hla_params &p) {
    auto ok = [](int x) { return x == 64 || x == 128; };
    return p.in_dtype == HLA_BF16 && ok(p.d) && ok(p.dv) && ok(p.chunk);
}

size_t fwd_tc_workspace(const hla_params &p, int num_sms) {
    if (p.n == 0) return 0;
    return tc::ws_layout(p, tc::make_plan(p, num_sms)).total;
}

cudaError_t fwd_tc_launch(const FwdArgs &a, cudaStream_t st, int num_sms) {
    const bool decay = (a.flags & HLA_DECAY) != 0, norm = (a.flags & HLA_NORMALIZE) != 0;
    if (decay)
        return norm ? tc::launch_flags<true, true>(a, st, num_sms) : tc::launch_flags<true, false>(a, st, num_sms);
    return norm ? tc::launch_flags<false, true>(a, st, num_sms) : tc::launch_flags<false, false>(a, st, num_sms);
}

}  // namespace hla
