// hla_fwd_tc.cu -- host entry of the tensor-core forward: support check,
// workspace size, and dispatch to the (decay, normalise, variant) launchers
// compiled in hla_fwd_tc_f0..f11.cu.  The masked variant at d = 64 runs the
// warp-specialised kernels: without decay on 128-token tiles (hla_fwd_ws2.cuh), with
// decay on the caller's chunk (hla_fwd_ws.cuh); every other shape and variant runs the
// kernel of hla_fwd_tc.cuh.
#include "hla_fwd_ws2.cuh"

namespace hla {
namespace tc {
extern template cudaError_t launch_flags<false, false, 0>(const FwdArgs &, cudaStream_t, int);
extern template cudaError_t launch_flags<false, false, 1>(const FwdArgs &, cudaStream_t, int);
extern template cudaError_t launch_flags<false, false, 2>(const FwdArgs &, cudaStream_t, int);
extern template cudaError_t launch_flags<false, true, 0>(const FwdArgs &, cudaStream_t, int);
extern template cudaError_t launch_flags<false, true, 1>(const FwdArgs &, cudaStream_t, int);
extern template cudaError_t launch_flags<false, true, 2>(const FwdArgs &, cudaStream_t, int);
extern template cudaError_t launch_flags<true, false, 0>(const FwdArgs &, cudaStream_t, int);
extern template cudaError_t launch_flags<true, false, 1>(const FwdArgs &, cudaStream_t, int);
extern template cudaError_t launch_flags<true, false, 2>(const FwdArgs &, cudaStream_t, int);
extern template cudaError_t launch_flags<true, true, 0>(const FwdArgs &, cudaStream_t, int);
extern template cudaError_t launch_flags<true, true, 1>(const FwdArgs &, cudaStream_t, int);
extern template cudaError_t launch_flags<true, true, 2>(const FwdArgs &, cudaStream_t, int);
}  // namespace tc
namespace ws {
extern template cudaError_t ws_launch_flags<false, false>(const FwdArgs &, cudaStream_t, int);
extern template cudaError_t ws_launch_flags<false, true>(const FwdArgs &, cudaStream_t, int);
extern template cudaError_t ws_launch_flags<true, false>(const FwdArgs &, cudaStream_t, int);
extern template cudaError_t ws_launch_flags<true, true>(const FwdArgs &, cudaStream_t, int);
}  // namespace ws
namespace ws2 {
extern template cudaError_t launch_flags<false>(const FwdArgs &, cudaStream_t, int);
extern template cudaError_t launch_flags<true>(const FwdArgs &, cudaStream_t, int);
}  // namespace ws2

bool fwd_tc_supported(const hla_params &p) {
    auto ok = [](int x) { return x == 64 || x == 128; };
    if ((p.flags & HLA_ASYMMETRIC) && p.dv > p.d) return false;  // its spare accumulator is d wide
    return p.in_dtype == HLA_BF16 && ok(p.d) && ok(p.dv) && ok(p.chunk);
}

size_t fwd_tc_workspace(const hla_params &p, int num_sms) {
    if (p.n == 0) return 0;
    if (ws2::ws2_supported(p)) return ws2::work_layout(p, ws2::work_plan(p, num_sms)).total;
    if (ws::ws_supported(p)) return ws::work_layout(p, ws::work_plan(p, num_sms)).total;
    return tc::ws_layout(p, tc::make_plan(p, num_sms)).total;
}

const char *fwd_tc_kernel_name(const hla_params &p) {
    if (ws2::ws2_supported(p)) return "fwd_ws2_kernel";
    if (ws::ws_supported(p)) return "fwd_ws_kernel";
    return "fwd_tc_kernel";
}

size_t fwd_tc_sync_bytes(const hla_params &p, int num_sms) {
    if (p.n == 0) return 0;
    if (ws2::ws2_supported(p)) return ws2::work_layout(p, ws2::work_plan(p, num_sms)).off_summ;
    if (ws::ws_supported(p)) return ws::work_layout(p, ws::work_plan(p, num_sms)).off_summ;
    return tc::ws_layout(p, tc::make_plan(p, num_sms)).off_summ;
}

cudaError_t fwd_tc_launch(const FwdArgs &a, cudaStream_t st, int num_sms) {
    const hla_params p{a.B, a.H, a.n, a.d, a.dv, a.chunk, a.in_dtype, a.flags, a.eps, a.gamma};
    if (ws2::ws2_supported(p))
        return (a.flags & HLA_NORMALIZE) ? ws2::launch_flags<true>(a, st, num_sms) : ws2::launch_flags<false>(a, st, num_sms);
    if (ws::ws_supported(p)) {
        const int wkey = ((a.flags & HLA_DECAY) ? 2 : 0) + ((a.flags & HLA_NORMALIZE) ? 1 : 0);
        switch (wkey) {
            case 0: return ws::ws_launch_flags<false, false>(a, st, num_sms);
            case 1: return ws::ws_launch_flags<false, true>(a, st, num_sms);
            case 2: return ws::ws_launch_flags<true, false>(a, st, num_sms);
            default: return ws::ws_launch_flags<true, true>(a, st, num_sms);
        }
    }
    const int var = (a.flags & HLA_UNMASKED) ? 1 : ((a.flags & HLA_ASYMMETRIC) ? 2 : 0);
    const int key = ((a.flags & HLA_DECAY) ? 6 : 0) + ((a.flags & HLA_NORMALIZE) ? 3 : 0) + var;
    switch (key) {
        case 0: return tc::launch_flags<false, false, 0>(a, st, num_sms);
        case 1: return tc::launch_flags<false, false, 1>(a, st, num_sms);
        case 2: return tc::launch_flags<false, false, 2>(a, st, num_sms);
        case 3: return tc::launch_flags<false, true, 0>(a, st, num_sms);
        case 4: return tc::launch_flags<false, true, 1>(a, st, num_sms);
        case 5: return tc::launch_flags<false, true, 2>(a, st, num_sms);
        case 6: return tc::launch_flags<true, false, 0>(a, st, num_sms);
        case 7: return tc::launch_flags<true, false, 1>(a, st, num_sms);
        case 8: return tc::launch_flags<true, false, 2>(a, st, num_sms);
        case 9: return tc::launch_flags<true, true, 0>(a, st, num_sms);
        case 10: return tc::launch_flags<true, true, 1>(a, st, num_sms);
        default: return tc::launch_flags<true, true, 2>(a, st, num_sms);
    }
}

}  // namespace hla
