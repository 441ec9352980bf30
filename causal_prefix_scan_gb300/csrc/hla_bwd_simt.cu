// hla_bwd_simt.cu -- shape checks, workspace size and dispatch of the backward
// kernels in hla_bwd_simt.cuh (instantiated per element type and chunk length in
// hla_bwd_<type>_c<chunk>.cu).
#include "hla_bwd_simt.cuh"

namespace hla {
namespace bwd {
#define HLA_BWD_EXTERN(T, C) extern template cudaError_t launch_d<T, C>(const BwdArgs &, cudaStream_t);
HLA_BWD_EXTERN(float, 16)
HLA_BWD_EXTERN(float, 32)
HLA_BWD_EXTERN(float, 64)
HLA_BWD_EXTERN(__nv_bfloat16, 16)
HLA_BWD_EXTERN(__nv_bfloat16, 32)
HLA_BWD_EXTERN(__nv_bfloat16, 64)
#undef HLA_BWD_EXTERN

namespace {
template <typename T>
cudaError_t launch_c(const BwdArgs &a, cudaStream_t st) {
    switch (a.chunk) {
        case 16: return launch_d<T, 16>(a, st);
        case 32: return launch_d<T, 32>(a, st);
        case 64: return launch_d<T, 64>(a, st);
    }
    return cudaErrorInvalidValue;
}
}  // namespace
}  // namespace bwd

bool bwd_simt_supported(const hla_params &p) {
    auto ok = [](int x) { return x == 16 || x == 32 || x == 64; };
    const int hkv = p.Hkv > 0 ? p.Hkv : p.H;
    const bool shape = (ok(p.d) && ok(p.dv) && ok(p.chunk)) || (p.d == 128 && p.chunk == 16 && (p.dv == 16 || p.dv == 32));
    return shape && p.H % hkv == 0 && !(p.flags & (HLA_UNMASKED | HLA_ASYMMETRIC));
}

// Local sums and chunk states, then (shared key/value heads only) the per-query-head
// dk, dv before their group sum.
size_t bwd_pair_offset(const hla_params &p) {
    const size_t nch = ((size_t)p.n + p.chunk - 1) / p.chunk;
    const bwd::BwdWs w{p.d, p.dv};
    return (size_t)p.B * p.H * nch * (w.loc_floats() + w.st_floats());
}

// ... then the adjoints at the first token of every pair (Lam, Om), for the gradient of
// a given initial state.
size_t bwd_adj0_offset(const hla_params &p) {
    const int hkv = p.Hkv > 0 ? p.Hkv : p.H;
    const size_t pair = hkv < p.H ? (size_t)p.B * p.H * p.n * ((size_t)p.d + p.dv) : 0;
    return bwd_pair_offset(p) + pair;
}

size_t bwd_simt_workspace(const hla_params &p) {
    const size_t adj = (size_t)p.B * p.H * ((size_t)p.d * p.dv + (size_t)p.d * p.d);
    return (bwd_adj0_offset(p) + adj) * sizeof(float);
}

cudaError_t bwd_simt_launch(const BwdArgs &a, cudaStream_t st) {
    if (a.n == 0) return cudaSuccess;
    return a.in_dtype == HLA_F32 ? bwd::launch_c<float>(a, st) : bwd::launch_c<__nv_bfloat16>(a, st);
}

}  // namespace hla
