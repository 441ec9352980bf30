// hla_api.cu -- the C ABI declared in hla.h: argument validation, workspace
// sizing, the sticky device status word, and dispatch to the kernels.
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>

#include "hla_internal.h"

namespace {

thread_local char g_msg[512] = "";

// Sticky device status word (DEV_OK / DEV_TIMEOUT), one per device.
__device__ unsigned g_dev_status = 0u;

hla_status fail(hla_status s, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
hla_status fail(hla_status s, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof g_msg, fmt, ap);
    va_end(ap);
    return s;
}

hla_status cuda_fail(cudaError_t e, const char *where) {
    return fail(HLA_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool width_ok(int x) { return x == 16 || x == 32 || x == 64 || x == 128; }

// Device address of the status word for the current device.
cudaError_t status_ptr(unsigned **p) {
    void *a = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&a, g_dev_status);
    *p = static_cast<unsigned *>(a);
    return e;
}

int num_sms_current() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) return 1;
    return n;
}

hla_status check_state(const hla_state *s, const char *name) {
    if (!s) return HLA_OK;
    if (!s->S || !s->C || !s->m || !s->G || !s->h) return fail(HLA_ERR_ARG, "%s: all five pointers must be set", name);
    if (!aligned16(s->S) || !aligned16(s->C) || !aligned16(s->m) || !aligned16(s->G) || !aligned16(s->h))
        return fail(HLA_ERR_ARG, "%s: pointers must be 16-byte aligned", name);
    return HLA_OK;
}

// The unmasked and asymmetric variants at dv = 128 with d <= 64 where no kernel takes the
// shape whole (the tensor-core AHLA needs dv <= d, the tensor cores d >= 64 and bf16, the
// CUDA-core kernel of these variants dv <= 64): two problems over the value columns
// [0,64) and [64,128).  The output's column j and the state's C, G columns j (C, and P, E
// of AHLA) depend on column j of v only; S, m, h (R, m^K, n of AHLA) on none.
hla_params fwd_half(const hla_params &p) {
    hla_params q = p;
    q.dv = 64;
    return q;
}
bool fwd_value_split(const hla_params &p) {
    if (!(p.flags & (HLA_ASYMMETRIC | HLA_UNMASKED)) || p.dv != 128 || p.d > 64) return false;
    if (hla::fwd_tc_supported(p) || hla::fwd_simt_supported(p)) return false;
    const hla_params h = fwd_half(p);
    return hla::fwd_tc_supported(h) || hla::fwd_simt_supported(h);
}

hla_status check_params(const hla_params *p) {
    if (!p) return fail(HLA_ERR_ARG, "params is NULL");
    if (p->B < 1 || p->H < 1 || p->n < 0) return fail(HLA_ERR_ARG, "need B >= 1, H >= 1, n >= 0");
    if (p->d < 1 || p->dv < 1 || p->chunk < 1) return fail(HLA_ERR_ARG, "need d, dv, chunk >= 1");
    if (p->in_dtype != HLA_F32 && p->in_dtype != HLA_BF16) return fail(HLA_ERR_ARG, "unknown in_dtype");
    if (p->flags & ~(unsigned)(HLA_NORMALIZE | HLA_DECAY | HLA_UNMASKED | HLA_ASYMMETRIC))
        return fail(HLA_ERR_ARG, "unknown flag bits");
    if ((p->flags & HLA_UNMASKED) && (p->flags & HLA_ASYMMETRIC))
        return fail(HLA_ERR_ARG, "HLA_UNMASKED and HLA_ASYMMETRIC exclude each other");
    if ((p->flags & HLA_DECAY) && !p->gamma) return fail(HLA_ERR_ARG, "HLA_DECAY needs gamma");
    if (p->Hkv < 0 || (p->Hkv > 0 && p->H % p->Hkv != 0))
        return fail(HLA_ERR_ARG, "Hkv must divide H (0 means Hkv = H)");
    if ((p->flags & HLA_NORMALIZE) && !(p->eps >= 0.f)) return fail(HLA_ERR_ARG, "eps must be >= 0");
    if ((long long)p->B * p->H * (long long)p->n * (p->d > p->dv ? p->d : p->dv) > (1LL << 40))
        return fail(HLA_ERR_ARG, "problem too large");
    if (fwd_value_split(*p)) return HLA_OK;
    if (!hla::fwd_tc_supported(*p) && !hla::fwd_simt_supported(*p))
        return fail(HLA_ERR_UNSUPPORTED, "unsupported shape: dtype=%d d=%d dv=%d chunk=%d", (int)p->in_dtype, p->d,
                    p->dv, p->chunk);
    if (p->in_dtype == HLA_F32 && !hla::fwd_simt_supported(*p))
        return fail(HLA_ERR_UNSUPPORTED, "fp32 inputs need d, dv, chunk in {16,32,64,128} (d, dv <= 64 for the unmasked and asymmetric variants)");
    return HLA_OK;
}

// One CTA waits, with the bounded barrier wait of the kernels (short poll limit), on a
// barrier whose phase nothing completes: the wait expires and raises the status word.
__global__ void expired_wait_kernel(unsigned *err) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        hla::mbar_init(&bar, 1);
        hla::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) hla::mbar_wait(&bar, 0u, err, 1u << 14);
}

}  // namespace

namespace hla {
// Record `msg` as this thread's last error and return `s` (used by entry points
// defined in other translation units).
hla_status report(hla_status s, const char *msg) { return fail(s, "%s", msg); }
}  // namespace hla

extern "C" {

const char *hla_status_string(hla_status s) {
    switch (s) {
        case HLA_OK: return "ok";
        case HLA_ERR_ARG: return "invalid argument";
        case HLA_ERR_UNSUPPORTED: return "unsupported configuration";
        case HLA_ERR_CUDA: return "CUDA error";
        case HLA_ERR_TIMEOUT: return "device wait timed out";
    }
    return "unknown status";
}

const char *hla_last_error(void) { return g_msg; }

}  // extern "C"

namespace {
size_t fwd_align256(size_t x) { return (x + 255) & ~size_t(255); }
// The forward split over value halves: the half problem's workspace, the gathered value half,
// the output half (input type), and the C, G halves (fp32) of state_in and state_out.
struct FwdSplit {
    size_t vh, oh, sin, sout, total;
};
FwdSplit fwd_split_layout(const hla_params &p, int nsm) {
    const hla_params h = fwd_half(p);
    const size_t el = p.in_dtype == HLA_F32 ? 4 : 2, hkv = p.Hkv > 0 ? p.Hkv : p.H;
    const size_t rq = (size_t)p.B * p.H * p.n, rkv = (size_t)p.B * hkv * p.n;
    const size_t half_cg = (size_t)p.B * p.H * p.d * 64 * 4;  // one half of C or G
    FwdSplit L;
    size_t o = fwd_align256(hla::fwd_tc_supported(h) && p.n > 0 ? hla::fwd_tc_workspace(h, nsm) : 0);
    L.vh = o; o = fwd_align256(o + rkv * 64 * el);
    L.oh = o; o = fwd_align256(o + rq * 64 * el);
    L.sin = o; o = fwd_align256(o + 2 * half_cg);
    L.sout = o; o = fwd_align256(o + 2 * half_cg);
    L.total = o;
    return L;
}
}  // namespace

extern "C" {

size_t hla_forward_workspace_size(const hla_params *p) {
    if (check_params(p) != HLA_OK) return 0;
    if (fwd_value_split(*p)) return p->n > 0 ? fwd_split_layout(*p, num_sms_current()).total : 0;
    if (hla::fwd_tc_supported(*p)) return hla::fwd_tc_workspace(*p, num_sms_current());
    return 0;
}

const char *hla_forward_kernel(const hla_params *p) {
    if (check_params(p) != HLA_OK || p->n == 0) return nullptr;
    if (fwd_value_split(*p)) {  // the kernel of each value half
        const hla_params h = fwd_half(*p);
        return hla::fwd_tc_supported(h) ? hla::fwd_tc_kernel_name(h) : "fwd_simt_kernel";
    }
    return hla::fwd_tc_supported(*p) ? hla::fwd_tc_kernel_name(*p) : "fwd_simt_kernel";
}

hla_status hla_forward_chunked(const hla_params *p, const void *q, const void *k, const void *v, void *o,
                               const hla_state *state_in, const hla_state *state_out, void *workspace,
                               size_t workspace_bytes, void *stream) {
    hla_status s = check_params(p);
    if (s != HLA_OK) return s;
    if ((s = check_state(state_in, "state_in")) != HLA_OK) return s;
    if ((s = check_state(state_out, "state_out")) != HLA_OK) return s;
    if (state_in && state_out &&
        (state_in->S == state_out->S || state_in->C == state_out->C || state_in->G == state_out->G))
        return fail(HLA_ERR_ARG, "state_out may not alias state_in");
    if (p->n > 0) {
        if (!q || !k || !v || !o) return fail(HLA_ERR_ARG, "q, k, v, o must be set when n > 0");
        if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
            return fail(HLA_ERR_ARG, "q, k, v, o must be 16-byte aligned");
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool tc = hla::fwd_tc_supported(*p);
    const int nsm = num_sms_current();
    if (tc && p->n > 0 && !fwd_value_split(*p)) {
        const size_t need = hla::fwd_tc_workspace(*p, nsm);
        if (!workspace || workspace_bytes < need)
            return fail(HLA_ERR_ARG, "workspace too small: need %zu bytes, got %zu", need, workspace_bytes);
        if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
            return fail(HLA_ERR_ARG, "workspace must be 256-byte aligned");
    }
    if (p->n == 0) {  // no tokens: state_out = state_in (or zeros); unmasked: G, h zero
        if (!state_out) return HLA_OK;
        const size_t BH = (size_t)p->B * p->H, D = p->d, DV = p->dv;
        const size_t sz[5] = {BH * D * D * 4, BH * D * DV * 4, BH * D * 4, BH * D * DV * 4, BH * D * 4};
        float *dst[5] = {state_out->S, state_out->C, state_out->m, state_out->G, state_out->h};
        const bool unmasked = (p->flags & HLA_UNMASKED) != 0;
        for (int i = 0; i < 5; ++i) {
            cudaError_t e;
            if (state_in && !(unmasked && i >= 3)) {
                const float *src[5] = {state_in->S, state_in->C, state_in->m, state_in->G, state_in->h};
                e = cudaMemcpyAsync(dst[i], src[i], sz[i], cudaMemcpyDeviceToDevice, st);
            } else {
                e = cudaMemsetAsync(dst[i], 0, sz[i], st);
            }
            if (e != cudaSuccess) return cuda_fail(e, "state copy");
        }
        return HLA_OK;
    }
    if (fwd_value_split(*p)) {  // two 64-column halves of the values, each written into its columns
        const FwdSplit L = fwd_split_layout(*p, nsm);
        if (!workspace || workspace_bytes < L.total)
            return fail(HLA_ERR_ARG, "workspace too small: need %zu bytes, got %zu", L.total, workspace_bytes);
        if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
            return fail(HLA_ERR_ARG, "workspace must be 256-byte aligned");
        const hla_params h = fwd_half(*p);
        uint8_t *w = static_cast<uint8_t *>(workspace);
        const size_t hkv = p->Hkv > 0 ? p->Hkv : p->H;
        const size_t rq = (size_t)p->B * p->H * p->n, rkv = (size_t)p->B * hkv * p->n;
        const size_t srows = (size_t)p->B * p->H * p->d, hs = srows * 64;
        float *ci = reinterpret_cast<float *>(w + L.sin), *co = reinterpret_cast<float *>(w + L.sout);
        cudaError_t e = cudaSuccess;
        for (int half = 0; half < 2 && e == cudaSuccess; ++half) {
            if ((e = hla::cols_part_copy(v, w + L.vh, rkv, p->in_dtype, 128, 64, half, true, st)) != cudaSuccess) break;
            hla_state si{}, so{};
            if (state_in) {
                si = *state_in;
                si.C = ci;
                si.G = ci + hs;
                if ((e = hla::cols_part_copy(state_in->C, si.C, srows, HLA_F32, 128, 64, half, true, st)) != cudaSuccess ||
                    (e = hla::cols_part_copy(state_in->G, si.G, srows, HLA_F32, 128, 64, half, true, st)) != cudaSuccess)
                    break;
            }
            if (state_out) {  // S, m, h come out the same from both halves
                so = *state_out;
                so.C = co;
                so.G = co + hs;
            }
            s = hla_forward_chunked(&h, q, k, w + L.vh, w + L.oh, state_in ? &si : nullptr,
                                    state_out ? &so : nullptr, w, L.vh, stream);
            if (s != HLA_OK) return s;
            if ((e = hla::cols_part_copy(w + L.oh, o, rq, p->in_dtype, 128, 64, half, false, st)) != cudaSuccess) break;
            if (state_out &&
                ((e = hla::cols_part_copy(so.C, state_out->C, srows, HLA_F32, 128, 64, half, false, st)) != cudaSuccess ||
                 (e = hla::cols_part_copy(so.G, state_out->G, srows, HLA_F32, 128, 64, half, false, st)) != cudaSuccess))
                break;
        }
        if (e != cudaSuccess) return cuda_fail(e, "forward over value halves");
        return HLA_OK;
    }
    hla::FwdArgs a;
    a.B = p->B; a.H = p->H; a.n = p->n; a.d = p->d; a.dv = p->dv; a.chunk = p->chunk;
    a.Hkv = p->Hkv > 0 ? p->Hkv : p->H;
    a.in_dtype = p->in_dtype; a.flags = p->flags; a.eps = p->eps; a.gamma = p->gamma;
    a.q = q; a.k = k; a.v = v; a.o = o;
    a.sin = hla::to_ptrs(state_in);
    a.sout = hla::to_ptrs(state_out);
    a.workspace = workspace;
    a.ws_bytes = workspace_bytes;
    cudaError_t e = status_ptr(&a.err);
    if (e != cudaSuccess) return cuda_fail(e, "status word");
    e = tc ? hla::fwd_tc_launch(a, st, nsm) : hla::fwd_simt_launch(a, st);
    if (e != cudaSuccess) return cuda_fail(e, "forward launch");
    return HLA_OK;
}

namespace {
// The shape the backward kernels run: a chunk of 128 tokens as two of 64 (the chunk
// length changes only the rounding), and dv = 128 as two 64-column halves of the values
// (hla_bwd_split.cu).  d = 128 runs in chunks of 16 tokens over slices of at most 32
// value columns: the CUDA-core gradient kernel holds its two d x d and two d x dv fp32
// states and the chunk's tiles in shared memory only at that size.
hla_params bwd_inner(const hla_params &p) {
    hla_params q = p;
    if (q.d == 128) {
        q.chunk = 16;
        if (q.dv > 32) q.dv = 32;
        return q;
    }
    if (q.chunk == 128) q.chunk = 64;
    if (q.dv == 128) q.dv = 64;
    return q;
}
// Value-column slices of the call (1: no split).
int bwd_slices(const hla_params &p) { return p.dv / bwd_inner(p).dv; }
bool bwd_split(const hla_params &p) { return bwd_slices(p) > 1; }

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Scratch of the unsplit problem: the kernels' workspace.
size_t bwd_inner_workspace(const hla_params &q) {
    if (q.flags & HLA_NORMALIZE) {
        if (q.n == 0) return 0;
        const size_t a = hla::bwd_norm_layout(q).total, b = hla::bwd_norm_tc_workspace(q);
        return a > b ? a : b;
    }
    return hla::bwd_simt_workspace(q);
}

// Split over value columns: the slice problem's workspace, then the gathered value and
// upstream slices, the slice's dq, dk, dv (input type) and the fp32 sums of dq and dk
// (byte offsets).
struct SplitLayout {
    size_t inner, vh, gh, dqh, dkh, dvh, acc_q, acc_k, total;
};
SplitLayout split_layout(const hla_params &p) {
    const hla_params q = bwd_inner(p);
    const size_t el = p.in_dtype == HLA_F32 ? 4 : 2, hkv = p.Hkv > 0 ? p.Hkv : p.H, w = q.dv;
    const size_t rq = (size_t)p.B * p.H * p.n, rkv = (size_t)p.B * hkv * p.n;
    SplitLayout L;
    size_t o = align256(bwd_inner_workspace(q));
    L.inner = 0;
    L.vh = o; o = align256(o + rkv * w * el);
    L.gh = o; o = align256(o + rq * w * el);
    L.dqh = o; o = align256(o + rq * p.d * el);
    L.dkh = o; o = align256(o + rkv * p.d * el);
    L.dvh = o; o = align256(o + rkv * w * el);
    L.acc_q = o; o = align256(o + rq * p.d * 4);
    L.acc_k = o; o = align256(o + rkv * p.d * 4);
    L.total = o;
    return L;
}

hla_status check_bwd_params(const hla_params *p) {
    if (!p) return fail(HLA_ERR_ARG, "params is NULL");
    if (p->B < 1 || p->H < 1 || p->n < 0) return fail(HLA_ERR_ARG, "need B >= 1, H >= 1, n >= 0");
    if (p->in_dtype != HLA_F32 && p->in_dtype != HLA_BF16) return fail(HLA_ERR_ARG, "unknown in_dtype");
    if (p->flags & ~(unsigned)(HLA_NORMALIZE | HLA_DECAY | HLA_UNMASKED | HLA_ASYMMETRIC))
        return fail(HLA_ERR_ARG, "unknown flag bits");
    if ((p->flags & HLA_DECAY) && !p->gamma) return fail(HLA_ERR_ARG, "HLA_DECAY needs gamma");
    if ((p->flags & HLA_NORMALIZE) && !(p->eps >= 0.f)) return fail(HLA_ERR_ARG, "eps must be >= 0");
    if (p->Hkv < 0 || (p->Hkv > 0 && p->H % p->Hkv != 0))
        return fail(HLA_ERR_ARG, "Hkv must divide H (0 means Hkv = H)");
    if ((long long)p->B * p->H * (long long)p->n * (p->d > p->dv ? p->d : p->dv) > (1LL << 40))
        return fail(HLA_ERR_ARG, "problem too large");
    const bool dv_ok = p->dv == 16 || p->dv == 32 || p->dv == 64 || p->dv == 128;
    const bool c_ok = p->chunk == 16 || p->chunk == 32 || p->chunk == 64 || p->chunk == 128;
    if (!dv_ok || !c_ok || !hla::bwd_simt_supported(bwd_inner(*p)))
        return fail(HLA_ERR_UNSUPPORTED,
                    "backward supports flags 0, HLA_DECAY, HLA_NORMALIZE, d in {16,32,64,128}, dv and chunk in "
                    "{16,32,64,128} (got flags=%u Hkv=%d d=%d dv=%d chunk=%d)",
                    p->flags, p->Hkv, p->d, p->dv, p->chunk);
    return HLA_OK;
}
}  // namespace

size_t hla_backward_workspace_size(const hla_params *p) {
    if (check_bwd_params(p) != HLA_OK) return 0;
    if (bwd_split(*p)) return p->n > 0 ? split_layout(*p).total : 0;
    return bwd_inner_workspace(bwd_inner(*p));
}

namespace {
hla_status backward_impl(const hla_params *p, const void *q, const void *k, const void *v, const void *dout,
                         const hla_state *state_in, void *dq, void *dk, void *dv, const hla_state *d_state_in,
                         void *workspace, size_t workspace_bytes, void *stream, void *const *phase_events) {
    hla_status s = check_bwd_params(p);
    if (s != HLA_OK) return s;
    const bool norm = (p->flags & HLA_NORMALIZE) != 0;
    if ((s = check_state(state_in, "state_in")) != HLA_OK) return s;
    if ((s = check_state(d_state_in, "d_state_in")) != HLA_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t BH = (size_t)p->B * p->H, D = p->d, DV = p->dv;
    if (d_state_in && !norm) {  // m and h enter only the denominator: their gradient is zero here
        const size_t sz[2] = {BH * D * 4, BH * D * 4};
        float *dst[2] = {d_state_in->m, d_state_in->h};
        for (int i = 0; i < 2; ++i) {
            cudaError_t e = cudaMemsetAsync(dst[i], 0, sz[i], st);
            if (e != cudaSuccess) return cuda_fail(e, "state gradient clear");
        }
    }
    if (p->n == 0) {  // no tokens: the state gradient is zero
        if (d_state_in) {
            const size_t sz[5] = {BH * D * D * 4, BH * D * DV * 4, BH * D * DV * 4, BH * D * 4, BH * D * 4};
            float *dst[5] = {d_state_in->S, d_state_in->C, d_state_in->G, d_state_in->m, d_state_in->h};
            for (int i = 0; i < 5; ++i) {
                cudaError_t e = cudaMemsetAsync(dst[i], 0, sz[i], st);
                if (e != cudaSuccess) return cuda_fail(e, "state gradient clear");
            }
        }
        return HLA_OK;
    }
    if (!q || !k || !v || !dout || !dq || !dk || !dv)
        return fail(HLA_ERR_ARG, "q, k, v, dout, dq, dk, dv must be set when n > 0");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dout) || !aligned16(dq) || !aligned16(dk) ||
        !aligned16(dv))
        return fail(HLA_ERR_ARG, "tensor pointers must be 16-byte aligned");
    const size_t need = hla_backward_workspace_size(p);
    if (!workspace || workspace_bytes < need)
        return fail(HLA_ERR_ARG, "workspace too small: need %zu bytes, got %zu", need, workspace_bytes);
    const bool split = bwd_split(*p);
    if ((norm || split) ? (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 : !aligned16(workspace))
        return fail(HLA_ERR_ARG, "workspace must be 256-byte aligned with HLA_NORMALIZE or a split over value "
                                 "columns (dv = 128; d = 128 with dv > 32), else 16-byte aligned");
    if (phase_events) {
        for (int i = 0; i < 4; ++i)
            if (!phase_events[i]) return fail(HLA_ERR_ARG, "phase_events must hold four events");
    }
    if (split) {  // slices of the value columns: dq, dk add up, dv side by side
        if (state_in || d_state_in)
            return fail(HLA_ERR_UNSUPPORTED, "a backward split over value columns (dv = 128; d = 128 with dv > 32) "
                                             "from a given state or with its gradient is not supported");
        const hla_params in = bwd_inner(*p);
        const SplitLayout L = split_layout(*p);
        uint8_t *w = static_cast<uint8_t *>(workspace);
        const size_t hkv = p->Hkv > 0 ? p->Hkv : p->H;
        const size_t rq = (size_t)p->B * p->H * p->n, rkv = (size_t)p->B * hkv * p->n;
        auto ev = [&](int i) {
            return phase_events ? cudaEventRecord(static_cast<cudaEvent_t>(phase_events[i]), st) : cudaSuccess;
        };
        const int parts = bwd_slices(*p), pw = in.dv;
        cudaError_t e = ev(0);
        for (int h = 0; h < parts && e == cudaSuccess; ++h) {
            if ((e = hla::cols_part_copy(v, w + L.vh, rkv, p->in_dtype, p->dv, pw, h, true, st)) != cudaSuccess) break;
            if ((e = hla::cols_part_copy(dout, w + L.gh, rq, p->in_dtype, p->dv, pw, h, true, st)) != cudaSuccess)
                break;
            s = backward_impl(&in, q, k, w + L.vh, w + L.gh, nullptr, w + L.dqh, w + L.dkh, w + L.dvh, nullptr,
                              w + L.inner, L.vh, stream, nullptr);
            if (s != HLA_OK) return s;
            if ((e = hla::acc_add(reinterpret_cast<float *>(w + L.acc_q), w + L.dqh, rq * p->d, p->in_dtype, h == 0,
                                  st)) != cudaSuccess ||
                (e = hla::acc_add(reinterpret_cast<float *>(w + L.acc_k), w + L.dkh, rkv * p->d, p->in_dtype, h == 0,
                                  st)) != cudaSuccess)
                break;
            e = hla::cols_part_copy(w + L.dvh, dv, rkv, p->in_dtype, p->dv, pw, h, false, st);
        }
        if (e == cudaSuccess) e = hla::acc_store(dq, reinterpret_cast<const float *>(w + L.acc_q), rq * p->d,
                                                 p->in_dtype, st);
        if (e == cudaSuccess) e = hla::acc_store(dk, reinterpret_cast<const float *>(w + L.acc_k), rkv * p->d,
                                                 p->in_dtype, st);
        for (int i = 1; i < 4 && e == cudaSuccess; ++i) e = ev(i);
        if (e != cudaSuccess) return cuda_fail(e, "backward over value-column slices");
        return HLA_OK;
    }
    const hla_params inner = bwd_inner(*p);
    p = &inner;
    hla::BwdArgs a;
    a.B = p->B; a.H = p->H; a.n = p->n; a.d = p->d; a.dv = p->dv; a.chunk = p->chunk;
    a.Hkv = p->Hkv > 0 ? p->Hkv : p->H;
    a.in_dtype = p->in_dtype; a.flags = p->flags & HLA_DECAY; a.gamma = p->gamma;
    a.q = q; a.k = k; a.v = v; a.go = dout;
    a.grad_q = dq; a.grad_k = dk; a.grad_v = dv;
    a.workspace = static_cast<float *>(workspace);
    a.dk_pair = a.Hkv < a.H ? a.workspace + hla::bwd_pair_offset(*p) : nullptr;
    a.dv_pair = a.Hkv < a.H ? a.dk_pair + (size_t)p->B * p->H * p->n * p->d : nullptr;
    a.sin_S = state_in ? state_in->S : nullptr;
    a.sin_C = state_in ? state_in->C : nullptr;
    a.sin_G = state_in ? state_in->G : nullptr;
    a.sin_m = state_in ? state_in->m : nullptr;
    a.sin_h = state_in ? state_in->h : nullptr;
    a.dS = d_state_in ? d_state_in->S : nullptr;
    a.dC = d_state_in ? d_state_in->C : nullptr;
    a.dG = d_state_in ? d_state_in->G : nullptr;
    a.dm = d_state_in ? d_state_in->m : nullptr;
    a.dh = d_state_in ? d_state_in->h : nullptr;
    a.adj0 = d_state_in ? a.workspace + hla::bwd_adj0_offset(*p) : nullptr;
    a.events = reinterpret_cast<cudaEvent_t const *>(phase_events);
    cudaError_t e = status_ptr(&a.err);
    if (e != cudaSuccess) return cuda_fail(e, "status word");
    if (norm) {
        if (hla::bwd_norm_tc_supported(*p, a)) return hla::bwd_norm_tc_launch(*p, a, st);
        return hla::bwd_norm_launch(*p, a, workspace, st);
    }
    e = hla::bwd_simt_launch(a, st);
    if (e != cudaSuccess) return cuda_fail(e, "backward launch");
    return HLA_OK;
}
}  // namespace

hla_status hla_backward_chunked(const hla_params *p, const void *q, const void *k, const void *v, const void *dout,
                                void *dq, void *dk, void *dv, void *workspace, size_t workspace_bytes,
                                void *stream) {
    return backward_impl(p, q, k, v, dout, nullptr, dq, dk, dv, nullptr, workspace, workspace_bytes, stream, nullptr);
}

hla_status hla_backward_chunked_traced(const hla_params *p, const void *q, const void *k, const void *v,
                                       const void *dout, void *dq, void *dk, void *dv, void *workspace,
                                       size_t workspace_bytes, void *stream, void *const *phase_events) {
    return backward_impl(p, q, k, v, dout, nullptr, dq, dk, dv, nullptr, workspace, workspace_bytes, stream,
                         phase_events);
}

hla_status hla_backward_chunked_state(const hla_params *p, const void *q, const void *k, const void *v,
                                      const void *dout, const hla_state *state_in, void *dq, void *dk, void *dv,
                                      const hla_state *d_state_in, void *workspace, size_t workspace_bytes,
                                      void *stream) {
    return backward_impl(p, q, k, v, dout, state_in, dq, dk, dv, d_state_in, workspace, workspace_bytes, stream,
                         nullptr);
}

namespace {
// The shape the third-order kernels run: a 128-token chunk as two of 64 and dv = 128 as
// two 64-column halves of the values (the output's column j and the state's P, T, M^QP
// columns j depend on the values' column j only; S^K, S^Q, M^KQ and the unit column's
// m, h, mqm on none), each half written into its columns (hla_bwd_split.cu copies).
// d = 128 runs in 16-token chunks over slices of at most 32 value columns: the CUDA-core
// output kernel holds S^K_p (128 x 128 fp32) beside P_p, T_p and the chunk's tiles only
// at that size.
hla_params fwd3_inner(const hla_params &p) {
    hla_params q = p;
    if (q.d == 128) {
        q.chunk = 16;
        if (q.dv > 32) q.dv = 32;
        return q;
    }
    if (q.chunk == 128) q.chunk = 64;
    if (q.dv == 128) q.dv = 64;
    return q;
}
// Value-column slices of the call (1: no split).
int fwd3_slices(const hla_params &p) { return p.dv / fwd3_inner(p).dv; }

// Split over value columns: the slice problem's workspace, the gathered value slice, the
// output slice, and the value-column slices (P, T, M^QP, fp32) of state_in and of
// state_out (byte offsets).
struct Split3 {
    size_t vh, oh, sin, sout, total;
};
Split3 split3_layout(const hla_params &p) {
    const hla_params q = fwd3_inner(p);
    const size_t el = p.in_dtype == HLA_F32 ? 4 : 2, rows = (size_t)p.B * p.H * p.n, w = q.dv;
    const size_t slice_state = (size_t)p.B * p.H * p.d * w * 4;
    Split3 L;
    size_t o = align256(hla::fwd3_workspace(q));
    L.vh = o; o = align256(o + rows * w * el);
    L.oh = o; o = align256(o + rows * w * el);
    L.sin = o; o = align256(o + 3 * slice_state);
    L.sout = o; o = align256(o + 3 * slice_state);
    L.total = o;
    return L;
}

hla_status forward3_impl(const hla_params *p, const void *q, const void *k, const void *v, void *o,
                         const hla_state3 *state_in, const hla_state3 *state_out, void *workspace,
                         size_t workspace_bytes, void *stream, void *const *phase_events);

hla_status check_fwd3_params(const hla_params *p) {
    if (!p) return fail(HLA_ERR_ARG, "params is NULL");
    if (p->B < 1 || p->H < 1 || p->n < 0) return fail(HLA_ERR_ARG, "need B >= 1, H >= 1, n >= 0");
    if (p->in_dtype != HLA_F32 && p->in_dtype != HLA_BF16) return fail(HLA_ERR_ARG, "unknown in_dtype");
    if (p->flags & ~(unsigned)(HLA_NORMALIZE | HLA_DECAY | HLA_UNMASKED | HLA_ASYMMETRIC))
        return fail(HLA_ERR_ARG, "unknown flag bits");
    if (p->Hkv < 0 || (p->Hkv > 0 && p->H % p->Hkv != 0))
        return fail(HLA_ERR_ARG, "Hkv must divide H (0 means Hkv = H)");
    if ((long long)p->B * p->H * (long long)p->n * (p->d > p->dv ? p->d : p->dv) > (1LL << 40))
        return fail(HLA_ERR_ARG, "problem too large");
    const bool dv_ok = p->dv == 16 || p->dv == 32 || p->dv == 64 || p->dv == 128;
    const bool c_ok = p->chunk == 16 || p->chunk == 32 || p->chunk == 64 || p->chunk == 128;
    if (!dv_ok || !c_ok || !hla::fwd3_supported(fwd3_inner(*p)))
        return fail(HLA_ERR_UNSUPPORTED,
                    "third order supports flags HLA_DECAY, HLA_NORMALIZE, Hkv dividing H, d, dv and chunk in "
                    "{16,32,64,128} (got flags=%u Hkv=%d d=%d dv=%d chunk=%d)",
                    p->flags, p->Hkv, p->d, p->dv, p->chunk);
    if ((p->flags & HLA_NORMALIZE) && !(p->eps >= 0.f)) return fail(HLA_ERR_ARG, "need eps >= 0");
    if ((p->flags & HLA_DECAY) && !p->gamma) return fail(HLA_ERR_ARG, "HLA_DECAY needs gamma");
    return HLA_OK;
}

hla_status check_state3(const hla_state3 *s, const char *name, bool normalize, bool maps = false) {
    if (!s) return HLA_OK;
    if (!s->S || !s->P || !s->T) return fail(HLA_ERR_ARG, "%s: S, P, T must be set", name);
    if (!aligned16(s->S) || !aligned16(s->P) || !aligned16(s->T))
        return fail(HLA_ERR_ARG, "%s: pointers must be 16-byte aligned", name);
    if (normalize && (!s->m || !s->h)) return fail(HLA_ERR_ARG, "%s: m and h must be set with HLA_NORMALIZE", name);
    if (maps && (!s->SQ || !s->MQP || !s->MKQ || (normalize && !s->mqm)))
        return fail(HLA_ERR_ARG, "%s: the segment maps SQ, MQP, MKQ (and mqm with HLA_NORMALIZE) must be set", name);
    return HLA_OK;
}
}  // namespace

size_t hla_forward3_workspace_size(const hla_params *p) {
    if (check_fwd3_params(p) != HLA_OK) return 0;
    if (fwd3_slices(*p) > 1) return split3_layout(*p).total;
    return hla::fwd3_workspace(fwd3_inner(*p));
}

hla_status hla_forward3_chunked(const hla_params *p, const void *q, const void *k, const void *v, void *o,
                                const hla_state3 *state_in, const hla_state3 *state_out, void *workspace,
                                size_t workspace_bytes, void *stream) {
    return hla_forward3_chunked_traced(p, q, k, v, o, state_in, state_out, workspace, workspace_bytes, stream,
                                       nullptr);
}

hla_status hla_forward3_chunked_traced(const hla_params *p, const void *q, const void *k, const void *v, void *o,
                                       const hla_state3 *state_in, const hla_state3 *state_out, void *workspace,
                                       size_t workspace_bytes, void *stream, void *const *phase_events) {
    return forward3_impl(p, q, k, v, o, state_in, state_out, workspace, workspace_bytes, stream, phase_events);
}

namespace {
hla_status forward3_impl(const hla_params *p, const void *q, const void *k, const void *v, void *o,
                         const hla_state3 *state_in, const hla_state3 *state_out, void *workspace,
                         size_t workspace_bytes, void *stream, void *const *phase_events) {
    hla_status s = check_fwd3_params(p);
    if (s != HLA_OK) return s;
    const bool norm = (p->flags & HLA_NORMALIZE) != 0;
    const bool maps = state_out && state_out->SQ;  // the segment maps are wanted
    if ((s = check_state3(state_in, "state_in", norm, maps)) != HLA_OK) return s;
    if ((s = check_state3(state_out, "state_out", norm, maps)) != HLA_OK) return s;
    if (state_in && state_out && (state_in->S == state_out->S || state_in->P == state_out->P || state_in->T == state_out->T ||
                                  (norm && (state_in->m == state_out->m || state_in->h == state_out->h))))
        return fail(HLA_ERR_ARG, "state_out may not alias state_in");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (p->n == 0) {  // no tokens: state_out = state_in (or zeros)
        if (!state_out) return HLA_OK;
        const size_t BH = (size_t)p->B * p->H, D = p->d, DV = p->dv;
        const size_t sz[9] = {BH * D * D * 4, BH * D * DV * 4, BH * D * DV * 4, BH * D * 4, BH * D * 4,
                              BH * D * D * 4, BH * D * DV * 4, BH * D * D * 4, BH * D * 4};
        float *dst[9] = {state_out->S, state_out->P, state_out->T, state_out->m, state_out->h,
                         state_out->SQ, state_out->MQP, state_out->MKQ, state_out->mqm};
        const bool used[9] = {true, true, true, norm, norm, maps, maps, maps, maps && norm};
        for (int i = 0; i < 9; ++i) {
            if (!used[i]) continue;
            cudaError_t e;
            if (state_in) {
                const float *src[9] = {state_in->S, state_in->P, state_in->T, state_in->m, state_in->h,
                                       state_in->SQ, state_in->MQP, state_in->MKQ, state_in->mqm};
                e = cudaMemcpyAsync(dst[i], src[i], sz[i], cudaMemcpyDeviceToDevice, st);
            } else {
                e = cudaMemsetAsync(dst[i], 0, sz[i], st);
            }
            if (e != cudaSuccess) return cuda_fail(e, "state copy");
        }
        return HLA_OK;
    }
    if (!q || !k || !v || !o) return fail(HLA_ERR_ARG, "q, k, v, o must be set when n > 0");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
        return fail(HLA_ERR_ARG, "q, k, v, o must be 16-byte aligned");
    const size_t need = hla_forward3_workspace_size(p);
    if (!workspace || workspace_bytes < need)
        return fail(HLA_ERR_ARG, "workspace too small: need %zu bytes, got %zu", need, workspace_bytes);
    if (!aligned16(workspace)) return fail(HLA_ERR_ARG, "workspace must be 16-byte aligned");
    const bool split = fwd3_slices(*p) > 1;
    if ((norm || split) && (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return fail(HLA_ERR_ARG, "workspace must be 256-byte aligned with HLA_NORMALIZE or a split over value "
                                 "columns (dv = 128; d = 128 with dv > 32)");
    if (phase_events) {
        for (int i = 0; i < 4; ++i)
            if (!phase_events[i]) return fail(HLA_ERR_ARG, "phase_events must hold four events");
    }
    if (split) {  // slices of the value columns, each written into its columns
        const hla_params in = fwd3_inner(*p);
        const Split3 L = split3_layout(*p);
        const int parts = fwd3_slices(*p), pw = in.dv;
        uint8_t *w = static_cast<uint8_t *>(workspace);
        const size_t rows = (size_t)p->B * p->H * p->n, srows = (size_t)p->B * p->H * p->d;
        const size_t kv_rows = (size_t)p->B * (p->Hkv > 0 ? p->Hkv : p->H) * p->n;
        const size_t hs = srows * pw;  // floats of one slice array of the state
        float *ti = reinterpret_cast<float *>(w + L.sin), *to = reinterpret_cast<float *>(w + L.sout);
        auto ev = [&](int i) {
            return phase_events ? cudaEventRecord(static_cast<cudaEvent_t>(phase_events[i]), st) : cudaSuccess;
        };
        cudaError_t e = ev(0);
        for (int h = 0; h < parts && e == cudaSuccess; ++h) {
            if ((e = hla::cols_part_copy(v, w + L.vh, kv_rows, p->in_dtype, p->dv, pw, h, true, st)) != cudaSuccess)
                break;
            hla_state3 si{}, so{};
            if (state_in) {
                si = *state_in;
                si.P = ti;
                si.T = ti + hs;
                si.MQP = maps ? ti + 2 * hs : nullptr;
                const float *src[3] = {state_in->P, state_in->T, state_in->MQP};
                for (int i = 0; i < (maps ? 3 : 2) && e == cudaSuccess; ++i)
                    e = hla::cols_part_copy(src[i], ti + i * hs, srows, HLA_F32, p->dv, pw, h, true, st);
                if (e != cudaSuccess) break;
            }
            if (state_out) {
                so = *state_out;
                so.P = to;
                so.T = to + hs;
                so.MQP = maps ? to + 2 * hs : nullptr;
            }
            s = forward3_impl(&in, q, k, w + L.vh, w + L.oh, state_in ? &si : nullptr, state_out ? &so : nullptr, w,
                              L.vh, stream, nullptr);
            if (s != HLA_OK) return s;
            if ((e = hla::cols_part_copy(w + L.oh, o, rows, p->in_dtype, p->dv, pw, h, false, st)) != cudaSuccess)
                break;
            if (state_out) {
                float *dst[3] = {state_out->P, state_out->T, state_out->MQP};
                for (int i = 0; i < (maps ? 3 : 2) && e == cudaSuccess; ++i)
                    e = hla::cols_part_copy(to + i * hs, dst[i], srows, HLA_F32, p->dv, pw, h, false, st);
            }
        }
        for (int i = 1; i < 4 && e == cudaSuccess; ++i) e = ev(i);
        if (e != cudaSuccess) return cuda_fail(e, "third-order forward over value-column slices");
        return HLA_OK;
    }
    const hla_params inner = fwd3_inner(*p);
    p = &inner;
    hla::Fwd3Args a;
    a.B = p->B; a.H = p->H; a.n = p->n; a.d = p->d; a.dv = p->dv; a.chunk = p->chunk;
    a.Hkv = p->Hkv > 0 ? p->Hkv : p->H;
    a.in_dtype = p->in_dtype;
    a.gamma = (p->flags & HLA_DECAY) ? p->gamma : nullptr;
    a.q = q; a.k = k; a.v = v; a.o = o;
    a.sin_S = state_in ? state_in->S : nullptr;
    a.sin_P = state_in ? state_in->P : nullptr;
    a.sin_T = state_in ? state_in->T : nullptr;
    a.sout_S = state_out ? state_out->S : nullptr;
    a.sout_P = state_out ? state_out->P : nullptr;
    a.sout_T = state_out ? state_out->T : nullptr;
    a.sin_SQ = maps && state_in ? state_in->SQ : nullptr;
    a.sin_MQP = maps && state_in ? state_in->MQP : nullptr;
    a.sin_MKQ = maps && state_in ? state_in->MKQ : nullptr;
    a.sout_SQ = maps ? state_out->SQ : nullptr;
    a.sout_MQP = maps ? state_out->MQP : nullptr;
    a.sout_MKQ = maps ? state_out->MKQ : nullptr;
    a.workspace = static_cast<float *>(workspace);
    a.events = reinterpret_cast<cudaEvent_t const *>(phase_events);
    cudaError_t e = status_ptr(&a.err);
    if (e != cudaSuccess) return cuda_fail(e, "status word");
    if (norm) {
        hla::Norm3 nm;
        nm.m_in = state_in ? state_in->m : nullptr;
        nm.h_in = state_in ? state_in->h : nullptr;
        nm.m_out = state_out ? state_out->m : nullptr;
        nm.h_out = state_out ? state_out->h : nullptr;
        nm.mqm_in = maps && state_in ? state_in->mqm : nullptr;
        nm.mqm_out = maps ? state_out->mqm : nullptr;
        nm.eps = p->eps;
        e = hla::fwd3_norm_launch(a, nm, st);
    } else {
        e = hla::fwd3_launch(a, st);
    }
    if (e != cudaSuccess) return cuda_fail(e, "third-order forward launch");
    return HLA_OK;
}
}  // namespace

hla_status hla_state3_combine(int count, int d, int dv, unsigned flags, const hla_state3 *A, const hla_state3 *B,
                              const hla_state3 *out, const float *decay_pow, void *stream) {
    if (count < 0) return fail(HLA_ERR_ARG, "need count >= 0");
    if (!width_ok(d) || !width_ok(dv))
        return fail(HLA_ERR_UNSUPPORTED, "d and dv must be in {16,32,64,128} (got %d, %d)", d, dv);
    if (flags & ~(unsigned)HLA_NORMALIZE) return fail(HLA_ERR_UNSUPPORTED, "flags must be 0 or HLA_NORMALIZE");
    if (!A || !B || !out) return fail(HLA_ERR_ARG, "A, B, out must be set");
    const bool norm = (flags & HLA_NORMALIZE) != 0;
    hla_status s;
    if ((s = check_state3(A, "A", norm, true)) != HLA_OK) return s;
    if ((s = check_state3(B, "B", norm, true)) != HLA_OK) return s;
    if ((s = check_state3(out, "out", norm, true)) != HLA_OK) return s;
    cudaError_t e = hla::state3_combine_launch(count, d, dv, norm, *A, *B, *out, decay_pow,
                                               static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "third-order combine launch");
    return HLA_OK;
}

hla_status hla_decode3_step(int N, int H, int d, int dv, hla_dtype dtype, unsigned flags, float eps,
                            const float *gamma, const hla_state3 *state, const void *q, const void *k, const void *v,
                            void *o, void *stream) {
    if (N < 0 || H < 1) return fail(HLA_ERR_ARG, "need N >= 0, H >= 1");
    if (!width_ok(d) || !width_ok(dv)) return fail(HLA_ERR_UNSUPPORTED, "d, dv must be in {16,32,64,128}");
    if (dtype != HLA_F32 && dtype != HLA_BF16) return fail(HLA_ERR_ARG, "unknown dtype");
    if (flags & ~(unsigned)(HLA_DECAY | HLA_NORMALIZE))
        return fail(HLA_ERR_UNSUPPORTED, "third-order decode supports HLA_DECAY and HLA_NORMALIZE (got %u)", flags);
    if ((flags & HLA_DECAY) && !gamma) return fail(HLA_ERR_ARG, "HLA_DECAY needs gamma");
    const bool norm = (flags & HLA_NORMALIZE) != 0;
    if (norm && !(eps >= 0.f)) return fail(HLA_ERR_ARG, "need eps >= 0");
    if (!state) return fail(HLA_ERR_ARG, "state must be set");
    hla_status s = check_state3(state, "state", norm);
    if (s != HLA_OK) return s;
    if (N > 0 && (!q || !k || !v || !o)) return fail(HLA_ERR_ARG, "q, k, v, o must be set");
    hla::Decode3Args a;
    a.N = N; a.H = H; a.d = d; a.dv = dv; a.dtype = dtype;
    a.gamma = (flags & HLA_DECAY) ? gamma : nullptr;
    a.eps = eps;
    a.m = norm ? state->m : nullptr;
    a.h = norm ? state->h : nullptr;
    a.S = state->S; a.P = state->P; a.T = state->T;
    a.q = q; a.k = k; a.v = v; a.o = o;
    cudaError_t e = hla::decode3_launch(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "third-order decode launch");
    return HLA_OK;
}

hla_status hla_state_combine(int count, int d, int dv, unsigned flags, const hla_state *A, const hla_state *B,
                             const hla_state *out, const float *decay_pow, void *stream) {
    if (count < 0) return fail(HLA_ERR_ARG, "count must be >= 0");
    if ((flags & HLA_UNMASKED) && (flags & HLA_ASYMMETRIC))
        return fail(HLA_ERR_ARG, "HLA_UNMASKED and HLA_ASYMMETRIC exclude each other");
    if (!width_ok(d) || !width_ok(dv)) return fail(HLA_ERR_UNSUPPORTED, "d, dv must be in {16,32,64,128}");
    if (!A || !B || !out) return fail(HLA_ERR_ARG, "A, B, out must be set");
    hla_status s;
    if ((s = check_state(A, "A")) != HLA_OK || (s = check_state(B, "B")) != HLA_OK ||
        (s = check_state(out, "out")) != HLA_OK)
        return s;
    hla::CombineArgs a;
    a.count = count; a.d = d; a.dv = dv; a.flags = flags;
    a.A = hla::to_ptrs(A); a.B = hla::to_ptrs(B); a.out = hla::to_ptrs(out);
    a.decay_pow = decay_pow;
    cudaError_t e = hla::combine_launch(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "combine launch");
    return HLA_OK;
}

hla_status hla_decode_step(int N, int H, int Hkv, int d, int dv, hla_dtype dtype, unsigned flags, float eps,
                           const float *gamma, const hla_state *state, const void *q, const void *k,
                           const void *v, void *o, void *stream) {
    if (N < 0 || H < 1 || (N % H) != 0) return fail(HLA_ERR_ARG, "need N >= 0, H >= 1, N %% H == 0");
    if (Hkv < 0 || (Hkv > 0 && H % Hkv != 0)) return fail(HLA_ERR_ARG, "Hkv must divide H (0 means Hkv = H)");
    if (!width_ok(d) || !width_ok(dv)) return fail(HLA_ERR_UNSUPPORTED, "d, dv must be in {16,32,64,128}");
    if (dtype != HLA_F32 && dtype != HLA_BF16) return fail(HLA_ERR_ARG, "unknown dtype");
    if (flags & ~(unsigned)(HLA_NORMALIZE | HLA_DECAY | HLA_UNMASKED | HLA_ASYMMETRIC))
        return fail(HLA_ERR_ARG, "unknown flag bits");
    if ((flags & HLA_UNMASKED) && (flags & HLA_ASYMMETRIC))
        return fail(HLA_ERR_ARG, "HLA_UNMASKED and HLA_ASYMMETRIC exclude each other");
    if ((flags & HLA_DECAY) && !gamma) return fail(HLA_ERR_ARG, "HLA_DECAY needs gamma");
    if (!state) return fail(HLA_ERR_ARG, "state must be set");
    hla_status s;
    if (flags & HLA_UNMASKED) {  // G, h are not part of the unmasked state
        if (!state->S || !state->C || !state->m) return fail(HLA_ERR_ARG, "state: S, C, m must be set");
        if (!aligned16(state->S) || !aligned16(state->C) || !aligned16(state->m))
            return fail(HLA_ERR_ARG, "state: pointers must be 16-byte aligned");
    } else if ((s = check_state(state, "state")) != HLA_OK) {
        return s;
    }
    if (N > 0 && (!q || !k || !v || !o)) return fail(HLA_ERR_ARG, "q, k, v, o must be set");
    hla::DecodeArgs a;
    a.N = N; a.H = H; a.d = d; a.dv = dv; a.dtype = dtype; a.flags = flags; a.eps = eps; a.gamma = gamma;
    a.Hkv = Hkv > 0 ? Hkv : H;
    a.st = hla::to_ptrs(state);
    a.q = q; a.k = k; a.v = v; a.o = o;
    cudaError_t e = hla::decode_launch(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    return HLA_OK;
}

hla_status hla_selftest_expired_wait(void *stream) {
    unsigned *err = nullptr;
    cudaError_t e = status_ptr(&err);
    if (e != cudaSuccess) return cuda_fail(e, "status word");
    expired_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(err);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
    return HLA_OK;
}

hla_status hla_sync_status(void *stream) {
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
    unsigned v = 0;
    e = cudaMemcpyFromSymbol(&v, g_dev_status, sizeof v);
    if (e != cudaSuccess) return cuda_fail(e, "read status word");
    if (v != 0u) {
        const unsigned zero = 0u;
        e = cudaMemcpyToSymbol(g_dev_status, &zero, sizeof zero);
        if (e != cudaSuccess) return cuda_fail(e, "clear status word");
        return fail(HLA_ERR_TIMEOUT, "a bounded device wait expired (status 0x%x)", v);
    }
    return HLA_OK;
}

}  // extern "C"
