// hla_noalloc.cu -- hla_forward_chunked_noalloc: the chunked forward for
// callers that cannot allocate device memory.
//
// Such callers (code running inside an allocator hook, allocation-free
// real-time loops, hosts that hand out device memory only up front) cannot give
// hla_forward_chunked its workspace.  Here the workspace is one file-scope
// device array, so the call allocates nothing: it looks up the array's device
// address for the current device's context and passes it to the ordinary forward.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdio>
#include <mutex>

#include "hla_internal.h"

namespace {

constexpr size_t kScratchBytes = HLA_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// The scratch.  In host code this name is only a stand-in for the symbol, never
// a usable device address: kernels get the address from cudaGetSymbolAddress.
// Zero at module load; every forward call leaves its ordering header and flags ready for the next.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_mu;
struct Cached {
    CUcontext ctx = nullptr;  // context the address belongs to
    void *ptr = nullptr;
};
Cached g_scratch[kMaxDevices];

// The CUDA driver's cuCtxGetCurrent, reached through the runtime (no link to libcuda).
PFN_cuCtxGetCurrent_v4000 ctx_getter() {
    static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    }
    return fn;
}

hla_status cuda_err(cudaError_t e, const char *where) {
    char msg[256];
    snprintf(msg, sizeof msg, "%s: %s", where, cudaGetErrorString(e));
    return hla::report(HLA_ERR_CUDA, msg);
}

// Device address of the scratch for the current device.  The lookup runs on the
// first call on a device and again whenever that device's current context differs
// from the one the cached address was taken in (after cudaDeviceReset the module,
// and with it the array, is loaded anew).  Also returns the device index.
hla_status scratch_address(void **out, int *dev_out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_err(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return hla::report(HLA_ERR_UNSUPPORTED, "device index out of range");
    auto get = ctx_getter();
    if (!get) return hla::report(HLA_ERR_CUDA, "no-alloc forward: cuCtxGetCurrent unavailable");
    CUcontext ctx = nullptr;  // NULL before the runtime has set up this device
    if (get(&ctx) != CUDA_SUCCESS) return hla::report(HLA_ERR_CUDA, "no-alloc forward: cannot read the context");
    std::lock_guard<std::mutex> lock(g_mu);
    Cached &c = g_scratch[dev];
    if (!c.ptr || !ctx || c.ctx != ctx) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);  // sets up the primary context if needed
        if (e != cudaSuccess || !p) return cuda_err(e, "no-alloc scratch address lookup");
        if (get(&ctx) != CUDA_SUCCESS || !ctx)
            return hla::report(HLA_ERR_CUDA, "no-alloc forward: no current context after the lookup");
        c.ctx = ctx;
        c.ptr = p;
    }
    *out = c.ptr;
    *dev_out = dev;
    return HLA_OK;
}

}  // namespace

extern "C" hla_status hla_forward_chunked_noalloc(const hla_params *p, const void *q, const void *k,
                                                  const void *v, void *o, const hla_state *state_in,
                                                  const hla_state *state_out, void *stream) {
    if (!p) return hla::report(HLA_ERR_ARG, "params is NULL");
    const size_t need = hla_forward_workspace_size(p);
    if (need == 0)  // invalid parameters (reported by the forward) or a path without scratch
        return hla_forward_chunked(p, q, k, v, o, state_in, state_out, nullptr, 0, stream);
    if (need > kScratchBytes) {
        char msg[256];
        snprintf(msg, sizeof msg, "no-alloc forward needs %zu bytes of scratch; its fixed array holds %zu",
                 need, kScratchBytes);
        return hla::report(HLA_ERR_UNSUPPORTED, msg);
    }
    void *scratch = nullptr;
    int dev = 0;
    hla_status s = scratch_address(&scratch, &dev);
    if (s != HLA_OK) return s;
    // The forward's ordering header and release flags (one per sequence and piece)
    // start each call at zero here: each call would leave them ready for the next,
    // but they are cleared anyway in case an earlier call on this array did not
    // finish.  Their size comes from the same work plan the forward uses.
    int nsm = 0;
    cudaError_t e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess || nsm < 1) return cuda_err(e, "SM count");
    const size_t clear = hla::fwd_tc_sync_bytes(*p, nsm);
    if (clear > 0) {
        e = cudaMemsetAsync(scratch, 0, clear < need ? clear : need, static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return cuda_err(e, "scratch clear");
    }
    return hla_forward_chunked(p, q, k, v, o, state_in, state_out, scratch, kScratchBytes, stream);
}
