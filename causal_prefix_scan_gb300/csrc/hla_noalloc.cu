// hla_noalloc.cu -- hla_forward_chunked_noalloc: the chunked forward for
// callers that cannot allocate device memory.
//
// Such callers (code running inside an allocator hook, allocation-free
// real-time loops, hosts that hand out device memory only up front) cannot give
// hla_forward_chunked its workspace.  Here the workspace is one file-scope
// device array, so the call allocates nothing: it looks up the array's device
// address once per device and passes it to the ordinary forward.
#include <cstdio>
#include <mutex>

#include "hla_internal.h"

namespace {

constexpr size_t kScratchBytes = HLA_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// The scratch.  In host code this name is only a stand-in for the symbol, never
// a usable device address: kernels get the address from cudaGetSymbolAddress.
// Zero at module load; every forward call leaves its ordering header zero again.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device (looked up once per device).
hla_status scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return hla::report(HLA_ERR_CUDA, cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return hla::report(HLA_ERR_UNSUPPORTED, "device index out of range");
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            char msg[256];
            snprintf(msg, sizeof msg, "no-alloc scratch address lookup failed: %s", cudaGetErrorString(e));
            return hla::report(HLA_ERR_CUDA, msg);
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
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
    hla_status s = scratch_address(&scratch);
    if (s != HLA_OK) return s;
    // The ordering header and per-segment flags at the front must start at zero;
    // the forward leaves them zero, clear them anyway in case an earlier call on
    // this array did not finish.  256 bytes of header plus one flag per
    // (pair, segment), at most max(B*H, SM count) of them.
    int dev = 0, nsm = 1;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    const size_t bh = (size_t)p->B * (size_t)p->H;
    size_t clear = 256 + 4 * (bh > (size_t)nsm ? bh : (size_t)nsm);
    clear = (clear + 255) & ~(size_t)255;
    if (clear > need) clear = need;
    cudaError_t e = cudaMemsetAsync(scratch, 0, clear, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return hla::report(HLA_ERR_CUDA, cudaGetErrorString(e));
    return hla_forward_chunked(p, q, k, v, o, state_in, state_out, scratch, kScratchBytes, stream);
}
