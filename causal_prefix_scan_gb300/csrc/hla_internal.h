// hla_internal.h -- argument bundles and launcher declarations shared by the
// C-ABI layer (hla_api.cu) and the kernel translation units.
#pragma once

#include <cstddef>
#include <cuda_runtime.h>

#include "hla.h"
#include "hla_common.cuh"

namespace hla {

struct StatePtrs {
    float *S = nullptr, *C = nullptr, *m = nullptr, *G = nullptr, *h = nullptr;
};

inline StatePtrs to_ptrs(const hla_state *s) {
    StatePtrs p;
    if (s) { p.S = s->S; p.C = s->C; p.m = s->m; p.G = s->G; p.h = s->h; }
    return p;
}

struct FwdArgs {
    int B, H, n, d, dv, chunk;
    int Hkv;  // key/value heads (H % Hkv == 0)
    hla_dtype in_dtype;
    unsigned flags;
    float eps;
    const float *gamma;
    const void *q, *k, *v;
    void *o;
    StatePtrs sin, sout;
    void *workspace;
    size_t ws_bytes;
    unsigned *err;  // sticky device status word
};

// CUDA-core path (fp32 arithmetic; d, dv, chunk in {16,32,64}).
bool fwd_simt_supported(const hla_params &p);
cudaError_t fwd_simt_launch(const FwdArgs &a, cudaStream_t st);

// Tensor-core path (bf16 inputs; d, dv, chunk in {64,128}; asymmetric: dv <= d).
bool fwd_tc_supported(const hla_params &p);
size_t fwd_tc_workspace(const hla_params &p, int num_sms);
const char *fwd_tc_kernel_name(const hla_params &p);
// Bytes at the start of the tensor-core forward's workspace that hold its ordering
// header and release flags: zero before the first call on a workspace; each call leaves
// them ready for the next (its generation in the header, its tag on the flags).
size_t fwd_tc_sync_bytes(const hla_params &p, int num_sms);
cudaError_t fwd_tc_launch(const FwdArgs &a, cudaStream_t st, int num_sms);

struct CombineArgs {
    int count, d, dv;
    unsigned flags;  // 0, HLA_UNMASKED or HLA_ASYMMETRIC: which concatenation rule
    StatePtrs A, B, out;
    const float *decay_pow;
};
cudaError_t combine_launch(const CombineArgs &a, cudaStream_t st);

struct DecodeArgs {
    int N, H, d, dv;
    int Hkv;  // key/value heads per sequence (H % Hkv == 0)
    hla_dtype dtype;
    unsigned flags;
    float eps;
    const float *gamma;
    StatePtrs st;
    const void *q, *k, *v;
    void *o;
};
cudaError_t decode_launch(const DecodeArgs &a, cudaStream_t st);

struct BwdArgs {
    int B, H, n, d, dv, chunk;
    int Hkv;  // key/value heads (H % Hkv == 0); below H, dk and dv are summed over each group
    hla_dtype in_dtype;
    unsigned flags;  // 0 or HLA_DECAY
    const float *gamma;
    const void *q, *k, *v, *go;    // inputs and the gradient of the output
    void *grad_q, *grad_k, *grad_v;  // outputs
    float *workspace;
    float *dk_pair, *dv_pair;  // Hkv < H: fp32 dk, dv of every query head before the group sum
    // the state before the first token (NULL: zeros), fp32 [B*H][d][d], [B*H][d][dv] x 2
    const float *sin_S, *sin_C, *sin_G;
    const float *sin_m, *sin_h;  // with ratio normalisation: the rest of the state
    // its gradient (dS NULL: not wanted), and the per-pair adjoints at the first token
    // the scan leaves for it (Lam [d][dv], then Om [d][d])
    float *dS, *dC, *dG, *adj0;
    float *dm, *dh;  // with ratio normalisation
    cudaEvent_t const *events;  // NULL or four events recorded at the phase boundaries
    unsigned *err;              // sticky device status word (bounded waits of the tensor-core kernels)
};

// Backward of the masked forward on CUDA cores (d, dv, chunk in {16,32,64}).
bool bwd_simt_supported(const hla_params &p);
size_t bwd_simt_workspace(const hla_params &p);
size_t bwd_pair_offset(const hla_params &p);  // floats before the per-query-head dk, dv
size_t bwd_adj0_offset(const hla_params &p);  // floats before the adjoints at the first token
cudaError_t bwd_simt_launch(const BwdArgs &a, cudaStream_t st);

// Backward through the ratio normalisation: two unnormalised fp32 forwards (values and
// a unit-value tile), the augmented upstream gradients, two unnormalised fp32 backwards
// and a sum of their dq, dk.  Byte offsets into the caller's workspace (256-byte
// aligned); the *32 buffers exist for bf16 inputs only.
struct NormLayout {
    int w1;  // width of the unit-value tile
    size_t fwd_ws, fwd_ws_bytes, num, den1, unit, gn, g1, dq1, dk1, dv1, bwd_ws;
    size_t q32, k32, v32, g32, dq32, dk32, dv32;
    int P;              // segments per sequence of the fp32 forwards (1: no split)
    size_t grep, seg, pre;  // decay rates repeated per segment; segment states; their prefixes
    // a given initial state: the unit-value pass's C and G (m, h in column 0), its state
    // gradient (S, C, G), and a zero d-vector per pair (the m, h the unnormalised passes ignore)
    size_t ce, ge, ds2, dce, dge, zvec;
    size_t total;
};
NormLayout bwd_norm_layout(const hla_params &p);
hla_status bwd_norm_launch(const hla_params &p, const BwdArgs &a, void *workspace, cudaStream_t st);
// A call split over value columns (hla_bwd_split.cu; the backward and the third-order
// forward at dv = 128 or d = 128): columns [part_width part, part_width (part + 1)) of
// [rows][width] elements of type dt gathered into [rows][part_width] (or scattered back;
// part_width elements a multiple of 16 bytes), and the fp32 sum of the slices' dq, dk
// (first: overwrite) with its final rounding.
cudaError_t cols_part_copy(const void *src, void *dst, size_t rows, hla_dtype dt, int width, int part_width,
                           int part, bool gather, cudaStream_t st);
cudaError_t acc_add(float *acc, const void *src, size_t count, hla_dtype dt, bool first, cudaStream_t st);
cudaError_t acc_store(void *dst, const float *acc, size_t count, hla_dtype dt, cudaStream_t st);
// The same on the tensor cores (hla_bwd_norm_tc.cu): bf16, d = dv = chunk = 64 (the shape),
// no given initial state and no state gradient (supported); workspace bytes, 0 off the shape.
bool bwd_norm_tc_shape(const hla_params &p);
bool bwd_norm_tc_supported(const hla_params &p, const BwdArgs &a);
size_t bwd_norm_tc_workspace(const hla_params &p);
hla_status bwd_norm_tc_launch(const hla_params &p, const BwdArgs &a, cudaStream_t st);

struct Fwd3Args {
    int B, H, n, d, dv, chunk;
    int Hkv;  // key/value heads (query head h reads h / (H / Hkv))
    hla_dtype in_dtype;
    const float *gamma;  // [H] decay per head, or NULL (none)
    const void *q, *k, *v;
    void *o;
    const float *sin_S, *sin_P, *sin_T;  // state before the first token (all NULL: zeros)
    float *sout_S, *sout_P, *sout_T;     // state after the last token (all NULL: skip)
    // segment maps S^Q, M^QP, M^KQ: written with the state when sout_SQ is set, composed
    // onto those of state_in (NULL: a state_in without maps, or none)
    const float *sin_SQ, *sin_MQP, *sin_MKQ;
    float *sout_SQ, *sout_MQP, *sout_MKQ;
    float *workspace;
    cudaEvent_t const *events;  // NULL or four events recorded at the phase boundaries
    unsigned *err;              // sticky device status word (bounded waits of the tensor-core kernels)
};

struct Decode3Args {
    int N, H, d, dv;
    hla_dtype dtype;
    const float *gamma;  // [H] decay per head (pair u uses gamma[u % H]), or NULL
    float eps;
    float *S, *P, *T;
    float *m, *h;        // with ratio normalisation: key mass and the unit-value column of T; else NULL
    const void *q, *k, *v;
    void *o;
};

// Masked third-order forward and decode on CUDA cores.
bool fwd3_supported(const hla_params &p);
size_t fwd3_workspace(const hla_params &p);
cudaError_t fwd3_launch(const Fwd3Args &a, cudaStream_t st);
// Ratio-normalised third order: the forward of the values (into o), the forward of a
// unit-value tile (the denominator) with the same S, then o /= den + eps.  m, h: the
// key mass and the unit-value column of T per pair ([B*H][d]), before (in) and after
// (out) the tokens; NULL for zeros / not wanted.  The workspace is fwd3_workspace(p)
// with HLA_NORMALIZE.
struct Norm3 {
    const float *m_in, *h_in, *mqm_in;
    float *m_out, *h_out, *mqm_out;  // mqm: the M^QP of a unit value (with the maps only)
    float eps;
};
cudaError_t fwd3_norm_launch(const Fwd3Args &a, const Norm3 &nm, cudaStream_t st);
// The segment maps of a forward that has run (its local sums and prefix states are in
// a.workspace) into a.sout_SQ, a.sout_MQP, a.sout_MKQ.
cudaError_t fwd3_maps_launch(const Fwd3Args &a, cudaStream_t st);
// hla_state3_combine on the device (d, dv in {16,32,64}).
cudaError_t state3_combine_launch(int count, int d, int dv, bool norm, const hla_state3 &A, const hla_state3 &B,
                                  const hla_state3 &out, const float *decay_pow, cudaStream_t st);
cudaError_t decode3_launch(const Decode3Args &a, cudaStream_t st);

// Set this thread's last-error message and return `s`.
hla_status report(hla_status s, const char *msg);

}  // namespace hla
