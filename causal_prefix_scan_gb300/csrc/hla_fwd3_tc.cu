// hla_fwd3_tc.cu -- tensor-core (tcgen05 MMA, TMEM accumulators) kernels for the
// chunk-local sums and the outputs of masked third-order HLA, bf16 inputs,
// d = dv = chunk = 64.  The chunk algebra is that of hla_fwd3_simt.cuh
// ("Higher-order Linear Attention", gist.science summary, sections 3 and 4):
//   A~ = tril(Q K^T),  U = Q S^K_p + A~ K,  W = Q P_p + A~ V,  M = tril(Q U^T),
//   O = Q T_p + M W;
//   local sums (zero prefix): S^K = K^T K, S^Q = Q^T Q, M^KQ = U^T Q, P = K^T V,
//   T = U^T W, M^QP = Q^T W.
// One CTA (8 warps, two per TMEM lane quadrant) per chunk; every product is a
// 64-row tcgen05.mma group issued by thread 0 from 128-byte-swizzled bf16 tiles.
// The fp32 prefix states enter as bf16 hi + lo pairs (two MMAs each), so their
// rounding is that of fp32; A~, U, W and M are rounded to bf16 between products.
// The scan between the two kernels stays on the CUDA cores (hla_fwd3_simt.cuh).
#include "hla_chunk_tc.cuh"
#include "hla_fwd3_simt.cuh"

namespace hla {
namespace fwd3tc {
using fwd3::Ws3;
using namespace chunktc;
namespace {

// tiles of the local-sums kernel
enum { L_Q, L_K, L_V, L_A, L_U, L_W, L_N };
// tiles of the output kernel
enum { O_Q, O_K, O_V, O_SH, O_SL, O_PH, O_PL, O_TH, O_TL, O_A, O_U, O_W, O_N };

__global__ void __launch_bounds__(kTc, 2) fwd3_local_tc_kernel(const __grid_constant__ Fwd3Args a,
                                                                 const __grid_constant__ ChunkMaps tm) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    Ctx x;
    if (!setup(x, smem_raw, L_N, a.err)) return;
    const int nch = (a.n + 63) / 64, u = blockIdx.x / nch, ch = blockIdx.x % nch;
    const int t0 = ch * 64, L = min(64, a.n - t0);
    const size_t r0 = ((size_t)u * a.n + t0) * 64;
    {
        const CUtensorMap *m[3] = {&tm.q, &tm.k, &tm.v};
        const int kvu = (u / a.H) * a.Hkv + (u % a.H) / (a.H / a.Hkv);  // key/value head
        const int un[3] = {u, kvu, kvu};
        uint8_t *dst[3] = {x.tile(L_Q), x.tile(L_K), x.tile(L_V)};
        tma_issue<3>(x, m, un, t0, dst);
    }
    const bool loaded = tma_wait(x);
    x.publish();
    float v[16];
    do {
        if (!loaded) break;
        // A~ = tril(Q K^T)
        if (x.tid == 0) mma_kk(x.tb, x.tile(L_Q), x.tile(L_K), false);
        x.commit();
        if (!x.wait()) break;
        x.ld_row(0, v);
        store_tril(x, x.tile(L_A), v);
        x.publish();
        // U = A~ K, W = A~ V (no earlier state)
        if (x.tid == 0) {
            mma_km(x.tb + 64, x.tile(L_A), x.tile(L_K), false);
            mma_km(x.tb + 128, x.tile(L_A), x.tile(L_V), false);
        }
        x.commit();
        if (!x.wait()) break;
        x.ld_row(64, v);
        tile_store_row16(x.tile(L_U), 64, x.row, x.c0, v);
        x.ld_row(128, v);
        tile_store_row16(x.tile(L_W), 64, x.row, x.c0, v);
        x.publish();
        // S^K = K^T K, S^Q = Q^T Q, M^KQ = U^T Q, P = K^T V (rows = feature index)
        if (x.tid == 0) {
            mma_mm(x.tb + 0, x.tile(L_K), x.tile(L_K));
            mma_mm(x.tb + 64, x.tile(L_Q), x.tile(L_Q));
            mma_mm(x.tb + 128, x.tile(L_U), x.tile(L_Q));
            mma_mm(x.tb + 192, x.tile(L_K), x.tile(L_V));
        }
        x.commit();
        if (!x.wait()) break;
        const Ws3 ws{64, 64};
        float *out = a.workspace + ((size_t)u * nch + ch) * ws.loc_floats();
        const size_t ro = (size_t)x.row * 64 + x.c0;
        x.ld_row(0, v);
        st_row16(out + ws.o_sk() + ro, v);
        x.ld_row(64, v);
        st_row16(out + ws.o_sq() + ro, v);
        x.ld_row(128, v);
        st_row16(out + ws.o_mkq() + ro, v);
        x.ld_row(192, v);
        st_row16(out + ws.o_p() + ro, v);
        x.publish();  // the reads of columns 0-127 precede their reuse
        // T = U^T W, M^QP = Q^T W
        if (x.tid == 0) {
            mma_mm(x.tb + 0, x.tile(L_U), x.tile(L_W));
            mma_mm(x.tb + 64, x.tile(L_Q), x.tile(L_W));
        }
        x.commit();
        if (!x.wait()) break;
        x.ld_row(0, v);
        st_row16(out + ws.o_t() + ro, v);
        x.ld_row(64, v);
        st_row16(out + ws.o_mqp() + ro, v);
    } while (false);
    teardown(x);
}

__global__ void __launch_bounds__(kTc, 2) fwd3_out_tc_kernel(const __grid_constant__ Fwd3Args a,
                                                               const __grid_constant__ ChunkMaps tm) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    Ctx x;
    if (!setup(x, smem_raw, O_N, a.err)) return;
    const int nch = (a.n + 63) / 64, u = blockIdx.x / nch, ch = blockIdx.x % nch;
    const int t0 = ch * 64, L = min(64, a.n - t0);
    const size_t r0 = ((size_t)u * a.n + t0) * 64;
    const Ws3 ws{64, 64};
    const float *so = a.workspace + (size_t)a.B * a.H * nch * ws.loc_floats() + ((size_t)u * nch + ch) * ws.st_floats();
    {  // the bf16 inputs by TMA while the threads convert the states
        const CUtensorMap *m[3] = {&tm.q, &tm.k, &tm.v};
        const int kvu = (u / a.H) * a.Hkv + (u % a.H) / (a.H / a.Hkv);  // key/value head
        const int un[3] = {u, kvu, kvu};
        uint8_t *dst[3] = {x.tile(O_Q), x.tile(O_K), x.tile(O_V)};
        tma_issue<3>(x, m, un, t0, dst);
        const float *ss[3] = {so + ws.s_sk(), so + ws.s_p(), so + ws.s_t()};
        uint8_t *hi[3] = {x.tile(O_SH), x.tile(O_PH), x.tile(O_TH)}, *lo[3] = {x.tile(O_SL), x.tile(O_PL), x.tile(O_TL)};
        load_tiles_hilo<3>(ss, hi, lo);
    }
    const bool loaded = tma_wait(x);
    x.publish();
    constexpr uint32_t SA = 0, SU = 64, SW = 128, SO = 192;
    float v[16];
    do {
        if (!loaded) break;
        // A~ = Q K^T, and the prefix-state terms Q S^K_p, Q P_p, Q T_p
        if (x.tid == 0) {
            mma_kk(x.tb + SA, x.tile(O_Q), x.tile(O_K), false);
            mma_km(x.tb + SU, x.tile(O_Q), x.tile(O_SH), false);
            mma_km(x.tb + SU, x.tile(O_Q), x.tile(O_SL), true);
            mma_km(x.tb + SW, x.tile(O_Q), x.tile(O_PH), false);
            mma_km(x.tb + SW, x.tile(O_Q), x.tile(O_PL), true);
            mma_km(x.tb + SO, x.tile(O_Q), x.tile(O_TH), false);
            mma_km(x.tb + SO, x.tile(O_Q), x.tile(O_TL), true);
        }
        x.commit();
        if (!x.wait()) break;
        x.ld_row(SA, v);
        store_tril(x, x.tile(O_A), v);
        x.publish();
        // U += A~ K, W += A~ V
        if (x.tid == 0) {
            mma_km(x.tb + SU, x.tile(O_A), x.tile(O_K), true);
            mma_km(x.tb + SW, x.tile(O_A), x.tile(O_V), true);
        }
        x.commit();
        if (!x.wait()) break;
        x.ld_row(SU, v);
        tile_store_row16(x.tile(O_U), 64, x.row, x.c0, v);
        x.ld_row(SW, v);
        tile_store_row16(x.tile(O_W), 64, x.row, x.c0, v);
        x.publish();
        // M = tril(Q U^T)
        if (x.tid == 0) mma_kk(x.tb + SA, x.tile(O_Q), x.tile(O_U), false);
        x.commit();
        if (!x.wait()) break;
        x.ld_row(SA, v);
        store_tril(x, x.tile(O_A), v);
        x.publish();
        // O += M W
        if (x.tid == 0) mma_km(x.tb + SO, x.tile(O_A), x.tile(O_W), true);
        x.commit();
        if (!x.wait()) break;
        x.ld_row(SO, v);
        if (x.row < L) {
            __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(a.o) + r0 + (size_t)x.row * 64 + x.c0;
            uint4 p0, p1;
            p0.x = pack_bf16(v[0], v[1]);   p0.y = pack_bf16(v[2], v[3]);
            p0.z = pack_bf16(v[4], v[5]);   p0.w = pack_bf16(v[6], v[7]);
            p1.x = pack_bf16(v[8], v[9]);   p1.y = pack_bf16(v[10], v[11]);
            p1.z = pack_bf16(v[12], v[13]); p1.w = pack_bf16(v[14], v[15]);
            reinterpret_cast<uint4 *>(o)[0] = p0;
            reinterpret_cast<uint4 *>(o)[1] = p1;
        }
    } while (false);
    teardown(x);
}

constexpr size_t kLocalSmem = L_N * TILE + 64, kOutSmem = O_N * TILE + 64;

}  // namespace

cudaError_t local_tc(const Fwd3Args &a, cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(fwd3_local_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kLocalSmem);
    if (e != cudaSuccess) return e;
    const int nch = (a.n + 63) / 64;
    ChunkMaps m;
    if (!chunk_maps(m, a.q, a.k, a.v, nullptr, a.n, a.B * a.H, a.B * a.Hkv)) return cudaErrorInvalidValue;
    fwd3_local_tc_kernel<<<a.B * a.H * nch, kTc, kLocalSmem, st>>>(a, m);
    return cudaGetLastError();
}

cudaError_t out_tc(const Fwd3Args &a, cudaStream_t st) {
    cudaError_t e =
        cudaFuncSetAttribute(fwd3_out_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kOutSmem);
    if (e != cudaSuccess) return e;
    const int nch = (a.n + 63) / 64;
    ChunkMaps m;
    if (!chunk_maps(m, a.q, a.k, a.v, nullptr, a.n, a.B * a.H, a.B * a.Hkv)) return cudaErrorInvalidValue;
    fwd3_out_tc_kernel<<<a.B * a.H * nch, kTc, kOutSmem, st>>>(a, m);
    return cudaGetLastError();
}

}  // namespace fwd3tc
}  // namespace hla
