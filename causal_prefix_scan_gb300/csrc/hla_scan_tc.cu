// hla_scan_tc.cu -- the scans over chunks of the backward pass and of the third-order
// forward for bf16 inputs with d = dv = chunk = 64, without a chain of dependent
// matrix products.
//
// Both recursions are linear in the state they carry, with increments that depend only
// on plain (decayed) prefix sums:
//   backward ("Higher-order Linear Attention", reverse mode of the masked recurrence):
//     S_p(B)     = sum_{B' < B} g^{...} S_loc(B')                 (prefix, factor g^L)
//     X_p(B)     = sum_{B' < B} g^{...} [S_p(B') C_q(B') + X_loc(B')]   (prefix, g^{2L})
//     Lam_n(B)   = sum_{B' > B} g^{...} L_loc(B')                 (suffix, g^{2L})
//     Om_n(B)    = sum_{B' > B} g^{...} [O_loc(B') + Lam_n(B') W(B')]   (suffix, g^L)
//   third order (section 4, "Derde-orde scans": composition through segment maps):
//     S^K_p, P_p plain prefix sums;
//     T_p(B) = T_in + sum_{B' < B} [T_B' + S^K_p(B') (M^QP_B' + S^Q_B' P_p(B')) + M^KQ_B' P_p(B')].
// So each scan runs as (1) an elementwise prefix / suffix sum over chunks, (2) one
// tensor-core kernel per chunk forming the increments (operands as bf16 hi + lo pairs,
// three MMAs per product: fp32-level accuracy), (3) a second elementwise scan.
#include "hla_bwd_simt.cuh"
#include "hla_chunk_tc.cuh"
#include "hla_fwd3_simt.cuh"

namespace hla {
namespace scantc {
using namespace chunktc;
namespace {

constexpr int kPrefixThreads = 256;

// Each thread scans four consecutive elements (count a multiple of 4, 16-byte aligned).
__global__ void __launch_bounds__(kPrefixThreads) chunk_prefix_kernel(const __grid_constant__ PrefixArgs a) {
    const PrefixJob &j = a.job[blockIdx.y];
    const int per_unit = (j.count / 4 + kPrefixThreads - 1) / kPrefixThreads;
    const int u = blockIdx.x / per_unit, e = ((blockIdx.x % per_unit) * kPrefixThreads + threadIdx.x) * 4;
    if (u >= a.units || e >= j.count) return;
    const float lg = a.gamma ? log2f(a.gamma[u % a.H]) : 0.f;
    float4 R = j.init ? *reinterpret_cast<const float4 *>(j.init + (size_t)u * j.count + e) : make_float4(0, 0, 0, 0);
    const float *in = j.in + (size_t)u * a.nch * j.in_stride + j.in_off + e;
    float *out = j.out + (size_t)u * a.nch * j.out_stride + j.out_off + e;
    // walk the chunks with pointer steps: forward +stride, reverse -stride from the last chunk
    const long long sin = j.reverse ? -(long long)j.in_stride : (long long)j.in_stride;
    const long long sout = j.reverse ? -(long long)j.out_stride : (long long)j.out_stride;
    if (j.reverse) {
        in += (size_t)(a.nch - 1) * j.in_stride;
        out += (size_t)(a.nch - 1) * j.out_stride;
    }
    constexpr int U = 8;  // loads of U chunks issued before their dependent updates
    for (int i0 = 0; i0 < a.nch; i0 += U) {
        float4 v[U];
#pragma unroll
        for (int k = 0; k < U; ++k)
            v[k] = i0 + k < a.nch ? __ldcg(reinterpret_cast<const float4 *>(in + (long long)k * sin))
                                  : make_float4(0, 0, 0, 0);
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const int it = i0 + k;
            if (it < a.nch) {
                *reinterpret_cast<float4 *>(out + (long long)k * sout) = R;
                float f = 1.f;
                if (a.gamma) {
                    const int ch = j.reverse ? a.nch - 1 - it : it;
                    f = gpow(lg, (float)(j.power * min(a.chunk, a.n - ch * a.chunk)));
                }
                R.x = f * R.x + v[k].x; R.y = f * R.y + v[k].y; R.z = f * R.z + v[k].z; R.w = f * R.w + v[k].w;
            }
        }
        in += U * sin;
        out += U * sout;
    }
    if (j.fin) *reinterpret_cast<float4 *>(j.fin + (size_t)u * j.count + e) = R;
}

}  // namespace
}  // namespace scantc

cudaError_t chunktc::chunk_prefix(const PrefixArgs &a, cudaStream_t st) {
    using namespace scantc;
    int mx = 0;
    for (int i = 0; i < a.njobs; ++i) mx = max(mx, (a.job[i].count / 4 + kPrefixThreads - 1) / kPrefixThreads);
    dim3 grid((unsigned)(a.units * mx), (unsigned)a.njobs);
    chunk_prefix_kernel<<<grid, kPrefixThreads, 0, st>>>(a);
    return cudaGetLastError();
}

namespace scantc {
namespace {

// D (+)= A B with A, B fp32 given as hi + lo tiles: hi.hi + hi.lo + lo.hi
__device__ __forceinline__ void mma3_km(uint32_t d, const uint8_t *ah, const uint8_t *al, const uint8_t *bh,
                                        const uint8_t *bl, bool acc) {
    mma_km(d, ah, bh, acc);
    mma_km(d, ah, bl, true);
    mma_km(d, al, bh, true);
}

// ---- backward increments: X_loc <- S_p C_q + X_loc,  O_loc <- O_loc + Lam_n W (in place)
enum { B_SH, B_SL, B_CH, B_CL, B_LH, B_LL, B_WH, B_WL, B_N };

__global__ void __launch_bounds__(kTc, 2) bwd_incr_tc_kernel(const __grid_constant__ BwdArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    Ctx x;
    if (!setup(x, smem_raw, B_N, a.err)) return;
    const int nch = (a.n + 63) / 64, u = blockIdx.x / nch, ch = blockIdx.x % nch;
    const bwd::BwdWs ws{64, 64};
    float *lc = a.workspace + ((size_t)u * nch + ch) * ws.loc_floats();
    const float *so =
        a.workspace + (size_t)a.B * a.H * nch * ws.loc_floats() + ((size_t)u * nch + ch) * ws.st_floats();
    {
        const float *ss[4] = {so + ws.o_sp(), lc + ws.o_cq(), so + ws.o_lam(), lc + ws.o_w()};
        uint8_t *hi[4] = {x.tile(B_SH), x.tile(B_CH), x.tile(B_LH), x.tile(B_WH)};
        uint8_t *lo[4] = {x.tile(B_SL), x.tile(B_CL), x.tile(B_LL), x.tile(B_WL)};
        load_tiles_hilo<4>(ss, hi, lo);
    }
    x.publish();
    // the addends of the epilogue, fetched while the products run
    const size_t ro = (size_t)x.row * 64 + x.c0;
    float xa[16], oa[16];
    ld_row16(lc + ws.o_xloc() + ro, xa);
    ld_row16(lc + ws.o_oloc() + ro, oa);
    do {
        // S_p C_q (rows = key feature), Lam_n W (rows = key feature)
        if (x.tid == 0) {
            mma3_km(x.tb + 0, x.tile(B_SH), x.tile(B_SL), x.tile(B_CH), x.tile(B_CL), false);
            mma3_km(x.tb + 64, x.tile(B_LH), x.tile(B_LL), x.tile(B_WH), x.tile(B_WL), false);
        }
        x.commit();
        if (!x.wait()) break;
        float r[16];
        x.ld_row(0, r);
#pragma unroll
        for (int i = 0; i < 16; ++i) r[i] += xa[i];
        st_row16(lc + ws.o_xloc() + ro, r);
        x.ld_row(64, r);
#pragma unroll
        for (int i = 0; i < 16; ++i) r[i] += oa[i];
        st_row16(lc + ws.o_oloc() + ro, r);
    } while (false);
    teardown(x);
}

// ---- third-order increments: T_loc <- T_B + S^K_p (M^QP_B + S^Q_B P_p) + M^KQ_B P_p (in place)
enum { T_QH, T_QL, T_MH, T_ML, T_KH, T_KL, T_PH, T_PL, T_XH, T_XL, T_N };

__global__ void __launch_bounds__(kTc, 2) fwd3_incr_tc_kernel(const __grid_constant__ Fwd3Args a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    Ctx x;
    if (!setup(x, smem_raw, T_N, a.err)) return;
    const int nch = (a.n + 63) / 64, u = blockIdx.x / nch, ch = blockIdx.x % nch;
    const fwd3::Ws3 ws{64, 64};
    float *lc = a.workspace + ((size_t)u * nch + ch) * ws.loc_floats();
    const float *so =
        a.workspace + (size_t)a.B * a.H * nch * ws.loc_floats() + ((size_t)u * nch + ch) * ws.st_floats();
    {
        const float *ss[4] = {lc + ws.o_sq(), lc + ws.o_mkq(), so + ws.s_sk(), so + ws.s_p()};
        uint8_t *hi[4] = {x.tile(T_QH), x.tile(T_MH), x.tile(T_KH), x.tile(T_PH)};
        uint8_t *lo[4] = {x.tile(T_QL), x.tile(T_ML), x.tile(T_KL), x.tile(T_PL)};
        load_tiles_hilo<4>(ss, hi, lo);
    }
    x.publish();
    const size_t ro = (size_t)x.row * 64 + x.c0;
    float r[16], qa[16], ta[16];  // epilogue addends M^QP_B and T_B, fetched while the products run
    ld_row16(lc + ws.o_mqp() + ro, qa);
    ld_row16(lc + ws.o_t() + ro, ta);
    do {
        // S^Q_B P_p, M^KQ_B P_p
        if (x.tid == 0) {
            mma3_km(x.tb + 0, x.tile(T_QH), x.tile(T_QL), x.tile(T_PH), x.tile(T_PL), false);
            mma3_km(x.tb + 64, x.tile(T_MH), x.tile(T_ML), x.tile(T_PH), x.tile(T_PL), false);
        }
        x.commit();
        if (!x.wait()) break;
        // X = M^QP_B + S^Q_B P_p as hi + lo tiles (rows = contraction index of S^K_p X)
        x.ld_row(0, r);
        {
            float h[16], l[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float s = r[i] + qa[i];
                h[i] = __bfloat162float(__float2bfloat16_rn(s));
                l[i] = s - h[i];
            }
            tile_store_row16(x.tile(T_XH), 64, x.row, x.c0, h);
            tile_store_row16(x.tile(T_XL), 64, x.row, x.c0, l);
        }
        x.publish();
        // + S^K_p X into the second accumulator
        if (x.tid == 0) mma3_km(x.tb + 64, x.tile(T_KH), x.tile(T_KL), x.tile(T_XH), x.tile(T_XL), true);
        x.commit();
        if (!x.wait()) break;
        x.ld_row(64, r);
#pragma unroll
        for (int i = 0; i < 16; ++i) r[i] += ta[i];
        st_row16(lc + ws.o_t() + ro, r);
    } while (false);
    teardown(x);
}

constexpr size_t kBwdIncrSmem = B_N * TILE + 64, kFwd3IncrSmem = T_N * TILE + 64;

}  // namespace

// Backward: S_p and Lam_n, the increments, then X_p and Om_n.
cudaError_t bwd_scan(const BwdArgs &a, cudaStream_t st) {
    const int nch = (a.n + 63) / 64, units = a.B * a.H;
    const bwd::BwdWs ws{64, 64};
    float *loc = a.workspace, *sta = a.workspace + (size_t)units * nch * ws.loc_floats();
    const float *gamma = (a.flags & HLA_DECAY) ? a.gamma : nullptr;
    PrefixArgs p{};
    p.njobs = 2; p.units = units; p.nch = nch; p.n = a.n; p.chunk = 64; p.H = a.H; p.gamma = gamma;
    p.job[0] = PrefixJob{loc, ws.loc_floats(), ws.o_sloc(), sta, ws.st_floats(), ws.o_sp(), nullptr, nullptr, 64 * 64, 0, 1};
    p.job[1] = PrefixJob{loc, ws.loc_floats(), ws.o_lloc(), sta, ws.st_floats(), ws.o_lam(), nullptr, nullptr, 64 * 64, 1, 2};
    cudaError_t e = chunk_prefix(p, st);
    if (e != cudaSuccess) return e;
    if ((e = cudaFuncSetAttribute(bwd_incr_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)kBwdIncrSmem)) != cudaSuccess)
        return e;
    bwd_incr_tc_kernel<<<units * nch, kTc, kBwdIncrSmem, st>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    p.job[0] = PrefixJob{loc, ws.loc_floats(), ws.o_xloc(), sta, ws.st_floats(), ws.o_xp(), nullptr, nullptr, 64 * 64, 0, 2};
    p.job[1] = PrefixJob{loc, ws.loc_floats(), ws.o_oloc(), sta, ws.st_floats(), ws.o_om(), nullptr, nullptr, 64 * 64, 1, 1};
    return chunk_prefix(p, st);
}

// Third order: S^K_p and P_p (and the final S^K, P), the increments, then T_p (and the final T).
cudaError_t fwd3_scan(const Fwd3Args &a, cudaStream_t st) {
    const int nch = (a.n + 63) / 64, units = a.B * a.H;
    const fwd3::Ws3 ws{64, 64};
    float *loc = a.workspace, *sta = a.workspace + (size_t)units * nch * ws.loc_floats();
    PrefixArgs p{};
    p.njobs = 2; p.units = units; p.nch = nch; p.n = a.n; p.chunk = 64; p.H = a.H; p.gamma = nullptr;
    p.job[0] = PrefixJob{loc, ws.loc_floats(), ws.o_sk(), sta, ws.st_floats(), ws.s_sk(), a.sin_S, a.sout_S, 64 * 64, 0, 1};
    p.job[1] = PrefixJob{loc, ws.loc_floats(), ws.o_p(), sta, ws.st_floats(), ws.s_p(), a.sin_P, a.sout_P, 64 * 64, 0, 1};
    cudaError_t e = chunk_prefix(p, st);
    if (e != cudaSuccess) return e;
    if ((e = cudaFuncSetAttribute(fwd3_incr_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)kFwd3IncrSmem)) != cudaSuccess)
        return e;
    fwd3_incr_tc_kernel<<<units * nch, kTc, kFwd3IncrSmem, st>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    p.njobs = 1;
    p.job[0] = PrefixJob{loc, ws.loc_floats(), ws.o_t(), sta, ws.st_floats(), ws.s_t(), a.sin_T, a.sout_T, 64 * 64, 0, 1};
    return chunk_prefix(p, st);
}

}  // namespace scantc
}  // namespace hla
