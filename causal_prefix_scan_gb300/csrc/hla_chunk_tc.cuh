// hla_chunk_tc.cuh -- shared machinery of the per-chunk tensor-core kernels (third
// order, backward): one CTA of 8 warps (two per TMEM lane quadrant) per chunk of 64
// tokens, 64 x 64 bf16 operand tiles in 128-byte-swizzled shared memory, 64-row
// tcgen05.mma groups issued by thread 0 into 64-column TMEM accumulators, bounded
// mbarrier waits that raise the sticky status flag instead of hanging.
#pragma once
#include "hla_internal.h"

namespace hla {
namespace chunktc {

// One elementwise scan over the chunks of every pair: out[ch] = R, R = f_ch R + in[ch],
// f_ch = g^{power * L_ch} (1 without decay), in chunk order (reverse: last chunk first).
struct PrefixJob {
    const float *in;
    size_t in_stride, in_off;  // element e of chunk ch of pair u at in[(u * nch + ch) * in_stride + in_off + e]
    float *out;
    size_t out_stride, out_off;
    const float *init;  // [units][count] or null (zeros)
    float *fin;         // [units][count] or null
    int count, reverse, power;
};

struct PrefixArgs {
    PrefixJob job[2];
    int njobs, units, nch, n, chunk, H;
    const float *gamma;  // per head, or null (no decay)
};

// Launches the elementwise scans of `a` (hla_scan_tc.cu).
cudaError_t chunk_prefix(const PrefixArgs &a, cudaStream_t st);

namespace {

constexpr int kTc = 256;
constexpr int N64 = 64;
constexpr int TILE = 64 * 64 * 2;  // one bf16 64 x 64 swizzled tile
constexpr uint32_t kCols = 256;    // TMEM columns: four 64-column accumulators

struct Ctx {
    uint8_t *base;
    uint64_t *bar;
    uint32_t tb, ph;
    int tid, warp, lane, quad, half;
    int row, c0;  // the accumulator row this thread reads and its first of 16 columns
    unsigned *err;

    __device__ uint8_t *tile(int i) const { return base + i * TILE; }
    __device__ uint32_t taddr(uint32_t slot, int col) const {
        return tb + slot + ((uint32_t)(32 * quad) << 16) + (uint32_t)col;
    }
    // 16 columns [c0, c0 + 16) of row `row` of the 64-row accumulator at `slot`
    __device__ void ld_row(uint32_t slot, float (&v)[16]) const {
        tmem_ld16x2<16>(taddr(slot, half * 32), v);
        tmem_wait_ld();
    }
    // shared-memory and TMEM writes of all threads visible to the MMAs issued next
    __device__ void publish() const {
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }
    __device__ void commit() const {
        if (tid == 0) umma_commit(bar);
    }
    // false: the bounded wait expired (status flag raised); uniform across the CTA
    __device__ bool wait() {
        const bool ok = mbar_wait(bar, ph, err);
        ph ^= 1u;
        tc_fence_after();
        return !__syncthreads_or(!ok);
    }
};

// ---- MMA groups (thread 0).  Every operand is one 64 x 64 tile.
// A K-major [64 x 64] (rows = M), B K-major [N x 64]
__device__ __forceinline__ void mma_kk(uint32_t d, const uint8_t *a, const uint8_t *b, bool acc) {
    constexpr uint32_t id = make_idesc(64, N64, false, false);
    const uint64_t da = make_sdesc(smem_u32(a), 16u, 1024u), db = make_sdesc(smem_u32(b), 16u, 1024u);
#pragma unroll
    for (int k = 0; k < 64; k += 16) {
        const uint32_t kk = ((uint32_t)k * 2u) >> 4;
        umma_f16(d, da + kk, db + kk, id, (acc || k > 0) ? 1u : 0u);
    }
}
// A K-major [64 x 64], B MN-major [64 (contraction) x N]
__device__ __forceinline__ void mma_km(uint32_t d, const uint8_t *a, const uint8_t *b, bool acc) {
    constexpr uint32_t id = make_idesc(64, N64, false, true);
    const uint64_t da = make_sdesc(smem_u32(a), 16u, 1024u), db = make_sdesc(smem_u32(b), 64u * 128u, 1024u);
#pragma unroll
    for (int k = 0; k < 64; k += 16)
        umma_f16(d, da + (((uint32_t)k * 2u) >> 4), db + (uint32_t)(k * 8), id, (acc || k > 0) ? 1u : 0u);
}
// A MN-major [64 (contraction) x 64] read as 64 x 64, B MN-major [64 (contraction) x N]
__device__ __forceinline__ void mma_mm(uint32_t d, const uint8_t *a, const uint8_t *b, bool acc = false) {
    constexpr uint32_t id = make_idesc(64, N64, true, true);
    const uint64_t da = make_sdesc(smem_u32(a), 64u * 128u, 1024u), db = make_sdesc(smem_u32(b), 64u * 128u, 1024u);
#pragma unroll
    for (int k = 0; k < 64; k += 16)
        umma_f16(d, da + (uint32_t)(k * 8), db + (uint32_t)(k * 8), id, (acc || k > 0) ? 1u : 0u);
}

// L rows of 64 bf16 (row-major) into a swizzled tile; rows >= L are zero.
__device__ __forceinline__ void load_tile_bf16(const __nv_bfloat16 *src, int L, uint8_t *tile) {
    for (int e = threadIdx.x; e < 64 * 8; e += kTc) {
        const int r = e >> 3, c = (e & 7) * 8;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (r < L) v = *reinterpret_cast<const uint4 *>(src + (size_t)r * 64 + c);
        *reinterpret_cast<uint4 *>(tile + tile_off(64, r, c)) = v;
    }
}
// A 64 x 64 fp32 matrix (row-major) into bf16 hi and lo tiles (hi + lo = the value to
// about 2^-17 relative).
__device__ __forceinline__ void load_tile_hilo(const float *src, uint8_t *hi, uint8_t *lo) {
    for (int e = threadIdx.x; e < 64 * 4; e += kTc) {
        const int r = e >> 2, c = (e & 3) * 16;
        float v[16], h[16], l[16];
#pragma unroll
        for (int i = 0; i < 16; i += 4) {
            const float4 x = *reinterpret_cast<const float4 *>(src + (size_t)r * 64 + c + i);
            v[i] = x.x; v[i + 1] = x.y; v[i + 2] = x.z; v[i + 3] = x.w;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            h[i] = __bfloat162float(__float2bfloat16_rn(v[i]));
            l[i] = v[i] - h[i];
        }
        tile_store_row16(hi, 64, r, c, h);
        tile_store_row16(lo, 64, r, c, l);
    }
}

// Block setup shared by both kernels: barrier, TMEM allocation.  Returns false if
// the shared window is not 1024-byte aligned (then nothing was allocated).
__device__ bool setup(Ctx &x, uint8_t *smem, int ntiles, unsigned *err) {
    x.base = smem;
    x.bar = reinterpret_cast<uint64_t *>(smem + ntiles * TILE);
    uint32_t *tptr = reinterpret_cast<uint32_t *>(smem + ntiles * TILE + 8);
    int *bad = reinterpret_cast<int *>(smem + ntiles * TILE + 12);
    x.tid = threadIdx.x;
    x.warp = x.tid >> 5;
    x.lane = x.tid & 31;
    x.quad = x.warp & 3;
    x.half = x.warp >> 2;
    x.row = 16 * x.quad + (x.lane & 15);
    x.c0 = x.half * 32 + (x.lane >> 4) * 16;
    x.ph = 0;
    x.err = err;
    if (x.tid == 0) {
        *bad = (smem_u32(smem) & 1023u) != 0;
        mbar_init(x.bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (*bad) {
        if (x.tid == 0) atomicOr(err, DEV_TIMEOUT);
        return false;
    }
    if (x.warp == 0) {
        tmem_alloc(tptr, kCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    x.tb = *tptr;
    return true;
}

__device__ void teardown(const Ctx &x) {
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (x.warp == 0) tmem_dealloc(x.tb, kCols);
}

// 16 accumulator values of this thread's row into a tile, lower triangle kept
__device__ __forceinline__ void store_tril(const Ctx &x, uint8_t *tile, float (&v)[16]) {
#pragma unroll
    for (int i = 0; i < 16; ++i)
        if (x.c0 + i > x.row) v[i] = 0.f;
    tile_store_row16(tile, 64, x.row, x.c0, v);
}

// N tiles of L rows of 64 bf16 each (row-major) into swizzled tiles, rows >= L zero;
// every global load of the batch is issued before the first shared store.
template <int N>
__device__ __forceinline__ void load_tiles_bf16(const __nv_bfloat16 *const (&src)[N], int L, uint8_t *const (&tile)[N]) {
    uint4 v[N][2];
#pragma unroll
    for (int t = 0; t < N; ++t)
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            const int e = threadIdx.x + p * kTc, r = e >> 3, c = (e & 7) * 8;
            v[t][p] = r < L ? *reinterpret_cast<const uint4 *>(src[t] + (size_t)r * 64 + c) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
    for (int t = 0; t < N; ++t)
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            const int e = threadIdx.x + p * kTc, r = e >> 3, c = (e & 7) * 8;
            *reinterpret_cast<uint4 *>(tile[t] + tile_off(64, r, c)) = v[t][p];
        }
}
// N fp32 64 x 64 matrices (row-major) into bf16 hi and lo tiles; all loads first.
template <int N>
__device__ __forceinline__ void load_tiles_hilo(const float *const (&src)[N], uint8_t *const (&hi)[N],
                                                uint8_t *const (&lo)[N]) {
    const int r = threadIdx.x >> 2, c = (threadIdx.x & 3) * 16;  // kTc == 256: one row segment each
    float4 v[N][4];
#pragma unroll
    for (int t = 0; t < N; ++t)
#pragma unroll
        for (int i = 0; i < 4; ++i) v[t][i] = *reinterpret_cast<const float4 *>(src[t] + (size_t)r * 64 + c + 4 * i);
#pragma unroll
    for (int t = 0; t < N; ++t) {
        float h[16], l[16];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float x[4] = {v[t][i].x, v[t][i].y, v[t][i].z, v[t][i].w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                h[4 * i + k] = __bfloat162float(__float2bfloat16_rn(x[k]));
                l[4 * i + k] = x[k] - h[4 * i + k];
            }
        }
        tile_store_row16(hi[t], 64, r, c, h);
        tile_store_row16(lo[t], 64, r, c, l);
    }
}

// L rows of 64 bf16 scaled by w[r] into a swizzled tile (bf16 after scaling); rows >= L zero.
__device__ __forceinline__ void load_tile_scaled(const __nv_bfloat16 *src, int L, const float *w, uint8_t *tile) {
    for (int e = threadIdx.x; e < 64 * 4; e += kTc) {
        const int r = e >> 2, c = (e & 3) * 16;
        float v[16];
        const float s = r < L ? w[r] : 0.f;
#pragma unroll
        for (int i = 0; i < 16; i += 8) {
            uint4 u = make_uint4(0, 0, 0, 0);
            if (r < L) u = *reinterpret_cast<const uint4 *>(src + (size_t)r * 64 + c + i);
            const uint32_t p[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                v[i + 2 * j] = s * __uint_as_float(p[j] << 16);
                v[i + 2 * j + 1] = s * __uint_as_float(p[j] & 0xFFFF0000u);
            }
        }
        tile_store_row16(tile, 64, r, c, v);
    }
}
// 16 accumulator values of this thread's row into a tile, lower triangle kept and
// weighted by gp[step * (row - col)] (powers of the decay factor)
__device__ __forceinline__ void store_tril_decay(const Ctx &x, uint8_t *tile, float (&v)[16], const float *gp, int step) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int dlt = x.row - (x.c0 + i);
        v[i] = dlt >= 0 ? gp[step * dlt] * v[i] : 0.f;
    }
    tile_store_row16(tile, 64, x.row, x.c0, v);
}
// 16 consecutive fp32 values from global memory
__device__ __forceinline__ void ld_row16(const float *src, float (&v)[16]) {
#pragma unroll
    for (int i = 0; i < 16; i += 4) {
        const float4 x = *reinterpret_cast<const float4 *>(src + i);
        v[i] = x.x; v[i + 1] = x.y; v[i + 2] = x.z; v[i + 3] = x.w;
    }
}
// 16 fp32 values as bf16 to global memory (two 16-byte stores)
__device__ __forceinline__ void st_row16_bf16(__nv_bfloat16 *dst, const float (&v)[16]) {
    uint4 p0, p1;
    p0.x = pack_bf16(v[0], v[1]);   p0.y = pack_bf16(v[2], v[3]);
    p0.z = pack_bf16(v[4], v[5]);   p0.w = pack_bf16(v[6], v[7]);
    p1.x = pack_bf16(v[8], v[9]);   p1.y = pack_bf16(v[10], v[11]);
    p1.z = pack_bf16(v[12], v[13]); p1.w = pack_bf16(v[14], v[15]);
    reinterpret_cast<uint4 *>(dst)[0] = p0;
    reinterpret_cast<uint4 *>(dst)[1] = p1;
}

__device__ __forceinline__ void st_row16(float *dst, const float (&v)[16]) {
#pragma unroll
    for (int i = 0; i < 16; i += 4) *reinterpret_cast<float4 *>(dst + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
}

}  // namespace
}  // namespace chunktc
}  // namespace hla
