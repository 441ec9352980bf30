// hla_chunk_tc.cuh -- shared machinery of the per-chunk tensor-core kernels (third
// order, backward): one CTA of 8 warps (two per TMEM lane quadrant) per chunk of 64
// tokens, 64 x 64 bf16 operand tiles in 128-byte-swizzled shared memory (the bf16 inputs
// brought in by TMA, the fp32 states converted by the threads), 64-row tcgen05.mma groups
// issued by thread 0 into 64-column TMEM accumulators, bounded mbarrier waits that raise
// the sticky status flag instead of hanging.
#pragma once
#include "hla_internal.h"
#include "hla_tmap.h"

namespace hla {
namespace chunktc {

// Tensor maps of the bf16 inputs a chunk kernel loads: [units][n][64], boxes of 64 token
// rows of one unit (q and the output gradient over query heads, k and v over key/value heads).
struct ChunkMaps {
    CUtensorMap q, k, v, g;
};
// false if the CUDA driver's tensor-map encoder is unavailable or rejects a tensor; g may be null
inline bool chunk_maps(ChunkMaps &m, const void *q, const void *k, const void *v, const void *g, int n, int units,
                       int kv_units) {
    return tc::encode_3d(&m.q, q, 64, n, units, 64) && tc::encode_3d(&m.k, k, 64, n, kv_units, 64) &&
           tc::encode_3d(&m.v, v, 64, n, kv_units, 64) && (!g || tc::encode_3d(&m.g, g, 64, n, units, 64));
}

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
    uint64_t *bar, *tbar;  // MMA completion; TMA tile arrival
    uint32_t tb, ph, tph;
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

// Block setup shared by both kernels: barrier, TMEM allocation.  Returns false if
// the shared window is not 1024-byte aligned (then nothing was allocated).
__device__ bool setup(Ctx &x, uint8_t *smem, int ntiles, unsigned *err) {
    x.base = smem;
    x.bar = reinterpret_cast<uint64_t *>(smem + ntiles * TILE);
    x.tbar = reinterpret_cast<uint64_t *>(smem + ntiles * TILE + 16);
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
    x.tph = 0;
    x.err = err;
    if (x.tid == 0) {
        *bad = (smem_u32(smem) & 1023u) != 0;
        mbar_init(x.bar, 1);
        mbar_init(x.tbar, 1);
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

// N tiles of 64 token rows by TMA (thread 0 issues): map m[i] at (feature 0, token t0,
// unit u[i]) into tile d[i]; rows past the sequence arrive as zeros.  Wait with tma_wait.
template <int N>
__device__ __forceinline__ void tma_issue(const Ctx &x, const CUtensorMap *const (&m)[N], const int (&u)[N], int t0,
                                          uint8_t *const (&d)[N]) {
    if (x.tid == 0) {
        mbar_expect_tx(x.tbar, N * TILE);
#pragma unroll
        for (int i = 0; i < N; ++i) tma_load_3d(d[i], m[i], x.tbar, 0, t0, u[i]);
    }
}
// Every thread: bounded wait for the tiles of the last tma_issue; false (uniform) if it expired.
__device__ __forceinline__ bool tma_wait(Ctx &x) {
    const bool ok = mbar_wait(x.tbar, x.tph, x.err);
    x.tph ^= 1u;
    return !__syncthreads_or(!ok);
}
// A bf16 tile with row r scaled by w[r] (zero for r >= L) into another tile.
__device__ __forceinline__ void scale_tile(const uint8_t *src, int L, const float *w, uint8_t *dst) {
    for (int e = threadIdx.x; e < 64 * 4; e += kTc) {
        const int r = e >> 2, c = (e & 3) * 16;
        const float s = r < L ? w[r] : 0.f;
        float a[8], b[8], v[16];
        tile_load_row8(src, 64, r, c, a);
        tile_load_row8(src, 64, r, c + 8, b);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            v[i] = s * a[i];
            v[8 + i] = s * b[i];
        }
        tile_store_row16(dst, 64, r, c, v);
    }
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
