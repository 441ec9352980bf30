// hla_common.cuh -- device helpers shared by the HLA kernels: inline-PTX
// wrappers for mbarriers, TMA tile loads, tcgen05 (TMEM allocation, MMA,
// TMEM loads/stores), the shared-memory operand layout, and bounded waits.
//
// Shared-memory operand layout ("tile"): a rows x cols bf16 matrix stored as
// cols/64 column blocks, each block holding `rows` rows of 128 bytes with the
// 128-byte XOR swizzle (16-byte chunk j of row r sits at chunk j ^ (r % 8)).
// It is exactly what a TMA load with CU_TENSOR_MAP_SWIZZLE_128B and a 64-column
// box writes.  The same bytes serve as a K-major operand (contraction over the
// columns) or as an MN-major operand (contraction over the rows); only the
// matrix descriptor differs.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#define HLA_DEVICE __device__ __forceinline__

namespace hla {

// ---------------------------------------------------------------- error flag
// Sticky device-side status: set when a bounded wait expires.
enum : unsigned { DEV_OK = 0u, DEV_TIMEOUT = 1u };

// Upper bound on polls of a flag (cross-CTA waits) before the wait is declared failed.
// With the sleep in those loops this is several seconds, far beyond any legitimate wait.
constexpr uint32_t kWaitLimit = 1u << 24;
// Time limit of a barrier wait, in microseconds: far beyond any legitimate wait.
constexpr uint32_t kWaitLimitUs = 2000000u;
// Suspend hint of one barrier poll (ns): the polling thread sleeps in hardware until the
// phase completes or this time passes, so waiting warps take no issue slots.
constexpr uint32_t kSuspendNs = 1u << 20;

HLA_DEVICE uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
HLA_DEVICE uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier
HLA_DEVICE void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
HLA_DEVICE void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
HLA_DEVICE void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
// One poll: true once the phase with the given parity has completed; otherwise the
// thread may sleep up to `hint_ns` (or until the phase completes) before it returns false.
HLA_DEVICE bool mbar_try_wait(uint64_t *bar, uint32_t parity, uint32_t hint_ns = kSuspendNs) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}
// Bounded wait for the phase with the given parity to complete.  Returns false (and
// raises the sticky flag) if it does not within `limit_us` microseconds.
HLA_DEVICE bool mbar_wait(uint64_t *bar, uint32_t parity, unsigned *err, uint32_t limit_us = kWaitLimitUs) {
    const uint32_t hint = limit_us * 1000u < kSuspendNs ? limit_us * 1000u : kSuspendNs;
    if (mbar_try_wait(bar, parity, hint)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < (uint64_t)limit_us * 1000u) {
        if (mbar_try_wait(bar, parity, hint)) return true;
    }
    atomicOr(err, DEV_TIMEOUT);
    return false;
}

// ---------------------------------------------------------------- TMA
HLA_DEVICE void tma_prefetch_desc(const void *tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}
// 3-D tiled load (coordinates innermost first) completing on `bar`.
HLA_DEVICE void tma_load_3d(void *dst, const void *tmap, uint64_t *bar, int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
        "l"(tmap), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// 3-D tiled store of a shared-memory tile (coordinates innermost first); rows
// outside the tensor are not written.  Tracked by the issuing thread's bulk groups.
HLA_DEVICE void tma_store_3d(const void *src, const void *tmap, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(tmap),
                 "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}
HLA_DEVICE void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until the issuing thread's bulk stores have read their shared-memory source ...
HLA_DEVICE void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// ... or have completed.
HLA_DEVICE void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Make generic-proxy shared-memory writes visible to the async proxy (tensor cores, TMA).
HLA_DEVICE void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// ---------------------------------------------------------------- tcgen05
HLA_DEVICE void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
HLA_DEVICE void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
HLA_DEVICE void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
HLA_DEVICE void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
HLA_DEVICE void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem], kind::f16 (bf16 inputs, fp32 accumulate).
HLA_DEVICE void umma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Warp-level forms: executed by all 32 lanes of a converged warp with warp-uniform
// operands; elect.sync picks the one lane that issues.  Keeping the whole warp on the
// issuing path lets the operands stay in uniform registers.
HLA_DEVICE void umma_f16_warp(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p, e;\n elect.sync _|e, 0xffffffff;\n setp.ne.b32 p, %4, 0;\n"
        " @e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
HLA_DEVICE void umma_commit_warp(uint64_t *bar) {
    asm volatile(
        "{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n"
        " @e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}\n" ::"r"(smem_u32(bar))
        : "memory");
}
// Arrive on `bar` once every previously issued tcgen05.mma of this thread completes.
HLA_DEVICE void umma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// 32 lanes x 16 columns of 32-bit words: thread l of the warp gets lane (base lane + l).
HLA_DEVICE void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
HLA_DEVICE void tmem_st16(uint32_t taddr, const float (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15]))
        : "memory");
}
// 16 lanes x 16 columns, two column groups: threads 0-15 read lanes base..base+15 at
// columns [c, c+16), threads 16-31 the same lanes at [c+OFF, c+OFF+16).  Suits
// accumulators with 64 rows, which use lanes 0-15 of each lane quadrant.
template <int OFF>
HLA_DEVICE void tmem_ld16x2(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.16x32bx2.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16], %17;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr), "n"(OFF));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
template <int OFF>
HLA_DEVICE void tmem_st16x2(uint32_t taddr, const float (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.16x32bx2.x16.b32 [%0], %1, {%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17};" ::"r"(
            taddr),
        "n"(OFF), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15]))
        : "memory");
}
HLA_DEVICE void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
HLA_DEVICE void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------- descriptors
// Shared-memory matrix descriptor (tcgen05 format): start address, leading and
// stride byte offsets (16-byte units), version 1, 128-byte swizzle.
HLA_DEVICE uint64_t make_sdesc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1u << 46;  // descriptor version for tcgen05
    d |= (uint64_t)2u << 61;  // SWIZZLE_128B
    return d;
}

// K-major operand (contraction over the tile's columns): rows of the tile are the
// M (or N) index.  `k0` is the first contraction column of this instruction (a
// multiple of 16).
HLA_DEVICE uint64_t desc_kmajor(const void *tile, int rows, int k0) {
    const uint32_t base = smem_u32(tile) + (uint32_t)(k0 >> 6) * (uint32_t)rows * 128u + (uint32_t)(k0 & 63) * 2u;
    return make_sdesc(base, 16u, 1024u);
}
// MN-major operand (contraction over the tile's rows): columns of the tile are the
// M (or N) index.  `k0` is the first contraction row of this instruction (a
// multiple of 16).  LBO = distance between 64-column blocks, SBO = 8 rows.
HLA_DEVICE uint64_t desc_mnmajor(const void *tile, int rows, int k0) {
    const uint32_t base = smem_u32(tile) + (uint32_t)k0 * 128u;
    return make_sdesc(base, (uint32_t)rows * 128u, 1024u);
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 D, dense.
// a_mn / b_mn: operand is MN-major.  M in {64,128}, N multiple of 8 (M=64) or 16.
__host__ __device__ constexpr uint32_t make_idesc(int M, int N, bool a_mn, bool b_mn) {
    return (1u << 4)                       // D format: f32
           | (1u << 7)                     // A format: bf16
           | (1u << 10)                    // B format: bf16
           | ((a_mn ? 1u : 0u) << 15)      // A major-ness
           | ((b_mn ? 1u : 0u) << 16)      // B major-ness
           | ((uint32_t)(N >> 3) << 17)    // N / 8
           | ((uint32_t)(M >> 4) << 24);   // M / 16
}

// ---------------------------------------------------------------- tile I/O
// Byte offset of element (r, c) inside a swizzled tile with `rows` rows.
HLA_DEVICE uint32_t tile_off(int rows, int r, int c) {
    return (uint32_t)(c >> 6) * (uint32_t)rows * 128u + (uint32_t)r * 128u +
           ((uint32_t)(((c & 63) >> 3) ^ (r & 7)) << 4) + (uint32_t)(c & 7) * 2u;
}
HLA_DEVICE uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}
// Write 16 consecutive fp32 values (columns c0..c0+15, c0 % 16 == 0) of row r as bf16.
HLA_DEVICE void tile_store_row16(uint8_t *tile, int rows, int r, int c0, const float (&v)[16]) {
    uint4 a, b;
    a.x = pack_bf16(v[0], v[1]);   a.y = pack_bf16(v[2], v[3]);
    a.z = pack_bf16(v[4], v[5]);   a.w = pack_bf16(v[6], v[7]);
    b.x = pack_bf16(v[8], v[9]);   b.y = pack_bf16(v[10], v[11]);
    b.z = pack_bf16(v[12], v[13]); b.w = pack_bf16(v[14], v[15]);
    *reinterpret_cast<uint4 *>(tile + tile_off(rows, r, c0)) = a;
    *reinterpret_cast<uint4 *>(tile + tile_off(rows, r, c0 + 8)) = b;
}
// Read 8 consecutive bf16 (columns c0..c0+7, c0 % 8 == 0) of row r as fp32.
HLA_DEVICE void tile_load_row8(const uint8_t *tile, int rows, int r, int c0, float (&v)[8]) {
    const uint4 u = *reinterpret_cast<const uint4 *>(tile + tile_off(rows, r, c0));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}
HLA_DEVICE float tile_load(const uint8_t *tile, int rows, int r, int c) {
    const uint16_t u = *reinterpret_cast<const uint16_t *>(tile + tile_off(rows, r, c));
    return __uint_as_float((uint32_t)u << 16);
}

// ---------------------------------------------------------------- TMEM row mapping
// Accumulator with M rows: which TMEM lane holds row r, and which row (if any)
// thread `tid` of a 128-thread group owns.  M = 128: row r in lane r.  M = 64:
// rows 16w..16w+15 in lanes 32w..32w+15 of lane quadrant w.
template <int M>
HLA_DEVICE int owned_row(int tid) {
    if constexpr (M == 128) {
        return tid;
    } else {
        const int l = tid & 31;
        return l < 16 ? (tid >> 5) * 16 + l : -1;
    }
}
// TMEM address of this warp's lane quadrant at column `col`.
HLA_DEVICE uint32_t tmem_warp_addr(uint32_t base, int warp, int col) {
    return base + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)col;
}

// ---------------------------------------------------------------- math helpers
// 2^y with the hardware approximation (PTX ex2.approx: relative error ~2^-22,
// 2^-inf = 0).
HLA_DEVICE float ex2_approx(float y) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(y));
    return r;
}
// g^x for x >= 0 with g in [0,1]; lg = log2(g) (may be -inf).  0^0 = 1.
HLA_DEVICE float gpow(float lg, float x) { return x == 0.f ? 1.f : ex2_approx(lg * x); }

// Per-call ordering of the CTAs of a forward launch through its workspace header.
// Header words 0-1 form one 64-bit word: the count of tickets taken (low half) and the
// call generation g (high half); word 2 counts finished CTAs in the one call that
// needs it.  Every CTA takes its ticket and g in one atomic, and the release flags of
// this call carry the tag g + 1, which a zero (never written) flag and every flag of an
// earlier call differ from.  The CTA that takes the last ticket starts generation g + 1
// at once: every ticket of this call is out, and the next launch on the workspace
// begins after this one ends, so no CTA clears anything when the call ends.  The tag
// 0xFFFFFFFF is the exception: that call keeps the header, and its last CTA to finish
// zeroes every flag and the header (generation 0), so a tag returns only after the
// flags have been cleared.
struct CallTicket {
    unsigned ticket, tag;
};
constexpr unsigned kTagWrap = 0xFFFFFFFFu;

// One thread per CTA.
HLA_DEVICE CallTicket take_ticket(unsigned *hdr) {
    unsigned long long *w = reinterpret_cast<unsigned long long *>(hdr);
    const unsigned long long old = atomicAdd(w, 1ull);
    CallTicket t;
    t.ticket = (unsigned)old;
    t.tag = (unsigned)(old >> 32) + 1u;
    if (t.ticket == gridDim.x - 1 && t.tag != kTagWrap) atomicExch(w, (unsigned long long)t.tag << 32);
    return t;
}

// End of the call with tag kTagWrap (a no-op for every other tag): the CTA that finishes
// last zeroes the flags and the header.  Every thread of the CTA calls this once the CTA
// has read its last flag; the last CTA's threads share the clearing stores.  fb may be null.
HLA_DEVICE void finish_call(unsigned *hdr, unsigned tag, unsigned *fa, unsigned *fb, int nflags,
                            volatile unsigned *s_last) {
    if (tag != kTagWrap) return;
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned done = atomicAdd(hdr + 2, 1u);
        __threadfence();
        *s_last = (done == gridDim.x - 1) ? 1u : 0u;
    }
    __syncthreads();
    if (*s_last) {
        for (int i = threadIdx.x; i < nflags; i += blockDim.x) {
            fa[i] = 0u;
            if (fb) fb[i] = 0u;
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            __threadfence();
            *reinterpret_cast<unsigned long long *>(hdr) = 0ull;
            hdr[2] = 0u;
            __threadfence();
        }
    }
}

}  // namespace hla
