// common.cuh — sm_103a device helpers shared by the kernels: bf16 epilogue,
// mbarrier waits with a time limit, TMA tile loads, tcgen05 / TMEM, clusters.
//
// Every spin-wait in this library goes through mbar_wait(), which gives up
// after a wall-clock limit (%globaltimer), records the first failure in the
// device status word, and returns false so the kernel can unwind to its common
// exit path instead of hanging the GPU.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "bf16_linear.h"

namespace bf16l {

// ---------------------------------------------------------------------------
// Status word: the first kernel wait that gives up stores its code there.
// code = (uint8)BF16L_ETIMEOUT | site << 8.  Kernels receive its address as a
// parameter (the word itself is defined once, in api.cu).
// ---------------------------------------------------------------------------

// Wait sites (recorded in the status word).
enum WaitSite : int32_t {
    kSiteFull = 1,       // MMA issuer waiting for a TMA stage
    kSiteEmpty = 2,      // TMA producer waiting for a free stage
    kSiteAccum = 3,      // epilogue waiting for the accumulator
    kSiteTmemEmpty = 4,  // MMA issuer waiting for the epilogue to drain TMEM
    kSiteDrain = 5,      // exit path draining copies still in flight
    kSiteSelftest = 6,   // bf16_linear_selftest_wait
    kSiteRecv = 7,       // split-K owner waiting for its peers' partials
    kSiteStage = 8,      // dot-product CTA waiting for its copy of x
    kSitePairTmem = 9,   // the two CTAs of a pair got different TMEM addresses (gave up before any MMA)
    kSiteScale = 10      // MXFP8 tile: scale-staging warps waiting for a free ring slot
};

// Default limit for one wait: 1 s of wall-clock time.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

__host__ __device__ constexpr int32_t timeout_code(int32_t site) {
    return (int32_t)((uint32_t)(uint8_t)(int8_t)BF16L_ETIMEOUT | ((uint32_t)site << 8));
}

__device__ __forceinline__ void record_timeout(int32_t *status, int32_t site) {
    atomicCAS(status, 0, timeout_code(site));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------------------
// bf16 epilogue: fp32 -> bf16 round-to-nearest-even (CUDA's conversion).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// acc += x.lo * w.lo, then acc += x.hi * w.hi, for two packed bf16 pairs, with
// the fp32-accumulating mixed-precision fma (sm_100+).  A product of two bf16
// values is exact in fp32, so each step equals fmaf(float(x), float(w), acc)
// bit for bit; only the widening instructions go away.
__device__ __forceinline__ float fma2_bf16(uint32_t x2, uint32_t w2, float acc) {
    asm("{\n\t.reg .b16 xl, xh, wl, wh;\n\t"
        "mov.b32 {xl, xh}, %1;\n\t"
        "mov.b32 {wl, wh}, %2;\n\t"
        "fma.rn.f32.bf16 %0, xl, wl, %0;\n\t"
        "fma.rn.f32.bf16 %0, xh, wh, %0;\n\t}"
        : "+f"(acc)
        : "r"(x2), "r"(w2));
    return acc;
}
__device__ __forceinline__ float bf16_to_f32(uint16_t v) { return __uint_as_float((uint32_t)v << 16); }
__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
    __nv_bfloat16 b = __float2bfloat16_rn(f);
    return *reinterpret_cast<uint16_t *>(&b);
}

// Output element stores for the two output types: bf16 (RNE) and fp32 (the
// router-logits variant).  `four` needs 4-element alignment of the index;
// `eight` needs 8-element alignment.
template <typename OutT>
struct OutStore;

template <>
struct OutStore<uint16_t> {
    static __device__ __forceinline__ void one(uint16_t *p, float v) { *p = f32_to_bf16(v); }
    static __device__ __forceinline__ void four(uint16_t *p, float a, float b, float c, float d) {
        uint2 pk;
        pk.x = pack_bf16x2(a, b);
        pk.y = pack_bf16x2(c, d);
        *reinterpret_cast<uint2 *>(p) = pk;
    }
    static __device__ __forceinline__ void eight(uint16_t *p, const float *v) {
        uint4 pk;
        pk.x = pack_bf16x2(v[0], v[1]);
        pk.y = pack_bf16x2(v[2], v[3]);
        pk.z = pack_bf16x2(v[4], v[5]);
        pk.w = pack_bf16x2(v[6], v[7]);
        *reinterpret_cast<uint4 *>(p) = pk;
    }
};

template <>
struct OutStore<float> {
    static __device__ __forceinline__ void one(float *p, float v) { *p = v; }
    static __device__ __forceinline__ void four(float *p, float a, float b, float c, float d) {
        *reinterpret_cast<float4 *>(p) = make_float4(a, b, c, d);
    }
    static __device__ __forceinline__ void eight(float *p, const float *v) {
        reinterpret_cast<float4 *>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
        reinterpret_cast<float4 *>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
    }
};

// floor(a * b / c) for 0 <= a, 0 <= b <= c and 0 < c < 65536, exactly, in
// 32-bit arithmetic (a 64-bit division is a long software routine, and these
// bounds sit in front of a kernel's first weight load): with a = q c + r,
// a b / c = q b + r b / c, where q b <= a and r b < c * c.
__device__ __forceinline__ int mul_div(int a, int b, int c) {
    const unsigned ua = (unsigned)a, ub = (unsigned)b, uc = (unsigned)c;
    const unsigned q = ua / uc, r = ua - q * uc;
    return (int)(q * ub + (r * ub) / uc);
}

// ---------------------------------------------------------------------------
// Shared-memory addresses and mbarriers.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make mbarrier initialisation visible to the async proxy (TMA, tcgen05) and the cluster.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar_addr, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar_addr), "r"(parity)
        : "memory");
    return ok != 0;
}

// As mbar_try_wait, with acquire semantics at cluster scope (for data other
// CTAs wrote with st.async).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar_addr, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar_addr), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_wait_cluster(uint64_t *bar, uint32_t parity, int32_t *status, int32_t site,
                                                  uint64_t limit_ns = kWaitLimitNs) {
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait_cluster(a, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait_cluster(a, parity)) return true;
        if (globaltimer_ns() - t0 > limit_ns) {
            record_timeout(status, site);
            return false;
        }
    }
}

// Wait until the phase with the given parity has completed, for at most
// limit_ns.  Returns false (after recording the site) when the limit passes.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, int32_t *status, int32_t site,
                                          uint64_t limit_ns = kWaitLimitNs) {
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait(a, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(a, parity)) return true;
        if (globaltimer_ns() - t0 > limit_ns) {
            record_timeout(status, site);
            return false;
        }
    }
}

// ---------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor) tile loads into this CTA's shared memory.
// c0 is the innermost (K) coordinate in elements, c1 the row coordinate.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar, int32_t c0,
                                            int32_t c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
        : "memory");
}

// Three-dimensional tile load (c0 innermost).  With the chunked weight/activation
// maps (make_tmap_bf16_chunks: {64 elements, rows, K / 64 chunks}) one box
// brings kc consecutive 64-wide K chunks of box_rows rows, laid out in shared
// memory as kc ordinary 128-byte-swizzled chunk tiles one after the other.
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, uint64_t *bar, int32_t c0,
                                            int32_t c1, int32_t c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

__device__ __forceinline__ void tma_load_2d_hint(void *dst, const CUtensorMap *map, uint64_t *bar, int32_t c0,
                                                 int32_t c1, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %5;"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1),
        "l"(policy)
        : "memory");
}

// Untiled bulk copy global -> this CTA's shared memory (both addresses 16-byte
// aligned, bytes a multiple of 16), completion counted on `bar`.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ---------------------------------------------------------------------------
// tcgen05: TMEM allocation, MMA, commit, loads.
// ---------------------------------------------------------------------------
// Whole warp: allocate `ncols` TMEM columns (power of two >= 32); address -> *dst (shared).
__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor for a K-major bf16 tile stored as rows of
// 64 elements (128 bytes) in the 128-byte swizzle layout TMA writes with
// CU_TENSOR_MAP_SWIZZLE_128B: 8-row groups of 1024 bytes (stride byte offset),
// start address 1024-byte aligned.  Fields: start>>4 [0,14), leading byte
// offset>>4 [16,30) (unused for this layout), stride byte offset>>4 [32,46),
// descriptor version 1 [46,48), swizzle mode 2 = 128B [61,64).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major,
// N>>3 at bit 17, M>>4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int mma_m, int mma_n) {
    return (1u << 4)                      // D format: f32
           | (1u << 7)                    // A format: bf16
           | (1u << 10)                   // B format: bf16
           | ((uint32_t)(mma_n >> 3) << 17) | ((uint32_t)(mma_m >> 4) << 24);
}

// Instruction descriptor, kind::f8f6f4 with both operands e4m3 (format code 0):
// D fp32, K-major A and B, N>>3 at bit 17, M>>4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int mma_m, int mma_n) {
    return (1u << 4) | ((uint32_t)(mma_n >> 3) << 17) | ((uint32_t)(mma_m >> 4) << 24);
}

// One e4m3 MMA (K = 32 codes per instruction): D[tmem] (+)= A[smem] * B[smem]^T.
__device__ __forceinline__ void mma_e4m3(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// One MMA: D[tmem] (+)= A[smem] * B[smem]^T, issued by a single thread.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on `bar` once every tcgen05 op issued so far by this thread has completed.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 32 lanes x 32 bits, 16 consecutive columns: thread t of the warp gets lane
// (quarter base + t), columns [col, col+16).  The registers are not valid
// until tmem_ld_wait16() on the same array: that wait names them as in-out
// operands, so the compiler cannot read them before it.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait16(uint32_t (&r)[16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                   "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                   "+r"(r[14]), "+r"(r[15])
                 :
                 : "memory");
}

// 32 lanes x 32 bits, 4 consecutive columns from registers: thread t of the warp
// writes lane (quarter base + t).  Complete before a later read once
// tmem_st_wait() has returned.
__device__ __forceinline__ void tmem_st4(uint32_t taddr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(a), "r"(b),
                 "r"(c), "r"(d)
                 : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Instruction descriptor of the block-scaled e4m3 MMA (kind::mxf8f6f4): A and B
// e4m3 (format 0), K-major, N>>3 at bit 17, scale format E8M0 at bit 23, M>>4 at
// bit 24; the byte of each 32-bit scale word to use (the scale factor id, 0..3)
// at bits 4-5 for B and 29-30 for A.  D is fp32.
__host__ __device__ constexpr uint32_t idesc_mxf8_f32(int mma_m, int mma_n, int sf_id) {
    return ((uint32_t)sf_id << 4) | ((uint32_t)(mma_n >> 3) << 17) | (1u << 23) | ((uint32_t)(mma_m >> 4) << 24) |
           ((uint32_t)sf_id << 29);
}

// One block-scaled e4m3 MMA, K = 32 codes (one scale block): D[tmem] (+)= (A * sA) (B * sB)^T.
// Scale words in TMEM: for A row m, lane m of column sfa + m / 32; for B column
// n, lane n % 32 of column sfb + n / 32, replicated in every lane quarter (the
// quarter of the D row being computed is the one read).  The byte used is the
// descriptor's scale factor id.  Keep sfa and sfb at columns that are
// multiples of 4 (sfa at a multiple of 8): other columns fault the GPU.
__device__ __forceinline__ void mma_mxf8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// ---- CTA pairs (cta_group::2): two CTAs of a cluster share one MMA ----
// Both CTAs of the pair allocate together: one warp in each (the same warp
// index) executes the alloc, and each CTA's TMEM gets the columns at the
// address written to its own shared memory.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t *dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Pair MMA, issued by one thread of the even CTA: D (rows split 128/128 over
// the two CTAs' TMEM) (+)= A (each CTA's own 128 rows) x B^T (each CTA holds
// half of the N rows), operands at the same shared-memory offsets in both CTAs.
__device__ __forceinline__ void mma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                              uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on the mbarrier at this shared-memory offset in every CTA of `mask`
// once the pair MMAs issued so far by this thread have completed.
__device__ __forceinline__ void mma_commit_pair(uint64_t *bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
        ::"r"(smem_u32(bar)), "h"(mask)
        : "memory");
}

// TMA tile load into this CTA's shared memory whose completion is counted on
// an mbarrier that may sit in the peer CTA of the pair (cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void *dst, const CUtensorMap *map, uint32_t bar_cluster,
                                                 int32_t c0, int32_t c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%3, %4}], [%2];"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1)
        : "memory");
}

// Arrive (release, cluster scope) on an mbarrier in another CTA of the cluster.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}

// ---------------------------------------------------------------------------
// Thread-block clusters and distributed shared memory.
// ---------------------------------------------------------------------------
// Index of this CTA's cluster in the grid (x), and the number of clusters along x.
__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_count_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %nclusterid.x;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %cluster_ctarank;" : "=r"(r));
    return r;
}

// Non-.aligned forms: correct even if threads of a warp reach them apart
// (the vLLM PR #42562 review found the .aligned forms hung when the DMA warps
// took another branch).
__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}
// Arrive without ordering memory (for phases that publish nothing).
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
}
__device__ __forceinline__ void cluster_sync() {
    cluster_arrive_release();
    cluster_wait_acquire();
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

// Asynchronous 16-byte store into another CTA's shared memory; the bytes are
// counted on that CTA's mbarrier (complete_tx), so the receiver can wait for
// all of them without a cluster barrier.
__device__ __forceinline__ void st_async_f4(uint32_t remote_addr, float a, float b, float c, float d,
                                            uint32_t remote_bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];"
                 ::"r"(remote_addr), "f"(a), "f"(b), "f"(c), "f"(d), "r"(remote_bar)
                 : "memory");
}

// Bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned) from
// this CTA's shared memory into another CTA's shared memory; the bytes are
// counted on the destination CTA's mbarrier.
__device__ __forceinline__ void bulk_copy_to_peer(uint32_t remote_dst, const void *local_src, uint32_t bytes,
                                                  uint32_t remote_bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(remote_dst), "r"(smem_u32(local_src)), "r"(bytes), "r"(remote_bar)
        : "memory");
}

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy accesses (bulk copies, TMA) of the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

// ---------------------------------------------------------------------------
// Global loads.
// ---------------------------------------------------------------------------
// Warp-level tensor-core MMAs (mma.sync) used by the kernels that feed their
// operands straight from 16-byte loads.
// D (16x8 fp32) += A (16x16 bf16, row-major) * B (16x8 bf16, column-major).
// Lane (g = lane / 4, t = lane % 4): A {a0: row g, k 2t..2t+1; a1: row g+8, k 2t..;
// a2: row g, k 2t+8..; a3: row g+8, k 2t+8..}; B {b0: k 2t..2t+1, col g;
// b1: k 2t+8.., col g}; D {(g, 2t), (g, 2t+1), (g+8, 2t), (g+8, 2t+1)}.
__device__ __forceinline__ void mma_m16n8k16_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                                  uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// The e4m3 form: 4 codes per register, 32 k positions per instruction, the
// fragments in the same registers as above.
__device__ __forceinline__ void mma_m16n8k32_e4m3(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                                  uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------------------
// 16-byte streaming load that bypasses L1 allocation (weights: read once).
__device__ __forceinline__ uint4 ldg_stream_v4(const void *p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Launch modes from the BF16L_FLAG_* bits (host side).  Every launch uses
// programmatic dependent launch unless BF16L_FLAG_SERIAL: the kernel may be
// scheduled while the previous kernel on the stream finishes, and waits for it
// (griddepcontrol.wait) before it reads anything.  With BF16L_FLAG_PDL the
// weight (and bias) loads may go out before that wait.
inline int pdl_attr_of(uint32_t flags) { return (flags & BF16L_FLAG_SERIAL) ? 0 : 1; }
inline int w_early_of(uint32_t flags) { return (flags & BF16L_FLAG_PDL) ? 1 : 0; }

// Ask L2 to fetch [p, p + bytes) (p 16-byte aligned, bytes a multiple of 16), in
// requests of at most 64 KB.  No data comes back to the thread and nothing is
// cached nearer than L2, the device's point of coherence for global memory: a
// kernel may issue it for its weights before the grid-dependency wait, and a
// write the previous kernel makes to them afterwards still reaches every load
// issued after the wait.
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
    const char *c = static_cast<const char *>(p);
    while (bytes) {
        const uint32_t n = bytes < 65536u ? bytes : 65536u;
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(c), "r"(n) : "memory");
        c += n;
        bytes -= n;
    }
}

// Bias of one 32-column slice n0..n0+31 of the output, one value per lane
// (lane l holds bias[n0 + l], 0 past N or without bias): one coalesced load per
// warp instead of 32 scalar loads per thread.  bias_add32 hands the values to
// every lane with shuffles; both must be called by all 32 lanes of the warp.
__device__ __forceinline__ float bias_lane(const uint16_t *bias, int n0, int N) {
    const int n = n0 + (int)(threadIdx.x & 31u);
    return (bias && n < N) ? bf16_to_f32(__ldg(bias + n)) : 0.0f;
}
__device__ __forceinline__ void bias_add32(float (&v)[32], float lane_bias) {
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] += __shfl_sync(0xFFFFFFFFu, lane_bias, j);
}

// Programmatic dependent launch hooks (no-ops when the launch did not enable PDL).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Host: 2-D bf16 tensor map (row-major [rows][cols], cols contiguous) with a
// box of box_rows x box_cols elements.  Defined in api.cu.  Returns a
// CUresult value (0 on success).
// ---------------------------------------------------------------------------
int make_tmap_bf16_2d(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                      uint32_t box_cols, CUtensorMapSwizzle swizzle, CUtensorMapL2promotion promo);
// A row-major bf16 matrix [rows][K] (K % 64 == 0) seen as {64, rows, K / 64}:
// element (k, r) at chunk k / 64, offset k % 64.  Strides: 2K bytes between
// rows, 128 bytes between chunks.  Box {64, box_rows, kc}, 128-byte swizzle:
// one load brings kc consecutive K chunks of box_rows rows (chunks past K / 64
// are zero-filled).
int make_tmap_bf16_chunks(CUtensorMap *map, const void *base, uint64_t rows, uint64_t K, uint32_t box_rows,
                          uint32_t kc);
// The same for one-byte elements (e4m3 codes): cols in bytes.
int make_tmap_u8_2d(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                    uint32_t box_cols, CUtensorMapSwizzle swizzle, CUtensorMapL2promotion promo);

}  // namespace bf16l
