// dotprod.cuh — CUDA-core dot-product kernel for the smallest token counts
// (templated on the output type; instantiated by dotprod.cu for bf16 and by
// dotprod_f32.cu for the fp32-logits variant).
//
// Prior art: the LLBf16Dotprod kernel on the vLLM PR #42562 page ("实现拆解"
// item 1 and its source excerpt): one CTA per expert row, 128-bit weight
// loads, each weight vector widened to fp32 once and used for every token,
// warp-shuffle then shared-memory reduction; chosen for M <= 4 or K < 2048.
//
// This kernel keeps that structure and adds what GB300 needs to keep enough
// bytes in flight at such small sizes:
//   * a CTA owns R consecutive W rows, so each x vector is reused R times;
//   * every thread issues the 16-byte weight loads of its first batch (up to
//     8 vectors per row) before anything else, while one thread copies x (all
//     MT token rows, a few KB to ~100 KB) into shared memory with one bulk
//     copy per row (a single L2 round trip, counted on an mbarrier); the
//     multiply-adds then read x from shared memory instead of waiting on L2
//     once per (vector, token);
//   * rows whose length is not a multiple of 8 elements (K % 8 != 0, so not
//     16-byte aligned) take a scalar path that reads x from global memory.
// Tokens are processed MT at a time.  With gridDim.y == 1 a CTA loops over the
// token groups, streaming its rows again for each; with gridDim.y = G token
// groups, CTA (b, y) takes groups y, y + G, ... of the same rows, so groups run
// side by side and the weight bytes of the later readers come from L2.
//
// Arithmetic: the products go through the mixed-precision fma
// (fma.rn.f32.bf16: bf16 x bf16 + fp32 -> fp32), so neither operand is widened
// by a separate instruction; the product of two bf16 values is exact in fp32,
// so this is fmaf(float(x), float(w), acc) bit for bit.
// fp32 products and sums (each thread sums its k-slice in
// ascending order, then a fixed shuffle tree and a fixed in-order sum over
// warps), bias added in fp32, one RNE rounding to bf16.  Deterministic.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace bf16l {

namespace {

constexpr int kXSmemMax = 160 * 1024;  // largest x slab staged in shared memory

template <int VEC>
struct Vec;
template <>
struct Vec<8> {  // 8 bf16 in 16 bytes
    uint4 v;
    __device__ __forceinline__ void load_stream(const uint16_t *p) { v = ldg_stream_v4(p); }
    __device__ __forceinline__ void load_cached(const uint16_t *p) { v = __ldg(reinterpret_cast<const uint4 *>(p)); }
    __device__ __forceinline__ float get(int e) const {
        const uint32_t w = (e < 2) ? v.x : (e < 4) ? v.y : (e < 6) ? v.z : v.w;
        return (e & 1) ? bf16_hi(w) : bf16_lo(w);
    }
};
template <>
struct Vec<1> {  // one bf16 (rows not 16-byte aligned when K % 8 != 0)
    uint16_t v;
    __device__ __forceinline__ void load_stream(const uint16_t *p) { v = __ldg(p); }
    __device__ __forceinline__ void load_cached(const uint16_t *p) { v = __ldg(p); }
    __device__ __forceinline__ float get(int) const { return bf16_to_f32(v); }
};

}  // namespace

template <int MT, int R, int VEC, bool XSMEM, typename OutT>
__global__ void __launch_bounds__(256) dotprod_kernel(const uint16_t *__restrict__ x,
                                                      const uint16_t *__restrict__ W,
                                                      const uint16_t *__restrict__ bias,
                                                      OutT *__restrict__ out, int M, int N, int K,
                                                      int32_t *status, int w_early) {
    if (!w_early) {
        // Default launch: nothing is read before the previous kernel has finished.  Meanwhile this
        // row slice's weights are fetched into L2 (one request per row; K % 8 == 0 for 16-byte rows).
        if (blockIdx.y == 0 && (K & 7) == 0 && (int)threadIdx.x < R && (int)blockIdx.x * R + (int)threadIdx.x < N)
            prefetch_l2(W + (size_t)((int)blockIdx.x * R + (int)threadIdx.x) * K, (uint32_t)K * 2u);
        pdl_wait();
    }
    constexpr int U = (VEC == 8) ? 8 : 4;  // vectors per row a thread loads before computing
    __shared__ float red[8][R * MT];
    __shared__ __align__(8) uint64_t xbar;
    extern __shared__ uint4 xs[];  // XSMEM: x[m0 + m][k] as 16-byte vectors, [MT][K / 8]

    const int tid = threadIdx.x;
    const int nt = blockDim.x;
    const int warp = tid >> 5, lane = tid & 31, nwarps = nt >> 5;
    const int n0 = blockIdx.x * R;
    const int nvec = K / VEC;

    const uint16_t *wrow[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int n = min(n0 + r, N - 1);  // rows past N re-read the last row and are not stored
        wrow[r] = W + (size_t)n * K;
    }

    Vec<VEC> wv[U][R];
    auto load_batch = [&](int v0) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int v = v0 + u * nt;
            if (v < nvec) {
#pragma unroll
                for (int r = 0; r < R; ++r) wv[u][r].load_stream(wrow[r] + (size_t)v * VEC);
            }
        }
    };
    // the first pass's first weight batch is in flight before the barrier set-up and before x is touched
    if ((int)blockIdx.y * MT < M) load_batch(tid);

    if constexpr (XSMEM) {
        if (tid == 0) {
            mbar_init(&xbar, 1);
            fence_barrier_init();
        }
        __syncthreads();
    }

    for (int m0 = (int)blockIdx.y * MT, pass = 0; m0 < M; m0 += MT * (int)gridDim.y, ++pass) {
        float acc[R][MT];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int m = 0; m < MT; ++m) acc[r][m] = 0.f;

        if (pass > 0) load_batch(tid);  // this pass's first weight batch
        if (pass == 0) {
            pdl_launch_dependents();  // (no-ops unless launched with programmatic serialization)
            pdl_wait();               // x may be written by the previous kernel; out may still be read by it
        }

        if constexpr (XSMEM) {
            // Stage the token rows of this pass in shared memory: one bulk copy
            // per row.  Rows past M are left stale: they only feed accumulators
            // that are never stored.
            if (tid == 0) {
                const int rows = (M - m0) < MT ? (M - m0) : MT;
                mbar_arrive_expect_tx(&xbar, (uint32_t)(rows * K * 2));
                for (int r = 0; r < rows; ++r)
                    bulk_load(xs + (size_t)r * nvec, x + (size_t)(m0 + r) * K, (uint32_t)(K * 2), &xbar);
            }
            mbar_wait(&xbar, (uint32_t)(pass & 1), status, kSiteStage);
        }

        for (int v0 = tid; v0 < nvec; v0 += U * nt) {
            if (v0 != tid) load_batch(v0);
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int v = v0 + u * nt;
                if (v < nvec) {
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        if (XSMEM || m0 + m < M) {
                            Vec<VEC> xv;
                            if constexpr (XSMEM)
                                xv.v = xs[m * nvec + v];
                            else
                                xv.load_cached(x + (size_t)(m0 + m) * K + (size_t)v * VEC);
                            if constexpr (VEC == 8) {  // bf16 x bf16 + fp32 in one instruction per product
#pragma unroll
                                for (int r = 0; r < R; ++r) {
                                    float a_ = acc[r][m];
                                    a_ = fma2_bf16(xv.v.x, wv[u][r].v.x, a_);
                                    a_ = fma2_bf16(xv.v.y, wv[u][r].v.y, a_);
                                    a_ = fma2_bf16(xv.v.z, wv[u][r].v.z, a_);
                                    a_ = fma2_bf16(xv.v.w, wv[u][r].v.w, a_);
                                    acc[r][m] = a_;
                                }
                            } else {
#pragma unroll
                                for (int e = 0; e < VEC; ++e) {
                                    const float xe = xv.get(e);
#pragma unroll
                                    for (int r = 0; r < R; ++r) acc[r][m] = fmaf(xe, wv[u][r].get(e), acc[r][m]);
                                }
                            }
                        }
                    }
                }
            }
        }

        // Block reduction: shuffle tree within each warp, then warps in order.
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                float v = acc[r][m];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
                if (lane == 0) red[warp][r * MT + m] = v;
            }
        __syncthreads();
        if (tid < R * MT) {
            const int r = tid / MT, m = tid % MT;
            float s = 0.f;
            for (int w = 0; w < nwarps; ++w) s += red[w][tid];
            const int n = n0 + r, mm = m0 + m;
            if (n < N && mm < M) {
                if (bias) s += bf16_to_f32(bias[n]);
                OutStore<OutT>::one(out + (size_t)mm * N + n, s);
            }
        }
        __syncthreads();  // red[] and xs[] are reused by the next pass
    }
}

namespace dot_detail {

template <typename OutT>
using DotFn = void (*)(const uint16_t *, const uint16_t *, const uint16_t *, OutT *, int, int, int, int32_t *, int);

// kind: 0 = 16-byte vectors with x in shared memory, 1 = 16-byte vectors with
// x from global memory, 2 = scalar (K % 8 != 0).
template <int MT, int R, typename OutT>
DotFn<OutT> pick_kind(int kind) {
    switch (kind) {
        case 0: return dotprod_kernel<MT, R, 8, true, OutT>;
        case 1: return dotprod_kernel<MT, R, 8, false, OutT>;
        default: return dotprod_kernel<MT, R, 1, false, OutT>;
    }
}

template <int MT, typename OutT>
DotFn<OutT> pick_rows(int R, int kind) {
    switch (R) {
        case 1: return pick_kind<MT, 1, OutT>(kind);
        case 2: return pick_kind<MT, 2, OutT>(kind);
        case 4: return pick_kind<MT, 4, OutT>(kind);
        default: return nullptr;
    }
}

template <typename OutT>
DotFn<OutT> pick(int MT, int R, int kind) {
    switch (MT) {
        case 1: return pick_rows<1, OutT>(R, kind);
        case 2: return pick_rows<2, OutT>(R, kind);
        case 3: return pick_rows<3, OutT>(R, kind);
        case 4: return pick_rows<4, OutT>(R, kind);
        case 5: return pick_rows<5, OutT>(R, kind);
        case 6: return pick_rows<6, OutT>(R, kind);
        case 7: return pick_rows<7, OutT>(R, kind);
        case 8: return pick_rows<8, OutT>(R, kind);
        default: return nullptr;
    }
}

template <typename OutT>
int init_dotprod_t() {
    for (int MT = 1; MT <= kDotMaxTokens; ++MT)
        for (int R : kDotRows) {
            const int e = (int)cudaFuncSetAttribute(pick<OutT>(MT, R, 0),
                                                    cudaFuncAttributeMaxDynamicSharedMemorySize, kXSmemMax);
            if (e) return e;
        }
    return (int)cudaSuccess;
}

template <typename OutT>
int launch_dotprod_t(const LaunchArgs &a, const bf16l_plan &p) {
    const int t = p.tokens_per_cta > 0 ? p.tokens_per_cta : kDotMaxTokens;
    const int MT = a.M < t ? a.M : t;
    const size_t xbytes = (size_t)MT * a.K * 2;
    // x from shared memory when it fits, unless the plan asks for x straight from L2 (stages == 1)
    const int kind = (a.K % 8 != 0) ? 2 : ((xbytes <= (size_t)kXSmemMax && p.stages == 0) ? 0 : 1);
    DotFn<OutT> fn = pick<OutT>(MT, p.rows_per_cta, kind);
    if (!fn) return (int)cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((a.N + p.rows_per_cta - 1) / p.rows_per_cta),
                       (unsigned)dot_token_groups(a.M, p.tokens_per_cta));
    cfg.blockDim = dim3((unsigned)p.threads);
    cfg.dynamicSmemBytes = kind == 0 ? xbytes : 0;
    cfg.stream = (cudaStream_t)a.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl_attr_of((uint32_t)p.flags);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return (int)cudaLaunchKernelEx(&cfg, fn, static_cast<const uint16_t *>(a.x), static_cast<const uint16_t *>(a.W),
                                   static_cast<const uint16_t *>(a.bias), static_cast<OutT *>(a.out), a.M, a.N,
                                   a.K, a.status, w_early_of((uint32_t)p.flags));
}

}  // namespace dot_detail

}  // namespace bf16l
