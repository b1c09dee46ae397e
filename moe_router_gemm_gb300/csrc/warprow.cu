// warprow.cu — persistent warp-per-row kernel for few tokens and many W rows
// (decode projections, MLP weights: N in the thousands, M <= 8).
//
// Prior art: the dot-product router kernel on the vLLM PR #42562 page (128-bit
// weight loads, each weight vector widened once and used for every token,
// shuffle reduction).  That kernel gives each CTA one expert row and reduces
// over the whole block; for weights of 30-120 MB it launches tens of thousands
// of short CTAs, and every one pays its launch, its first DRAM round trip and
// a block-wide reduction.
//
// On GB300 the fastest way found to stream such a weight from HBM is plain
// 16-byte loads from as many resident warps as the register file holds (about
// 70% of the copy bandwidth for 30 MB and 90% for 117 MB, above bulk copies
// and 2-D TMA boxes).  So this kernel keeps every SM full of warps for the
// whole call and removes the block-wide steps:
//   * persistent grid (a few CTAs per SM); CTA b owns the contiguous W rows
//     [N*b/G, N*(b+1)/G);
//   * a group of WPR warps computes one row at a time (WPR = 1: a warp per row,
//     no barrier at all); each warp of the group takes a fixed K slice, each
//     lane U 16-byte weight vectors per batch;
//   * x (M <= 8 token rows) is staged once per CTA in shared memory by bulk
//     copies; the weight loads of the first batch are issued before that, and
//     before the programmatic-launch wait;
//   * products with the fp32-accumulating bf16 fma (exact products), per-lane
//     sums in ascending k, a fixed shuffle tree, then (WPR > 1) the group's
//     warps summed in order: deterministic for a given plan.
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

namespace bf16l {

namespace {

constexpr int kWrMaxWarps = 32;

}  // namespace

int warprow_smem_bytes(int M, int K) { return M * K * 2; }

// NT = the block size the instance is compiled for; two instances (512 and
// 1024) both keep 1024 threads per SM resident (64 registers a thread).
template <int MT, int WPR, int NT, typename OutT>
__global__ void __launch_bounds__(NT, 1024 / NT)
    warprow_kernel(const uint16_t *__restrict__ x, const uint16_t *__restrict__ W, const uint16_t *__restrict__ bias,
                   OutT *__restrict__ out, int M, int N, int K, int32_t *status, int w_early) {
    if (!w_early) {
        // Default launch: nothing is read before the previous kernel has finished.  Meanwhile the first
        // 32 KB of this CTA's contiguous row range are fetched into L2.
        if (threadIdx.x == 0) {
            const int p0 = mul_div(N, (int)blockIdx.x, (int)gridDim.x), p1 = mul_div(N, (int)blockIdx.x + 1, (int)gridDim.x);
            const uint32_t bytes = (uint32_t)(p1 - p0) * (uint32_t)K * 2u;
            if (p1 > p0) prefetch_l2(W + (size_t)p0 * K, bytes < 32768u ? bytes : 32768u);
        }
        pdl_wait();
    }
    constexpr int U = 8;  // 16-byte weight vectors per lane per batch (128 KB in flight per SM)
    extern __shared__ uint4 xs[];          // x[m][k] as 16-byte vectors, [MT][K / 8]
    __shared__ float part[kWrMaxWarps][MT];
    __shared__ __align__(8) uint64_t xbar;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nw = (int)blockDim.x >> 5;
    const int groups = nw / WPR;
    const int g = warp / WPR, gw = warp - g * WPR;
    const int nvec = K >> 3;
    const int per = (nvec + WPR - 1) / WPR;
    const int kv0 = gw * per, kv1 = (kv0 + per) < nvec ? (kv0 + per) : nvec;
    const int G = (int)gridDim.x, b = (int)blockIdx.x;
    const int r0 = mul_div(N, b, G), r1 = mul_div(N, b + 1, G);

    if (tid == 0) {
        mbar_init(&xbar, 1);
        fence_barrier_init();
    }

    // First batch of this group's first row: in flight before anything waits.
    int n = r0 + g;
    uint4 wv[U];
    auto load_batch = [&](int row, int v) {
        const uint4 *wr = reinterpret_cast<const uint4 *>(W + (size_t)row * K);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int vv = v + 32 * u;
            wv[u] = vv < kv1 ? ldg_stream_v4(wr + vv) : make_uint4(0u, 0u, 0u, 0u);
        }
    };
    if (n < r1) load_batch(n, kv0 + lane);

    pdl_launch_dependents();
    pdl_wait();  // x may be written, and out still read, by the previous kernel
    __syncthreads();
    if (tid == 0 && r1 > r0) {
        mbar_arrive_expect_tx(&xbar, (uint32_t)(M * K * 2));
        for (int m = 0; m < M; ++m) bulk_load(xs + (size_t)m * nvec, x + (size_t)m * K, (uint32_t)(K * 2), &xbar);
    }
    const bool staged = r1 > r0 ? mbar_wait(&xbar, 0, status, kSiteStage) : true;
    if (!__syncthreads_and(staged)) return;  // the whole CTA leaves together (only after a timeout)

    for (bool first = true; n < r1; n += groups, first = false) {
        // two independent fma chains per token (the low and the high 8 bytes of each vector), summed at the end
        float acc[MT], acc2[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[m] = acc2[m] = 0.f;
        for (int v = kv0 + lane; v < kv1; v += 32 * U) {
            if (!(first && v == kv0 + lane)) load_batch(n, v);
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int vv = v + 32 * u;
                if (vv < kv1) {
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        const uint4 xv = xs[m * nvec + vv];
                        float a = acc[m], a2 = acc2[m];
                        a = fma2_bf16(xv.x, wv[u].x, a);
                        a2 = fma2_bf16(xv.z, wv[u].z, a2);
                        a = fma2_bf16(xv.y, wv[u].y, a);
                        a2 = fma2_bf16(xv.w, wv[u].w, a2);
                        acc[m] = a;
                        acc2[m] = a2;
                    }
                }
            }
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            acc[m] += acc2[m];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc[m] += __shfl_xor_sync(0xffffffffu, acc[m], off);
        }
        if constexpr (WPR == 1) {
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                if (lane == m && m < M) {
                    float s = acc[m];
                    if (bias) s += bf16_to_f32(bias[n]);
                    OutStore<OutT>::one(out + (size_t)m * N + n, s);
                }
            }
        } else {
#pragma unroll
            for (int m = 0; m < MT; ++m)
                if (lane == m) part[warp][m] = acc[m];
            asm volatile("bar.sync %0, %1;" ::"r"(1 + g), "r"(WPR * 32) : "memory");
            if (gw == 0 && lane < MT && lane < M) {
                float s = 0.f;
#pragma unroll
                for (int w = 0; w < WPR; ++w) s += part[g * WPR + w][lane];
                if (bias) s += bf16_to_f32(bias[n]);
                OutStore<OutT>::one(out + (size_t)lane * N + n, s);
            }
            asm volatile("bar.sync %0, %1;" ::"r"(1 + g), "r"(WPR * 32) : "memory");  // part[] is reused
        }
    }
}

namespace {

template <typename OutT>
using WrFn = void (*)(const uint16_t *, const uint16_t *, const uint16_t *, OutT *, int, int, int, int32_t *, int);

template <int MT, int WPR, typename OutT>
WrFn<OutT> pick_nt(int threads) {
    return threads > 512 ? warprow_kernel<MT, WPR, 1024, OutT> : warprow_kernel<MT, WPR, 512, OutT>;
}

template <int MT, typename OutT>
WrFn<OutT> pick_wpr(int wpr, int threads) {
    switch (wpr) {
        case 1: return pick_nt<MT, 1, OutT>(threads);
        case 2: return pick_nt<MT, 2, OutT>(threads);
        case 4: return pick_nt<MT, 4, OutT>(threads);
        default: return nullptr;
    }
}

template <typename OutT>
WrFn<OutT> pick_wr(int MT, int wpr, int threads) {
    switch (MT) {
        case 1: return pick_wpr<1, OutT>(wpr, threads);
        case 2: return pick_wpr<2, OutT>(wpr, threads);
        case 3: return pick_wpr<3, OutT>(wpr, threads);
        case 4: return pick_wpr<4, OutT>(wpr, threads);
        case 5: return pick_wpr<5, OutT>(wpr, threads);
        case 6: return pick_wpr<6, OutT>(wpr, threads);
        case 7: return pick_wpr<7, OutT>(wpr, threads);
        case 8: return pick_wpr<8, OutT>(wpr, threads);
        default: return nullptr;
    }
}

template <typename OutT>
int set_wr_attrs() {
    for (int MT = 1; MT <= kWarpRowMaxTokens; ++MT)
        for (int wpr : {1, 2, 4})
            for (int t : {512, 1024}) {
                const int e = (int)cudaFuncSetAttribute(pick_wr<OutT>(MT, wpr, t),
                                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                        kWarpRowMaxSmem);
                if (e) return e;
            }
    return 0;
}

template <typename OutT>
int launch_wr_t(const LaunchArgs &a, const bf16l_plan &p) {
    WrFn<OutT> fn = pick_wr<OutT>(a.M, p.rows_per_cta, p.threads);
    if (!fn) return (int)cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.grid);
    cfg.blockDim = dim3((unsigned)p.threads);
    cfg.dynamicSmemBytes = (size_t)warprow_smem_bytes(a.M, a.K);
    cfg.stream = (cudaStream_t)a.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl_attr_of((uint32_t)p.flags);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return (int)cudaLaunchKernelEx(&cfg, fn, static_cast<const uint16_t *>(a.x), static_cast<const uint16_t *>(a.W),
                                   static_cast<const uint16_t *>(a.bias), static_cast<OutT *>(a.out), a.M, a.N, a.K,
                                   a.status, w_early_of((uint32_t)p.flags));
}

}  // namespace

int init_warprow() {
    int e = set_wr_attrs<uint16_t>();
    if (!e) e = set_wr_attrs<float>();
    return e;
}

int launch_warprow(const LaunchArgs &a, const bf16l_plan &p) {
    return a.out_f32 ? launch_wr_t<float>(a, p) : launch_wr_t<uint16_t>(a, p);
}

}  // namespace bf16l
