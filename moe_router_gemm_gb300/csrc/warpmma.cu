// warpmma.cu — persistent warp-level tensor-core kernel for M <= 16 tokens and
// many W rows (decode projections, MLP weights).
//
// The warp-per-row kernel (warprow.cu) streams W at close to the copy
// bandwidth, but its CUDA-core arithmetic (one fma per weight and token) costs
// as much as the streaming once M reaches 4: a 30 MB weight (15 M elements)
// times 8 tokens is 120 M fmas, about 3 us of issue on all 152 SMs.
// This kernel keeps the same data movement — 16-byte weight loads straight into
// registers from a full SM of warps, the fastest way found to stream such
// weights here — and hands the arithmetic to the tensor cores with the
// warp-level mma.sync.m16n8k16 (bf16 x bf16 -> fp32), whose B operand is the
// very registers the loads filled.  (tcgen05.mma reads B only from shared
// memory: using it would mean staging W through shared memory, with 2-D TMA
// boxes that stream these weights measurably slower than 16-byte loads.)
//
//   * a group of WPR warps owns 8 consecutive W rows (the MMA N) at a time;
//     each warp of the group takes a fixed K slice of whole 32-wide blocks;
//   * per 32-wide K block, lane (g = lane / 4, t = lane % 4) loads the 16 bytes
//     W[n0 + g][kb + 8t, kb + 8t + 8) and the same 16 bytes of x tokens g and
//     g + 8 from shared memory.  The MMA's k index runs over a permutation of
//     the block's 32 positions, the same for A and B, in two m16n8k16 steps;
//   * tokens sit on the MMA M side (rows 0..15; rows past M are zero);
//   * D lane (g, t) ends with out[token g (and g + 8)][rows n0 + 2t, n0 + 2t + 1];
//     with WPR > 1 the group's warps are summed in order through shared memory;
//   * x staged once per CTA by bulk copies (M * K * 2 bytes); the first weight
//     batch is issued before the programmatic-launch wait.
// The tensor core's internal summation order is fixed, so a plan is bitwise
// reproducible.
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

namespace bf16l {

namespace {

constexpr int kWmMaxWarps = 32;

}  // namespace

int warpmma_smem_bytes(int M, int K) { return M * K * 2; }

// NT: block size the instance is compiled for (512 or 1024; a 256-thread block
// runs the 512 instance); all keep 1024 threads per SM resident.  HI: M > 8
// (tokens 8..15 in the MMA's upper rows).  XR: x fragments loaded from L2 into
// registers with each weight batch instead of staged in shared memory (for x
// too large to stage, e.g. 16 tokens of K = 7168); 512 threads per SM then, as
// the batch of x fragments takes another 64 registers a thread.  F8: x and W
// are e4m3 codes (m16n8k32 MMAs on the same registers; the sum is scaled by
// *scale_x * *scale_w before bias).  NG: 8-row groups a warp covers with each
// x fragment it reads (1, 2 or 4; with 2 the x bytes read per weight byte halve,
// which matters once 9..16 tokens make x twice the weight bytes a warp moves).
// Rows of x and W are RB bytes.
template <int WPR, int NT, bool HI, bool XR, bool F8, typename OutT, int NG = 1>
__global__ void __launch_bounds__(NT, XR ? 1 : 1024 / NT)
    warpmma_kernel(const uint8_t *__restrict__ x, const uint8_t *__restrict__ W, const uint16_t *__restrict__ bias,
                   OutT *__restrict__ out, int M, int N, int RB, int32_t *status, const float *__restrict__ scale_x,
                   const float *__restrict__ scale_w, int w_early) {
    constexpr int U = 8 / NG;                      // K blocks (4 x 16 bytes across a lane quad) per lane per batch
    extern __shared__ uint4 xs[];                  // x[m] rows as 16-byte vectors, [M][RB / 16]
    __shared__ float part[WPR > 1 ? kWmMaxWarps : 1][32][4];  // WPR > 1: every lane's four sums
    __shared__ __align__(8) uint64_t xbar;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    const int nw = (int)blockDim.x >> 5;
    const int groups = nw / WPR;
    const int grp = warp / WPR, gw = warp - grp * WPR;
    const int nvec = RB >> 4;
    // this warp's K slice in 16-byte vectors, whole 32-wide blocks (4 vectors)
    const int nblk = (nvec + 3) >> 2;
    const int per = (nblk + WPR - 1) / WPR;
    const int vb0 = 4 * gw * per;
    const int vb1 = min(nvec, 4 * (gw + 1) * per);
    // CTA b owns the (8 NG)-row slabs [RS*b/G, RS*(b+1)/G)
    const int RS = (N + 8 * NG - 1) / (8 * NG);
    const int G = (int)gridDim.x, b = (int)blockIdx.x;
    const int q0 = mul_div(RS, b, G), q1 = mul_div(RS, b + 1, G);
    const bool tok_lo = g < M, tok_hi = HI && (g + 8 < M);
    if (!w_early) {
        // Default launch: nothing is read before the previous kernel has finished.  Meanwhile the first
        // 32 KB of this CTA's contiguous rows are fetched into L2.
        if (tid == 0 && q1 > q0) {
            const int p0 = 8 * NG * q0, p1 = min(N, 8 * NG * q1);
            const uint32_t bytes = (uint32_t)(p1 - p0) * (uint32_t)RB;
            if (p1 > p0) prefetch_l2(W + (size_t)p0 * RB, bytes < 32768u ? bytes : 32768u);
        }
        pdl_wait();
    }

    if (tid == 0) {
        mbar_init(&xbar, 1);
        fence_barrier_init();
    }

    uint4 wv[U][NG];
    auto load_batch = [&](int n0, int vb) {  // the batch of blocks starting at vector vb
#pragma unroll
        for (int j = 0; j < NG; ++j) {
            const int row = n0 + 8 * j + g;
            const uint4 *wr = reinterpret_cast<const uint4 *>(W + (size_t)(row < N ? row : N - 1) * RB);
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int vv = vb + 4 * u + t;
                wv[u][j] = (vv < vb1 && row < N) ? ldg_stream_v4(wr + vv) : make_uint4(0u, 0u, 0u, 0u);
            }
        }
    };
    // One L2 prefetch per lane of a batch's 32 lines (8 NG rows x U / 2 lines of 128 bytes), issued one batch
    // ahead so the next loads find their lines in L2.
    auto prefetch_batch = [&](int qn, int vb) {
        if (qn >= q1 || vb >= vb1) return;
        const int row = 8 * NG * qn + lane / (U / 2);
        const int v = vb + 8 * (lane % (U / 2));  // first 16-byte vector of this lane's 128-byte line
        if (row < N && v < vb1)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(W + (size_t)row * RB + (size_t)v * 16));
    };
    int q = q0 + grp;
    if (q < q1) load_batch(8 * NG * q, vb0);

    pdl_launch_dependents();
    pdl_wait();  // x may be written, and out still read, by the previous kernel
    __syncthreads();
    if constexpr (!XR) {
        if (tid == 0 && q1 > q0) {
            mbar_arrive_expect_tx(&xbar, (uint32_t)(M * RB));
            for (int m = 0; m < M; ++m)
                bulk_load(xs + (size_t)m * nvec, x + (size_t)m * RB, (uint32_t)RB, &xbar);
        }
        const bool staged = q1 > q0 ? mbar_wait(&xbar, 0, status, kSiteStage) : true;
        if (!__syncthreads_and(staged)) return;  // the whole CTA leaves together (only after a timeout)
    }

    const uint4 *xlo = xs + (size_t)(tok_lo ? g : 0) * nvec;
    const uint4 *xhi = xs + (size_t)(tok_hi ? g + 8 : 0) * nvec;
    const uint4 *glo = reinterpret_cast<const uint4 *>(x + (size_t)(tok_lo ? g : 0) * RB);
    const uint4 *ghi = reinterpret_cast<const uint4 *>(x + (size_t)(tok_hi ? g + 8 : 0) * RB);
    for (bool first = true; q < q1; q += groups, first = false) {
        const int n0 = 8 * NG * q;
        // per 8-row group, two independent accumulator chains: step s of every block goes to chain
        // s (the same order whether x comes from shared memory or L2), summed at the end
        float c[NG][2][4];
#pragma unroll
        for (int j = 0; j < NG; ++j)
#pragma unroll
            for (int i = 0; i < 2; ++i) c[j][i][0] = c[j][i][1] = c[j][i][2] = c[j][i][3] = 0.f;
        for (int vb = vb0; vb < vb1; vb += 4 * U) {  // warp-uniform trip count: mma.sync is warp-wide
            if (!(first && vb == vb0)) load_batch(n0, vb);
            if (vb + 4 * U < vb1)
                prefetch_batch(q, vb + 4 * U);
            else
                prefetch_batch(q + groups, vb0);
            uint4 xl[XR ? U : 1], xh[XR ? U : 1];
            if constexpr (XR) {  // this batch's x fragments, in flight with the weights
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int vv = vb + 4 * u + t;
                    const bool in = vv < vb1;
                    xl[u] = (tok_lo && in) ? __ldg(glo + vv) : make_uint4(0u, 0u, 0u, 0u);
                    xh[u] = (HI && tok_hi && in) ? __ldg(ghi + vv) : make_uint4(0u, 0u, 0u, 0u);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int vv = vb + 4 * u + t;
                const bool in = vv < vb1;
                uint4 lo, hi = make_uint4(0u, 0u, 0u, 0u);
                if constexpr (XR) {
                    lo = xl[u];
                    hi = xh[u];
                } else {
                    lo = (tok_lo && in) ? xlo[vv] : make_uint4(0u, 0u, 0u, 0u);
                    if constexpr (HI) {
                        if (tok_hi && in) hi = xhi[vv];
                    }
                }
                // this lane's 16 block bytes: step 0 takes the first 8, step 1 the last 8; the same
                // x fragment feeds every 8-row group of the slab
#pragma unroll
                for (int j = 0; j < NG; ++j) {
                    if constexpr (F8) {
                        mma_m16n8k32_e4m3(c[j][0], lo.x, hi.x, lo.y, hi.y, wv[u][j].x, wv[u][j].y);
                        mma_m16n8k32_e4m3(c[j][1], lo.z, hi.z, lo.w, hi.w, wv[u][j].z, wv[u][j].w);
                    } else {
                        mma_m16n8k16_bf16(c[j][0], lo.x, hi.x, lo.y, hi.y, wv[u][j].x, wv[u][j].y);
                        mma_m16n8k16_bf16(c[j][1], lo.z, hi.z, lo.w, hi.w, wv[u][j].z, wv[u][j].w);
                    }
                }
            }
        }
#pragma unroll
        for (int jg = 0; jg < NG; ++jg) {  // each 8-row group of the slab: reduce over the WPR warps, store
            float d[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) d[j] = c[jg][0][j] + c[jg][1][j];
            if constexpr (WPR > 1) {
#pragma unroll
                for (int j = 0; j < 4; ++j) part[warp][lane][j] = d[j];
                asm volatile("bar.sync %0, %1;" ::"r"(1 + grp), "r"(WPR * 32) : "memory");
                if (gw == 0) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        float s = 0.f;
                        for (int w = 0; w < WPR; ++w) s += part[grp * WPR + w][lane][j];
                        d[j] = s;
                    }
                }
            }
            if (WPR == 1 || gw == 0) {
                if constexpr (F8) {  // per-tensor scales (read after the grid-dependency wait)
                    const float sxw = __ldg(scale_x) * __ldg(scale_w);
#pragma unroll
                    for (int j = 0; j < 4; ++j) d[j] *= sxw;
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int m = g + (j >> 1) * 8, n = n0 + 8 * jg + 2 * t + (j & 1);
                    if (m < M && n < N) {
                        float s = d[j];
                        if (bias) s += bf16_to_f32(bias[n]);
                        OutStore<OutT>::one(out + (size_t)m * N + n, s);
                    }
                }
            }
            if constexpr (WPR > 1) asm volatile("bar.sync %0, %1;" ::"r"(1 + grp), "r"(WPR * 32) : "memory");
        }
    }
}

namespace {

template <typename OutT>
using WmFn = void (*)(const uint8_t *, const uint8_t *, const uint16_t *, OutT *, int, int, int, int32_t *,
                      const float *, const float *, int);

template <int WPR, bool HI, bool XR, bool F8, typename OutT, int NG>
WmFn<OutT> pick_nt(int threads) {
    if constexpr (XR) {
        return warpmma_kernel<WPR, 512, HI, true, F8, OutT, NG>;  // at most 512 threads
    } else {
        return threads > 512 ? warpmma_kernel<WPR, 1024, HI, false, F8, OutT, NG>
                             : warpmma_kernel<WPR, 512, HI, false, F8, OutT, NG>;
    }
}

template <bool HI, bool XR, bool F8, typename OutT, int NG = 1>
WmFn<OutT> pick_wpr(int wpr, int threads) {
    switch (wpr) {
        case 1: return pick_nt<1, HI, XR, F8, OutT, NG>(threads);
        case 2: return pick_nt<2, HI, XR, F8, OutT, NG>(threads);
        case 4: return pick_nt<4, HI, XR, F8, OutT, NG>(threads);
        case 8: return pick_nt<8, HI, XR, F8, OutT, NG>(threads);
        case 16: return pick_nt<16, HI, XR, F8, OutT, NG>(threads);
        default: return nullptr;
    }
}

// ng: 8-row groups per warp (2 or 4 only with x from L2, whose 128 registers hold the groups' weights).
template <typename OutT>
WmFn<OutT> pick_wm(int M, int wpr, int threads, bool xr, int ng = 1) {
    if (xr && ng == 4)
        return M > 8 ? pick_wpr<true, true, false, OutT, 4>(wpr, threads)
                     : pick_wpr<false, true, false, OutT, 4>(wpr, threads);
    if (xr && ng == 2)
        return M > 8 ? pick_wpr<true, true, false, OutT, 2>(wpr, threads)
                     : pick_wpr<false, true, false, OutT, 2>(wpr, threads);
    if (xr)
        return M > 8 ? pick_wpr<true, true, false, OutT>(wpr, threads) : pick_wpr<false, true, false, OutT>(wpr, threads);
    return M > 8 ? pick_wpr<true, false, false, OutT>(wpr, threads) : pick_wpr<false, false, false, OutT>(wpr, threads);
}

// e4m3 operands: x staged in shared memory, bf16 out.
WmFn<uint16_t> pick_wm_f8(int M, int wpr, int threads) {
    return M > 8 ? pick_wpr<true, false, true, uint16_t>(wpr, threads)
                 : pick_wpr<false, false, true, uint16_t>(wpr, threads);
}

template <typename OutT>
int set_wm_attrs() {
    for (int M : {8, 16})
        for (int wpr : {1, 2, 4, 8, 16})
            for (int t : {512, 1024}) {
                const int e = (int)cudaFuncSetAttribute(pick_wm<OutT>(M, wpr, t, false),
                                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                        kWarpMmaMaxSmem);
                if (e) return e;
            }
    return 0;
}

template <typename OutT>
int launch_wm_common(WmFn<OutT> fn, const void *x, const void *W, const void *bias, OutT *out, int M, int N,
                     int RB, int grid, int threads, size_t smem, uint32_t flags, void *stream, int32_t *status,
                     const float *sx, const float *sw) {
    if (!fn) return (int)cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = (cudaStream_t)stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl_attr_of(flags);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return (int)cudaLaunchKernelEx(&cfg, fn, static_cast<const uint8_t *>(x), static_cast<const uint8_t *>(W),
                                   static_cast<const uint16_t *>(bias), out, M, N, RB, status, sx, sw,
                                   w_early_of(flags));
}

template <typename OutT>
int launch_wm_t(const LaunchArgs &a, const bf16l_plan &p) {
    const bool xr = p.split_k == 1;
    const int ng = p.tokens_per_cta > 1 ? p.tokens_per_cta : 1;
    return launch_wm_common(pick_wm<OutT>(a.M, p.rows_per_cta, p.threads, xr, ng), a.x, a.W, a.bias,
                            static_cast<OutT *>(a.out), a.M, a.N, a.K * 2, p.grid, p.threads,
                            xr ? 0 : (size_t)warpmma_smem_bytes(a.M, a.K), (uint32_t)p.flags, a.stream, a.status,
                            nullptr, nullptr);
}

}  // namespace

int init_warpmma() {
    int e = set_wm_attrs<uint16_t>();
    if (!e) e = set_wm_attrs<float>();
    for (int M : {8, 16})
        for (int wpr : {1, 2, 4, 8, 16})
            for (int t : {512, 1024})
                if (!e)
                    e = (int)cudaFuncSetAttribute(pick_wm_f8(M, wpr, t), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                  kWarpMmaMaxSmem);
    return e;
}

int launch_warpmma(const LaunchArgs &a, const bf16l_plan &p) {
    if (p.split_k >= 2) return launch_warpmma_ks(a, p);  // the cluster form (warpmma_ks.cu)
    return a.out_f32 ? launch_wm_t<float>(a, p) : launch_wm_t<uint16_t>(a, p);
}

int launch_warpmma_fp8(const void *xq, const void *wq, const float *sx, const float *sw, const void *bias, void *out,
                       int M, int N, int K, int wpr, int threads, int grid, uint32_t flags, void *stream,
                       int32_t *status) {
    return launch_wm_common(pick_wm_f8(M, wpr, threads), xq, wq, bias, static_cast<uint16_t *>(out), M, N, K, grid,
                            threads, (size_t)M * K, flags, stream, status, sx, sw);
}

}  // namespace bf16l
