// dotmma.cu — router-sized N with up to 16 tokens: 8 W rows per CTA, K split
// over a cluster of S CTAs, warp-level tensor-core MMAs fed by 16-byte loads.
//
// Prior art: the cluster split-K router kernel on the vLLM PR #42562 page
// ("实现拆解" items 2-3): K split over the CTAs of a cluster, fp32 partials
// summed by one CTA through distributed shared memory, for 4 < M <= 64.
//
// For M = 9..16 on router weights (N = 128..384 rows, 1-6 MB) the dot-product
// kernel does M fmas per weight element on CUDA cores and the tcgen05 split-K
// kernel pays TMEM allocation, tensor-map fetches and a 64-row MMA for <= 16
// tokens.  This kernel keeps the split-K shape and takes the arithmetic from the
// warp-MMA kernel: lane (g, t) of a warp loads the 16 bytes
// W[n0 + g][kb + 8t, +8) of each 32-wide K block — its B fragment for two
// mma.sync.m16n8k16 steps under a permutation of the block's k positions — and
// the same 16 bytes of tokens g and g + 8 from shared memory as its A fragment.
//   * grid (S, ceil(N / 8)); CTA (r, q) owns rows 8q..8q+7 and the r-th of S
//     equal runs of 32-wide K blocks; its warps split that run;
//   * x: each CTA stages only its K slice of the M token rows (bulk copies),
//     or (XR) each lane loads its x fragments from L2 next to its weights;
//     the weight loads of the first batch go out before that and before the
//     programmatic-launch wait;
//   * warps' partial tiles summed in warp order in shared memory; ranks 1..S-1
//     send theirs (a 16 x 8 fp32 tile, 512 bytes) to rank 0 with st.async, counted on
//     rank 0's mbarrier; rank 0 sums in rank order, adds bias, rounds, stores.
// Two cluster barrier phases (non-.aligned): "receive barrier initialised"
// (arrived at start, waited before sending) and "all received" (before exit).
// Cluster-free form (WS, BF16L_KERNEL_DOTMMA_WS): the S CTAs of a row group
// are independent; each writes its tile to a caller workspace, fences and takes
// a ticket from the group's counter; the last to arrive sums the S tiles in
// rank order, stores, and resets the counter for the next call.
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

namespace bf16l {

namespace {

constexpr int kDmWarps = 8;  // at most 256 threads

// K blocks (of 4 16-byte vectors = 32 elements) of CTA rank r out of S.
__host__ __device__ inline int dm_blk(int nblk, int r, int S) { return (int)(((long long)nblk * r) / S); }

}  // namespace

// Workspace of the cluster-free form: per-group arrival counters (rounded up
// to 256 bytes), then the tiles [groups][S][32 lanes] of float4.
size_t dotmma_ws_counter_bytes(int groups) { return ((size_t)groups * 4 + 255) / 256 * 256; }
size_t dotmma_ws_bytes(int N, const bf16l_plan &p) {
    if (p.kernel != BF16L_KERNEL_DOTMMA_WS || p.split_k <= 0) return 0;
    const int groups = (N + 7) / 8;
    return dotmma_ws_counter_bytes(groups) + (size_t)groups * p.split_k * 32 * 16;
}

// Dynamic shared memory: x slice [M][vectors of the largest slice] as 16-byte
// vectors (K in bf16 elements; an e4m3 row of K codes is K / 2 of them).
int dotmma_smem_bytes(int M, int K, int S) {
    const int nvec = K / 8, nblk = (nvec + 3) / 4;
    int most = 0;
    for (int r = 0; r < S; ++r) {
        const int v0 = 4 * dm_blk(nblk, r, S);
        const int v1 = 4 * dm_blk(nblk, r + 1, S) < nvec ? 4 * dm_blk(nblk, r + 1, S) : nvec;
        if (v1 - v0 > most) most = v1 - v0;
    }
    return M * most * 16;
}

// HI: M > 8 (tokens 8..15 on the MMA's upper rows).  XR: x fragments loaded
// from global memory (L2) straight into registers next to the weights, instead
// of a bulk copy of the CTA's x slice into shared memory.  F8: x and W are e4m3
// codes (per-tensor FP8; the sum is scaled by *scale_x * *scale_w before bias).
// Rows of x and W are RB bytes (K * 2 for bf16, K for e4m3).  grid.z: groups of
// 16 tokens (CTA z takes tokens 16z..16z+15).
template <bool HI, bool XR, bool WS, bool F8, typename OutT>
__global__ void __launch_bounds__(kDmWarps * 32)
    dotmma_kernel(const uint8_t *__restrict__ x, const uint8_t *__restrict__ W, const uint16_t *__restrict__ bias,
                  OutT *__restrict__ out, int M, int N, int RB, int S, int32_t *status, uint32_t *counters,
                  float4 *tiles, const float *__restrict__ scale_x, const float *__restrict__ scale_w,
                  int w_early) {
    constexpr int U = 8;  // K blocks (4 x 16 bytes across the lane quad) per lane per batch
    extern __shared__ uint4 xs[];
    __shared__ float4 part[kDmWarps][32];  // per warp, lane (g, t): tokens g, g+8 x rows 2t, 2t+1
    __shared__ float4 recv[kDotMmaMaxCluster][32];
    __shared__ __align__(8) uint64_t xbar, rbar;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    const int nw = (int)blockDim.x >> 5;
    {  // this CTA's group of 16 tokens
        const int m0 = 16 * (int)blockIdx.z;
        x += (size_t)m0 * RB;
        out += (size_t)m0 * N;
        M = (M - m0) < 16 ? (M - m0) : 16;
    }
    const bool clus = !WS && S > 1;
    const int rank = WS ? (int)blockIdx.x : (S > 1 ? (int)cluster_ctarank() : 0);
    const int n0 = 8 * (int)blockIdx.y;
    const int nvec = RB >> 4, nblk = (nvec + 3) >> 2;
    // this CTA's vectors [cv0, cv1) and this warp's blocks
    const int cb0 = mul_div(nblk, rank, S), cb1 = mul_div(nblk, rank + 1, S);  // = dm_blk
    const int cv0 = 4 * cb0, cv1 = min(nvec, 4 * cb1);
    const int wb0 = cb0 + mul_div(cb1 - cb0, warp, nw);
    const int wb1 = cb0 + mul_div(cb1 - cb0, warp + 1, nw);
    const int wv0 = 4 * wb0, wv1 = min(cv1, 4 * wb1);
    const int sv = cv1 - cv0;  // vectors in this CTA's x slice
    if (!w_early) {
        // Default launch: nothing is read before the previous kernel has finished.  Meanwhile this CTA's
        // slice of its 8 rows is fetched into L2 (one request per row, by the first token group only).
        if (blockIdx.z == 0 && tid < 8 && n0 + tid < N && sv > 0)
            prefetch_l2(W + (size_t)(n0 + tid) * RB + (size_t)cv0 * 16, (uint32_t)sv * 16u);
        pdl_wait();
    }
    const bool tok_lo = g < M, tok_hi = HI && (g + 8 < M);
    const int row = n0 + g;
    const uint4 *wr = reinterpret_cast<const uint4 *>(W + (size_t)(row < N ? row : N - 1) * RB);

    uint4 wv[U];
    auto load_batch = [&](int vb) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int vv = vb + 4 * u + t;
            wv[u] = (vv < wv1 && row < N) ? ldg_stream_v4(wr + vv) : make_uint4(0u, 0u, 0u, 0u);
        }
    };
    load_batch(wv0);  // in flight before anything waits, the barrier set-up included

    if (tid == 0) {
        mbar_init(&xbar, 1);
        mbar_init(&rbar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (clus) cluster_arrive_relaxed();  // phase 1: "my receive barrier is initialised"

    pdl_launch_dependents();
    pdl_wait();  // x may be written, and out still read, by the previous kernel
    bool ok = true;
    if constexpr (!XR) {
        if (tid == 0 && sv > 0) {
            mbar_arrive_expect_tx(&xbar, (uint32_t)(M * sv * 16));
            for (int m = 0; m < M; ++m)
                bulk_load(xs + (size_t)m * sv, x + (size_t)m * RB + (size_t)cv0 * 16, (uint32_t)(sv * 16), &xbar);
        }
        const bool staged = sv > 0 ? mbar_wait(&xbar, 0, status, kSiteStage) : true;
        ok = __syncthreads_and(staged) != 0;
    }

    // two independent accumulator chains: step s of every block goes to chain s
    float c[2][4];
#pragma unroll
    for (int i = 0; i < 2; ++i) c[i][0] = c[i][1] = c[i][2] = c[i][3] = 0.f;
    if (ok) {
        const uint4 *xlo = xs + (size_t)(tok_lo ? g : 0) * sv;  // indexed by vector - cv0
        const uint4 *xhi = xs + (size_t)(tok_hi ? g + 8 : 0) * sv;
        const uint4 *glo = reinterpret_cast<const uint4 *>(x + (size_t)(tok_lo ? g : 0) * RB);
        const uint4 *ghi = reinterpret_cast<const uint4 *>(x + (size_t)(tok_hi ? g + 8 : 0) * RB);
        for (int vb = wv0; vb < wv1; vb += 4 * U) {  // warp-uniform trip count: mma.sync is warp-wide
            if (vb != wv0) load_batch(vb);
            uint4 xl[U], xh[U];
            if constexpr (XR) {  // this batch's x fragments, in flight together
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int vv = vb + 4 * u + t;
                    const bool in = vv < wv1;
                    xl[u] = (tok_lo && in) ? __ldg(glo + vv) : make_uint4(0u, 0u, 0u, 0u);
                    xh[u] = (HI && tok_hi && in) ? __ldg(ghi + vv) : make_uint4(0u, 0u, 0u, 0u);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int vv = vb + 4 * u + t;
                const bool in = vv < wv1;
                uint4 lo, hi = make_uint4(0u, 0u, 0u, 0u);
                if constexpr (XR) {
                    lo = xl[u];
                    hi = xh[u];
                } else {
                    lo = (tok_lo && in) ? xlo[vv - cv0] : make_uint4(0u, 0u, 0u, 0u);
                    if constexpr (HI) {
                        if (tok_hi && in) hi = xhi[vv - cv0];
                    }
                }
                if constexpr (F8) {
                    mma_m16n8k32_e4m3(c[0], lo.x, hi.x, lo.y, hi.y, wv[u].x, wv[u].y);
                    mma_m16n8k32_e4m3(c[1], lo.z, hi.z, lo.w, hi.w, wv[u].z, wv[u].w);
                } else {
                    mma_m16n8k16_bf16(c[0], lo.x, hi.x, lo.y, hi.y, wv[u].x, wv[u].y);
                    mma_m16n8k16_bf16(c[1], lo.z, hi.z, lo.w, hi.w, wv[u].z, wv[u].w);
                }
            }
        }
    }
    float d[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) d[j] = c[0][j] + c[1][j];
    part[warp][lane] = make_float4(d[0], d[1], d[2], d[3]);
    __syncthreads();
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    if (warp == 0) {
        for (int w = 0; w < nw; ++w) {  // warps in order
            const float4 p = part[w][lane];
            s.x += p.x;
            s.y += p.y;
            s.z += p.z;
            s.w += p.w;
        }
    }

    bool have = ok;
    bool store = rank == 0;
    if constexpr (WS) {
        // ---- cluster-free: tile to the workspace, ticket, the last CTA reduces ----
        __shared__ uint32_t ticket;
        const int q = (int)blockIdx.y;
        if (warp == 0) {
            __stcg(&tiles[((size_t)q * S + rank) * 32 + lane], s);
            __threadfence();
            __syncwarp();
            if (lane == 0) ticket = atomicAdd(&counters[q], 1u);
        }
        __syncthreads();
        store = ticket == (uint32_t)(S - 1);
        if (store && warp == 0) {
            __threadfence();
            s = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int r = 0; r < S; ++r) {  // ranks in order
                const float4 p = __ldcg(&tiles[((size_t)q * S + r) * 32 + lane]);
                s.x += p.x;
                s.y += p.y;
                s.z += p.z;
                s.w += p.w;
            }
            if (lane == 0) counters[q] = 0u;  // ready for the next call
        }
    } else if (S > 1) {
        cluster_wait_acquire();  // phase 1 done: rank 0's receive barrier exists
        if (rank != 0) {
            if (warp == 0)
                st_async_f4(mapa_shared(smem_u32(&recv[rank][lane]), 0), s.x, s.y, s.z, s.w,
                            mapa_shared(smem_u32(&rbar), 0));
        } else {
            if (tid == 0) mbar_arrive_expect_tx(&rbar, (uint32_t)((S - 1) * 32 * 16));
            if (warp == 0) {
                have = mbar_wait_cluster(&rbar, 0, status, kSiteRecv) && have;
                for (int r = 1; r < S; ++r) {  // ranks in order
                    const float4 p = recv[r][lane];
                    s.x += p.x;
                    s.y += p.y;
                    s.z += p.z;
                    s.w += p.w;
                }
            }
        }
        cluster_arrive_relaxed();  // phase 2: everything this CTA sends or receives has landed (rank 0)
    }
    if (store && warp == 0 && have) {
        float v[4] = {s.x, s.y, s.z, s.w};
        if constexpr (F8) {  // per-tensor scales (read after the grid-dependency wait)
            const float sxw = __ldg(scale_x) * __ldg(scale_w);
#pragma unroll
            for (int j = 0; j < 4; ++j) v[j] *= sxw;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int m = g + (j >> 1) * 8, n = n0 + 2 * t + (j & 1);
            if (m < M && n < N) {
                float r = v[j];
                if (bias) r += bf16_to_f32(bias[n]);
                OutStore<OutT>::one(out + (size_t)m * N + n, r);
            }
        }
    }
    if (clus) cluster_wait_acquire();  // phase 2 done: rank 0 holds every partial; all may exit
}

namespace {

template <typename OutT>
using DmFn = void (*)(const uint8_t *, const uint8_t *, const uint16_t *, OutT *, int, int, int, int, int32_t *,
                      uint32_t *, float4 *, const float *, const float *, int);

template <bool WS, typename OutT>
DmFn<OutT> pick_dm_ws(int M, bool xr) {
    if (xr) return M > 8 ? dotmma_kernel<true, true, WS, false, OutT> : dotmma_kernel<false, true, WS, false, OutT>;
    return M > 8 ? dotmma_kernel<true, false, WS, false, OutT> : dotmma_kernel<false, false, WS, false, OutT>;
}

template <typename OutT>
DmFn<OutT> pick_dm(int M, bool xr, bool ws) {
    return ws ? pick_dm_ws<true, OutT>(M, xr) : pick_dm_ws<false, OutT>(M, xr);
}

// e4m3 operands: x fragments from L2, clusters along K, bf16 out.
DmFn<uint16_t> pick_dm_f8(int M) {
    return M > 8 ? dotmma_kernel<true, true, false, true, uint16_t> : dotmma_kernel<false, true, false, true, uint16_t>;
}

template <typename OutT>
int set_dm_attrs() {
    for (int M : {8, 16})
        for (bool xr : {false, true})
            for (bool ws : {false, true}) {
                int e = (int)cudaFuncSetAttribute(pick_dm<OutT>(M, xr, ws),
                                                  cudaFuncAttributeMaxDynamicSharedMemorySize, kDotMmaMaxSmem);
                if (!e && !ws)
                    e = (int)cudaFuncSetAttribute(pick_dm<OutT>(M, xr, ws),
                                                  cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
                if (e) return e;
            }
    return 0;
}

template <typename OutT>
int launch_dm_common(DmFn<OutT> fn, const void *x, const void *W, const void *bias, OutT *out, int M, int N, int RB,
                     int S, int threads, size_t smem, bool cluster, uint32_t flags, void *stream, int32_t *status,
                     uint32_t *counters, float4 *tiles, const float *sx, const float *sw) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)S, (unsigned)((N + 7) / 8), (unsigned)((M + 15) / 16));
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = (cudaStream_t)stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl_attr_of(flags);
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)S;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = cluster ? 2 : 1;
    return (int)cudaLaunchKernelEx(&cfg, fn, static_cast<const uint8_t *>(x), static_cast<const uint8_t *>(W),
                                   static_cast<const uint16_t *>(bias), out, M, N, RB, S, status, counters, tiles,
                                   sx, sw, w_early_of(flags));
}

template <typename OutT>
int launch_dm_t(const LaunchArgs &a, const bf16l_plan &p) {
    const int S = p.split_k;
    const bool ws = p.kernel == BF16L_KERNEL_DOTMMA_WS;
    uint32_t *counters = nullptr;
    float4 *tiles = nullptr;
    if (ws) {
        const int groups = (a.N + 7) / 8;
        if (!a.workspace || a.workspace_bytes < dotmma_ws_bytes(a.N, p)) return (int)cudaErrorInvalidValue;
        counters = static_cast<uint32_t *>(a.workspace);
        tiles = reinterpret_cast<float4 *>(static_cast<uint8_t *>(a.workspace) + dotmma_ws_counter_bytes(groups));
    }
    const bool xr = p.stages == 1;
    const size_t smem = xr ? 0 : (size_t)dotmma_smem_bytes(a.M < 16 ? a.M : 16, a.K, S);  // one token group
    return launch_dm_common(pick_dm<OutT>(a.M, xr, ws), a.x, a.W, a.bias, static_cast<OutT *>(a.out), a.M, a.N,
                            a.K * 2, S, p.threads, smem, S > 1 && !ws, (uint32_t)p.flags, a.stream, a.status,
                            counters, tiles, nullptr, nullptr);
}

}  // namespace

int init_dotmma() {
    int e = set_dm_attrs<uint16_t>();
    if (!e) e = set_dm_attrs<float>();
    for (int M : {8, 16})
        if (!e) e = (int)cudaFuncSetAttribute(pick_dm_f8(M), cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return e;
}

int launch_dotmma(const LaunchArgs &a, const bf16l_plan &p) {
    return a.out_f32 ? launch_dm_t<float>(a, p) : launch_dm_t<uint16_t>(a, p);
}

int launch_dotmma_fp8(const void *xq, const void *wq, const float *sx, const float *sw, const void *bias, void *out,
                      int M, int N, int K, int S, int threads, uint32_t flags, void *stream, int32_t *status) {
    return launch_dm_common(pick_dm_f8(M), xq, wq, bias, static_cast<uint16_t *>(out), M, N, K, S, threads, 0,
                            S > 1, flags, stream, status, nullptr, nullptr, sx, sw);
}

}  // namespace bf16l
