// warpmma_ks.cu — the persistent warp-level tensor-core kernel with K split
// over a thread-block cluster (2..16 CTAs), for decode-sized weights and up to 64 tokens.
//
// Prior art: the cluster split-K kernel on the vLLM PR #42562 page ("实现拆解"
// items 2-3): K spread over the CTAs of a cluster, fp32 partial tiles reduced
// through distributed shared memory in a fixed order.
//
// Why a third form of the warp-MMA kernel: with the whole of x staged per CTA
// (warpmma.cu) 16 tokens of K = 7168 (229 KB) do not fit in shared memory, and
// loading x fragments from L2 next to every weight batch moves twice as many
// bytes through L2 as the weights themselves.  Splitting K over S CTAs of a
// cluster shrinks each CTA's x slice S times, so it is staged once per CTA and
// read from shared memory for every weight row the CTA streams.
//   * grid = C clusters of S CTAs; cluster c owns the 8-row groups
//     [RG*c/C, RG*(c+1)/C) of the RG = ceil(N/8); rank r of the cluster owns the
//     r-th of S equal runs of 32-wide K blocks, for every one of those groups;
//   * inside a CTA, groups of WPR warps take one 8-row group at a time and
//     split the rank's K run between them; per 32-wide K block lane (g, t)
//     loads W[n0 + g][kb + 8t, +8) (16 bytes) and the same 16 bytes of tokens
//     16j + g and 16j + g + 8 from the staged slice, for each 16-token tile j
//     (up to 4), and issues two mma.sync.m16n8k16 per tile on them;
//   * the WPR warps' tiles are summed in warp order in shared memory; the
//     group's partial goes to the rank that finishes it (the group's index in
//     the cluster modulo S), by st.async into that rank's receive slot, counted
//     on its mbarrier (a rank's own partial is a plain shared store);
//   * at the end each rank waits for the partials of its own groups, sums the
//     S of them in rank order, adds the bias, rounds and stores;
//   * the next group's first weight batch is loaded before the reductions, and
//     the first one before the programmatic-launch wait and the x copy.
// Two cluster barrier phases (non-.aligned): "receive barrier initialised"
// (arrived at start, waited before any partial is sent) and "done" (before
// exit).  The summation order is fixed, so a plan is bitwise reproducible.
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace bf16l {

namespace {

// Row stride of the staged x slice in 16-byte vectors: 4 (mod 8), so that the
// two token rows a quarter-warp reads land in different halves of the banks.
__host__ __device__ inline int ks_stride(int sv) { return sv + (12 - sv % 8) % 8; }

// Dynamic shared memory: x slice [M][stride], the warps' partial tiles
// [warps][TT][32] float4 (WPR > 1), the receive slots [slots][S][TT][32] float4.
struct KsLayout {
    int part_off, recv_off, bytes;
};
__host__ __device__ inline KsLayout ks_layout(int M, int N, int RB, int S, int C, int nw, int wpr, int tt) {
    const int nvec = RB >> 4, nblk = (nvec + 3) >> 2;
    const int stride_max = 4 * ((nblk + S - 1) / S) + 7;  // >= ks_stride of any rank's slice
    const int RG = (N + 7) >> 3, gmax = (RG + C - 1) / C, slots = (gmax + S - 1) / S;
    KsLayout L;
    L.part_off = M * stride_max * 16;
    L.recv_off = L.part_off + (wpr > 1 ? nw * tt * 512 : 0);
    L.bytes = L.recv_off + slots * S * tt * 512;
    return L;
}

}  // namespace

// WPR warps per 8-row group; NT: block size the instance is compiled for (a
// smaller block runs the 512 instance); TT: 16-token tiles (1, 2 or 4).  TT = 1
// keeps 64 registers a thread (1024 threads per SM); TT > 1 takes 128.
template <int WPR, int NT, int TT, typename OutT>
__global__ void __launch_bounds__(NT, TT == 1 ? 1024 / NT : 1)
    warpmma_ks_kernel(const uint8_t *__restrict__ x, const uint8_t *__restrict__ W, const uint16_t *__restrict__ bias,
                      OutT *__restrict__ out, int M, int N, int RB, int S, int32_t *status, int w_early) {
    constexpr int U = 8;  // K blocks (4 x 16 bytes across a lane quad) per lane per batch
    extern __shared__ __align__(16) uint8_t ks_smem[];
    __shared__ __align__(8) uint64_t xbar, rbar;

    // Only what the first weight batch needs comes before it is issued (all 32-bit).
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    const int grp = warp / WPR, gw = warp - grp * WPR;
    const int rank = (int)cluster_ctarank(), c = (int)cluster_id_x(), C = (int)cluster_count_x();
    // this rank's vectors [cv0, cv1) of every row, and this warp's share of them
    const int nvec = RB >> 4, nblk = (nvec + 3) >> 2;
    const int cb0 = mul_div(nblk, rank, S), cb1 = mul_div(nblk, rank + 1, S);  // floor(nblk * r / S)
    const int cv1 = min(nvec, 4 * cb1);
    const int wb0 = cb0 + (cb1 - cb0) * gw / WPR, wb1 = cb0 + (cb1 - cb0) * (gw + 1) / WPR;
    const int wv0 = 4 * wb0, wv1 = min(cv1, 4 * wb1);
    // this cluster's 8-row groups; rank r finishes local groups i with i % S == r
    const int RG = (N + 7) >> 3;
    const int q0 = mul_div(RG, c, C), q1 = mul_div(RG, c + 1, C);
    if (!w_early) {
        // Default launch: nothing is read before the previous kernel has finished.  Meanwhile this rank's
        // K slice of the rows of its cluster's first 8-row group is fetched into L2 (one request a row).
        const int row = 8 * q0 + tid;
        if (tid < 8 && q1 > q0 && row < N && cv1 > 4 * cb0)
            prefetch_l2(W + (size_t)row * RB + (size_t)cb0 * 64, (uint32_t)(cv1 - 4 * cb0) * 16u);
        pdl_wait();
    }

    uint4 wv[U];
    auto load_batch = [&](int n0, int vb) {  // the batch of blocks starting at vector vb
        const int row = n0 + g;
        const uint4 *wr = reinterpret_cast<const uint4 *>(W + (size_t)(row < N ? row : N - 1) * RB);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int vv = vb + 4 * u + t;
            wv[u] = (vv < wv1 && row < N) ? ldg_stream_v4(wr + vv) : make_uint4(0u, 0u, 0u, 0u);
        }
    };
    // One L2 prefetch per lane of a batch's 32 lines (8 rows x 4 lines of 128 bytes), issued one batch ahead
    // so the next loads find their lines in L2.
    auto prefetch_batch = [&](int qn, int vb) {
        if (qn >= q1 || vb >= wv1) return;
        const int row = 8 * qn + lane / (U / 2);
        const int v = vb + 8 * (lane % (U / 2));  // first 16-byte vector of this lane's line
        if (row < N && v < wv1)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(W + (size_t)row * RB + (size_t)v * 16));
    };
    int q = q0 + grp;
    bool pre = q < q1;
    if (pre) load_batch(8 * q, wv0);

    const int nw = (int)blockDim.x >> 5;
    const int GW = nw / WPR;  // 8-row groups in flight in this CTA
    const KsLayout L = ks_layout(M, N, RB, S, C, nw, WPR, TT);
    uint4 *xs = reinterpret_cast<uint4 *>(ks_smem);
    float4 *part = reinterpret_cast<float4 *>(ks_smem + L.part_off);
    float4 *recv = reinterpret_cast<float4 *>(ks_smem + L.recv_off);
    const int cv0 = 4 * cb0, sv = cv1 - cv0, sp = ks_stride(sv);
    const int own = (q1 - q0) > rank ? (q1 - q0 - rank + S - 1) / S : 0;

    if (tid == 0) {
        mbar_init(&xbar, 1);
        mbar_init(&rbar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (tid == 0 && own > 0) mbar_arrive_expect_tx(&rbar, (uint32_t)(own * (S - 1) * TT * 512));
    cluster_arrive_relaxed();  // phase 1: "my receive barrier is initialised"

    pdl_launch_dependents();
    pdl_wait();  // x may be written, and out still read, by the previous kernel
    const bool stage = q1 > q0 && sv > 0;
    if (tid == 0 && stage) {
        mbar_arrive_expect_tx(&xbar, (uint32_t)(M * sv * 16));
        for (int m = 0; m < M; ++m)
            bulk_load(xs + (size_t)m * sp, x + (size_t)m * RB + (size_t)cv0 * 16, (uint32_t)(sv * 16), &xbar);
    }
    const bool staged = stage ? mbar_wait(&xbar, 0, status, kSiteStage) : true;
    const bool ok = __syncthreads_and(staged) != 0;
    cluster_wait_acquire();  // phase 1 done: every rank's receive barrier exists

    // this lane's token rows in the staged slice, indexed by vector: tokens 16j + g (lo) and 16j + g + 8 (hi)
    const uint4 *xlo = xs + (g * sp - cv0), *xhi = xs + ((g + 8) * sp - cv0);
    const int tstep = 16 * sp;  // vectors from one 16-token tile to the next
    for (; q < q1; q += GW) {
        const int n0 = 8 * q;
        float d[TT][4];
#pragma unroll
        for (int j = 0; j < TT; ++j) d[j][0] = d[j][1] = d[j][2] = d[j][3] = 0.f;
        if (ok) {
            for (int vb = wv0; vb < wv1; vb += 4 * U) {  // warp-uniform trip count: mma.sync is warp-wide
                if (!(pre && vb == wv0)) load_batch(n0, vb);
                if (vb + 4 * U < wv1)
                    prefetch_batch(q, vb + 4 * U);
                else
                    prefetch_batch(q + GW, wv0);
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int vv = vb + 4 * u + t;
                    const bool in = vv < wv1;
#pragma unroll
                    for (int j = 0; j < TT; ++j) {
                        const uint4 lo = (in && 16 * j + g < M) ? xlo[j * tstep + vv] : make_uint4(0u, 0u, 0u, 0u);
                        const uint4 hi = (in && 16 * j + g + 8 < M) ? xhi[j * tstep + vv] : make_uint4(0u, 0u, 0u, 0u);
                        // this lane's 16 block bytes: step 0 takes the first 8, step 1 the last 8
                        mma_m16n8k16_bf16(d[j], lo.x, hi.x, lo.y, hi.y, wv[u].x, wv[u].y);
                        mma_m16n8k16_bf16(d[j], lo.z, hi.z, lo.w, hi.w, wv[u].z, wv[u].w);
                    }
                }
            }
        }
        // the next group's first batch streams in during the reductions
        pre = ok && q + GW < q1;
        if (pre) load_batch(8 * (q + GW), wv0);
        if constexpr (WPR > 1) {
#pragma unroll
            for (int j = 0; j < TT; ++j)
                part[((size_t)warp * TT + j) * 32 + lane] = make_float4(d[j][0], d[j][1], d[j][2], d[j][3]);
            asm volatile("bar.sync %0, %1;" ::"r"(1 + grp), "r"(WPR * 32) : "memory");
            if (gw == 0) {
#pragma unroll
                for (int j = 0; j < TT; ++j) {
                    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
                    for (int w = 0; w < WPR; ++w) {  // warps in order
                        const float4 p = part[((size_t)(grp * WPR + w) * TT + j) * 32 + lane];
                        s0 += p.x;
                        s1 += p.y;
                        s2 += p.z;
                        s3 += p.w;
                    }
                    d[j][0] = s0, d[j][1] = s1, d[j][2] = s2, d[j][3] = s3;
                }
            }
        }
        if (gw == 0) {  // the group's partial to the rank that finishes it
            const int i = q - q0, owner = i % S, slot = i / S;
#pragma unroll
            for (int j = 0; j < TT; ++j) {
                float4 *dst = recv + (((size_t)slot * S + rank) * TT + j) * 32 + lane;
                if (owner == rank)
                    *dst = make_float4(d[j][0], d[j][1], d[j][2], d[j][3]);
                else
                    st_async_f4(mapa_shared(smem_u32(dst), (uint32_t)owner), d[j][0], d[j][1], d[j][2], d[j][3],
                                mapa_shared(smem_u32(&rbar), (uint32_t)owner));
            }
        }
        if constexpr (WPR > 1) asm volatile("bar.sync %0, %1;" ::"r"(1 + grp), "r"(WPR * 32) : "memory");
    }

    // ---- finish this rank's groups: S partials in rank order, bias, round, store ----
    __syncthreads();  // this CTA's own partials are in place
    const int items = own * TT * 32;
    if (tid < items) {
        const bool have = S > 1 ? mbar_wait_cluster(&rbar, 0, status, kSiteRecv) : true;
        for (int it = tid; have && it < items; it += (int)blockDim.x) {
            const int slot = it / (TT * 32), j = (it / 32) % TT, ln = it % 32;
            const int qq = q0 + slot * S + rank;
            float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int r = 0; r < S; ++r) {  // ranks in order
                const float4 p = recv[(((size_t)slot * S + r) * TT + j) * 32 + ln];
                s.x += p.x;
                s.y += p.y;
                s.z += p.z;
                s.w += p.w;
            }
            const float v[4] = {s.x, s.y, s.z, s.w};
            const int gg = ln >> 2, tt = ln & 3;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int m = 16 * j + gg + (e >> 1) * 8, n = 8 * qq + 2 * tt + (e & 1);
                if (m < M && n < N) {
                    float o = v[e];
                    if (bias) o += bf16_to_f32(bias[n]);
                    OutStore<OutT>::one(out + (size_t)m * N + n, o);
                }
            }
        }
    }
    cluster_arrive_relaxed();  // phase 2: this CTA has received everything it waits for
    cluster_wait_acquire();    // every CTA has: all may exit
}

namespace {

template <typename OutT>
using KsFn = void (*)(const uint8_t *, const uint8_t *, const uint16_t *, OutT *, int, int, int, int, int32_t *, int);

// 16-token tiles an instance covers for M tokens (3 tiles run the 4-tile instance).
int ks_tiles(int M) {
    const int tt = (M + 15) / 16;
    return tt <= 2 ? (tt < 1 ? 1 : tt) : 4;
}

template <int WPR, int TT, typename OutT>
KsFn<OutT> pick_ks_nt(int threads) {
    if constexpr (TT == 1)
        return threads > 512 ? warpmma_ks_kernel<WPR, 1024, 1, OutT> : warpmma_ks_kernel<WPR, 512, 1, OutT>;
    return warpmma_ks_kernel<WPR, 512, TT, OutT>;
}

template <int TT, typename OutT>
KsFn<OutT> pick_ks_wpr(int wpr, int threads) {
    switch (wpr) {
        case 1: return pick_ks_nt<1, TT, OutT>(threads);
        case 2: return pick_ks_nt<2, TT, OutT>(threads);
        case 4: return pick_ks_nt<4, TT, OutT>(threads);
        case 8: return pick_ks_nt<8, TT, OutT>(threads);
        case 16: return pick_ks_nt<16, TT, OutT>(threads);
        default: return nullptr;
    }
}

template <typename OutT>
KsFn<OutT> pick_ks(int M, int wpr, int threads) {
    switch (ks_tiles(M)) {
        case 1: return pick_ks_wpr<1, OutT>(wpr, threads);
        case 2: return pick_ks_wpr<2, OutT>(wpr, threads);
        default: return pick_ks_wpr<4, OutT>(wpr, threads);
    }
}

template <typename OutT>
int set_ks_attrs() {
    for (int M : {16, 32, 64})
        for (int wpr : {1, 2, 4, 8, 16})
            for (int t : {512, 1024}) {
                int e = (int)cudaFuncSetAttribute(pick_ks<OutT>(M, wpr, t),
                                                  cudaFuncAttributeMaxDynamicSharedMemorySize, kWarpMmaKsMaxSmem);
                if (!e)
                    e = (int)cudaFuncSetAttribute(pick_ks<OutT>(M, wpr, t),
                                                  cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
                if (e) return e;
            }
    return 0;
}

// Co-resident clusters per (instance, cluster size, block, shared memory,
// device), from the occupancy calculator, kept after the first query.
struct KsOcc {
    const void *fn;
    int S, threads, smem, dev, clusters;
};
std::mutex g_ks_mu;
KsOcc g_ks_occ[64];
int g_ks_nocc = 0;

int ks_max_clusters(const void *fn, int S, int threads, int smem, int dev) {
    std::lock_guard<std::mutex> lock(g_ks_mu);
    for (int i = 0; i < g_ks_nocc; ++i) {
        const KsOcc &o = g_ks_occ[i];
        if (o.fn == fn && o.S == S && o.threads == threads && o.smem == smem && o.dev == dev) return o.clusters;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(S * kGb300Sms));
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    // A failed query only loses the clamp (the launch then uses the plan's grid).
    if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
        n = 0;
        (void)cudaGetLastError();
    }
    if (g_ks_nocc < 64) g_ks_occ[g_ks_nocc++] = KsOcc{fn, S, threads, smem, dev, n};
    return n;
}

template <typename OutT>
int launch_ks_t(const LaunchArgs &a, const bf16l_plan &p) {
    const int S = p.split_k, threads = p.threads, wpr = p.rows_per_cta;
    const KsFn<OutT> fn = pick_ks<OutT>(a.M, wpr, threads);
    if (!fn || S < 2 || p.grid < S) return (int)cudaErrorInvalidValue;
    const int tt = ks_tiles(a.M), nw = threads / 32;
    int C = p.grid / S;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return (int)cudaErrorInvalidDevice;
    // A cluster that cannot be resident with the others would run its groups
    // after them: never launch more clusters than fit at once.
    const int occ = ks_max_clusters(reinterpret_cast<const void *>(fn), S, threads,
                                    ks_layout(a.M, a.N, 2 * a.K, S, C, nw, wpr, tt).bytes, dev);
    if (occ > 0 && C > occ) C = occ;
    const int smem = ks_layout(a.M, a.N, 2 * a.K, S, C, nw, wpr, tt).bytes;
    if (smem > kWarpMmaKsMaxSmem) return (int)cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(C * S));
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = (cudaStream_t)a.stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = pdl_attr_of((uint32_t)p.flags);
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return (int)cudaLaunchKernelEx(&cfg, fn, static_cast<const uint8_t *>(a.x), static_cast<const uint8_t *>(a.W),
                                   static_cast<const uint16_t *>(a.bias), static_cast<OutT *>(a.out), a.M, a.N,
                                   a.K * 2, S, a.status, w_early_of((uint32_t)p.flags));
}

}  // namespace

int warpmma_ks_smem_bytes(int M, int N, int K, int S, int clusters, int threads, int wpr) {
    if (S < 1 || clusters < 1 || threads < 32) return 1 << 30;
    return ks_layout(M, N, 2 * K, S, clusters, threads / 32, wpr, ks_tiles(M)).bytes;
}

int init_warpmma_ks() {
    int e = set_ks_attrs<uint16_t>();
    if (!e) e = set_ks_attrs<float>();
    return e;
}

int launch_warpmma_ks(const LaunchArgs &a, const bf16l_plan &p) {
    return a.out_f32 ? launch_ks_t<float>(a, p) : launch_ks_t<uint16_t>(a, p);
}

}  // namespace bf16l
