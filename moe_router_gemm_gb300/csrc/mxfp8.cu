// mxfp8.cu — MXFP8: block-scaled e4m3 operands (32 elements along K share one
// power-of-two E8M0 scale byte).  The quantisation of bf16 activations, and the
// block-scaled linear on warp-level tensor-core MMAs.
//
// Source: the sglang PR #34042 page ("执行摘要", "实现拆解" items 2-3): a dense
// MXFP8 GEMM on SM10x, whose small-batch decode kernels the page reports 2-5x
// faster; weights carry block scales, activations are quantised the same way.
// The format is read as the OCP microscaling MXFP8 format (the page does not
// spell it out): block scale 2^(e - 127) from its byte e, e4m3 elements.
//
// Quantisation (bf16_quant_mxfp8): four threads per 32-value block, eight values
// each.  The block's largest magnitude comes from a quad shuffle; its binary
// exponent L = floor(log2 max|v|) is read from the fp32 exponent field (0 for
// zero and for fp32 subnormals, whose L is below -126 anyway), the scale
// exponent is s = max(L - 8, -127) (8: the exponent of e4m3's largest binade,
// 448 = 1.75 * 2^8), the byte e = s + 127, and each value is multiplied by the
// exact power of two 2^-s and converted with cvt.rn.satfinite.e4m3x2 (round
// to nearest even, saturating at +-448).
//
// Linear (bf16_linear_mxfp8): out = sum over blocks b of 2^(sx[m][b]-127) *
// 2^(sw[n][b]-127) * sum_{k in b} e4m3(xq[m][k]) e4m3(wq[n][k]), + bias, one
// rounding to bf16.  One mma.sync.m16n8k32 e4m3 step is exactly one block:
//   * grid (S, ceil(N/8), ceil(M/16)), clusters of S CTAs along K; CTA (r, q, z)
//     owns W rows 8q..8q+7, tokens 16z..16z+15 and the r-th of S runs of blocks,
//     which its warps split;
//   * lane (g, t) loads 8 bytes of W row g, and of x rows g and g+8, at codes
//     [32b + 8t, +8) of block b: the B fragment and the two A fragment rows of
//     the block's MMA under the k permutation "MMA k 4t+j <-> code 8t+j, MMA k
//     16+4t+j <-> code 8t+4+j" (the same for A and B, so the sum is the block's
//     dot product);
//   * each block's MMA runs on a zeroed fragment, which is scaled by the two
//     scales of its token row and W column (exact powers of two, so only the
//     fp32 accumulation rounds) and added to the running fp32 sum;
//   * warps' sums in warp order in shared memory; ranks 1..S-1 send theirs to
//     rank 0 with st.async counted on its mbarrier; rank 0 sums in rank order,
//     adds bias, rounds, stores.  Two non-.aligned cluster barrier phases, as in
//     the bf16 router kernel.
// The default launch waits for the previous kernel before any read; with
// BF16L_FLAG_PDL the weight codes and scales of the first batch are loaded
// before that wait.
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

namespace bf16l {

namespace {

constexpr int kMxWarps = 8;     // at most 256 threads
constexpr int kMxU = 4;         // blocks per lane per batch (loads in flight)
constexpr int kMxMaxCluster = 16;

// Two fp32 values -> two e4m3 codes, lo in the low byte.
__device__ __forceinline__ uint16_t mx_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// 2^(e - 127) as fp32: a normal number for e >= 1, the subnormal 2^-127 for e == 0.
__device__ __forceinline__ float e8m0_f32(uint32_t e) {
    return e ? __uint_as_float(e << 23) : __uint_as_float(0x00400000u);
}

__global__ void __launch_bounds__(256) quant_mxfp8_kernel(const uint16_t *__restrict__ x, uint8_t *__restrict__ q,
                                                          uint8_t *__restrict__ scales, long long nvec) {
    pdl_launch_dependents();
    pdl_wait();  // x may be written by the previous kernel
    const long long stride = (long long)gridDim.x * blockDim.x;
    // nvec (8-value vectors) is a multiple of 4, and so is stride (256-thread blocks): every
    // quad of lanes stays together through the loop, as the shuffles need.
    for (long long v = (long long)blockIdx.x * blockDim.x + threadIdx.x; v < nvec; v += stride) {
        const uint4 w = __ldg(reinterpret_cast<const uint4 *>(x) + v);
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
        float f[8];
        float amax = 0.0f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            f[2 * j] = bf16_to_f32((uint16_t)(u[j] & 0xFFFFu));
            f[2 * j + 1] = bf16_to_f32((uint16_t)(u[j] >> 16));
            amax = fmaxf(amax, fmaxf(fabsf(f[2 * j]), fabsf(f[2 * j + 1])));
        }
        // the quad's four lanes are in or out of the loop together (nvec % 4 == 0, stride % 4 == 0),
        // but the warp's other quads may have left it: shuffle within the quad only
        const unsigned quad = 0xFu << (threadIdx.x & 28u);
        amax = fmaxf(amax, __shfl_xor_sync(quad, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(quad, amax, 2));
        const int ef = (int)((__float_as_uint(amax) >> 23) & 0xFFu);
        int s = ef == 0 ? -127 : (ef - 127) - 8;
        s = s < -127 ? -127 : s;
        const float inv = __uint_as_float((uint32_t)(127 - s) << 23);  // 2^-s, s in [-127, 119]
        uint16_t c[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) c[j] = mx_e4m3x2(f[2 * j] * inv, f[2 * j + 1] * inv);
        uint2 o;
        o.x = (uint32_t)c[0] | ((uint32_t)c[1] << 16);
        o.y = (uint32_t)c[2] | ((uint32_t)c[3] << 16);
        reinterpret_cast<uint2 *>(q)[v] = o;
        if ((threadIdx.x & 3) == 0) scales[v >> 2] = (uint8_t)(s + 127);
    }
}

template <bool HI, typename OutT>
__global__ void __launch_bounds__(kMxWarps * 32)
    mxfp8_linear_kernel(const uint8_t *__restrict__ xq, const uint8_t *__restrict__ xs,
                        const uint8_t *__restrict__ wq, const uint8_t *__restrict__ ws,
                        const uint16_t *__restrict__ bias, OutT *__restrict__ out, int M, int N, int K, int S,
                        int32_t *status, int w_early) {
    __shared__ float4 part[kMxWarps][32];
    __shared__ float4 recv[kMxMaxCluster][32];
    __shared__ __align__(8) uint64_t rbar;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    const int nw = (int)blockDim.x >> 5;
    const int nb = K >> 5;  // blocks per row
    {  // this CTA's group of 16 tokens
        const int m0 = 16 * (int)blockIdx.z;
        xq += (size_t)m0 * K;
        xs += (size_t)m0 * nb;
        out += (size_t)m0 * N;
        M = (M - m0) < 16 ? (M - m0) : 16;
    }
    const bool clus = S > 1;
    const int rank = clus ? (int)cluster_ctarank() : 0;
    const int n0 = 8 * (int)blockIdx.y;
    const int cb0 = mul_div(nb, rank, S), cb1 = mul_div(nb, rank + 1, S);
    const int b0 = cb0 + mul_div(cb1 - cb0, warp, nw), b1 = cb0 + mul_div(cb1 - cb0, warp + 1, nw);
    if (!w_early) {
        // Default launch: nothing is read before the previous kernel has finished.  Meanwhile this CTA's
        // codes of its 8 rows are fetched into L2 (one request per row, by the first token group only).
        if (blockIdx.z == 0 && tid < 8 && n0 + tid < N && cb1 > cb0)
            prefetch_l2(wq + (size_t)(n0 + tid) * K + (size_t)cb0 * 32, (uint32_t)(cb1 - cb0) * 32u);
        pdl_wait();
    }
    const bool tok_lo = g < M, tok_hi = HI && (g + 8 < M);
    const int row = n0 + g;                                  // this lane's W row (B column g)
    const int na = n0 + 2 * t, nb1 = n0 + 2 * t + 1;         // this lane's accumulator columns
    const uint8_t *wr = wq + (size_t)(row < N ? row : N - 1) * K + 8 * t;
    const uint8_t *xlo = xq + (size_t)(tok_lo ? g : 0) * K + 8 * t;
    const uint8_t *xhi = xq + (size_t)(tok_hi ? g + 8 : 0) * K + 8 * t;
    const uint8_t *wsa = ws + (size_t)(na < N ? na : N - 1) * nb, *wsb = ws + (size_t)(nb1 < N ? nb1 : N - 1) * nb;
    const uint8_t *xsl = xs + (size_t)(tok_lo ? g : 0) * nb, *xsh = xs + (size_t)(tok_hi ? g + 8 : 0) * nb;

    uint2 wv[kMxU];
    uint32_t swa[kMxU], swb[kMxU];
    auto load_w = [&](int bb) {
#pragma unroll
        for (int u = 0; u < kMxU; ++u) {
            const int b = bb + u;
            const bool in = b < b1;
            wv[u] = (in && row < N) ? __ldg(reinterpret_cast<const uint2 *>(wr + 32 * (size_t)b)) : make_uint2(0u, 0u);
            swa[u] = in ? __ldg(wsa + b) : 127u;
            swb[u] = in ? __ldg(wsb + b) : 127u;
        }
    };
    load_w(b0);  // the first batch (after the wait unless the weights may be read early)

    if (tid == 0) {
        mbar_init(&rbar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (clus) cluster_arrive_relaxed();  // phase 1: "my receive barrier is initialised"
    pdl_launch_dependents();
    pdl_wait();  // x may be written, and out still read, by the previous kernel

    float c[4] = {0.f, 0.f, 0.f, 0.f};
    for (int bb = b0; bb < b1; bb += kMxU) {  // warp-uniform trip count: mma.sync is warp-wide
        if (bb != b0) load_w(bb);
        uint2 al[kMxU], ah[kMxU];
        uint32_t sxl[kMxU], sxh[kMxU];
#pragma unroll
        for (int u = 0; u < kMxU; ++u) {
            const int b = bb + u;
            const bool in = b < b1;
            al[u] = (tok_lo && in) ? __ldg(reinterpret_cast<const uint2 *>(xlo + 32 * (size_t)b)) : make_uint2(0u, 0u);
            ah[u] = (HI && tok_hi && in) ? __ldg(reinterpret_cast<const uint2 *>(xhi + 32 * (size_t)b))
                                         : make_uint2(0u, 0u);
            sxl[u] = in ? __ldg(xsl + b) : 127u;
            sxh[u] = (HI && in) ? __ldg(xsh + b) : 127u;
        }
#pragma unroll
        for (int u = 0; u < kMxU; ++u) {
            float d[4] = {0.f, 0.f, 0.f, 0.f};
            // a0 / a2: token g, codes 8t..8t+3 / 8t+4..8t+7; a1 / a3: token g+8; b0 / b1: W row g
            mma_m16n8k32_e4m3(d, al[u].x, ah[u].x, al[u].y, ah[u].y, wv[u].x, wv[u].y);
            const float fl = e8m0_f32(sxl[u]), fh = e8m0_f32(sxh[u]);
            const float fa = e8m0_f32(swa[u]), fb = e8m0_f32(swb[u]);
            c[0] += (d[0] * fl) * fa;
            c[1] += (d[1] * fl) * fb;
            c[2] += (d[2] * fh) * fa;
            c[3] += (d[3] * fh) * fb;
        }
    }
    part[warp][lane] = make_float4(c[0], c[1], c[2], c[3]);
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
    bool have = true;
    if (clus) {
        cluster_wait_acquire();  // phase 1 done: rank 0's receive barrier exists
        if (rank != 0) {
            if (warp == 0)
                st_async_f4(mapa_shared(smem_u32(&recv[rank][lane]), 0), s.x, s.y, s.z, s.w,
                            mapa_shared(smem_u32(&rbar), 0));
        } else {
            if (tid == 0) mbar_arrive_expect_tx(&rbar, (uint32_t)((S - 1) * 32 * 16));
            if (warp == 0) {
                have = mbar_wait_cluster(&rbar, 0, status, kSiteRecv);
                for (int r = 1; r < S; ++r) {  // ranks in order
                    const float4 p = recv[r][lane];
                    s.x += p.x;
                    s.y += p.y;
                    s.z += p.z;
                    s.w += p.w;
                }
            }
        }
        cluster_arrive_relaxed();  // phase 2: everything rank 0 receives has landed
    }
    if (rank == 0 && warp == 0 && have) {
        const float v[4] = {s.x, s.y, s.z, s.w};
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

using MxFn = void (*)(const uint8_t *, const uint8_t *, const uint8_t *, const uint8_t *, const uint16_t *,
                      uint16_t *, int, int, int, int, int32_t *, int);

MxFn pick_mx(int M) { return M > 8 ? mxfp8_linear_kernel<true, uint16_t> : mxfp8_linear_kernel<false, uint16_t>; }

}  // namespace

int init_mxfp8() {
    for (int M : {8, 16}) {
        const int e = (int)cudaFuncSetAttribute(pick_mx(M), cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e) return e;
    }
    return 0;
}

int mxfp8_split(int M, int N, int K, int threads, int num_sms) {
    // The smallest power of two K split that gives about two CTAs per SM, at most 16,
    // with at least one block per warp.
    if (M <= 0 || N <= 0 || K < 32 || num_sms <= 0) return 1;
    const long long base = (long long)((N + 7) / 8) * ((M + 15) / 16);
    const int nb = K / 32, nw = threads / 32;
    int S = 1;
    while (S < 16 && 2 * S * nw <= nb && base * S < 2LL * num_sms) S *= 2;
    return S;
}

int launch_mxfp8(const void *xq, const void *xs, const void *wq, const void *ws, const void *bias, void *out, int M,
                 int N, int K, int S, int threads, uint32_t flags, void *stream, int32_t *status) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)S, (unsigned)((N + 7) / 8), (unsigned)((M + 15) / 16));
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = (cudaStream_t)stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl_attr_of(flags);
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)S;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = S > 1 ? 2 : 1;
    return (int)cudaLaunchKernelEx(&cfg, pick_mx(M), static_cast<const uint8_t *>(xq), static_cast<const uint8_t *>(xs),
                                   static_cast<const uint8_t *>(wq), static_cast<const uint8_t *>(ws),
                                   static_cast<const uint16_t *>(bias), static_cast<uint16_t *>(out), M, N, K, S,
                                   status, w_early_of(flags));
}

int launch_quant_mxfp8(const void *x, void *q, void *scales, long long n, int num_sms, uint32_t flags,
                       void *stream) {
    const long long nvec = n / 8;
    long long blocks = (nvec + 255) / 256;
    const long long cap = 8LL * num_sms;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(256);
    cfg.stream = (cudaStream_t)stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl_attr_of(flags);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return (int)cudaLaunchKernelEx(&cfg, quant_mxfp8_kernel, static_cast<const uint16_t *>(x),
                                   static_cast<uint8_t *>(q), static_cast<uint8_t *>(scales), nvec);
}

}  // namespace bf16l
