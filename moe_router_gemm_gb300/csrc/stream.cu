// stream.cu — persistent weight-streaming kernel for few tokens and large N.
//
// Prior art: the dot-product router kernel on the vLLM PR #42562 page (one CTA
// per expert, 128-bit weight loads, fp32 FMA over every token, warp-shuffle and
// shared-memory reduction).  That layout launches one CTA per row; for decode
// and MLP weights (N = 2K..14K rows, 30..120 MB) it runs in many waves and each
// wave pays the full DRAM latency again.
//
// This kernel keeps the CUDA-core arithmetic and changes the data movement:
//   * one CTA per SM (persistent) owns a contiguous range of W rows, which is
//     one contiguous byte range of the row-major weight;
//   * a producer warp streams that range through a `stages`-deep ring in
//     row-groups of RG rows — each group is contiguous, so one untiled bulk
//     copy (cp.async.bulk, no tensor-map descriptor) fills a stage — and refills
//     a stage as soon as the compute warps release it;
//   * the 8 compute warps split K: warp w always handles the same K slice, so
//     its lanes hold their slice of x (MT <= 4 tokens) in registers for the
//     whole kernel and read only W from shared memory;
//   * per row-group each warp writes its MT x RG partial sums to shared memory
//     and one warp sums the 8 partials in warp order (deterministic), adds the
//     bias, rounds and stores.
//   * Programmatic dependent launch: the first weight stages go out before the
//     grid-dependency wait; x and out are touched only after it.
#include "common.cuh"
#include "kernels.h"

namespace bf16l {

namespace {

constexpr int kStreamComputeWarps = 8;
static_assert(kStreamThreads == (kStreamComputeWarps + 1) * 32, "8 compute warps + one producer warp");
constexpr int kStreamMaxRG = kStreamMaxRows;

struct StreamShared {
    uint64_t full[kStreamMaxStages];
    uint64_t empty[kStreamMaxStages];
    float red[2][kStreamComputeWarps][kStreamMaxRG * kStreamMaxTokens];  // double-buffered partials
};

}  // namespace

int stream_smem_bytes(int K, int rg, int stages) {
    return 128 /*alignment*/ + stages * rg * K * 2 + (int)sizeof(StreamShared);
}

template <int MT, int RG, typename OutT>
__global__ void __launch_bounds__(kStreamThreads, 1)
    stream_kernel(const uint16_t *__restrict__ x, const uint16_t *__restrict__ W, const uint16_t *__restrict__ bias,
                  OutT *__restrict__ out, int M, int N, int K, int rg_unused, int stages, int32_t *status,
                  int w_early) {
    if (!w_early) {
        // Default launch: nothing is read before the previous kernel has finished.  Meanwhile the start of
        // this CTA's contiguous row range is fetched into L2.
        if (threadIdx.x == 0) {
            const int p0 = mul_div(N, (int)blockIdx.x, (int)gridDim.x), p1 = mul_div(N, (int)blockIdx.x + 1, (int)gridDim.x);
            const uint32_t bytes = (uint32_t)(p1 - p0) * (uint32_t)K * 2u;  // at most the first 64 KB
            if (p1 > p0) prefetch_l2(W + (size_t)p0 * K, bytes < 65536u ? bytes : 65536u);
        }
        pdl_wait();
    }
    constexpr int rg = RG;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *ring = smem_raw + (((raw + 127u) & ~127u) - raw);
    const int stage_bytes = rg * K * 2;
    StreamShared &sh = *reinterpret_cast<StreamShared *>(ring + stages * stage_bytes);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = (int)gridDim.x, b = (int)blockIdx.x;
    const int r0 = mul_div(N, b, G), r1 = mul_div(N, b + 1, G);
    const int nrows = r1 - r0;
    const int ngroups = (nrows + rg - 1) / rg;
    const int first = ngroups < stages ? ngroups : stages;
    const int nvec = K / 8;

    if (tid == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&sh.full[s], 1);
            mbar_init(&sh.empty[s], kStreamComputeWarps);
        }
        fence_barrier_init();
        for (int g = 0; g < first; ++g) {
            const int rows = (nrows - g * rg) < rg ? (nrows - g * rg) : rg;
            const uint32_t bytes = (uint32_t)(rows * K * 2);
            mbar_arrive_expect_tx(&sh.full[g], bytes);
            bulk_load(ring + g * stage_bytes, W + (size_t)(r0 + g * rg) * K, bytes, &sh.full[g]);
        }
    }
    pdl_launch_dependents();
    pdl_wait();  // x may be written, and out still read, by the previous kernel
    __syncthreads();

    if (warp == kStreamComputeWarps) {
        if (lane == 0) {  // ---- producer: refill each stage once its row-group is consumed ----
            for (int g = first; g < ngroups; ++g) {
                const int s = g % stages;
                if (!mbar_wait(&sh.empty[s], ((g / stages) - 1) & 1, status, kSiteEmpty)) break;
                const int rows = (nrows - g * rg) < rg ? (nrows - g * rg) : rg;
                const uint32_t bytes = (uint32_t)(rows * K * 2);
                mbar_arrive_expect_tx(&sh.full[s], bytes);
                bulk_load(ring + s * stage_bytes, W + (size_t)(r0 + g * rg) * K, bytes, &sh.full[s]);
            }
        }
        return;  // the producer takes no part in the compute warps' barriers below
    }

    // ---- compute warps: warp w owns K vectors [v0, v1) for every row ----
    const int per_warp = (nvec + kStreamComputeWarps - 1) / kStreamComputeWarps;
    const int v0 = warp * per_warp;
    const int v1 = (v0 + per_warp) < nvec ? (v0 + per_warp) : nvec;
    constexpr int kMaxVec = kStreamMaxK / (8 * 32 * kStreamComputeWarps);  // x vectors per lane in registers
    uint4 xv[kMaxVec][MT];
#pragma unroll
    for (int i = 0; i < kMaxVec; ++i) {
        const int v = v0 + lane + 32 * i;
#pragma unroll
        for (int m = 0; m < MT; ++m)
            xv[i][m] = (v < v1 && m < M) ? __ldg(reinterpret_cast<const uint4 *>(x + (size_t)m * K) + v)
                                         : make_uint4(0u, 0u, 0u, 0u);
    }

    for (int g = 0; g < ngroups; ++g) {
        const int s = g % stages;
        const int rows = (nrows - g * rg) < rg ? (nrows - g * rg) : rg;
        const bool ok = mbar_wait(&sh.full[s], (g / stages) & 1, status, kSiteFull);
        const uint4 *wst = reinterpret_cast<const uint4 *>(ring + s * stage_bytes);
        float acc[RG][MT];
#pragma unroll
        for (int r = 0; r < RG; ++r)
#pragma unroll
            for (int m = 0; m < MT; ++m) acc[r][m] = 0.f;
        if (ok) {
#pragma unroll
            for (int i = 0; i < kMaxVec; ++i) {
                const int v = v0 + lane + 32 * i;
                if (v >= v1) break;
#pragma unroll
                for (int r = 0; r < RG; ++r) {
                    if (r >= rows) break;
                    const uint4 w = wst[(size_t)r * nvec + v];
#pragma unroll
                    for (int m = 0; m < MT; ++m) {  // mixed-precision fma: exact products, fp32 sums
                        const uint4 xx = xv[i][m];
                        float a = acc[r][m];
                        a = fma2_bf16(xx.x, w.x, a);
                        a = fma2_bf16(xx.y, w.y, a);
                        a = fma2_bf16(xx.z, w.z, a);
                        a = fma2_bf16(xx.w, w.w, a);
                        acc[r][m] = a;
                    }
                }
            }
        }
        // Warp reduction, then this warp's partials to shared memory; the stage is free.
        float(*red)[kStreamMaxRG * kStreamMaxTokens] = sh.red[g & 1];
#pragma unroll
        for (int r = 0; r < RG; ++r)
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                float v = acc[r][m];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
                if (lane == 0 && r < rows) red[warp][r * MT + m] = v;
            }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.empty[s]);
        // All compute warps' partials of this group are in: warp 0 finishes the outputs.
        asm volatile("bar.sync 1, %0;" ::"n"(kStreamComputeWarps * 32) : "memory");
        if (warp == 0 && lane < rows * MT) {
            const int r = lane / MT, m = lane % MT;
            if (m < M) {
                float sum = 0.f;
#pragma unroll
                for (int w = 0; w < kStreamComputeWarps; ++w) sum += red[w][lane];
                const int n = r0 + g * rg + r;
                if (bias) sum += bf16_to_f32(bias[n]);
                OutStore<OutT>::one(out + (size_t)m * N + n, sum);
            }
        }
    }
}

namespace {

template <typename OutT>
using StreamFn = void (*)(const uint16_t *, const uint16_t *, const uint16_t *, OutT *, int, int, int, int, int,
                          int32_t *, int);

template <int MT, typename OutT>
StreamFn<OutT> pick_rg(int RG) {
    switch (RG) {
        case 1: return stream_kernel<MT, 1, OutT>;
        case 2: return stream_kernel<MT, 2, OutT>;
        case 4: return stream_kernel<MT, 4, OutT>;
        default: return nullptr;
    }
}

template <typename OutT>
StreamFn<OutT> pick_stream(int MT, int RG) {
    switch (MT) {
        case 1: return pick_rg<1, OutT>(RG);
        case 2: return pick_rg<2, OutT>(RG);
        case 3: return pick_rg<3, OutT>(RG);
        case 4: return pick_rg<4, OutT>(RG);
        default: return nullptr;
    }
}

template <typename OutT>
int launch_stream_t(const LaunchArgs &a, const bf16l_plan &p) {
    StreamFn<OutT> fn = pick_stream<OutT>(a.M, p.rows_per_cta);
    if (!fn) return (int)cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.grid);
    cfg.blockDim = dim3(kStreamThreads);
    cfg.dynamicSmemBytes = (size_t)stream_smem_bytes(a.K, p.rows_per_cta, p.stages);
    cfg.stream = (cudaStream_t)a.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl_attr_of((uint32_t)p.flags);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return (int)cudaLaunchKernelEx(&cfg, fn, static_cast<const uint16_t *>(a.x), static_cast<const uint16_t *>(a.W),
                                   static_cast<const uint16_t *>(a.bias), static_cast<OutT *>(a.out), a.M, a.N, a.K,
                                   p.rows_per_cta, p.stages, a.status, w_early_of((uint32_t)p.flags));
}

template <typename OutT>
int set_stream_attrs() {
    for (int MT = 1; MT <= kStreamMaxTokens; ++MT)
        for (int RG : {1, 2, 4}) {
            const int e = (int)cudaFuncSetAttribute(pick_stream<OutT>(MT, RG),
                                                    cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
            if (e) return e;
        }
    return 0;
}

}  // namespace

int init_stream() {
    int e = set_stream_attrs<uint16_t>();
    if (!e) e = set_stream_attrs<float>();
    return e;
}

int launch_stream(const LaunchArgs &a, const bf16l_plan &p) {
    return a.out_f32 ? launch_stream_t<float>(a, p) : launch_stream_t<uint16_t>(a, p);
}

}  // namespace bf16l
