// splitk.cu — cluster split-K kernel on the 5th-generation tensor cores.
//
// Prior art: the LLBf16SplitK kernel on the vLLM PR #42562 page ("实现拆解"
// item 2 and its source excerpt): K split over the CTAs of one thread-block
// cluster (8 by default), a warp-specialised DMA/MMA pipeline, fp32 partial
// tiles reduced across the cluster through distributed shared memory
// (st.shared::cluster), non-.aligned cluster barriers (its review found the
// .aligned forms hung), fp32 logits out.
//
// On sm_103a this is rebuilt around tcgen05 instead of mma.sync:
//   * swap-AB: 128 weight rows sit on the MMA M side and the (few) tokens,
//     padded to TOK = 16..64, on the MMA N side, so one 128 x TOK x 16
//     tcgen05.mma does the work of a whole warpgroup of m16n8k16 MMAs and the
//     fp32 accumulator lives in TMEM (TOK columns), not in registers;
//   * one thread issues TMA tile loads (128-byte swizzle, out-of-bounds rows
//     and K-columns zero-filled) of W[n0:n0+128, kslice] and x[0:TOK, kslice]
//     into a `stages`-deep ring of 64-wide K chunks, all issued at once when
//     the slice fits, so every CTA has its whole weight slice in flight;
//   * one thread issues the MMAs and frees each stage with tcgen05.commit;
//   * all four warps then move the accumulator TMEM -> registers -> shared
//     memory, and after a cluster barrier each CTA reduces a 1/S share of the
//     tile by reading the S partials over DSMEM (ld.shared::cluster) in rank
//     order (deterministic), adds the bias, rounds to bf16 and stores.
//
// Grid: (S, ceil(N/128)) with cluster dims (S, 1, 1); rank r of a cluster
// takes K chunks [r*C/S, (r+1)*C/S) of the C = ceil(K/64) chunks.
#include "common.cuh"
#include "kernels.h"

namespace bf16l {

namespace {

constexpr int kRows = kSplitRows;               // 128 W rows per CTA (MMA M)
constexpr int kSmemPerSm = 233472;              // 228 KB of shared memory per SM on sm_103
constexpr int kWTileBytes = kRows * kChunkK * 2;  // 16 KB per stage

template <int TOK>
struct SplitCfg {
    static constexpr int kXTileBytes = TOK * kChunkK * 2;
    static constexpr int kStageBytes = kWTileBytes + kXTileBytes;  // multiple of 1024
    static constexpr int kPartBytes = TOK * kRows * 4;            // fp32 partial tile [TOK][128]
    static constexpr int kTmemCols = TOK <= 32 ? 32 : 64;
    static constexpr uint32_t kIdesc = idesc_bf16_f32(kRows, TOK);
    // Shared memory per CTA.  Padded so that the CTAs that fit on one SM can
    // never ask for more than the SM's 512 TMEM columns between them (an
    // allocation that cannot be satisfied would stall its CTA).
    static int smem_bytes(int stages) {
        const int ring = stages * kStageBytes;
        int bytes = 1024 /*alignment slack*/ + (ring > kPartBytes ? ring : kPartBytes) + 256 /*barriers*/;
        const int min_bytes = kSmemPerSm / (512 / kTmemCols);
        return bytes > min_bytes ? bytes : min_bytes;
    }
};

struct SplitShared {  // bookkeeping placed after the ring
    uint64_t full[kSplitMaxStages];
    uint64_t empty[kSplitMaxStages];
    uint64_t accum;
    uint32_t tmem_base;
    int32_t aborted;   // set when a wait gave up: skip the rest of the math
    int32_t issued;    // TMA chunks issued by the producer
    int32_t consumed;  // chunks whose data the MMA issuer saw arrive
};

}  // namespace

template <int TOK>
__global__ void __launch_bounds__(kSplitThreads, 1)
    splitk_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                  const uint16_t *__restrict__ bias, uint16_t *__restrict__ out, int M, int N, int K, int stages,
                  int32_t *status) {
    using Cfg = SplitCfg<TOK>;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned ring (required by the 128-byte swizzle layout).
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *ring = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const int ring_bytes = stages * Cfg::kStageBytes > Cfg::kPartBytes ? stages * Cfg::kStageBytes : Cfg::kPartBytes;
    SplitShared &sh = *reinterpret_cast<SplitShared *>(ring + ring_bytes);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank();
    const int S = (int)gridDim.x;  // cluster spans the whole x dimension of the grid
    const int n0 = blockIdx.y * kRows;
    const int C = (K + kChunkK - 1) / kChunkK;
    const int c_begin = (int)(((long long)rank * C) / S);
    const int c_end = (int)(((long long)(rank + 1) * C) / S);
    const int nchunks = c_end - c_begin;

    if (tid == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&sh.full[s], 1);
            mbar_init(&sh.empty[s], 1);
        }
        mbar_init(&sh.accum, 1);
        sh.aborted = 0;
        sh.issued = 0;
        sh.consumed = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(&sh.tmem_base, Cfg::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;

    if (warp == 0) {
        if (lane == 0) {  // ---- TMA producer ----
            tma_prefetch_desc(&tm_w);
            tma_prefetch_desc(&tm_x);
            int i = 0;
            for (; i < nchunks; ++i) {
                const int s = i % stages;
                if (i >= stages && !mbar_wait(&sh.empty[s], ((i / stages) - 1) & 1, status, kSiteEmpty)) {
                    atomicExch(&sh.aborted, 1);
                    break;
                }
                uint8_t *st = ring + s * Cfg::kStageBytes;
                mbar_arrive_expect_tx(&sh.full[s], Cfg::kStageBytes);
                const int kc = (c_begin + i) * kChunkK;
                tma_load_2d(st, &tm_w, &sh.full[s], kc, n0);
                tma_load_2d(st + kWTileBytes, &tm_x, &sh.full[s], kc, 0);
            }
            sh.issued = i;
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {  // ---- MMA issuer ----
            int i = 0;
            for (; i < nchunks; ++i) {
                const int s = i % stages;
                if (!mbar_wait(&sh.full[s], (i / stages) & 1, status, kSiteFull)) {
                    atomicExch(&sh.aborted, 1);
                    break;
                }
                tc_fence_after();
                const uint8_t *st = ring + s * Cfg::kStageBytes;
                const uint64_t adesc = smem_desc_sw128(smem_u32(st));
                const uint64_t bdesc = smem_desc_sw128(smem_u32(st + kWTileBytes));
#pragma unroll
                for (int kk = 0; kk < kChunkK / 16; ++kk)  // 4 MMAs of K = 16 (32 bytes) each
                    mma_bf16(tmem, adesc + 2 * kk, bdesc + 2 * kk, Cfg::kIdesc, (i > 0 || kk > 0) ? 1u : 0u);
                mma_commit(&sh.empty[s]);
            }
            sh.consumed = i;
            if (i == nchunks)
                mma_commit(&sh.accum);  // accumulator complete
            else
                mbar_arrive(&sh.accum);  // gave up: release the epilogue at once
        }
        __syncwarp();
    }

    // ---- epilogue, all four warps: TMEM -> shared partial [TOK][128] ----
    float *part = reinterpret_cast<float *>(ring);  // overlays the (consumed) ring
    const bool ok = mbar_wait(&sh.accum, 0, status, kSiteAccum);
    tc_fence_after();
    if (ok && !*((volatile int32_t *)&sh.aborted)) {
        const int row = warp * 32 + lane;  // TMEM lane == W row within the tile
#pragma unroll
        for (int c = 0; c < TOK; c += 16) {
            float v[16];
            tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c, v);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j) part[(c + j) * kRows + row] = v[j];
        }
    }
    tc_fence_before();
    cluster_sync();  // every CTA's partial is written and visible cluster-wide

    // ---- distributed reduction: this CTA owns items [r*T/S, (r+1)*T/S) of T = M*32 float4s ----
    const bool aborted = *((volatile int32_t *)&sh.aborted) != 0;
    if (!aborted) {
        const int T = M * (kRows / 4);
        const int it0 = (int)(((long long)rank * T) / S), it1 = (int)(((long long)(rank + 1) * T) / S);
        const uint32_t part_addr = smem_u32(part);
        for (int it = it0 + tid; it < it1; it += kSplitThreads) {
            const int m = it / (kRows / 4), g = it % (kRows / 4);
            const uint32_t off = (uint32_t)((m * kRows + 4 * g) * 4);
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int q = 0; q < S; ++q) {
                const float4 v = ld_dsmem_f4(mapa_shared(part_addr + off, (uint32_t)q));
                acc.x += v.x;
                acc.y += v.y;
                acc.z += v.z;
                acc.w += v.w;
            }
            const int n = n0 + 4 * g;
            float r4[4] = {acc.x, acc.y, acc.z, acc.w};
            if (bias) {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (n + j < N) r4[j] += bf16_to_f32(bias[n + j]);
            }
            const size_t o = (size_t)m * N + n;
            if (n + 3 < N && (o & 3) == 0) {
                uint2 pk;
                pk.x = pack_bf16x2(r4[0], r4[1]);
                pk.y = pack_bf16x2(r4[2], r4[3]);
                *reinterpret_cast<uint2 *>(out + o) = pk;
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (n + j < N) out[o + j] = f32_to_bf16(r4[j]);
            }
        }
    }

    // Drain TMA copies that were issued but never consumed (only after a timeout).
    if (tid == 0) {
        for (int i = sh.consumed; i < sh.issued; ++i)
            mbar_wait(&sh.full[i % stages], (i / stages) & 1, status, kSiteDrain);
    }
    cluster_sync();  // peers have finished reading this CTA's partial
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, Cfg::kTmemCols);
    }
}

namespace {

template <int TOK>
int set_attrs() {
    auto fn = splitk_kernel<TOK>;
    int e = (int)cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      SplitCfg<TOK>::smem_bytes(kSplitMaxStages));
    if (!e) e = (int)cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return e;
}

template <int TOK>
int launch(const LaunchArgs &a, const bf16l_plan &p) {
    CUtensorMap tw, tx;
    int r = make_tmap_bf16_2d(&tw, a.W, (uint64_t)a.N, (uint64_t)a.K, kRows, kChunkK, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    if (r) return (int)cudaErrorInvalidValue;
    r = make_tmap_bf16_2d(&tx, a.x, (uint64_t)a.M, (uint64_t)a.K, TOK, kChunkK, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    if (r) return (int)cudaErrorInvalidValue;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.split_k, (unsigned)((a.N + kRows - 1) / kRows), 1);
    cfg.blockDim = dim3(kSplitThreads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)SplitCfg<TOK>::smem_bytes(p.stages);
    cfg.stream = (cudaStream_t)a.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)p.split_k;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return (int)cudaLaunchKernelEx(&cfg, splitk_kernel<TOK>, tw, tx, static_cast<const uint16_t *>(a.bias),
                                   static_cast<uint16_t *>(a.out), a.M, a.N, a.K, p.stages, a.status);
}

}  // namespace

int init_splitk() {
    int e = set_attrs<16>();
    if (!e) e = set_attrs<32>();
    if (!e) e = set_attrs<48>();
    if (!e) e = set_attrs<64>();
    return e;
}

int launch_splitk(const LaunchArgs &a, const bf16l_plan &p) {
    switch (p.tokens_per_cta) {
        case 16: return launch<16>(a, p);
        case 32: return launch<32>(a, p);
        case 48: return launch<48>(a, p);
        case 64: return launch<64>(a, p);
        default: return (int)cudaErrorInvalidValue;
    }
}

}  // namespace bf16l
