// tile.cu — persistent warp-specialised tcgen05 tile GEMM for large M.
//
// Prior art: the TGV BF16 GEMM kernel on the sglang PR #30117 page (header
// comment of cutedsl_bf16_gemm.py): 256 threads in 8 warps — warp 0 loads A
// with TMA, warp 1 loads B with TMA (and waits on the programmatic grid
// dependency), warp 2 issues tcgen05.mma into TMEM and owns its
// allocation, warps 4-7 run the epilogue TMEM -> registers -> bf16 ->
// st.global; K tiles of 128; a table of (cta_m, cta_n, stages, 2-CTA) tactics.
//
// This kernel keeps the roles and rebuilds the rest for large-M prefill on
// GB300, where the problem is a dense contraction bound by the tensor pipe:
//   * tile 128 (x rows, MMA M) x 256 (W rows, MMA N), K in 64-wide chunks
//     (one 128-byte swizzle row), a 4-stage TMA ring of 48 KB stages;
//   * one producer thread loads both operands (one expect_tx per stage);
//   * one MMA thread issues 4 x tcgen05.mma (128 x 256 x 16) per chunk and
//     frees the stage with tcgen05.commit;
//   * the fp32 accumulator is double-buffered in TMEM (2 x 256 columns = all
//     512), so the epilogue of tile i overlaps the MMAs of tile i+1;
//   * persistent grid (one CTA per SM) walking the tiles in groups of 8 N-tiles
//     (N fastest inside a group, then M), so the ~150 CTAs running together
//     cover about 19 x-tiles times 8 W-tiles and both operands are re-read
//     from L2 rather than HBM;
//   * epilogue: 4 warps, TMEM lane = output row; 32 columns at a time ->
//     + bias -> bf16 (RNE) -> 16-byte stores.
// Waits are bounded (1 s) and record their site in the status word.
#include "common.cuh"
#include "kernels.h"

namespace bf16l {

namespace {

constexpr int kBM = kTileBM;                     // 128
constexpr int kBN = kTileBN;                     // 256
constexpr int kABytes = kBM * kChunkK * 2;       // 16 KB
constexpr int kBBytes = kBN * kChunkK * 2;       // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;   // 48 KB
constexpr int kAccCols = kBN;                    // fp32 accumulator columns per buffer
constexpr int kTmemCols = 2 * kAccCols;          // double buffer = all 512 columns
constexpr uint32_t kIdesc = idesc_bf16_f32(kBM, kBN);
constexpr uint32_t kIdescF8 = idesc_e4m3_f32(kBM, kBN);
constexpr int kGroupN = 8;                       // N tiles per raster group

struct TileShared {
    uint64_t full[kTileMaxStages];
    uint64_t empty[kTileMaxStages];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint32_t tmem_base;
    int32_t aborted;
    int32_t issued;    // chunks the producer put in flight
    int32_t consumed;  // chunks whose arrival the MMA thread saw
};

__device__ __forceinline__ void tile_coords(int t, int m_tiles, int n_tiles, int &m0, int &n0) {
    // Groups of kGroupN N-tiles; inside a group N varies fastest, then M.
    const int per_group = kGroupN * m_tiles;
    const int g = t / per_group, r = t - g * per_group;
    const int gn = (n_tiles - g * kGroupN) < kGroupN ? (n_tiles - g * kGroupN) : kGroupN;
    const int mi = r / gn, ni = g * kGroupN + (r - mi * gn);
    m0 = mi * kBM;
    n0 = ni * kBN;
}

}  // namespace

// F8: x and W are e4m3 codes (per-tensor FP8).  A 128-byte swizzle row then
// holds 128 codes instead of 64 bf16 values, each MMA (kind::f8f6f4) takes 32
// of them, and the epilogue scales the fp32 sum by *scale_x * *scale_w before
// bias; the shared-memory geometry of a stage is the same.  K counts elements.
template <typename OutT, bool F8 = false>
__global__ void __launch_bounds__(kTileThreads, 1)
    tile_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                const uint16_t *__restrict__ bias, OutT *__restrict__ out, int M, int N, int K, int stages,
                int32_t *status, const float *__restrict__ scale_x = nullptr,
                const float *__restrict__ scale_w = nullptr) {
    constexpr int kChunk = F8 ? 2 * kChunkK : kChunkK;  // elements per 128-byte row
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *ring = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    TileShared &sh = *reinterpret_cast<TileShared *>(ring + stages * kStageBytes);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int m_tiles = (M + kBM - 1) / kBM, n_tiles = (N + kBN - 1) / kBN;
    const int num_tiles = m_tiles * n_tiles;
    const int C = (K + kChunk - 1) / kChunk;

    if (tid == 0) {
        tma_prefetch_desc(&tm_x);
        tma_prefetch_desc(&tm_w);
        for (int s = 0; s < stages; ++s) {
            mbar_init(&sh.full[s], 1);
            mbar_init(&sh.empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sh.acc_full[b], 1);
            mbar_init(&sh.acc_empty[b], 4);  // one arrival per epilogue warp
        }
        sh.aborted = 0;
        sh.issued = 0;
        sh.consumed = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(&sh.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;
    pdl_launch_dependents();

    if (warp == 0) {
        if (lane == 0) {  // ---- TMA producer ----
            pdl_wait();
            int it = 0;  // global chunk counter across tiles (ring position)
            for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
                int m0, n0;
                tile_coords(t, m_tiles, n_tiles, m0, n0);
                for (int c = 0; c < C; ++c, ++it) {
                    const int s = it % stages;
                    if (it >= stages && !mbar_wait(&sh.empty[s], ((it / stages) - 1) & 1, status, kSiteEmpty)) {
                        atomicExch(&sh.aborted, 1);
                        goto producer_done;
                    }
                    if (*((volatile int32_t *)&sh.aborted)) goto producer_done;
                    uint8_t *st = ring + s * kStageBytes;
                    mbar_arrive_expect_tx(&sh.full[s], kStageBytes);
                    tma_load_2d(st, &tm_x, &sh.full[s], c * kChunk, m0);
                    tma_load_2d(st + kABytes, &tm_w, &sh.full[s], c * kChunk, n0);
                }
            }
        producer_done:
            sh.issued = it;
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {  // ---- MMA issuer ----
            int it = 0, tile_iter = 0;
            for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++tile_iter) {
                sh.consumed = it;
                const int b = tile_iter & 1;
                const uint32_t acc = tmem + (uint32_t)(b * kAccCols);
                // Wait for the epilogue to have drained this buffer (used two tiles ago).
                if (tile_iter >= 2 &&
                    !mbar_wait(&sh.acc_empty[b], ((tile_iter / 2) - 1) & 1, status, kSiteTmemEmpty)) {
                    atomicExch(&sh.aborted, 1);
                    break;
                }
                tc_fence_after();
                bool ok = true;
                for (int c = 0; c < C; ++c, ++it) {
                    const int s = it % stages;
                    if (!mbar_wait(&sh.full[s], (it / stages) & 1, status, kSiteFull)) {
                        atomicExch(&sh.aborted, 1);
                        sh.consumed = it;
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint8_t *st = ring + s * kStageBytes;
                    const uint64_t adesc = smem_desc_sw128(smem_u32(st));
                    const uint64_t bdesc = smem_desc_sw128(smem_u32(st + kABytes));
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {  // 32 bytes of each row per MMA
                        if constexpr (F8)
                            mma_e4m3(acc, adesc + 2 * kk, bdesc + 2 * kk, kIdescF8, (c > 0 || kk > 0) ? 1u : 0u);
                        else
                            mma_bf16(acc, adesc + 2 * kk, bdesc + 2 * kk, kIdesc, (c > 0 || kk > 0) ? 1u : 0u);
                    }
                    mma_commit(&sh.empty[s]);
                }
                if (!ok) {
                    mbar_arrive(&sh.acc_full[b]);  // release the epilogue at once
                    break;
                }
                mma_commit(&sh.acc_full[b]);
            }
            sh.consumed = it;
        }
        __syncwarp();
    } else {
        // ---- epilogue: warps 2..5; TMEM lane quarter = warp % 4 ----
        const int q = warp & 3;
        const int row = q * 32 + lane;
        int tile_iter = 0;
        const bool vec_ok = (N % 8) == 0;
        for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++tile_iter) {
            int m0, n0;
            tile_coords(t, m_tiles, n_tiles, m0, n0);
            const int b = tile_iter & 1;
            const bool ok = mbar_wait(&sh.acc_full[b], (tile_iter / 2) & 1, status, kSiteAccum);
            tc_fence_after();
            const bool have = ok && !*((volatile int32_t *)&sh.aborted);
            const int m = m0 + row;
            const uint32_t acc = tmem + (uint32_t)(b * kAccCols) + ((uint32_t)(q * 32) << 16);
            if (have) {
                pdl_wait();
                const float sxw = F8 ? __ldg(scale_x) * __ldg(scale_w) : 1.0f;
#pragma unroll 1
                for (int c = 0; c < kBN; c += 32) {
                    uint32_t r0[16], r1[16];
                    tmem_ld16(acc + (uint32_t)c, r0);
                    tmem_ld16(acc + (uint32_t)(c + 16), r1);
                    tmem_ld_wait16(r0);
                    tmem_ld_wait16(r1);
                    const int n = n0 + c;
                    if (m < M && n < N) {
                        float v[32];
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            v[j] = __uint_as_float(r0[j]);
                            v[16 + j] = __uint_as_float(r1[j]);
                        }
                        if constexpr (F8) {
#pragma unroll
                            for (int j = 0; j < 32; ++j) v[j] *= sxw;
                        }
                        if (bias) {
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                if (n + j < N) v[j] += bf16_to_f32(bias[n + j]);
                        }
                        OutT *o = out + (size_t)m * N + n;
                        if (vec_ok && n + 32 <= N) {
#pragma unroll
                            for (int j = 0; j < 32; j += 8) OutStore<OutT>::eight(o + j, v + j);
                        } else {
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                if (n + j < N) OutStore<OutT>::one(o + j, v[j]);
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.acc_empty[b]);
            if (!have) break;
        }
    }

    tc_fence_before();
    __syncthreads();
    // Drain TMA copies that were issued but never consumed (only after a timeout).
    if (tid == 0) {
        for (int i = sh.consumed; i < sh.issued; ++i)
            mbar_wait(&sh.full[i % stages], (i / stages) & 1, status, kSiteDrain);
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

int tile_smem_bytes(int stages) { return 1024 + stages * kStageBytes + 256; }

int init_tile() {
    int e = (int)cudaFuncSetAttribute(tile_kernel<uint16_t>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      tile_smem_bytes(kTileMaxStages));
    if (!e)
        e = (int)cudaFuncSetAttribute(tile_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      tile_smem_bytes(kTileMaxStages));
    if (!e)
        e = (int)cudaFuncSetAttribute(tile_kernel<uint16_t, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      tile_smem_bytes(kTileMaxStages));
    return e;
}

template <typename OutT>
static int launch_tile_t(const LaunchArgs &a, const bf16l_plan &p) {
    CUtensorMap tx, tw;
    int r = make_tmap_bf16_2d(&tx, a.x, (uint64_t)a.M, (uint64_t)a.K, kBM, kChunkK, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    if (r) return (int)cudaErrorInvalidValue;
    r = make_tmap_bf16_2d(&tw, a.W, (uint64_t)a.N, (uint64_t)a.K, kBN, kChunkK, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    if (r) return (int)cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.grid);
    cfg.blockDim = dim3(kTileThreads);
    cfg.dynamicSmemBytes = (size_t)tile_smem_bytes(p.stages);
    cfg.stream = (cudaStream_t)a.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = (p.flags & BF16L_FLAG_PDL) ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return (int)cudaLaunchKernelEx(&cfg, tile_kernel<OutT>, tx, tw, static_cast<const uint16_t *>(a.bias),
                                   static_cast<OutT *>(a.out), a.M, a.N, a.K, p.stages, a.status,
                                   static_cast<const float *>(nullptr), static_cast<const float *>(nullptr));
}

int launch_tile(const LaunchArgs &a, const bf16l_plan &p) {
    return a.out_f32 ? launch_tile_t<float>(a, p) : launch_tile_t<uint16_t>(a, p);
}

int launch_tile_fp8(const void *xq, const void *wq, const float *sx, const float *sw, const void *bias, void *out,
                    int M, int N, int K, int stages, int grid, uint32_t flags, void *stream, int32_t *status) {
    CUtensorMap tx, tw;  // 128-byte rows of 128 codes, as the bf16 form's 64 values
    int r = make_tmap_u8_2d(&tx, xq, (uint64_t)M, (uint64_t)K, kBM, 2 * kChunkK, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    if (r) return (int)cudaErrorInvalidValue;
    r = make_tmap_u8_2d(&tw, wq, (uint64_t)N, (uint64_t)K, kBN, 2 * kChunkK, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    if (r) return (int)cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kTileThreads);
    cfg.dynamicSmemBytes = (size_t)tile_smem_bytes(stages);
    cfg.stream = (cudaStream_t)stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = (flags & BF16L_FLAG_PDL) ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return (int)cudaLaunchKernelEx(&cfg, tile_kernel<uint16_t, true>, tx, tw, static_cast<const uint16_t *>(bias),
                                   static_cast<uint16_t *>(out), M, N, K, stages, status, sx, sw);
}

}  // namespace bf16l
