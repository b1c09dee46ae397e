// tile.cuh — persistent warp-specialised tcgen05 tile GEMM, templated on the
// tile width, in two orientations.  Instantiated by tile.cu (x rows on the MMA
// M side) and tile_t.cu (the swap-AB form: W rows on the MMA M side).
//
// Prior art: the TGV BF16 GEMM kernel on the sglang PR #30117 page (header
// comment of cutedsl_bf16_gemm.py and its tactic table): 256 threads in 8 warps
// — warp 0 loads A with TMA, warp 1 loads B with TMA (and waits on the
// programmatic grid dependency), warp 2 issues tcgen05.mma into TMEM and owns
// its allocation, warps 4-7 run the epilogue TMEM -> registers -> bf16 ->
// st.global; K tiles of 128; a table of (cta_m, cta_n, stages, 2-CTA) tactics
// with cta_m in {64, 128} and cta_n from 8 to 256.
//
// This kernel keeps the roles and rebuilds the rest for GB300:
//   * tile 128 (MMA M) x BN (MMA N), K in 64-wide chunks (one 128-byte swizzle
//     row) through a ring of `stages` TMA stages of (128 + BN) x 128 bytes; with
//     KC = 2 a stage holds two chunks, brought by one 3-D box per operand (the
//     matrix seen as {64, rows, K / 64}), so half as many loads are issued;
//   * orientation: P is the operand on the MMA M side (128 rows per tile), Q
//     the one on the N side (BN rows per tile).  Plain form (tile.cu): P = x,
//     Q = W, so each tile is 128 tokens x BN weight rows.  Swap-AB form
//     (tile_t.cu, SWAP): P = W, Q = x, so each tile is 128 weight rows x BN
//     tokens, the orientation the TGV table's small cta_n entries serve
//     (few tokens, many weight rows);
//   * one producer thread loads both operands (one expect_tx per stage);
//   * one MMA thread issues 4 x tcgen05.mma (128 x BN x 16) per chunk and
//     frees the stage with tcgen05.commit;
//   * the fp32 accumulator is double-buffered in TMEM (two buffers at a
//     power-of-two column stride), so the epilogue of tile i overlaps the
//     MMAs of tile i+1;
//   * persistent grid (at most one CTA per SM) walking the tiles in raster
//     groups of `group` Q-tiles (Q fastest inside a group, then P), so the
//     CTAs running together share both operands in L2;
//   * epilogue: 4 warps, TMEM lane = P row; the tile's bias read before the
//     accumulator wait (one coalesced load per 32 columns, handed to the lanes
//     by shuffles); 16 or 32 columns at a time -> + bias -> bf16 (RNE) ->
//     stores (16-byte vectors along a row of out in the plain form; in the
//     swap form each column is one token's row of
//     out, and a warp's 32 lanes store 32 consecutive outputs of it).
// Waits are bounded (1 s) and record their site in the status word.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace bf16l {

constexpr int kTileBP = kTileBM;               // 128 P rows per tile (the MMA M)
constexpr int kTileABytes = kTileBP * 128;     // 16 KB: 128 rows of one 128-byte swizzle row

__host__ __device__ constexpr int tile_stage_bytes(int bn) { return kTileABytes + bn * 128; }
// TMEM column stride between the two accumulator buffers, and the allocation.
__host__ __device__ constexpr int tile_acc_stride(int bn) {
    return bn <= 32 ? 32 : bn <= 64 ? 64 : bn <= 128 ? 128 : 256;
}

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

// Tile t -> (P row, Q row) origins: groups of `group` Q-tiles; inside a group
// Q varies fastest, then P.
__device__ __forceinline__ void tile_coords(int t, int p_tiles, int q_tiles, int group, int bq, int &p0, int &q0) {
    const int per_group = group * p_tiles;
    const int g = t / per_group, r = t - g * per_group;
    const int gq = (q_tiles - g * group) < group ? (q_tiles - g * group) : group;
    const int pi = r / gq, qi = g * group + (r - pi * gq);
    p0 = pi * kTileBP;
    q0 = qi * bq;
}

// F8: x and W are e4m3 codes (per-tensor FP8).  A 128-byte swizzle row then
// holds 128 codes instead of 64 bf16 values, each MMA (kind::f8f6f4) takes 32
// of them, and the epilogue scales the fp32 sum by *scale_x * *scale_w before
// bias; the shared-memory geometry of a stage is the same.  K counts elements.
template <int BN, bool SWAP, typename OutT, bool F8 = false, int KC = 1>
__global__ void __launch_bounds__(kTileThreads, 1)
    tile_kernel(const __grid_constant__ CUtensorMap tm_p, const __grid_constant__ CUtensorMap tm_q,
                const uint16_t *__restrict__ bias, OutT *__restrict__ out, int M, int N, int K, int stages,
                int group, int32_t *status, const float *__restrict__ scale_x,
                const float *__restrict__ scale_w) {
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N: a multiple of 16 up to 256");
    static_assert(!(SWAP && F8), "the e4m3 form is plain only");
    static_assert(KC == 1 || (KC == 2 && !F8), "two-chunk stages: bf16 only");
    constexpr int kc = KC;  // K chunks per ring stage (a template parameter: the issue loops stay minimal)
    constexpr int kChunk = F8 ? 2 * kChunkK : kChunkK;  // elements per 128-byte row
    constexpr int kQBytes = BN * 128;  // one chunk of the N-side operand
    constexpr int kAccStride = tile_acc_stride(BN);
    constexpr int kTmemCols = 2 * kAccStride;
    constexpr uint32_t kIdesc = F8 ? idesc_e4m3_f32(kTileBP, BN) : idesc_bf16_f32(kTileBP, BN);
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *ring = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    // A stage holds kc consecutive K chunks: kc P chunk tiles, then kc Q chunk tiles.
    constexpr int stage_bytes = kc * tile_stage_bytes(BN);
    TileShared &sh = *reinterpret_cast<TileShared *>(ring + stages * stage_bytes);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int p_rows = SWAP ? N : M, q_rows = SWAP ? M : N;
    const int p_tiles = (p_rows + kTileBP - 1) / kTileBP, q_tiles = (q_rows + BN - 1) / BN;
    const int num_tiles = p_tiles * q_tiles;
    const int C = (K + kChunk * kc - 1) / (kChunk * kc);  // ring stages per tile (the last one zero-filled past K)
    const int G = group > 0 ? group : q_tiles;

    if (tid == 0) {
        tma_prefetch_desc(&tm_p);
        tma_prefetch_desc(&tm_q);
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
                int p0, q0;
                tile_coords(t, p_tiles, q_tiles, G, BN, p0, q0);
                for (int c = 0; c < C; ++c, ++it) {
                    const int s = it % stages;
                    if (it >= stages && !mbar_wait(&sh.empty[s], ((it / stages) - 1) & 1, status, kSiteEmpty)) {
                        atomicExch(&sh.aborted, 1);
                        goto producer_done;
                    }
                    if (*((volatile int32_t *)&sh.aborted)) goto producer_done;
                    uint8_t *st = ring + s * stage_bytes;
                    mbar_arrive_expect_tx(&sh.full[s], (uint32_t)stage_bytes);
                    if constexpr (kc == 1) {
                        tma_load_2d(st, &tm_p, &sh.full[s], c * kChunk, p0);
                        tma_load_2d(st + kTileABytes, &tm_q, &sh.full[s], c * kChunk, q0);
                    } else {  // chunked maps: {64, rows, chunks}
                        tma_load_3d(st, &tm_p, &sh.full[s], 0, p0, c * kc);
                        tma_load_3d(st + kc * kTileABytes, &tm_q, &sh.full[s], 0, q0, c * kc);
                    }
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
                const uint32_t acc = tmem + (uint32_t)(b * kAccStride);
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
                    const uint8_t *st = ring + s * stage_bytes;
#pragma unroll
                    for (int j = 0; j < kc; ++j) {
                        const uint64_t adesc = smem_desc_sw128(smem_u32(st + j * kTileABytes));
                        const uint64_t bdesc = smem_desc_sw128(smem_u32(st + kc * kTileABytes + j * kQBytes));
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {  // 32 bytes of each row per MMA
                            const uint32_t accum = (c > 0 || j > 0 || kk > 0) ? 1u : 0u;
                            if constexpr (F8)
                                mma_e4m3(acc, adesc + 2 * kk, bdesc + 2 * kk, kIdesc, accum);
                            else
                                mma_bf16(acc, adesc + 2 * kk, bdesc + 2 * kk, kIdesc, accum);
                        }
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
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        int tile_iter = 0;
        const bool vec_ok = (N % 8) == 0;
        for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++tile_iter) {
            int p0, q0;
            tile_coords(t, p_tiles, q_tiles, G, BN, p0, q0);
            const int b = tile_iter & 1;
            const int p = p0 + row;  // x row (plain) or W row (swap) of this thread
            // The tile's bias, read while the MMAs run: plain form one value per lane and 32-column slice
            // (bias_lane), swap form this thread's W row.
            pdl_wait();  // bias may be written by the previous kernel
            constexpr int kSlices = (BN + 31) / 32;
            float lbs[kSlices];
#pragma unroll
            for (int i = 0; i < kSlices; ++i) lbs[i] = SWAP ? 0.0f : bias_lane(bias, q0 + 32 * i, N);
            const float bias_row = (SWAP && bias && p < N) ? bf16_to_f32(bias[p]) : 0.0f;
            const bool ok = mbar_wait(&sh.acc_full[b], (tile_iter / 2) & 1, status, kSiteAccum);
            tc_fence_after();
            // warp-uniform, so that the bias shuffles below run on all 32 lanes
            const bool have = __all_sync(0xFFFFFFFFu, ok && !*((volatile int32_t *)&sh.aborted));
            const uint32_t acc = tmem + (uint32_t)(b * kAccStride) + ((uint32_t)(quarter * 32) << 16);
            if (have) {
                const float sxw = F8 ? __ldg(scale_x) * __ldg(scale_w) : 1.0f;
                // cnt (16 or 32) accumulator columns starting at column c, this thread's row;
                // lb: the plain form's bias for columns q0 + c + lane (bias_lane)
                auto emit = [&](int c, const float *vin, int cnt, float lb) {
                    float v[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = j < cnt ? vin[j] * sxw : 0.0f;
                    if constexpr (SWAP) {
                        if (p < N) {
#pragma unroll
                            for (int j = 0; j < 32; ++j) {
                                const int m = q0 + c + j;
                                if (j < cnt && m < M) OutStore<OutT>::one(out + (size_t)m * N + p, v[j] + bias_row);
                            }
                        }
                    } else {
                        const int n = q0 + c;
                        if (bias && n < N) bias_add32(v, lb);  // warp-uniform condition
                        if (p < M && n < N) {
                            OutT *o = out + (size_t)p * N + n;
                            if (vec_ok && n + cnt <= N) {
#pragma unroll
                                for (int j = 0; j < 32; j += 8)
                                    if (j < cnt) OutStore<OutT>::eight(o + j, v + j);
                            } else {
#pragma unroll
                                for (int j = 0; j < 32; ++j)
                                    if (j < cnt && n + j < N) OutStore<OutT>::one(o + j, v[j]);
                            }
                        }
                    }
                };
#pragma unroll
                for (int c = 0; c + 32 <= BN; c += 32) {
                    const float lb = lbs[c / 32];
                    uint32_t r0[16], r1[16];
                    tmem_ld16(acc + (uint32_t)c, r0);
                    tmem_ld16(acc + (uint32_t)(c + 16), r1);
                    tmem_ld_wait16(r0);
                    tmem_ld_wait16(r1);
                    float v[32];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        v[j] = __uint_as_float(r0[j]);
                        v[16 + j] = __uint_as_float(r1[j]);
                    }
                    emit(c, v, 32, lb);
                }
                if constexpr (BN % 32 != 0) {  // the last 16 columns
                    const float lb = lbs[kSlices - 1];  // columns BN - 16 .. BN - 1: lanes 0..15
                    uint32_t r0[16];
                    tmem_ld16(acc + (uint32_t)(BN - 16), r0);
                    tmem_ld_wait16(r0);
                    float v[32];
#pragma unroll
                    for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r0[j]);
                    emit(BN - 16, v, 16, lb);
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

// Dynamic shared memory of a launch: 1 KB alignment slack, the ring, the
// barriers; at least 116 KB, so that no two CTAs share an SM (a second one
// would find the TMEM columns taken and wait in tcgen05.alloc until the first
// CTA is done with all of its tiles).
inline int tile_smem_bytes_bn(int stages, int bn, int kc = 1) {
    const int need = 1024 + stages * kc * tile_stage_bytes(bn) + 256;
    return need > 116 * 1024 ? need : 116 * 1024;
}

template <int BN, bool SWAP, typename OutT>
int tile_set_attr() {
    const int bytes = tile_smem_bytes_bn(tile_max_stages(BN), BN);  // covers every valid (stages, chunks)
    int e = (int)cudaFuncSetAttribute(tile_kernel<BN, SWAP, OutT, false, 1>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (!e)
        e = (int)cudaFuncSetAttribute(tile_kernel<BN, SWAP, OutT, false, 2>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    return e;
}

// One launch of the bf16 form: P rows of 128 from tm_p, Q rows of BN from tm_q, KC chunks per stage.
template <int BN, bool SWAP, typename OutT, int KC>
int tile_launch_kc(const LaunchArgs &a, const bf16l_plan &p) {
    CUtensorMap tp, tq;
    const void *pb = SWAP ? a.W : a.x, *qb = SWAP ? a.x : a.W;
    const uint64_t pr = SWAP ? (uint64_t)a.N : (uint64_t)a.M, qr = SWAP ? (uint64_t)a.M : (uint64_t)a.N;
    int r;
    if (KC == 1) {
        r = make_tmap_bf16_2d(&tp, pb, pr, (uint64_t)a.K, kTileBP, kChunkK, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
        if (!r)
            r = make_tmap_bf16_2d(&tq, qb, qr, (uint64_t)a.K, BN, kChunkK, CU_TENSOR_MAP_SWIZZLE_128B,
                                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    } else {  // the chunked view: one box brings KC chunks (the plan check asked for K % 64 == 0)
        r = make_tmap_bf16_chunks(&tp, pb, pr, (uint64_t)a.K, kTileBP, (uint32_t)KC);
        if (!r) r = make_tmap_bf16_chunks(&tq, qb, qr, (uint64_t)a.K, BN, (uint32_t)KC);
    }
    if (r) return (int)cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.grid);
    cfg.blockDim = dim3(kTileThreads);
    cfg.dynamicSmemBytes = (size_t)tile_smem_bytes_bn(p.stages, BN, KC);
    cfg.stream = (cudaStream_t)a.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl_attr_of((uint32_t)p.flags);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return (int)cudaLaunchKernelEx(&cfg, tile_kernel<BN, SWAP, OutT, false, KC>, tp, tq,
                                   static_cast<const uint16_t *>(a.bias), static_cast<OutT *>(a.out), a.M, a.N, a.K,
                                   p.stages, p.split_k > 0 ? p.split_k : (SWAP ? 0 : kTileDefaultGroup), a.status,
                                   static_cast<const float *>(nullptr), static_cast<const float *>(nullptr));
}

template <int BN, bool SWAP, typename OutT>
int tile_launch_bn(const LaunchArgs &a, const bf16l_plan &p) {
    return p.chunks_per_stage == 2 ? tile_launch_kc<BN, SWAP, OutT, 2>(a, p) : tile_launch_kc<BN, SWAP, OutT, 1>(a, p);
}

}  // namespace bf16l
