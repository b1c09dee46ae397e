// tile2.cu — CTA-pair (cta_group::2) tcgen05 tile GEMM for large M.
//
// Prior art: the TGV BF16 GEMM on the sglang PR #30117 page lists 2-CTA
// tactics beside its 1-CTA ones (the "2-CTA" column of its tactic table).
//
// Why a pair on GB300: the 1-CTA tile (tile.cu, 128 x 256 per CTA) has every
// CTA write a whole 48 KB stage into its shared memory and the tensor core
// read all of it back — about 192 bytes of shared-memory traffic per clock at
// the full MMA rate, more than one SM's shared memory delivers.  Here two CTAs
// of a cluster compute one 256 x 256 tile with pair MMAs: each CTA stages only
// its own 128 x rows and its own 128 W rows (32 KB per 64-wide K chunk) and the
// tensor cores of both SMs read each half once.  Per SM that is two thirds of
// the staging traffic for the same flops, and a 32 KB stage leaves room for a
// 6-deep ring.
//
//   * cluster of 2; the even CTA (rank 0) issues all MMAs; both CTAs allocate
//     TMEM together and receive their 128 accumulator rows in their own TMEM;
//   * one producer thread per CTA loads its A half (x rows m0 + 128 * rank) and
//     B half (W rows n0 + 128 * rank); both count their bytes on the leader's
//     `full` barrier, which expects the whole 64 KB of a stage;
//   * the leader's commits arrive on `empty` (stage free) and `acc_full`
//     (accumulator ready) in both CTAs at once (multicast commit);
//   * each CTA's 4 epilogue warps drain their own TMEM rows and arrive on the
//     leader's `acc_empty` (8 arrivals free an accumulator buffer);
//   * fp32 accumulators double-buffered in TMEM (2 x 256 columns);
//   * persistent: each cluster walks 256 x 256 tiles in groups of 8 N-tiles;
//   * a 256 x 192 pair tile (each CTA staging 96 W rows, 28 KB stages) is the
//     other instance: for a bandwidth-bound M = 256 it makes N = 14336 into 75
//     tiles, one per pair of SMs, instead of 56 that leave 40 SMs idle.
// Cross-CTA lifetime: a cluster barrier after set-up (every barrier exists
// before any remote arrival) and one before TMEM is freed and the CTAs exit
// (no remote arrival or copy is left in flight).  Every wait is bounded.
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace bf16l {

namespace {

constexpr int kHalf = 128;                              // rows of A per CTA
constexpr int kPairBM = 2 * kHalf;                      // x rows per pair tile
constexpr int kHalfBytes = kHalf * kChunkK * 2;         // 16 KB: the A half of a stage
// BN: W rows per pair tile (256, or 192 so that N = 14336 makes 75 tiles: one per
// pair of SMs); each CTA stages BN / 2 of them per chunk.
template <int BN>
struct Pair {
    static constexpr int kBHalfBytes = (BN / 2) * kChunkK * 2;        // 16 or 12 KB
    static constexpr int kStageBytes = kHalfBytes + kBHalfBytes;      // 32 or 28 KB per CTA
    static constexpr int kAccCols = BN;                               // fp32 columns of one accumulator
    static constexpr uint32_t kIdesc = idesc_bf16_f32(kPairBM, BN);
};
constexpr int kGroup2N = 8;
constexpr int kEpiWarps = 4;
// TMEM accumulator buffers: 2 lets the epilogue of one tile overlap the MMAs
// of the next (2 x 256 = all 512 columns); 1 uses half the columns.
#ifndef BF16L_TILE2_ACC_BUFS
#define BF16L_TILE2_ACC_BUFS 2
#endif
constexpr int kAccBufs = BF16L_TILE2_ACC_BUFS;
static_assert(kAccBufs == 1 || kAccBufs == 2, "one or two accumulator buffers");
// TMEM columns to allocate: a power of two that holds the accumulator buffers.
__host__ __device__ constexpr uint32_t tmem_cols_for(int cols) { return cols <= 256 ? 256u : 512u; }

struct Tile2Shared {
    uint64_t full[kTile2MaxStages];   // leader only: all 64 KB of a stage (both CTAs) landed
    uint64_t empty[kTile2MaxStages];  // both: the pair MMAs reading the stage are done
    uint64_t acc_full[2];             // both: accumulator buffer holds a finished tile
    uint64_t acc_empty[2];            // leader only: both CTAs' epilogues drained the buffer
    uint32_t tmem_base;
    int32_t bad_pair;  // the pair disagrees on the TMEM address: do nothing
    int32_t aborted;
    int32_t issued;    // chunks this CTA's producer put in flight
    int32_t consumed;  // leader: chunks whose arrival the MMA thread saw
};

__device__ __forceinline__ void tile2_coords(int u, int mp_tiles, int n_tiles, int bn, int &m0, int &n0) {
    const int per_group = kGroup2N * mp_tiles;
    const int g = u / per_group, r = u - g * per_group;
    const int gn = (n_tiles - g * kGroup2N) < kGroup2N ? (n_tiles - g * kGroup2N) : kGroup2N;
    const int mi = r / gn, ni = g * kGroup2N + (r - mi * gn);
    m0 = mi * kPairBM;
    n0 = ni * bn;
}

}  // namespace

template <typename OutT, int BN>
__global__ void __launch_bounds__(kTileThreads, 1)
    tile2_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                 const uint16_t *__restrict__ bias, OutT *__restrict__ out, int M, int N, int K, int stages,
                 int32_t *status) {
    using P = Pair<BN>;
    constexpr int kStage2Bytes = P::kStageBytes, kAcc2Cols = P::kAccCols, kPairBN = BN;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *ring = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    Tile2Shared &sh = *reinterpret_cast<Tile2Shared *>(ring + stages * kStage2Bytes);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int mp_tiles = (M + kPairBM - 1) / kPairBM, n_tiles = (N + kPairBN - 1) / kPairBN;
    const int units = mp_tiles * n_tiles;
    const int cl = (int)blockIdx.x >> 1, ncl = (int)gridDim.x >> 1;
    const int C = (K + kChunkK - 1) / kChunkK;
    constexpr uint32_t kCols = tmem_cols_for(kAccBufs * kAcc2Cols);

    if (tid == 0) {
        tma_prefetch_desc(&tm_x);
        tma_prefetch_desc(&tm_w);
        for (int s = 0; s < stages; ++s) {
            mbar_init(&sh.full[s], 1);   // the leader producer's arrive.expect_tx
            mbar_init(&sh.empty[s], 1);  // the leader's multicast commit
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sh.acc_full[b], 1);
            mbar_init(&sh.acc_empty[b], 2 * kEpiWarps);
        }
        sh.aborted = 0;
        sh.issued = 0;
        sh.consumed = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(&sh.tmem_base, kCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    // Both CTAs' barriers and TMEM exist before any cross-CTA arrival or copy.
    cluster_arrive_release();
    cluster_wait_acquire();
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;
    // The pair MMA writes the same TMEM address in both CTAs: check that the
    // joint allocation gave both the same columns (each CTA reads the other's).
    if (tid == 0) {
        uint32_t other;
        asm volatile("ld.shared::cluster.u32 %0, [%1];"
                     : "=r"(other)
                     : "r"(mapa_shared(smem_u32(&sh.tmem_base), rank ^ 1u))
                     : "memory");
        sh.bad_pair = other != tmem;
        if (other != tmem) record_timeout(status, kSitePairTmem);
    }
    __syncthreads();
    const bool bad_pair = sh.bad_pair != 0;  // the same verdict in both CTAs
    pdl_launch_dependents();

    if (bad_pair) {
        // nothing issued: fall through to the exit barrier
    } else if (warp == 0) {
        if (lane == 0) {  // ---- TMA producer (both CTAs) ----
            pdl_wait();
            const uint32_t full0 = mapa_shared(smem_u32(&sh.full[0]), 0);  // leader's full[0]
            int it = 0;
            for (int u = cl; u < units; u += ncl) {
                int m0, n0;
                tile2_coords(u, mp_tiles, n_tiles, BN, m0, n0);
                const int am = m0 + (int)rank * kHalf, bn = n0 + (int)rank * (BN / 2);
                for (int c = 0; c < C; ++c, ++it) {
                    const int s = it % stages;
                    if (it >= stages && !mbar_wait(&sh.empty[s], ((it / stages) - 1) & 1, status, kSiteEmpty)) {
                        atomicExch(&sh.aborted, 1);
                        goto producer_done;
                    }
                    if (*((volatile int32_t *)&sh.aborted)) goto producer_done;
                    uint8_t *st = ring + s * kStage2Bytes;
                    if (leader) mbar_arrive_expect_tx(&sh.full[s], 2 * kStage2Bytes);
                    const uint32_t fb = full0 + (uint32_t)(s * sizeof(uint64_t));
                    tma_load_2d_pair(st, &tm_x, fb, c * kChunkK, am);
                    tma_load_2d_pair(st + kHalfBytes, &tm_w, fb, c * kChunkK, bn);
                }
            }
        producer_done:
            sh.issued = it;
            // Every commit that arrives on this CTA's `empty` barriers has
            // landed before the exit barrier (the last `stages` chunks).
            if (!*((volatile int32_t *)&sh.aborted)) {
                for (int i = (it > stages ? it - stages : 0); i < it; ++i)
                    if (!mbar_wait(&sh.empty[i % stages], (i / stages) & 1, status, kSiteDrain)) break;
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0 && leader) {  // ---- MMA issuer (leader only) ----
            int it = 0, tile_iter = 0;
            for (int u = cl; u < units; u += ncl, ++tile_iter) {
                sh.consumed = it;
                const int b = tile_iter % kAccBufs;
                const uint32_t acc = tmem + (uint32_t)(b * kAcc2Cols);
                // Both CTAs' epilogues drained this buffer (used kAccBufs tiles ago).
                if (tile_iter >= kAccBufs &&
                    !mbar_wait(&sh.acc_empty[b], ((tile_iter / kAccBufs) - 1) & 1, status, kSiteTmemEmpty)) {
                    atomicExch(&sh.aborted, 1);
                    mbar_arrive(&sh.acc_full[b]);
                    mbar_arrive_cluster(mapa_shared(smem_u32(&sh.acc_full[b]), 1));
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
                    const uint8_t *st = ring + s * kStage2Bytes;
                    const uint64_t adesc = smem_desc_sw128(smem_u32(st));
                    const uint64_t bdesc = smem_desc_sw128(smem_u32(st + kHalfBytes));
#pragma unroll
                    for (int kk = 0; kk < kChunkK / 16; ++kk)
                        mma_bf16_pair(acc, adesc + 2 * kk, bdesc + 2 * kk, P::kIdesc, (c > 0 || kk > 0) ? 1u : 0u);
                    mma_commit_pair(&sh.empty[s], (uint16_t)0x3);
                }
                if (!ok) {  // release both epilogues at once
                    mbar_arrive(&sh.acc_full[b]);
                    mbar_arrive_cluster(mapa_shared(smem_u32(&sh.acc_full[b]), 1));
                    break;
                }
                mma_commit_pair(&sh.acc_full[b], (uint16_t)0x3);
            }
            sh.consumed = it;
        }
        __syncwarp();
    } else {
        // ---- epilogue: warps 2..5 of both CTAs; TMEM lane quarter = warp % 4 ----
        const int q = warp & 3;
        const int row = q * 32 + lane;
        int tile_iter = 0;
        const bool vec_ok = (N % 8) == 0;
        const uint32_t acc_empty0 = mapa_shared(smem_u32(&sh.acc_empty[0]), 0);
        for (int u = cl; u < units; u += ncl, ++tile_iter) {
            int m0, n0;
            tile2_coords(u, mp_tiles, n_tiles, BN, m0, n0);
            const int b = tile_iter % kAccBufs;
            // The tile's bias, one value per lane and 32-column slice, read while the MMAs run.
            pdl_wait();  // bias may be written by the previous kernel
            float lbs[kPairBN / 32];
#pragma unroll
            for (int i = 0; i < kPairBN / 32; ++i) lbs[i] = bias_lane(bias, n0 + 32 * i, N);
            const bool ok = mbar_wait(&sh.acc_full[b], (tile_iter / kAccBufs) & 1, status, kSiteAccum);
            tc_fence_after();
            // warp-uniform, so that the bias shuffles below run on all 32 lanes
            const bool have = __all_sync(0xFFFFFFFFu, ok && !*((volatile int32_t *)&sh.aborted));
            const int m = m0 + (int)rank * kHalf + row;
            const uint32_t acc = tmem + (uint32_t)(b * kAcc2Cols) + ((uint32_t)(q * 32) << 16);
            if (have) {
#pragma unroll
                for (int c = 0; c < kPairBN; c += 32) {
                    const float lb = lbs[c / 32];
                    uint32_t r0[16], r1[16];
                    tmem_ld16(acc + (uint32_t)c, r0);
                    tmem_ld16(acc + (uint32_t)(c + 16), r1);
                    tmem_ld_wait16(r0);
                    tmem_ld_wait16(r1);
                    const int n = n0 + c;
                    float v[32];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        v[j] = __uint_as_float(r0[j]);
                        v[16 + j] = __uint_as_float(r1[j]);
                    }
                    if (bias && n < N) bias_add32(v, lb);  // warp-uniform condition
                    if (m < M && n < N) {
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
            if (lane == 0) {
                if (leader)
                    mbar_arrive(&sh.acc_empty[b]);
                else
                    mbar_arrive_cluster(acc_empty0 + (uint32_t)(b * sizeof(uint64_t)));
            }
            if (!have) break;
        }
    }

    tc_fence_before();
    __syncthreads();
    // Drain TMA copies that were issued but never consumed (only after a timeout).
    if (tid == 0 && leader) {
        for (int i = sh.consumed; i < sh.issued; ++i)
            if (!mbar_wait(&sh.full[i % stages], (i / stages) & 1, status, kSiteDrain)) break;
    }
    // No remote arrival, copy or MMA operand read is left in flight past here.
    cluster_arrive_release();
    cluster_wait_acquire();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, kCols);
    }
}

// At least 116 KB, so that no two CTAs share an SM: each holds all 512 TMEM
// columns, and two pairs waiting on each other's SMs for TMEM must not happen.
int tile2_smem_bytes(int stages, int bn) {
    const int need = 1024 + stages * (bn == 192 ? Pair<192>::kStageBytes : Pair<256>::kStageBytes) + 256;
    return need > 116 * 1024 ? need : 116 * 1024;
}

namespace {

constexpr int kMaxDev2 = 64;
int g_pair_clusters[kMaxDev2];  // co-resident clusters of 2 at the largest ring, per device

template <typename OutT>
int set_tile2_attrs() {
    int e = (int)cudaFuncSetAttribute(tile2_kernel<OutT, 256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      tile2_smem_bytes(kTile2MaxStages, 256));
    if (!e)
        e = (int)cudaFuncSetAttribute(tile2_kernel<OutT, 192>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      tile2_smem_bytes(kTile2MaxStages, 192));
    return e;
}

}  // namespace

int init_tile2() {
    int e = set_tile2_attrs<uint16_t>();
    if (!e) e = set_tile2_attrs<float>();
    if (e) return e;
    int dev = 0;
    e = (int)cudaGetDevice(&dev);
    if (e || dev < 0 || dev >= kMaxDev2) return e ? e : (int)cudaErrorInvalidDevice;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * kGb300Sms);
    cfg.blockDim = dim3(kTileThreads);
    cfg.dynamicSmemBytes = (size_t)tile2_smem_bytes(kTile2MaxStages, 256);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    // A failed query only loses the clamp (launches then use the plan's grid).
    if (cudaOccupancyMaxActiveClusters(&n, tile2_kernel<uint16_t, 256>, &cfg) != cudaSuccess) {
        n = 0;
        (void)cudaGetLastError();
    }
    g_pair_clusters[dev] = n;
    return 0;
}

template <typename OutT, int BN>
static int launch_tile2_t(const LaunchArgs &a, const bf16l_plan &p) {
    CUtensorMap tx, tw;
    int r = make_tmap_bf16_2d(&tx, a.x, (uint64_t)a.M, (uint64_t)a.K, kHalf, kChunkK, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    if (r) return (int)cudaErrorInvalidValue;
    r = make_tmap_bf16_2d(&tw, a.W, (uint64_t)a.N, (uint64_t)a.K, BN / 2, kChunkK, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    if (r) return (int)cudaErrorInvalidValue;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev2) return (int)cudaErrorInvalidDevice;
    // A cluster that cannot be resident with the others would run its tiles
    // after them: never launch more clusters than fit at once.
    int clusters = p.grid / 2;
    if (g_pair_clusters[dev] > 0 && clusters > g_pair_clusters[dev]) clusters = g_pair_clusters[dev];
    if (clusters < 1) return (int)cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * clusters));
    cfg.blockDim = dim3(kTileThreads);
    cfg.dynamicSmemBytes = (size_t)tile2_smem_bytes(p.stages, BN);
    cfg.stream = (cudaStream_t)a.stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = pdl_attr_of((uint32_t)p.flags);
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return (int)cudaLaunchKernelEx(&cfg, tile2_kernel<OutT, BN>, tx, tw, static_cast<const uint16_t *>(a.bias),
                                   static_cast<OutT *>(a.out), a.M, a.N, a.K, p.stages, a.status);
}

int launch_tile2(const LaunchArgs &a, const bf16l_plan &p) {
    if (p.rows_per_cta == 192) return a.out_f32 ? launch_tile2_t<float, 192>(a, p) : launch_tile2_t<uint16_t, 192>(a, p);
    return a.out_f32 ? launch_tile2_t<float, 256>(a, p) : launch_tile2_t<uint16_t, 256>(a, p);
}

}  // namespace bf16l
