// splitk.cu — cluster split-K kernel on the 5th-generation tensor cores.
//
// Prior art: the LLBf16SplitK kernel on the vLLM PR #42562 page ("实现拆解"
// item 2 and its source excerpt): K split over the CTAs of one thread-block
// cluster (8 by default), a warp-specialised DMA/MMA pipeline, fp32 partial
// tiles reduced across the cluster through distributed shared memory
// (st.shared::cluster), non-.aligned cluster barriers (its review found the
// .aligned forms hung), tile_m = 16 tokens, tile_n = 16 weight rows.
//
// Rebuilt for sm_103a around what limits a skinny GEMM on GB300: one CTA's TMA
// intake is only some tens of GB/s, so the weights must be spread over 100+
// CTAs, each streaming a few tens of KB, and the prologue / epilogue chain
// must be short.
//   * MMA shape: tokens on the MMA M side (M = 64; only the first TOKP rows of
//     the A tile hold x, the rest is whatever follows in shared memory and only
//     feeds accumulator rows that are never read), BN = 16..256 weight rows on
//     the N side.  So a CTA's weight tile can be as small as 16 rows and the
//     grid can have hundreds of CTAs even for N = 128..384.  With M = 64 the
//     accumulator row of token t sits in TMEM lane 32*(t/16) + t%16.
//   * One thread issues TMA tile loads (128-byte swizzle; rows past N, tokens
//     past M and K past the end are zero-filled) into a `stages`-deep ring of
//     64-wide K chunks: the weight halves first, before anything else, then
//     (after the programmatic-launch wait, when enabled) the x halves.
//   * One thread issues tcgen05.mma (128 x BN x 16, fp32 accumulate in TMEM)
//     and frees each stage with tcgen05.commit.
//   * Exchange, push-based: the tile's M x BN partial sums are cut into
//     float4 items (token-major); rank d of the cluster owns a contiguous 1/S
//     of them.  Each token's thread reads its row of the accumulator from
//     TMEM and st.async-s every item straight into its owner's receive buffer,
//     whose mbarrier counts the bytes.  The owner sums the S partials in rank
//     order (deterministic), adds the bias, rounds to bf16 and stores 4
//     outputs at a time.
//   * Programmatic dependent launch (optional): weights are read before
//     griddepcontrol.wait, x and the output only after it, and every CTA lets
//     the next kernel start as soon as its own weight loads are issued.
//
//   * Two-chunk stages (kc = 2, K % 64 == 0): one 3-D box per operand brings two
//     consecutive K chunks (the matrix seen as {64, rows, K / 64}); the ranks then
//     split K in units of two chunks.
//
// Grid: (S, ceil(N/BN)) with cluster dims (S, 1, 1); rank r takes ring stages
// [r*C/S, (r+1)*C/S) of the C = ceil(K / (64 kc)) stages.
#include "common.cuh"
#include "kernels.h"

namespace bf16l {

namespace {

constexpr int kSmemPerSm = 233472;  // 228 KB of shared memory per SM on sm_103
constexpr int kSmemPerCta = 232448; // 227 KB usable by one CTA
constexpr int kMmaM = 64;           // MMA rows (tokens, zero- or garbage-padded)
constexpr int kATileBytes = kMmaM * kChunkK * 2;  // the 8 KB the MMA reads as A per chunk

struct SplitShared {  // bookkeeping placed after the receive buffer (<= 512 bytes)
    uint64_t full[kSplitMaxStages];
    uint64_t empty[kSplitMaxStages];
    uint64_t accum;
    uint64_t recv;
    uint32_t tmem_base;
    int32_t aborted;   // set when a wait gave up: skip the rest of the math
    int32_t issued;    // TMA chunks issued by the producer
    int32_t consumed;  // chunks whose data the MMA issuer saw arrive
    int32_t last;      // (workspace mode) this CTA arrived last for its tile
};

__device__ __forceinline__ int part_begin(int d, int T, int S) { return mul_div(T, d, S); }

}  // namespace

static_assert(sizeof(SplitShared) <= 512, "bookkeeping must fit its reserved space");

// Host-visible layout arithmetic (shared with the planner through kernels.h).
int split_stage_bytes(int tokens, int rows, int kc) { return kc * (tokens + rows) * kChunkK * 2; }

int split_recv_bytes(int tokens, int rows) {
    // S partials of this CTA's share: at most S * ceil(T / S) <= T + S items of 16 bytes.
    return (tokens * rows / 4 + kSplitMaxCluster) * 16;
}

// Independent accumulators per CTA: consecutive MMAs of a chunk rotate over
// them, so a short MMA does not wait for the previous one to finish adding
// into the same TMEM tile.  Summed in fixed order in the epilogue.
__host__ __device__ constexpr int split_acc_count(int rows) { return rows <= 64 ? 4 : rows <= 128 ? 2 : 1; }

int split_tmem_cols(int rows) {
    const int need = split_acc_count(rows) * rows;
    return need <= 32 ? 32 : need <= 64 ? 64 : need <= 128 ? 128 : 256;
}

int split_ring_bytes(int tokens, int rows, int stages, int kc) {
    // The ring, which the accumulator staging (tokens x rows fp32) reuses once the MMAs are done.
    const int ring = stages * split_stage_bytes(tokens, rows, kc), acc = tokens * rows * 4;
    return ring > acc ? ring : acc;
}

int split_smem_bytes(int tokens, int rows, int stages, int kc) {
    const int stage = split_stage_bytes(tokens, rows, kc);
    int body = split_ring_bytes(tokens, rows, stages, kc) + split_recv_bytes(tokens, rows) + 512 /*bookkeeping*/;
    // The MMA reads a full 64-row A window from the last stage's last x chunk on.
    const int window = (stages - 1) * stage + (kc - 1) * tokens * kChunkK * 2 + kATileBytes;
    if (window > body) body = window;
    int bytes = 1024 /*alignment slack*/ + body;
    // Pad so that the CTAs that fit on one SM never ask for more than its 512
    // TMEM columns between them (an allocation that cannot be met would stall).
    const int cols = split_tmem_cols(rows);
    const int min_bytes = kSmemPerSm / (512 / cols + 1) + 1;
    return bytes > min_bytes ? bytes : min_bytes;
}

int split_max_stages(int tokens, int rows, int kc) {
    int s = kSplitMaxStages;
    while (s > 1 && split_smem_bytes(tokens, rows, s, kc) > kSmemPerCta) --s;
    return split_smem_bytes(tokens, rows, s, kc) <= kSmemPerCta ? s : 0;
}

// kClus: the S CTAs that share a tile form a thread-block cluster and reduce
// through distributed shared memory.  !kClus: no cluster; every CTA writes its
// fp32 partial tile to the workspace `ws` and bumps the tile's counter; the
// last CTA to arrive sums the S partials in rank order and resets the counter.
template <int BN, typename OutT, bool kClus>
__global__ void __launch_bounds__(kSplitThreads, 1)
    splitk_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                  const uint16_t *__restrict__ bias, OutT *__restrict__ out, int M, int N, int K, int tokp,
                  int stages, int32_t *status, float *__restrict__ ws, uint32_t *__restrict__ counters,
                  int w_early, int kc) {
    constexpr uint32_t kIdesc = idesc_bf16_f32(kMmaM, BN);
    constexpr int kAcc = split_acc_count(BN);
    constexpr int kCols = kAcc * BN <= 32 ? 32 : kAcc * BN <= 64 ? 64 : kAcc * BN <= 128 ? 128 : 256;
    constexpr int kWBytes = BN * kChunkK * 2;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *ring = smem_raw + (((raw + 1023u) & ~1023u) - raw);  // 1024-aligned (128-byte swizzle atoms)
    const int xbytes = tokp * kChunkK * 2;
    const int stage_bytes = kc * (xbytes + kWBytes);  // kc x chunk tiles, then kc weight chunk tiles
    const int T = M * (BN / 4);  // float4 items of the tile's partial sums
    const int ring_bytes = stages * stage_bytes > tokp * BN * 4 ? stages * stage_bytes : tokp * BN * 4;
    float4 *stage_out = reinterpret_cast<float4 *>(ring);  // accumulator staging, [M][BN] fp32, after the MMAs
    float4 *recv = reinterpret_cast<float4 *>(ring + ring_bytes);
    const int recv_bytes = (tokp * BN / 4 + kSplitMaxCluster) * 16;  // as split_recv_bytes()
    SplitShared &sh = *reinterpret_cast<SplitShared *>(ring + ring_bytes + recv_bytes);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rank = kClus ? (int)cluster_ctarank() : (int)blockIdx.x;
    const int S = (int)gridDim.x;  // the K split spans the whole x dimension of the grid
    const int n0 = blockIdx.y * BN;
    // K moves in ring stages of kc 64-wide chunks (the last one zero-filled past K); the ranks split the stages.
    const int C = (K + kChunkK * kc - 1) / (kChunkK * kc);
    const int c_begin = mul_div(C, rank, S);
    const int nchunks = mul_div(C, rank + 1, S) - c_begin;
    const int first = nchunks < stages ? nchunks : stages;  // stages whose weights go out at once
    // Default launch: nothing is read before the previous kernel has finished.  (An L2 prefetch of the
    // first ring's weight boxes here, as the CUDA-core kernels issue, measured 2-4% slower on the decode
    // and MLP shapes this kernel serves.)
    if (!w_early) pdl_wait();

    if (tid == 0) {
        tma_prefetch_desc(&tm_w);
        tma_prefetch_desc(&tm_x);
        for (int s = 0; s < stages; ++s) {
            mbar_init(&sh.full[s], 1);
            mbar_init(&sh.empty[s], 1);
        }
        mbar_init(&sh.accum, 1);
        mbar_init(&sh.recv, 1);
        sh.aborted = 0;
        sh.issued = 0;
        sh.consumed = 0;
        fence_barrier_init();
        // Weights do not depend on the previous kernel: put them in flight first.
        for (int i = 0; i < first; ++i) {
            uint8_t *st = ring + i * stage_bytes;
            mbar_arrive_expect_tx(&sh.full[i], (uint32_t)stage_bytes);
            if (kc == 1)
                tma_load_2d(st + xbytes, &tm_w, &sh.full[i], (c_begin + i) * kChunkK, n0);
            else
                tma_load_3d(st + kc * xbytes, &tm_w, &sh.full[i], 0, n0, (c_begin + i) * kc);
        }
        pdl_launch_dependents();  // the next kernel may start its own weight loads now
        pdl_wait();               // x may be written by the previous kernel
        for (int i = 0; i < first; ++i) {
            if (kc == 1)
                tma_load_2d(ring + i * stage_bytes, &tm_x, &sh.full[i], (c_begin + i) * kChunkK, 0);
            else
                tma_load_3d(ring + i * stage_bytes, &tm_x, &sh.full[i], 0, 0, (c_begin + i) * kc);
        }
    }
    if (warp == 1) {
        tmem_alloc(&sh.tmem_base, kCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_launch_dependents();
    if constexpr (kClus) cluster_arrive_relaxed();  // phase 1: "my receive barrier is initialised"
    const uint32_t tmem = sh.tmem_base;

    if (warp == 0) {
        if (lane == 0) {  // ---- TMA producer: ring refills beyond the first `stages` chunks ----
            int i = first;
            for (; i < nchunks; ++i) {
                const int s = i % stages;
                if (!mbar_wait(&sh.empty[s], ((i / stages) - 1) & 1, status, kSiteEmpty)) {
                    atomicExch(&sh.aborted, 1);
                    break;
                }
                uint8_t *st = ring + s * stage_bytes;
                mbar_arrive_expect_tx(&sh.full[s], (uint32_t)stage_bytes);
                if (kc == 1) {
                    const int k0 = (c_begin + i) * kChunkK;
                    tma_load_2d(st + xbytes, &tm_w, &sh.full[s], k0, n0);
                    tma_load_2d(st, &tm_x, &sh.full[s], k0, 0);
                } else {
                    tma_load_3d(st + kc * xbytes, &tm_w, &sh.full[s], 0, n0, (c_begin + i) * kc);
                    tma_load_3d(st, &tm_x, &sh.full[s], 0, 0, (c_begin + i) * kc);
                }
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
                const uint8_t *st = ring + s * stage_bytes;
#pragma unroll 1
                for (int j = 0; j < kc; ++j) {
                    const uint64_t adesc = smem_desc_sw128(smem_u32(st + j * xbytes));
                    const uint64_t bdesc = smem_desc_sw128(smem_u32(st + kc * xbytes + j * kWBytes));
#pragma unroll
                    for (int kk = 0; kk < kChunkK / 16; ++kk) {  // 4 MMAs of K = 16 (32 bytes) each
                        const int q = j * (kChunkK / 16) + kk;  // MMA index in the stage: accumulator q % kAcc
                        mma_bf16(tmem + (uint32_t)((q % kAcc) * BN), adesc + 2 * kk, bdesc + 2 * kk, kIdesc,
                                 (i > 0 || q >= kAcc) ? 1u : 0u);
                    }
                }
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

    if constexpr (!kClus) {
        // ---- epilogue without a cluster: partial tile -> workspace; the last CTA reduces ----
        const bool ok = mbar_wait(&sh.accum, 0, status, kSiteAccum);
        tc_fence_after();
        const bool have = ok && !*((volatile int32_t *)&sh.aborted);
        pdl_wait();  // the workspace and `out` may still be in use by the previous kernel
        float4 *part = reinterpret_cast<float4 *>(ws) + (size_t)(blockIdx.y * S + rank) * T;
        if (warp * 16 < M) {  // warp w holds tokens 16w..16w+15 in its lanes 0..15
            const int t = warp * 16 + lane;
#pragma unroll 1
            for (int c = 0; c < BN; c += 16) {
                uint32_t r[16];
                if (have) {
                    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c;
                    tmem_ld16(lane_base, r);
                    tmem_ld_wait16(r);
#pragma unroll
                    for (int a = 1; a < kAcc; ++a) {
                        uint32_t r2[16];
                        tmem_ld16(lane_base + (uint32_t)(a * BN), r2);
                        tmem_ld_wait16(r2);
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            r[j] = __float_as_uint(__uint_as_float(r[j]) + __uint_as_float(r2[j]));
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) r[j] = 0u;
                }
                if (lane < 16 && t < M) {
                    float4 *dst = part + (t * BN + c) / 4;
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4)
                        __stcg(dst + q4, make_float4(__uint_as_float(r[4 * q4]), __uint_as_float(r[4 * q4 + 1]),
                                                     __uint_as_float(r[4 * q4 + 2]), __uint_as_float(r[4 * q4 + 3])));
                }
            }
            __threadfence();  // this CTA's partial is visible GPU-wide before the counter moves
        }
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            const uint32_t prev = atomicAdd(&counters[blockIdx.y], 1u);
            *reinterpret_cast<volatile int32_t *>(&sh.last) = (prev == (uint32_t)(S - 1)) ? 1 : 0;
            __threadfence();
        }
        __syncthreads();
        if (*reinterpret_cast<volatile int32_t *>(&sh.last)) {
            const float4 *pt = reinterpret_cast<const float4 *>(ws) + (size_t)blockIdx.y * S * T;
            for (int j = tid; j < T; j += kSplitThreads) {
                float4 acc = __ldcg(pt + j);
                for (int q = 1; q < S; ++q) {  // rank order: deterministic
                    const float4 v = __ldcg(pt + (size_t)q * T + j);
                    acc.x += v.x;
                    acc.y += v.y;
                    acc.z += v.z;
                    acc.w += v.w;
                }
                const int m = j / (BN / 4);
                const int n = n0 + 4 * (j % (BN / 4));
                float r4[4] = {acc.x, acc.y, acc.z, acc.w};
                if (bias) {
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (n + e < N) r4[e] += bf16_to_f32(bias[n + e]);
                }
                const size_t o = (size_t)m * N + n;
                if (n + 3 < N && (o & 3) == 0) {
                    OutStore<OutT>::four(out + o, r4[0], r4[1], r4[2], r4[3]);
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (n + e < N) OutStore<OutT>::one(out + o + e, r4[e]);
                }
            }
            if (tid == 0) counters[blockIdx.y] = 0u;  // ready for the next call
        }
    } else {
    // ---- epilogue: accumulator -> local staging [M][BN] -> one bulk copy per owner ----
    cluster_wait_acquire();  // phase 1 done (long since): every CTA's receive barrier exists
    const bool ok = mbar_wait(&sh.accum, 0, status, kSiteAccum);
    tc_fence_after();
    const bool have = ok && !*((volatile int32_t *)&sh.aborted);
    if (warp * 16 < M) {  // warp w holds tokens 16w..16w+15 in its lanes 0..15
        const int t = warp * 16 + lane;
#pragma unroll 1
        for (int c = 0; c < BN; c += 16) {
            uint32_t r[16];
            if (have) {
                const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c;
                tmem_ld16(lane_base, r);
                tmem_ld_wait16(r);
#pragma unroll
                for (int a = 1; a < kAcc; ++a) {  // fixed order: accumulator 0, 1, ...
                    uint32_t r2[16];
                    tmem_ld16(lane_base + (uint32_t)(a * BN), r2);
                    tmem_ld_wait16(r2);
#pragma unroll
                    for (int j = 0; j < 16; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) + __uint_as_float(r2[j]));
                }
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j) r[j] = 0u;
            }
            if (lane < 16 && t < M) {
                float4 *dst = stage_out + (t * BN + c) / 4;
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4)
                    dst[q4] = make_float4(__uint_as_float(r[4 * q4]), __uint_as_float(r[4 * q4 + 1]),
                                          __uint_as_float(r[4 * q4 + 2]), __uint_as_float(r[4 * q4 + 3]));
            }
        }
        fence_proxy_async_smem();  // the bulk copies below read the staging through the async proxy
    }
    tc_fence_before();
    __syncthreads();
    if (tid < S) {  // thread d sends owner d its slice [it0(d), it1(d)) of the items
        const int d = tid;
        const int d0 = part_begin(d, T, S);
        const int nd = part_begin(d + 1, T, S) - d0;
        if (nd > 0)
            bulk_copy_to_peer(mapa_shared(smem_u32(recv + rank * nd), (uint32_t)d), stage_out + d0,
                              (uint32_t)(nd * 16), mapa_shared(smem_u32(&sh.recv), (uint32_t)d));
    }

    // ---- owner: S partials of my items -> bias -> bf16 -> out ----
    const int it0 = part_begin(rank, T, S);
    const int mine = part_begin(rank + 1, T, S) - it0;
    if (tid == 0) mbar_arrive_expect_tx(&sh.recv, (uint32_t)(S * mine * 16));
    const bool got = mbar_wait_cluster(&sh.recv, 0, status, kSiteRecv);
    // Every copy into this CTA has landed, so every peer's copy out of its own
    // staging has been read: phase 2 lets all of them exit.
    cluster_arrive_relaxed();
    pdl_wait();  // the previous kernel may still read `out`
    if (got && !*((volatile int32_t *)&sh.aborted)) {
        for (int j = tid; j < mine; j += kSplitThreads) {
            float4 acc = recv[j];
            for (int q = 1; q < S; ++q) {
                const float4 v = recv[q * mine + j];
                acc.x += v.x;
                acc.y += v.y;
                acc.z += v.z;
                acc.w += v.w;
            }
            const int item = it0 + j;
            const int m = item / (BN / 4);
            const int n = n0 + 4 * (item % (BN / 4));
            float r4[4] = {acc.x, acc.y, acc.z, acc.w};
            if (bias) {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (n + e < N) r4[e] += bf16_to_f32(bias[n + e]);
            }
            const size_t o = (size_t)m * N + n;
            if (n + 3 < N && (o & 3) == 0) {
                OutStore<OutT>::four(out + o, r4[0], r4[1], r4[2], r4[3]);
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (n + e < N) OutStore<OutT>::one(out + o + e, r4[e]);
            }
        }
    }

    }  // kClus

    // Drain TMA copies that were issued but never consumed (only after a timeout).
    if (tid == 0) {
        for (int i = sh.consumed; i < sh.issued; ++i)
            mbar_wait(&sh.full[i % stages], (i / stages) & 1, status, kSiteDrain);
    }
    if constexpr (kClus) cluster_wait_acquire();  // phase 2 done: no copy into or out of this CTA is pending
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kCols);
    }
}

namespace {

template <typename OutT, bool kClus>
using SplitFn = void (*)(CUtensorMap, CUtensorMap, const uint16_t *, OutT *, int, int, int, int, int, int32_t *,
                         float *, uint32_t *, int, int);

template <typename OutT, bool kClus>
SplitFn<OutT, kClus> pick(int BN) {
    switch (BN) {
        case 16: return splitk_kernel<16, OutT, kClus>;
        case 32: return splitk_kernel<32, OutT, kClus>;
        case 48: return splitk_kernel<48, OutT, kClus>;
        case 64: return splitk_kernel<64, OutT, kClus>;
        case 96: return splitk_kernel<96, OutT, kClus>;
        case 128: return splitk_kernel<128, OutT, kClus>;
        case 192: return splitk_kernel<192, OutT, kClus>;
        case 256: return splitk_kernel<256, OutT, kClus>;
        default: return nullptr;
    }
}

template <typename OutT, bool kClus>
int set_split_attrs() {
    for (int BN : {16, 32, 48, 64, 96, 128, 192, 256}) {
        auto fn = pick<OutT, kClus>(BN);
        int e = (int)cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemPerCta);
        if (!e && kClus) e = (int)cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e) return e;
    }
    return 0;
}

template <typename OutT, bool kClus>
int launch_split_t(const LaunchArgs &a, const bf16l_plan &p) {
    SplitFn<OutT, kClus> fn = pick<OutT, kClus>(p.rows_per_cta);
    if (!fn) return (int)cudaErrorInvalidValue;
    CUtensorMap tw, tx;
    const int kc = p.chunks_per_stage == 2 ? 2 : 1;  // validated by the plan check (K % 64 == 0)
    int r;
    if (kc == 1) {
        r = make_tmap_bf16_2d(&tw, a.W, (uint64_t)a.N, (uint64_t)a.K, (uint32_t)p.rows_per_cta, kChunkK,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
        if (!r)
            r = make_tmap_bf16_2d(&tx, a.x, (uint64_t)a.M, (uint64_t)a.K, (uint32_t)p.tokens_per_cta, kChunkK,
                                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    } else {
        r = make_tmap_bf16_chunks(&tw, a.W, (uint64_t)a.N, (uint64_t)a.K, (uint32_t)p.rows_per_cta, (uint32_t)kc);
        if (!r)
            r = make_tmap_bf16_chunks(&tx, a.x, (uint64_t)a.M, (uint64_t)a.K, (uint32_t)p.tokens_per_cta,
                                      (uint32_t)kc);
    }
    if (r) return (int)cudaErrorInvalidValue;

    const int tiles = (a.N + p.rows_per_cta - 1) / p.rows_per_cta;
    uint32_t *counters = nullptr;
    float *parts = nullptr;
    if (!kClus) {
        if (!a.workspace || a.workspace_bytes < split_ws_bytes(a.M, a.N, p)) return (int)cudaErrorInvalidValue;
        counters = static_cast<uint32_t *>(a.workspace);
        parts = reinterpret_cast<float *>(static_cast<uint8_t *>(a.workspace) + split_ws_counter_bytes(tiles));
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.split_k, (unsigned)tiles, 1);
    cfg.blockDim = dim3(kSplitThreads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)split_smem_bytes(p.tokens_per_cta, p.rows_per_cta, p.stages, kc);
    cfg.stream = (cudaStream_t)a.stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = pdl_attr_of((uint32_t)p.flags);
    ++na;
    if (kClus) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = (unsigned)p.split_k;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return (int)cudaLaunchKernelEx(&cfg, fn, tw, tx, static_cast<const uint16_t *>(a.bias),
                                   static_cast<OutT *>(a.out), a.M, a.N, a.K, p.tokens_per_cta, p.stages,
                                   a.status, parts, counters, w_early_of((uint32_t)p.flags), kc);
}

}  // namespace

size_t split_ws_counter_bytes(int tiles) { return ((size_t)tiles * 4 + 255) / 256 * 256; }

size_t split_ws_bytes(int M, int N, const bf16l_plan &p) {
    if (p.kernel != BF16L_KERNEL_SPLITK_WS || p.rows_per_cta <= 0) return 0;
    const int tiles = (N + p.rows_per_cta - 1) / p.rows_per_cta;
    return split_ws_counter_bytes(tiles) + (size_t)tiles * p.split_k * M * p.rows_per_cta * 4;
}

bool split_rows_supported(int rows) { return pick<uint16_t, true>(rows) != nullptr; }

int init_splitk() {
    int e = set_split_attrs<uint16_t, true>();
    if (!e) e = set_split_attrs<float, true>();
    if (!e) e = set_split_attrs<uint16_t, false>();
    if (!e) e = set_split_attrs<float, false>();
    return e;
}

int launch_splitk(const LaunchArgs &a, const bf16l_plan &p) {
    const bool clus = p.kernel == BF16L_KERNEL_SPLITK;
    if (a.out_f32) return clus ? launch_split_t<float, true>(a, p) : launch_split_t<float, false>(a, p);
    return clus ? launch_split_t<uint16_t, true>(a, p) : launch_split_t<uint16_t, false>(a, p);
}

}  // namespace bf16l
