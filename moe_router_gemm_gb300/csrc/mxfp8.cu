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
// before that wait.  For large M the tile form below (tcgen05 block-scaled
// MMAs, scales in TMEM) takes over.
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

// ---------------------------------------------------------------------------
// The tile form for large M: tcgen05.mma.kind::mxf8f6f4.block_scale, one
// instruction per 32-code scale block, scales applied by the tensor core.
//   * tile 128 x rows (MMA M) x BQ W rows (MMA N, 128 or 256); a stage is one
//     128-code chunk of both operands (128-byte swizzle rows, TMA) = four
//     scale blocks;
//   * warp 0 loads the codes (TMA), warp 1 issues the MMAs and owns TMEM,
//     warps 2-5 run the epilogue (TMEM lane = x row; bias, bf16 store), warps
//     6-9 stage each chunk's scale words into TMEM ahead of the MMAs: the word
//     of row r for chunk c is the four bytes xs[r][4c..4c+3] (k-blocks 0..3 of
//     the chunk), so MMA step kk selects byte kk (the descriptor's scale id);
//     the words of the next four chunks are always in flight;
//   * TMEM: the accumulator (two BQ-column buffers for BQ = 128, one for 256,
//     whose epilogue then runs between tiles), then one scale slot per ring
//     stage at a column that is a multiple of 8 (the MMA takes scale addresses
//     at aligned columns only).  The MMA reads A row m's word from lane m of
//     column sfa + m / 32 and B row n's from lane n % 32 of column sfb + n / 32
//     in the lane quarter of the D row it computes: a slot holds A's 4 columns
//     (quarter q's words in column q) and then, from column 4 (BQ = 128) or 8
//     (BQ = 256), B's BQ / 32 columns, written by all four scale warps (every
//     quarter a copy).
// ---------------------------------------------------------------------------
constexpr int kMxtThreads = 320;
constexpr int kMxtBP = 128, kMxtChunk = 128;  // codes per stage
constexpr int kMxtMaxStages = 6;

__host__ __device__ constexpr int mxt_stage_bytes(int bq) { return (kMxtBP + bq) * 128; }

struct MxtShared {
    uint64_t full[kMxtMaxStages];
    uint64_t empty[kMxtMaxStages];
    uint64_t sfull[kMxtMaxStages];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint32_t tmem_base;
    int32_t aborted;
    int32_t issued;
    int32_t consumed;
};

__device__ __forceinline__ void mxt_coords(int t, int p_tiles, int q_tiles, int group, int bq, int &p0, int &q0) {
    const int per_group = group * p_tiles;
    const int g = t / per_group, r = t - g * per_group;
    const int gq = (q_tiles - g * group) < group ? (q_tiles - g * group) : group;
    const int pi = r / gq, qi = g * group + (r - pi * gq);
    p0 = pi * kMxtBP;
    q0 = qi * bq;
}

// V4: the scale rows are read 16 bytes (four chunks' words) at a time (K % 512 == 0, xs and ws 16-byte
// aligned).  One 4-byte word per lane and chunk, from rows 128 or 256 bytes apart (K = 4096 or 8192),
// measured 40% slower over the whole kernel than at any neighbouring K.
template <int BQ, bool V4>
__global__ void __launch_bounds__(kMxtThreads, 1)
    mxtile_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                  const uint8_t *__restrict__ xs, const uint8_t *__restrict__ ws, const uint16_t *__restrict__ bias,
                  uint16_t *__restrict__ out, int M, int N, int K, int stages, int group, int32_t *status) {
    constexpr int kNbuf = BQ == 128 ? 2 : 1;          // accumulator buffers
    constexpr int kBcols = BQ / 32;                   // B scale columns per ring slot
    constexpr int kSlot = 4 + kBcols <= 8 ? 8 : 16;   // columns per slot (a multiple of 8)
    constexpr int kBoff = kBcols <= 4 ? 4 : 8;        // B's columns within a slot (8-aligned when it has 8)
    constexpr int kSf = kNbuf * BQ;                   // the scale slots start after the accumulators
    constexpr int kStageBytes = mxt_stage_bytes(BQ);
    static_assert(kSf + kMxtMaxStages * kSlot <= 512, "TMEM columns");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *ring = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    MxtShared &sh = *reinterpret_cast<MxtShared *>(ring + stages * kStageBytes);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int p_tiles = (M + kMxtBP - 1) / kMxtBP, q_tiles = (N + BQ - 1) / BQ;
    const int num_tiles = p_tiles * q_tiles;
    const int C = K / kMxtChunk;
    const int nb = K >> 5;  // scale bytes per row
    const int G = group > 0 ? group : 8;

    if (tid == 0) {
        tma_prefetch_desc(&tm_x);
        tma_prefetch_desc(&tm_w);
        for (int s = 0; s < stages; ++s) {
            mbar_init(&sh.full[s], 1);
            mbar_init(&sh.empty[s], 1);
            mbar_init(&sh.sfull[s], 4);  // one arrival per scale warp
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
        tmem_alloc(&sh.tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;
    pdl_launch_dependents();

    if (warp == 0) {
        if (lane == 0) {  // ---- TMA producer: the codes ----
            pdl_wait();
            int it = 0;
            for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
                int p0, q0;
                mxt_coords(t, p_tiles, q_tiles, G, BQ, p0, q0);
                for (int c = 0; c < C; ++c, ++it) {
                    const int s = it % stages;
                    if (it >= stages && !mbar_wait(&sh.empty[s], ((it / stages) - 1) & 1, status, kSiteEmpty)) {
                        atomicExch(&sh.aborted, 1);
                        goto producer_done;
                    }
                    if (*((volatile int32_t *)&sh.aborted)) goto producer_done;
                    uint8_t *st = ring + s * kStageBytes;
                    mbar_arrive_expect_tx(&sh.full[s], kStageBytes);
                    tma_load_2d(st, &tm_x, &sh.full[s], c * kMxtChunk, p0);
                    tma_load_2d(st + kMxtBP * 128, &tm_w, &sh.full[s], c * kMxtChunk, q0);
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
                const int b = tile_iter % kNbuf, use = tile_iter / kNbuf;
                const uint32_t acc = tmem + (uint32_t)(b * BQ);
                // wait for the epilogue to have drained this buffer (its previous use)
                if (use >= 1 && !mbar_wait(&sh.acc_empty[b], (use - 1) & 1, status, kSiteTmemEmpty)) {
                    atomicExch(&sh.aborted, 1);
                    break;
                }
                tc_fence_after();
                bool ok = true;
                for (int c = 0; c < C; ++c, ++it) {
                    const int s = it % stages;
                    if (!mbar_wait(&sh.full[s], (it / stages) & 1, status, kSiteFull) ||
                        !mbar_wait(&sh.sfull[s], (it / stages) & 1, status, kSiteFull)) {
                        atomicExch(&sh.aborted, 1);
                        sh.consumed = it;
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint8_t *st = ring + s * kStageBytes;
                    const uint64_t adesc = smem_desc_sw128(smem_u32(st));
                    const uint64_t bdesc = smem_desc_sw128(smem_u32(st + kMxtBP * 128));
                    const uint32_t sfa = tmem + (uint32_t)(kSf + kSlot * s), sfb = sfa + kBoff;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)  // one 32-code scale block per MMA, its byte of the words
                        mma_mxf8(acc, adesc + 2 * kk, bdesc + 2 * kk, idesc_mxf8_f32(kMxtBP, BQ, kk), sfa, sfb,
                                 (c > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(&sh.empty[s]);  // frees the codes and the scale slot
                }
                if (!ok) {
                    mbar_arrive(&sh.acc_full[b]);
                    break;
                }
                mma_commit(&sh.acc_full[b]);
            }
            sh.consumed = it;
        }
        __syncwarp();
    } else if (warp < 6) {
        // ---- epilogue: warps 2..5; TMEM lane quarter = warp % 4 ----
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        int tile_iter = 0;
        const bool vec_ok = (N % 8) == 0;
        for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++tile_iter) {
            int p0, q0;
            mxt_coords(t, p_tiles, q_tiles, G, BQ, p0, q0);
            const int b = tile_iter % kNbuf, use = tile_iter / kNbuf;
            // The tile's bias, one value per lane and 32-column slice, read while the MMAs run.
            pdl_wait();  // bias may be written by the previous kernel
            float lbs[BQ / 32];
#pragma unroll
            for (int i = 0; i < BQ / 32; ++i) lbs[i] = bias_lane(bias, q0 + 32 * i, N);
            const bool ok = mbar_wait(&sh.acc_full[b], use & 1, status, kSiteAccum);
            tc_fence_after();
            // warp-uniform, so that the bias shuffles below run on all 32 lanes
            const bool have = __all_sync(0xFFFFFFFFu, ok && !*((volatile int32_t *)&sh.aborted));
            const int m = p0 + row;
            const uint32_t acc = tmem + (uint32_t)(b * BQ) + ((uint32_t)(quarter * 32) << 16);
            if (have) {
#pragma unroll
                for (int c = 0; c < BQ; c += 32) {
                    const float lb = lbs[c / 32];
                    uint32_t r0[16], r1[16];
                    tmem_ld16(acc + (uint32_t)c, r0);
                    tmem_ld16(acc + (uint32_t)(c + 16), r1);
                    tmem_ld_wait16(r0);
                    tmem_ld_wait16(r1);
                    const int n = q0 + c;
                    float v[32];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        v[j] = __uint_as_float(r0[j]);
                        v[16 + j] = __uint_as_float(r1[j]);
                    }
                    if (bias && n < N) bias_add32(v, lb);  // warp-uniform condition
                    if (m < M && n < N) {
                        uint16_t *o = out + (size_t)m * N + n;
                        if (vec_ok && n + 32 <= N) {
#pragma unroll
                            for (int j = 0; j < 32; j += 8) OutStore<uint16_t>::eight(o + j, v + j);
                        } else {
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                if (n + j < N) OutStore<uint16_t>::one(o + j, v[j]);
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.acc_empty[b]);
            if (!have) break;
        }
    } else {
        // ---- scale staging: warps 6..9, one per TMEM lane quarter ----
        const int quarter = warp & 3;
        const uint32_t qlane = (uint32_t)(quarter * 32) << 16;
        pdl_wait();  // the scales may be written by the previous kernel
        int it = 0;
        for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
            int p0, q0;
            mxt_coords(t, p_tiles, q_tiles, G, BQ, p0, q0);
            const int ra = p0 + quarter * 32 + lane;  // this lane's x row (A scales, its own quarter)
            const uint32_t *wa = reinterpret_cast<const uint32_t *>(xs + (size_t)(ra < M ? ra : 0) * nb);
            const uint32_t *wb[kBcols];
            bool inb[kBcols];
#pragma unroll
            for (int j = 0; j < kBcols; ++j) {
                const int rb = q0 + 32 * j + lane;  // W rows of B scale column j (every quarter holds them)
                inb[j] = rb < N;
                wb[j] = reinterpret_cast<const uint32_t *>(ws + (size_t)(inb[j] ? rb : 0) * nb);
            }
            if constexpr (V4) {
                // words of chunks 4g..4g+3 in one 16-byte load per row; group g + 1 is in flight while g is used
                const uint4 kOne = make_uint4(0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
                const int ng = C / 4;
                const uint4 *ga = reinterpret_cast<const uint4 *>(wa);
                const uint4 *gb[kBcols];
#pragma unroll
                for (int j = 0; j < kBcols; ++j) gb[j] = reinterpret_cast<const uint4 *>(wb[j]);
                uint4 ca = (ng > 0 && ra < M) ? __ldg(ga) : kOne, na = (ng > 1 && ra < M) ? __ldg(ga + 1) : kOne;
                uint4 cbw[kBcols], nbw[kBcols];
#pragma unroll
                for (int j = 0; j < kBcols; ++j) {
                    cbw[j] = (ng > 0 && inb[j]) ? __ldg(gb[j]) : kOne;
                    nbw[j] = (ng > 1 && inb[j]) ? __ldg(gb[j] + 1) : kOne;
                }
                auto pick = [](const uint4 &v, int k) { return k == 0 ? v.x : k == 1 ? v.y : k == 2 ? v.z : v.w; };
                bool stop = false;
                for (int c = 0; c < C; ++c, ++it) {
                    const int s = it % stages;
                    if (it >= stages && !mbar_wait(&sh.empty[s], ((it / stages) - 1) & 1, status, kSiteScale)) {
                        atomicExch(&sh.aborted, 1);
                        stop = true;
                    }
                    stop = __any_sync(0xffffffffu, stop) || *((volatile int32_t *)&sh.aborted);
                    if (stop) break;
                    const int k = c & 3;
                    const uint32_t sf = tmem + (uint32_t)(kSf + kSlot * s) + qlane;
                    const uint32_t aw = pick(ca, k);
                    tmem_st4(sf, aw, aw, aw, aw);  // column `quarter` of the four is the one read
#pragma unroll
                    for (int j = 0; j < kBcols; j += 4)
                        tmem_st4(sf + kBoff + j, pick(cbw[j], k), pick(cbw[j + 1], k), pick(cbw[j + 2], k),
                                 pick(cbw[j + 3], k));
                    if (k == 3) {  // next group; fetch the one after
                        const int gn = c / 4 + 2;
                        ca = na;
                        na = (gn < ng && ra < M) ? __ldg(ga + gn) : kOne;
#pragma unroll
                        for (int j = 0; j < kBcols; ++j) {
                            cbw[j] = nbw[j];
                            nbw[j] = (gn < ng && inb[j]) ? __ldg(gb[j] + gn) : kOne;
                        }
                    }
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sh.sfull[s]);
                }
                if (stop) break;
                continue;
            }
            // The words of chunks c..c+3 are in flight together (a[d], bw[j][d] = chunk c + d), so the
            // L2 round trip of a chunk's words overlaps the three chunks before it.
            constexpr int PD = 4;
            uint32_t a[PD], bw[kBcols][PD];
#pragma unroll
            for (int d = 0; d < PD; ++d) {
                a[d] = (d < C && ra < M) ? __ldg(wa + d) : 0x7F7F7F7Fu;
#pragma unroll
                for (int j = 0; j < kBcols; ++j) bw[j][d] = (d < C && inb[j]) ? __ldg(wb[j] + d) : 0x7F7F7F7Fu;
            }
            bool stop = false;
            for (int c = 0; c < C; ++c, ++it) {
                const int s = it % stages;
                if (it >= stages && !mbar_wait(&sh.empty[s], ((it / stages) - 1) & 1, status, kSiteScale)) {
                    atomicExch(&sh.aborted, 1);
                    stop = true;
                }
                stop = __any_sync(0xffffffffu, stop) || *((volatile int32_t *)&sh.aborted);
                if (stop) break;
                const uint32_t sf = tmem + (uint32_t)(kSf + kSlot * s) + qlane;
                tmem_st4(sf, a[0], a[0], a[0], a[0]);  // column `quarter` of the four is the one read
#pragma unroll
                for (int j = 0; j < kBcols; j += 4)
                    tmem_st4(sf + kBoff + j, bw[j][0], bw[j + 1][0], bw[j + 2][0], bw[j + 3][0]);
                // shift the window and fetch chunk c + PD
#pragma unroll
                for (int d = 0; d + 1 < PD; ++d) {
                    a[d] = a[d + 1];
#pragma unroll
                    for (int j = 0; j < kBcols; ++j) bw[j][d] = bw[j][d + 1];
                }
                const int cn = c + PD;
                a[PD - 1] = (cn < C && ra < M) ? __ldg(wa + cn) : 0x7F7F7F7Fu;
#pragma unroll
                for (int j = 0; j < kBcols; ++j) bw[j][PD - 1] = (cn < C && inb[j]) ? __ldg(wb[j] + cn) : 0x7F7F7F7Fu;
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sh.sfull[s]);
            }
            if (stop) break;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
        for (int i = sh.consumed; i < sh.issued; ++i)
            mbar_wait(&sh.full[i % stages], (i / stages) & 1, status, kSiteDrain);
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

using MxFn = void (*)(const uint8_t *, const uint8_t *, const uint8_t *, const uint8_t *, const uint16_t *,
                      uint16_t *, int, int, int, int, int32_t *, int);

MxFn pick_mx(int M) { return M > 8 ? mxfp8_linear_kernel<true, uint16_t> : mxfp8_linear_kernel<false, uint16_t>; }

}  // namespace

int mxtile_smem_bytes(int stages, int bq) {
    const int need = 1024 + stages * mxt_stage_bytes(bq) + 256;
    return need > 116 * 1024 ? need : 116 * 1024;  // one CTA per SM (each allocates all 512 TMEM columns)
}

int mxtile_max_stages(int bq) {
    const int fit = (232448 - 1024 - 256) / mxt_stage_bytes(bq);
    return fit < kMxtMaxStages ? fit : kMxtMaxStages;
}

int init_mxfp8() {
    for (int M : {8, 16}) {
        const int e = (int)cudaFuncSetAttribute(pick_mx(M), cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e) return e;
    }
    int e = (int)cudaFuncSetAttribute(mxtile_kernel<128, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      mxtile_smem_bytes(mxtile_max_stages(128), 128));
    if (!e)
        e = (int)cudaFuncSetAttribute(mxtile_kernel<256, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      mxtile_smem_bytes(mxtile_max_stages(256), 256));
    if (!e)
        e = (int)cudaFuncSetAttribute(mxtile_kernel<128, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      mxtile_smem_bytes(mxtile_max_stages(128), 128));
    if (!e)
        e = (int)cudaFuncSetAttribute(mxtile_kernel<256, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      mxtile_smem_bytes(mxtile_max_stages(256), 256));
    return e;
}

int launch_mxfp8_tile(const void *xq, const void *xs, const void *wq, const void *ws, const void *bias, void *out,
                      int M, int N, int K, int bq, int stages, int group, int grid, uint32_t flags, void *stream,
                      int32_t *status) {
    if ((bq != 128 && bq != 256) || stages < 2 || stages > mxtile_max_stages(bq)) return (int)cudaErrorInvalidValue;
    CUtensorMap tx, tw;  // 128-byte rows of 128 codes
    int r = make_tmap_u8_2d(&tx, xq, (uint64_t)M, (uint64_t)K, kMxtBP, kMxtChunk, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    if (r) return (int)cudaErrorInvalidValue;
    r = make_tmap_u8_2d(&tw, wq, (uint64_t)N, (uint64_t)K, (uint32_t)bq, kMxtChunk, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    if (r) return (int)cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kMxtThreads);
    cfg.dynamicSmemBytes = (size_t)mxtile_smem_bytes(stages, bq);
    cfg.stream = (cudaStream_t)stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl_attr_of(flags);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // 16-byte scale reads when every scale row starts on a 16-byte boundary
    const bool v4 = K % 512 == 0 && ((reinterpret_cast<uintptr_t>(xs) | reinterpret_cast<uintptr_t>(ws)) & 15u) == 0;
    auto fn = bq == 128 ? (v4 ? mxtile_kernel<128, true> : mxtile_kernel<128, false>)
                        : (v4 ? mxtile_kernel<256, true> : mxtile_kernel<256, false>);
    return (int)cudaLaunchKernelEx(&cfg, fn, tx, tw,
                                   static_cast<const uint8_t *>(xs), static_cast<const uint8_t *>(ws),
                                   static_cast<const uint16_t *>(bias), static_cast<uint16_t *>(out), M, N, K, stages,
                                   group, status);
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
