// kernels.h — internal interface between the C ABI (api.cu), the planner
// (plan.cpp) and the three kernels.  Host-only declarations: no CUDA headers,
// so the planner builds and runs without a GPU.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include "bf16_linear.h"

namespace bf16l {

// ---- parameter limits shared by the planner and the launchers ----

// Dot-product kernel: tokens handled per pass over W (one template instance
// per count), W rows per CTA, and block sizes.
constexpr int kDotMaxTokens = 8;
constexpr int kDotRows[] = {1, 2, 4};
constexpr int kDotThreads[] = {64, 128, 256};
// CTAs along y of a dot-product launch: one per token group of `tokens`
// (0 = a single CTA row that loops over groups of kDotMaxTokens).
inline int dot_token_groups(int M, int tokens) {
    if (tokens <= 0 || M <= 0) return 1;
    const int mt = M < tokens ? M : tokens;
    return (M + mt - 1) / mt;
}

// Cluster split-K kernel: tokens (M <= 64, padded to a multiple of 8) on the
// MMA M side, 16..256 weight rows per CTA on the N side, K split over up to 16
// CTAs of one cluster, up to 16 ring stages.
constexpr int kSplitMaxTokens = 64;
constexpr int kSplitMaxCluster = 16;
constexpr int kSplitMaxStages = 16;
constexpr int kSplitThreads = 128;
// Shared-memory layout arithmetic of the split-K kernel (defined in splitk.cu).
int split_stage_bytes(int tokens, int rows, int kc = 1);  // kc: 64-wide K chunks per ring stage
int split_recv_bytes(int tokens, int rows);
int split_smem_bytes(int tokens, int rows, int stages, int kc = 1);
int split_max_stages(int tokens, int rows, int kc = 1);  // 0 when even one stage does not fit
int split_tmem_cols(int rows);
bool split_rows_supported(int rows);         // a kernel instance exists for this many rows
constexpr int kSplitWsMaxSplit = 64;         // K splits of the cluster-free (workspace) variant
// Workspace layout of the cluster-free split-K: per-tile arrival counters
// (rounded up to 256 bytes), then the fp32 partial tiles [tiles][S][M][rows].
size_t split_ws_counter_bytes(int tiles);
size_t split_ws_bytes(int M, int N, const bf16l_plan &p);

// Streaming kernel: M <= 4 tokens, K <= 8192 (x slice held in registers),
// 1, 2 or 4 W rows per ring stage (4 only for M <= 3), one CTA per SM.
constexpr int kStreamMaxTokens = 4;
constexpr int kStreamMaxStages = 16;
constexpr int kStreamMaxRows = 4;
constexpr int kStreamMaxK = 8192;
constexpr int kStreamThreads = 288;
int stream_smem_bytes(int K, int rows, int stages);
int init_stream();

// Tile kernel: 128 rows of one operand on the MMA M side by BN rows of the
// other on the N side, 64-wide K chunks.  Plain form (BF16L_KERNEL_TILE): x rows
// on M, BN W rows on N; swap-AB form (BF16L_KERNEL_TILE_T): W rows on M, BN
// tokens on N.  The ring takes as many stages as fit 227 KB, at most 8.
constexpr int kTileBM = 128;
constexpr int kTileBN = 256;
constexpr int kTileMinStages = 2;
constexpr int kTileMaxStages = 8;
constexpr int kTileThreads = 192;
constexpr int kTileDefaultGroup = 8;  // raster group (N-tiles) of the plain form when a plan gives 0
constexpr int kTileBNs[] = {128, 192, 224, 240, 256};  // plain form: W rows per tile
constexpr int kTileTBNs[] = {32, 64, 128, 192, 256};   // swap-AB form: tokens per tile
constexpr int tile_max_stages(int bn) {
    return (232448 - 1024 - 256) / (128 * 128 + bn * 128) < kTileMaxStages
               ? (232448 - 1024 - 256) / (128 * 128 + bn * 128)
               : kTileMaxStages;
}
int tile_smem_bytes(int stages, int bn);
int init_tile_t();

// Warp-per-row kernel: M <= 8 tokens staged in shared memory (M*K*2 bytes),
// 256/512/1024 threads, 1/2/4 warps per row, a few CTAs per SM.
constexpr int kWarpRowMaxTokens = 8;
constexpr int kWarpRowMaxSmem = 200 * 1024;
int warprow_smem_bytes(int M, int K);
int init_warprow();

// Warp-level tensor-core kernel: M <= 16 tokens staged in shared memory,
// 8 W rows per group of 1..16 warps.
constexpr int kWarpMmaMaxTokens = 16;
constexpr int kWarpMmaMaxSmem = 200 * 1024;
int warpmma_smem_bytes(int M, int K);
int init_warpmma();
// Its cluster form (WARPMMA plans with split_k = S >= 2): K split over S CTAs
// of a cluster, each staging its K slice of up to 64 tokens; partial tiles
// summed through distributed shared memory.  `clusters` of S CTAs.
constexpr int kWarpMmaKsMaxTokens = 64;
constexpr int kWarpMmaKsMaxCluster = 16;  // above 8: a non-portable cluster size
constexpr int kWarpMmaKsMaxSmem = 231424;  // 226 KB dynamic: the kernel has static barriers too
int warpmma_ks_smem_bytes(int M, int N, int K, int S, int clusters, int threads, int wpr);
int init_warpmma_ks();

// Router split-K on warp-level MMAs: 8 W rows per CTA, K over a cluster of
// 1, 2, 4 or 8 CTAs, M <= 16, each CTA stages its K slice of x.
constexpr int kDotMmaMaxTokens = 16;
constexpr int kDotMmaMaxCluster = 16;
constexpr int kDotMmaMaxSmem = 200 * 1024;
int dotmma_smem_bytes(int M, int K, int S);
constexpr int kDotMmaWsMaxSplit = 64;  // K splits of the cluster-free (workspace) form
size_t dotmma_ws_counter_bytes(int groups);
size_t dotmma_ws_bytes(int N, const bf16l_plan &p);
// Workspace bytes a plan needs (0 for every kernel but the two cluster-free forms).
inline size_t plan_ws_bytes(int M, int N, const bf16l_plan &p) { return split_ws_bytes(M, N, p) + dotmma_ws_bytes(N, p); }
int init_dotmma();

// Pair tile kernel (cta_group::2): 256 x rows x 256 W rows per cluster of 2,
// 32 KB ring stages per CTA.
constexpr int kTile2MinStages = 2;
constexpr int kTile2MaxStages = 6;
int tile2_smem_bytes(int stages, int bn);  // bn: W rows per pair tile, 256 or 192
int init_tile2();

constexpr int kChunkK = 64;  // K elements per TMA box row (128 bytes, the swizzle width)

// GB300 default device description (cc 10.3, 152 SMs).
constexpr int kGb300Sms = 152;

// The current device, initialised once (kernel attributes) and checked to be
// compute capability 10.3: BF16L_OK and *dev filled, else the status to return
// (a failed CUDA call is recorded for bf16_linear_cuda_error).  Defined in api.cu.
int current_device_checked(bf16l_device *dev);
// Record a CUDA error code for bf16_linear_cuda_error (0 is ignored); returns it.
int note_cuda_error(int cuda_err);

// BF16L_FLAG_* bits a call may pass: known bits only, and not PDL with SERIAL.
inline bool flags_valid(uint32_t f) {
    return (f & ~(BF16L_FLAG_PDL | BF16L_FLAG_SERIAL)) == 0 && (f & (BF16L_FLAG_PDL | BF16L_FLAG_SERIAL)) !=
                                                                    (BF16L_FLAG_PDL | BF16L_FLAG_SERIAL);
}

// Validate a plan against a shape; BF16L_OK or the error to return.  Fills
// plan->grid.  Pure host logic.
int check_plan(int M, int N, int K, const bf16l_device &dev, bf16l_plan *plan);

// Device-side launchers (defined in the .cu files).
struct LaunchArgs {
    const void *x;
    const void *W;
    const void *bias;
    void *out;
    int M, N, K;
    void *stream;     // cudaStream_t
    int num_sms;
    int32_t *status;  // device address of the kernel status word
    int out_f32;      // 1: out is fp32 [M][N] (router logits); 0: bf16
    void *workspace;  // caller's scratch for workspace plans (zeroed once before first use), or null
    size_t workspace_bytes;
};

// Each returns a cudaError_t value (0 on success).
int launch_dotprod(const LaunchArgs &a, const bf16l_plan &p);
int launch_splitk(const LaunchArgs &a, const bf16l_plan &p);
int launch_tile(const LaunchArgs &a, const bf16l_plan &p);   // both tile forms
int launch_tile_swap(const LaunchArgs &a, const bf16l_plan &p);
int launch_stream(const LaunchArgs &a, const bf16l_plan &p);
int launch_tile2(const LaunchArgs &a, const bf16l_plan &p);
int launch_warprow(const LaunchArgs &a, const bf16l_plan &p);
int launch_warpmma(const LaunchArgs &a, const bf16l_plan &p);
int launch_warpmma_ks(const LaunchArgs &a, const bf16l_plan &p);
int launch_dotmma(const LaunchArgs &a, const bf16l_plan &p);
// Per-tensor FP8: the router MMA split-K kernel with e4m3 operands (K in bytes
// = codes; grid.z covers any M in groups of 16 tokens), and the static
// quantisation of bf16 values with a per-tensor scale.
int launch_dotmma_fp8(const void *xq, const void *wq, const float *sx, const float *sw, const void *bias, void *out,
                      int M, int N, int K, int S, int threads, uint32_t flags, void *stream, int32_t *status);
int launch_warpmma_fp8(const void *xq, const void *wq, const float *sx, const float *sw, const void *bias, void *out,
                       int M, int N, int K, int wpr, int threads, int grid, uint32_t flags, void *stream,
                       int32_t *status);
int launch_tile_fp8(const void *xq, const void *wq, const float *sx, const float *sw, const void *bias, void *out,
                    int M, int N, int K, int stages, int grid, uint32_t flags, void *stream, int32_t *status);
int launch_quant_fp8(const void *x, const float *scale, void *q, long long n, int num_sms, uint32_t flags,
                     void *stream);
// MXFP8 (mxfp8.cu): block quantisation (n values, n % 32 == 0) and the block-scaled linear on warp-level
// e4m3 MMAs (K % 32 == 0; grid.z covers any M in groups of 16 tokens; S: CTAs per cluster along K, 1..16).
int init_mxfp8();
int mxfp8_split(int M, int N, int K, int threads, int num_sms);
int launch_quant_mxfp8(const void *x, void *q, void *scales, long long n, int num_sms, uint32_t flags, void *stream);
int launch_mxfp8(const void *xq, const void *xs, const void *wq, const void *ws, const void *bias, void *out, int M,
                 int N, int K, int S, int threads, uint32_t flags, void *stream, int32_t *status);
// The MXFP8 tile form (tcgen05 block-scaled MMAs): 128 x rows by bq (128 or 256) W rows per tile,
// K % 128 == 0, 320 threads, 2 up to mxtile_max_stages(bq) stages, persistent grid of at most one CTA per
// SM; group: raster group of W tiles (0 = 8).
constexpr int kMxTileThreads = 320;
int mxtile_max_stages(int bq);
int launch_mxfp8_tile(const void *xq, const void *xs, const void *wq, const void *ws, const void *bias, void *out,
                      int M, int N, int K, int bq, int stages, int group, int grid, uint32_t flags, void *stream,
                      int32_t *status);

// One-time per-device kernel attribute setup (dynamic shared memory limits,
// non-portable cluster sizes).  Returns a cudaError_t value.
int init_dotprod();
int init_dotprod_f32();
int launch_dotprod_f32(const LaunchArgs &a, const bf16l_plan &p);
int init_splitk();
int init_tile();

}  // namespace bf16l
