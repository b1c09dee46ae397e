// plan.cpp — shape -> kernel dispatch (pure host code, no CUDA calls).
//
// Structure follows the vLLM LL-BF16 router GEMM dispatcher (vLLM PR #48774
// page, LLBf16Gemm.dispatch / _arch_tuned_configs): a table keyed by (K, N)
// with one entry per M, measured on the target GPU, decides; anything not in
// the table falls back to size rules.  The page's own rule (dot product when
// M <= 4 or K < 2048, split-K otherwise, default (split_k, num_stages) =
// (6, 4)) was tuned on other hardware; here the table is re-measured on GB300
// (dispatch_table.inc, written by the sweep in bench.py) and the size rules
// are only the starting point for shapes it does not list.
#include <stdint.h>

#include <initializer_list>

#include "bf16_linear.h"
#include "kernels.h"

namespace bf16l {

namespace {

struct TableEntry {
    int K, N, M;
    int kernel, threads, rows_per_cta, tokens_per_cta, split_k, stages;
    int chunks_per_stage;  // 0 when the entry leaves it out
};

// Measured on GB300 (sm_103a, 152 SMs).  Regenerate with `python bench.py --sweep`.
const TableEntry kTable[] = {
#include "dispatch_table.inc"
    {0, 0, 0, 0, 0, 0, 0, 0, 0}  // sentinel
};

int ceil_div(int a, int b) { return (a + b - 1) / b; }

int round_up(int a, int b) { return ceil_div(a, b) * b; }

bool in_list(int v, const int *list, int n) {
    for (int i = 0; i < n; ++i)
        if (list[i] == v) return true;
    return false;
}

void plan_dotprod(int M, int N, int K, const bf16l_device &dev, bf16l_plan *p) {
    (void)K;
    // GB300 sweep: one W row per CTA for a single token on small N, two rows
    // otherwise (each x vector then serves two rows), four on very large N.
    p->kernel = BF16L_KERNEL_DOTPROD;
    p->threads = (N >= 16 * dev.num_sms) ? 128 : 256;
    p->rows_per_cta = (M == 1 && N < 8 * dev.num_sms) ? 1 : (N < 64 * dev.num_sms ? 2 : 4);
}

void plan_splitk(int M, int N, int K, const bf16l_device &dev, bf16l_plan *p) {
    // GB300 sweep: 64 weight rows x a 16-CTA cluster for router-sized N; for
    // large N, 256 rows and as many K splits as give about half a CTA per SM
    // (each CTA then streams a deep ring).
    const int chunks = ceil_div(K, kChunkK);
    int rows, split;
    if (N <= 512) {
        rows = 64;
        split = kSplitMaxCluster;
    } else {
        rows = 256;
        const int tiles = ceil_div(N, rows);
        split = ceil_div(dev.num_sms / 2, tiles);
        if (split < 1) split = 1;
        if (split > 8) split = 8;
    }
    if (split > chunks) split = chunks;
    p->kernel = BF16L_KERNEL_SPLITK;
    p->threads = kSplitThreads;
    p->rows_per_cta = rows;
    p->tokens_per_cta = round_up(M, 8);
    p->split_k = split;
    const int per_cta = ceil_div(chunks, split);
    const int max_stages = split_max_stages(p->tokens_per_cta, rows);
    p->stages = per_cta < max_stages ? per_cta : max_stages;
}

void plan_tile(int M, int N, int K, const bf16l_device &dev, bf16l_plan *p) {
    (void)M;
    (void)N;
    (void)K;
    (void)dev;
    p->kernel = BF16L_KERNEL_TILE;
    p->threads = kTileThreads;
    p->rows_per_cta = kTileBN;
    p->tokens_per_cta = kTileBM;
    p->stages = tile_max_stages(kTileBN);
}

}  // namespace

int check_plan(int M, int N, int K, const bf16l_device &dev, bf16l_plan *p) {
    if (M < 0 || N <= 0 || K <= 0) return BF16L_EINVAL;
    if (!flags_valid((uint32_t)p->flags)) return BF16L_EINVAL;
    const int kc = p->chunks_per_stage;
    if (kc < 0 || kc > 2) return BF16L_EINVAL;
    const bool ring_kernel = p->kernel == BF16L_KERNEL_SPLITK || p->kernel == BF16L_KERNEL_SPLITK_WS ||
                             p->kernel == BF16L_KERNEL_TILE || p->kernel == BF16L_KERNEL_TILE_T;
    if (kc == 2 && !ring_kernel) return BF16L_EINVAL;
    if (kc == 2 && K % kChunkK != 0) return BF16L_EUNSUPPORTED;  // the chunked tensor maps need whole chunks
    const int kcs = kc == 2 ? 2 : 1;
    switch (p->kernel) {
        case BF16L_KERNEL_DOTPROD: {
            if (!in_list(p->threads, kDotThreads, 3) || !in_list(p->rows_per_cta, kDotRows, 3))
                return BF16L_EINVAL;
            if (p->tokens_per_cta < 0 || p->tokens_per_cta > kDotMaxTokens) return BF16L_EINVAL;
            if (p->stages != 0 && p->stages != 1) return BF16L_EINVAL;  // 1: x read from L2, not staged
            p->grid = M == 0 ? 0 : ceil_div(N, p->rows_per_cta) * dot_token_groups(M, p->tokens_per_cta);
            return BF16L_OK;
        }
        case BF16L_KERNEL_SPLITK:
        case BF16L_KERNEL_SPLITK_WS: {
            const int max_split = p->kernel == BF16L_KERNEL_SPLITK ? kSplitMaxCluster : kSplitWsMaxSplit;
            if (K % 8 != 0) return BF16L_EUNSUPPORTED;  // TMA needs 16-byte row strides
            if (M > kSplitMaxTokens) return BF16L_EUNSUPPORTED;
            const int chunks = ceil_div(K, kChunkK);
            if (p->threads != kSplitThreads || !split_rows_supported(p->rows_per_cta)) return BF16L_EINVAL;
            if (p->tokens_per_cta < 8 || p->tokens_per_cta > kSplitMaxTokens || p->tokens_per_cta % 8 != 0 ||
                p->tokens_per_cta < M)
                return BF16L_EINVAL;
            // every rank needs at least one ring stage of kcs chunks
            if (p->split_k < 1 || p->split_k > max_split || p->split_k > ceil_div(chunks, kcs)) return BF16L_EINVAL;
            if (p->stages < 1 || p->stages > split_max_stages(p->tokens_per_cta, p->rows_per_cta, kcs))
                return BF16L_EINVAL;
            const int64_t grid = (int64_t)ceil_div(N, p->rows_per_cta) * p->split_k;
            if (ceil_div(N, p->rows_per_cta) > 65535) return BF16L_EUNSUPPORTED;
            p->grid = M == 0 ? 0 : (int)grid;
            return BF16L_OK;
        }
        case BF16L_KERNEL_STREAM: {
            if (K % 8 != 0 || K > kStreamMaxK || M > kStreamMaxTokens) return BF16L_EUNSUPPORTED;
            if (p->threads != kStreamThreads ||
                (p->rows_per_cta != 1 && p->rows_per_cta != 2 && p->rows_per_cta != 4) ||
                (p->rows_per_cta == 4 && M > 3))
                return BF16L_EINVAL;
            if (p->stages < 1 || p->stages > kStreamMaxStages ||
                stream_smem_bytes(K, p->rows_per_cta, p->stages) > 232448)
                return BF16L_EINVAL;
            p->grid = M == 0 ? 0 : (N < dev.num_sms ? N : dev.num_sms);
            return BF16L_OK;
        }
        case BF16L_KERNEL_TILE:
        case BF16L_KERNEL_TILE_T: {
            // plain: 128 x rows by rows_per_cta W rows per tile; swap-AB: 128 W rows by tokens_per_cta tokens
            if (K % 8 != 0) return BF16L_EUNSUPPORTED;
            const bool swap = p->kernel == BF16L_KERNEL_TILE_T;
            const int bn = swap ? p->tokens_per_cta : p->rows_per_cta;
            if (p->threads != kTileThreads || (swap ? p->rows_per_cta : p->tokens_per_cta) != kTileBM ||
                !(swap ? in_list(bn, kTileTBNs, 5) : in_list(bn, kTileBNs, 5)))
                return BF16L_EINVAL;
            if (p->stages < kTileMinStages || p->stages * kcs > tile_max_stages(bn)) return BF16L_EINVAL;
            if (p->split_k < 0 || p->split_k > 1024) return BF16L_EINVAL;  // raster group
            const int64_t tiles = swap ? (int64_t)ceil_div(N, kTileBM) * ceil_div(M, bn)
                                       : (int64_t)ceil_div(M, kTileBM) * ceil_div(N, bn);
            const int64_t grid = tiles < dev.num_sms ? tiles : dev.num_sms;
            p->grid = M == 0 ? 0 : (int)grid;
            return BF16L_OK;
        }
        case BF16L_KERNEL_WARPROW: {
            if (K % 8 != 0 || M > kWarpRowMaxTokens || warprow_smem_bytes(M, K) > kWarpRowMaxSmem)
                return BF16L_EUNSUPPORTED;
            const int t = p->threads, wpr = p->rows_per_cta, cps = p->stages;
            if ((t != 128 && t != 256 && t != 512 && t != 1024) || (wpr != 1 && wpr != 2 && wpr != 4) ||
                (t / 32) % wpr != 0)
                return BF16L_EINVAL;
            // a named barrier per row group (ids 1..15) when warps share a row
            if (wpr > 1 && (t / 32) / wpr > 15) return BF16L_EINVAL;
            if (cps < 1 || cps > 8 || t * cps > 2048 ||
                cps * (warprow_smem_bytes(M, K) + 2048) > 232448)
                return BF16L_EINVAL;
            const int64_t ctas = (int64_t)dev.num_sms * cps;
            p->grid = M == 0 ? 0 : (int)(ctas < N ? ctas : N);
            return BF16L_OK;
        }
        case BF16L_KERNEL_WARPMMA: {
            if (p->split_k >= 2) {
                // the cluster form: K over S CTAs, up to 64 tokens; 1024-thread blocks only for <= 16 tokens
                // (64 registers a thread), otherwise at most 512 threads per SM (128 registers)
                const int S = p->split_k, t = p->threads, wpr = p->rows_per_cta, cps = p->stages;
                if (K % 8 != 0 || M > kWarpMmaKsMaxTokens) return BF16L_EUNSUPPORTED;
                if ((t != 128 && t != 256 && t != 512 && t != 1024) || (t == 1024 && M > 16) ||
                    (wpr != 1 && wpr != 2 && wpr != 4 && wpr != 8 && wpr != 16) || (t / 32) % wpr != 0 ||
                    (wpr > 1 && (t / 32) / wpr > 15) || S > kWarpMmaKsMaxCluster || S > ceil_div(K / 8, 4) ||
                    cps < 1 || cps > 8 || t * cps > (M > 16 ? 512 : 1024))
                    return BF16L_EINVAL;
                int64_t clusters = (int64_t)dev.num_sms * cps / S;
                const int64_t groups = ceil_div(N, 8);
                if (clusters > groups) clusters = groups;
                // tokens_per_cta > 0: that many 8-row groups per cluster (fewer clusters, one x slice per CTA
                // serving several groups)
                if (p->tokens_per_cta < 0) return BF16L_EINVAL;
                if (p->tokens_per_cta > 0 && ceil_div(groups, p->tokens_per_cta) < clusters)
                    clusters = ceil_div(groups, p->tokens_per_cta);
                if (clusters < 1) return BF16L_EINVAL;
                const int smem = warpmma_ks_smem_bytes(M, N, K, S, (int)clusters, t, wpr);
                if (smem > kWarpMmaKsMaxSmem || (int64_t)cps * (smem + 1024) > 233472) return BF16L_EINVAL;
                p->grid = M == 0 ? 0 : (int)(clusters * S);
                return BF16L_OK;
            }
            // split_k 1: x fragments from L2 into registers (no shared-memory x, at most 512 threads per SM)
            const bool xr = p->split_k == 1;
            if (K % 8 != 0 || M > kWarpMmaMaxTokens || (!xr && warpmma_smem_bytes(M, K) > kWarpMmaMaxSmem))
                return BF16L_EUNSUPPORTED;
            const int t = p->threads, wpr = p->rows_per_cta, cps = p->stages;
            if ((t != 128 && t != 256 && t != 512 && t != 1024) ||
                (wpr != 1 && wpr != 2 && wpr != 4 && wpr != 8 && wpr != 16) || (t / 32) % wpr != 0 ||
                (p->split_k != 0 && p->split_k != 1))
                return BF16L_EINVAL;
            if (wpr > 1 && (t / 32) / wpr > 15) return BF16L_EINVAL;  // named barriers 1..15
            // tokens_per_cta: 8-row groups per warp, 0/1, 2 or 4 (2 and 4 only with x from L2)
            const int ng = p->tokens_per_cta > 1 ? p->tokens_per_cta : 1;
            if (p->tokens_per_cta < 0 || p->tokens_per_cta == 3 || p->tokens_per_cta > 4 || (ng > 1 && !xr))
                return BF16L_EINVAL;
            const int static_smem = (wpr > 1 ? 32 * 32 * 4 * 4 : 512) + 1024;
            if (cps < 1 || cps > 8 || t * cps > (xr ? 512 : 1024) ||
                cps * ((xr ? 0 : warpmma_smem_bytes(M, K)) + static_smem) > 232448)
                return BF16L_EINVAL;
            const int64_t ctas = (int64_t)dev.num_sms * cps, groups = ceil_div(N, 8 * ng);
            p->grid = M == 0 ? 0 : (int)(ctas < groups ? ctas : groups);
            return BF16L_OK;
        }
        case BF16L_KERNEL_DOTMMA:
        case BF16L_KERNEL_DOTMMA_WS: {
            // the cluster form takes up to 64 tokens in groups of 16 (grid.z); the workspace form 16
            if (K % 8 != 0 || M > (p->kernel == BF16L_KERNEL_DOTMMA ? 4 * kDotMmaMaxTokens : kDotMmaMaxTokens))
                return BF16L_EUNSUPPORTED;
            const int S = p->split_k;
            // clusters: 1..16 CTAs along K; the workspace form: any power of two up to 64
            const bool s_ok = p->kernel == BF16L_KERNEL_DOTMMA
                                  ? (S == 1 || S == 2 || S == 4 || S == 8 || S == 16)
                                  : (S >= 2 && S <= kDotMmaWsMaxSplit && (S & (S - 1)) == 0);
            if ((p->threads != 128 && p->threads != 256) || p->rows_per_cta != 8 || !s_ok ||
                S > ceil_div(K / 8, 4) || (p->stages != 0 && p->stages != 1))
                return BF16L_EINVAL;
            // stages 1: x straight from global memory; 0: the CTA's x slice staged in shared memory
            const int mg = M < kDotMmaMaxTokens ? M : kDotMmaMaxTokens;  // tokens of one group
            if (p->stages == 0 && dotmma_smem_bytes(mg, K, S) > kDotMmaMaxSmem) return BF16L_EUNSUPPORTED;
            p->grid = M == 0 ? 0 : S * ceil_div(N, 8) * ceil_div(M, kDotMmaMaxTokens);
            return BF16L_OK;
        }
        case BF16L_KERNEL_TILE2: {
            // A pair tile is 256 x rows x rows_per_cta W rows (256, or 192: 75 tiles for N = 14336, one per
            // pair of SMs); threads and the x rows are fixed.
            if (K % 8 != 0) return BF16L_EUNSUPPORTED;
            if (p->threads != kTileThreads || (p->rows_per_cta != 2 * kTileBM && p->rows_per_cta != 192) ||
                p->tokens_per_cta != 2 * kTileBM)
                return BF16L_EINVAL;
            if (p->stages < kTile2MinStages || p->stages > kTile2MaxStages) return BF16L_EINVAL;
            const int64_t units = (int64_t)ceil_div(M, 2 * kTileBM) * ceil_div(N, p->rows_per_cta);
            const int64_t pairs = dev.num_sms / 2;
            p->grid = M == 0 ? 0 : 2 * (int)(units < pairs ? units : pairs);
            return BF16L_OK;
        }
        default:
            return BF16L_EINVAL;
    }
}

}  // namespace bf16l

extern "C" int bf16_linear_plan_ws(int M, int N, int K, const bf16l_device *devp, size_t workspace_bytes,
                                   bf16l_plan *plan) {
    using namespace bf16l;
    if (!plan || M < 0 || N <= 0 || K <= 0) return BF16L_EINVAL;
    const bf16l_device gb300 = {10, 3, kGb300Sms};
    const bf16l_device &dev = devp ? *devp : gb300;
    if (dev.cc_major != 10 || dev.cc_minor != 3) return BF16L_EARCH;
    if (dev.num_sms <= 0) return BF16L_EINVAL;

    // The table lists, per shape, the fastest plan first; when that one needs
    // a workspace it is followed by the fastest plan that needs none.
    bf16l_plan p = {};
    bool from_table = false;
    for (const TableEntry *e = kTable; e->K != 0 && !from_table; ++e) {
        if (e->K != K || e->N != N || e->M != M) continue;
        p = bf16l_plan{};
        p.kernel = e->kernel;
        p.threads = e->threads;
        p.rows_per_cta = e->rows_per_cta;
        p.tokens_per_cta = e->tokens_per_cta;
        p.split_k = e->split_k;
        p.stages = e->stages;
        p.chunks_per_stage = e->chunks_per_stage;
        from_table = check_plan(M, N, K, dev, &p) == BF16L_OK && plan_ws_bytes(M, N, p) <= workspace_bytes;
    }
    if (!from_table) {
        p = bf16l_plan{};
        // The pages' rule was M <= 4 or K < 2048 for the dot product; on GB300
        // the dot product stays ahead up to M = 8 (one pass over W).
        if (K % 8 != 0 || M <= kDotMaxTokens || (M <= 16 && K < 2048))
            plan_dotprod(M, N, K, dev, &p);
        else if (M <= kSplitMaxTokens)
            plan_splitk(M, N, K, dev, &p);
        else
            plan_tile(M, N, K, dev, &p);
        const int st = check_plan(M, N, K, dev, &p);
        if (st != BF16L_OK) return st;
    }
    *plan = p;
    return BF16L_OK;
}

extern "C" int bf16_linear_plan_for_device(int M, int N, int K, const bf16l_device *devp, bf16l_plan *plan) {
    return bf16_linear_plan_ws(M, N, K, devp, 0, plan);
}

extern "C" int bf16_linear_plan(int M, int N, int K, bf16l_plan *out_plan) {
    return bf16_linear_plan_ws(M, N, K, nullptr, 0, out_plan);
}

extern "C" size_t bf16_linear_workspace_size(int M, int N, int K, const bf16l_plan *plan) {
    using namespace bf16l;
    if (M < 0 || N <= 0 || K <= 0) return 0;
    if (plan) return plan_ws_bytes(M, N, *plan);
    bf16l_plan p;
    if (bf16_linear_plan_ws(M, N, K, nullptr, (size_t)-1, &p) != BF16L_OK) return 0;
    return plan_ws_bytes(M, N, p);
}

extern "C" int bf16_linear_plan_check(int M, int N, int K, const bf16l_device *devp, bf16l_plan *plan) {
    using namespace bf16l;
    if (!plan) return BF16L_EINVAL;
    const bf16l_device gb300 = {10, 3, kGb300Sms};
    const bf16l_device &dev = devp ? *devp : gb300;
    if (dev.cc_major != 10 || dev.cc_minor != 3) return BF16L_EARCH;
    if (dev.num_sms <= 0) return BF16L_EINVAL;
    return check_plan(M, N, K, dev, plan);
}
