// api.cu — the C ABI: argument validation, per-device initialisation, the
// kernel status word, TMA descriptor encoding and the launch itself.
//
// Validation follows the contract in bf16_linear.h: sizes and pointers are
// checked before any CUDA call (so the checks also run on hosts without a GPU),
// then the device is checked (compute capability 10.3 only), then the plan is
// made and exactly one kernel is launched.  Nothing here allocates device
// memory or synchronises a stream.
#include <cudaTypedefs.h>
#include <stdint.h>

#include <functional>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace bf16l {

// The kernel status word (one per device, in this module's device image).
__device__ int32_t g_status = 0;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceState {
    std::once_flag once;
    int err = 0;  // cudaError_t of the initialisation
    bf16l_device dev = {0, 0, 0};
    int32_t *status = nullptr;
};
DeviceState g_devices[kMaxDevices];

thread_local int t_last_cuda_error = 0;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

int note(int cuda_err) {
    if (cuda_err != 0) t_last_cuda_error = cuda_err;
    return cuda_err;
}

void init_device(DeviceState &s) {
    int d = 0;
    int e = (int)cudaGetDevice(&d);
    if (!e) e = (int)cudaDeviceGetAttribute(&s.dev.cc_major, cudaDevAttrComputeCapabilityMajor, d);
    if (!e) e = (int)cudaDeviceGetAttribute(&s.dev.cc_minor, cudaDevAttrComputeCapabilityMinor, d);
    if (!e) e = (int)cudaDeviceGetAttribute(&s.dev.num_sms, cudaDevAttrMultiProcessorCount, d);
    if (!e && s.dev.cc_major == 10 && s.dev.cc_minor == 3) {
        // Host code cannot take the address of a __device__ variable directly:
        // ask the runtime for this device's copy.
        void *p = nullptr;
        e = (int)cudaGetSymbolAddress(&p, g_status);
        s.status = static_cast<int32_t *>(p);
        if (!e) e = init_dotprod();
        if (!e) e = init_dotprod_f32();
        if (!e) e = init_splitk();
        if (!e) e = init_tile();
        if (!e) e = init_stream();
        if (!e) e = init_tile2();
        if (!e) e = init_warprow();
        if (!e) e = init_warpmma();
        if (!e) e = init_warpmma_ks();
        if (!e) e = init_dotmma();
        if (!e) e = init_mxfp8();
    }
    s.err = e;
}

// Current device's state, initialised once.  Returns a bf16l_status.
int current_device(DeviceState **out) {
    int d = 0;
    const int e = (int)cudaGetDevice(&d);
    if (e) {
        note(e);
        return BF16L_ELAUNCH;
    }
    if (d < 0 || d >= kMaxDevices) return BF16L_ELAUNCH;
    DeviceState &s = g_devices[d];
    std::call_once(s.once, init_device, std::ref(s));
    if (s.err) {
        note(s.err);
        return BF16L_ELAUNCH;
    }
    if (s.dev.cc_major != 10 || s.dev.cc_minor != 3) return BF16L_EARCH;
    *out = &s;
    return BF16L_OK;
}

bool misaligned(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

bool overlaps(const void *a, uint64_t abytes, const void *b, uint64_t bbytes) {
    if (!a || !b || abytes == 0 || bbytes == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + bbytes && b0 < a0 + abytes;
}

// Size and pointer checks that need no GPU.  BF16L_OK means "go on".
int check_args(const void *x, const void *W, const void *bias, void *out, int M, int N, int K, int out_elem) {
    if (M < 0 || N <= 0 || K <= 0) return BF16L_EINVAL;
    if (M == 0) return BF16L_OK;
    if (!x || !W || !out) return BF16L_EINVAL;
    if (misaligned(x) || misaligned(W) || misaligned(out) || (bias && misaligned(bias))) return BF16L_EALIGN;
    const uint64_t xb = 2ull * (uint64_t)M * (uint64_t)K, wb = 2ull * (uint64_t)N * (uint64_t)K;
    const uint64_t ob = (uint64_t)out_elem * (uint64_t)M * (uint64_t)N, bb = bias ? 2ull * (uint64_t)N : 0;
    if (overlaps(out, ob, x, xb) || overlaps(out, ob, W, wb) || overlaps(out, ob, bias, bb)) return BF16L_EINVAL;
    return BF16L_OK;
}

int run(const bf16l_call &c) {
    const bf16l_plan *forced = c.plan;
    const uint32_t flags = forced ? (uint32_t)forced->flags : c.flags;
    int st = check_args(c.x, c.W, c.bias, c.out, c.M, c.N, c.K, c.out_f32 ? 4 : 2);
    if (st != BF16L_OK) return st;
    if (!flags_valid(flags)) return BF16L_EINVAL;
    if (c.workspace && (reinterpret_cast<uintptr_t>(c.workspace) & 255u)) return BF16L_EALIGN;
    if (c.M == 0) return BF16L_OK;
    if (forced) {
        // Check the requested plan's shape rules before touching the device.
        bf16l_plan tmp = *forced;
        const bf16l_device any = {10, 3, kGb300Sms};
        st = check_plan(c.M, c.N, c.K, any, &tmp);
        if (st != BF16L_OK) return st;
        if (plan_ws_bytes(c.M, c.N, tmp) > (c.workspace ? c.workspace_bytes : 0)) return BF16L_EINVAL;
    }
    DeviceState *ds = nullptr;
    st = current_device(&ds);
    if (st != BF16L_OK) return st;

    bf16l_plan p;
    if (forced) {
        p = *forced;
        st = check_plan(c.M, c.N, c.K, ds->dev, &p);
    } else {
        st = bf16_linear_plan_ws(c.M, c.N, c.K, &ds->dev, c.workspace ? c.workspace_bytes : 0, &p);
        p.flags = (int32_t)flags;
    }
    if (st != BF16L_OK) return st;

    LaunchArgs a = {c.x,      c.W,          c.bias, c.out, c.M, c.N, c.K, c.stream, ds->dev.num_sms, ds->status,
                    c.out_f32, c.workspace, c.workspace ? c.workspace_bytes : 0};
    int e = 0;
    switch (p.kernel) {
        case BF16L_KERNEL_DOTPROD: e = launch_dotprod(a, p); break;
        case BF16L_KERNEL_SPLITK:
        case BF16L_KERNEL_SPLITK_WS: e = launch_splitk(a, p); break;
        case BF16L_KERNEL_TILE:
        case BF16L_KERNEL_TILE_T: e = launch_tile(a, p); break;
        case BF16L_KERNEL_STREAM: e = launch_stream(a, p); break;
        case BF16L_KERNEL_TILE2: e = launch_tile2(a, p); break;
        case BF16L_KERNEL_WARPROW: e = launch_warprow(a, p); break;
        case BF16L_KERNEL_WARPMMA: e = launch_warpmma(a, p); break;
        case BF16L_KERNEL_DOTMMA:
        case BF16L_KERNEL_DOTMMA_WS: e = launch_dotmma(a, p); break;
        default: return BF16L_EINVAL;
    }
    if (e) {
        note(e);
        return BF16L_ELAUNCH;
    }
    return BF16L_OK;
}

int run(const void *x, const void *W, const void *bias, void *out, int M, int N, int K, const bf16l_plan *forced,
        uint32_t flags, bf16l_stream_t stream, int out_f32 = 0) {
    bf16l_call c = {};
    c.x = x;
    c.W = W;
    c.bias = bias;
    c.out = out;
    c.M = M;
    c.N = N;
    c.K = K;
    c.out_f32 = out_f32;
    c.flags = flags;
    c.plan = forced;
    c.stream = stream;
    return run(c);
}

// One thread waits on an mbarrier that nothing arrives on, for limit_ns.
__global__ void selftest_wait_kernel(int32_t *status, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    mbar_init(&bar, 1);
    fence_barrier_init();
    mbar_wait(&bar, 0, status, kSiteSelftest, limit_ns);
    // Complete the barrier's phase ourselves so nothing is left pending.
    mbar_arrive(&bar);
}

}  // namespace

int current_device_checked(bf16l_device *dev) {
    DeviceState *ds = nullptr;
    const int st = current_device(&ds);
    if (st == BF16L_OK && dev) *dev = ds->dev;
    return st;
}

int note_cuda_error(int cuda_err) { return note(cuda_err); }

// cuTensorMapEncodeTiled, looked up once from the driver.
static PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode;
}

static int make_tmap_2d(CUtensorMap *map, CUtensorMapDataType dtype, uint64_t esize, const void *base,
                        uint64_t rows, uint64_t cols, uint32_t box_rows, uint32_t box_cols,
                        CUtensorMapSwizzle swizzle, CUtensorMapL2promotion promo) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
    if (!enc) return (int)CUDA_ERROR_NOT_FOUND;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * esize};  // bytes between rows
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return (int)enc(map, dtype, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle, promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

int make_tmap_bf16_2d(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                      uint32_t box_cols, CUtensorMapSwizzle swizzle, CUtensorMapL2promotion promo) {
    return make_tmap_2d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, rows, cols, box_rows, box_cols, swizzle,
                        promo);
}

int make_tmap_bf16_chunks(CUtensorMap *map, const void *base, uint64_t rows, uint64_t K, uint32_t box_rows,
                          uint32_t kc) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
    if (!enc) return (int)CUDA_ERROR_NOT_FOUND;
    if (K % kChunkK != 0 || kc < 1) return (int)CUDA_ERROR_INVALID_VALUE;
    const cuuint64_t dims[3] = {(cuuint64_t)kChunkK, rows, K / kChunkK};
    const cuuint64_t strides[2] = {K * 2, (cuuint64_t)kChunkK * 2};  // bytes between rows, between chunks
    const cuuint32_t box[3] = {(cuuint32_t)kChunkK, box_rows, kc};
    const cuuint32_t estr[3] = {1, 1, 1};
    return (int)enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

int make_tmap_u8_2d(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                    uint32_t box_cols, CUtensorMapSwizzle swizzle, CUtensorMapL2promotion promo) {
    return make_tmap_2d(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, base, rows, cols, box_rows, box_cols, swizzle, promo);
}

}  // namespace bf16l

// ---------------------------------------------------------------------------
// Exported entry points.
// ---------------------------------------------------------------------------
extern "C" int bf16_linear(const void *x, const void *W, const void *bias, void *out, int M, int N, int K,
                           bf16l_stream_t stream) {
    return bf16l::run(x, W, bias, out, M, N, K, nullptr, 0u, stream);
}

extern "C" int bf16_linear_ex(const void *x, const void *W, const void *bias, void *out, int M, int N, int K,
                              uint32_t flags, bf16l_stream_t stream) {
    return bf16l::run(x, W, bias, out, M, N, K, nullptr, flags, stream);
}

namespace {
size_t up256(size_t v) { return (v + 255) / 256 * 256; }
}  // namespace

extern "C" size_t bf16_linear_host_staging_bytes(int M, int N, int K, int with_bias) {
    if (M < 0 || N <= 0 || K <= 0) return 0;
    return up256(2ull * (size_t)M * (size_t)K) + up256(2ull * (size_t)N * (size_t)K) +
           (with_bias ? up256(2ull * (size_t)N) : 0) + up256(2ull * (size_t)M * (size_t)N);
}

extern "C" int bf16_linear_host(const void *x, const void *W, const void *bias, void *out, int M, int N, int K,
                                void *staging, size_t staging_bytes, uint32_t flags, bf16l_stream_t stream) {
    using namespace bf16l;
    if (M < 0 || N <= 0 || K <= 0 || !flags_valid(flags)) return BF16L_EINVAL;
    if (M == 0) return BF16L_OK;
    if (!x || !W || !out || !staging) return BF16L_EINVAL;
    if (reinterpret_cast<uintptr_t>(staging) & 255u) return BF16L_EALIGN;
    if (staging_bytes < bf16_linear_host_staging_bytes(M, N, K, bias != nullptr)) return BF16L_EINVAL;
    const size_t bx = 2ull * (size_t)M * (size_t)K, bw = 2ull * (size_t)N * (size_t)K, bb = 2ull * (size_t)N,
                 bo = 2ull * (size_t)M * (size_t)N;
    uint8_t *dx = static_cast<uint8_t *>(staging);
    uint8_t *dw = dx + up256(bx);
    uint8_t *db = bias ? dw + up256(bw) : nullptr;
    uint8_t *dout = dw + up256(bw) + (bias ? up256(bb) : 0);
    const cudaStream_t s = (cudaStream_t)stream;
    int e = (int)cudaMemcpyAsync(dx, x, bx, cudaMemcpyHostToDevice, s);
    if (!e) e = (int)cudaMemcpyAsync(dw, W, bw, cudaMemcpyHostToDevice, s);
    if (!e && bias) e = (int)cudaMemcpyAsync(db, bias, bb, cudaMemcpyHostToDevice, s);
    if (e) {
        note(e);
        return BF16L_ELAUNCH;
    }
    const int st = bf16l::run(dx, dw, db, dout, M, N, K, nullptr, flags, stream);
    if (st != BF16L_OK) return st;
    e = (int)cudaMemcpyAsync(out, dout, bo, cudaMemcpyDeviceToHost, s);
    if (e) {
        note(e);
        return BF16L_ELAUNCH;
    }
    return BF16L_OK;
}

extern "C" int bf16_linear_f32out(const void *x, const void *W, const void *bias, float *out, int M, int N, int K,
                                  uint32_t flags, bf16l_stream_t stream) {
    return bf16l::run(x, W, bias, out, M, N, K, nullptr, flags, stream, 1);
}

extern "C" int bf16_linear_f32out_with_plan(const void *x, const void *W, const void *bias, float *out, int M, int N,
                                            int K, const bf16l_plan *plan, bf16l_stream_t stream) {
    if (!plan) return BF16L_EINVAL;
    return bf16l::run(x, W, bias, out, M, N, K, plan, (uint32_t)plan->flags, stream, 1);
}

extern "C" int bf16_linear_with_plan(const void *x, const void *W, const void *bias, void *out, int M, int N,
                                     int K, const bf16l_plan *plan, bf16l_stream_t stream) {
    if (!plan) return BF16L_EINVAL;
    return bf16l::run(x, W, bias, out, M, N, K, plan, (uint32_t)plan->flags, stream);
}

extern "C" int bf16_linear_run(const bf16l_call *call) {
    if (!call) return BF16L_EINVAL;
    return bf16l::run(*call);
}

// ---- per-tensor FP8 ----

extern "C" int bf16_linear_fp8_split(int M, int N, int K, int num_sms) {
    // K splits of the FP8 kernel: the smallest power of two that gives about two
    // CTAs per SM, at most 8 (16-CTA clusters measured slower on every shape)
    // and at most one 64-code block each.
    if (M <= 0 || N <= 0 || K <= 0 || num_sms <= 0) return 1;
    const long long base = (long long)((N + 7) / 8) * ((M + 15) / 16);
    const int nblk = (K / 16 + 3) / 4;
    int S = 1;
    while (S < 8 && 2 * S <= nblk && base * S < 2LL * num_sms) S *= 2;
    return S;
}

extern "C" int bf16_linear_fp8_with_plan(const void *xq, const void *wq, const float *scale_x,
                                         const float *scale_w, const void *bias, void *out, int M, int N, int K,
                                         const bf16l_plan *plan, bf16l_stream_t stream);

extern "C" int bf16_linear_fp8(const void *xq, const void *wq, const float *scale_x, const float *scale_w,
                               const void *bias, void *out, int M, int N, int K, uint32_t flags,
                               bf16l_stream_t stream) {
    bf16l_plan p = {};
    p.kernel = BF16L_KERNEL_DOTMMA;
    p.threads = 0;  // chosen below, with the split, for this shape
    p.flags = (int32_t)flags;
    return bf16_linear_fp8_with_plan(xq, wq, scale_x, scale_w, bias, out, M, N, K, &p, stream);
}

extern "C" int bf16_linear_fp8_with_plan(const void *xq, const void *wq, const float *scale_x,
                                         const float *scale_w, const void *bias, void *out, int M, int N, int K,
                                         const bf16l_plan *plan, bf16l_stream_t stream) {
    using namespace bf16l;
    if (!plan) return BF16L_EINVAL;
    if (plan->chunks_per_stage != 0 && plan->chunks_per_stage != 1) return BF16L_EINVAL;
    const uint32_t flags = (uint32_t)plan->flags;
    if (M < 0 || N <= 0 || K <= 0) return BF16L_EINVAL;
    if (!flags_valid(flags)) return BF16L_EINVAL;
    if (M == 0) return BF16L_OK;
    if (!xq || !wq || !out || !scale_x || !scale_w) return BF16L_EINVAL;
    if (misaligned(xq) || misaligned(wq) || misaligned(out) || (bias && misaligned(bias)) ||
        (reinterpret_cast<uintptr_t>(scale_x) & 3u) || (reinterpret_cast<uintptr_t>(scale_w) & 3u))
        return BF16L_EALIGN;
    if (K % 16 != 0) return BF16L_EUNSUPPORTED;  // 16-byte rows of e4m3 codes
    const uint64_t ob = 2ull * (uint64_t)M * (uint64_t)N;
    if (overlaps(out, ob, xq, (uint64_t)M * K) || overlaps(out, ob, wq, (uint64_t)N * K) ||
        overlaps(out, ob, bias, bias ? 2ull * N : 0))
        return BF16L_EINVAL;
    DeviceState *ds = nullptr;
    const int st = current_device(&ds);
    if (st != BF16L_OK) return st;
    int kernel = plan->kernel, S = plan->split_k, threads = plan->threads, wpr = plan->rows_per_cta,
        cps = plan->stages;
    if (threads == 0) {  // the entry point's own choice
        const long long tiles = (long long)((M + kTileBM - 1) / kTileBM) * ((N + kTileBN - 1) / kTileBN);
        if (M > 16 && tiles >= 32) {  // a dense contraction with enough tiles: the tcgen05 tile form
            kernel = BF16L_KERNEL_TILE;
            threads = kTileThreads;
            cps = tile_max_stages(kTileBN);
        } else if (M <= kWarpMmaMaxTokens && (size_t)M * K <= (size_t)kWarpMmaMaxSmem && N >= 1024) {
            // Many rows: the persistent warp-MMA form.  Measured on GB300: more,
            // smaller CTAs per SM win where x is small enough to stage that often.
            kernel = BF16L_KERNEL_WARPMMA;
            const long long xs = (long long)M * K + 32 * 32 * 4 * 4 + 1024;
            if (N >= 8192 && M <= 4 && 4 * xs <= 232448) {
                threads = 256, wpr = 2, cps = 4;
            } else if (2 * xs <= 232448) {
                threads = 512, wpr = N >= 8192 ? 4 : 8, cps = 2;
            } else {
                threads = 1024, wpr = 8, cps = 1;
            }
        } else {
            kernel = BF16L_KERNEL_DOTMMA;
            S = bf16_linear_fp8_split(M, N, K, ds->dev.num_sms);
            threads = 128;
        }
    }
    int e = 0;
    if (kernel == BF16L_KERNEL_DOTMMA) {
        if ((threads != 128 && threads != 256) || (S != 1 && S != 2 && S != 4 && S != 8 && S != 16) ||
            S > (K / 16 + 3) / 4)
            return BF16L_EINVAL;
        e = launch_dotmma_fp8(xq, wq, scale_x, scale_w, bias, out, M, N, K, S, threads, flags, stream, ds->status);
    } else if (kernel == BF16L_KERNEL_WARPMMA) {
        // x (M x K codes) staged in shared memory; 8 W rows per group of wpr warps
        if (M > kWarpMmaMaxTokens || (size_t)M * K > (size_t)kWarpMmaMaxSmem) return BF16L_EUNSUPPORTED;
        const int static_smem = (wpr > 1 ? 32 * 32 * 4 * 4 : 512) + 1024;
        if ((threads != 256 && threads != 512 && threads != 1024) ||
            (wpr != 1 && wpr != 2 && wpr != 4 && wpr != 8 && wpr != 16) || (threads / 32) % wpr != 0 ||
            (wpr > 1 && (threads / 32) / wpr > 15) || S != 0 || cps < 1 || cps > 4 || threads * cps > 1024 ||
            (long long)cps * ((long long)M * K + static_smem) > 232448)
            return BF16L_EINVAL;
        const long long ctas = (long long)ds->dev.num_sms * cps, groups = (N + 7) / 8;
        e = launch_warpmma_fp8(xq, wq, scale_x, scale_w, bias, out, M, N, K, wpr, threads,
                               (int)(ctas < groups ? ctas : groups), flags, stream, ds->status);
    } else if (kernel == BF16L_KERNEL_TILE) {
        // stages = ring depth; tiles of 128 x rows by 256 W rows, 128 codes per 128-byte swizzle row
        if (threads != kTileThreads || cps < kTileMinStages || cps > tile_max_stages(kTileBN)) return BF16L_EINVAL;
        const long long tiles = (long long)((M + kTileBM - 1) / kTileBM) * ((N + kTileBN - 1) / kTileBN);
        const int grid = (int)(tiles < ds->dev.num_sms ? tiles : ds->dev.num_sms);
        e = launch_tile_fp8(xq, wq, scale_x, scale_w, bias, out, M, N, K, cps, grid, flags, stream, ds->status);
    } else {
        return BF16L_EINVAL;
    }
    if (e) {
        note(e);
        return BF16L_ELAUNCH;
    }
    return BF16L_OK;
}

extern "C" int bf16_quant_fp8(const void *x, const float *scale, void *xq, int64_t n, uint32_t flags,
                              bf16l_stream_t stream) {
    using namespace bf16l;
    if (n < 0 || !flags_valid(flags)) return BF16L_EINVAL;
    if (n == 0) return BF16L_OK;
    if (!x || !scale || !xq) return BF16L_EINVAL;
    if ((reinterpret_cast<uintptr_t>(x) & 1u) || (reinterpret_cast<uintptr_t>(scale) & 3u)) return BF16L_EALIGN;
    if (overlaps(xq, (uint64_t)n, x, 2ull * (uint64_t)n)) return BF16L_EINVAL;
    DeviceState *ds = nullptr;
    const int st = current_device(&ds);
    if (st != BF16L_OK) return st;
    const int e = launch_quant_fp8(x, scale, xq, (long long)n, ds->dev.num_sms, flags, stream);
    if (e) {
        note(e);
        return BF16L_ELAUNCH;
    }
    return BF16L_OK;
}

// ---- MXFP8 ----

extern "C" int bf16_linear_mxfp8_split(int M, int N, int K, int threads, int num_sms) {
    return bf16l::mxfp8_split(M, N, K, threads, num_sms);
}

extern "C" int bf16_quant_mxfp8(const void *x, int64_t rows, int K, void *xq, void *xs, uint32_t flags,
                                bf16l_stream_t stream) {
    using namespace bf16l;
    if (rows < 0 || K <= 0 || !flags_valid(flags)) return BF16L_EINVAL;
    if (K % 32 != 0) return BF16L_EUNSUPPORTED;
    if (rows == 0) return BF16L_OK;
    if (!x || !xq || !xs) return BF16L_EINVAL;
    if (misaligned(x) || misaligned(xq)) return BF16L_EALIGN;
    const uint64_t n = (uint64_t)rows * (uint64_t)K;
    if (n > (1ull << 40)) return BF16L_EINVAL;
    if (overlaps(xq, n, x, 2 * n) || overlaps(xs, n / 32, x, 2 * n) || overlaps(xs, n / 32, xq, n))
        return BF16L_EINVAL;
    DeviceState *ds = nullptr;
    const int st = current_device(&ds);
    if (st != BF16L_OK) return st;
    const int e = launch_quant_mxfp8(x, xq, xs, (long long)n, ds->dev.num_sms, flags, stream);
    if (e) {
        note(e);
        return BF16L_ELAUNCH;
    }
    return BF16L_OK;
}

extern "C" int bf16_linear_mxfp8_with_plan(const void *xq, const void *xs, const void *wq, const void *ws,
                                           const void *bias, void *out, int M, int N, int K, const bf16l_plan *plan,
                                           bf16l_stream_t stream) {
    using namespace bf16l;
    if (!plan) return BF16L_EINVAL;
    if (plan->chunks_per_stage != 0 && plan->chunks_per_stage != 1) return BF16L_EINVAL;
    const uint32_t flags = (uint32_t)plan->flags;
    if (M < 0 || N <= 0 || K <= 0 || !flags_valid(flags)) return BF16L_EINVAL;
    if (K % 32 != 0) return BF16L_EUNSUPPORTED;  // whole 32-element scale blocks
    if (M == 0) return BF16L_OK;
    if (!xq || !xs || !wq || !ws || !out) return BF16L_EINVAL;
    if (misaligned(xq) || misaligned(wq) || misaligned(out) || (bias && misaligned(bias))) return BF16L_EALIGN;
    if ((N + 7) / 8 > 65535 || (M + 15) / 16 > 65535) return BF16L_EUNSUPPORTED;
    const uint64_t ob = 2ull * (uint64_t)M * (uint64_t)N, nb = (uint64_t)(K / 32);
    if (overlaps(out, ob, xq, (uint64_t)M * K) || overlaps(out, ob, wq, (uint64_t)N * K) ||
        overlaps(out, ob, xs, (uint64_t)M * nb) || overlaps(out, ob, ws, (uint64_t)N * nb) ||
        overlaps(out, ob, bias, bias ? 2ull * N : 0))
        return BF16L_EINVAL;
    int kernel = plan->kernel, threads = plan->threads, S = plan->split_k, stages = plan->stages;
    int bq = plan->rows_per_cta;
    if (threads == 0) {  // the entry point's own choice
        const long long tiles256 = (long long)((M + 127) / 128) * ((N + 255) / 256);
        if (M > 16 && K % 128 == 0 && tiles256 >= 32) {  // a dense contraction: the tcgen05 tile form
            kernel = BF16L_KERNEL_TILE;
            threads = kMxTileThreads;
            bq = 256;
            stages = 3;  // measured: 8-10% faster than the deepest ring (4) on the prefill shapes
            S = 0;
        } else {
            kernel = BF16L_KERNEL_DOTMMA;
            threads = 128;
            S = mxfp8_split(M, N, K, threads, kGb300Sms);
        }
    }
    if (kernel == BF16L_KERNEL_TILE) {
        // 128 x 128 tiles of whole 128-code chunks; scale rows read as 32-bit words (4-byte aligned)
        if (K % 128 != 0) return BF16L_EUNSUPPORTED;
        if (threads != kMxTileThreads || (bq != 128 && bq != 256) || stages < 2 || stages > mxtile_max_stages(bq) ||
            S < 0 || S > 1024)
            return BF16L_EINVAL;
        if ((reinterpret_cast<uintptr_t>(xs) & 3u) || (reinterpret_cast<uintptr_t>(ws) & 3u)) return BF16L_EALIGN;
    } else if (kernel == BF16L_KERNEL_DOTMMA) {
        if ((threads != 128 && threads != 256) || (S != 1 && S != 2 && S != 4 && S != 8 && S != 16) || S > K / 32)
            return BF16L_EINVAL;
    } else {
        return BF16L_EINVAL;
    }
    DeviceState *ds = nullptr;
    const int st = current_device(&ds);
    if (st != BF16L_OK) return st;
    int e = 0;
    if (kernel == BF16L_KERNEL_TILE) {
        const long long tiles = (long long)((M + 127) / 128) * ((N + bq - 1) / bq);
        const int grid = (int)(tiles < ds->dev.num_sms ? tiles : ds->dev.num_sms);
        e = launch_mxfp8_tile(xq, xs, wq, ws, bias, out, M, N, K, bq, stages, S, grid, flags, stream, ds->status);
    } else {
        if (plan->threads == 0) S = mxfp8_split(M, N, K, threads, ds->dev.num_sms);
        e = launch_mxfp8(xq, xs, wq, ws, bias, out, M, N, K, S, threads, flags, stream, ds->status);
    }
    if (e) {
        note(e);
        return BF16L_ELAUNCH;
    }
    return BF16L_OK;
}

extern "C" int bf16_linear_mxfp8(const void *xq, const void *xs, const void *wq, const void *ws, const void *bias,
                                 void *out, int M, int N, int K, uint32_t flags, bf16l_stream_t stream) {
    bf16l_plan p = {};
    p.kernel = BF16L_KERNEL_DOTMMA;
    p.threads = 0;  // the entry point's own choice
    p.flags = (int32_t)flags;
    return bf16_linear_mxfp8_with_plan(xq, xs, wq, ws, bias, out, M, N, K, &p, stream);
}

extern "C" int bf16_linear_device_status(int32_t *status, int clear) {
    using namespace bf16l;
    if (!status) return BF16L_EINVAL;
    DeviceState *ds = nullptr;
    const int st = current_device(&ds);
    if (st != BF16L_OK) return st;
    int32_t v = 0;
    int e = (int)cudaMemcpy(&v, ds->status, sizeof v, cudaMemcpyDeviceToHost);
    if (!e && clear) {
        const int32_t zero = 0;
        e = (int)cudaMemcpy(ds->status, &zero, sizeof zero, cudaMemcpyHostToDevice);
    }
    if (e) {
        note(e);
        return BF16L_ELAUNCH;
    }
    *status = v;
    return BF16L_OK;
}

extern "C" int bf16_linear_selftest_wait(uint32_t limit_us, bf16l_stream_t stream) {
    using namespace bf16l;
    DeviceState *ds = nullptr;
    const int st = current_device(&ds);
    if (st != BF16L_OK) return st;
    selftest_wait_kernel<<<1, 1, 0, (cudaStream_t)stream>>>(ds->status, (uint64_t)limit_us * 1000ull);
    const int e = (int)cudaGetLastError();
    if (e) {
        note(e);
        return BF16L_ELAUNCH;
    }
    return BF16L_OK;
}

extern "C" const char *bf16_linear_strerror(int status) {
    switch (status) {
        case BF16L_OK: return "ok";
        case BF16L_EINVAL: return "invalid argument";
        case BF16L_EALIGN: return "pointer not 16-byte aligned";
        case BF16L_EARCH: return "device is not compute capability 10.3 (GB300)";
        case BF16L_ELAUNCH: return "CUDA launch or device query failed";
        case BF16L_ETIMEOUT: return "a kernel wait timed out";
        case BF16L_EUNSUPPORTED: return "the requested kernel does not support this shape";
        case BF16L_ENOSCRATCH: return "the shape needs more scratch than the fixed no-allocation array holds";
        default: return "unknown status";
    }
}

extern "C" int bf16_linear_cuda_error(void) { return bf16l::t_last_cuda_error; }

extern "C" int bf16_linear_version(void) { return 1 * 10000 + 0 * 100 + 0; }
