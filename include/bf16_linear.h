/*
 * bf16_linear.h — C ABI of the GB300 (sm_103a) skinny BF16 linear layer.
 *
 *     out[M,N] = x[M,K] @ W[N,K]^T (+ bias[N])
 *
 * Operation: the unquantised serving linear layer defined in the header comment
 * of the TGV BF16 GEMM kernel (sglang PR #30117 page, "关键源码片段": out[M, N]
 * = x[M, K] @ weight[N, K].T (+ bias[N]); bf16 inputs and output, fp32
 * accumulation inside).  Its hot regime is the decode / MoE-router shape with
 * M <= 16 tokens (vLLM PR #42562 page, "实现拆解" items 1-4), where reading W
 * from HBM sets the cost.
 *
 * Conventions shared by every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller, on the
 *    current CUDA device (bf16_linear_host alone takes host buffers).  The library keeps no reference after the call
 *    returns (the launch is asynchronous: buffers must stay valid until the
 *    stream reaches it).
 *  - Layouts are dense row-major with no padding: x[M][K], W[N][K] (the
 *    nn.Linear weight layout), out[M][N], bias[N].  Elements are IEEE bfloat16
 *    (the upper 16 bits of a binary32), except out of bf16_linear_f32out (fp32).
 *  - Pointers must be 16-byte aligned (the vLLM PR #42562 review lowered the
 *    assumed alignment of these kernels to 16 bytes).  out must not overlap
 *    x, W or bias.
 *  - Arithmetic: every product and sum in fp32, then out = RNE_bf16(acc + bias)
 *    (bias, when given, is added in fp32 before the single rounding).  The
 *    summation order depends on the kernel the plan picks; for a fixed plan the
 *    result is bitwise deterministic from run to run.
 *  - Nothing allocates device memory, nothing synchronises the stream, and the
 *    calls are safe to make from several host threads at once.  (Plans that
 *    need scratch memory run only when the caller passes a workspace to
 *    bf16_linear_run.)  A call may be
 *    captured in a CUDA graph once the device has been initialised by one
 *    earlier non-captured call on it (initialisation sets kernel attributes).
 *  - Device: compute capability 10.3 (GB300) only; any other device returns
 *    BF16L_EARCH (the TGV page notes its kernel is built for SM10x only and
 *    errors elsewhere; this library is built for sm_103a alone).
 *  - Errors are reported by return value; no entry point aborts the process.
 */
#ifndef BF16_LINEAR_H
#define BF16_LINEAR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* CUDA stream handle (a cudaStream_t / CUstream); NULL means the legacy default stream. */
typedef void *bf16l_stream_t;

typedef enum {
    BF16L_OK = 0,
    BF16L_EINVAL = -1,       /* bad size, NULL required pointer, or a plan that cannot run this shape */
    BF16L_EALIGN = -2,       /* a pointer is not 16-byte aligned */
    BF16L_EARCH = -3,        /* current device is not compute capability 10.3 */
    BF16L_ELAUNCH = -4,      /* the CUDA launch (or device query) failed; see bf16_linear_cuda_error */
    BF16L_ETIMEOUT = -5,     /* a kernel's bounded wait gave up (read via bf16_linear_device_status) */
    BF16L_EUNSUPPORTED = -6, /* the requested kernel does not support this shape (e.g. K % 8 != 0 for a TMA kernel) */
    BF16L_ENOSCRATCH = -7    /* bf16_linear_noalloc: the shape needs more scratch than its fixed array holds */
} bf16l_status;

/* Kernels behind the dispatcher. */
typedef enum {
    BF16L_KERNEL_DOTPROD = 0, /* CUDA-core dot product, 128-bit weight loads, one CTA per slice of W rows */
    BF16L_KERNEL_SPLITK = 1,  /* TMA -> tcgen05 (weights on the MMA M side), K split over a thread-block
                                 cluster, fp32 partials reduced through distributed shared memory */
    BF16L_KERNEL_TILE = 2,    /* persistent warp-specialised TMA -> tcgen05 -> TMEM tile GEMM */
    BF16L_KERNEL_SPLITK_WS = 3, /* the split-K kernel without a cluster: K split over up to 64 CTAs, fp32
                                   partials reduced through a caller-provided workspace (see bf16_linear_run) */
    BF16L_KERNEL_STREAM = 4,   /* persistent CUDA-core kernel for M <= 4 and K <= 8192: one CTA per SM streams
                                  a contiguous row range through a bulk-copy ring (large N: decode, MLP) */
    BF16L_KERNEL_TILE2 = 5,    /* persistent tcgen05 tile GEMM on CTA pairs (cta_group::2, clusters of 2):
                                  256 x 256 (or 256 x 192) tiles, each CTA stages half of each operand; large M */
    BF16L_KERNEL_WARPROW = 6,  /* persistent CUDA-core kernel for M <= 8 and many rows: a group of 1, 2 or 4
                                  warps computes one W row at a time from 16-byte loads, x in shared memory */
    BF16L_KERNEL_WARPMMA = 7,  /* persistent kernel for M <= 16 and many rows: 16-byte weight loads feed the
                                  warp-level tensor-core MMA (m16n8k16) directly; 8 W rows per group of warps.
                                  With split_k >= 2, its cluster form: K over S CTAs of a cluster, M <= 64, each
                                  CTA staging its K slice of x, partial tiles summed over DSMEM in rank order */
    BF16L_KERNEL_DOTMMA = 8,   /* router-sized N, M <= 64 (16-token groups): 8 W rows per CTA, K over a cluster of 1..16 CTAs,
                                  16-byte loads feed m16n8k16 MMAs, partials summed by rank 0 over DSMEM */
    BF16L_KERNEL_DOTMMA_WS = 9, /* the same without a cluster: K split over 2..64 CTAs whose partial tiles meet in
                                  a caller-provided workspace (see bf16_linear_run); the last CTA reduces */
    BF16L_KERNEL_TILE_T = 10   /* the tile kernel in the swap-AB orientation: 128 W rows on the MMA M side,
                                  tokens_per_cta tokens (32, 64, 128, 192 or 256) on the N side; mid-size M */
} bf16l_kernel;

/*
 * A launch plan: which kernel and its parameters.  Mirrors the dispatch key of
 * the vLLM LL-BF16 router GEMM (vLLM PR #42562 page, LLBf16Gemm.CompileKey:
 * backend, M, K, bs, split_k, num_stages), extended with the fields the
 * tcgen05 kernels need.  Fields a kernel does not use are 0.
 */
typedef struct {
    int32_t kernel;        /* bf16l_kernel */
    int32_t threads;       /* threads per CTA */
    int32_t rows_per_cta;  /* W rows per CTA (DOTPROD 1/2/4; SPLITK 16..256, the MMA N); TILE: W rows per tile
                              (the MMA N: 128, 192, 224, 240 or 256); TILE_T: 128 (the MMA M);
                              TILE2: W rows per pair tile (256 or 192);
                              STREAM: W rows per ring stage (1, 2, or 4 when M <= 3);
                              WARPROW: warps that share one row (1, 2 or 4);
                              WARPMMA: warps that share one group of 8 rows (1, 2, 4, 8 or 16) */
    int32_t tokens_per_cta;/* SPLITK: x rows loaded per chunk (M rounded up to 8, <= 64);  TILE: x rows per tile
                              (128); TILE_T: tokens per tile (the MMA N: 32, 64, 128, 192 or 256);
                              DOTPROD: tokens per CTA, 1..8 (0 = min(M, 8)); ceil(M / tokens) CTAs then share each
                              row slice, one token group each, instead of one CTA looping over the groups;
                              WARPMMA: 8-row groups a warp covers per x fragment, 1, 2 or 4 (2 and 4 only with
                              split_k = 1; 0 = 1); WARPMMA cluster form: 8-row groups per cluster (0 = as many clusters as fit) */
    int32_t split_k;       /* SPLITK: CTAs per cluster along K (1..16); SPLITK_WS: CTAs along K (1..64);
                              TILE / TILE_T: raster group, the N-side tiles walked together before the next row
                              of M-side tiles (0 = 8 for TILE, all of them for TILE_T);
                              DOTMMA: CTAs per cluster along K (1, 2, 4, 8 or 16);
                              DOTMMA_WS: CTAs along K (a power of two, 2..64);
                              WARPMMA: 1 = x fragments loaded from global memory into registers (512 threads per
                              SM at most), 0 = x staged in shared memory, S = 2..16: the cluster form (K over S
                              CTAs; 1024-thread blocks only for M <= 16, else at most 512 threads per SM) */
    int32_t stages;        /* SPLITK / TILE / TILE_T: shared-memory ring depth, in stages of chunks_per_stage
                              64-wide K chunks (TILE and TILE_T: 2 up to what fits 227 KB, stages x chunks at
                              most 8); DOTPROD: 1 = x read
                              from global memory (L2) instead of staged in shared memory;
                              WARPROW / WARPMMA: CTAs per SM; DOTMMA: 1 = x fragments loaded from global
                              memory into registers, 0 = each CTA's x slice staged in shared memory */
    int32_t grid;          /* CTAs launched (informational; computed by the plan) */
    int32_t flags;         /* BF16L_FLAG_* bits the launch uses */
    int32_t chunks_per_stage; /* SPLITK / SPLITK_WS / TILE / TILE_T: 64-wide K chunks per ring stage, 0 or 1 = one,
                              2 = two (K % 64 == 0; each stage is then one TMA box per operand holding two chunk
                              tiles, so a CTA issues half as many loads; `stages` counts these double stages, and
                              SPLITK / SPLITK_WS need split_k <= ceil(K / 128)); every other kernel: 0 or 1 */
} bf16l_plan;

/*
 * Launch modes.  By default every kernel is launched with programmatic
 * dependent launch (the mode the sglang PR #28333 page turns on wherever the
 * GPU supports it): it may be scheduled while the kernel before it on the
 * stream finishes, runs its set-up, and then waits for that kernel to complete
 * (griddepcontrol.wait) before it reads x, W or bias or writes out.  This is
 * always correct, whatever the previous kernel does; it hides the launch cost
 * of back-to-back calls.  It also lets the next kernel on the stream be
 * scheduled early; a kernel of another library that is launched with
 * programmatic dependent launch after this one must wait before it reads out,
 * as that launch mode requires.
 *
 * BF16L_FLAG_PDL: in addition, the kernel reads W and bias (and issues its
 * weight copies) BEFORE that wait, overlapping the weight fetch with the end
 * of the previous kernel.  Use only when W and bias are not written by the
 * kernel launched just before this call on the same stream (true for
 * weights).  x is still read, and out written, only after the wait.
 *
 * BF16L_FLAG_SERIAL: launch without programmatic dependent launch (the call
 * starts only once everything before it on the stream has completed).
 * BF16L_FLAG_PDL and BF16L_FLAG_SERIAL together are refused (BF16L_EINVAL).
 */
#define BF16L_FLAG_PDL 1u
#define BF16L_FLAG_SERIAL 2u

/*
 * Describe the device a plan is made for.  bf16_linear() fills this from the
 * current device; tests pass fake devices (the mock-device pattern of the
 * sglang PR #34042 page's backend tests).
 */
typedef struct {
    int32_t cc_major;      /* compute capability, 10 */
    int32_t cc_minor;      /* 3 for GB300 */
    int32_t num_sms;       /* streaming multiprocessors (152 on GB300) */
} bf16l_device;

/*
 * bf16_linear_plan — choose the kernel and parameters for (M, N, K) on a GB300
 * (cc 10.3, 152 SMs).
 *
 * Pure host code: makes no CUDA call and touches no device.  Rules (vLLM PR
 * #48774 page, LLBf16Gemm.dispatch and _arch_tuned_configs, with the
 * thresholds re-measured on GB300): a table measured on GB300 keyed by (K, N)
 * with one entry per M decides; shapes not in the table use size rules (dot
 * product for tiny M or K % 8 != 0, cluster split-K for skinny M, the tile
 * kernel for large M).
 *
 * Returns BF16L_OK and fills *out_plan; BF16L_EINVAL for M < 0, N <= 0, K <= 0
 * or out_plan == NULL.  M == 0 yields a plan with grid == 0 (nothing to launch).
 */
int bf16_linear_plan(int M, int N, int K, bf16l_plan *out_plan);

/*
 * bf16_linear_plan_for_device — bf16_linear_plan for the device `dev`
 * describes (NULL = a GB300).  The device is data, not a query, so tests can
 * plan for fake devices (the mock-device pattern of the sglang PR #34042
 * page's backend tests).  Same returns as bf16_linear_plan, plus BF16L_EARCH
 * when dev is not compute capability 10.3 and BF16L_EINVAL for
 * dev->num_sms <= 0.
 */
int bf16_linear_plan_for_device(int M, int N, int K, const bf16l_device *dev, bf16l_plan *plan);

/*
 * bf16_linear_plan_check — validate an explicit plan for (M, N, K) on `dev`
 * (NULL = GB300) and fill plan->grid.  Pure host code.  Returns BF16L_OK,
 * BF16L_EINVAL (a parameter outside the kernel's limits, or a shared-memory
 * ring that does not fit), BF16L_EUNSUPPORTED (the kernel cannot run this
 * shape, e.g. K % 8 != 0 for the TMA kernels) or BF16L_EARCH.
 */
int bf16_linear_plan_check(int M, int N, int K, const bf16l_device *dev, bf16l_plan *plan);

/*
 * bf16_linear — out = x @ W^T (+ bias), bf16 out, on `stream`.
 *
 * x: device bf16 [M][K]; W: device bf16 [N][K]; bias: device bf16 [N] or NULL;
 * out: device bf16 [M][N], written in full (every element), never read.
 * Asynchronous: returns after enqueueing one kernel launch (none when M == 0).
 * Returns BF16L_OK, BF16L_EINVAL (sizes, NULL x/W/out), BF16L_EALIGN,
 * BF16L_EARCH, or BF16L_ELAUNCH.
 */
int bf16_linear(const void *x, const void *W, const void *bias, void *out,
                int M, int N, int K, bf16l_stream_t stream);

/*
 * bf16_linear_ex — as bf16_linear, with BF16L_FLAG_* launch flags (0 = the
 * same as bf16_linear).  Unknown flag bits, or BF16L_FLAG_PDL together with
 * BF16L_FLAG_SERIAL, return BF16L_EINVAL.
 */
int bf16_linear_ex(const void *x, const void *W, const void *bias, void *out,
                   int M, int N, int K, uint32_t flags, bf16l_stream_t stream);

/*
 * bf16_linear_host — bf16_linear_ex on HOST buffers: copies x, W and bias from
 * host memory into a caller-provided device staging buffer, runs the planned
 * kernel there, and copies out back to host memory, all enqueued on `stream`
 * (one cudaMemcpyAsync per buffer, in that order).
 *
 * x: host bf16 [M][K]; W: host bf16 [N][K]; bias: host bf16 [N] or NULL;
 * out: host bf16 [M][N], written in full once the stream reaches the copy.
 * Page-locked host memory gives asynchronous copies; pageable memory works
 * but the driver then stages each copy synchronously.  staging: memory of the
 * current device (the one `stream` belongs to) of at least
 * bf16_linear_host_staging_bytes(M, N, K, bias != NULL) bytes,
 * 256-byte aligned, owned by the caller; the library lays out x, W, bias and
 * out in it at 256-byte aligned offsets and allocates nothing.  The host
 * buffers and the staging must stay valid, and unread/unwritten by the caller,
 * until the stream passes the final copy.
 * Returns BF16L_OK (M == 0: nothing enqueued), BF16L_EINVAL (sizes, NULL
 * x/W/out/staging, staging too small, unknown flags), BF16L_EALIGN (staging
 * not 256-byte aligned), BF16L_EARCH, or BF16L_ELAUNCH (a copy or the launch
 * failed; bf16_linear_cuda_error has the CUDA code).
 */
int bf16_linear_host(const void *x, const void *W, const void *bias, void *out, int M, int N, int K,
                     void *staging, size_t staging_bytes, uint32_t flags, bf16l_stream_t stream);

/* Device staging bytes bf16_linear_host needs for this shape (0 for invalid sizes).  Pure host code. */
size_t bf16_linear_host_staging_bytes(int M, int N, int K, int with_bias);

/*
 * bf16_linear_f32out — the router-logits variant: the same product and bias,
 * but out is fp32 [M][N] (each output is the fp32 accumulation plus the bias,
 * not rounded to bf16).  The vLLM PR #42562 page's split-K router kernel
 * writes fp32 (LLBf16SplitK, out_dtype=cutlass.Float32) so that top-k expert
 * selection sees unrounded logits.  Same plans, kernels, arguments, flags and
 * errors as bf16_linear_ex; out must be 16-byte aligned and not overlap the
 * inputs.
 */
int bf16_linear_f32out(const void *x, const void *W, const void *bias, float *out,
                       int M, int N, int K, uint32_t flags, bf16l_stream_t stream);

/* bf16_linear_f32out with an explicit plan (no fallback, as bf16_linear_with_plan). */
int bf16_linear_f32out_with_plan(const void *x, const void *W, const void *bias, float *out,
                                 int M, int N, int K, const bf16l_plan *plan, bf16l_stream_t stream);

/*
 * bf16_linear_with_plan — as bf16_linear, but run exactly `plan` (for tests,
 * sweeps and benchmarks).  No fallback: a plan that cannot run this shape
 * returns BF16L_EINVAL or BF16L_EUNSUPPORTED without launching (an explicit
 * request errors rather than silently falling back, as the sglang PR #34042
 * page's backend resolution does).
 */
int bf16_linear_with_plan(const void *x, const void *W, const void *bias, void *out,
                          int M, int N, int K, const bf16l_plan *plan, bf16l_stream_t stream);

/*
 * bf16_linear_device_status — read (and optionally clear) the current device's
 * kernel status word.  0 means no kernel gave up; otherwise the first failing
 * wait's code (BF16L_ETIMEOUT in the low byte, the wait site above it).
 * Sites: 1 MMA waiting for a stage, 2 producer waiting for a free stage,
 * 3 epilogue waiting for the accumulator, 4 MMA waiting for the epilogue,
 * 5 exit drain, 6 self-test, 7 split-K owner waiting for partials, 8 dot
 * product waiting for x, 9 the two CTAs of a pair (BF16L_KERNEL_TILE2) got
 * different TMEM addresses and gave up before any MMA.
 * Synchronises the device (reads device memory).  Returns BF16L_OK or
 * BF16L_ELAUNCH.
 */
int bf16_linear_device_status(int32_t *status, int clear);

/*
 * bf16_linear_selftest_wait — diagnostic for the bounded-wait path.  Launches
 * one thread that waits on a shared-memory barrier nothing ever completes and
 * gives up after limit_us microseconds, recording BF16L_ETIMEOUT (wait site 6)
 * in the device status word, exactly as a kernel whose wait ran out would.
 * The GPU stays usable.  Asynchronous; returns BF16L_OK, BF16L_EARCH or
 * BF16L_ELAUNCH.
 */
int bf16_linear_selftest_wait(uint32_t limit_us, bf16l_stream_t stream);

/*
 * The general entry point.  Every other launch entry point is a special case
 * of this one.
 *
 * workspace: device scratch for plans that need it (kernel
 * BF16L_KERNEL_SPLITK_WS), or NULL.  It must be 256-byte aligned, zero-filled
 * before its first use (one cudaMemset), and not shared by calls that can run
 * at the same time on different streams.  Consecutive calls on one stream may
 * share one, with or without BF16L_FLAG_PDL (a kernel touches the workspace
 * only after its grid-dependency wait).  Every completed call leaves the
 * workspace's counters zero again, so no clearing is needed between calls.  With plan == NULL the dispatcher may pick
 * a workspace plan only when workspace_bytes is large enough for it
 * (bf16_linear_workspace_size); otherwise it picks the best plan that needs
 * none.  With an explicit workspace plan and too small a workspace the call
 * returns BF16L_EINVAL.
 */
typedef struct {
    const void *x;            /* bf16 [M][K] */
    const void *W;            /* bf16 [N][K] */
    const void *bias;         /* bf16 [N] or NULL */
    void *out;                /* bf16 [M][N], or fp32 [M][N] when out_f32 */
    int32_t M, N, K;
    int32_t out_f32;          /* 0: bf16 out; 1: fp32 out (router logits) */
    uint32_t flags;           /* BF16L_FLAG_* (ignored when plan != NULL: plan->flags is used) */
    const bf16l_plan *plan;   /* NULL: the dispatcher chooses */
    void *workspace;          /* see above; may be NULL */
    size_t workspace_bytes;
    bf16l_stream_t stream;
} bf16l_call;

int bf16_linear_run(const bf16l_call *call);

/*
 * Bytes of workspace a call needs: for `plan` when given, else for the plan
 * the dispatcher picks for (M, N, K) on a GB300 when any workspace is
 * allowed.  0 when the plan needs none.  Pure host code.
 */
size_t bf16_linear_workspace_size(int M, int N, int K, const bf16l_plan *plan);

/*
 * The dispatcher's choice when `workspace_bytes` of workspace are available
 * (bf16_linear_plan_for_device is this with workspace_bytes == 0).  Pure host code.
 */
int bf16_linear_plan_ws(int M, int N, int K, const bf16l_device *dev, size_t workspace_bytes, bf16l_plan *plan);

/*
 * bf16_linear_noalloc — the same operation for callers that cannot allocate
 * device memory.  (No counterpart on the pages: it exists for callers such as
 * a plug-in that receives its input and output buffers from a host program
 * owning all device memory, and so has no way to obtain a workspace.)
 *
 * It runs the cluster-free split-K kernel (BF16L_KERNEL_SPLITK_WS) with its
 * scratch in a fixed array of bf16_linear_noalloc_scratch_bytes() (4 MiB)
 * that is part of the library's device image: every GPU that loads the
 * library holds it until the process exits.  Nothing is allocated or freed.
 * x, W, bias, out: as bf16_linear (bf16 out).  Requires M <= 64 and
 * K % 8 == 0 (else BF16L_EUNSUPPORTED); the plan takes fewer K splits until
 * its scratch fits, and a shape that does not fit even unsplit (about
 * M * N * 4 bytes > 4 MiB) returns BF16L_ENOSCRATCH.
 *
 * The first call on a device looks up the array's device address (with that
 * device current) and keeps it; make that first call before any stream
 * capture.  A lookup that fails returns BF16L_ELAUNCH (the CUDA code through
 * bf16_linear_cuda_error) and is tried again on the next call.  As every
 * entry point, it returns BF16L_EARCH on a device that is not a GB300,
 * before touching the device.
 * Each call clears the array's counters on `stream` before its launch (a
 * memset, which starts only once everything before it on the stream has
 * completed, so consecutive calls on one stream never overlap).  All calls
 * share the one array, so calls on different streams that can run at the same
 * time race and give wrong results; issue them on one stream.
 */
int bf16_linear_noalloc(const void *x, const void *W, const void *bias, void *out,
                        int M, int N, int K, bf16l_stream_t stream);

/* Size in bytes of the fixed scratch array behind bf16_linear_noalloc. */
size_t bf16_linear_noalloc_scratch_bytes(void);

/*
 * ---- Per-tensor FP8 (e4m3) ----
 *
 * Source: the sglang PR #28333 page, "关键源码片段": apply_fp8_linear_bmm_flashinfer
 * quantises the input with a given per-tensor scale (static_quant_fp8), multiplies
 * the e4m3 operands with per-tensor x_scale and weight_scale (bmm_fp8) and adds
 * bias; the quantisation kernel forms 1 / scale and stores clamp(y * (1 / scale),
 * -448, 448) as e4m3.
 *
 * bf16_quant_fp8 — static quantisation of n bf16 values x to e4m3 codes xq:
 *   xq[i] = e4m3_rne(clamp(float(x[i]) * (1.0f / *scale), -448, 448)),
 *   the reciprocal and the product in binary32.  scale: device pointer to one
 *   fp32 (read on the device, after the programmatic-launch wait when `flags`
 *   has BF16L_FLAG_PDL).  x 2-byte aligned (16-byte alignment of x and xq takes
 *   the vector path), xq must not overlap x.  Asynchronous; BF16L_EINVAL for a
 *   negative n, NULL pointers or unknown flags; BF16L_EALIGN.
 *
 * bf16_linear_fp8 — out[M,N] (bf16) =
 *   bf16_rne(*scale_x * *scale_w * sum_k e4m3(xq[m,k]) e4m3(wq[n,k]) (+ bias[n]))
 *   with fp32 accumulation; bias (bf16, may be NULL) enters before the one
 *   rounding.  xq[M,K] and wq[N,K] are row-major e4m3 codes (one byte each),
 *   K % 16 == 0 (16-byte rows, else BF16L_EUNSUPPORTED); all data pointers
 *   16-byte aligned (BF16L_EALIGN); scale_x, scale_w device pointers to one fp32
 *   each.  Any M (groups of 16 tokens); launches one kernel (warp-level e4m3
 *   MMAs, K split over a cluster), allocates nothing.
 *
 * bf16_linear_fp8_with_plan — the same with an explicit plan: kernel
 *   BF16L_KERNEL_DOTMMA (threads 128 or 256, split_k 1/2/4/8/16, at most one
 *   64-code block per CTA; any M) or BF16L_KERNEL_WARPMMA (the persistent
 *   warp-MMA form: threads 256/512/1024, rows_per_cta = warps per 8-row group,
 *   stages = CTAs per SM, split_k 0; M <= 16 and M * K <= 200 KB) or
 *   BF16L_KERNEL_TILE (the tcgen05 kind::f8f6f4 tile form: threads 192,
 *   stages 2..4; any M), flags; threads == 0 means the entry point's own
 *   choice (the tile form for M > 16 with at least 32 tiles of 128 x 256, else
 *   the warp-MMA form for N >= 1024 when it applies, else the split form).
 *   BF16L_EINVAL for any other plan.
 *
 * bf16_linear_fp8_split — the K split bf16_linear_fp8 uses for a shape on a
 *   device with num_sms SMs (pure host logic; for tests and tuning).
 */
int bf16_quant_fp8(const void *x, const float *scale, void *xq, int64_t n, uint32_t flags, bf16l_stream_t stream);
int bf16_linear_fp8(const void *xq, const void *wq, const float *scale_x, const float *scale_w, const void *bias,
                    void *out, int M, int N, int K, uint32_t flags, bf16l_stream_t stream);
int bf16_linear_fp8_with_plan(const void *xq, const void *wq, const float *scale_x, const float *scale_w,
                              const void *bias, void *out, int M, int N, int K, const bf16l_plan *plan,
                              bf16l_stream_t stream);
int bf16_linear_fp8_split(int M, int N, int K, int num_sms);

/*
 * bf16_linear_probe_read — a measurement probe, not part of the linear layer
 * (no counterpart on the pages).  Launches `grid` CTAs of `threads` threads
 * that read the `bytes` bytes at `src` once, with the 16-byte loads the
 * weight-streaming kernels use; CTA b XORs every 32-bit word it read into
 * sink[b] (sink: device uint32[grid], zeroed by the caller if it wants the
 * checksum, which is then the XOR of the grid words).  Nothing else is
 * computed, so its time for a W-sized buffer is the floor of any kernel that
 * must read that weight, launched the same way: by default as the library's
 * kernels are (programmatic dependent launch, each CTA's share prefetched into
 * L2 before the grid-dependency wait), serially with BF16L_FLAG_SERIAL (the
 * only flag it takes).  With bytes == 0 it is an empty launch (src and sink
 * may then be NULL), whose time in a graph of back-to-back launches is the
 * per-call launch cost.  bytes % 16 == 0, src 16-byte aligned, sink 4-byte
 * aligned, 1 <= grid, threads a multiple of 32 in 32..1024.  Asynchronous;
 * returns BF16L_OK, BF16L_EINVAL, BF16L_EALIGN, BF16L_EARCH or BF16L_ELAUNCH.
 */
int bf16_linear_probe_read(const void *src, size_t bytes, int grid, int threads, uint32_t *sink, uint32_t flags,
                           bf16l_stream_t stream);

/*
 * ---- MXFP8: block-scaled e4m3 ----
 *
 * Source: the sglang PR #34042 page ("执行摘要", "实现拆解" items 2-3): the dense
 * MXFP8 GEMM on SM10x (weights with block scales, activations quantised the
 * same way), whose small-batch decode kernels the page reports 2-5x faster.
 * The page does not spell the format out; it is read as the OCP
 * microscaling MXFP8 format: each run of 32 consecutive elements along K
 * shares one E8M0 scale byte e (value 2^(e - 127)), the elements are e4m3
 * codes (as for the per-tensor FP8 entry points).  Scales are row-major
 * [rows][K / 32] bytes (no swizzle).
 *
 * bf16_quant_mxfp8 — quantise x[rows][K] (bf16, K % 32 == 0) into codes
 *   xq[rows][K] and scales xs[rows][K / 32]: per block, s = floor(log2(max
 *   |v|)) - 8 clamped below at -127 (an all-zero block gets s = -127),
 *   xs = s + 127, xq = e4m3 of v * 2^-s rounded to nearest even, saturating
 *   at +-448.  x and xq 16-byte aligned; no two buffers may overlap.
 *   Asynchronous; BF16L_EINVAL (sizes, NULL, flags, overlap), BF16L_EALIGN,
 *   BF16L_EUNSUPPORTED (K % 32 != 0), BF16L_EARCH, BF16L_ELAUNCH.
 *
 * bf16_linear_mxfp8 — out[M][N] (bf16) = RNE_bf16( sum over blocks b of
 *   2^(xs[m][b]-127) * 2^(ws[n][b]-127) * sum_{k in b} e4m3(xq[m][k])
 *   e4m3(wq[n][k]) (+ bias[n]) ), fp32 accumulation, bias before the one
 *   rounding.  xq[M][K], wq[N][K] codes and xs[M][K/32], ws[N][K/32] scales
 *   as above; K % 32 == 0 (else BF16L_EUNSUPPORTED); xq, wq, out and bias
 *   16-byte aligned; out must not overlap the inputs.  Any M.  Small M:
 *   warp-level e4m3 MMAs, one per scale block, K split over a cluster, in
 *   groups of 16 tokens.  M > 16 with at least 32 tiles of 128 x 256 and
 *   K % 128 == 0: the tcgen05 tile form (256 W rows per tile, a three-stage
 *   ring), one block-scaled MMA
 *   (kind::mxf8f6f4.block_scale) per scale block with the scales staged into
 *   tensor memory (xs and ws 4-byte aligned, else BF16L_EALIGN).  Launches one
 *   kernel, allocates nothing.  Block-scale products 2^(xs+ws-254) outside
 *   the fp32 range are not supported by the warp-level form (quantised data
 *   stays far inside it).
 *
 * bf16_linear_mxfp8_with_plan — the same with an explicit plan: kernel
 *   BF16L_KERNEL_DOTMMA (the warp-level form: threads 128 or 256, split_k 1,
 *   2, 4, 8 or 16, at most K / 32) or BF16L_KERNEL_TILE (the tile form:
 *   threads 320, rows_per_cta = W rows per tile, 128 or 256, stages 2..6
 *   for 128 and 2..4 for 256, split_k = raster group of W tiles, 0 = 8;
 *   K % 128 == 0, else BF16L_EUNSUPPORTED), flags; threads == 0 means the
 *   entry point's own choice.  BF16L_EINVAL for any other plan.
 *
 * bf16_linear_mxfp8_split — the K split the entry point uses with `threads`
 *   threads per CTA on a device with num_sms SMs (pure host logic).
 */
int bf16_quant_mxfp8(const void *x, int64_t rows, int K, void *xq, void *xs, uint32_t flags, bf16l_stream_t stream);
int bf16_linear_mxfp8(const void *xq, const void *xs, const void *wq, const void *ws, const void *bias, void *out,
                      int M, int N, int K, uint32_t flags, bf16l_stream_t stream);
int bf16_linear_mxfp8_with_plan(const void *xq, const void *xs, const void *wq, const void *ws, const void *bias,
                                void *out, int M, int N, int K, const bf16l_plan *plan, bf16l_stream_t stream);
int bf16_linear_mxfp8_split(int M, int N, int K, int threads, int num_sms);

/* Human-readable name of a status code (static string, never NULL). */
const char *bf16_linear_strerror(int status);

/* The last CUDA error code seen by the library on this host thread (0 if none). */
int bf16_linear_cuda_error(void);

/* Library version, as major * 10000 + minor * 100 + patch. */
int bf16_linear_version(void);

#ifdef __cplusplus
}
#endif

#endif /* BF16_LINEAR_H */
