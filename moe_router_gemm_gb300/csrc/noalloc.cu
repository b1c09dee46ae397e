// noalloc.cu — bf16_linear_noalloc: the linear layer for callers that cannot
// allocate device memory.
//
// Who needs this: code that is handed device buffers for its inputs and
// outputs but has no way to obtain scratch of its own — a plug-in inside an
// inference engine whose memory is reserved up front by the host program, a
// component that must not touch the global allocator while other work owns
// the device memory budget, or any caller for whom cudaMalloc is simply not
// available.  Such callers cannot provide the workspace that the cluster-free
// split-K kernel (BF16L_KERNEL_SPLITK_WS) reduces through.
//
// What it does instead: the scratch lives in a fixed-size array that is part
// of this library's device image (`g_noalloc_scratch` below, kNoAllocBytes).
// Every GPU that loads the library holds that memory until the process exits.
// No call here allocates or frees anything.  The first call on a device looks
// up the array's device address (cudaGetSymbolAddress, with that device
// current) and keeps it; make that first call before any stream capture.
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

// The scratch array: 4 MiB, enough for the arrival counters plus the fp32
// partial tiles of one call (see bf16_linear_noalloc for the shapes that fit).
// In host code this name is only a stand-in for the device symbol, never a
// device address: the address comes from cudaGetSymbolAddress in
// noalloc_scratch().
#define BF16L_NOALLOC_BYTES (4u << 20)
static __device__ __align__(256) uint8_t g_noalloc_scratch[BF16L_NOALLOC_BYTES];

namespace bf16l {

namespace {

constexpr size_t kNoAllocBytes = BF16L_NOALLOC_BYTES;
constexpr int kNoAllocMaxDevices = 64;

struct NoAllocDevice {
    std::mutex mu;
    void *scratch = nullptr;  // set once the lookup has succeeded; never cleared
};
NoAllocDevice g_noalloc_devices[kNoAllocMaxDevices];

// The array's device address on the current device, looked up on first use.
// Only a successful lookup is kept: a failed one (for example, made during a
// stream capture) is reported and retried on the next call.  Returns a
// cudaError_t value.
int noalloc_scratch(int device, void **out) {
    NoAllocDevice &d = g_noalloc_devices[device];
    std::lock_guard<std::mutex> lock(d.mu);
    if (!d.scratch) {
        void *p = nullptr;
        const int e = (int)cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e) {
            (void)cudaGetLastError();  // leave no sticky error behind for the caller's next check
            return e;
        }
        d.scratch = p;
    }
    *out = d.scratch;
    return 0;
}

int ceil_div(int a, int b) { return (a + b - 1) / b; }

}  // namespace

}  // namespace bf16l

/*
 * See bf16_linear.h.  Runs the cluster-free split-K kernel with a plan sized to
 * the device and shrunk (fewer K splits) until its scratch fits the fixed
 * array; shapes that do not fit even unsplit return BF16L_ENOSCRATCH.
 */
extern "C" int bf16_linear_noalloc(const void *x, const void *W, const void *bias, void *out, int M, int N, int K,
                                   bf16l_stream_t stream) {
    using namespace bf16l;
    if (M < 0 || N <= 0 || K <= 0) return BF16L_EINVAL;
    if (M == 0) return BF16L_OK;
    if (!x || !W || !out) return BF16L_EINVAL;
    const uintptr_t align = reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(W) |
                            reinterpret_cast<uintptr_t>(out) | reinterpret_cast<uintptr_t>(bias);
    if (align & 15u) return BF16L_EALIGN;
    if (M > kSplitMaxTokens || K % 8 != 0) return BF16L_EUNSUPPORTED;

    // The device check of every entry point (compute capability 10.3, kernel
    // attributes set) comes before anything else touches the device.
    bf16l_device dev = {};
    const int st = current_device_checked(&dev);
    if (st != BF16L_OK) return st;
    int device = 0;
    int e = (int)cudaGetDevice(&device);
    if (e) {
        note_cuda_error(e);
        return BF16L_ELAUNCH;
    }
    if (device < 0 || device >= kNoAllocMaxDevices) return BF16L_ELAUNCH;
    void *scratch = nullptr;
    e = noalloc_scratch(device, &scratch);
    if (e) {
        note_cuda_error(e);
        return BF16L_ELAUNCH;
    }

    // Plan: tokens on the MMA M side, 64 weight rows per CTA (128 for large N),
    // about one CTA per SM, then as few K splits as needed to fit the array.
    bf16l_plan p = {};
    p.kernel = BF16L_KERNEL_SPLITK_WS;
    p.threads = kSplitThreads;
    p.rows_per_cta = N <= 512 ? 64 : 128;
    p.tokens_per_cta = ((M + 7) / 8) * 8;
    const int tiles = ceil_div(N, p.rows_per_cta);
    const int chunks = ceil_div(K, kChunkK);
    int split = dev.num_sms / tiles;
    if (split < 1) split = 1;
    if (split > kSplitWsMaxSplit) split = kSplitWsMaxSplit;
    if (split > chunks) split = chunks;
    for (;; --split) {
        p.split_k = split;
        const int per_cta = ceil_div(chunks, split);
        const int max_stages = split_max_stages(p.tokens_per_cta, p.rows_per_cta);
        p.stages = per_cta < max_stages ? per_cta : max_stages;
        if (bf16_linear_workspace_size(M, N, K, &p) <= kNoAllocBytes) break;
        if (split == 1) return BF16L_ENOSCRATCH;
    }

    // The array keeps the last call's contents; the arrival counters must
    // start at zero, so clear them (stream-ordered, nothing allocated).
    e = (int)cudaMemsetAsync(scratch, 0, split_ws_counter_bytes(tiles), (cudaStream_t)stream);
    if (e) {
        note_cuda_error(e);
        return BF16L_ELAUNCH;
    }

    bf16l_call c = {};
    c.x = x;
    c.W = W;
    c.bias = bias;
    c.out = out;
    c.M = M;
    c.N = N;
    c.K = K;
    c.plan = &p;
    c.workspace = scratch;
    c.workspace_bytes = kNoAllocBytes;
    c.stream = stream;
    return bf16_linear_run(&c);
}

extern "C" size_t bf16_linear_noalloc_scratch_bytes(void) { return bf16l::kNoAllocBytes; }
