// probe.cu — the read-floor probe: a kernel that only streams a buffer from
// memory with the same 16-byte loads the weight-streaming kernels use, and
// does no arithmetic beyond folding the words it read into one checksum.
//
// What it is for: the skinny linear layer's cost is reading W, so the time of
// a pure read of a W-sized buffer, launched the same way (back to back in a
// CUDA graph, rotated over copies larger than L2), is the floor no kernel of
// the library can go below for that weight.  It is launched as the library's
// kernels are (programmatic dependent launch, the buffer prefetched into L2
// before the grid-dependency wait), or serially on request.  With bytes == 0
// it is an empty launch: the per-call launch cost of a graph of back-to-back
// kernels.  The benchmark reports both beside its own numbers.
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

namespace bf16l {

namespace {

// Grid-stride loop over 16-byte vectors, four independent loads in flight per
// thread.  The XOR of every 32-bit word a CTA read is folded per warp, then
// across the CTA's warps, and XORed into the CTA's own word sink[blockIdx.x]
// by one thread (no two CTAs touch the same word, so the checksum costs no
// contended atomics; the loads cannot be removed, and a test can check them).
__global__ void __launch_bounds__(1024) read_probe_kernel(const uint4 *__restrict__ src, size_t nvec,
                                                          uint32_t *__restrict__ sink) {
    __shared__ uint32_t warp_acc[32];
    // Launched like the library's kernels: the CTA's share of the buffer is fetched into L2 while the
    // previous kernel finishes, and nothing is read before the grid-dependency wait (a no-op when the
    // launch is serial).
    if (threadIdx.x == 0 && nvec != 0) {
        const size_t v0 = nvec * blockIdx.x / gridDim.x, v1 = nvec * (blockIdx.x + 1) / gridDim.x;
        size_t bytes = (v1 - v0) * 16;
        const char *p = reinterpret_cast<const char *>(src + v0);
        while (bytes) {
            const uint32_t n = bytes < (1u << 30) ? (uint32_t)bytes : (1u << 30);
            prefetch_l2(p, n);
            p += n;
            bytes -= n;
        }
    }
    pdl_launch_dependents();
    pdl_wait();
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    uint32_t acc = 0;
    for (; i + 3 * stride < nvec; i += 4 * stride) {
        const uint4 a = ldg_stream_v4(src + i), b = ldg_stream_v4(src + i + stride);
        const uint4 c = ldg_stream_v4(src + i + 2 * stride), d = ldg_stream_v4(src + i + 3 * stride);
        acc ^= a.x ^ a.y ^ a.z ^ a.w ^ b.x ^ b.y ^ b.z ^ b.w ^ c.x ^ c.y ^ c.z ^ c.w ^ d.x ^ d.y ^ d.z ^ d.w;
    }
    for (; i < nvec; i += stride) {
        const uint4 a = ldg_stream_v4(src + i);
        acc ^= a.x ^ a.y ^ a.z ^ a.w;
    }
    if (nvec == 0) return;  // the empty launch
    for (int o = 16; o > 0; o >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, o);
    const int warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    if ((threadIdx.x & 31) == 0) warp_acc[warp] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t v = 0;
        for (int w = 0; w < nw; ++w) v ^= warp_acc[w];
        sink[blockIdx.x] ^= v;
    }
}

}  // namespace

}  // namespace bf16l

/* See bf16_linear.h. */
extern "C" int bf16_linear_probe_read(const void *src, size_t bytes, int grid, int threads, uint32_t *sink,
                                      uint32_t flags, bf16l_stream_t stream) {
    using namespace bf16l;
    if (grid < 1 || threads < 32 || threads > 1024 || threads % 32 != 0 || (bytes % 16) != 0) return BF16L_EINVAL;
    if (flags & ~BF16L_FLAG_SERIAL) return BF16L_EINVAL;
    if (bytes != 0 && (!src || !sink)) return BF16L_EINVAL;
    if ((reinterpret_cast<uintptr_t>(src) & 15u) || (reinterpret_cast<uintptr_t>(sink) & 3u)) return BF16L_EALIGN;
    bf16l_device dev = {};
    const int st = current_device_checked(&dev);
    if (st != BF16L_OK) return st;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)threads);
    cfg.stream = (cudaStream_t)stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl_attr_of(flags);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int e = (int)cudaLaunchKernelEx(&cfg, read_probe_kernel, static_cast<const uint4 *>(src), bytes / 16, sink);
    if (!e) e = (int)cudaGetLastError();
    if (e) {
        note_cuda_error(e);
        return BF16L_ELAUNCH;
    }
    return BF16L_OK;
}
