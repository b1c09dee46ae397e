// tile.cu — the plain orientation of the tcgen05 tile GEMM (tile.cuh): 128 x
// rows (MMA M) by BN W rows (MMA N) per tile, for large M; and its e4m3 form.
#include "tile.cuh"

namespace bf16l {

int tile_smem_bytes(int stages, int bn) { return tile_smem_bytes_bn(stages, bn); }

int init_tile() {
    int e = 0;
    if (!e) e = tile_set_attr<128, false, uint16_t>();
    if (!e) e = tile_set_attr<192, false, uint16_t>();
    if (!e) e = tile_set_attr<224, false, uint16_t>();
    if (!e) e = tile_set_attr<240, false, uint16_t>();
    if (!e) e = tile_set_attr<256, false, uint16_t>();
    if (!e) e = tile_set_attr<128, false, float>();
    if (!e) e = tile_set_attr<192, false, float>();
    if (!e) e = tile_set_attr<224, false, float>();
    if (!e) e = tile_set_attr<240, false, float>();
    if (!e) e = tile_set_attr<256, false, float>();
    if (!e)
        e = (int)cudaFuncSetAttribute(tile_kernel<256, false, uint16_t, true>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      tile_smem_bytes_bn(tile_max_stages(256), 256));
    if (!e) e = init_tile_t();
    return e;
}

template <typename OutT>
static int launch_tile_t(const LaunchArgs &a, const bf16l_plan &p) {
    switch (p.rows_per_cta) {
        case 128: return tile_launch_bn<128, false, OutT>(a, p);
        case 192: return tile_launch_bn<192, false, OutT>(a, p);
        case 224: return tile_launch_bn<224, false, OutT>(a, p);
        case 240: return tile_launch_bn<240, false, OutT>(a, p);
        case 256: return tile_launch_bn<256, false, OutT>(a, p);
        default: return (int)cudaErrorInvalidValue;
    }
}

int launch_tile(const LaunchArgs &a, const bf16l_plan &p) {
    if (p.kernel == BF16L_KERNEL_TILE_T) return launch_tile_swap(a, p);
    return a.out_f32 ? launch_tile_t<float>(a, p) : launch_tile_t<uint16_t>(a, p);
}

int launch_tile_fp8(const void *xq, const void *wq, const float *sx, const float *sw, const void *bias, void *out,
                    int M, int N, int K, int stages, int grid, uint32_t flags, void *stream, int32_t *status) {
    CUtensorMap tx, tw;  // 128-byte rows of 128 codes, as the bf16 form's 64 values
    int r = make_tmap_u8_2d(&tx, xq, (uint64_t)M, (uint64_t)K, kTileBP, 2 * kChunkK, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    if (r) return (int)cudaErrorInvalidValue;
    r = make_tmap_u8_2d(&tw, wq, (uint64_t)N, (uint64_t)K, kTileBN, 2 * kChunkK, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    if (r) return (int)cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kTileThreads);
    cfg.dynamicSmemBytes = (size_t)tile_smem_bytes_bn(stages, kTileBN);
    cfg.stream = (cudaStream_t)stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl_attr_of(flags);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return (int)cudaLaunchKernelEx(&cfg, tile_kernel<256, false, uint16_t, true>, tx, tw,
                                   static_cast<const uint16_t *>(bias), static_cast<uint16_t *>(out), M, N, K, stages,
                                   kTileDefaultGroup, status, sx, sw);
}

}  // namespace bf16l
