// tile_t.cu — the swap-AB orientation of the tcgen05 tile GEMM (tile.cuh): 128
// W rows (MMA M) by BN tokens (MMA N) per tile, for mid-size M (tens to a few
// hundred tokens) where a 128-token tile would be mostly padding.
#include "tile.cuh"

namespace bf16l {

int init_tile_t() {
    int e = 0;
    if (!e) e = tile_set_attr<32, true, uint16_t>();
    if (!e) e = tile_set_attr<64, true, uint16_t>();
    if (!e) e = tile_set_attr<128, true, uint16_t>();
    if (!e) e = tile_set_attr<192, true, uint16_t>();
    if (!e) e = tile_set_attr<256, true, uint16_t>();
    if (!e) e = tile_set_attr<32, true, float>();
    if (!e) e = tile_set_attr<64, true, float>();
    if (!e) e = tile_set_attr<128, true, float>();
    if (!e) e = tile_set_attr<192, true, float>();
    if (!e) e = tile_set_attr<256, true, float>();
    return e;
}

template <typename OutT>
static int launch_swap_t(const LaunchArgs &a, const bf16l_plan &p) {
    switch (p.tokens_per_cta) {
        case 32: return tile_launch_bn<32, true, OutT>(a, p);
        case 64: return tile_launch_bn<64, true, OutT>(a, p);
        case 128: return tile_launch_bn<128, true, OutT>(a, p);
        case 192: return tile_launch_bn<192, true, OutT>(a, p);
        case 256: return tile_launch_bn<256, true, OutT>(a, p);
        default: return (int)cudaErrorInvalidValue;
    }
}

int launch_tile_swap(const LaunchArgs &a, const bf16l_plan &p) {
    return a.out_f32 ? launch_swap_t<float>(a, p) : launch_swap_t<uint16_t>(a, p);
}

}  // namespace bf16l
