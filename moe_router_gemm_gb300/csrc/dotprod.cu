// dotprod.cu — bf16-output instances of the dot-product kernel (dotprod.cuh)
// and the dispatch between the bf16 and fp32-output launchers.
#include "dotprod.cuh"

namespace bf16l {

int init_dotprod() { return dot_detail::init_dotprod_t<uint16_t>(); }

int launch_dotprod(const LaunchArgs &a, const bf16l_plan &p) {
    return a.out_f32 ? launch_dotprod_f32(a, p) : dot_detail::launch_dotprod_t<uint16_t>(a, p);
}

}  // namespace bf16l
