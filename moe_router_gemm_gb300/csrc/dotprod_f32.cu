// dotprod_f32.cu — fp32-output (router logits) instances of the dot-product
// kernel in dotprod.cuh, in their own translation unit so both output types
// compile in parallel.
#include "dotprod.cuh"

namespace bf16l {

int init_dotprod_f32() { return dot_detail::init_dotprod_t<float>(); }

int launch_dotprod_f32(const LaunchArgs &a, const bf16l_plan &p) { return dot_detail::launch_dotprod_t<float>(a, p); }

}  // namespace bf16l
