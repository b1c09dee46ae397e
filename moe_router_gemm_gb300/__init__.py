"""GB300-native skinny BF16 linear layer: out[M,N] = x[M,K] @ W[N,K]^T (+ bias[N]).

The product is the C-ABI library ``libbf16_linear.so`` (include/bf16_linear.h):
hand-written sm_103a kernels (CUDA-core dot product and weight streaming,
warp-level tensor-core kernels fed by 16-byte loads, tcgen05 cluster split-K
with a DSMEM reduction, 1-CTA (plain and swap-AB) and CTA-pair tcgen05
tile GEMMs) behind a
measured shape dispatcher, plus per-tensor FP8 and block-scaled MXFP8 paths.  This package is its thin Python binding; build the library with
``python -m moe_router_gemm_gb300.build``.
"""
from ._binding import (BF16LinearError, Call, Device, KERNEL_DOTPROD, KERNEL_NAMES, KERNEL_SPLITK,  # noqa: F401
                       KERNEL_SPLITK_WS, KERNEL_STREAM, KERNEL_TILE2, KERNEL_WARPROW,
                       KERNEL_WARPMMA, KERNEL_DOTMMA, KERNEL_DOTMMA_WS, KERNEL_TILE_T, new_workspace, plan_ws, run, workspace_size,
                       KERNEL_TILE, LIB_PATH, FLAG_PDL, FLAG_SERIAL, Plan, bf16_linear, bf16_linear_ex, bf16_linear_f32out,
                       bf16_linear_noalloc, bf16_linear_fp8, quant_fp8, fp8_split, quant_mxfp8, bf16_linear_mxfp8,
                       mxfp8_split, bf16_linear_host,
                       host_staging_bytes, new_host_staging,
                       bf16_linear_with_plan, device_status,
                       load, make_plan, plan, plan_check, probe_read, selftest_wait, strerror, version)
