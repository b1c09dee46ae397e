"""Seeded synthetic inputs and the workload shapes, shared by tests and bench.

This module holds no arithmetic of the method: it only draws random inputs
(and names the shapes).  Both the CUDA path and the CPU oracle consume what it
produces, as torch bf16 tensors or as their uint16 bit patterns.

Recipe (same for every workload):
  x    ~ N(0, 1)          drawn in fp32, cast to bf16   shape [M, K], row-major
  W    ~ N(0, 1/K)        drawn in fp32, cast to bf16   shape [N, K], row-major (nn.Linear layout)
  bias ~ U(-0.1, 0.1)     drawn in fp32, cast to bf16   shape [N]   (only where a workload has bias)
drawn in that order from one ``torch.Generator`` seeded per shape.

Shapes are those of the serving linear layers the pages discuss: MoE router
gates (N = 128..384 experts, hidden K = 2048..7168; vLLM PR #42562 and #48774
pages), the DeepSeek attention-input projection (N = 1536 + 512 + 64 = 2112;
sglang PR #30117 page, prepare_qkv_latent), a dense MLP projection and
prefill-size contractions.
"""
from __future__ import annotations

import numpy as np
import torch

# (K, N) pairs of the MoE router sweep; K = 2880 is the non-tile-aligned case
# the vLLM PR #42562 tests call out.
ROUTER_KN = [(4096, 256), (6144, 256), (7168, 256), (7168, 384), (2880, 128)]
ROUTER_M = list(range(1, 17))

DECODE_M = [1, 2, 4, 8, 16, 32, 64]
DECODE_KN = (7168, 2112)

MLP_M = [1, 8, 64, 256]
MLP_KN = (4096, 14336)

PREFILL_M = [2048, 8192]
PREFILL_KN = [(7168, 2112), (4096, 14336), (7168, 7168)]


def router_smallest():
    """Smallest router case: M=4, K=2048, N=256, no bias, seed 0."""
    return [dict(name="router_smallest", M=4, K=2048, N=256, bias=False, seed=0)]


def router_sweep():
    """MoE router sweep: M = 1..16 x five (K, N) pairs, no bias (80 points)."""
    pts = []
    for i, (K, N) in enumerate(ROUTER_KN):
        for M in ROUTER_M:
            pts.append(dict(name=f"router_K{K}_N{N}_M{M}", M=M, K=K, N=N, bias=False,
                            seed=1000 + 100 * i + M))
    return pts


def decode_proj():
    """Decode attention-input projection: K=7168, N=2112, no bias."""
    K, N = DECODE_KN
    return [dict(name=f"decode_M{M}", M=M, K=K, N=N, bias=False, seed=2000 + M)
            for M in DECODE_M]


def mlp_bias():
    """Dense MLP linear with bias: K=4096, N=14336."""
    K, N = MLP_KN
    return [dict(name=f"mlp_M{M}", M=M, K=K, N=N, bias=True, seed=3000 + M)
            for M in MLP_M]


def prefill():
    """Prefill-size contractions, bias on and off."""
    pts = []
    for i, (K, N) in enumerate(PREFILL_KN):
        for M in PREFILL_M:
            for b in (False, True):
                pts.append(dict(name=f"prefill_K{K}_N{N}_M{M}_{'bias' if b else 'nobias'}",
                                M=M, K=K, N=N, bias=b, seed=4000 + 100 * i + M // 1024 + (50 if b else 0)))
    return pts


def make_inputs(M: int, N: int, K: int, seed: int, bias: bool = False):
    """Draw (x, W, bias_or_None) as CPU bf16 tensors, contiguous row-major."""
    g = torch.Generator().manual_seed(int(seed))
    x = torch.randn(M, K, generator=g, dtype=torch.float32).to(torch.bfloat16)
    W = (torch.randn(N, K, generator=g, dtype=torch.float32) * (K ** -0.5)).to(torch.bfloat16)
    b = None
    if bias:
        b = (torch.rand(N, generator=g, dtype=torch.float32) * 0.2 - 0.1).to(torch.bfloat16)
    return x.contiguous(), W.contiguous(), (b.contiguous() if b is not None else None)


def bits(t: torch.Tensor | None) -> np.ndarray | None:
    """uint16 bit patterns of a CPU bf16 tensor (no copy of the values' meaning)."""
    if t is None:
        return None
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def from_bits(a: np.ndarray) -> torch.Tensor:
    """CPU bf16 tensor with the given uint16 bit patterns."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).view(torch.bfloat16)
