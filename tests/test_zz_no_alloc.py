"""bf16_linear_noalloc: the entry point for callers that cannot allocate device memory.

Some callers get their input and output buffers from a host program that owns
all device memory (a plug-in inside an inference engine, say) and have no way
to obtain a workspace of their own.  bf16_linear_noalloc gives them the
workspace split-K kernel with its scratch in the library's fixed device array.
These tests call it through the C ABI and check its output against the CPU
oracle on calls in a row (and, as an extra check, against the regular
bf16_linear entry point), including a shape whose plan must take fewer K
splits to fit the array, and that a shape too large for the array is refused
with its own error code.

This file sorts last so that a run stopping at the first failure has already
run every other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tolerance import check_close, tensor_bits

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _noalloc(lib, x, W, b, out):
    L = lib.load()
    return L.bf16_linear_noalloc(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(W.data_ptr()),
                                 ctypes.c_void_p(b.data_ptr()) if b is not None else None,
                                 ctypes.c_void_p(out.data_ptr()), x.shape[0], W.shape[0], x.shape[1],
                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _split_needed(M, N, K, lib):
    """K splits of the workspace split-K plan the entry point starts from (about one CTA per SM), and
    whether its partial tiles overflow the 4 MiB array there, so that the plan has to shrink."""
    rows = 64 if N <= 512 else 128
    tiles = -(-N // rows)
    split = min(152 // tiles, -(-K // 64), 64)
    p = lib.make_plan("splitk_ws", threads=128, rows_per_cta=rows, tokens_per_cta=-(-M // 8) * 8, split_k=split,
                      stages=1)
    return split, lib.workspace_size(M, N, K, p) > lib.load().bf16_linear_noalloc_scratch_bytes()


def test_noalloc_matches_oracle_on_calls_in_a_row(lib):
    assert lib.load().bf16_linear_noalloc_scratch_bytes() == 4 << 20
    # the last shape starts at 8 K splits (about 4.46 MB of partials) and must drop to 7 to fit
    split, overflow = _split_needed(64, 2112, 7168, lib)
    assert split == 8 and overflow
    cases = [(16, 384, 7168, False, 1), (9, 2112, 7168, True, 2), (64, 2112, 7168, True, 3)]
    # consecutive calls of different shapes: each reuses the array the previous one left behind
    for (M, N, K, bias, seed) in cases:
        x, W, b = wl.make_inputs(M, N, K, seed, bias)
        xd, Wd = x.to(DEV), W.to(DEV)
        bd = b.to(DEV) if b is not None else None
        out = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
        assert _noalloc(lib, xd, Wd, bd, out) == 0
        ref = lib.bf16_linear(xd, Wd, bd)
        torch.cuda.synchronize()
        want = oracle.linear_bf16(wl.bits(x), wl.bits(W), wl.bits(b))
        check_close(tensor_bits(out), want, f"noalloc vs oracle M={M} N={N} K={K} bias={bias}")
        check_close(tensor_bits(out), tensor_bits(ref), f"noalloc vs bf16_linear M={M} N={N} K={K}")
    # and the same shape twice more: bit-identical through the shared array
    for _ in range(2):
        out2 = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
        assert _noalloc(lib, xd, Wd, bd, out2) == 0
        torch.cuda.synchronize()
        assert np.array_equal(tensor_bits(out2), tensor_bits(out))


def test_noalloc_refuses_what_does_not_fit(lib):
    # M * N * 4 bytes of unsplit partials exceed the 4 MiB array
    M, N, K = 64, 40000, 1024
    x = torch.randn(M, K, device=DEV).to(torch.bfloat16)
    W = torch.randn(N, K, device=DEV).to(torch.bfloat16)
    out = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    assert _noalloc(lib, x, W, None, out) == -7
    assert "scratch" in lib.strerror(-7)
    # shapes outside the kernel's limits are refused, not sent elsewhere
    x2 = torch.randn(65, K, device=DEV).to(torch.bfloat16)
    assert _noalloc(lib, x2, W[:8].contiguous(), None, torch.empty(65, 8, dtype=torch.bfloat16, device=DEV)) == -6
