"""bf16_linear_noalloc: the entry point for callers that cannot allocate device memory.

Some callers get their input and output buffers from a host program that owns
all device memory (a plug-in inside an inference engine, say) and have no way
to obtain a workspace of their own.  bf16_linear_noalloc gives them the
workspace split-K kernel with its scratch in the library's fixed device array.
These tests call it through the C ABI and check that two calls in a row agree
with the regular bf16_linear entry point, within the parity tolerance, and that
a shape too large for the fixed array is refused with its own error code.

This file sorts last so that a run stopping at the first failure has already
run every other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

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


def test_noalloc_matches_bf16_linear_twice_in_a_row(lib):
    assert lib.load().bf16_linear_noalloc_scratch_bytes() == 4 << 20
    # two calls in a row: different shapes, so the second reuses the array the first left behind
    for (M, N, K, bias, seed) in [(16, 384, 7168, False, 1), (9, 2112, 7168, True, 2)]:
        x, W, b = wl.make_inputs(M, N, K, seed, bias)
        xd, Wd = x.to(DEV), W.to(DEV)
        bd = b.to(DEV) if b is not None else None
        out = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
        assert _noalloc(lib, xd, Wd, bd, out) == 0
        ref = lib.bf16_linear(xd, Wd, bd)
        torch.cuda.synchronize()
        check_close(tensor_bits(out), tensor_bits(ref), f"noalloc vs bf16_linear M={M} N={N} K={K}")
    # and the same shape again: deterministic through the shared array
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
