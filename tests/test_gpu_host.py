"""GPU parity of bf16_linear_host: host buffers in and out, copies and kernel on the caller's stream.

The result must equal the device entry point's (the same plan on the same bits)
and the oracle within tolerance; page-locked and pageable host memory both
work; a side stream is honoured; a staging buffer that is too small or not
256-byte aligned is rejected before anything is enqueued.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tolerance import check_close, tensor_bits

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.mark.parametrize("shape", [(16, 384, 7168, False), (4, 2112, 7168, True), (64, 2112, 7168, False),
                                   (300, 1000, 520, True), (3, 7, 16, True)], ids=lambda s: "x".join(map(str, s)))
def test_host_entry_matches_device_entry_and_oracle(lib, shape):
    M, N, K, bias = shape
    x, W, b = wl.make_inputs(M, N, K, M + N, bias)
    hx, hW = x.pin_memory(), W.pin_memory()
    hb = b.pin_memory() if b is not None else None
    st = lib.new_host_staging(M, N, K, bias, device=DEV)
    out = lib.bf16_linear_host(hx, hW, hb, staging=st)
    torch.cuda.synchronize()
    dev = lib.bf16_linear(x.to(DEV), W.to(DEV), b.to(DEV) if b is not None else None)
    torch.cuda.synchronize()
    assert np.array_equal(tensor_bits(out), tensor_bits(dev))
    rows = np.unique(np.array([0, M // 2, M - 1]))
    check_close(tensor_bits(out)[rows], oracle.linear_bf16(wl.bits(x)[rows], wl.bits(W), wl.bits(b)), f"host {shape}")


def test_host_entry_pageable_and_side_stream(lib):
    M, N, K = 8, 2112, 4096
    x, W, _ = wl.make_inputs(M, N, K, 3, False)
    st = lib.new_host_staging(M, N, K, False, device=DEV)
    s = torch.cuda.Stream(DEV)
    out = torch.empty(M, N, dtype=torch.bfloat16)  # pageable
    lib.bf16_linear_host(x, W, None, out, staging=st, stream=s)
    s.synchronize()
    want = lib.bf16_linear(x.to(DEV), W.to(DEV))
    torch.cuda.synchronize()
    assert np.array_equal(tensor_bits(out), tensor_bits(want))


def test_host_entry_rejects(lib):
    M, N, K = 4, 256, 2048
    x, W, _ = wl.make_inputs(M, N, K, 1, False)
    need = lib.host_staging_bytes(M, N, K, False)
    small = torch.empty(need - 256, dtype=torch.uint8, device=DEV)
    with pytest.raises(lib.BF16LinearError):
        lib.bf16_linear_host(x, W, staging=small)
    big = torch.empty(need + 512, dtype=torch.uint8, device=DEV)
    with pytest.raises(lib.BF16LinearError):
        lib.bf16_linear_host(x, W, staging=big[16:])  # 16 bytes past a 256-byte boundary
    empty = lib.bf16_linear_host(torch.empty(0, K, dtype=torch.bfloat16), W, staging=big)
    assert tuple(empty.shape) == (0, N)
