"""torch's F.linear (cuBLAS) beside the library, on one shape of every workload: a comparator, not the gate.

The gate is the oracle (the same element-wise bound as every parity test).  cuBLAS
sums in its own order and may round its fp32 result differently, so the two GPU
results are only expected to agree to about one bf16 ulp; the test reports the
largest ulp distance between them, the share of elements that differ, and each
one's largest error against the oracle (as test properties and on stdout), so
that a regression shows up beside a known library.  The only assertion on the
comparator is that it runs and is finite.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import workloads as wl
from tolerance import bits_to_f64, check_close, tensor_bits

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

CASES = [
    # M, N, K, bias: router, decode, MLP (bias), and a prefill shape checked on sampled rows
    (16, 256, 7168, False),
    (8, 2112, 7168, False),
    (64, 14336, 4096, True),
    (2048, 2112, 7168, True),
]


def _ordered(bits):
    """bf16 bit patterns -> integers that are ordered like the values (for ulp distances)."""
    b = np.asarray(bits, dtype=np.int32)
    return np.where(b & 0x8000, 0x8000 - b, b)


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_against_cublas(lib, case, record_property):
    M, N, K, bias = case
    x, W, b = wl.make_inputs(M, N, K, 11 + M + N, bias)
    xd, Wd, bd = x.to(DEV), W.to(DEV), (b.to(DEV) if b is not None else None)
    ours = tensor_bits(lib.bf16_linear(xd, Wd, bd))
    ref = tensor_bits(F.linear(xd, Wd, bd))
    torch.cuda.synchronize()
    assert np.isfinite(bits_to_f64(ref)).all()
    rows = np.arange(M) if M * N * K <= 2e9 else np.unique(np.r_[0:M:128, 127:M:128, M - 1])
    want = (oracle.linear_bf16(wl.bits(x), wl.bits(W), wl.bits(b)) if len(rows) == M else
            oracle.linear_rows_bf16(wl.bits(x), wl.bits(W), wl.bits(b), rows.astype(np.int64)))
    err_ours = check_close(ours[rows], want, f"library {case}")  # the gate
    o = bits_to_f64(want)
    err_cublas = float(np.abs(bits_to_f64(ref[rows]) - o).max())
    ulps = np.abs(_ordered(ours[rows]) - _ordered(ref[rows]))
    stats = {"max_ulp_vs_cublas": int(ulps.max()), "share_differing": float((ulps > 0).mean()),
             "max_err_library": err_ours, "max_err_cublas": err_cublas}
    for k, v in stats.items():
        record_property(k, v)
    print(f"{case}: {stats}")
