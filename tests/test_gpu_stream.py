"""The persistent weight-streaming kernel (BF16L_KERNEL_STREAM) against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tolerance import check_close, tensor_bits

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def stream_plan(lib, rows, stages):
    return lib.make_plan("stream", threads=288, rows_per_cta=rows, stages=stages)


CASES = [
    # M, N, K, rows per stage, stages
    (1, 2112, 7168, 2, 8),
    (4, 2112, 7168, 1, 12),
    (2, 14336, 4096, 4, 6),       # many row groups per CTA: the ring wraps
    (3, 256, 7168, 4, 4),         # fewer rows than CTAs x rows: short and empty CTAs
    (1, 5, 8, 1, 1),              # N < SM count: one row per CTA
    (4, 1000, 8192, 2, 6),        # the largest K the kernel takes
    (2, 777, 1032, 2, 3),         # ragged row ranges, K not a multiple of 64
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_stream_parity(lib, case):
    M, N, K, rows, stages = case
    p = stream_plan(lib, rows, stages)
    for bias in (False, True):
        x, W, b = wl.make_inputs(M, N, K, M + N + K, bias)
        xd, Wd = x.to(DEV), W.to(DEV)
        bd = b.to(DEV) if b is not None else None
        got = [tensor_bits(lib.run(xd, Wd, bd, plan_=p)) for _ in range(2)]
        torch.cuda.synchronize()
        check_close(got[0], oracle.linear_bf16(wl.bits(x), wl.bits(W), wl.bits(b)), f"stream {case} bias={bias}")
        assert np.array_equal(got[0], got[1])
        o32 = lib.run(xd, Wd, bd, plan_=p, out_f32=True)
        assert torch.equal(o32.to(torch.bfloat16).cpu(), torch.from_numpy(got[0].view(np.int16)).view(torch.bfloat16))


def test_stream_exact_and_limits(lib):
    M, N, K = 3, 500, 4096
    p = stream_plan(lib, 2, 6)
    _, W, b = wl.make_inputs(M, N, K, 1, True)
    ks = np.random.default_rng(3).integers(0, K, M)
    x = torch.zeros(M, K, dtype=torch.bfloat16)
    x[torch.arange(M), torch.from_numpy(ks)] = 1.0
    assert np.array_equal(tensor_bits(lib.run(x.to(DEV), W.to(DEV), plan_=p)), wl.bits(W)[:, ks].T)
    z = lib.run(torch.zeros_like(x).to(DEV), W.to(DEV), b.to(DEV), plan_=p)
    assert np.array_equal(tensor_bits(z), np.broadcast_to(wl.bits(b), (M, N)))
    with pytest.raises(lib.BF16LinearError) as e:    # more tokens than the kernel holds in registers
        lib.run(torch.randn(5, K, device=DEV).to(torch.bfloat16), W.to(DEV), plan_=p)
    assert e.value.status == -6
    with pytest.raises(lib.BF16LinearError) as e:    # K beyond 8192
        lib.run(torch.randn(1, 8200, device=DEV).to(torch.bfloat16),
                torch.randn(16, 8200, device=DEV).to(torch.bfloat16), plan_=p)
    assert e.value.status == -6
