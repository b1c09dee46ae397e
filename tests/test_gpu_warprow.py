"""GPU parity of the warp-per-row kernel (BF16L_KERNEL_WARPROW) against the oracle.

The kernel is persistent: CTA b owns a contiguous range of W rows and groups of
1, 2 or 4 warps compute one row at a time.  The cases cover every group size
and block size, CTAs that own no row at all (N smaller than the grid), K tails
inside a lane batch, bias on and off, M = 1..8, the decode and MLP shapes, and
the fp32 epilogue (which must round to the bf16 result of the same plan bit for
bit).  Results for one plan are bitwise reproducible.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tolerance import check_close, tensor_bits

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _plan(lib, threads=512, wpr=1, cps=1):
    return lib.make_plan("warprow", threads=threads, rows_per_cta=wpr, stages=cps)


def _run(lib, x, W, b, plan, f32=False):
    xd, Wd = x.to(DEV), W.to(DEV)
    bd = b.to(DEV) if b is not None else None
    out = (lib.bf16_linear_f32out(xd, Wd, bd, plan_=plan) if f32
           else lib.bf16_linear_with_plan(xd, Wd, bd, plan_=plan))
    torch.cuda.synchronize()
    return out


def _check(lib, M, N, K, seed, bias, plan, rows=None):
    x, W, b = wl.make_inputs(M, N, K, seed, bias)
    got = tensor_bits(_run(lib, x, W, b, plan))
    want = oracle.linear_bf16(wl.bits(x), wl.bits(W), wl.bits(b))
    check_close(got, want, f"warprow M={M} N={N} K={K} bias={bias} plan={plan}")
    return x, W, b, got


@pytest.mark.parametrize("cfg", [(512, 1, 1), (512, 2, 1), (512, 4, 1), (1024, 1, 1), (1024, 4, 1),
                                 (256, 1, 4), (256, 2, 2), (512, 2, 2), (128, 1, 8), (128, 4, 8)],
                         ids=lambda c: "t%d_wpr%d_cps%d" % c)
@pytest.mark.parametrize("shape", [(1, 300, 1032), (3, 517, 2880), (8, 64, 4096), (5, 1000, 136), (2, 5, 64)],
                         ids=lambda s: "x".join(map(str, s)))
def test_warprow_forced(lib, shape, cfg):
    M, N, K = shape
    if cfg[2] * (M * K * 2 + 2048) > 232448:
        # the planner refuses a ring of CTAs whose staged x does not fit one SM
        with pytest.raises(lib.BF16LinearError):
            lib.plan_check(M, N, K, _plan(lib, *cfg))
        return
    for bias in (False, True):
        _check(lib, M, N, K, seed=M + N + K, bias=bias, plan=_plan(lib, *cfg))


@pytest.mark.parametrize("M", [1, 2, 4, 8])
def test_warprow_decode_shape(lib, M):
    _check(lib, M, 2112, 7168, seed=40 + M, bias=False, plan=_plan(lib, 512, 2, 2 if M <= 4 else 1))


def test_warprow_mlp_shape(lib):
    _check(lib, 8, 14336, 4096, seed=7, bias=True, plan=_plan(lib, 1024, 1, 1))


def test_warprow_deterministic_and_f32(lib):
    M, N, K = 4, 1500, 3000
    x, W, b = wl.make_inputs(M, N, K, 2, True)
    p = _plan(lib, 512, 4, 2)
    a = tensor_bits(_run(lib, x, W, b, p))
    assert np.array_equal(a, tensor_bits(_run(lib, x, W, b, p)))
    f = _run(lib, x, W, b, p, f32=True)
    assert np.array_equal(tensor_bits(f.to(torch.bfloat16)), a)
    assert lib.device_status() == 0


def test_warprow_exact_cases(lib):
    M, N, K = 6, 700, 2048
    _, W, b = wl.make_inputs(M, N, K, 3, True)
    ks = np.random.default_rng(5).integers(0, K, M)
    x = torch.zeros(M, K, dtype=torch.bfloat16)
    x[torch.arange(M), torch.from_numpy(ks)] = 1.0
    p = _plan(lib, 512, 2, 1)
    assert torch.equal(_run(lib, x, W, None, p).cpu(), W[:, torch.from_numpy(ks)].T.contiguous())
    assert torch.equal(_run(lib, torch.zeros_like(x), W, b, p).cpu(), b.expand(M, N))
    ones = _run(lib, torch.ones(M, K, dtype=torch.bfloat16), torch.ones(N, K, dtype=torch.bfloat16), None, p)
    assert (ones.cpu().float() == float(K)).all()


def test_warprow_pdl_matches(lib):
    M, N, K = 4, 2112, 7168
    x, W, b = wl.make_inputs(M, N, K, 9, False)
    p = _plan(lib, 512, 2, 2)
    ref = tensor_bits(_run(lib, x, W, None, p))
    p.flags = lib.FLAG_PDL
    xd, Wd = x.to(DEV), W.to(DEV)
    outs = [lib.bf16_linear_with_plan(xd, Wd, None, plan_=p) for _ in range(3)]
    torch.cuda.synchronize()
    for o in outs:
        assert np.array_equal(tensor_bits(o), ref)
