"""GPU parity of the fp32-logits variant (bf16_linear_f32out) against the oracle.

The oracle's result for this variant is the f64 sum rounded once to binary32
(oracle.linear_f32).  The kernels accumulate in fp32 in their own order, so
the bound is the classical worst case of a K-term fp32 sum,
    |gpu - oracle| <= (K + 2) * 2^-24 * sum_k |x_k w_k| + 2^-24 * |bias|,
computed per element from |x| @ |W|^T.  Exact cases (one-hot rows, all ones,
x = 0) must match bitwise, and for any plan the fp32 output rounded to bf16
must equal the bf16 output of the same plan bit for bit (one accumulation,
two epilogues).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _f32_bits(t):
    return t.detach().contiguous().cpu().numpy().view(np.uint32)


def _bf16_f64(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).double().numpy()


def _check_f32(lib, M, N, K, seed, bias, plan=None):
    x, W, b = wl.make_inputs(M, N, K, seed, bias)
    xd, Wd = x.to(DEV), W.to(DEV)
    bd = b.to(DEV) if b is not None else None
    out = lib.bf16_linear_f32out(xd, Wd, bd, plan_=plan)
    torch.cuda.synchronize()
    got = out.cpu().double().numpy()
    want = oracle.linear_f32(wl.bits(x), wl.bits(W), wl.bits(b)).view(np.float32).astype(np.float64)
    scale = np.abs(_bf16_f64(wl.bits(x))) @ np.abs(_bf16_f64(wl.bits(W))).T
    bound = (K + 2) * 2.0 ** -24 * scale + (2.0 ** -24 * np.abs(_bf16_f64(wl.bits(b)))[None, :] if bias else 0.0)
    bound = bound + 2.0 ** -24 * np.abs(want)
    bad = np.abs(got - want) > bound
    assert not bad.any(), f"{int(bad.sum())} fp32 outputs out of the summation bound (M={M} N={N} K={K})"
    return x, W, b, out


def _plans(lib, M):
    plans = [None, lib.make_plan("dotprod", threads=128, rows_per_cta=2)]
    if M <= 64:
        plans.append(lib.make_plan("splitk", threads=128, rows_per_cta=32, tokens_per_cta=max(8, -(-M // 8) * 8),
                                   split_k=4, stages=2))
    if M > 32:
        plans.append(lib.make_plan("tile", threads=192, rows_per_cta=256, tokens_per_cta=128, stages=4))
    return plans


@pytest.mark.parametrize("shape", [(1, 256, 7168), (4, 256, 2048), (16, 384, 7168), (9, 128, 2880),
                                   (64, 2112, 7168), (200, 520, 1024)], ids=lambda s: "x".join(map(str, s)))
def test_f32out_parity_and_same_accumulation(lib, shape):
    M, N, K = shape
    for plan in _plans(lib, M):
        x, W, b, out = _check_f32(lib, M, N, K, seed=M + N, bias=True, plan=plan)
        # same plan, bf16 epilogue: must be the fp32 result rounded to bf16, bit for bit
        xd, Wd, bd = x.to(DEV), W.to(DEV), b.to(DEV)
        ob = (lib.bf16_linear(xd, Wd, bd) if plan is None else lib.bf16_linear_with_plan(xd, Wd, bd, plan_=plan))
        torch.cuda.synchronize()
        assert torch.equal(out.to(torch.bfloat16).cpu(), ob.cpu()), f"epilogues disagree for plan {plan}"


def test_f32out_exact_cases(lib):
    M, N, K = 8, 300, 2048
    _, W, b = wl.make_inputs(M, N, K, 5, True)
    rng = np.random.default_rng(1)
    ks = rng.integers(0, K, M)
    x = torch.zeros(M, K, dtype=torch.bfloat16)
    x[torch.arange(M), torch.from_numpy(ks)] = 1.0
    for plan in _plans(lib, M):
        out = lib.bf16_linear_f32out(x.to(DEV), W.to(DEV), plan_=plan)
        want = W.float()[:, torch.from_numpy(ks)].T.contiguous()
        assert torch.equal(out.cpu(), want), f"one-hot not exact, plan {plan}"
        z = lib.bf16_linear_f32out(torch.zeros_like(x).to(DEV), W.to(DEV), b.to(DEV), plan_=plan)
        assert torch.equal(z.cpu(), b.float().expand(M, N)), f"x = 0 must give the bias, plan {plan}"
        ones = lib.bf16_linear_f32out(torch.ones(M, K, dtype=torch.bfloat16, device=DEV),
                                      torch.ones(N, K, dtype=torch.bfloat16, device=DEV), plan_=plan)
        assert (ones.cpu() == float(K)).all()


def test_f32out_rejects_bad_out(lib):
    x = torch.randn(4, 64, device=DEV).to(torch.bfloat16)
    W = torch.randn(8, 64, device=DEV).to(torch.bfloat16)
    with pytest.raises(ValueError):
        lib.bf16_linear_f32out(x, W, out=torch.empty(4, 8, dtype=torch.bfloat16, device=DEV))
