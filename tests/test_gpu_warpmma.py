"""GPU parity of the warp-level tensor-core kernel (BF16L_KERNEL_WARPMMA) against the oracle.

Groups of 1..16 warps own 8 W rows at a time and feed 16-byte weight loads to
mma.sync.m16n8k16 with the tokens on the MMA's 16 rows.  The cases cover every
group size and block size, N not a multiple of 8 and smaller than the grid, K
tails inside a 32-wide block and inside a lane batch, M = 1..16 (tokens 8..15 in
the MMA's upper rows), bias on and off, the decode and MLP shapes, and the fp32
epilogue (which must round to the bf16 result of the same plan bit for bit).
Results for one plan are bitwise reproducible.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tolerance import check_close, tensor_bits

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

CFGS = [(128, 4, 8), (128, 1, 8), (512, 1, 2), (512, 2, 2), (512, 4, 2), (512, 16, 1), (1024, 1, 1), (1024, 4, 1), (1024, 8, 1),
        (256, 1, 4), (256, 8, 4)]
SHAPES = [(1, 300, 1032), (3, 517, 2880), (8, 64, 4096), (5, 1000, 136), (2, 5, 64), (16, 203, 1024),
          (12, 96, 2056), (9, 1, 40)]


def _plan(lib, threads=512, wpr=1, cps=1, xr=0):
    return lib.make_plan("warpmma", threads=threads, rows_per_cta=wpr, stages=cps, split_k=xr)


def _fits(M, K, cfg):
    static = (32 * 32 * 4 * 4 if cfg[1] > 1 else 512) + 1024
    return cfg[2] * (M * K * 2 + static) <= 232448


def _run(lib, x, W, b, plan, f32=False):
    xd, Wd = x.to(DEV), W.to(DEV)
    bd = b.to(DEV) if b is not None else None
    out = (lib.bf16_linear_f32out(xd, Wd, bd, plan_=plan) if f32
           else lib.bf16_linear_with_plan(xd, Wd, bd, plan_=plan))
    torch.cuda.synchronize()
    return out


def _check(lib, M, N, K, seed, bias, plan):
    x, W, b = wl.make_inputs(M, N, K, seed, bias)
    got = tensor_bits(_run(lib, x, W, b, plan))
    want = oracle.linear_bf16(wl.bits(x), wl.bits(W), wl.bits(b))
    check_close(got, want, f"warpmma M={M} N={N} K={K} bias={bias} plan={plan}")
    return got


@pytest.mark.parametrize("cfg", CFGS, ids=lambda c: "t%d_wpr%d_cps%d" % c)
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_warpmma_forced(lib, shape, cfg):
    M, N, K = shape
    if not _fits(M, K, cfg):
        with pytest.raises(lib.BF16LinearError):
            lib.plan_check(M, N, K, _plan(lib, *cfg))
        return
    for bias in (False, True):
        _check(lib, M, N, K, seed=M + N + K, bias=bias, plan=_plan(lib, *cfg))


XR_CFGS = [(512, 1, 1), (512, 4, 1), (512, 16, 1), (256, 2, 2), (256, 8, 2)]


@pytest.mark.parametrize("cfg", XR_CFGS, ids=lambda c: "xreg_t%d_wpr%d_cps%d" % c)
@pytest.mark.parametrize("shape", SHAPES + [(16, 333, 7168)], ids=lambda s: "x".join(map(str, s)))
def test_warpmma_x_from_l2(lib, shape, cfg):
    """x fragments loaded from L2 with each weight batch (no shared-memory x): any K, M <= 16."""
    M, N, K = shape
    for bias in (False, True):
        _check(lib, M, N, K, seed=M + N + K + 1, bias=bias, plan=_plan(lib, *cfg, xr=1))


@pytest.mark.parametrize("ng", [2, 4])
@pytest.mark.parametrize("cfg", XR_CFGS + [(128, 4, 4)], ids=lambda c: "t%d_wpr%d_cps%d" % c)
@pytest.mark.parametrize("shape", SHAPES + [(16, 333, 7168), (13, 2112, 7168)], ids=lambda s: "x".join(map(str, s)))
def test_warpmma_groups_per_warp(lib, shape, cfg, ng):
    """x from L2, each x fragment feeding 2 or 4 8-row groups (16 or 32 W rows per warp, slabs past N ragged)."""
    M, N, K = shape
    p = _plan(lib, *cfg, xr=1)
    p.tokens_per_cta = ng
    for bias in (False, True):
        _check(lib, M, N, K, seed=M + N + K + 2, bias=bias, plan=p)


def test_warpmma_groups_per_warp_f32_and_pdl(lib):
    # the fp32 epilogue rounds to the bf16 result of the same plan; the launch flag changes nothing
    M, N, K = 14, 1000, 3000
    x, W, b = wl.make_inputs(M, N, K, 6, True)
    for ng in (2, 4):
        p = _plan(lib, 256, 8, 2, 1)
        p.tokens_per_cta = ng
        a = tensor_bits(_run(lib, x, W, b, p))
        f = _run(lib, x, W, b, p, f32=True)
        assert np.array_equal(tensor_bits(f.to(torch.bfloat16)), a)
        p.flags = lib.FLAG_PDL
        assert np.array_equal(tensor_bits(_run(lib, x, W, b, p)), a)


def test_warpmma_x_paths_agree(lib):
    # the same fragments reach the same MMAs in the same order from shared memory or from L2, one
    # or two 8-row groups per warp: the same bits
    x, W, b = wl.make_inputs(12, 2112, 4096, 4, True)
    a = tensor_bits(_run(lib, x, W, b, _plan(lib, 512, 4, 1, 0)))
    assert np.array_equal(a, tensor_bits(_run(lib, x, W, b, _plan(lib, 512, 4, 1, 1))))
    for ng in (2, 4):
        p = _plan(lib, 512, 4, 1, 1)
        p.tokens_per_cta = ng
        assert np.array_equal(a, tensor_bits(_run(lib, x, W, b, p)))


@pytest.mark.parametrize("M", [9, 16])
def test_warpmma_decode_16_tokens(lib, M):
    # 9..16 tokens of K = 7168 (> 115 KB) can still fit, 16 do not: the L2 path takes any
    if M * 7168 * 2 > 200 * 1024:
        with pytest.raises(lib.BF16LinearError):
            lib.plan_check(M, 2112, 7168, _plan(lib, 512, 4, 1, 0))
    _check(lib, M, 2112, 7168, seed=77, bias=False, plan=_plan(lib, 512, 4, 1, 1))


@pytest.mark.parametrize("M", [1, 2, 4, 8])
def test_warpmma_decode_shape(lib, M):
    _check(lib, M, 2112, 7168, seed=60 + M, bias=False, plan=_plan(lib, 512, 4, 2 if M <= 4 else 1))


@pytest.mark.parametrize("M", [8, 16])
def test_warpmma_mlp_shape(lib, M):
    _check(lib, M, 14336, 4096, seed=8 + M, bias=True, plan=_plan(lib, 1024, 4, 1))


def test_warpmma_deterministic_and_f32(lib):
    M, N, K = 11, 1500, 3000
    x, W, b = wl.make_inputs(M, N, K, 2, True)
    p = _plan(lib, 512, 4, 1)
    a = tensor_bits(_run(lib, x, W, b, p))
    assert np.array_equal(a, tensor_bits(_run(lib, x, W, b, p)))
    f = _run(lib, x, W, b, p, f32=True)
    assert np.array_equal(tensor_bits(f.to(torch.bfloat16)), a)
    assert lib.device_status() == 0


def test_warpmma_exact_cases(lib):
    M, N, K = 16, 700, 2048
    _, W, b = wl.make_inputs(M, N, K, 3, True)
    ks = np.random.default_rng(5).integers(0, K, M)
    x = torch.zeros(M, K, dtype=torch.bfloat16)
    x[torch.arange(M), torch.from_numpy(ks)] = 1.0
    p = _plan(lib, 512, 2, 1)
    assert torch.equal(_run(lib, x, W, None, p).cpu(), W[:, torch.from_numpy(ks)].T.contiguous())
    assert torch.equal(_run(lib, torch.zeros_like(x), W, b, p).cpu(), b.expand(M, N))
    ones = _run(lib, torch.ones(M, K, dtype=torch.bfloat16), torch.ones(N, K, dtype=torch.bfloat16), None, p)
    assert (ones.cpu().float() == float(K)).all()


def test_warpmma_pdl_matches(lib):
    M, N, K = 8, 2112, 7168
    x, W, b = wl.make_inputs(M, N, K, 9, False)
    p = _plan(lib, 512, 4, 1)
    ref = tensor_bits(_run(lib, x, W, None, p))
    p.flags = lib.FLAG_PDL
    xd, Wd = x.to(DEV), W.to(DEV)
    outs = [lib.bf16_linear_with_plan(xd, Wd, None, plan_=p) for _ in range(3)]
    torch.cuda.synchronize()
    for o in outs:
        assert np.array_equal(tensor_bits(o), ref)
