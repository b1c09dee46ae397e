"""GPU parity of the cluster form of the warp-MMA kernel (WARPMMA plans with split_k >= 2).

K is split over S = 2..16 CTAs of a cluster; each stages its K slice of up to 64
tokens (1 to 4 tiles of 16 on the MMA rows) and the partial tiles of every
8-row group are summed, in rank order, by the rank that finishes the group.
The cases cover every group size, 256/512/1024-thread blocks, one and two CTAs
per SM, S from 2 to 16 (a non-portable cluster size above 8), K runs that end inside a 32-wide block or leave a rank a
single block, N not a multiple of 8 and smaller than the cluster count, M from
1 to 64 (ragged last tile, 3 tiles on the 4-tile instance), bias on and off,
the decode and MLP shapes (sampled rows at M = 64 of the MLP weight), the fp32
epilogue, bitwise reproducibility and the programmatic-launch flag.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tolerance import check_close, tensor_bits

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

# (threads, warps per 8-row group, CTAs per SM, cluster size)
CFGS = [(1024, 8, 1, 2), (1024, 4, 1, 4), (1024, 16, 1, 2), (512, 4, 1, 8), (512, 1, 1, 2), (256, 2, 2, 4),
        (512, 16, 1, 3), (256, 8, 1, 8), (256, 2, 4, 16), (128, 2, 8, 4)]
SHAPES = [(1, 300, 1032), (3, 517, 2880), (16, 203, 1024), (12, 96, 2056), (9, 1, 40), (20, 1000, 2048),
          (33, 77, 4096), (64, 130, 1024), (48, 2112, 512), (17, 2112, 7168)]


def _plan(lib, threads, wpr, cps, S):
    return lib.make_plan("warpmma", threads=threads, rows_per_cta=wpr, stages=cps, split_k=S)


def _valid(lib, M, N, K, p):
    try:
        lib.plan_check(M, N, K, p)
        return True
    except lib.BF16LinearError:
        return False


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
    xb = wl.bits(x) if rows is None else wl.bits(x)[rows]
    want = oracle.linear_bf16(xb, wl.bits(W), wl.bits(b))
    check_close(got if rows is None else got[rows], want, f"warpmma cluster M={M} N={N} K={K} bias={bias} plan={plan}")
    return got


@pytest.mark.parametrize("cfg", CFGS, ids=lambda c: "t%d_wpr%d_cps%d_S%d" % c)
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_warpmma_cluster_forced(lib, shape, cfg):
    M, N, K = shape
    p = _plan(lib, *cfg)
    if not _valid(lib, M, N, K, p):
        pytest.skip("plan outside the form's limits (checked on the CPU)")
    for bias in (False, True):
        _check(lib, M, N, K, seed=M + N + K + cfg[3], bias=bias, plan=p)
    assert lib.device_status() == 0


@pytest.mark.parametrize("M", [4, 8, 16, 32, 64])
def test_warpmma_cluster_decode_shape(lib, M):
    p = _plan(lib, 1024, 8, 1, 2) if M <= 16 else _plan(lib, 512, 4, 1, 8)
    _check(lib, M, 2112, 7168, seed=90 + M, bias=False, plan=p)


def test_warpmma_cluster_mlp_sampled(lib):
    rows = np.array([0, 1, 15, 16, 30, 31])
    _check(lib, 32, 14336, 4096, seed=64, bias=True, plan=_plan(lib, 512, 4, 1, 4), rows=rows)
    # 64 tokens: the receive slots for 48 row groups per cluster (96 KB) and the x slice do not fit
    with pytest.raises(lib.BF16LinearError):
        lib.plan_check(64, 14336, 4096, _plan(lib, 512, 4, 1, 4))


@pytest.mark.parametrize("gpc", [1, 2, 3, 5])
def test_warpmma_cluster_groups_per_cluster(lib, gpc):
    # fewer clusters, each CTA's x slice serving several row groups (more groups than warp groups too)
    p = _plan(lib, 256, 2, 4, 8)
    p.tokens_per_cta = gpc
    for M, N, K in ((16, 256, 7168), (7, 384, 4096), (13, 203, 2880)):
        _check(lib, M, N, K, seed=gpc + M, bias=True, plan=p)


def test_warpmma_cluster_agrees_across_forms(lib):
    # the same K slices in another cluster size give another summation order: both within tolerance,
    # each bitwise reproducible
    M, N, K = 13, 1500, 3000
    x, W, b = wl.make_inputs(M, N, K, 2, True)
    want = oracle.linear_bf16(wl.bits(x), wl.bits(W), wl.bits(b))
    for p in (_plan(lib, 1024, 8, 1, 2), _plan(lib, 512, 2, 1, 4)):
        a = tensor_bits(_run(lib, x, W, b, p))
        check_close(a, want, f"plan={p}")
        assert np.array_equal(a, tensor_bits(_run(lib, x, W, b, p)))
        f = _run(lib, x, W, b, p, f32=True)
        assert np.array_equal(tensor_bits(f.to(torch.bfloat16)), a)
    assert lib.device_status() == 0


def test_warpmma_cluster_exact_cases(lib):
    M, N, K = 40, 700, 2048
    _, W, b = wl.make_inputs(M, N, K, 3, True)
    ks = np.random.default_rng(5).integers(0, K, M)
    x = torch.zeros(M, K, dtype=torch.bfloat16)
    x[torch.arange(M), torch.from_numpy(ks)] = 1.0
    p = _plan(lib, 512, 2, 1, 4)
    assert torch.equal(_run(lib, x, W, None, p).cpu(), W[:, torch.from_numpy(ks)].T.contiguous())
    assert torch.equal(_run(lib, torch.zeros_like(x), W, b, p).cpu(), b.expand(M, N))
    ones = _run(lib, torch.ones(M, K, dtype=torch.bfloat16), torch.ones(N, K, dtype=torch.bfloat16), None, p)
    assert (ones.cpu().float() == float(K)).all()


def test_warpmma_cluster_pdl_matches(lib):
    M, N, K = 16, 2112, 7168
    x, W, _ = wl.make_inputs(M, N, K, 9, False)
    p = _plan(lib, 1024, 8, 1, 2)
    ref = tensor_bits(_run(lib, x, W, None, p))
    p.flags = lib.FLAG_PDL
    xd, Wd = x.to(DEV), W.to(DEV)
    outs = [lib.bf16_linear_with_plan(xd, Wd, None, plan_=p) for _ in range(3)]
    torch.cuda.synchronize()
    for o in outs:
        assert np.array_equal(tensor_bits(o), ref)
