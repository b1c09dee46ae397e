"""GPU parity of the CTA-pair tile kernel (BF16L_KERNEL_TILE2) against the oracle.

A pair tile is 256 x rows by 256 W rows; each CTA of the pair stages half of
each operand and the even CTA issues the pair MMAs.  The cases span one pair
tile, a pair whose odd half lies wholly past M (its A rows are TMA zero fill),
ragged N and K, rings that wrap, persistent clusters taking several tiles, bias
on and off, and the fp32-logits epilogue (which must round to the bf16 output of
the same plan bit for bit).  Large shapes are checked on sampled rows that
include the first and last row of every 128-row half tile.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tolerance import check_close, tensor_bits

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _plan(lib, stages=4, bn=256):
    return lib.make_plan("tile2", threads=192, rows_per_cta=bn, tokens_per_cta=256, stages=stages)


def _run(lib, x, W, b, plan, f32=False):
    xd, Wd = x.to(DEV), W.to(DEV)
    bd = b.to(DEV) if b is not None else None
    if f32:
        out = lib.bf16_linear_f32out(xd, Wd, bd, plan_=plan)
    else:
        out = lib.bf16_linear_with_plan(xd, Wd, bd, plan_=plan)
    torch.cuda.synchronize()
    return out


def _rows(M):
    rows = set()
    for m0 in range(0, M, 128):
        rows.update({m0, min(m0 + 127, M - 1), min(m0 + 64, M - 1)})
    return sorted(r for r in rows if r < M)


def _check(lib, M, N, K, seed, bias, plan, sampled=False):
    x, W, b = wl.make_inputs(M, N, K, seed, bias)
    got = tensor_bits(_run(lib, x, W, b, plan))
    if sampled:
        rows = _rows(M)
        want = oracle.linear_rows_bf16(wl.bits(x), wl.bits(W), wl.bits(b), np.array(rows, dtype=np.int64))
        check_close(got[rows], want, f"tile2 M={M} N={N} K={K} rows={len(rows)}")
    else:
        want = oracle.linear_bf16(wl.bits(x), wl.bits(W), wl.bits(b))
        check_close(got, want, f"tile2 M={M} N={N} K={K} bias={bias}")
    return x, W, b, got


def test_tile2_one_pair_tile(lib):
    # the smallest case: one cluster, one tile, one K chunk
    for bias in (False, True):
        _check(lib, 256, 256, 64, seed=1, bias=bias, plan=_plan(lib, 2))
    assert lib.device_status() == 0


CASES = [
    # M, N, K, stages
    (256, 256, 1024, 4),     # ring wraps
    (130, 300, 520, 2),      # odd half of the pair wholly past M; K tail inside a chunk
    (384, 2112, 2880, 6),    # N tail (2112 = 8.25 x 256), K = 2880 (45 chunks)
    (1000, 700, 136, 3),     # ragged everything, 3 chunks on a 3-deep ring
    (512, 1024, 4096, 5),
    (129, 257, 72, 2),       # one row and one W row past a tile
]


@pytest.mark.parametrize("bn", [256, 192])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_tile2_forced(lib, case, bn):
    M, N, K, st = case
    for bias in (False, True):
        _check(lib, M, N, K, seed=M + N + K, bias=bias, plan=_plan(lib, st, bn))


def test_tile2_192_mlp_shape(lib):
    # the bandwidth-bound M = 256 MLP weight: 75 pair tiles of 256 x 192 (the last one 128 rows past N)
    _check(lib, 256, 14336, 4096, seed=13, bias=True, plan=_plan(lib, 6, 192), sampled=True)
    x, W, b = wl.make_inputs(200, 400, 1024, 14, True)
    a = tensor_bits(_run(lib, x, W, b, _plan(lib, 4, 192)))
    check_close(a, oracle.linear_bf16(wl.bits(x), wl.bits(W), wl.bits(b)), "tile2 192 ragged")
    f = _run(lib, x, W, b, _plan(lib, 4, 192), f32=True)
    assert np.array_equal(tensor_bits(f.to(torch.bfloat16)), a)


def test_tile2_persistent_many_tiles(lib):
    # more tiles than clusters: every cluster walks several 256 x 256 tiles
    _check(lib, 4096, 4864, 1024, seed=11, bias=True, plan=_plan(lib, 6), sampled=True)


def test_tile2_prefill_shape(lib):
    _check(lib, 2048, 7168, 7168, seed=12, bias=False, plan=_plan(lib, 6), sampled=True)


def test_tile2_deterministic_and_f32_epilogue(lib):
    M, N, K = 600, 520, 1032
    x, W, b = wl.make_inputs(M, N, K, 5, True)
    p = _plan(lib, 4)
    a = tensor_bits(_run(lib, x, W, b, p))
    assert np.array_equal(a, tensor_bits(_run(lib, x, W, b, p)))
    f = _run(lib, x, W, b, p, f32=True)
    assert np.array_equal(tensor_bits(f.to(torch.bfloat16)), a)


def test_tile2_exact_cases(lib):
    M, N, K = 300, 260, 640
    _, W, b = wl.make_inputs(M, N, K, 3, True)
    rng = np.random.default_rng(4)
    ks = rng.integers(0, K, M)
    x = torch.zeros(M, K, dtype=torch.bfloat16)
    x[torch.arange(M), torch.from_numpy(ks)] = 1.0
    p = _plan(lib, 3)
    out = _run(lib, x, W, None, p)
    assert torch.equal(out.cpu(), W[:, torch.from_numpy(ks)].T.contiguous()), "one-hot rows must copy W exactly"
    z = _run(lib, torch.zeros_like(x), W, b, p)
    assert torch.equal(z.cpu(), b.expand(M, N)), "x = 0 must give the bias"
    ones = _run(lib, torch.ones(M, K, dtype=torch.bfloat16), torch.ones(N, K, dtype=torch.bfloat16), None, p)
    assert (ones.cpu().float() == float(K)).all()
    assert lib.device_status() == 0


def test_tile2_pdl_matches(lib):
    M, N, K = 512, 768, 2048
    x, W, b = wl.make_inputs(M, N, K, 9, True)
    p = _plan(lib, 4)
    ref = tensor_bits(_run(lib, x, W, b, p))
    p.flags = lib.FLAG_PDL
    xd, Wd, bd = x.to(DEV), W.to(DEV), b.to(DEV)
    outs = [lib.bf16_linear_with_plan(xd, Wd, bd, plan_=p) for _ in range(3)]
    torch.cuda.synchronize()
    for o in outs:
        assert np.array_equal(tensor_bits(o), ref)
