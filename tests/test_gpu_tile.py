"""GPU parity of the 1-CTA tcgen05 tile kernel (BF16L_KERNEL_TILE), forced, against the oracle.

The tile is 128 x rows by 256 W rows, K in 64-wide chunks through a 2..4-deep
ring, persistent over the tiles.  The cases put the tails where the dispatcher's
prefill shapes never do: M below one tile and one row past a tile (x rows past M
are TMA zero fill), N not a multiple of 256, K not a multiple of 64 (the last
chunk's columns past K are zero fill on both operands), a ring deeper than the
chunk count, and more tiles than SMs (CTAs that take a second tile reuse the
double-buffered accumulator).  Each runs with bias on and off; large shapes are
checked on sampled rows covering the first, middle and last row of every
128-row tile.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tolerance import check_close, tensor_bits

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _plan(lib, stages=4):
    return lib.make_plan("tile", threads=192, rows_per_cta=256, tokens_per_cta=128, stages=stages)


def _rows(M):
    rows = set()
    for m0 in range(0, M, 128):
        rows.update({m0, min(m0 + 64, M - 1), min(m0 + 127, M - 1)})
    return sorted(r for r in rows if r < M)


CASES = [
    # M, N, K, stages
    (130, 300, 520, 2),      # M one tile plus two rows, N tail of 44, K = 8 chunks + 8
    (1000, 700, 136, 3),     # ragged M, N and K; three chunks on a three-deep ring
    (129, 257, 72, 2),       # one row and one W row past a tile; K = one chunk + 8
    (384, 2112, 2056, 4),    # N = 8.25 tiles, K = 32 chunks + 8, ring wraps
    (77, 130, 8, 4),         # K = 8: one partial chunk, ring deeper than the chunk count
    (64, 1000, 4096, 4),     # half a tile of rows, K a multiple of 64
    (1100, 5000, 200, 3),    # 9 x 20 = 180 tiles on 152 SMs: some CTAs take two
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_tile_forced_ragged(lib, case):
    M, N, K, st = case
    plan = _plan(lib, st)
    sampled = M * N * K > 2e9
    for bias in (False, True):
        x, W, b = wl.make_inputs(M, N, K, M + N + K + st + bias, bias)
        out = lib.bf16_linear_with_plan(x.to(DEV), W.to(DEV), b.to(DEV) if b is not None else None, plan_=plan)
        torch.cuda.synchronize()
        got = tensor_bits(out)
        if sampled:
            rows = _rows(M)
            want = oracle.linear_rows_bf16(wl.bits(x), wl.bits(W), wl.bits(b), np.array(rows, dtype=np.int64))
            check_close(got[rows], want, f"tile M={M} N={N} K={K} bias={bias} rows={len(rows)}")
        else:
            want = oracle.linear_bf16(wl.bits(x), wl.bits(W), wl.bits(b))
            check_close(got, want, f"tile M={M} N={N} K={K} stages={st} bias={bias}")
    assert lib.device_status() == 0


def test_tile_ragged_stage_depths_agree(lib):
    """The ring depth changes scheduling, not the per-tile MMA order: every depth gives the same bits."""
    M, N, K = 130, 300, 520
    x, W, b = wl.make_inputs(M, N, K, 5, True)
    xd, Wd, bd = x.to(DEV), W.to(DEV), b.to(DEV)
    outs = [tensor_bits(lib.bf16_linear_with_plan(xd, Wd, bd, plan_=_plan(lib, s))) for s in (2, 3, 4)]
    torch.cuda.synchronize()
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_tile_ragged_f32_logits(lib):
    """The fp32 epilogue of the same forced plan on a ragged shape: within the fp32 bound of the
    oracle's unrounded value, and rounding it to bf16 reproduces the bf16 epilogue bit for bit."""
    M, N, K = 129, 257, 72
    x, W, b = wl.make_inputs(M, N, K, 11, True)
    xd, Wd, bd = x.to(DEV), W.to(DEV), b.to(DEV)
    f32 = lib.bf16_linear_f32out(xd, Wd, bd, plan_=_plan(lib, 2))
    bf = lib.bf16_linear_with_plan(xd, Wd, bd, plan_=_plan(lib, 2))
    torch.cuda.synchronize()
    assert np.array_equal(tensor_bits(f32.to(torch.bfloat16)), tensor_bits(bf))
    exact = oracle.linear_f64(wl.bits(x), wl.bits(W), wl.bits(b))
    got = f32.double().cpu().numpy()
    # |fp32 sum - exact| <= K * 2^-24 * sum_k |x_k w_k| (+ the bias term): a loose, always-valid bound
    xf, Wf = x.double().numpy(), W.double().numpy()
    mag = np.abs(xf) @ np.abs(Wf).T + np.abs(b.double().numpy())[None, :]
    assert np.all(np.abs(got - exact) <= (K + 2) * 2.0 ** -24 * mag + 1e-30)


# ---- the tactic space: tile widths, ring depths, raster groups, and the swap-AB form ----

WIDTH_CASES = [
    # BN (W rows per tile), M, N, K, stages, raster group
    (128, 130, 300, 520, 7, 0),
    (192, 1000, 700, 136, 5, 1),
    (224, 129, 2112, 2056, 4, 3),
    (240, 384, 2112, 1032, 4, 16),
    (256, 300, 1000, 200, 2, 1),
]


@pytest.mark.parametrize("case", WIDTH_CASES, ids=lambda c: "x".join(map(str, c)))
def test_tile_widths(lib, case):
    """Every plain-form width, with ragged M, N and K, against the oracle; the raster group only
    reorders tiles, so it must not change a bit (checked against group 0)."""
    bn, M, N, K, st, grp = case
    plan = lib.make_plan("tile", threads=192, rows_per_cta=bn, tokens_per_cta=128, stages=st, split_k=grp)
    base = lib.make_plan("tile", threads=192, rows_per_cta=bn, tokens_per_cta=128, stages=2, split_k=0)
    for bias in (False, True):
        x, W, b = wl.make_inputs(M, N, K, bn + M + bias, bias)
        xd, Wd, bd = x.to(DEV), W.to(DEV), (b.to(DEV) if b is not None else None)
        got = tensor_bits(lib.bf16_linear_with_plan(xd, Wd, bd, plan_=plan))
        ref = tensor_bits(lib.bf16_linear_with_plan(xd, Wd, bd, plan_=base))
        torch.cuda.synchronize()
        check_close(got, oracle.linear_bf16(wl.bits(x), wl.bits(W), wl.bits(b)),
                    f"tile BN={bn} M={M} N={N} K={K} stages={st} group={grp} bias={bias}")
        assert np.array_equal(got, ref)
    assert lib.device_status() == 0


SWAP_CASES = [
    # BN (tokens per tile), M, N, K, stages, raster group
    (32, 17, 300, 520, 8, 0),       # one partial token tile, N tail inside a W tile, K tail
    (64, 64, 2112, 7168, 8, 0),     # decode M = 64: one token tile, 16.5 W tiles
    (64, 100, 1000, 136, 6, 1),     # two token tiles (the second partial), raster one token tile at a time
    (128, 200, 257, 72, 5, 0),      # one W row past a tile
    (192, 256, 14336, 1024, 5, 0),  # MLP-like N: 112 W tiles, 2 token tiles, more tiles than SMs
    (256, 256, 520, 4096, 4, 0),    # MLP M = 256 in one token tile
    (256, 40, 384, 2880, 3, 2),     # tokens far fewer than the tile: TMA zero fill past M
]


@pytest.mark.parametrize("case", SWAP_CASES, ids=lambda c: "x".join(map(str, c)))
def test_tile_swap_ab(lib, case):
    """The swap-AB form (W rows on the MMA M side, tokens on N) against the oracle, bias on and off;
    its fp32 epilogue rounds to its bf16 epilogue bit for bit."""
    bn, M, N, K, st, grp = case
    plan = lib.make_plan("tile_t", threads=192, rows_per_cta=128, tokens_per_cta=bn, stages=st, split_k=grp)
    sampled = M * N * K > 2e9
    for bias in (False, True):
        x, W, b = wl.make_inputs(M, N, K, 3 * bn + M + bias, bias)
        xd, Wd, bd = x.to(DEV), W.to(DEV), (b.to(DEV) if b is not None else None)
        out = lib.bf16_linear_with_plan(xd, Wd, bd, plan_=plan)
        f32 = lib.bf16_linear_f32out(xd, Wd, bd, plan_=plan)
        torch.cuda.synchronize()
        got = tensor_bits(out)
        assert np.array_equal(tensor_bits(f32.to(torch.bfloat16)), got)
        if sampled:
            rows = sorted({0, M // 2, M - 1})
            want = oracle.linear_rows_bf16(wl.bits(x), wl.bits(W), wl.bits(b), np.array(rows, dtype=np.int64))
            check_close(got[rows], want, f"tile_t BN={bn} M={M} N={N} K={K} rows={rows}")
        else:
            check_close(got, oracle.linear_bf16(wl.bits(x), wl.bits(W), wl.bits(b)),
                        f"tile_t BN={bn} M={M} N={N} K={K} stages={st} bias={bias}")
    assert lib.device_status() == 0


def test_tile_swap_ab_exact_cases(lib):
    """One-hot token rows reproduce W^T bit for bit and x = 0 gives the bias, through the transposed
    epilogue (a swapped index would put W[n, k] at the wrong output)."""
    M, N, K = 48, 320, 256
    plan = lib.make_plan("tile_t", threads=192, rows_per_cta=128, tokens_per_cta=64, stages=4)
    _, W, b = wl.make_inputs(1, N, K, 9, True)
    x = torch.zeros(M, K, dtype=torch.bfloat16)
    ks = [(7 * m + 3) % K for m in range(M)]
    for m, k in enumerate(ks):
        x[m, k] = 1.0
    out = tensor_bits(lib.bf16_linear_with_plan(x.to(DEV), W.to(DEV), None, plan_=plan))
    want = tensor_bits(W[:, ks].t().contiguous())
    assert np.array_equal(out, want)
    zero = tensor_bits(lib.bf16_linear_with_plan(torch.zeros(M, K, dtype=torch.bfloat16, device=DEV), W.to(DEV),
                                                 b.to(DEV), plan_=plan))
    assert np.array_equal(zero, np.broadcast_to(tensor_bits(b), (M, N)))
