"""GPU parity of two-chunk ring stages (chunks_per_stage = 2) in the tcgen05 ring kernels.

With two chunks per stage each operand arrives as one three-dimensional TMA box
holding two consecutive 64-wide K chunks, through the chunked view
{64, rows, K / 64} of the row-major matrix.  The cases put the ragged parts
where that view can go wrong: an odd chunk count (the second chunk of the last
stage lies past K and is TMA zero fill), rows past M or N (zero fill in the row
dimension), a single chunk, more tiles than SMs, and, for the split-K forms,
K splits whose ranks get one stage each or whose last stage is half fill.

The tile forms keep the MMA order of the one-chunk ring (chunk after chunk, four
K = 16 steps each), so their results must equal the one-chunk plan's bit for bit;
the split-K forms split K in units of two chunks, so they are checked against the
oracle.  Every case runs with bias on and off.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tolerance import check_close, tensor_bits

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _inputs(M, N, K, seed, bias):
    x, W, b = wl.make_inputs(M, N, K, seed, bias)
    return x, W, b, x.to(DEV), W.to(DEV), (b.to(DEV) if b is not None else None)


TILE_CASES = [
    # M, N, K, stages (of two chunks), W rows per tile
    (130, 300, 576, 2, 256),     # 9 chunks: the last stage's second chunk is fill; M and N tails
    (1000, 700, 128, 2, 192),    # one stage per tile
    (77, 130, 64, 2, 256),       # a single chunk: one stage, half fill
    (1100, 5000, 192, 2, 128),   # 9 x 40 = 360 tiles on 152 SMs; 3 chunks
    (256, 14336, 4096, 2, 192),  # the MLP weight at M = 256, sampled
]


def _rows(M):
    rows = set()
    for m0 in range(0, M, 128):
        rows.update({m0, min(m0 + 64, M - 1), min(m0 + 127, M - 1)})
    return sorted(r for r in rows if r < M)


@pytest.mark.parametrize("case", TILE_CASES, ids=lambda c: "x".join(map(str, c)))
def test_tile_two_chunk_stages(lib, case):
    M, N, K, st, bn = case
    p2 = lib.make_plan("tile", threads=192, rows_per_cta=bn, tokens_per_cta=128, stages=st, chunks_per_stage=2)
    p1 = lib.make_plan("tile", threads=192, rows_per_cta=bn, tokens_per_cta=128, stages=2 * st)
    for bias in (False, True):
        x, W, b, xd, Wd, bd = _inputs(M, N, K, M + N + K + bias, bias)
        got = tensor_bits(lib.bf16_linear_with_plan(xd, Wd, bd, plan_=p2))
        ref = tensor_bits(lib.bf16_linear_with_plan(xd, Wd, bd, plan_=p1))
        torch.cuda.synchronize()
        assert np.array_equal(got, ref), f"two-chunk stages differ from one-chunk stages: {case} bias={bias}"
        if M * N * K > 2e9:
            rows = _rows(M)
            want = oracle.linear_rows_bf16(wl.bits(x), wl.bits(W), wl.bits(b), np.array(rows, dtype=np.int64))
            check_close(got[rows], want, f"tile x2 {case} bias={bias} rows={len(rows)}")
        else:
            check_close(got, oracle.linear_bf16(wl.bits(x), wl.bits(W), wl.bits(b)), f"tile x2 {case} bias={bias}")
    assert lib.device_status() == 0


TILE_T_CASES = [
    # M, N, K, stages (of two chunks), tokens per tile
    (40, 1000, 576, 2, 64),      # 9 chunks; N tail of 104 W rows; 24 token rows of fill
    (64, 3584, 4096, 4, 64),     # the MLP width / 4, the ring depth the sweep tries
    (100, 300, 64, 2, 128),      # a single chunk
    (200, 2112, 7168, 3, 32),    # 7 token tiles x 17 W tiles
]


@pytest.mark.parametrize("case", TILE_T_CASES, ids=lambda c: "x".join(map(str, c)))
def test_tile_t_two_chunk_stages(lib, case):
    M, N, K, st, bn = case
    p2 = lib.make_plan("tile_t", threads=192, rows_per_cta=128, tokens_per_cta=bn, stages=st, chunks_per_stage=2)
    p1 = lib.make_plan("tile_t", threads=192, rows_per_cta=128, tokens_per_cta=bn, stages=2 * st)
    for bias in (False, True):
        x, W, b, xd, Wd, bd = _inputs(M, N, K, 3 * M + N + K + bias, bias)
        got = tensor_bits(lib.bf16_linear_with_plan(xd, Wd, bd, plan_=p2))
        ref = tensor_bits(lib.bf16_linear_with_plan(xd, Wd, bd, plan_=p1))
        torch.cuda.synchronize()
        assert np.array_equal(got, ref), f"two-chunk stages differ from one-chunk stages: {case} bias={bias}"
        check_close(got, oracle.linear_bf16(wl.bits(x), wl.bits(W), wl.bits(b)), f"tile_t x2 {case} bias={bias}")
    assert lib.device_status() == 0


SPLIT_CASES = [
    # kernel, M, N, K, W rows per CTA, K splits, stages (of two chunks)
    ("splitk", 16, 2112, 7168, 64, 8, 4),     # decode: 56 stages over 8 ranks
    ("splitk", 33, 300, 576, 32, 4, 2),       # 5 stages over 4 ranks, the last one half fill; ragged N
    ("splitk", 1, 128, 2880, 16, 16, 1),      # 23 stages over 16 ranks: ranks of one and two stages
    ("splitk", 64, 2112, 7168, 96, 12, 2),    # the decode M = 64 form: 264 CTAs, two per SM
    ("splitk", 64, 14336, 4096, 96, 2, 4),    # the MLP width at M = 64
    ("splitk_ws", 9, 384, 7168, 32, 16, 3),
    ("splitk_ws", 5, 130, 192, 48, 2, 1),     # 3 chunks: 2 stages over 2 ranks, the last half fill
    ("splitk_ws", 12, 256, 6144, 64, 48, 1),  # 48 stages over 48 ranks: one stage each
]


@pytest.mark.parametrize("case", SPLIT_CASES, ids=lambda c: "x".join(map(str, c)))
def test_splitk_two_chunk_stages(lib, case):
    kernel, M, N, K, rows, split, st = case
    p = lib.make_plan(kernel, threads=128, rows_per_cta=rows, tokens_per_cta=max(8, -(-M // 8) * 8),
                      split_k=split, stages=st, chunks_per_stage=2)
    ws = lib.new_workspace(lib.workspace_size(M, N, K, p), DEV) if kernel == "splitk_ws" else None
    for bias in (False, True):
        x, W, b, xd, Wd, bd = _inputs(M, N, K, 5 * M + N + split + bias, bias)
        outs = [tensor_bits(lib.run(xd, Wd, bd, plan_=p, workspace=ws)) for _ in range(2)]
        torch.cuda.synchronize()
        check_close(outs[0], oracle.linear_bf16(wl.bits(x), wl.bits(W), wl.bits(b)), f"{case} bias={bias}")
        assert np.array_equal(outs[0], outs[1]), "not deterministic across calls"
    assert lib.device_status() == 0


def test_splitk_two_chunk_exact(lib):
    """One-hot x rows select W columns exactly through two-chunk stages (a dropped or doubled chunk, or a
    chunk read from the wrong K offset, changes the selected column)."""
    M, N, K = 7, 300, 576
    p = lib.make_plan("splitk", threads=128, rows_per_cta=32, tokens_per_cta=8, split_k=3, stages=2,
                      chunks_per_stage=2)
    _, W, _ = wl.make_inputs(M, N, K, 11, False)
    ks = np.array([0, 63, 64, 127, 128, 511, 575])
    x = torch.zeros(M, K, dtype=torch.bfloat16)
    x[torch.arange(M), torch.from_numpy(ks)] = 1.0
    got = tensor_bits(lib.run(x.to(DEV), W.to(DEV), plan_=p))
    torch.cuda.synchronize()
    assert np.array_equal(got, wl.bits(W)[:, ks].T)
