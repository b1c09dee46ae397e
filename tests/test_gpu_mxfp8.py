"""GPU parity of the MXFP8 path (bf16_quant_mxfp8, bf16_linear_mxfp8) against the oracle.

Quantisation must match the oracle bit for bit (codes and scale bytes) on seeded
inputs and on the edge cases (all-zero blocks, values that saturate, bf16
subnormals, blocks spanning many binades).  The linear is compared element by
element with the oracle's block-scaled result within the parity tolerance, on
operands quantised by the oracle from seeded bf16 data and on random codes with
random scale bytes (a wrong block index would misapply a scale), over router,
decode and ragged shapes, every K split and block size of the explicit-plan
entry point, bias on and off.  The early-weights launch flag must not change a
bit.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tolerance import check_close, tensor_bits

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _u8(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).to(DEV)


def _bf16_tensor(vals):
    return torch.tensor(vals, dtype=torch.float64).to(torch.bfloat16)


@pytest.mark.parametrize("rows,K,seed", [(1, 32, 1), (7, 2880, 2), (16, 7168, 3), (3, 96, 4)])
def test_quant_matches_oracle(lib, rows, K, seed):
    g = torch.Generator().manual_seed(seed)
    mag = torch.exp2(torch.randint(-40, 40, (rows, K // 32), generator=g).double()).repeat_interleave(32, dim=1)
    x = (torch.randn(rows, K, generator=g, dtype=torch.float64) * mag).to(torch.bfloat16)
    q, s = lib.quant_mxfp8(x.to(DEV))
    torch.cuda.synchronize()
    wq, ws = oracle.quant_mxfp8(wl.bits(x))
    assert np.array_equal(s.cpu().numpy(), ws)
    assert np.array_equal(q.cpu().numpy(), wq)


def test_quant_edge_blocks(lib):
    blocks = [[0.0] * 32,                                       # all zero: scale byte 0, codes 0
              [480.0] + [1.0] * 31,                             # saturates to 448
              [-470.0, 300.0] + [0.25] * 30,
              [2.0 ** -130, -(2.0 ** -133)] + [0.0] * 30,       # bf16 subnormals: the exponent clamps at -127
              [2.0 ** 100, 2.0 ** 90, -(2.0 ** 80)] + [3.0] * 29,  # values that underflow e4m3 next to a large one
              [1.0] * 31 + [-(2.0 ** 127) * 1.5]]               # the largest binade of bf16
    x = _bf16_tensor(blocks)
    q, s = lib.quant_mxfp8(x.to(DEV))
    torch.cuda.synchronize()
    wq, ws = oracle.quant_mxfp8(wl.bits(x))
    assert np.array_equal(s.cpu().numpy(), ws)
    assert np.array_equal(q.cpu().numpy(), wq)
    assert int(ws[0, 0]) == 0 and int(ws[1, 0]) == 127 and int(wq[1, 0]) == 0x7E


def _quantised_inputs(M, N, K, seed, bias):
    x, W, b = wl.make_inputs(M, N, K, seed, bias)
    xq, xs = oracle.quant_mxfp8(wl.bits(x))
    wq, ws = oracle.quant_mxfp8(wl.bits(W))
    return xq, xs, wq, ws, b


def _run(lib, xq, xs, wq, ws, b, plan=None, flags=0):
    out = lib.bf16_linear_mxfp8(_u8(xq), _u8(xs), _u8(wq), _u8(ws), b.to(DEV) if b is not None else None,
                                flags=flags, plan_=plan)
    torch.cuda.synchronize()
    return tensor_bits(out)


SHAPES = [(1, 256, 7168), (4, 256, 2048), (16, 384, 7168), (9, 128, 2880), (5, 33, 96), (17, 300, 1024),
          (8, 2112, 7168), (40, 520, 512)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_linear_matches_oracle(lib, shape):
    M, N, K = shape
    for bias in (False, True):
        xq, xs, wq, ws, b = _quantised_inputs(M, N, K, M + N + K + bias, bias)
        got = _run(lib, xq, xs, wq, ws, b)
        want = oracle.linear_mxfp8(xq, xs, wq, ws, wl.bits(b))
        check_close(got, want, f"mxfp8 M={M} N={N} K={K} bias={bias}")
    assert lib.device_status() == 0


def test_linear_random_scales(lib):
    """Random codes and scale bytes (2^-17 .. 2^17 per block): each block's scale must reach its own MMA."""
    rng = np.random.default_rng(5)
    M, N, K = 13, 72, 640
    finite = [c for c in range(256) if (c & 0x7F) != 0x7F]
    xq = rng.choice(finite, size=(M, K)).astype(np.uint8)
    wq = rng.choice(finite, size=(N, K)).astype(np.uint8)
    xs = rng.integers(110, 145, size=(M, K // 32)).astype(np.uint8)
    ws = rng.integers(110, 145, size=(N, K // 32)).astype(np.uint8)
    for S, threads in [(1, 128), (4, 256), (16, 128)]:
        plan = lib.make_plan("dotmma", threads=threads, split_k=S)
        got = _run(lib, xq, xs, wq, ws, None, plan=plan)
        check_close(got, oracle.linear_mxfp8(xq, xs, wq, ws), f"mxfp8 random scales S={S} threads={threads}")


@pytest.mark.parametrize("S", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("threads", [128, 256])
def test_linear_forced_plans(lib, S, threads):
    M, N, K = 11, 130, 2880
    xq, xs, wq, ws, b = _quantised_inputs(M, N, K, 3 * S + threads, True)
    plan = lib.make_plan("dotmma", threads=threads, split_k=S)
    got = _run(lib, xq, xs, wq, ws, b, plan=plan)
    check_close(got, oracle.linear_mxfp8(xq, xs, wq, ws, wl.bits(b)), f"mxfp8 S={S} threads={threads}")


def test_linear_large_n_sampled_rows(lib):
    """The MLP-sized weight (N = 14336) at M = 8: every row against the oracle's selected-rows form."""
    M, N, K = 8, 14336, 4096
    xq, xs, wq, ws, b = _quantised_inputs(M, N, K, 77, True)
    got = _run(lib, xq, xs, wq, ws, b)
    rows = np.array([0, 3, 7], dtype=np.int64)
    want = oracle.linear_rows_mxfp8(xq, xs, wq, ws, wl.bits(b), rows)
    check_close(got[rows], want, "mxfp8 M=8 N=14336 K=4096 sampled rows")


def test_early_weights_flag_same_bits(lib):
    M, N, K = 16, 256, 7168
    xq, xs, wq, ws, b = _quantised_inputs(M, N, K, 9, True)
    base = _run(lib, xq, xs, wq, ws, b)
    for flags in (lib.FLAG_PDL, lib.FLAG_SERIAL):
        assert np.array_equal(_run(lib, xq, xs, wq, ws, b, flags=flags), base)


def test_quant_then_linear_end_to_end(lib):
    """bf16 activations quantised on the GPU, then the linear: equal to the oracle on the oracle's codes."""
    M, N, K = 6, 384, 7168
    x, W, b = wl.make_inputs(M, N, K, 31, True)
    wq, ws = oracle.quant_mxfp8(wl.bits(W))
    xq_d, xs_d = lib.quant_mxfp8(x.to(DEV))
    out = lib.bf16_linear_mxfp8(xq_d, xs_d, _u8(wq), _u8(ws), b.to(DEV))
    torch.cuda.synchronize()
    xq, xs = oracle.quant_mxfp8(wl.bits(x))
    check_close(tensor_bits(out), oracle.linear_mxfp8(xq, xs, wq, ws, wl.bits(b)), "mxfp8 quant + linear")


def test_rejects_bad_arguments(lib):
    xq = torch.zeros(4, 80, dtype=torch.uint8, device=DEV)   # K = 80: not whole 32-element blocks
    xs = torch.zeros(4, 2, dtype=torch.uint8, device=DEV)
    with pytest.raises(lib.BF16LinearError) as e:
        lib.bf16_linear_mxfp8(xq, xs, xq, xs)
    assert e.value.status == -6
    with pytest.raises(lib.BF16LinearError):
        lib.bf16_linear_mxfp8(_u8(np.zeros((4, 64))), _u8(np.zeros((4, 2))), _u8(np.zeros((4, 64))),
                              _u8(np.zeros((4, 2))), plan_=lib.make_plan("dotmma", threads=128, split_k=3))


# ---- the tile form (tcgen05 block-scaled MMAs, scales staged into tensor memory) ----

def _tile_plan(lib, stages=4, group=0, bq=256):
    return lib.make_plan("tile", threads=320, rows_per_cta=bq, stages=stages, split_k=group)


TILE_CASES = [
    # W rows per tile, M, N, K, stages, raster group
    (128, 128, 128, 128, 2, 0),     # one tile, one chunk (four scale blocks)
    (128, 130, 300, 1024, 6, 0),    # ragged M and N, the ring wraps
    (256, 256, 520, 4096, 4, 1),
    (128, 1000, 700, 256, 3, 2),    # ragged everything, two chunks on a three-deep ring
    (256, 1000, 700, 256, 3, 2),    # the same with 256-row weight tiles (one accumulator buffer)
    (256, 129, 129, 384, 2, 16),    # one row past a tile, N inside one weight tile
    (256, 600, 2112, 7168, 4, 0),   # 5 x 9 tiles, K = 56 chunks, sampled rows
    (128, 600, 2112, 7168, 6, 0),
]


@pytest.mark.parametrize("case", TILE_CASES, ids=lambda c: "x".join(map(str, c)))
def test_tile_matches_oracle(lib, case):
    bq, M, N, K, st, grp = case
    plan = _tile_plan(lib, st, grp, bq)
    sampled = M * N * K > 2e9
    for bias in (False, True):
        xq, xs, wq, ws, b = _quantised_inputs(M, N, K, M + N + K + st + bias, bias)
        got = _run(lib, xq, xs, wq, ws, b, plan=plan)
        if sampled:
            rows = np.array(sorted({0, 127, 128, M // 2, M - 1}), dtype=np.int64)
            check_close(got[rows], oracle.linear_rows_mxfp8(xq, xs, wq, ws, wl.bits(b), rows),
                        f"mxfp8 tile M={M} N={N} K={K} sampled rows")
        else:
            check_close(got, oracle.linear_mxfp8(xq, xs, wq, ws, wl.bits(b)),
                        f"mxfp8 tile M={M} N={N} K={K} stages={st} group={grp} bias={bias}")
    assert lib.device_status() == 0


def test_tile_random_scales_and_one_hot(lib):
    """Random codes with random scale bytes, and one-hot rows: each block's scale must reach its own
    MMA step and each row and column its own scale word."""
    rng = np.random.default_rng(23)
    M, N, K = 200, 264, 512
    finite = [c for c in range(256) if (c & 0x7F) != 0x7F]
    xq = rng.choice(finite, size=(M, K)).astype(np.uint8)
    wq = rng.choice(finite, size=(N, K)).astype(np.uint8)
    xs = rng.integers(110, 145, size=(M, K // 32)).astype(np.uint8)
    ws = rng.integers(110, 145, size=(N, K // 32)).astype(np.uint8)
    for bq in (128, 256):
        got = _run(lib, xq, xs, wq, ws, None, plan=_tile_plan(lib, bq=bq))
        check_close(got, oracle.linear_mxfp8(xq, xs, wq, ws), f"mxfp8 tile random scales bq={bq}")
    # one-hot rows: x[m] = 1.0 at k_m (one block), so out[m, n] = e4m3(w[n, k_m]) * 2^(xs[m, b] + ws[n, b] - 254)
    xo = np.zeros((M, K), dtype=np.uint8)
    ks = (np.arange(M) * 37 + 5) % K
    xo[np.arange(M), ks] = 0x38
    for bq in (128, 256):
        got = _run(lib, xo, xs, wq, ws, None, plan=_tile_plan(lib, bq=bq))
        assert np.array_equal(got, oracle.linear_mxfp8(xo, xs, wq, ws))


def test_tile_is_the_large_m_choice(lib):
    """At prefill size the entry point's own choice is the tile form; sampled rows against the oracle."""
    M, N, K = 2048, 2112, 7168
    xq, xs, wq, ws, b = _quantised_inputs(M, N, K, 41, True)
    got = _run(lib, xq, xs, wq, ws, b)
    rows = np.array([0, 127, 128, 1023, 2047], dtype=np.int64)
    check_close(got[rows], oracle.linear_rows_mxfp8(xq, xs, wq, ws, wl.bits(b), rows), "mxfp8 prefill sampled rows")
    forced = _run(lib, xq, xs, wq, ws, b, plan=_tile_plan(lib))
    assert np.array_equal(got, forced)


def test_tile_rejects_partial_chunks(lib):
    xq, xs, wq, ws, _ = _quantised_inputs(64, 128, 96, 3, False)   # K = 96: not whole 128-code chunks
    with pytest.raises(lib.BF16LinearError) as e:
        _run(lib, xq, xs, wq, ws, None, plan=_tile_plan(lib))
    assert e.value.status == -6
