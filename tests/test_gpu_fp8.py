"""GPU parity of the per-tensor FP8 path (bf16_quant_fp8, bf16_linear_fp8) against the oracle.

The quantisation must match oracle.quant_fp8 bit for bit (the same binary32
reciprocal and product, clamp, round to nearest even), on the vector path and
the scalar one, with tails.  The FP8 linear is compared with oracle.linear_fp8
under the same tolerance as the bf16 linear (its fp32 accumulation is the only
difference from the exact sum); one-hot rows with power-of-two scales must be
exact.  Shapes span router, decode and MLP weights, M over several 16-token
groups with a ragged last one, N not a multiple of 8, bias on and off.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tolerance import check_close, tensor_bits

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _scale(v):
    return torch.tensor([v], dtype=torch.float32, device=DEV)


def _fp8_inputs(M, N, K, seed, bias):
    """Seeded bf16 inputs, quantised on the CPU by the oracle with scales from their max."""
    x, W, b = wl.make_inputs(M, N, K, seed, bias)
    sx = float(np.float32(x.float().abs().max().item() / 448.0))
    sw = float(np.float32(W.float().abs().max().item() / 448.0))
    xq = oracle.quant_fp8(wl.bits(x), sx)
    wq = oracle.quant_fp8(wl.bits(W), sw)
    return x, W, b, xq, wq, sx, sw


@pytest.mark.parametrize("n", [8, 4096, 4097, 12345, 1, 7])
@pytest.mark.parametrize("s", [1.0, 0.0123, 7.0, 1.7])
def test_quant_matches_oracle(lib, n, s):
    rng = np.random.default_rng(n)
    x = torch.from_numpy(rng.standard_normal(n).astype(np.float32) * 4).to(torch.bfloat16)
    if n > 4:
        x[:4] = torch.tensor([1e4, -1e4, 0.0, -0.0]).to(torch.bfloat16)
    got = lib.quant_fp8(x.to(DEV), _scale(s))
    torch.cuda.synchronize()
    want = oracle.quant_fp8(wl.bits(x), s)
    assert np.array_equal(got.cpu().numpy(), want)


def test_quant_unaligned_takes_the_scalar_path(lib):
    x = torch.from_numpy(np.random.default_rng(1).standard_normal(1001).astype(np.float32)).to(torch.bfloat16)
    xd = x.to(DEV)
    out = torch.zeros(1001, dtype=torch.uint8, device=DEV)
    lib.quant_fp8(xd[1:], _scale(0.05), out=out[1:])  # both 2 / 1 bytes past a 16-byte boundary
    torch.cuda.synchronize()
    assert np.array_equal(out[1:].cpu().numpy(), oracle.quant_fp8(wl.bits(x[1:]), 0.05))
    assert out[0].item() == 0


SHAPES = [(1, 256, 7168), (16, 384, 7168), (4, 2112, 7168), (33, 300, 1024), (8, 14336, 4096), (2, 7, 16),
          (64, 256, 2048)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_linear_fp8_matches_oracle(lib, shape):
    M, N, K = shape
    for bias in (False, True):
        x, W, b, xq, wq, sx, sw = _fp8_inputs(M, N, K, M + N + K, bias)
        bd = b.to(DEV) if b is not None else None
        out = lib.bf16_linear_fp8(torch.from_numpy(xq).to(DEV), torch.from_numpy(wq).to(DEV), _scale(sx),
                                  _scale(sw), bd)
        torch.cuda.synchronize()
        want = oracle.linear_fp8(xq, wq, sx, sw, wl.bits(b))
        check_close(tensor_bits(out), want, f"fp8 M={M} N={N} K={K} bias={bias}")
    assert lib.device_status() == 0


def test_quant_then_linear_end_to_end(lib):
    M, N, K = 12, 2112, 7168
    x, W, _ = wl.make_inputs(M, N, K, 5, False)
    sx, sw = 0.01, 0.002
    wq = oracle.quant_fp8(wl.bits(W), sw)
    xq = lib.quant_fp8(x.to(DEV), _scale(sx))
    out = lib.bf16_linear_fp8(xq, torch.from_numpy(wq).to(DEV), _scale(sx), _scale(sw))
    torch.cuda.synchronize()
    want = oracle.linear_fp8(oracle.quant_fp8(wl.bits(x), sx), wq, sx, sw)
    check_close(tensor_bits(out), want, "quant -> fp8 linear")


def test_linear_fp8_exact_cases(lib):
    M, N, K = 20, 260, 512
    rng = np.random.default_rng(3)
    wq = rng.integers(0, 256, (N, K)).astype(np.uint8)
    wq[(wq & 0x7F) == 0x7F] = 0x38
    ks = rng.integers(0, K, M)
    xq = np.zeros((M, K), dtype=np.uint8)
    xq[np.arange(M), ks] = 0x38  # 1.0
    out = lib.bf16_linear_fp8(torch.from_numpy(xq).to(DEV), torch.from_numpy(wq).to(DEV), _scale(0.5), _scale(0.25))
    torch.cuda.synchronize()
    # e4m3 values have 4 significant bits: times 1/8 they are exact in bf16
    assert np.array_equal(tensor_bits(out), oracle.linear_fp8(xq, wq, 0.5, 0.25))


def test_linear_fp8_deterministic_and_pdl(lib):
    M, N, K = 16, 384, 7168
    _, _, _, xq, wq, sx, sw = _fp8_inputs(M, N, K, 9, False)
    xd, wd = torch.from_numpy(xq).to(DEV), torch.from_numpy(wq).to(DEV)
    a = lib.bf16_linear_fp8(xd, wd, _scale(sx), _scale(sw))
    outs = [lib.bf16_linear_fp8(xd, wd, _scale(sx), _scale(sw), flags=lib.FLAG_PDL) for _ in range(3)]
    torch.cuda.synchronize()
    for o in outs:
        assert torch.equal(o, a)


WM_CFGS = [(1024, 8, 1), (512, 4, 2), (256, 1, 4), (1024, 16, 1), (512, 2, 1)]


@pytest.mark.parametrize("cfg", WM_CFGS, ids=lambda c: "t%d_wpr%d_cps%d" % c)
@pytest.mark.parametrize("shape", [(4, 2112, 7168), (16, 1000, 1024), (1, 14336, 4096), (9, 77, 2048)],
                         ids=lambda s: "x".join(map(str, s)))
def test_linear_fp8_warpmma_form(lib, shape, cfg):
    M, N, K = shape
    t, w, c = cfg
    p = lib.make_plan("warpmma", threads=t, rows_per_cta=w, stages=c)
    for bias in (False, True):
        x, W, b, xq, wq, sx, sw = _fp8_inputs(M, N, K, M + N + K + w, bias)
        bd = b.to(DEV) if b is not None else None
        xd, wd = torch.from_numpy(xq).to(DEV), torch.from_numpy(wq).to(DEV)
        out = lib.bf16_linear_fp8(xd, wd, _scale(sx), _scale(sw), bd, plan_=p)
        torch.cuda.synchronize()
        check_close(tensor_bits(out), oracle.linear_fp8(xq, wq, sx, sw, wl.bits(b)),
                    f"fp8 warpmma M={M} N={N} K={K} cfg={cfg} bias={bias}")


@pytest.mark.parametrize("S,t", [(1, 128), (4, 256), (8, 128), (16, 256)])
def test_linear_fp8_split_form(lib, S, t):
    M, N, K = 16, 256, 7168
    x, W, b, xq, wq, sx, sw = _fp8_inputs(M, N, K, S, True)
    out = lib.bf16_linear_fp8(torch.from_numpy(xq).to(DEV), torch.from_numpy(wq).to(DEV), _scale(sx), _scale(sw),
                              b.to(DEV), plan_=lib.make_plan("dotmma", threads=t, rows_per_cta=8, split_k=S))
    torch.cuda.synchronize()
    check_close(tensor_bits(out), oracle.linear_fp8(xq, wq, sx, sw, wl.bits(b)), f"fp8 split S={S} t={t}")


def _tile(lib, stages=4):
    return lib.make_plan("tile", threads=192, stages=stages)


@pytest.mark.parametrize("shape", [(128, 256, 128), (300, 520, 1040), (17, 2112, 7168), (256, 14336, 4096)],
                         ids=lambda s: "x".join(map(str, s)))
def test_linear_fp8_tile_form(lib, shape):
    M, N, K = shape
    for bias in (False, True):
        x, W, b, xq, wq, sx, sw = _fp8_inputs(M, N, K, M + N + K, bias)
        bd = b.to(DEV) if b is not None else None
        out = lib.bf16_linear_fp8(torch.from_numpy(xq).to(DEV), torch.from_numpy(wq).to(DEV), _scale(sx),
                                  _scale(sw), bd, plan_=_tile(lib, 2 if K <= 1040 else 4))
        torch.cuda.synchronize()
        rows = np.unique(np.concatenate([np.arange(0, M, 127), [M - 1], np.arange(0, M, 128)]))
        rows = rows[rows < M]
        want = oracle.linear_fp8(xq[rows], wq, sx, sw, wl.bits(b))
        check_close(tensor_bits(out)[rows], want, f"fp8 tile M={M} N={N} K={K} bias={bias}")


def test_linear_fp8_tile_prefill_sampled(lib):
    M, N, K = 2048, 7168, 7168
    x, W, _, xq, wq, sx, sw = _fp8_inputs(M, N, K, 21, False)
    out = lib.bf16_linear_fp8(torch.from_numpy(xq).to(DEV), torch.from_numpy(wq).to(DEV), _scale(sx), _scale(sw))
    torch.cuda.synchronize()
    rows = np.array([0, 1, 127, 128, 1000, 2047])
    check_close(tensor_bits(out)[rows], oracle.linear_fp8(xq[rows], wq, sx, sw), "fp8 prefill sampled rows")


def test_linear_fp8_tile_exact(lib):
    M, N, K = 200, 264, 384
    rng = np.random.default_rng(4)
    wq = rng.integers(0, 256, (N, K)).astype(np.uint8)
    wq[(wq & 0x7F) == 0x7F] = 0x38
    ks = rng.integers(0, K, M)
    xq = np.zeros((M, K), dtype=np.uint8)
    xq[np.arange(M), ks] = 0x38
    out = lib.bf16_linear_fp8(torch.from_numpy(xq).to(DEV), torch.from_numpy(wq).to(DEV), _scale(0.5), _scale(0.25),
                              plan_=_tile(lib, 3))
    torch.cuda.synchronize()
    assert np.array_equal(tensor_bits(out), oracle.linear_fp8(xq, wq, 0.5, 0.25))


def test_linear_fp8_rejects(lib):
    xq = torch.zeros(4, 40, dtype=torch.uint8, device=DEV)
    wq = torch.zeros(8, 40, dtype=torch.uint8, device=DEV)
    with pytest.raises(lib.BF16LinearError):
        lib.bf16_linear_fp8(xq, wq, _scale(1.0), _scale(1.0))  # K % 16 != 0
    xq = torch.zeros(4, 64, dtype=torch.uint8, device=DEV)
    wq = torch.zeros(8, 64, dtype=torch.uint8, device=DEV)
    with pytest.raises(ValueError):
        lib.bf16_linear_fp8(xq, wq, torch.ones(2, device=DEV), _scale(1.0))
    for p in (lib.make_plan("splitk", threads=256, split_k=2), lib.make_plan("stream", threads=256),
              lib.make_plan("tile2", threads=192, stages=4)):  # kernels the FP8 entry does not run
        with pytest.raises(lib.BF16LinearError):
            lib.bf16_linear_fp8(xq, wq, _scale(1.0), _scale(1.0), plan_=p)
    with pytest.raises(lib.BF16LinearError):  # the tile form needs a ring of at least two stages
        lib.bf16_linear_fp8(xq, wq, _scale(1.0), _scale(1.0), plan_=lib.make_plan("tile", threads=192, stages=1))
    with pytest.raises(lib.BF16LinearError):  # 17 tokens do not fit the warp-MMA form
        lib.bf16_linear_fp8(torch.zeros(17, 64, dtype=torch.uint8, device=DEV), wq, _scale(1.0), _scale(1.0),
                            plan_=lib.make_plan("warpmma", threads=512, rows_per_cta=4, stages=1))
