"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Every case draws seeded inputs from workloads.py, runs the library on cuda:0,
and compares element by element with the oracle under the tolerance in
tests/tolerance.py.  Kernels are exercised both through the dispatcher and
forced one by one with explicit plans, over shapes that span several tiles,
ragged tails in N, K and M, and the edge cases (M = 0, N = 1, K = 1, K % 8 != 0,
bias on and off).  Shapes too large for the oracle to evaluate in full are
checked on sampled rows (always including the first and last row of every
128-row M tile).
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
    return x, W, b


def _run(lib, x, W, b, plan=None):
    xd, Wd = x.to(DEV), W.to(DEV)
    bd = b.to(DEV) if b is not None else None
    if plan is None:
        out = lib.bf16_linear(xd, Wd, bd)
    else:
        out = lib.bf16_linear_with_plan(xd, Wd, bd, plan_=plan)
    torch.cuda.synchronize()
    return tensor_bits(out)


def _expect(x, W, b):
    return oracle.linear_bf16(wl.bits(x), wl.bits(W), wl.bits(b))


def _check(lib, M, N, K, seed=0, bias=False, plan=None, what=""):
    x, W, b = _inputs(M, N, K, seed, bias)
    got = _run(lib, x, W, b, plan)
    want = _expect(x, W, b)
    check_close(got, want, what or f"M={M} N={N} K={K} bias={bias} plan={plan}")
    return got, want


def splitk_plan(lib, M, split, stages, rows=32, tokens=None):
    return lib.make_plan("splitk", threads=128, rows_per_cta=rows,
                         tokens_per_cta=tokens or max(8, -(-M // 8) * 8), split_k=split, stages=stages)


def dot_plan(lib, R, threads=128):
    return lib.make_plan("dotprod", threads=threads, rows_per_cta=R)


# ---------------------------------------------------------------------------
# The workloads, through the dispatcher.
# ---------------------------------------------------------------------------

def test_router_smallest_matches_golden(lib):
    import os
    import sys
    sys.path.insert(0, os.path.join(os.path.dirname(__file__), "golden"))
    import make_golden
    meta, want = make_golden.read("router_smallest_seed0.txt")
    x, W, b = _inputs(meta["M"], meta["N"], meta["K"], meta["seed"], bool(meta["bias"]))
    # the fixture was written by the oracle from the same seeded inputs
    assert np.array_equal(_expect(x, W, b), want)
    check_close(_run(lib, x, W, b), want, "router smallest vs golden")


@pytest.mark.parametrize("pt", wl.router_sweep(), ids=lambda p: p["name"])
def test_router_sweep(lib, pt):
    _check(lib, pt["M"], pt["N"], pt["K"], pt["seed"], pt["bias"])


@pytest.mark.parametrize("pt", wl.decode_proj(), ids=lambda p: p["name"])
def test_decode_projection(lib, pt):
    _check(lib, pt["M"], pt["N"], pt["K"], pt["seed"], pt["bias"])


def _sample_rows(M, max_rows=24, seed=0):
    rows = {0, M - 1}
    for t in range(0, M, 128):
        rows |= {t, min(t + 127, M - 1)}
    rng = np.random.default_rng(seed)
    rows = sorted(rows)
    if len(rows) > max_rows:
        keep = [rows[0], rows[-1]] + list(rng.choice(rows[1:-1], max_rows - 2, replace=False))
        rows = sorted(set(keep))
    extra = rng.integers(0, M, 4)
    return np.array(sorted(set(rows) | set(int(e) for e in extra)), dtype=np.int64)


def _check_rows(lib, M, N, K, seed, bias, plan=None):
    x, W, b = _inputs(M, N, K, seed, bias)
    got = _run(lib, x, W, b, plan)
    rows = _sample_rows(M, seed=seed)
    want = oracle.linear_rows_bf16(wl.bits(x), wl.bits(W), wl.bits(b), rows)
    check_close(got[rows], want, f"sampled rows M={M} N={N} K={K} bias={bias}")
    assert np.isfinite(torch.from_numpy(got.view(np.int16)).view(torch.bfloat16).float().numpy()).all()


@pytest.mark.parametrize("pt", wl.mlp_bias(), ids=lambda p: p["name"])
def test_mlp_with_bias(lib, pt):
    if pt["M"] <= 8:
        _check(lib, pt["M"], pt["N"], pt["K"], pt["seed"], pt["bias"])
    else:
        _check_rows(lib, pt["M"], pt["N"], pt["K"], pt["seed"], pt["bias"])


@pytest.mark.parametrize("pt", wl.prefill(), ids=lambda p: p["name"])
def test_prefill_sampled_rows(lib, pt):
    _check_rows(lib, pt["M"], pt["N"], pt["K"], pt["seed"], pt["bias"])


# ---------------------------------------------------------------------------
# Each kernel forced, over ragged shapes.
# ---------------------------------------------------------------------------

DOT_SHAPES = [(1, 1, 8), (1, 1, 1), (3, 17, 2880), (4, 256, 2048), (2, 5, 7), (8, 130, 1000),
              (5, 33, 2881), (9, 40, 264), (13, 19, 101), (1, 300, 7168)]


@pytest.mark.parametrize("R", [1, 2, 4])
@pytest.mark.parametrize("shape", DOT_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_dotprod_forced(lib, shape, R):
    M, N, K = shape
    for bias in (False, True):
        _check(lib, M, N, K, seed=M * 7 + N + K, bias=bias, plan=dot_plan(lib, R, threads=128 if K > 64 else 64))


@pytest.mark.parametrize("case", [(9, 256, 4096, 5, 2), (16, 384, 7168, 8, 2), (13, 40, 2880, 4, 1),
                                  (16, 256, 6144, 3, 4), (6, 128, 2880, 2, 1), (11, 33, 1032, 7, 2),
                                  (5, 17, 101, 2, 1), (12, 300, 7168, 6, 4)],
                         ids=lambda c: "x".join(map(str, c)))
def test_dotprod_token_groups(lib, case):
    """Token groups side by side (grid.y = ceil(M / t)), including a ragged last group
    and the scalar K % 8 != 0 form."""
    M, N, K, t, R = case
    plan = lib.make_plan("dotprod", threads=128, rows_per_cta=R, tokens_per_cta=t)
    for bias in (False, True):
        got, _ = _check(lib, M, N, K, seed=M + N + K + t, bias=bias, plan=plan)
    # Each (row, token) output is summed in the same order whatever the grouping
    # (per-thread k-slices, shuffle tree, warps in order), so the bits must match
    # a single CTA row looping over groups of 8.
    x, W, b = _inputs(M, N, K, 3, True)
    loop = _run(lib, x, W, b, lib.make_plan("dotprod", threads=128, rows_per_cta=R, tokens_per_cta=0))
    assert np.array_equal(loop, _run(lib, x, W, b, plan))


@pytest.mark.parametrize("shape", [(1, 256, 7168), (4, 300, 2056), (3, 17, 2880)], ids=lambda s: "x".join(map(str, s)))
def test_dotprod_x_from_l2(lib, shape):
    """x read from L2 (stages = 1) instead of staged: the same products in the same order, the same bits."""
    M, N, K = shape
    x, W, b = _inputs(M, N, K, 8, True)
    staged = _run(lib, x, W, b, lib.make_plan("dotprod", threads=128, rows_per_cta=2))
    direct = _run(lib, x, W, b, lib.make_plan("dotprod", threads=128, rows_per_cta=2, stages=1))
    assert np.array_equal(staged, direct)
    check_close(direct, _expect(x, W, b), f"dotprod x from L2 M={M} N={N} K={K}")


@pytest.mark.parametrize("threads", [64, 256])
def test_dotprod_block_sizes(lib, threads):
    _check(lib, 4, 384, 7168, seed=5, plan=dot_plan(lib, 2, threads))


SPLIT_CASES = [
    # M, N, K, rows (MMA N), split, stages
    (5, 256, 4096, 32, 8, 5),
    (16, 256, 7168, 16, 9, 13),
    (16, 384, 7168, 32, 12, 10),
    (9, 128, 2880, 16, 8, 2),       # K = 2880: 45 chunks over 8 CTAs (uneven split), ring reuse
    (12, 256, 6144, 64, 6, 4),      # the pages' default (split_k, num_stages) = (6, 4)
    (1, 200, 64, 16, 1, 1),         # one chunk, one CTA, ragged N
    (3, 130, 136, 48, 1, 1),        # K tail inside the last chunk, one stage reused 3 times
    (32, 2112, 7168, 128, 8, 8),    # N tail (2112 = 16.5 x 128)
    (64, 2112, 7168, 128, 8, 3),    # 64 tokens, ring wraps several times
    (48, 300, 520, 96, 2, 2),
    (17, 129, 1032, 192, 5, 2),     # ragged everything
    (8, 14336, 4096, 256, 2, 4),
    (64, 1000, 1024, 256, 1, 2),
    (2, 64, 7168, 16, 16, 7),       # 16-CTA cluster, M = 2
]


@pytest.mark.parametrize("case", SPLIT_CASES, ids=lambda c: "x".join(map(str, c)))
def test_splitk_forced(lib, case):
    M, N, K, rows, split, stages = case
    for bias in (False, True):
        _check(lib, M, N, K, seed=M + N + K + split, bias=bias, plan=splitk_plan(lib, M, split, stages, rows=rows))


@pytest.mark.parametrize("tokens", [8, 16, 24, 40, 64])
def test_splitk_token_padding(lib, tokens):
    """Fewer tokens than the loaded x rows: padded rows are zero-filled and never stored."""
    _check(lib, 3, 256, 2048, seed=tokens, plan=splitk_plan(lib, 3, 4, 4, rows=32, tokens=tokens))


@pytest.mark.parametrize("rows", [16, 32, 48, 64, 96, 128, 192, 256])
def test_splitk_every_tile_width(lib, rows):
    _check(lib, 11, 520, 1536, seed=rows, bias=True, plan=splitk_plan(lib, 11, 3, 3, rows=rows))


def test_pdl_launch_matches(lib):
    """Programmatic dependent launch changes scheduling only, never the result."""
    import ctypes
    for (M, N, K) in [(16, 256, 7168), (2, 384, 7168), (64, 2112, 7168)]:
        x, W, b = _inputs(M, N, K, 21, True)
        xd, Wd, bd = x.to(DEV), W.to(DEV), b.to(DEV)
        plain = tensor_bits(lib.bf16_linear(xd, Wd, bd))
        outs = []
        for _ in range(3):
            o = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
            st = lib.load().bf16_linear_ex(ctypes.c_void_p(xd.data_ptr()), ctypes.c_void_p(Wd.data_ptr()),
                                           ctypes.c_void_p(bd.data_ptr()), ctypes.c_void_p(o.data_ptr()),
                                           M, N, K, 1, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
            assert st == 0
            outs.append(o)
        torch.cuda.synchronize()
        for o in outs:
            assert np.array_equal(tensor_bits(o), plain)


# ---------------------------------------------------------------------------
# Exact cases (bitwise on every kernel) and determinism.
# ---------------------------------------------------------------------------

def _plans_for(lib, M):
    plans = [None, dot_plan(lib, 2)]
    if M <= 64:
        plans.append(splitk_plan(lib, M, 4, 2, rows=32))
    return plans


@pytest.mark.parametrize("M", [1, 4, 16, 64])
def test_one_hot_rows_are_exact(lib, M):
    N, K = 256, 2048
    rng = np.random.default_rng(M)
    _, W, _ = _inputs(1, N, K, 99, False)
    ks = rng.integers(0, K, M)
    x = torch.zeros(M, K, dtype=torch.bfloat16)
    x[torch.arange(M), torch.from_numpy(ks)] = 1.0
    want = wl.bits(W)[:, ks].T
    for plan in _plans_for(lib, M):
        got = _run(lib, x, W, None, plan)
        assert np.array_equal(got, want), f"one-hot not exact with plan {plan}"


@pytest.mark.parametrize("K", [2048, 2880, 7168])
def test_all_ones_gives_K(lib, K):
    M, N = 8, 130
    x = torch.ones(M, K, dtype=torch.bfloat16)
    W = torch.ones(N, K, dtype=torch.bfloat16)
    b = torch.full((N,), 0.5, dtype=torch.bfloat16)
    for plan in _plans_for(lib, M):
        got = _run(lib, x, W, None, plan)
        assert (got == wl.bits(torch.tensor([float(K)], dtype=torch.bfloat16))[0]).all()
        gotb = _run(lib, x, W, b, plan)
        assert np.array_equal(gotb, oracle.linear_bf16(wl.bits(x), wl.bits(W), wl.bits(b)))


def test_zero_x_returns_bias(lib):
    M, N, K = 5, 300, 1024
    _, W, b = _inputs(M, N, K, 3, True)
    x = torch.zeros(M, K, dtype=torch.bfloat16)
    for plan in _plans_for(lib, M):
        assert np.array_equal(_run(lib, x, W, b, plan), np.broadcast_to(wl.bits(b), (M, N)))


def test_power_of_two_scaling_is_exact(lib):
    M, N, K = 16, 256, 4096
    x, W, _ = _inputs(M, N, K, 4, False)
    for plan in _plans_for(lib, M):
        base = _run(lib, x, W, None, plan)
        scaled = _run(lib, (x.float() * 8).to(torch.bfloat16), W, None, plan)
        b64 = torch.from_numpy(base.view(np.int16)).view(torch.bfloat16).double()
        s64 = torch.from_numpy(scaled.view(np.int16)).view(torch.bfloat16).double()
        assert torch.equal(s64, b64 * 8), f"x*8 not exactly 8*out with plan {plan}"


@pytest.mark.parametrize("shape", [(16, 384, 7168), (4, 2112, 7168), (64, 2112, 7168)])
def test_bitwise_deterministic(lib, shape):
    M, N, K = shape
    x, W, _ = _inputs(M, N, K, 8, False)
    xd, Wd = x.to(DEV), W.to(DEV)
    outs = []
    for _ in range(3):
        outs.append(tensor_bits(lib.bf16_linear(xd, Wd)))
    assert all(np.array_equal(outs[0], o) for o in outs[1:])


# ---------------------------------------------------------------------------
# Boundary behaviour on the device.
# ---------------------------------------------------------------------------

def test_no_write_outside_out(lib):
    """Poisoned guard bands around `out` stay untouched (every kernel)."""
    M, N, K = 5, 130, 2048
    x, W, b = _inputs(M, N, K, 11, True)
    xd, Wd, bd = x.to(DEV), W.to(DEV), b.to(DEV)
    for plan in _plans_for(lib, M):
        buf = torch.full((M * N + 2 * 64,), float("nan"), dtype=torch.bfloat16, device=DEV)
        out = buf[64:64 + M * N].view(M, N)
        if plan is None:
            lib.bf16_linear(xd, Wd, bd, out=out)
        else:
            lib.bf16_linear_with_plan(xd, Wd, bd, out=out, plan_=plan)
        torch.cuda.synchronize()
        assert torch.isnan(buf[:64]).all() and torch.isnan(buf[64 + M * N:]).all()
        check_close(tensor_bits(out), oracle.linear_bf16(wl.bits(x), wl.bits(W), wl.bits(b)), "guarded")


def test_m_zero_is_a_no_op(lib):
    x = torch.empty(0, 64, dtype=torch.bfloat16, device=DEV)
    W = torch.randn(8, 64, device=DEV).to(torch.bfloat16)
    out = lib.bf16_linear(x, W)
    assert out.shape == (0, 8)


def test_rejects_misaligned_and_wrong_dtype(lib):
    W = torch.randn(8, 72, device=DEV).to(torch.bfloat16)
    xbig = torch.randn(1, 80, device=DEV).to(torch.bfloat16)
    x = xbig[:, 8:].contiguous()[:, :72]  # aligned copy
    lib.bf16_linear(x.contiguous(), W)
    mis = xbig.view(-1)[1:73].view(1, 72)  # 2-byte offset
    with pytest.raises(lib.BF16LinearError) as e:
        lib.bf16_linear(mis, W)
    assert e.value.status == -2
    with pytest.raises(TypeError):
        lib.bf16_linear(x.float(), W)
    with pytest.raises(TypeError):
        lib.bf16_linear(x, W.float())


def test_explicit_plan_never_falls_back(lib):
    x = torch.randn(4, 2049, device=DEV).to(torch.bfloat16)
    W = torch.randn(16, 2049, device=DEV).to(torch.bfloat16)
    with pytest.raises(lib.BF16LinearError) as e:
        lib.bf16_linear_with_plan(x, W, plan_=splitk_plan(lib, 4, 2, 2))
    assert e.value.status == -6
    lib.bf16_linear(x, W)  # the dispatcher takes the dot product for K % 8 != 0


def test_status_word_clean_after_runs(lib):
    assert lib.device_status(clear=False) == 0


def test_bounded_wait_reports_timeout(lib):
    """A wait that nothing completes gives up after its limit; the GPU stays usable."""
    assert lib.device_status(clear=True) == 0
    lib.selftest_wait(2000)  # 2 ms
    torch.cuda.synchronize()
    st = lib.device_status(clear=True)
    assert st & 0xFF == (-5) & 0xFF and (st >> 8) == 6
    assert lib.device_status(clear=False) == 0
    _check(lib, 4, 256, 2048, seed=0)  # still works
