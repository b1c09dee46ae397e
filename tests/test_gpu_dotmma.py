"""GPU parity of the router split-K kernel on warp-level MMAs (BF16L_KERNEL_DOTMMA).

CTA (r, q) of a cluster of S computes rows 8q..8q+7 over the r-th K run with
mma.sync fed by 16-byte loads; rank 0 sums the S partial tiles received over
DSMEM.  The cases cover S = 1, 2, 4, 8 and both block sizes, M = 1..16 (tokens
8..15 in the MMA's upper rows), N not a multiple of 8, K tails inside a 32-wide
block, K runs too short to give every warp a block, bias on and off, the router
shapes, and the fp32 epilogue (which must round to the bf16 result of the same
plan bit for bit).  Results for one plan are bitwise reproducible.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tolerance import check_close, tensor_bits

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

SHAPES = [(16, 384, 7168), (9, 256, 4096), (13, 128, 2880), (4, 300, 1032), (1, 7, 136), (16, 20, 40),
          (11, 257, 6144)]


def _smem(M, K, S):
    nvec = K // 8
    nblk = -(-nvec // 4)
    most = max(min(nvec, 4 * (nblk * (r + 1) // S)) - 4 * (nblk * r // S) for r in range(S))
    return M * most * 16


def _plan(lib, S, threads=256, xr=0):
    return lib.make_plan("dotmma", threads=threads, rows_per_cta=8, split_k=S, stages=xr)


def _run(lib, x, W, b, plan, f32=False):
    xd, Wd = x.to(DEV), W.to(DEV)
    bd = b.to(DEV) if b is not None else None
    out = (lib.bf16_linear_f32out(xd, Wd, bd, plan_=plan) if f32
           else lib.bf16_linear_with_plan(xd, Wd, bd, plan_=plan))
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("xr", [0, 1], ids=["xsmem", "xreg"])
@pytest.mark.parametrize("threads", [128, 256])
@pytest.mark.parametrize("S", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_dotmma_forced(lib, shape, S, threads, xr):
    M, N, K = shape
    p = _plan(lib, S, threads, xr)
    # too few K blocks for the cluster, or (x in shared memory) the x slice does not fit
    if S > -(-(K // 8) // 4) or (not xr and _smem(M, K, S) > 200 * 1024):
        with pytest.raises(lib.BF16LinearError):
            lib.plan_check(M, N, K, p)
        return
    for bias in (False, True):
        x, W, b = wl.make_inputs(M, N, K, M + N + K + S, bias)
        got = tensor_bits(_run(lib, x, W, b, p))
        want = oracle.linear_bf16(wl.bits(x), wl.bits(W), wl.bits(b))
        check_close(got, want, f"dotmma M={M} N={N} K={K} S={S} threads={threads} bias={bias}")


@pytest.mark.parametrize("M", range(1, 17))
def test_dotmma_router_tokens(lib, M):
    x, W, b = wl.make_inputs(M, 256, 7168, 100 + M, False)
    want = oracle.linear_bf16(wl.bits(x), wl.bits(W), None)
    for xr in (0, 1):
        got = tensor_bits(_run(lib, x, W, b, _plan(lib, 4, 256, xr)))
        check_close(got, want, f"dotmma router M={M} xr={xr}")


def test_dotmma_x_paths_agree(lib):
    # x from shared memory or from registers: the same fragments, the same MMAs, the same bits
    for (M, N, K, S) in [(16, 384, 7168, 4), (5, 130, 2880, 2), (12, 256, 4096, 16)]:
        x, W, b = wl.make_inputs(M, N, K, 7, True)
        a = tensor_bits(_run(lib, x, W, b, _plan(lib, S, 128, 0)))
        assert np.array_equal(a, tensor_bits(_run(lib, x, W, b, _plan(lib, S, 128, 1))))


def _ws_run(lib, x, W, b, plan, f32=False):
    xd, Wd = x.to(DEV), W.to(DEV)
    bd = b.to(DEV) if b is not None else None
    ws = lib.new_workspace(lib.workspace_size(x.shape[0], W.shape[0], W.shape[1], plan), DEV)
    out = torch.empty(x.shape[0], W.shape[0], dtype=torch.float32 if f32 else torch.bfloat16, device=DEV)
    outs = []
    for _ in range(2):  # the counters reset themselves: a second call on the same workspace must agree
        lib.run(xd, Wd, bd, out, plan_=plan, workspace=ws)
        torch.cuda.synchronize()
        outs.append(out.clone())
    assert torch.equal(outs[0], outs[1])
    return outs[0]


@pytest.mark.parametrize("xr", [0, 1], ids=["xsmem", "xreg"])
@pytest.mark.parametrize("S", [2, 8, 32, 64])
@pytest.mark.parametrize("shape", [(16, 384, 7168), (9, 256, 4096), (4, 300, 2056), (13, 7, 4096)],
                         ids=lambda s: "x".join(map(str, s)))
def test_dotmma_workspace_form(lib, shape, S, xr):
    M, N, K = shape
    p = lib.make_plan("dotmma_ws", threads=128, rows_per_cta=8, split_k=S, stages=xr)
    if not xr and _smem(M, K, S) > 200 * 1024:
        with pytest.raises(lib.BF16LinearError):
            lib.plan_check(M, N, K, p)
        return
    x, W, b = wl.make_inputs(M, N, K, S + M, True)
    got = tensor_bits(_ws_run(lib, x, W, b, p))
    check_close(got, oracle.linear_bf16(wl.bits(x), wl.bits(W), wl.bits(b)), f"dotmma_ws M={M} N={N} K={K} S={S}")
    # the same partial tiles summed in the same rank order as the cluster form with the same split
    if S <= 16:
        c = _plan(lib, S, 128, xr)
        assert np.array_equal(got, tensor_bits(_run(lib, x, W, b, c)))


def test_dotmma_workspace_needs_workspace(lib):
    p = lib.make_plan("dotmma_ws", threads=128, rows_per_cta=8, split_k=8)
    assert lib.workspace_size(16, 384, 7168, p) == 256 + 48 * 8 * 512
    x = torch.zeros(16, 7168, dtype=torch.bfloat16, device=DEV)
    W = torch.zeros(384, 7168, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(lib.BF16LinearError):
        lib.bf16_linear_with_plan(x, W, None, plan_=p)  # no workspace given


@pytest.mark.parametrize("shape", [(32, 2112, 7168), (64, 256, 4096), (17, 300, 1032), (50, 128, 2880)],
                         ids=lambda s: "x".join(map(str, s)))
def test_dotmma_token_groups(lib, shape):
    """More than 16 tokens: groups of 16 along grid.z, the last one ragged."""
    M, N, K = shape
    for xr in (0, 1):
        x, W, b = wl.make_inputs(M, N, K, M + N, True)
        got = tensor_bits(_run(lib, x, W, b, _plan(lib, 4, 256, xr)))
        want = oracle.linear_bf16(wl.bits(x), wl.bits(W), wl.bits(b))
        check_close(got, want, f"dotmma token groups M={M} N={N} K={K} xr={xr}")


def test_dotmma_deterministic_and_f32(lib):
    M, N, K = 14, 384, 7168
    x, W, b = wl.make_inputs(M, N, K, 2, True)
    p = _plan(lib, 8)
    a = tensor_bits(_run(lib, x, W, b, p))
    assert np.array_equal(a, tensor_bits(_run(lib, x, W, b, p)))
    f = _run(lib, x, W, b, p, f32=True)
    assert np.array_equal(tensor_bits(f.to(torch.bfloat16)), a)
    assert lib.device_status() == 0


def test_dotmma_exact_cases(lib):
    M, N, K = 16, 260, 2048
    _, W, b = wl.make_inputs(M, N, K, 3, True)
    ks = np.random.default_rng(5).integers(0, K, M)
    x = torch.zeros(M, K, dtype=torch.bfloat16)
    x[torch.arange(M), torch.from_numpy(ks)] = 1.0
    p = _plan(lib, 4)
    assert torch.equal(_run(lib, x, W, None, p).cpu(), W[:, torch.from_numpy(ks)].T.contiguous())
    assert torch.equal(_run(lib, torch.zeros_like(x), W, b, p).cpu(), b.expand(M, N))
    ones = _run(lib, torch.ones(M, K, dtype=torch.bfloat16), torch.ones(N, K, dtype=torch.bfloat16), None, p)
    assert (ones.cpu().float() == float(K)).all()


def test_dotmma_pdl_matches(lib):
    M, N, K = 12, 256, 6144
    x, W, b = wl.make_inputs(M, N, K, 9, False)
    p = _plan(lib, 4)
    ref = tensor_bits(_run(lib, x, W, None, p))
    p.flags = lib.FLAG_PDL
    xd, Wd = x.to(DEV), W.to(DEV)
    outs = [lib.bf16_linear_with_plan(xd, Wd, None, plan_=p) for _ in range(3)]
    torch.cuda.synchronize()
    for o in outs:
        assert np.array_equal(tensor_bits(o), ref)
