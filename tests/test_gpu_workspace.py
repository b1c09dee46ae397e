"""The cluster-free split-K kernel (BF16L_KERNEL_SPLITK_WS): partial tiles reduced
through a caller-provided workspace by the last CTA to arrive."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tolerance import check_close, tensor_bits

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def ws_plan(lib, M, rows, split, stages, tokens=None):
    return lib.make_plan("splitk_ws", threads=128, rows_per_cta=rows,
                         tokens_per_cta=tokens or max(8, -(-M // 8) * 8), split_k=split, stages=stages)


CASES = [
    # M, N, K, rows, split, stages
    (16, 256, 7168, 64, 32, 4),
    (9, 384, 7168, 32, 16, 7),
    (1, 128, 2880, 16, 45, 1),       # one chunk per CTA, 45 CTAs along K
    (64, 2112, 7168, 128, 16, 7),    # N tail
    (5, 130, 200, 48, 2, 2),         # ragged everything
    (33, 1000, 4096, 256, 8, 4),
    (12, 256, 6144, 64, 64, 2),      # the deepest split
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_workspace_splitk_parity(lib, case):
    M, N, K, rows, split, stages = case
    p = ws_plan(lib, M, rows, split, stages)
    ws = lib.new_workspace(lib.workspace_size(M, N, K, p), DEV)
    for bias in (False, True):
        x, W, b = wl.make_inputs(M, N, K, M + N + split, bias)
        xd, Wd = x.to(DEV), W.to(DEV)
        bd = b.to(DEV) if b is not None else None
        outs = [tensor_bits(lib.run(xd, Wd, bd, plan_=p, workspace=ws)) for _ in range(3)]
        torch.cuda.synchronize()
        want = oracle.linear_bf16(wl.bits(x), wl.bits(W), wl.bits(b))
        check_close(outs[0], want, f"workspace split-K {case} bias={bias}")
        assert all(np.array_equal(outs[0], o) for o in outs[1:]), "not deterministic across calls"
        # fp32 logits through the same plan, rounded to bf16, equal the bf16 result bit for bit
        o32 = lib.run(xd, Wd, bd, plan_=p, workspace=ws, out_f32=True)
        assert torch.equal(o32.to(torch.bfloat16).cpu(), torch.from_numpy(outs[0].view(np.int16)).view(torch.bfloat16))
    # every completed call leaves the arrival counters at zero
    tiles = -(-N // rows)
    assert int(ws[: 4 * tiles].view(torch.int32).abs().sum().item()) == 0


def test_workspace_exact_cases(lib):
    M, N, K = 7, 300, 2048
    p = ws_plan(lib, M, 32, 16, 2)
    ws = lib.new_workspace(lib.workspace_size(M, N, K, p), DEV)
    _, W, b = wl.make_inputs(M, N, K, 3, True)
    x = torch.zeros(M, K, dtype=torch.bfloat16)
    ks = np.random.default_rng(2).integers(0, K, M)
    x[torch.arange(M), torch.from_numpy(ks)] = 1.0
    got = tensor_bits(lib.run(x.to(DEV), W.to(DEV), plan_=p, workspace=ws))
    assert np.array_equal(got, wl.bits(W)[:, ks].T)
    got = tensor_bits(lib.run(torch.zeros_like(x).to(DEV), W.to(DEV), b.to(DEV), plan_=p, workspace=ws))
    assert np.array_equal(got, np.broadcast_to(wl.bits(b), (M, N)))


def test_workspace_errors(lib):
    M, N, K = 16, 256, 2048
    x = torch.randn(M, K, device=DEV).to(torch.bfloat16)
    W = torch.randn(N, K, device=DEV).to(torch.bfloat16)
    p = ws_plan(lib, M, 64, 8, 4)
    need = lib.workspace_size(M, N, K, p)
    with pytest.raises(lib.BF16LinearError) as e:
        lib.run(x, W, plan_=p)                                   # no workspace
    assert e.value.status == -1
    with pytest.raises(lib.BF16LinearError) as e:
        lib.run(x, W, plan_=p, workspace=lib.new_workspace(need - 256, DEV))   # too small
    assert e.value.status == -1
    big = lib.new_workspace(need + 512, DEV)
    with pytest.raises(lib.BF16LinearError) as e:
        lib.run(x, W, plan_=p, workspace=big[16:])               # not 256-byte aligned
    assert e.value.status == -2
    lib.run(x, W, plan_=p, workspace=big)                       # fine


def test_dispatcher_with_workspace_matches_oracle(lib):
    """With a workspace the dispatcher may choose the cluster-free plan; results stay in tolerance."""
    for (M, N, K) in [(16, 256, 7168), (64, 2112, 7168), (8, 14336, 4096)]:
        x, W, _ = wl.make_inputs(M, N, K, 9, False)
        ws = lib.new_workspace(max(256, lib.workspace_size(M, N, K)), DEV)
        got = tensor_bits(lib.run(x.to(DEV), W.to(DEV), workspace=ws))
        check_close(got, oracle.linear_bf16(wl.bits(x), wl.bits(W)), f"dispatcher+workspace {M},{N},{K}")
