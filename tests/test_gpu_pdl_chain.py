"""Programmatic dependent launch across a real producer -> consumer chain.

Every launch of the library uses programmatic dependent launch unless told
otherwise: the kernel may start before the previous kernel on its stream has
finished and waits for it before reading anything (the default), or, with
BF16L_FLAG_PDL, reads W (and issues its weight copies) early and only x and out
wait.  The hazard either mode brings in is a consumer reading its x before the
producer has written it, or writing its out while the producer still reads it.
Each case here chains two launches on one stream:

    A (the dispatcher's plan):  y  = x0 @ W1^T          y [M, K1]
    B (one kernel family):      x0 = y @ W2^T + b2      B's out overwrites A's input

so B reads what A writes (read after write) and writes what A reads (write after
read).  A runs with BF16L_FLAG_PDL; B runs in each mode (early weights, and the
default).  y is poisoned before A runs.  The results are checked against the
oracle: A's output against oracle(x0, W1), B's output against the oracle applied
to A's GPU output and against the oracle applied to A's oracle output.  The same
chain also runs as a captured CUDA graph, replayed with fresh inputs.  The
kernel families are every kernel that honours the flag.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tolerance import check_close, tensor_bits

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
POISON = 3.0e4  # what a read of y before A wrote it would see


def _families(lib):
    mk = lib.make_plan
    # name: (plan, M, K0 = N of B, K1 = N of A = K of B)
    return {
        "dotprod": (mk("dotprod", threads=128, rows_per_cta=2), 4, 256, 2048),
        "dotprod_x_l2": (mk("dotprod", threads=128, rows_per_cta=2, stages=1), 3, 256, 2048),
        "dotprod_groups": (mk("dotprod", threads=128, rows_per_cta=2, tokens_per_cta=4), 11, 256, 2048),
        "stream": (mk("stream", threads=288, rows_per_cta=2, stages=4), 4, 256, 2048),
        "warprow": (mk("warprow", threads=512, rows_per_cta=1, stages=2), 2, 2112, 2048),
        "warpmma": (mk("warpmma", threads=512, rows_per_cta=4, stages=2), 8, 2112, 2048),
        "warpmma_x_l2": (mk("warpmma", threads=512, rows_per_cta=8, stages=1, split_k=1, tokens_per_cta=2),
                         16, 2112, 2048),
        "warpmma_cluster": (mk("warpmma", threads=256, rows_per_cta=2, stages=4, split_k=4), 16, 384, 2048),
        "warpmma_cluster_m40": (mk("warpmma", threads=256, rows_per_cta=2, stages=2, split_k=4), 40, 384, 2048),
        "dotmma": (mk("dotmma", threads=128, rows_per_cta=8, split_k=4, stages=0), 12, 256, 2048),
        "dotmma_x_l2": (mk("dotmma", threads=128, rows_per_cta=8, split_k=4, stages=1), 16, 256, 2048),
        "dotmma_m40": (mk("dotmma", threads=128, rows_per_cta=8, split_k=4, stages=1), 40, 256, 2048),
        "dotmma_ws": (mk("dotmma_ws", threads=128, rows_per_cta=8, split_k=8, stages=0), 12, 256, 2048),
        "splitk": (mk("splitk", threads=128, rows_per_cta=32, tokens_per_cta=16, split_k=4, stages=4), 16, 256, 2048),
        "splitk_ws": (mk("splitk_ws", threads=128, rows_per_cta=32, tokens_per_cta=16, split_k=8, stages=4),
                      16, 256, 2048),
        "tile": (mk("tile", threads=192, rows_per_cta=256, tokens_per_cta=128, stages=4), 256, 512, 1024),
        "tile2": (mk("tile2", threads=192, rows_per_cta=256, tokens_per_cta=256, stages=4), 256, 512, 1024),
        "tile_t": (mk("tile_t", threads=192, rows_per_cta=128, tokens_per_cta=64, stages=4), 64, 512, 1024),
    }


NAMES = ["dotprod", "dotprod_x_l2", "dotprod_groups", "stream", "warprow", "warpmma", "warpmma_x_l2",
         "warpmma_cluster", "warpmma_cluster_m40", "dotmma", "dotmma_x_l2", "dotmma_m40", "dotmma_ws", "splitk",
         "splitk_ws", "tile", "tile2", "tile_t"]


def test_family_list_is_complete(lib):
    """Every kernel the library launches appears in the chain."""
    fams = _families(lib)
    assert sorted(fams) == sorted(NAMES)
    kernels = {lib.KERNEL_NAMES[p.kernel] for p, *_ in fams.values()}
    assert kernels == set(lib.KERNEL_NAMES.values())


class Chain:
    def __init__(self, lib, name, seed, flags):
        plan, M, K0, K1 = _families(lib)[name]
        self.lib, self.name, self.M, self.K0, self.K1 = lib, name, M, K0, K1
        self.plan = plan
        self.plan.flags = flags
        lib.plan_check(M, K0, K1, self.plan)  # B: x[M, K1] @ W2[K0, K1]^T
        _, W1, _ = wl.make_inputs(1, K1, K0, seed, False)
        _, W2, b2 = wl.make_inputs(1, K0, K1, seed + 1, True)
        self.W1, self.W2, self.b2 = W1, W2, b2
        self.W1d, self.W2d, self.b2d = W1.to(DEV), W2.to(DEV), b2.to(DEV)
        self.x0 = torch.empty(M, K0, dtype=torch.bfloat16, device=DEV)
        self.src = torch.empty(M, K0, dtype=torch.bfloat16, device=DEV)
        self.y = torch.empty(M, K1, dtype=torch.bfloat16, device=DEV)
        self.ws = lib.new_workspace(max(256, lib.workspace_size(M, K0, K1, self.plan)), DEV)

    def enqueue(self, stream):
        """x0 <- src; poison y; A; B: four launches on `stream`, the last two with PDL."""
        with torch.cuda.stream(stream):
            self.x0.copy_(self.src)
            self.y.fill_(POISON)
            self.lib.bf16_linear_ex(self.x0, self.W1d, None, out=self.y, flags=self.lib.FLAG_PDL, stream=stream)
            self.lib.run(self.y, self.W2d, self.b2d, self.x0, plan_=self.plan, workspace=self.ws, stream=stream)

    def check(self, x_in):
        y_gpu = tensor_bits(self.y)
        out = tensor_bits(self.x0)
        y_want = oracle.linear_bf16(wl.bits(x_in), wl.bits(self.W1), None)
        check_close(y_gpu, y_want, f"{self.name}: A's output (x0 read before B overwrote it)")
        b_bits = wl.bits(self.b2)
        check_close(out, oracle.linear_bf16(y_gpu, wl.bits(self.W2), b_bits),
                    f"{self.name}: B on A's GPU output (y read after A wrote it)")
        check_close(out, oracle.linear_bf16(y_want, wl.bits(self.W2), b_bits),
                    f"{self.name}: B on A's oracle output")


def _fresh_x(M, K0, seed):
    x, _, _ = wl.make_inputs(M, 1, K0, seed, False)
    return x


MODES = {"early_weights": 1, "default": 0}


@pytest.mark.parametrize("mode", list(MODES))
@pytest.mark.parametrize("name", NAMES)
def test_pdl_chain(lib, name, mode):
    ch = Chain(lib, name, seed=37 * NAMES.index(name), flags=MODES[mode])
    stream = torch.cuda.Stream(DEV)
    for rep in range(2):
        x = _fresh_x(ch.M, ch.K0, 100 + rep)
        ch.src.copy_(x.to(DEV))
        torch.cuda.synchronize()
        ch.enqueue(stream)
        stream.synchronize()
        ch.check(x)
    assert lib.device_status() == 0


@pytest.mark.parametrize("mode", list(MODES))
@pytest.mark.parametrize("name", NAMES)
def test_pdl_chain_in_graph(lib, name, mode):
    ch = Chain(lib, name, seed=500 + 37 * NAMES.index(name), flags=MODES[mode])
    stream = torch.cuda.Stream(DEV)
    ch.src.copy_(_fresh_x(ch.M, ch.K0, 7).to(DEV))
    torch.cuda.synchronize()
    ch.enqueue(stream)  # initialise outside the capture
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        ch.enqueue(stream)
    for rep in range(2):
        x = _fresh_x(ch.M, ch.K0, 200 + rep)
        ch.src.copy_(x.to(DEV))
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            g.replay()
        stream.synchronize()
        ch.check(x)
    assert lib.device_status() == 0
