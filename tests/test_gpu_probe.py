"""The read-floor probe (bf16_linear_probe_read) reads every byte it is given once.

Its checksum (the XOR of all 32-bit words, one partial per CTA) must equal
numpy's over the same bytes, for buffer sizes that do and do not fill the unrolled main loop, and an
empty launch must leave the sink untouched.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.mark.parametrize("nbytes,grid,threads", [(16, 1, 32), (4096 * 16 + 48, 3, 64), (1 << 22, 152, 256),
                                                 ((1 << 20) + 16 * 7, 608, 128), (3 << 20, 152 * 4, 1024)])
def test_probe_checksum(lib, nbytes, grid, threads):
    rng = np.random.default_rng(nbytes)
    host = rng.integers(0, 2 ** 32, size=nbytes // 4, dtype=np.uint64).astype(np.uint32)
    src = torch.from_numpy(host.view(np.int32)).to(DEV)
    want = np.bitwise_xor.reduce(host)
    for flags in (0, lib.FLAG_SERIAL):  # the library's launch mode (L2 prefetch, PDL) and serial
        sink = torch.zeros(grid, dtype=torch.int32, device=DEV)
        lib.probe_read(src, grid, threads, sink, flags=flags)
        torch.cuda.synchronize()
        assert int(np.bitwise_xor.reduce(sink.cpu().numpy().view(np.uint32))) == int(want)


def test_probe_empty_launch(lib):
    sink = torch.full((152,), 1234, dtype=torch.int32, device=DEV)
    lib.probe_read(None, 152, 32, sink)
    torch.cuda.synchronize()
    assert bool((sink == 1234).all())
