"""Host-side checks of the C ABI that need no GPU: exports, plan(), validation."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")


def declared_functions():
    names = set()
    for fn in os.listdir(HEADER_DIR):
        if fn.endswith(".h"):
            text = open(os.path.join(HEADER_DIR, fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"^[A-Za-z_][\w \*]*?\b(bf16_linear\w*)\s*\(", text, flags=re.M))
    return sorted(names)


def test_header_declares_entry_points():
    names = declared_functions()
    for want in ("bf16_linear", "bf16_linear_plan", "bf16_linear_with_plan", "bf16_linear_strerror"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    so = ctypes.CDLL(lib.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(so, n)]
    assert not missing, f"declared but not exported: {missing}"


def test_version_and_strerror(lib):
    assert lib.version() >= 10000
    for st in range(0, -7, -1):
        assert lib.strerror(st) and lib.strerror(st) != "unknown status"
    assert lib.strerror(12345) == "unknown status"


# ---- plan(): the dispatch rules, on fake devices (no CUDA call is made) ----

def test_plan_refuses_other_architectures(lib):
    for dev in [(9, 0, 132), (10, 0, 148), (12, 0, 84), (10, 1, 100)]:
        with pytest.raises(lib.BF16LinearError) as e:
            lib.plan(4, 256, 2048, device=dev)
        assert e.value.status == -3


def test_plan_rejects_bad_sizes(lib):
    for s in [(-1, 4, 4), (1, 0, 4), (1, 4, 0), (1, -3, 4)]:
        with pytest.raises(lib.BF16LinearError) as e:
            lib.plan(*s)
        assert e.value.status == -1


def test_plan_size_rules(lib):
    # tiny M -> dot product (the pages' default rule M <= 4), any K % 8 != 0 -> dot product
    # (K = 3000 has no measured table entry, so the size rules decide)
    assert lib.plan(4, 256, 3000).kernel == lib.KERNEL_DOTPROD
    assert lib.plan(40, 256, 2881).kernel == lib.KERNEL_DOTPROD
    assert lib.plan(300, 256, 2881).kernel == lib.KERNEL_DOTPROD
    # large M -> tile kernel (K = 4104: no measured table entry, so the size rules decide)
    p = lib.plan(8192, 14336, 4104)
    assert p.kernel == lib.KERNEL_TILE and p.grid == 152
    p = lib.plan(8192, 14336, 4104, device=(10, 3, 100))
    assert p.grid == 100


def test_plan_m_zero_launches_nothing(lib):
    assert lib.plan(0, 256, 2048).grid == 0


def test_plan_is_valid_everywhere(lib):
    """Every plan the dispatcher returns for the workload shapes is a valid plan."""
    import workloads as wl
    pts = wl.router_sweep() + wl.decode_proj() + wl.mlp_bias() + wl.prefill() + wl.router_smallest()
    for pt in pts:
        p = lib.plan(pt["M"], pt["N"], pt["K"])
        assert p.grid > 0
        if p.kernel == lib.KERNEL_SPLITK:
            assert p.tokens_per_cta >= pt["M"] and p.tokens_per_cta % 8 == 0
            assert 1 <= p.split_k <= 16 and p.split_k <= -(-pt["K"] // 64)
            assert p.grid == p.split_k * -(-pt["N"] // p.rows_per_cta)
        if p.kernel == lib.KERNEL_DOTPROD:
            t = p.tokens_per_cta
            groups = 1 if t == 0 else -(-pt["M"] // min(t, pt["M"]))
            assert 0 <= t <= 8 and p.grid == -(-pt["N"] // p.rows_per_cta) * groups


# ---- bf16_linear(): argument validation happens before any CUDA call ----

def _raw(lib):
    return lib.load()


def test_validation_without_gpu(lib):
    L = _raw(lib)
    A = ctypes.c_void_p(0x10000)      # never dereferenced: rejected before any CUDA call
    B = ctypes.c_void_p(0x20000000)
    O = ctypes.c_void_p(0x40000000)
    # sizes
    assert L.bf16_linear(A, B, None, O, -1, 4, 8, None) == -1
    assert L.bf16_linear(A, B, None, O, 1, 0, 8, None) == -1
    assert L.bf16_linear(A, B, None, O, 1, 4, 0, None) == -1
    # M == 0: nothing to do
    assert L.bf16_linear(None, None, None, None, 0, 4, 8, None) == 0
    # NULL required pointers
    assert L.bf16_linear(None, B, None, O, 1, 4, 8, None) == -1
    assert L.bf16_linear(A, None, None, O, 1, 4, 8, None) == -1
    assert L.bf16_linear(A, B, None, None, 1, 4, 8, None) == -1
    # misalignment
    assert L.bf16_linear(ctypes.c_void_p(0x10008), B, None, O, 1, 4, 8, None) == -2
    assert L.bf16_linear(A, B, ctypes.c_void_p(0x30000002), O, 1, 4, 8, None) == -2
    # out overlapping an input
    assert L.bf16_linear(A, B, None, ctypes.c_void_p(0x10000), 1, 4, 8, None) == -1


def test_fp8_validation_and_split_without_gpu(lib):
    L = _raw(lib)
    A, B, O = ctypes.c_void_p(0x10000), ctypes.c_void_p(0x20000000), ctypes.c_void_p(0x40000000)
    S1, S2 = ctypes.c_void_p(0x50000000), ctypes.c_void_p(0x50000010)
    f = L.bf16_linear_fp8
    assert f(A, B, S1, S2, None, O, 0, 8, 64, 0, None) == 0            # M == 0: nothing to do
    assert f(A, B, S1, S2, None, O, -1, 8, 64, 0, None) == -1
    assert f(A, B, None, S2, None, O, 4, 8, 64, 0, None) == -1          # scales required
    assert f(A, B, S1, S2, None, O, 4, 8, 64, 4, None) == -1            # unknown flag
    assert f(A, B, S1, S2, None, O, 4, 8, 64, 3, None) == -1            # PDL with SERIAL
    assert f(ctypes.c_void_p(0x10008), B, S1, S2, None, O, 4, 8, 64, 0, None) == -2
    assert f(A, B, ctypes.c_void_p(0x50000002), S2, None, O, 4, 8, 64, 0, None) == -2
    assert f(A, B, S1, S2, None, O, 4, 8, 40, 0, None) == -6            # K % 16 != 0
    assert f(A, B, S1, S2, None, ctypes.c_void_p(0x10000), 4, 8, 64, 0, None) == -1  # out overlaps xq
    q = L.bf16_quant_fp8
    assert q(A, S1, O, 0, 0, None) == 0
    assert q(A, S1, O, -5, 0, None) == -1
    assert q(ctypes.c_void_p(0x10001), S1, O, 8, 0, None) == -2
    assert q(A, S1, ctypes.c_void_p(0x10004), 8, 0, None) == -1          # codes over their own input
    # K split: about two CTAs per SM, a power of two, at most 8 and one 64-code block each
    assert lib.fp8_split(16, 384, 7168) == 8       # 48 row groups x 8 >= 304
    assert lib.fp8_split(1, 14336, 4096) == 1      # 1792 row groups already
    assert lib.fp8_split(4, 8, 64) == 1            # a single 64-code block
    assert lib.fp8_split(4, 8, 4096, num_sms=1000) == 8


def test_forced_plan_rules_without_gpu(lib):
    L = _raw(lib)
    A, B, O = ctypes.c_void_p(0x10000), ctypes.c_void_p(0x20000000), ctypes.c_void_p(0x40000000)

    def run(M, N, K, **plan):
        p = lib.make_plan(**plan)
        return L.bf16_linear_with_plan(A, B, None, O, M, N, K, ctypes.byref(p), None)

    split = dict(kernel="splitk", threads=128, rows_per_cta=32, tokens_per_cta=16, split_k=4, stages=2)
    assert run(8, 256, 2049, **split) == -6            # TMA kernels need K % 8 == 0
    assert run(65, 256, 2048, **{**split, "tokens_per_cta": 64}) == -6  # split-K holds at most 64 tokens
    assert run(20, 256, 2048, **split) == -1           # tokens_per_cta < M
    assert run(8, 256, 2048, **{**split, "split_k": 17}) == -1
    assert run(8, 256, 128, **{**split, "split_k": 3}) == -1  # more CTAs than 64-wide K chunks
    assert run(8, 256, 2048, **{**split, "stages": 17}) == -1
    assert run(8, 256, 2048, **{**split, "tokens_per_cta": 12}) == -1   # not a multiple of 8
    assert run(8, 256, 2048, **{**split, "rows_per_cta": 24}) == -1     # no kernel for 24 rows
    assert run(8, 256, 2048, **{**split, "rows_per_cta": 512}) == -1
    assert run(8, 256, 2048, **{**split, "flags": 4}) == -1             # unknown launch flag
    assert run(8, 256, 2048, **{**split, "flags": 3}) == -1             # early weights with serial
    assert run(8, 256, 2048, kernel="dotprod", threads=96, rows_per_cta=2) == -1
    assert run(8, 256, 2048, kernel="dotprod", threads=128, rows_per_cta=3) == -1
    assert run(8, 256, 2048, kernel="tile", threads=192, rows_per_cta=256, tokens_per_cta=128, stages=9) == -1
    assert run(8, 256, 2049, kernel="tile", threads=192, rows_per_cta=256, tokens_per_cta=128, stages=4) == -6
    p = lib.make_plan(kernel=7)
    assert L.bf16_linear_with_plan(A, B, None, O, 8, 256, 2048, ctypes.byref(p), None) == -1
    assert L.bf16_linear_with_plan(A, B, None, O, 8, 256, 2048, None, None) == -1


def test_plan_check_accepts_and_rejects(lib):
    p = lib.make_plan("splitk", threads=128, rows_per_cta=64, tokens_per_cta=16, split_k=16, stages=7)
    assert lib.plan_check(16, 256, 7168, p).grid == 64
    with pytest.raises(lib.BF16LinearError):
        lib.plan_check(16, 256, 7168, lib.make_plan("splitk", threads=128, rows_per_cta=64, tokens_per_cta=16,
                                                    split_k=16, stages=40))
    with pytest.raises(lib.BF16LinearError):
        lib.plan_check(16, 256, 7168, p, device=(9, 0, 132))
    # every plan the dispatcher makes passes its own check
    for (M, N, K) in [(1, 256, 2048), (16, 384, 7168), (64, 2112, 7168), (300, 1000, 520), (5, 7, 9)]:
        q = lib.plan(M, N, K)
        assert lib.plan_check(M, N, K, q).grid == q.grid


def test_dotprod_token_groups_on_cpu(lib):
    # ceil(N / R) row slices x ceil(M / t) token groups
    assert lib.plan_check(16, 256, 7168, lib.make_plan("dotprod", threads=128, rows_per_cta=2,
                                                       tokens_per_cta=8)).grid == 128 * 2
    assert lib.plan_check(13, 256, 7168, lib.make_plan("dotprod", threads=128, rows_per_cta=1,
                                                       tokens_per_cta=4)).grid == 256 * 4
    assert lib.plan_check(3, 256, 7168, lib.make_plan("dotprod", threads=128, rows_per_cta=1,
                                                      tokens_per_cta=8)).grid == 256
    # 0 = one CTA row looping over groups of 8
    assert lib.plan_check(16, 256, 7168, lib.make_plan("dotprod", threads=128, rows_per_cta=2)).grid == 128
    for bad in (-1, 9):
        with pytest.raises(lib.BF16LinearError):
            lib.plan_check(16, 256, 7168, lib.make_plan("dotprod", threads=128, rows_per_cta=2, tokens_per_cta=bad))


def test_pair_tile_plans_on_cpu(lib):
    p = lib.make_plan("tile2", threads=192, rows_per_cta=256, tokens_per_cta=256, stages=6)
    # 8 x 28 pair tiles of 256 x 256; 76 clusters of 2 on 152 SMs
    assert lib.plan_check(2048, 7168, 7168, p).grid == 152
    assert lib.plan_check(256, 256, 64, p).grid == 2
    assert lib.plan_check(300, 300, 64, p).grid == 2 * 2 * 2
    p192 = lib.make_plan("tile2", threads=192, rows_per_cta=192, tokens_per_cta=256, stages=6)
    assert lib.plan_check(256, 14336, 4096, p192).grid == 150  # 75 pair tiles of 256 x 192
    for bad in (dict(stages=7), dict(stages=1), dict(rows_per_cta=128), dict(rows_per_cta=224), dict(tokens_per_cta=128),
                dict(threads=128)):
        q = lib.make_plan("tile2", **dict(dict(threads=192, rows_per_cta=256, tokens_per_cta=256, stages=4), **bad))
        with pytest.raises(lib.BF16LinearError):
            lib.plan_check(2048, 7168, 7168, q)
    with pytest.raises(lib.BF16LinearError):
        lib.plan_check(2048, 7168, 7161, p)  # TMA needs K % 8 == 0


def test_warprow_plans_on_cpu(lib):
    mk = lambda t, w, c: lib.make_plan("warprow", threads=t, rows_per_cta=w, stages=c)
    assert lib.plan_check(1, 2112, 7168, mk(512, 2, 2)).grid == 304
    assert lib.plan_check(1, 100, 7168, mk(512, 2, 2)).grid == 100  # never more CTAs than rows
    assert lib.plan_check(1, 2112, 7168, mk(128, 2, 8)).grid == 1216  # eight 128-thread CTAs per SM
    for bad in (mk(64, 1, 1), mk(512, 3, 1), mk(1024, 1, 3), mk(512, 1, 5), mk(256, 1, 0), mk(128, 8, 1),
                mk(128, 1, 9)):
        with pytest.raises(lib.BF16LinearError):
            lib.plan_check(4, 2112, 7168, bad)
    with pytest.raises(lib.BF16LinearError):
        lib.plan_check(9, 2112, 7168, mk(512, 1, 1))   # at most 8 tokens
    with pytest.raises(lib.BF16LinearError):
        lib.plan_check(4, 2112, 7170, mk(512, 1, 1))   # 16-byte vectors need K % 8 == 0
    with pytest.raises(lib.BF16LinearError):
        lib.plan_check(8, 64, 16384, mk(512, 1, 1))    # x does not fit in shared memory


def test_warpmma_plans_on_cpu(lib):
    mk = lambda t, w, c: lib.make_plan("warpmma", threads=t, rows_per_cta=w, stages=c)
    assert lib.plan_check(16, 14336, 4096, mk(1024, 4, 1)).grid == 152
    assert lib.plan_check(4, 2112, 7168, mk(512, 4, 2)).grid == 264  # 264 groups of 8 rows < 304 CTAs
    assert lib.plan_check(1, 2112, 4096, mk(128, 4, 8)).grid == 264  # eight 128-thread CTAs per SM, 264 groups
    for bad in (mk(512, 3, 1), mk(256, 16, 1), mk(1024, 2, 1), mk(1024, 1, 2), mk(512, 1, 0), mk(64, 1, 1),
                mk(128, 8, 1), mk(128, 1, 9)):
        with pytest.raises(lib.BF16LinearError):
            lib.plan_check(4, 2112, 7168, bad)
    xr2 = lib.make_plan("warpmma", threads=256, rows_per_cta=8, stages=2, split_k=1, tokens_per_cta=2)
    assert lib.plan_check(16, 2112, 7168, xr2).grid == 132  # 16-row slabs: 132 < 304 CTAs
    for bad in (lib.make_plan("warpmma", threads=256, rows_per_cta=8, stages=2, split_k=0, tokens_per_cta=2),
                lib.make_plan("warpmma", threads=256, rows_per_cta=8, stages=2, split_k=1, tokens_per_cta=3),
                lib.make_plan("warpmma", threads=256, rows_per_cta=8, stages=2, split_k=1, tokens_per_cta=8)):
        with pytest.raises(lib.BF16LinearError):
            lib.plan_check(4, 2112, 7168, bad)           # several groups per warp only with x from L2; 1, 2 or 4
    with pytest.raises(lib.BF16LinearError):
        lib.plan_check(17, 2112, 4096, mk(512, 1, 1))   # at most 16 tokens
    with pytest.raises(lib.BF16LinearError):
        lib.plan_check(16, 2112, 7168, mk(512, 1, 1))   # x (229 KB) does not fit in shared memory


def test_host_staging_bytes(lib):
    # x, W, (bias,) out at 256-byte aligned offsets
    assert lib.host_staging_bytes(4, 256, 2048, False) == 16384 + 1048576 + 2048
    assert lib.host_staging_bytes(4, 256, 2048, True) == 16384 + 1048576 + 512 + 2048
    assert lib.host_staging_bytes(3, 5, 8, True) == 4 * 256
    assert lib.host_staging_bytes(0, 5, 8, False) == 256  # W only
    for bad in ((-1, 5, 8), (3, 0, 8), (3, 5, 0)):
        assert lib.host_staging_bytes(*bad, False) == 0


def test_warpmma_cluster_plans_on_cpu(lib):
    mk = lambda t, w, c, S: lib.make_plan("warpmma", threads=t, rows_per_cta=w, stages=c, split_k=S)
    assert lib.plan_check(16, 2112, 7168, mk(1024, 8, 1, 2)).grid == 152   # 76 clusters of 2
    assert lib.plan_check(64, 2112, 7168, mk(512, 4, 1, 8)).grid == 152    # 19 clusters of 8
    assert lib.plan_check(32, 2112, 7168, mk(256, 2, 2, 8)).grid == 304    # two 256-thread CTAs per SM
    assert lib.plan_check(5, 24, 4096, mk(512, 4, 1, 2)).grid == 6         # no more clusters than row groups
    assert lib.plan_check(16, 2112, 7168, mk(256, 2, 4, 16)).grid == 608  # 38 clusters of 16
    g4 = mk(256, 2, 4, 16)
    g4.tokens_per_cta = 4
    assert lib.plan_check(16, 256, 7168, g4).grid == 8 * 16              # 4 of the 32 row groups per cluster
    for bad in (mk(1024, 8, 1, 17), mk(512, 3, 1, 2), mk(512, 8, 0, 2), mk(512, 8, 3, 2), mk(1024, 2, 1, 2)):
        with pytest.raises(lib.BF16LinearError):
            lib.plan_check(16, 2112, 7168, bad)
    with pytest.raises(lib.BF16LinearError):
        lib.plan_check(32, 2112, 7168, mk(1024, 8, 1, 4))   # more than 16 tokens: at most 512 threads per SM
    with pytest.raises(lib.BF16LinearError):
        lib.plan_check(32, 2112, 7168, mk(512, 8, 2, 4))
    with pytest.raises(lib.BF16LinearError):
        lib.plan_check(65, 2112, 7168, mk(512, 4, 1, 8))    # at most 64 tokens
    with pytest.raises(lib.BF16LinearError):
        lib.plan_check(64, 2112, 7168, mk(512, 4, 1, 2))    # a 466 KB x slice does not fit
    with pytest.raises(lib.BF16LinearError):
        lib.plan_check(16, 2112, 7168, mk(512, 8, 2, 2))    # two 127 KB CTAs do not fit one SM
    with pytest.raises(lib.BF16LinearError):
        lib.plan_check(4, 64, 32, mk(512, 4, 1, 2))         # one 32-wide K block cannot be split


def test_dotmma_plans_on_cpu(lib):
    mk = lambda t, S: lib.make_plan("dotmma", threads=t, rows_per_cta=8, split_k=S)
    assert lib.plan_check(16, 384, 7168, mk(256, 4)).grid == 4 * 48
    assert lib.plan_check(3, 7, 4096, mk(128, 8)).grid == 8
    assert lib.plan_check(16, 384, 7168, mk(256, 16)).grid == 16 * 48
    for bad in (mk(512, 4), mk(256, 3), mk(256, 32), lib.make_plan("dotmma", threads=256, rows_per_cta=16, split_k=2),
                lib.make_plan("dotmma", threads=256, rows_per_cta=8, split_k=4, stages=2)):
        with pytest.raises(lib.BF16LinearError):
            lib.plan_check(16, 384, 7168, bad)
    with pytest.raises(lib.BF16LinearError):
        lib.plan_check(16, 384, 7168, mk(256, 1))   # x (229 KB) does not fit one CTA's shared memory
    xr = lib.make_plan("dotmma", threads=256, rows_per_cta=8, split_k=1, stages=1)
    assert lib.plan_check(16, 384, 7168, xr).grid == 48  # ... but x straight from L2 needs none
    assert lib.plan_check(17, 384, 4096, xr).grid == 48 * 2       # two groups of 16 tokens along grid.z
    assert lib.plan_check(64, 384, 4096, mk(256, 4)).grid == 4 * 48 * 4
    with pytest.raises(lib.BF16LinearError):
        lib.plan_check(65, 384, 4096, mk(256, 4))   # at most 64 tokens (4 groups)
    with pytest.raises(lib.BF16LinearError):
        lib.plan_check(17, 384, 4096, lib.make_plan("dotmma_ws", threads=256, rows_per_cta=8, split_k=4))
    with pytest.raises(lib.BF16LinearError):
        lib.plan_check(4, 384, 40, mk(256, 4))      # two 32-wide K blocks cannot feed 4 CTAs


def test_workspace_plans_on_cpu(lib):
    import ctypes
    p = lib.make_plan("splitk_ws", threads=128, rows_per_cta=64, tokens_per_cta=16, split_k=64, stages=2)
    assert lib.plan_check(16, 256, 7168, p).grid == 64 * 4
    with pytest.raises(lib.BF16LinearError):
        lib.plan_check(16, 256, 7168, lib.make_plan("splitk_ws", threads=128, rows_per_cta=64, tokens_per_cta=16,
                                                    split_k=65, stages=2))
    # counters (4 tiles, rounded up to 256 bytes) + partials [tiles][S][M][rows] fp32
    assert lib.workspace_size(16, 256, 7168, p) == 256 + 4 * 64 * 16 * 64 * 4
    assert lib.workspace_size(16, 256, 7168, lib.make_plan("dotprod", threads=128, rows_per_cta=2)) == 0
    # the dispatcher never needs a workspace it was not given
    assert lib.workspace_size(16, 256, 7168, lib.plan(16, 256, 7168)) == 0
    # a misaligned workspace is rejected before any CUDA call
    L = lib.load()
    c = lib.Call()
    c.x, c.W, c.out = 0x10000, 0x20000000, 0x40000000
    c.M, c.N, c.K = 16, 256, 7168
    c.workspace, c.workspace_bytes = 0x50000010, 1 << 20
    assert L.bf16_linear_run(ctypes.byref(c)) == -2
    assert L.bf16_linear_run(None) == -1


def test_probe_read_validates_before_touching_a_device(lib):
    import ctypes as C
    L = lib.load()
    for bytes_, grid, threads in [(17, 1, 32), (16, 0, 32), (16, 1, 48), (16, 1, 2048), (16, 1, 0)]:
        assert L.bf16_linear_probe_read(C.c_void_p(4096), bytes_, grid, threads, C.c_void_p(8192), 0, None) == -1
    assert L.bf16_linear_probe_read(None, 16, 1, 32, C.c_void_p(8192), 0, None) == -1   # NULL src with bytes
    assert L.bf16_linear_probe_read(C.c_void_p(4104), 16, 1, 32, C.c_void_p(8192), 0, None) == -2  # misaligned
    for bad_flags in (1, 4):  # only the serial flag applies
        assert L.bf16_linear_probe_read(C.c_void_p(4096), 16, 1, 32, C.c_void_p(8192), bad_flags, None) == -1


def test_tile_tactic_space(lib):
    """Plain tile widths 128..256 and swap-AB token widths 32..256; rings as deep as fit 227 KB (8 at
    most); any other width, or the wrong fixed side, is refused."""
    mk = lambda k, **f: lib.make_plan(k, **dict(dict(threads=192), **f))
    for bn, most in ((128, 7), (192, 5), (224, 5), (240, 4), (256, 4)):
        p = mk("tile", rows_per_cta=bn, tokens_per_cta=128, stages=most, split_k=2)
        assert lib.plan_check(2048, 7168, 7168, p).grid == 152
        with pytest.raises(lib.BF16LinearError):
            lib.plan_check(2048, 7168, 7168, mk("tile", rows_per_cta=bn, tokens_per_cta=128, stages=most + 1))
    for bn, most in ((32, 8), (64, 8), (128, 7), (192, 5), (256, 4)):
        p = mk("tile_t", rows_per_cta=128, tokens_per_cta=bn, stages=most)
        # 14336 / 128 = 112 W tiles times ceil(64 / bn) token tiles
        assert lib.plan_check(64, 14336, 4096, p).grid == min(152, 112 * -(-64 // bn))
    for bad in (mk("tile", rows_per_cta=160, tokens_per_cta=128, stages=4),
                mk("tile", rows_per_cta=256, tokens_per_cta=64, stages=4),
                mk("tile_t", rows_per_cta=256, tokens_per_cta=64, stages=4),
                mk("tile_t", rows_per_cta=128, tokens_per_cta=48, stages=4),
                mk("tile_t", rows_per_cta=128, tokens_per_cta=64, stages=1),
                mk("tile", rows_per_cta=256, tokens_per_cta=128, stages=4, split_k=-1)):
        with pytest.raises(lib.BF16LinearError):
            lib.plan_check(256, 14336, 4096, bad)
    with pytest.raises(lib.BF16LinearError) as e:  # K % 8 != 0: a TMA kernel cannot run it
        lib.plan_check(256, 1024, 1001, mk("tile_t", rows_per_cta=128, tokens_per_cta=64, stages=4))
    assert e.value.status == -6


def test_two_chunk_stage_rules(lib):
    """chunks_per_stage: 0 or 1 is one 64-wide K chunk per ring stage, 2 is two (the ring kernels only, K a
    multiple of 64); the stage count then counts double stages against the same shared memory, and a
    split-K plan may not have more ranks than double stages."""
    mk = lambda k, **f: lib.make_plan(k, **f)
    tile = dict(threads=192, rows_per_cta=192, tokens_per_cta=128)
    assert lib.plan_check(256, 14336, 4096, mk("tile", stages=2, chunks_per_stage=2, **tile)).grid == 150
    with pytest.raises(lib.BF16LinearError):  # 3 double stages of 40 KB chunks do not fit 227 KB
        lib.plan_check(256, 14336, 4096, mk("tile", stages=3, chunks_per_stage=2, **tile))
    tt = dict(threads=192, rows_per_cta=128, tokens_per_cta=64)
    assert lib.plan_check(64, 14336, 4096, mk("tile_t", stages=4, chunks_per_stage=2, **tt)).grid == 112
    with pytest.raises(lib.BF16LinearError):
        lib.plan_check(64, 14336, 4096, mk("tile_t", stages=5, chunks_per_stage=2, **tt))
    sk = dict(threads=128, rows_per_cta=64, tokens_per_cta=16)
    assert lib.plan_check(16, 2112, 7168, mk("splitk", split_k=8, stages=4, chunks_per_stage=2, **sk)).grid == 264
    # 2880 = 45 chunks = 23 double stages: 23 ranks at most
    assert lib.plan_check(1, 128, 2880, mk("splitk_ws", split_k=23, stages=1, chunks_per_stage=2, **sk)).grid == 46
    with pytest.raises(lib.BF16LinearError):
        lib.plan_check(1, 128, 2880, mk("splitk_ws", split_k=24, stages=1, chunks_per_stage=2, **sk))
    assert lib.plan_check(1, 128, 2880, mk("splitk_ws", split_k=45, stages=1, **sk)).grid == 90
    for bad in (dict(chunks_per_stage=3), dict(chunks_per_stage=-1)):
        with pytest.raises(lib.BF16LinearError):
            lib.plan_check(16, 2112, 7168, mk("splitk", split_k=8, stages=2, **dict(sk, **bad)))
    for other in (mk("dotprod", threads=128, rows_per_cta=2, chunks_per_stage=2),
                  mk("tile2", threads=192, rows_per_cta=256, tokens_per_cta=256, stages=4, chunks_per_stage=2),
                  mk("dotmma", threads=128, rows_per_cta=8, split_k=4, stages=1, chunks_per_stage=2)):
        with pytest.raises(lib.BF16LinearError) as e:
            lib.plan_check(16, 2112, 7168, other)
        assert e.value.status == -1
    with pytest.raises(lib.BF16LinearError) as e:  # K % 64 != 0: no chunked view of the matrices
        lib.plan_check(16, 2112, 7176, mk("splitk", split_k=8, stages=2, chunks_per_stage=2, **sk))
    assert e.value.status == -6
    assert lib.plan_check(16, 2112, 7176, mk("splitk", split_k=8, stages=2, chunks_per_stage=1, **sk)).grid == 264
    # the dispatcher's plans always pass their own check, whatever chunks they carry
    for (M, N, K) in [(16, 2112, 7168), (64, 14336, 4096), (256, 14336, 4096), (32, 2112, 7168)]:
        q = lib.plan(M, N, K)
        assert q.chunks_per_stage in (0, 1, 2)
        assert lib.plan_check(M, N, K, q).grid == q.grid


def test_launch_flags_validated_without_gpu(lib):
    """Unknown flag bits, and the early-weights mode together with the serial one, are refused before any
    CUDA call; the plan check applies the same rule to a plan's flags."""
    import ctypes as C
    L = lib.load()
    x, W, o = C.c_void_p(1 << 16), C.c_void_p(1 << 29), C.c_void_p(1 << 30)
    for bad in (4, 3, 0x80000000):
        assert L.bf16_linear_ex(x, W, None, o, 4, 256, 2048, bad, None) == -1
        assert L.bf16_quant_fp8(x, C.c_void_p(1 << 20), o, 64, bad, None) == -1
    p = lib.make_plan("dotprod", threads=128, rows_per_cta=2)
    for ok in (0, lib.FLAG_PDL, lib.FLAG_SERIAL):
        p.flags = ok
        lib.plan_check(4, 256, 2048, p)
    p.flags = lib.FLAG_PDL | lib.FLAG_SERIAL
    with pytest.raises(lib.BF16LinearError):
        lib.plan_check(4, 256, 2048, p)


def test_mxfp8_validation_and_split_without_gpu(lib):
    import ctypes as C
    L = lib.load()
    A, S1, B, S2, O = (C.c_void_p(v) for v in (1 << 16, 1 << 18, 1 << 20, 1 << 22, 1 << 24))
    f = L.bf16_linear_mxfp8
    assert f(A, S1, B, S2, None, O, 4, 8, 80, 0, None) == -6        # K % 32 != 0
    assert f(A, S1, B, S2, None, O, -1, 8, 64, 0, None) == -1
    assert f(A, S1, B, S2, None, O, 4, 8, 64, 3, None) == -1         # PDL with SERIAL
    assert f(C.c_void_p((1 << 16) + 8), S1, B, S2, None, O, 4, 8, 64, 0, None) == -2
    assert f(None, S1, B, S2, None, O, 4, 8, 64, 0, None) == -1
    assert f(A, S1, B, S2, None, O, 0, 8, 64, 0, None) == 0          # M == 0: nothing to do
    q = L.bf16_quant_mxfp8
    assert q(A, 4, 48, B, S2, 0, None) == -6
    assert q(A, -1, 64, B, S2, 0, None) == -1
    assert q(A, 4, 64, C.c_void_p(1 << 16), S2, 0, None) == -1      # codes overlap the input
    # the split: a power of two, at most 16, at least one scale block per warp
    for M, N, K in [(1, 256, 7168), (16, 384, 7168), (8, 14336, 4096), (64, 2112, 7168), (3, 8, 64)]:
        s = lib.mxfp8_split(M, N, K)
        assert s in (1, 2, 4, 8, 16) and s * 4 <= max(4, K // 32)
