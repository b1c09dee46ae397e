"""Pins for the oracle's MXFP8 functions, and planted mistakes they catch.

What fixes each function, independently of the oracle:
  * E8M0 decoding: 2^(e - 127) as an exact rational, for all 256 bytes (255 NaN);
  * block quantisation: exact rationals -- the block's scale exponent
    floor(log2 max|v|) - 8 (clamped at -127) from integer arithmetic, each code
    the nearest finite e4m3 value of v / 2^s (ties to an even significand,
    saturating at +-448), on random blocks and on the edge cases (all zero,
    a value past 448 after scaling, bf16 subnormals); and the round trip of
    blocks built as e4m3 values times 2^t;
  * the linear: exact rational sums of the block-scaled products on tiny shapes,
    rounded once to bf16; one-hot rows; doubling a row's or a column's scales
    doubles that row or column exactly; unit scales reduce it to the per-tensor
    FP8 linear with unit scales.
The mutants are built from a text-substituted copy of oracle.c in a temporary
directory; the committed oracle is untouched.
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from exact import bf16_bits_to_fraction, rne_bf16_bits_exact
from test_oracle_fp8 import FINITE, e4m3_by_definition, nearest_e4m3

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")


def floor_log2(a: Fraction) -> int:
    """floor(log2(a)) of a positive rational, by integer arithmetic."""
    lg = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** lg > a:
        lg -= 1
    assert Fraction(2) ** lg <= a < Fraction(2) ** (lg + 1)
    return lg


def quant_block_exact(vals):
    """(codes, scale byte) of one 32-value block from the definition, exact rationals."""
    amax = max(abs(v) for v in vals)
    s = -127 if amax == 0 else max(floor_log2(amax) - 8, -127)
    codes = []
    for v in vals:
        y = v / Fraction(2) ** s
        if y > 448:
            codes.append(0x7E)
        elif y < -448:
            codes.append(0xFE)
        else:
            codes.append(nearest_e4m3(y))
    return codes, s + 127


def bf16_of(values) -> np.ndarray:
    t = torch.tensor(values, dtype=torch.float64).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def check_e8m0(orc):
    got = orc.e8m0_to_f64(np.arange(256, dtype=np.uint8))
    assert np.isnan(got[255])
    for e in range(255):
        assert Fraction(got[e]) == Fraction(2) ** (e - 127), e


def check_quant_round_trip(orc, seed=11):
    rng = np.random.default_rng(seed)
    finite = [c for c, v in FINITE if c not in (0x80,)]   # no negative zero in the inputs
    top = [0x78, 0x79, 0x7A, 0x7B, 0x7C, 0x7D, 0x7E, 0xF8, 0xFE]  # |value| in [256, 448]
    rows = []
    ts = []
    codes = []
    for r in range(6):
        t = int(rng.integers(-20, 21))
        c = [int(rng.choice(finite)) for _ in range(32)]
        c[int(rng.integers(32))] = int(rng.choice(top))
        vals = [e4m3_by_definition(x) * Fraction(2) ** t for x in c]
        rows.append([float(v) for v in vals])
        ts.append(t)
        codes.append(c)
    x = bf16_of(rows)
    q, s = orc.quant_mxfp8(x)
    assert np.array_equal(s[:, 0], np.array(ts) + 127)
    assert np.array_equal(q, np.array(codes, dtype=np.uint8))


def check_quant_brute_force(orc, seed=13):
    rng = np.random.default_rng(seed)
    blocks = []
    for r in range(8):
        mag = 2.0 ** int(rng.integers(-30, 30))
        blocks.append(list(rng.standard_normal(32) * mag))
    blocks.append([0.0] * 32)                                   # all zero: scale byte 0
    blocks.append([480.0] + [1.0] * 31)                         # 480 / 2^0 saturates to 448
    blocks.append([-470.0, 300.0] + [0.25] * 30)
    blocks.append([2.0 ** -130, -(2.0 ** -133)] + [0.0] * 30)   # bf16 subnormals: the exponent clamps at -127
    x = bf16_of(blocks).reshape(len(blocks), 32)
    q, s = orc.quant_mxfp8(x)
    for r in range(len(blocks)):
        vals = bf16_bits_to_fraction(x[r])
        codes, sb = quant_block_exact(vals)
        assert int(s[r, 0]) == sb, (r, int(s[r, 0]), sb)
        assert [int(v) for v in q[r]] == codes, r
    assert int(s[8, 0]) == 0 and not q[8].any()
    assert int(s[9, 0]) == 127 and int(q[9, 0]) == 0x7E


def _mx_inputs(rng, M, N, K, lo=120, hi=134):
    finite = [c for c, v in FINITE]
    xq = rng.choice(finite, size=(M, K)).astype(np.uint8)
    wq = rng.choice(finite, size=(N, K)).astype(np.uint8)
    sx = rng.integers(lo, hi, size=(M, K // 32)).astype(np.uint8)
    sw = rng.integers(lo, hi, size=(N, K // 32)).astype(np.uint8)
    return xq, sx, wq, sw


def check_linear_brute_force(orc, seed=17):
    rng = np.random.default_rng(seed)
    for M, N, K, with_bias in [(2, 3, 64, False), (3, 2, 96, True), (1, 1, 32, True)]:
        xq, sx, wq, sw = _mx_inputs(rng, M, N, K)
        b = bf16_of(list(rng.uniform(-0.1, 0.1, N))) if with_bias else None
        out = orc.linear_mxfp8(xq, sx, wq, sw, b)
        acc = orc.linear_mxfp8_f64(xq, sx, wq, sw, b)
        bias = bf16_bits_to_fraction(b) if with_bias else [Fraction(0)] * N
        for m in range(M):
            for n in range(N):
                v = bias[n]
                for k in range(K):
                    v += (e4m3_by_definition(int(xq[m, k])) * e4m3_by_definition(int(wq[n, k]))
                          * Fraction(2) ** (int(sx[m, k // 32]) - 127) * Fraction(2) ** (int(sw[n, k // 32]) - 127))
                assert int(out[m, n]) == rne_bf16_bits_exact(v), (M, N, K, m, n)
                assert abs(Fraction(acc[m, n]) - v) <= abs(v) * Fraction(1, 2 ** 50) + Fraction(1, 2 ** 200)


def check_one_hot(orc, seed=19):
    rng = np.random.default_rng(seed)
    M, N, K = 4, 5, 96
    _, _, wq, sw = _mx_inputs(rng, M, N, K)
    xq = np.zeros((M, K), dtype=np.uint8)
    sx = np.full((M, K // 32), 127, dtype=np.uint8)
    ks = [5, 37, 70, 95]
    for m, k in enumerate(ks):
        xq[m, k] = 0x38                      # 1.0
        sx[m, k // 32] = 127 + m - 1         # 2^(m-1) on the one block that matters
    out = orc.linear_mxfp8(xq, sx, wq, sw)
    for m, k in enumerate(ks):
        for n in range(N):
            v = e4m3_by_definition(int(wq[n, k])) * Fraction(2) ** (m - 1 + int(sw[n, k // 32]) - 127)
            assert int(out[m, n]) == rne_bf16_bits_exact(v), (m, n)


def check_scale_doubling(orc, seed=23):
    rng = np.random.default_rng(seed)
    M, N, K = 3, 4, 128
    xq, sx, wq, sw = _mx_inputs(rng, M, N, K)
    base = orc.linear_mxfp8_f64(xq, sx, wq, sw)
    sx2 = sx.copy()
    sx2[1] += 1
    row = orc.linear_mxfp8_f64(xq, sx2, wq, sw)
    assert np.array_equal(row[1], 2 * base[1]) and np.array_equal(row[[0, 2]], base[[0, 2]])
    sw2 = sw.copy()
    sw2[2] += 1
    col = orc.linear_mxfp8_f64(xq, sx, wq, sw2)
    assert np.array_equal(col[:, 2], 2 * base[:, 2]) and np.array_equal(col[:, [0, 1, 3]], base[:, [0, 1, 3]])


def check_unit_scales_reduce_to_per_tensor(orc, seed=29):
    rng = np.random.default_rng(seed)
    M, N, K = 3, 4, 64
    xq, _, wq, _ = _mx_inputs(rng, M, N, K)
    ones_x = np.full((M, 2), 127, dtype=np.uint8)
    ones_w = np.full((N, 2), 127, dtype=np.uint8)
    assert np.array_equal(orc.linear_mxfp8(xq, ones_x, wq, ones_w), orc.linear_fp8(xq, wq, 1.0, 1.0))


MX_CHECKS = [check_e8m0, check_quant_round_trip, check_quant_brute_force, check_linear_brute_force, check_one_hot,
             check_scale_doubling, check_unit_scales_reduce_to_per_tensor]


@pytest.mark.parametrize("check", MX_CHECKS, ids=lambda c: c.__name__)
def test_mxfp8_oracle_pins(check):
    oracle.build()
    check(oracle.default())


MX_MUTANTS = [
    ("scale_bias_128", "pow2_exact((int)xs[k / 32] - 127)", "pow2_exact((int)xs[k / 32] - 128)"),
    ("w_scale_from_x", "pow2_exact((int)ws[k / 32] - 127)", "pow2_exact((int)xs[k / 32] - 127)"),
    ("w_scale_dropped", "*\n               pow2_exact((int)ws[k / 32] - 127);", ";"),
    ("emax_7", "s = lg - 8;", "s = lg - 7;"),
    ("emax_9", "s = lg - 8;", "s = lg - 9;"),
    ("no_saturation", "if (y > 448.0) y = 448.0;", "(void)0;"),
    ("zero_block_scale", "int s = -127;", "int s = 0;"),
    ("amax_half_block", "for (int i = 0; i < 32; ++i) {\n                const double f", "for (int i = 0; i < 16; ++i) {\n                const double f"),
    ("no_lower_clamp", "if (s < -127) s = -127;", "(void)0;"),
    ("e8m0_nan_as_value", "if (e == 255) {", "if (0) {"),
]


@pytest.mark.parametrize("name,old,new", MX_MUTANTS, ids=[m[0] for m in MX_MUTANTS])
def test_mxfp8_pins_catch_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    path = tmp_path / f"oracle_{name}.c"
    path.write_text(src.replace(old, new))
    orc = oracle.Oracle(oracle.compile_source(str(path), str(tmp_path / f"lib_{name}.so")))
    failed = []
    for check in MX_CHECKS:
        try:
            check(orc)
        except AssertionError:
            failed.append(check.__name__)
    assert failed, f"no pin caught the planted mistake {name!r}"
