"""Pins for the oracle's per-tensor FP8 functions, and planted mistakes they catch.

What fixes each function, independently of the oracle:
  * e4m3 decoding: the format definition written out here (sign, 4-bit
    exponent with bias 7, 3-bit significand, subnormals below 2^-6, 0x7F/0xFF
    NaN, no infinities) and torch's own float8_e4m3fn dtype, for all 256 codes;
  * rounding to e4m3: the nearest of the 253 finite values (exact rationals),
    ties to the code with an even significand;
  * static quantisation: torch doing the page's steps (binary32 reciprocal,
    binary32 product, clamp to +-448, cast to float8_e4m3fn), bit for bit;
  * the FP8 linear: exact rational sums on tiny shapes, one-hot rows, all-ones.
The mutants are built from a text-substituted copy of oracle.c in a temporary
directory; the committed oracle is untouched.
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from exact import bf16_bits_to_fraction, rne_fraction

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")


def e4m3_by_definition(c: int):
    """Exact value of an e4m3 code from the format definition (None for NaN)."""
    s, E, m = c >> 7, (c >> 3) & 15, c & 7
    if E == 15 and m == 7:
        return None
    v = Fraction(m, 8) * Fraction(1, 64) if E == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (E - 7)
    return -v if s else v


FINITE = [(c, e4m3_by_definition(c)) for c in range(256) if e4m3_by_definition(c) is not None]


def nearest_e4m3(v: Fraction) -> int:
    """Code of the finite e4m3 value nearest to v, ties to an even significand (|v| <= 448)."""
    best = None
    for c, val in FINITE:
        if val == 0 and c == 0x80 and v >= 0:
            continue  # +0 for non-negative inputs
        if val == 0 and c == 0x00 and v < 0:
            continue  # -0 for negative inputs
        d = abs(val - v)
        if best is None or d < best[0] or (d == best[0] and (c & 1) == 0):
            best = (d, c)
    return best[1]


def check_decode(orc):
    c = np.arange(256, dtype=np.uint8)
    got = orc.e4m3_to_f64(c)
    for code in range(256):
        want = e4m3_by_definition(code)
        if want is None:
            assert np.isnan(got[code]), hex(code)
        else:
            assert Fraction(float(got[code])) == want, hex(code)
    t = torch.from_numpy(c.copy()).view(torch.float8_e4m3fn).double().numpy()
    fin = ~np.isnan(t)
    assert np.array_equal(np.isnan(got), ~fin) and np.array_equal(got[fin], t[fin])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x08] == 2.0 ** -6 and got[0x38] == 1.0


def check_rne(orc, seed=3):
    rng = np.random.default_rng(seed)
    vals = [float(v) for _, v in FINITE]
    mids = [(a + b) / 2 for a, b in zip(sorted(vals), sorted(vals)[1:])]  # exact ties
    rand = list(rng.uniform(-448, 448, 300)) + list(rng.uniform(-0.02, 0.02, 300))
    probe = np.array(vals + mids + rand, dtype=np.float64)
    got = orc.rne_e4m3(probe)
    for v, g in zip(probe, got):
        assert int(g) == nearest_e4m3(Fraction(float(v))), (v, hex(int(g)))


def check_quant_vs_torch(orc, seed=5):
    rng = np.random.default_rng(seed)
    x = torch.from_numpy(rng.standard_normal(4000).astype(np.float32) * 3).to(torch.bfloat16)
    x[:4] = torch.tensor([1e4, -1e4, 0.0, -0.0]).to(torch.bfloat16)  # saturation and signed zeros
    bits = x.view(torch.int16).numpy().view(np.uint16)
    for s in (1.0, 0.5, 0.0123, 3.7, 1e-3, 0.3):
        inv = torch.tensor(1.0, dtype=torch.float32) / torch.tensor(s, dtype=torch.float32)
        want = (x.float() * inv).clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        got = orc.quant_fp8(bits, s)
        assert np.array_equal(got, want), f"scale {s}: {int((got != want).sum())} codes differ"
    # Every bf16 value in [2^-7, 2^9) and its negative, with scales 7 and 1.7:
    # there the binary32 reciprocal of the scale makes x * (1/s) land on the
    # other side of an e4m3 rounding boundary than x / s for some inputs, so
    # this pins the page's way of applying the scale (reciprocal, then product).
    b = np.arange(0x3C00, 0x4400, dtype=np.uint16)
    b = np.concatenate([b, b | 0x8000])
    xb = torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16)
    for s in (7.0, 1.7):
        inv = torch.tensor(1.0, dtype=torch.float32) / torch.tensor(s, dtype=torch.float32)
        want = (xb.float() * inv).clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(orc.quant_fp8(b, s), want), f"scale {s}: reciprocal-then-product codes differ"


def _codes(rng, shape):
    c = rng.integers(0, 256, shape).astype(np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x38  # no NaN codes
    return c


def check_brute_force(orc, seed=7):
    rng = np.random.default_rng(seed)
    for (M, N, K) in [(1, 1, 1), (2, 3, 5), (3, 2, 17), (4, 4, 8)]:
        xq, wq = _codes(rng, (M, K)), _codes(rng, (N, K))
        sx, sw = float(np.float32(rng.uniform(0.001, 2))), float(np.float32(rng.uniform(0.001, 2)))
        b = torch.from_numpy(rng.uniform(-0.5, 0.5, N).astype(np.float32)).to(torch.bfloat16)
        bbits = b.view(torch.int16).numpy().view(np.uint16)
        bf = bf16_bits_to_fraction(bbits)
        got = orc.linear_fp8(xq, wq, sx, sw, bbits)
        gotf = bf16_bits_to_fraction(got)
        for m in range(M):
            for n in range(N):
                acc = sum(e4m3_by_definition(int(xq[m, k])) * e4m3_by_definition(int(wq[n, k])) for k in range(K))
                v = acc * Fraction(sx) * Fraction(sw) + bf[n]
                r = rne_fraction(v, 8, 7)
                assert gotf[m * N + n] == r, (m, n)


def check_one_hot_and_ones(orc, seed=9):
    rng = np.random.default_rng(seed)
    M, N, K = 5, 7, 33
    wq = _codes(rng, (N, K))
    ks = rng.integers(0, K, M)
    xq = np.zeros((M, K), dtype=np.uint8)
    xq[np.arange(M), ks] = 0x38  # 1.0
    acc = orc.linear_fp8_f64(xq, wq, 1.0, 1.0)
    dec = np.array([[float(e4m3_by_definition(int(c))) for c in row] for row in wq])
    assert np.array_equal(acc, dec[:, ks].T)
    ones = orc.linear_fp8_f64(np.full((2, K), 0x38, np.uint8), np.full((3, K), 0x38, np.uint8), 0.5, 0.25)
    assert (ones == K * 0.125).all()


FP8_CHECKS = [check_decode, check_rne, check_quant_vs_torch, check_brute_force, check_one_hot_and_ones]


@pytest.mark.parametrize("check", FP8_CHECKS, ids=lambda c: c.__name__)
def test_fp8_oracle_pins(check):
    check(oracle.default())


FP8_MUTANTS = [
    ("decode_bias_8", "for (int i = 7; i < E; ++i) v *= 2.0;", "for (int i = 8; i < E; ++i) v *= 2.0;"),
    ("decode_subnormal_scale", "v = (double)m / 8.0 * 0.015625;", "v = (double)m / 8.0 * 0.03125;"),
    ("decode_sign_dropped", "return s ? -v : v;", "return v;"),
    ("e4m3_round_half_up", "if (rem > half || (rem == half && (kept & 1))) kept++;", "if (rem >= half) kept++;"),
    ("e4m3_exponent_field", "(((E + 7 - 1) << mbits) + (int)kept)", "(((E + 7) << mbits) + (int)kept)"),
    ("quant_no_clamp", "if (y > 448.0f) y = 448.0f;", "(void)0;"),
    ("quant_divides", "float y = (float)bf16_to_f64(x[i]) * inv;", "float y = (float)bf16_to_f64(x[i]) / scale;"),
    ("fp8_one_scale", "const double sxw = (double)sx * (double)sw;\n    for (int64_t m = 0; m < M; ++m)\n        for (int64_t n = 0; n < N; ++n)\n            out",
     "const double sxw = (double)sx;\n    for (int64_t m = 0; m < M; ++m)\n        for (int64_t n = 0; n < N; ++n)\n            out"),
    ("fp8_w_index", "e4m3_to_f64(wrow[k])", "e4m3_to_f64(wrow[0])"),
]


@pytest.mark.parametrize("name,old,new", FP8_MUTANTS, ids=[m[0] for m in FP8_MUTANTS])
def test_fp8_pins_catch_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    path = tmp_path / f"oracle_{name}.c"
    path.write_text(src.replace(old, new))
    orc = oracle.Oracle(oracle.compile_source(str(path), str(tmp_path / f"lib_{name}.so")))
    failed = []
    for check in FP8_CHECKS:
        try:
            check(orc)
        except AssertionError:
            failed.append(check.__name__)
    assert failed, f"no FP8 pin caught the planted mistake {name!r}"
