"""Pins for the CPU oracle: facts fixed by arithmetic, not by the oracle itself.

Each ``check_*`` takes an ``oracle.Oracle`` and raises AssertionError when the
oracle disagrees with a fact it must satisfy.  ``test_oracle_pins.py`` runs
them on the real oracle; ``test_oracle_mutants.py`` plants plausible mistakes
in a copy of oracle.c and checks that at least one pin fails for each.

What fixes each expected value:
  * rounding cases: the IEEE 754 binary format definition (bf16 = 1 sign bit,
    8 exponent bits with bias 127, 7 trailing significand bits), worked by hand
    in the comments; plus an exact-rational re-derivation and torch's own
    float32 -> bfloat16 cast, a library routine;
  * one-hot rows: x[m,:] = e_k makes out[m,n] = W[n,k] exactly;
  * all-ones: x = W = 1 gives out = RNE(K) (+ bias) exactly;
  * power-of-two scaling commutes with rounding (no overflow / subnormals);
  * linearity of the unrounded sum in x;
  * bias exactness: x = 0 gives out = bias;
  * exact-rational brute force on tiny shapes (sums exact in f64 by range);
  * numpy's float64 matmul (a different summation order) agrees to ~1e-13.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np
import torch

from exact import (bf16_bits_to_fraction, dyadic_bf16, exact_linear,
                   rne_bf16_bits_exact, rne_f32_bits_exact)

# ---------------------------------------------------------------------------
# Rounding: closed-form cases from the binary format definition.
# bf16 ulp at [1,2) is 2^-7; the smallest normal is 2^-126 (bits 0x0080);
# subnormals are multiples of 2^-133 (bits = multiple); the largest finite is
# (2 - 2^-7) * 2^127 (0x7F7F).  Ties go to the even trailing significand.
# ---------------------------------------------------------------------------
BF16_CASES = [
    (1.0, 0x3F80),                                  # exponent 127, significand 0
    (-2.0, 0xC000),
    (1 + 2**-8, 0x3F80),                            # tie 1 | 1+2^-7 -> even (0x..80)
    (1 + 3 * 2**-8, 0x3F82),                        # tie 1+2^-7 | 1+2^-6 -> even (0x..82)
    (1 + 2**-8 + 2**-30, 0x3F81),                   # just above the tie
    (1 + 2**-8 - 2**-30, 0x3F80),                   # just below the tie
    (2 - 2**-8, 0x4000),                            # tie 0x3FFF (odd) | 2.0 -> up, carries into exponent
    ((2 - 2**-7) * 2.0**127, 0x7F7F),               # largest finite
    ((2 - 2**-8) * 2.0**127, 0x7F80),               # tie largest (odd) | 2^128 -> infinity
    ((2 - 2**-8 - 2**-20) * 2.0**127, 0x7F7F),      # below that tie
    (2.0**128, 0x7F80),
    (2.0**-126, 0x0080),                            # smallest normal
    (2.0**-133, 0x0001),                            # smallest subnormal
    (2.0**-134, 0x0000),                            # tie 0 | 2^-133 -> even (0)
    (3 * 2.0**-135, 0x0001),                        # 0.75 ulp -> 1 ulp
    (3 * 2.0**-134, 0x0002),                        # 1.5 ulp tie -> even (2)
    (-(2.0**-134), 0x8000),                         # negative tie to zero keeps the sign
    (2.0**-126 - 2.0**-134, 0x0080),                # 127.5 subnormal ulps -> 128 = smallest normal
    (0.1, 0x3DCD),                                  # 1.6*2^-4: significand 76.8/128 -> 77
    (1e-300, 0x0000),
    (5e-324, 0x0000),                               # f64 subnormal
    (-0.0, 0x8000),
    (0.0, 0x0000),
    (math.inf, 0x7F80),
    (-math.inf, 0xFF80),
    (math.nan, 0x7FC0),                             # canonical quiet NaN
    (7168.0, 0x45E0),                               # 1.75 * 2^12
    (2049.0, 0x4500),                               # 2^11 (1 + 2^-11): below half an ulp (ulp 16)
    (2056.0, 0x4500),                               # 2048 + 8: tie -> even
    (2072.0, 0x4502),                               # 2048 + 24: tie 2064 | 2080 -> even
]

F32_CASES = [
    (0.1, 0x3DCCCCCD),
    (1 + 2**-24, 0x3F800000),                       # tie -> even
    (1 + 3 * 2**-24, 0x3F800002),                   # tie -> even
    (2.0**-149, 0x00000001),                        # smallest subnormal
    (2.0**-150, 0x00000000),                        # tie -> even (0)
    (3 * 2.0**-150, 0x00000002),                    # 1.5 ulp tie -> even (2)
    ((2 - 2**-24) * 2.0**127, 0x7F800000),          # tie at the top -> infinity
    (1e39, 0x7F800000),
    (-1.0, 0xBF800000),
]


def check_rne_cases(orc):
    for v, want in BF16_CASES:
        got = int(orc.rne_bf16([v])[0])
        assert got == want, f"RNE_bf16({v!r}) = {got:#06x}, want {want:#06x}"
    for v, want in F32_CASES:
        got = int(orc.rne_f32([v])[0])
        assert got == want, f"RNE_f32({v!r}) = {got:#010x}, want {want:#010x}"


def _rounding_probe_values(rng, n=4000):
    """f64 values that stress rounding: random binades incl. subnormal/overflow
    ranges, exact bf16 midpoints, and their f64 neighbours."""
    e = rng.integers(-140, 130, n)
    mant = rng.random(n) + 1.0
    sgn = np.where(rng.random(n) < 0.5, -1.0, 1.0)
    vals = list(sgn * mant * np.exp2(e.astype(np.float64)))
    # midpoints of adjacent bf16 values (exact in f64: 9 significant bits)
    bits = rng.integers(0, 0x7F7F, n // 4).astype(np.uint16)
    lo = bf16_bits_to_fraction(bits)
    hi = bf16_bits_to_fraction(bits + 1)
    for a, b in zip(lo, hi):
        mid = float((a + b) / 2)
        vals += [mid, np.nextafter(mid, np.inf), np.nextafter(mid, -np.inf), -mid]
    return [float(v) for v in vals]


def check_rne_vs_exact_rationals(orc, seed=11):
    rng = np.random.default_rng(seed)
    vals = _rounding_probe_values(rng)
    got_b = orc.rne_bf16(vals)
    got_f = orc.rne_f32(vals)
    for v, gb, gf in zip(vals, got_b, got_f):
        fv = Fraction(v)
        wb = rne_bf16_bits_exact(fv)
        assert int(gb) == wb, f"RNE_bf16({v!r}) = {int(gb):#06x}, exact rational gives {wb:#06x}"
        wf = rne_f32_bits_exact(fv)
        assert int(gf) == wf, f"RNE_f32({v!r}) = {int(gf):#010x}, exact rational gives {wf:#010x}"


def check_rne_vs_torch_cast(orc, seed=12):
    """torch's float32 -> bfloat16 cast is round-to-nearest-even: a library special case."""
    rng = np.random.default_rng(seed)
    n = 20000
    u = rng.integers(0, 2**32, n, dtype=np.uint64).astype(np.uint32)
    f = u.view(np.float32)
    f = f[np.isfinite(f)]
    want = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = orc.rne_bf16(f.astype(np.float64))
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, (f"{bad.size} mismatches vs torch cast, first: {float(f[bad[0]])!r} -> "
                           f"{int(got[bad[0]]):#06x} vs {int(want[bad[0]]):#06x}")
    # numpy's float64 -> float32 cast is round-to-nearest-even too
    d = rng.standard_normal(5000) * np.exp2(rng.integers(-150, 128, 5000).astype(np.float64))
    with np.errstate(over="ignore"):
        want32 = d.astype(np.float32).view(np.uint32)
    got32 = orc.rne_f32(d)
    assert np.array_equal(got32, want32), "RNE_f32 disagrees with numpy's float64->float32 cast"


# ---------------------------------------------------------------------------
# The linear map itself.
# ---------------------------------------------------------------------------
def _rand_bf16(rng, shape, scale=1.0):
    t = torch.from_numpy(rng.standard_normal(shape).astype(np.float32) * np.float32(scale))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _f64(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).double().numpy()


def check_one_hot(orc, seed=21):
    """x[m,:] = e_{k_m}  =>  out[m, n] = W[n, k_m] exactly (non-square: catches a transpose)."""
    rng = np.random.default_rng(seed)
    for (M, N, K) in [(3, 5, 7), (4, 256, 2048), (2, 17, 2880)]:
        W = _rand_bf16(rng, (N, K), K ** -0.5)
        ks = rng.integers(0, K, M)
        x = np.zeros((M, K), dtype=np.uint16)
        x[np.arange(M), ks] = 0x3F80  # 1.0
        out = orc.linear_bf16(x, W)
        assert np.array_equal(out, W[:, ks].T), f"one-hot rows do not reproduce W columns ({M},{N},{K})"
        # and with a bias: out = RNE(W[n,k] + b[n])
        b = _rand_bf16(rng, (N,), 0.05)
        outb = orc.linear_f64(x, W, b)
        assert np.array_equal(outb, _f64(W[:, ks].T) + _f64(b)[None, :]), "one-hot + bias"


def check_all_ones(orc):
    """x = W = 1  =>  out = RNE(K) (and RNE(K + b) with bias); K of every workload is exact in bf16."""
    for K, want in [(2048, 0x4500), (2880, 0x4534), (4096, 0x4580), (6144, 0x45C0),
                    (7168, 0x45E0), (2049, 0x4500), (2072, 0x4502), (1, 0x3F80)]:
        M, N = 2, 3
        x = np.full((M, K), 0x3F80, dtype=np.uint16)
        W = np.full((N, K), 0x3F80, dtype=np.uint16)
        out = orc.linear_bf16(x, W)
        assert (out == want).all(), f"all-ones K={K}: got {int(out[0,0]):#06x} want {want:#06x}"
        assert (orc.linear_f64(x, W) == float(K)).all(), f"all-ones K={K}: unrounded sum != K"
    # with bias 0.5 (0x3F00) and -3 (0xC040): K + b, rounded once
    K = 2880
    x = np.full((1, K), 0x3F80, dtype=np.uint16)
    W = np.full((2, K), 0x3F80, dtype=np.uint16)
    b = np.array([0x3F00, 0xC040], dtype=np.uint16)
    assert list(orc.linear_f64(x, W, b)[0]) == [2880.5, 2877.0]
    # 2880.5 -> ulp 16 at [2048,4096): 2880 exactly representable (0x4534); 2877 -> 2880
    assert list(orc.linear_bf16(x, W, b)[0]) == [0x4534, 0x4534]


def check_pow2_scaling(orc, seed=31):
    """out(2^j x) = 2^j out(x) bitwise: scaling by 2^j commutes with f64 sums and with RNE."""
    rng = np.random.default_rng(seed)
    M, N, K = 4, 64, 512
    x = _rand_bf16(rng, (M, K))
    W = _rand_bf16(rng, (N, K), K ** -0.5)
    base = _f64(orc.linear_bf16(x, W))
    for j in (3, -5):
        xs = (x.astype(np.int32) + (j << 7)).astype(np.uint16)  # add j to the exponent field
        assert np.array_equal(_f64(xs), _f64(x) * 2.0**j)
        got = _f64(orc.linear_bf16(xs, W))
        assert np.array_equal(got, base * 2.0**j), f"power-of-two scaling by 2^{j} not exact"


def check_linearity(orc, seed=41):
    """f(3*x1 + x2) = 3 f(x1) + f(x2) on the unrounded sums (small-integer x keep inputs exact)."""
    rng = np.random.default_rng(seed)
    M, N, K = 3, 40, 1000
    W = _rand_bf16(rng, (N, K), K ** -0.5)
    i1 = rng.integers(-16, 17, (M, K)).astype(np.float32)
    i2 = rng.integers(-16, 17, (M, K)).astype(np.float32)

    def b(a):
        return torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)

    f1 = orc.linear_f64(b(i1), W)
    f2 = orc.linear_f64(b(i2), W)
    f3 = orc.linear_f64(b(3 * i1 + i2), W)
    scale = np.abs(3 * i1 + i2).astype(np.float64) @ np.abs(_f64(W)).T + np.abs(i1) @ np.abs(_f64(W)).T
    assert np.all(np.abs(f3 - (3 * f1 + f2)) <= 1e-12 * scale + 1e-300), "not linear in x"


def check_bias_exact(orc, seed=51):
    """x = 0  =>  out = bias exactly (bias drawn without zeros, so no signed-zero question)."""
    rng = np.random.default_rng(seed)
    M, N, K = 3, 37, 96
    W = _rand_bf16(rng, (N, K), K ** -0.5)
    bias = _rand_bf16(rng, (N,), 0.05)
    bias[(bias & 0x7FFF) == 0] = 0x3F80
    x = np.zeros((M, K), dtype=np.uint16)
    out = orc.linear_bf16(x, W, bias)
    assert np.array_equal(out, np.broadcast_to(bias, (M, N))), "x=0 must return the bias exactly"
    assert np.array_equal(orc.linear_bf16(x, W), np.zeros((M, N), dtype=np.uint16)), "x=0, no bias must be +0"


def check_brute_force(orc, seed=61):
    """Tiny shapes: exact rational sums and an independent RNE equal the oracle bitwise.

    Values have |v| in [2^-8, 2^8), so every product is a multiple of 2^-30 below 2^16
    and any sum of <= 9 such terms is exact in f64: the oracle's f64 sum must equal
    the rational one, and so must the rounded results."""
    rng = np.random.default_rng(seed)
    for trial in range(40):
        M = int(rng.integers(1, 5))
        N = int(rng.integers(1, 9))
        K = int(rng.integers(1, 9))
        x = dyadic_bf16(rng, (M, K))
        W = dyadic_bf16(rng, (N, K))
        b = dyadic_bf16(rng, (N,)) if trial % 2 else None
        ex = exact_linear(x, W, b)
        acc = orc.linear_f64(x, W, b)
        out = orc.linear_bf16(x, W, b)
        out32 = orc.linear_f32(x, W, b)
        for m in range(M):
            for n in range(N):
                assert Fraction(float(acc[m, n])) == ex[m][n], f"f64 sum != exact at ({m},{n}) trial {trial}"
                assert int(out[m, n]) == rne_bf16_bits_exact(ex[m][n]), f"bf16 at ({m},{n}) trial {trial}"
                assert int(out32[m, n]) == rne_f32_bits_exact(ex[m][n]), f"f32 at ({m},{n}) trial {trial}"


def check_numpy_matmul(orc, seed=71):
    """numpy's float64 matmul (another summation order) agrees on the unrounded sums to ~1e-13,
    and the rounded results differ by at most one bf16 ulp, only next to ties."""
    rng = np.random.default_rng(seed)
    M, N, K = 4, 256, 2048
    x = _rand_bf16(rng, (M, K))
    W = _rand_bf16(rng, (N, K), K ** -0.5)
    b = _rand_bf16(rng, (N,), 0.05)
    acc = orc.linear_f64(x, W, b)
    ref = _f64(x) @ _f64(W).T + _f64(b)[None, :]
    scale = np.abs(_f64(x)) @ np.abs(_f64(W)).T + np.abs(_f64(b))[None, :]
    assert np.all(np.abs(acc - ref) <= 1e-13 * scale), "oracle f64 sum disagrees with numpy matmul"
    out = orc.linear_bf16(x, W, b)
    ref_bits = orc.rne_bf16(ref.ravel()).reshape(M, N)
    diff = np.abs(out.astype(np.int32) - ref_bits.astype(np.int32))
    assert diff.max() <= 1, "rounded results differ by more than one ulp"
    assert (diff != 0).sum() <= 2, "too many rounding disagreements for a 1e-13 perturbation"


def check_rows_variant(orc, seed=81):
    """The sampled-rows entry points equal the corresponding rows of the full result."""
    rng = np.random.default_rng(seed)
    M, N, K = 9, 33, 160
    x = _rand_bf16(rng, (M, K))
    W = _rand_bf16(rng, (N, K), K ** -0.5)
    b = _rand_bf16(rng, (N,), 0.05)
    rows = np.array([0, 4, 8, 4])
    assert np.array_equal(orc.linear_rows_bf16(x, W, b, rows), orc.linear_bf16(x, W, b)[rows])
    assert np.array_equal(orc.linear_rows_f64(x, W, b, rows), orc.linear_f64(x, W, b)[rows])


ALL_CHECKS = [check_rne_cases, check_rne_vs_exact_rationals, check_rne_vs_torch_cast,
              check_one_hot, check_all_ones, check_pow2_scaling, check_linearity,
              check_bias_exact, check_brute_force, check_numpy_matmul, check_rows_variant]
