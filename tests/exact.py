"""Exact-rational helpers for pinning the oracle, written independently of it.

Nothing here calls the oracle or the CUDA library.  bf16 values are decoded
with torch's own bfloat16 dtype and turned into exact ``Fraction`` objects;
rounding is re-derived on rationals: find the binade, scale by the unit in the
last place, take the floor, and break ties toward an even significand.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np
import torch

INF = float("inf")


def bf16_bits_to_fraction(bits) -> list[Fraction]:
    """Exact value of each finite bf16 bit pattern (decoded by torch)."""
    b = np.asarray(bits, dtype=np.uint16).ravel()
    f = torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    return [Fraction(float(v)) for v in f]


def rne_fraction(v: Fraction, ebits: int, mbits: int):
    """Nearest value of the (ebits, mbits) binary format, ties to even significand.

    Returns a Fraction, or +/-INF when the rounded magnitude reaches 2^(emax+1).
    """
    if v == 0:
        return Fraction(0)
    sgn = -1 if v < 0 else 1
    a = abs(v)
    bias = 2 ** (ebits - 1) - 1
    emin = 1 - bias
    E = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** E > a:
        E -= 1
    while Fraction(2) ** (E + 1) <= a:
        E += 1
    q = max(E, emin) - mbits
    scaled = a / (Fraction(2) ** q)
    n = scaled.numerator // scaled.denominator
    r = scaled - n
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and n % 2 == 1):
        n += 1
    val = n * Fraction(2) ** q
    if val >= Fraction(2) ** (bias + 1):
        return sgn * INF
    return sgn * val


_BF16_TABLE = None


def _bf16_table():
    """Map exact value -> bit pattern for every finite non-negative bf16."""
    global _BF16_TABLE
    if _BF16_TABLE is None:
        pos = np.arange(0, 0x7F80, dtype=np.uint16)  # +0 .. largest finite
        vals = bf16_bits_to_fraction(pos)
        _BF16_TABLE = {v: int(b) for v, b in zip(vals, pos)}
    return _BF16_TABLE


def rne_bf16_bits_exact(v: Fraction, negative_zero: bool = False) -> int:
    """bf16 bit pattern of RNE(v), derived on rationals."""
    r = rne_fraction(v, 8, 7)
    if r == INF:
        return 0x7F80
    if r == -INF:
        return 0xFF80
    if r == 0:
        return 0x8000 if (v < 0 or negative_zero) else 0x0000
    bits = _bf16_table()[abs(r)]
    return bits | (0x8000 if r < 0 else 0)


def rne_f32_bits_exact(v: Fraction) -> int:
    """binary32 bit pattern of RNE(v), derived on rationals."""
    r = rne_fraction(v, 8, 23)
    if r in (INF, -INF):
        return 0x7F800000 | (0x80000000 if r < 0 else 0)
    if r == 0:
        return 0x80000000 if v < 0 else 0
    f = np.float32(float(r))          # r has <= 24 significant bits: exact in f64 and f32
    assert Fraction(float(f)) == r
    return int(np.array([f], dtype=np.float32).view(np.uint32)[0])


def exact_linear(xb, Wb, bb=None) -> list[list[Fraction]]:
    """Exact rational out[m][n] = sum_k x[m,k] W[n,k] (+ b[n]) for tiny shapes."""
    xb = np.asarray(xb, dtype=np.uint16)
    Wb = np.asarray(Wb, dtype=np.uint16)
    M, K = xb.shape
    N = Wb.shape[0]
    xv = [bf16_bits_to_fraction(xb[m]) for m in range(M)]
    wv = [bf16_bits_to_fraction(Wb[n]) for n in range(N)]
    bv = bf16_bits_to_fraction(bb) if bb is not None else None
    out = []
    for m in range(M):
        row = []
        for n in range(N):
            s = sum((xv[m][k] * wv[n][k] for k in range(K)), Fraction(0))
            if bv is not None:
                s += bv[n]
            row.append(s)
        out.append(row)
    return out


def dyadic_bf16(rng: np.random.Generator, shape, emin=-8, emax=7) -> np.ndarray:
    """Random bf16 bit patterns with |v| in [2^emin, 2^(emax+1)): sign, exponent, 7-bit mantissa."""
    n = int(np.prod(shape))
    sign = rng.integers(0, 2, n).astype(np.uint16) << 15
    exp = (rng.integers(emin, emax + 1, n) + 127).astype(np.uint16) << 7
    man = rng.integers(0, 128, n).astype(np.uint16)
    return (sign | exp | man).reshape(shape)
