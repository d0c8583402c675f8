"""Shared test helpers: exact decoding, an independent RNE in rational
arithmetic, and the acceptance tolerance of the decode projection."""
from fractions import Fraction

import numpy as np

from skinny_bf16_split_gb300.synth import bf16_to_f32


def bf16_fraction(h: int) -> Fraction:
    """Exact value of finite BF16 bits, decoded through the FP32 hardware format."""
    f = np.array([int(h) << 16], dtype=np.uint32).view(np.float32)[0]
    assert np.isfinite(f)
    return Fraction(float(f))


def rne_bf16_fraction(s: Fraction) -> int:
    """Round an exact rational to BF16 bits, nearest, ties to even (independent of
    the oracle's limb arithmetic: works on Python rationals)."""
    if s == 0:
        return 0x0000
    sign = 0x8000 if s < 0 else 0
    a = abs(s)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    elif Fraction(2) ** (e + 1) <= a:
        e += 1
    qe = max(e - 7, -133)
    scaled = a / Fraction(2) ** qe
    M = scaled.numerator // scaled.denominator
    rem = scaled - M
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and M % 2 == 1):
        M += 1
    if M == 256:
        M, qe = 128, qe + 1
    if qe == -133 and M < 128:
        return sign | M
    field = qe + 134
    if field >= 255:
        return sign | 0x7F80
    return sign | (field << 7) | (M - 128)


def exact_bf16(v) -> int:
    """BF16 bits of a value that must be exactly representable."""
    f = np.float32(v)
    bits = int(np.array([f], dtype=np.float32).view(np.uint32)[0])
    assert bits & 0xFFFF == 0 and float(f) == float(v), f"{v} is not a BF16 value"
    return bits >> 16


def within_tolerance(y, ref):
    """|y - ref| <= 2^-7 |ref| + 1e-3 rms(ref), elementwise, rms over the call.

    Returns (ok, worst excess ratio, index of worst)."""
    yf = bf16_to_f32(y).astype(np.float64)
    rf = bf16_to_f32(ref).astype(np.float64)
    rms = np.sqrt(np.mean(rf * rf)) if rf.size else 0.0
    bound = 2.0 ** -7 * np.abs(rf) + 1e-3 * rms
    err = np.abs(yf - rf)
    both_nan = np.isnan(yf) & np.isnan(rf)
    same_inf = np.isinf(yf) & np.isinf(rf) & (yf == rf)
    bad = ~(both_nan | same_inf) & ~(err <= bound)
    if not bad.any():
        return True, 0.0, None
    ratio = np.where(bad, err / np.maximum(bound, 1e-300), 0)
    idx = np.unravel_index(int(np.nanargmax(ratio)), ratio.shape)
    return False, float(ratio[idx]), idx
