"""The group scale's shortcut to the exact result, checked on the host
against its definition (no GPU, no CUDA code): s = amax / 448 without a
division, q = RN(amax * RN(1/448)) and one fused multiply-add correction
s = RN(q + RN(amax - 448 q) * RN(1/448)) (correctly rounded division by a
constant known in advance, Brisebarre, Muller and Raina).  Checked against
IEEE fp32 division for every non-negative finite bf16 amax, with the two
fused multiply-adds evaluated exactly in rational arithmetic and rounded
once.  (The per-element code's shortcut is checked exhaustively in
test_corrected_quotient.py.)
"""
from fractions import Fraction

import numpy as np


F32 = np.float32


def rn32(v: Fraction) -> np.float32:
    """Round a rational to the nearest fp32 (ties to even), subnormals kept."""
    if v == 0:
        return F32(0.0)
    sign = -1 if v < 0 else 1
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    quantum = Fraction(2) ** (max(e, -126) - 23)
    n, rem = divmod(a, quantum)
    n = int(n)
    if rem * 2 > quantum or (rem * 2 == quantum and n % 2 == 1):
        n += 1
    return F32(sign * float(n * quantum))


def bf16_values(nonnegative: bool) -> np.ndarray:
    """Every finite bf16 value (as fp32); with `nonnegative`, sign bit clear
    (+0 but not -0: an amax is a maximum of magnitudes starting at +0)."""
    bits = np.arange(0, 0x8000 if nonnegative else 0x10000, dtype=np.uint32)
    vals = (bits << 16).view(np.float32)
    return vals[np.isfinite(vals)]


def test_scale_without_division_equals_ieee_division():
    R = F32(1.0) / F32(448.0)
    fr_R = Fraction(float(R))
    bad = []
    for amax in bf16_values(nonnegative=True):
        q = F32(amax) * R
        fr_q = Fraction(float(q))
        rem = rn32(Fraction(float(amax)) - fr_q * 448)
        s = rn32(fr_q + Fraction(float(rem)) * fr_R)
        want = F32(amax) / F32(448.0)
        if s.view(np.uint32) != want.view(np.uint32):
            bad.append(float(amax))
    assert not bad, bad[:8]
