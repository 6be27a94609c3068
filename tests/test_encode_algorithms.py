"""The two shortcuts the CUDA quantisers take to the exact result, checked on
the host against their definitions (no GPU, no CUDA code):

* the group scale s = amax / 448 without a division: q = RN(amax * RN(1/448))
  and one fused multiply-add correction s = RN(q + RN(amax - 448 q) * RN(1/448))
  (correctly rounded division by a constant known in advance, Brisebarre,
  Muller and Raina).  Checked against IEEE fp32 division for every
  non-negative finite bf16 amax, with the two fused multiply-adds evaluated
  exactly in rational arithmetic and rounded once.

* the code of fp32(x / s) from a reciprocal bracket: with r within about an
  ulp of 1/s, ra = RN(r (1 - 2^-21)) and rb = RN(r (1 + 2^-21)), whenever the
  E4M3 codes of RN(x ra) and RN(x rb) agree, that code is the code of
  RN(x / s).  Checked for every finite bf16 x against a spread of scales and
  three reciprocals per scale (RN(1/s) and its two neighbours), with the
  oracle's encoder as the reference.
"""
from fractions import Fraction

import numpy as np

import oracle

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


def test_reciprocal_bracket_codes_are_exact():
    saved = np.geterr()
    try:
        _bracket_check()
    finally:
        np.seterr(**saved)


def _bracket_check():
    x = bf16_values(nonnegative=False)
    # scales s = amax / 448 from a spread of normal amax values: powers of two,
    # the extremes of the normal range and seeded random bf16 magnitudes
    rng = np.random.default_rng(11)
    amaxes = [1.0, 448.0, 2.0 ** -100 * 448.0, 3.0e38, 1.5, 0.3, 1e-20, 7e15]
    # bf16 exponent fields 12 .. 254: amax >= 2^-115, so s = amax / 448 is normal
    amaxes += list((rng.integers(0x0600, 0x7F80, 12, dtype=np.uint32) << 16).view(np.float32))
    agreed = disagreed = 0
    # |x| far above a small group's amax overflows x / s and x * r to +-inf in
    # fp32; both then saturate to the +-448 code, as in the kernel
    np.seterr(over="ignore")
    for amax in amaxes:
        s = F32(amax) / F32(448.0)
        assert s >= F32(2.0 ** -126)           # normal scales take the bracket
        exact = oracle.e4m3_encode(x / s)      # fp32 IEEE division per element
        r0 = F32(1.0) / s
        for r in (np.nextafter(r0, F32(0.0)), r0, np.nextafter(r0, F32(np.inf))):
            ra = F32(r) * F32(float.fromhex("0x1.fffffp-1"))
            rb = F32(r) * F32(float.fromhex("0x1.000008p+0"))
            ca = oracle.e4m3_encode(x * ra)
            cb = oracle.e4m3_encode(x * rb)
            same = ca == cb
            assert np.array_equal(ca[same], exact[same]), (float(amax), float(r))
            agreed += int(same.sum())
            disagreed += int((~same).sum())
    # the exact fallback stays the rare path
    assert disagreed < 0.05 * (agreed + disagreed)
