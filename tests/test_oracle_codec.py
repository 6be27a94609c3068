"""Pins for the oracle's E4M3 codec (CPU only).

What pins it, independently of the oracle's own arithmetic:
  * code values printed in the OCP FP8 definition (golden file);
  * an exhaustive round trip of all 256 codes;
  * PyTorch's float8_e4m3fn decode (library routine) for all 256 codes;
  * a brute-force nearest-value search with the round-to-nearest-even tie
    rule, over every bf16 bit pattern and a large stratified sample of fp32
    patterns (all exact ties and their neighbours included);
  * PyTorch's float -> float8_e4m3fn cast for |v| <= 448.
"""
import numpy as np
import pytest
import torch

from conftest import read_golden
from e4m3_brute import TABLE, brute_encode


def _f32(bits):
    return np.asarray(bits, dtype=np.uint32).view(np.float32)


def test_golden_code_values(oracle_mod):
    rows = read_golden("e4m3_codes.txt")
    assert len(rows) >= 15
    codes = np.array([int(r[0], 16) for r in rows], dtype=np.uint8)
    dec = oracle_mod.e4m3_decode(codes)
    for (c, v), d in zip(rows, dec):
        if v == "nan":
            assert np.isnan(d), c
        elif v == "-0":
            assert d == 0.0 and np.signbit(d), c
        else:
            assert d == float(v), (c, v, d)


def test_decode_matches_library_decode(oracle_mod):
    dec = oracle_mod.e4m3_decode(np.arange(256, dtype=np.uint8))
    for c in range(256):
        if np.isnan(TABLE[c]):
            assert np.isnan(dec[c]), c
        else:
            assert dec[c] == TABLE[c] and np.signbit(dec[c]) == np.signbit(TABLE[c]), c


def test_round_trip_all_codes(oracle_mod):
    codes = np.arange(256, dtype=np.uint8)
    dec = oracle_mod.e4m3_decode(codes)
    finite = np.isfinite(dec)
    assert finite.sum() == 254           # 0x7f and 0xff are NaN
    back = oracle_mod.e4m3_encode(dec[finite].astype(np.float32))
    assert np.array_equal(back, codes[finite])
    # NaN encodes to the canonical NaN code
    assert oracle_mod.e4m3_encode(np.array([np.nan], np.float32))[0] == 0x7F


def test_value_order_and_symmetry(oracle_mod):
    dec = oracle_mod.e4m3_decode(np.arange(256, dtype=np.uint8))
    pos = dec[:0x7F]
    assert np.all(np.diff(pos) > 0)      # codes 0x00..0x7e strictly increasing
    assert pos[-1] == 448.0
    assert np.array_equal(dec[0x80:0xFF], -pos)


def test_encode_all_bf16_patterns_vs_brute_force(oracle_mod):
    bits = np.arange(65536, dtype=np.uint32) << 16
    vals = _f32(bits)
    keep = ~np.isnan(vals)
    vals = vals[keep]
    got = oracle_mod.e4m3_encode(vals)
    want = brute_encode(vals.astype(np.float64))
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(float(vals[i]), hex(got[i]), hex(want[i])) for i in bad[:8]]


def _fp32_sample(rng):
    parts = []
    # every exact tie between neighbouring finite E4M3 values, and the fp32
    # values just above and below it
    dec = np.unique(TABLE[np.isfinite(TABLE)])
    mids = ((dec[:-1] + dec[1:]) / 2).astype(np.float32)
    parts += [mids, np.nextafter(mids, np.float32(np.inf)), np.nextafter(mids, np.float32(-np.inf))]
    parts += [dec.astype(np.float32)]
    # dense random mantissas over the binades that matter (2^-12 .. 2^10)
    exps = rng.integers(127 - 12, 127 + 10, size=1 << 20, dtype=np.uint32)
    mant = rng.integers(0, 1 << 23, size=1 << 20, dtype=np.uint32)
    sign = rng.integers(0, 2, size=1 << 20, dtype=np.uint32)
    parts.append(_f32((sign << 31) | (exps << 23) | mant))
    # random full-range patterns (saturation, fp32 subnormals, huge values)
    parts.append(_f32(rng.integers(0, 1 << 32, size=1 << 18, dtype=np.uint64).astype(np.uint32)))
    parts.append(np.array([0.0, -0.0, np.inf, -np.inf, 448.0, -448.0, 463.99, 464.0, 464.01,
                           479.0, 480.0, 1e30, -1e30, np.finfo(np.float32).tiny,
                           _f32(1), -_f32(1)], dtype=np.float32))
    v = np.concatenate(parts).astype(np.float32)
    return v[~np.isnan(v)]


def test_encode_fp32_sample_vs_brute_force(oracle_mod):
    rng = np.random.default_rng(1234)
    vals = _fp32_sample(rng)
    got = oracle_mod.e4m3_encode(vals)
    want = brute_encode(vals.astype(np.float64))
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(float(vals[i]), hex(got[i]), hex(want[i])) for i in bad[:8]]


def test_encode_vs_library_cast(oracle_mod):
    """torch's float32 -> float8_e4m3fn cast (round to nearest even) agrees
    wherever it is defined without saturation (|v| <= 448)."""
    rng = np.random.default_rng(7)
    bits = np.arange(65536, dtype=np.uint32) << 16
    vals = np.concatenate([_f32(bits), _fp32_sample(rng)])
    vals = vals[np.isfinite(vals) & (np.abs(vals) <= 448.0)]
    lib = torch.from_numpy(vals.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle_mod.e4m3_encode(vals)
    bad = np.nonzero(got != lib)[0]
    assert bad.size == 0, [(float(vals[i]), hex(got[i]), hex(lib[i])) for i in bad[:8]]


def test_check_range_helper(oracle_mod):
    """The bulk comparison helper counts mismatches correctly."""
    lo = 0x3F800000                      # 1.0f
    vals = _f32(np.arange(lo, lo + 4096, dtype=np.uint64).astype(np.uint32))
    codes = brute_encode(vals.astype(np.float64))
    assert oracle_mod.e4m3_encode_check_range(lo, codes) == (0, -1)
    codes[100] ^= 1
    assert oracle_mod.e4m3_encode_check_range(lo, codes) == (1, 100)
