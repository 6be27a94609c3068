"""Pins for the oracle's group quantisers (CPU only).

Checked against what the definitions fix, not against a retyped formula:
  * hand-worked groups (golden files) with exact scales and every rounding
    case (ties to even, subnormals, underflow to signed zero, saturation);
  * each group's amax element maps to +-448 whenever its scale is normal;
  * all-zero groups give scale 0 and codes 0x00;
  * power-of-two scales reproduce E4M3-representable groups exactly;
  * with scale 1 every |x| <= 448 bf16 value encodes as the brute-force
    nearest E4M3 value;
  * the rounding error bound of a 3-bit-mantissa format;
  * layout invariants: row permutation equivariance, Q2(X) = Q1(X^T),
    Q3(W^T) = Q3(W)^T, transposed weight codes = codes^T.
"""
import numpy as np
import pytest
import torch

from conftest import read_golden
from e4m3_brute import TABLE, brute_encode


def bf16_bits(a):
    """float array -> bf16 bit patterns (exact for the values used here)."""
    t = torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_from_normal(shape, sigma, seed):
    g = torch.Generator().manual_seed(seed)
    t = (torch.randn(*shape, generator=g) * sigma).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def deq(q):
    return TABLE[q.astype(np.int64)]


def test_golden_worked_group(oracle_mod):
    rows = read_golden("group_1x128_worked.txt")
    assert rows[0][0] == "scale"
    scale = float(rows[0][1])
    x = np.zeros(128, dtype=np.float64)
    want = np.zeros(128, dtype=np.uint8)
    for idx, val, code, *_ in rows[1:]:
        x[int(idx)] = float(val)
        want[int(idx)] = int(code, 16)
    xb = bf16_bits(x)
    assert np.array_equal(oracle_mod.bf16_bits_to_f32(xb).astype(np.float64), x)  # exact inputs
    q, s = oracle_mod.quantize_act(xb.reshape(1, 128))
    assert s.shape == (1, 1) and s[0, 0] == np.float32(scale)
    bad = np.nonzero(q[0] != want)[0]
    assert bad.size == 0, [(int(i), x[i], hex(q[0, i]), hex(want[i])) for i in bad]


def test_golden_nonpow2_scale(oracle_mod):
    rows = read_golden("group_nonpow2_scale.txt")
    sbits = int(rows[0][1], 16)
    x = np.zeros(128, dtype=np.float64)
    want = np.zeros(128, dtype=np.uint8)
    for idx, val, code in rows[1:]:
        x[int(idx)] = float(val)
        want[int(idx)] = int(code, 16)
    q, s = oracle_mod.quantize_act(bf16_bits(x).reshape(1, 128))
    assert s.view(np.uint32)[0, 0] == sbits
    assert np.array_equal(q[0], want)


def _normal_scale_groups(s):
    return s >= np.float32(np.finfo(np.float32).tiny)


def test_amax_maps_to_448(oracle_mod):
    xb = bf16_from_normal((64, 512), 1.0, 0)
    x = oracle_mod.bf16_bits_to_f32(xb)
    q, s = oracle_mod.quantize_act(xb)
    for g in range(4):
        blk = x[:, g * 128:(g + 1) * 128]
        arg = np.argmax(np.abs(blk), axis=1)
        codes = q[np.arange(64), g * 128 + arg]
        sign = np.signbit(blk[np.arange(64), arg])
        assert np.all(codes == np.where(sign, 0xFE, 0x7E))
        assert np.all(_normal_scale_groups(s[g]))
    # transposed and weight quantisers too
    qt, st = oracle_mod.quantize_act_transposed(bf16_from_normal((256, 128), 1e-2, 1))
    assert np.all((np.max(qt & 0x7F, axis=1) == 0x7E))
    qw, sw, _ = oracle_mod.quantize_weight(bf16_from_normal((256, 256), 0.02, 2))
    for bn in range(2):
        for bk in range(2):
            blk = qw[bn * 128:(bn + 1) * 128, bk * 128:(bk + 1) * 128]
            assert (blk & 0x7F).max() == 0x7E


def test_tiny_amax_subnormal_scales(oracle_mod):
    """Very small groups: the scale is an fp32 subnormal (no flush to zero)
    and is still amax/448 rounded once."""
    x = np.zeros((1, 128), np.float32)
    x[0, 0] = 2.0 ** -130           # bf16 subnormal
    x[0, 1] = -(2.0 ** -131)
    xb = bf16_bits(x)
    q, s = oracle_mod.quantize_act(xb)
    want_s = np.float32(2.0 ** -130) / np.float32(448.0)
    assert s[0, 0] == want_s and s[0, 0] > 0
    assert s[0, 0] < np.finfo(np.float32).tiny
    # quotient is finite and the codes are the nearest E4M3 of the fp32 quotient
    xf = oracle_mod.bf16_bits_to_f32(xb)[0]
    quot = (xf / s[0, 0]).astype(np.float32)
    assert np.array_equal(q[0], brute_encode(quot.astype(np.float64)))


def test_zero_groups(oracle_mod):
    x = np.zeros((3, 256), np.float32)
    x[1, 130] = 1.5                  # only group 1 of row 1 is non-zero
    x[2, 5] = -0.0
    q, s = oracle_mod.quantize_act(bf16_bits(x))
    assert s[1, 1] == np.float32(1.5) / np.float32(448)
    s_mask = np.ones_like(s, dtype=bool)
    s_mask[1, 1] = False
    assert np.all(s[s_mask] == 0)
    assert np.count_nonzero(q) == 1 and q[1, 130] == 0x7E
    qt, st = oracle_mod.quantize_act_transposed(np.zeros((128, 128), np.uint16))
    assert not qt.any() and not st.any()
    qw, sw, qwt = oracle_mod.quantize_weight(np.zeros((128, 256), np.uint16), True)
    assert not qw.any() and not sw.any() and not qwt.any()


def test_power_of_two_scale_is_exact(oracle_mod):
    """A group made of E4M3 values times 2^e with 448*2^e present has
    s = 2^e exactly, so it quantises and dequantises without error."""
    rng = np.random.default_rng(3)
    finite = TABLE[np.isfinite(TABLE)]
    for e in (-20, -7, 0, 3):
        vals = rng.choice(finite, size=(4, 128))
        vals[:, 17] = 448.0
        x = vals * 2.0 ** e
        xb = bf16_bits(x)
        assert np.array_equal(oracle_mod.bf16_bits_to_f32(xb).astype(np.float64), x)
        q, s = oracle_mod.quantize_act(xb)
        assert np.all(s == np.float32(2.0 ** e))
        assert np.array_equal(deq(q) * 2.0 ** e, x)


def test_scale_one_all_bf16(oracle_mod):
    """With amax = 448 the scale is exactly 1, so each code is simply the
    nearest E4M3 value of the bf16 input: checked for every bf16 |x| <= 448."""
    bits = np.arange(65536, dtype=np.uint32) << 16
    v = oracle_mod.bf16_bits_to_f32((bits >> 16).astype(np.uint16))
    v = v[np.isfinite(v) & (np.abs(v) <= 448.0)]
    n = (v.size + 126) // 127 * 127
    pad = np.zeros(n, np.float32)
    pad[:v.size] = v
    rows = pad.reshape(-1, 127)
    x = np.concatenate([np.full((rows.shape[0], 1), 448.0, np.float32), rows], axis=1)
    q, s = oracle_mod.quantize_act(bf16_bits(x))
    assert np.all(s == 1.0)
    want = brute_encode(x.astype(np.float64))
    assert np.array_equal(q, want)


def test_error_bound(oracle_mod):
    """|deq - x| <= s * max(2^-4 |x/s|, 2^-10) (3 mantissa bits, RNE;
    subnormal quantum 2^-9), with slack for the fp32 quotient rounding."""
    xb = bf16_from_normal((128, 1024), 3.0, 11)
    x = oracle_mod.bf16_bits_to_f32(xb).astype(np.float64)
    q, s = oracle_mod.quantize_act(xb)
    sfull = np.repeat(s.T.astype(np.float64), 128, axis=1)
    err = np.abs(deq(q) * sfull - x)
    bound = sfull * np.maximum(2.0 ** -4 * np.abs(x) / sfull, 2.0 ** -10) * (1 + 2.0 ** -20)
    assert np.all(err <= bound)


def test_row_permutation_equivariance(oracle_mod):
    xb = bf16_from_normal((96, 384), 1.0, 5)
    perm = np.random.default_rng(0).permutation(96)
    q, s = oracle_mod.quantize_act(xb)
    qp, sp = oracle_mod.quantize_act(xb[perm])
    assert np.array_equal(qp, q[perm]) and np.array_equal(sp, s[:, perm])


def test_transposed_equals_act_of_transpose(oracle_mod):
    xb = bf16_from_normal((256, 384), 1e-2, 6)
    qt, st = oracle_mod.quantize_act_transposed(xb)
    q1, s1 = oracle_mod.quantize_act(np.ascontiguousarray(xb.T))
    assert qt.shape == (384, 256) and st.shape == (2, 384)
    assert np.array_equal(qt, q1) and np.array_equal(st, s1)


def test_weight_transpose_symmetry(oracle_mod):
    wb = bf16_from_normal((256, 384), 0.02, 8)
    q, s, qt = oracle_mod.quantize_weight(wb, True)
    q2, s2, _ = oracle_mod.quantize_weight(np.ascontiguousarray(wb.T), False)
    assert np.array_equal(qt, q.T)
    assert np.array_equal(q2, q.T) and np.array_equal(s2, s.T)


def test_threads_do_not_change_results(oracle_mod):
    xb = bf16_from_normal((300, 256), 1.0, 9)
    a = oracle_mod.quantize_act(xb)
    b = oracle_mod.quantize_act(xb, threads=4)
    assert all(np.array_equal(u, v) for u, v in zip(a, b))
    xt = bf16_from_normal((256, 384), 1.0, 10)
    a = oracle_mod.quantize_act_transposed(xt)
    b = oracle_mod.quantize_act_transposed(xt, threads=3)
    assert all(np.array_equal(u, v) for u, v in zip(a, b))
    wb = bf16_from_normal((384, 256), 0.02, 12)
    a = oracle_mod.quantize_weight(wb, True)
    b = oracle_mod.quantize_weight(wb, True, threads=3)
    assert all(np.array_equal(u, v) for u, v in zip(a, b))
