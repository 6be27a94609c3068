"""Pins for the parity bars themselves (test infrastructure the GEMM and
producer parity tests rest on).

  * ``bf16_ulp``: the spacing of bf16 numbers, checked against values the
    format fixes (8 significant bits, exponent range of fp32, subnormal
    spacing 2^-133) and against the spacing read off consecutive bf16 bit
    patterns for every positive finite bf16 value and the midpoints between
    them;
  * ``gemm_within_tolerance``: accepts the correctly rounded result, and
    rejects the results of plausible kernel mistakes planted in the oracle
    on the CPU (one K group dropped, a scale read one group off, a transposed
    scale index), on the tiny layer and on a 32-group contraction.
"""
import numpy as np
import pytest

import oracle
from e4m3_group_quantise_gb300 import synthetic as syn


# ---------------------------------------------------------------- bf16_ulp
@pytest.mark.parametrize("v,ulp", [
    (1.0, 2.0 ** -7), (1.99, 2.0 ** -7), (2.0, 2.0 ** -6), (-3.0, 2.0 ** -6), (0.75, 2.0 ** -8),
    (448.0, 2.0 ** 1), (3.0e38, 2.0 ** 120),
    (2.0 ** -126, 2.0 ** -133), (2.0 ** -130, 2.0 ** -133), (0.0, 2.0 ** -133), (-1e-42, 2.0 ** -133),
])
def test_bf16_ulp_values_the_format_fixes(v, ulp):
    assert oracle.bf16_ulp(np.array([v]))[0] == ulp


def test_bf16_ulp_matches_consecutive_bit_patterns():
    """For every positive finite bf16 value v below the largest, the distance to
    the next bf16 value up (bit pattern + 1) equals bf16_ulp(v) and
    bf16_ulp of the midpoint between them."""
    bits = np.arange(1, 0x7F7F, dtype=np.uint32)          # +min subnormal .. just below the largest finite
    v = oracle.bf16_bits_to_f32(bits.astype(np.uint16)).astype(np.float64)
    nxt = oracle.bf16_bits_to_f32((bits + 1).astype(np.uint16)).astype(np.float64)
    gap = nxt - v
    assert np.array_equal(oracle.bf16_ulp(v), gap)
    assert np.array_equal(oracle.bf16_ulp(-v), gap)
    assert np.array_equal(oracle.bf16_ulp(v + gap / 2), gap)


def test_bf16_within_ulp():
    ref = np.array([1.0, 1.0 + 2.0 ** -8, 3.0, -2.0 ** -128])
    got = syn.np_f32_to_bf16_bits(np.array([1.0, 1.0 + 2.0 ** -7, 3.0 + 2.0 ** -6, -2.0 ** -128], np.float32))
    ok, worst, idx = oracle.bf16_within_ulp(got, ref)
    assert ok and worst == 1.0 and idx == 2
    got2 = syn.np_f32_to_bf16_bits(np.array([1.0, 1.0, 3.0 + 2.0 ** -4, -2.0 ** -128], np.float32))
    ok, worst, idx = oracle.bf16_within_ulp(got2, ref)
    assert not ok and idx == 2


# ---------------------------------------------------------------- the GEMM bar
def _tiny(K=512, M=256, N=512, seed=0):
    x = syn.activation(M, K, seed=seed)
    w = syn.weight(N, K, seed=seed)
    qx, sx = oracle.quantize_act(syn.bf16_bits(x))
    qw, sw, _ = oracle.quantize_weight(syn.bf16_bits(w))
    return qx, sx, qw, sw


def _bf16(v):
    return oracle.bf16_bits_to_f32(syn.np_f32_to_bf16_bits(v.astype(np.float32))).astype(np.float64)


@pytest.mark.parametrize("K", [512, 4096])
def test_gemm_bar_accepts_the_rounded_result_and_rejects_planted_mistakes(K):
    M, N = (256, 512) if K == 512 else (128, 256)
    qx, sx, qw, sw = _tiny(K, M, N)
    ref, asum = oracle.gemm_fprop(qx, sx, qw, sw, threads=8)
    # the exact result rounded to bf16 (what a perfect kernel returns) passes
    ok, worst, _ = oracle.gemm_within_tolerance(_bf16(ref), ref, asum)
    assert ok and worst <= 0.5

    # one K group dropped (its activation scales zeroed)
    sx_drop = sx.copy()
    sx_drop[K // 256] = 0.0
    bad, _ = oracle.gemm_fprop(qx, sx_drop, qw, sw, threads=8)
    ok, worst, _ = oracle.gemm_within_tolerance(_bf16(bad), ref, asum)
    assert not ok, f"dropping one of {K // 128} groups stayed within the bar (worst {worst:.3g})"

    # activation scales read one group off (group g uses group g+1's scale)
    sx_shift = np.roll(sx, -1, axis=0)
    bad, _ = oracle.gemm_fprop(qx, sx_shift, qw, sw, threads=8)
    ok, worst, _ = oracle.gemm_within_tolerance(_bf16(bad), ref, asum)
    assert not ok, f"shifted scales stayed within the bar (worst {worst:.3g})"

    # weight block scales indexed transposed ([K/128][N/128] read as [N/128][K/128])
    if sw.shape[0] == sw.shape[1]:
        sw_t = np.ascontiguousarray(sw.T)
    else:
        sw_t = np.ascontiguousarray(sw.T.reshape(sw.shape))
    bad, _ = oracle.gemm_fprop(qx, sx, qw, sw_t, threads=8)
    ok, worst, _ = oracle.gemm_within_tolerance(_bf16(bad), ref, asum)
    assert not ok, f"transposed weight-scale index stayed within the bar (worst {worst:.3g})"
