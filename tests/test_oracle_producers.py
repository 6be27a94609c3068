"""Pins for the oracle's fused-producer definitions (RMSNorm and SwiGLU in
front of the linear layers, evaluated in fp64; their FP8 form is
quantize_act of a kernel's bf16 result).

Each function is checked against what mathematics and independent libraries
fix, not against a retyping of itself:
  * hand-worked values (tests/golden/rmsnorm_swiglu_examples.txt);
  * RMSNorm: closed forms (constant rows, one-hot rows, zero rows), exact
    power-of-two scale invariance, the gain applied last, the unit mean
    square of the normalised row, and PyTorch's own float64 rms_norm;
  * SwiGLU: silu(g) - silu(-g) = g, the limits, and PyTorch's float64 silu.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from conftest import read_golden

RNG = np.random.default_rng(2024)


def to_bf16_bits(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_to_f64(bits):
    return oracle.bf16_bits_to_f32(bits).astype(np.float64)


def _entries(tokens, H):
    """'i:v' or 'a-b:v' tokens -> dense float64 vector of length H."""
    v = np.zeros(H)
    for t in tokens:
        idx, val = t.split(":")
        if "-" in idx:
            a, b = (int(u) for u in idx.split("-"))
            v[a:b + 1] = float(val)
        else:
            v[int(idx)] = float(val)
    return v


def test_golden_examples():
    rows = read_golden("rmsnorm_swiglu_examples.txt")
    assert len(rows) >= 9
    for r in rows:
        arrow = r.index("->")
        if r[0] == "rmsnorm":
            H, eps, gain = int(r[1]), float(r[2]), float(r[3])
            x = _entries(r[4:arrow], H)
            want = _entries(r[arrow + 1:], H)
            got = oracle.rmsnorm(to_bf16_bits([x]), to_bf16_bits(np.full(H, gain)), eps)[0]
            np.testing.assert_allclose(got, want, rtol=4e-16, atol=0, err_msg=" ".join(r))
        else:
            g, u = float(r[1]), float(r[2])
            want = float(r[arrow + 1])
            got = oracle.swiglu(to_bf16_bits([[g, u]]))[0, 0]
            assert got == pytest.approx(want, rel=4e-16, abs=0), r


# ---------------------------------------------------------------- RMSNorm
def test_rmsnorm_closed_forms():
    H = 512
    ones = to_bf16_bits(np.ones(H))
    # a row of +-c (power of two), gain 1, eps 0: exactly +-1
    signs = RNG.choice([-1.0, 1.0], H)
    y = oracle.rmsnorm(to_bf16_bits([signs * 0.25]), ones, 0.0)[0]
    assert np.array_equal(y, signs)
    # a zero row with eps > 0: exactly 0
    y = oracle.rmsnorm(to_bf16_bits(np.zeros((1, H))), ones, 1e-5)
    assert not y.any()
    # one non-zero value a among H = 4096: rms = |a| / 64, y = 64 sign(a)
    x = np.zeros((1, 4096))
    x[0, 100] = -0.375
    y = oracle.rmsnorm(to_bf16_bits(x), to_bf16_bits(np.ones(4096)), 0.0)[0]
    assert y[100] == -64.0 and np.count_nonzero(y) == 1


def test_rmsnorm_invariants():
    H = 1024
    x = RNG.standard_normal((6, H)) * RNG.uniform(0.01, 100, (6, 1))
    g = to_bf16_bits(RNG.uniform(0.5, 1.5, H))
    ones = to_bf16_bits(np.ones(H))
    # eps = 0: scaling the row by a power of two changes nothing, bit for bit
    a = oracle.rmsnorm(to_bf16_bits(x), g, 0.0)
    b = oracle.rmsnorm(to_bf16_bits(x * 8.0), g, 0.0)
    assert np.array_equal(a, b)
    # the gain multiplies last: gain 2 doubles every output exactly
    a1 = oracle.rmsnorm(to_bf16_bits(x), ones, 1e-6)
    a2 = oracle.rmsnorm(to_bf16_bits(x), to_bf16_bits(np.full(H, 2.0)), 1e-6)
    assert np.array_equal(a2, 2 * a1)
    # with gain 1 and eps 0 the normalised row has mean square 1
    u = oracle.rmsnorm(to_bf16_bits(x), ones, 0.0)
    np.testing.assert_allclose(np.mean(u * u, axis=1), 1.0, rtol=1e-13)
    # eps enters under the root: mean square of y = ms / (ms + eps)
    xb = bf16_to_f64(to_bf16_bits(x))
    ms = np.mean(xb * xb, axis=1)
    eps = float(np.float32(0.5))
    v = oracle.rmsnorm(to_bf16_bits(x), ones, eps)
    np.testing.assert_allclose(np.mean(v * v, axis=1), ms / (ms + eps), rtol=1e-13)


@pytest.mark.parametrize("H", [256, 512, 4096, 5120])
def test_rmsnorm_against_torch_float64(H):
    """PyTorch's own rms_norm (an independent implementation) in float64."""
    x = to_bf16_bits(RNG.standard_normal((16, H)) * RNG.uniform(0.01, 100, (16, 1)))
    g = to_bf16_bits(RNG.uniform(0.5, 1.5, H))
    got = oracle.rmsnorm(x, g, 1e-6)
    xt = torch.from_numpy(bf16_to_f64(x))
    gt = torch.from_numpy(bf16_to_f64(g))
    ref = torch.nn.functional.rms_norm(xt, (H,), weight=gt, eps=float(np.float32(1e-6))).numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-300)


def test_rmsnorm_eps_taken_at_fp32():
    """The C-ABI passes eps as a float: the oracle rounds it the same way."""
    H = 256
    x = to_bf16_bits(np.zeros((1, H)))
    x[0, 0] = to_bf16_bits([1.0])[0]
    a = oracle.rmsnorm(x, to_bf16_bits(np.ones(H)), 0.1)
    b = oracle.rmsnorm(x, to_bf16_bits(np.ones(H)), float(np.float32(0.1)))
    assert np.array_equal(a, b)


def test_rmsnorm_rejects_bad_gain():
    with pytest.raises(ValueError):
        oracle.rmsnorm(to_bf16_bits(np.ones((1, 384))), to_bf16_bits(np.ones(256)), 1e-6)


# ---------------------------------------------------------------- SwiGLU
def test_swiglu_against_torch_float64():
    """PyTorch's float64 silu (an independent e^x) times up."""
    g = RNG.standard_normal((64, 512)) * 3
    u = RNG.standard_normal((64, 512))
    gu = to_bf16_bits(np.concatenate([g, u], axis=1))
    got = oracle.swiglu(gu)
    t = torch.from_numpy(bf16_to_f64(gu))
    ref = (torch.nn.functional.silu(t[:, :512]) * t[:, 512:]).numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-14, atol=1e-300)


def test_swiglu_odd_part_and_limits():
    # silu(g) - silu(-g) = g sigmoid(g) + g sigmoid(-g) = g
    g = bf16_to_f64(to_bf16_bits(RNG.uniform(-30, 30, 4096)))
    ones = np.ones_like(g)
    pos = oracle.swiglu(to_bf16_bits(np.concatenate([[g], [ones]], axis=1)))[0]
    neg = oracle.swiglu(to_bf16_bits(np.concatenate([[-g], [ones]], axis=1)))[0]
    np.testing.assert_allclose(pos - neg, g, rtol=1e-14, atol=1e-14)
    # limits: silu(g) -> g for large g, -> 0 (keeping the sign) for very negative g
    gu = to_bf16_bits([[100.0, -800.0, 0.0, 3.0, 2.0, 7.0, -5.0, 0.0]])
    y = oracle.swiglu(gu)[0]
    assert y[0] == 200.0                    # e^-100 vanishes next to 1
    assert y[1] == 0.0 and math.copysign(1.0, y[1]) < 0   # e^800 = inf: -800 / inf = -0
    assert y[2] == 0.0                      # silu(0) = 0
    assert y[3] == 0.0                      # up = 0
