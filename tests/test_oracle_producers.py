"""Pins for the oracle's fused-producer definitions (RMSNorm and SwiGLU in
front of the linear layers; their FP8 form is quantize_act of the result).

Each function is checked against what mathematics and independent libraries
fix, not against a retyping of itself:
  * fp32 -> bf16 rounding: PyTorch's own conversion, bit for bit, including
    exact ties and special values;
  * e^x: float64 numpy exp within 2 fp32 ulps over the whole normal range,
    exact special values, monotonicity;
  * SwiGLU: float64 silu(g) * u within one bf16 ulp, exact limits;
  * RMSNorm: float64 RMSNorm within one bf16 ulp, exact closed forms
    (constant rows, zero rows, power-of-two scale invariance).
"""
import numpy as np
import pytest
import torch

import oracle

RNG = np.random.default_rng(2024)


def bf16_to_f64(bits):
    return oracle.bf16_bits_to_f32(bits).astype(np.float64)


def bf16_ulp(v):
    return oracle.bf16_ulp(v)


def to_bf16_bits(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------- fp32 -> bf16
def test_float_to_bf16_matches_torch():
    bits = RNG.integers(0, 2**32, 1_000_000, dtype=np.uint64).astype(np.uint32)
    # exact ties and their neighbours, every exponent
    ties = (RNG.integers(0, 2**16, 100_000, dtype=np.uint64).astype(np.uint32) << 16) | 0x8000
    allb = np.concatenate([bits, ties, ties + 1, ties - 1]).astype(np.uint32)
    f = allb.view(np.float32)
    f = f[~np.isnan(f)]
    specials = np.array([0.0, -0.0, np.inf, -np.inf, 3.3895314e38, 3.4028235e38, 1e-45, -1e-45, 1.17549435e-38],
                        dtype=np.float32)
    f = np.concatenate([f, specials])
    assert np.array_equal(oracle.float_to_bf16_bits(f), to_bf16_bits(f))


# ---------------------------------------------------------------- exp
def test_exp_within_two_ulp_of_float64():
    x = np.concatenate([np.linspace(-87.0, 88.7, 2_000_001, dtype=np.float32),
                        RNG.uniform(-87, 88.7, 500_000).astype(np.float32),
                        RNG.uniform(-1, 1, 500_000).astype(np.float32)])
    got = oracle.exp_f32(x).astype(np.float64)
    ref = np.exp(x.astype(np.float64))
    ulp = np.spacing(ref.astype(np.float32)).astype(np.float64)
    err = np.abs(got - ref) / ulp
    assert err.max() <= 2.0, (err.max(), x[np.argmax(err)])
    assert np.mean(err <= 0.5) > 0.9             # mostly correctly rounded


def test_exp_special_values_and_monotone():
    e = oracle.exp_f32
    assert e(np.float32([0.0]))[0] == 1.0
    assert e(np.float32([-0.0]))[0] == 1.0
    assert np.isposinf(e(np.float32([89.0, 100.0, np.inf]))).all()
    assert (e(np.float32([-87.5, -100.0, -np.inf])) == 0.0).all()
    assert np.isnan(e(np.float32([np.nan])))[0]
    x = np.linspace(-87.0, 88.7, 1_000_001, dtype=np.float32)
    y = e(x)
    assert np.all(np.diff(y.astype(np.float64)) >= 0)


# ---------------------------------------------------------------- SwiGLU
def swiglu_f64(gu_bits):
    g64 = bf16_to_f64(gu_bits)
    I = g64.shape[1] // 2
    g, u = g64[:, :I], g64[:, I:]
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g)) * u


def test_swiglu_within_one_bf16_ulp():
    g = RNG.standard_normal((64, 512)) * 3
    u = RNG.standard_normal((64, 512))
    gu = to_bf16_bits(np.concatenate([g, u], axis=1))
    y = oracle.swiglu(gu)
    got = bf16_to_f64(y)
    ref = swiglu_f64(gu)
    assert np.all(np.abs(got - ref) <= bf16_ulp(ref) * 1.0001)
    # against PyTorch's own silu (an independent e^x)
    gt = torch.from_numpy(oracle.bf16_bits_to_f32(gu[:, :512]))
    ut = torch.from_numpy(oracle.bf16_bits_to_f32(gu[:, 512:]))
    tref = (torch.nn.functional.silu(gt) * ut).double().numpy()
    assert np.all(np.abs(got - tref) <= bf16_ulp(tref) * 1.0001)


def test_swiglu_exact_limits():
    g = np.float32([[0.0, 20.0, -100.0, 100.0, -0.0, 1.0]])
    u = np.float32([[3.0, 1.5, 2.0, -0.25, 5.0, 0.0]])
    gu = to_bf16_bits(np.concatenate([g, u], axis=1))
    y = oracle.bf16_bits_to_f32(oracle.swiglu(gu))[0]
    assert y[0] == 0.0                     # silu(0) = 0
    assert y[1] == 30.0                    # e^-20 vanishes next to 1: silu(g) = g exactly
    assert y[2] == 0.0 and np.signbit(y[2])   # e^100 = inf: sigmoid 0, silu(-100) = -0
    assert y[3] == -25.0
    assert y[5] == 0.0


# ---------------------------------------------------------------- RMSNorm
def rmsnorm_f64(x_bits, g_bits, eps):
    x = bf16_to_f64(x_bits)
    g = bf16_to_f64(g_bits)
    return x / np.sqrt(np.mean(x * x, axis=1, keepdims=True) + eps) * g


@pytest.mark.parametrize("H", [256, 512, 4096, 5120])
def test_rmsnorm_within_one_bf16_ulp(H):
    x = to_bf16_bits(RNG.standard_normal((16, H)) * RNG.uniform(0.01, 100, (16, 1)))
    g = to_bf16_bits(RNG.uniform(0.5, 1.5, H))
    y = oracle.rmsnorm(x, g, 1e-6)
    got = bf16_to_f64(y)
    ref = rmsnorm_f64(x, g, 1e-6)
    assert np.all(np.abs(got - ref) <= bf16_ulp(ref) * 1.0001)


def test_rmsnorm_closed_forms():
    H = 512
    ones = to_bf16_bits(np.ones(H))
    # a row of +-c (power of two), gain 1, eps 0: exactly +-1
    c = 0.25
    signs = RNG.choice([-1.0, 1.0], H)
    y = oracle.bf16_bits_to_f32(oracle.rmsnorm(to_bf16_bits([signs * c]), ones, 0.0))[0]
    assert np.array_equal(y, signs.astype(np.float32))
    # a zero row with eps > 0: exactly 0
    y = oracle.rmsnorm(to_bf16_bits(np.zeros((1, H))), ones, 1e-5)
    assert not y.any() or np.all((y & 0x7FFF) == 0)
    # eps = 0: scaling the row by a power of two changes nothing, bit for bit
    x = RNG.standard_normal((4, H))
    g = to_bf16_bits(RNG.uniform(0.5, 1.5, H))
    a = oracle.rmsnorm(to_bf16_bits(x), g, 0.0)
    b = oracle.rmsnorm(to_bf16_bits(x * 8.0), g, 0.0)
    assert np.array_equal(a, b)
    # the gain multiplies last: gain 2 doubles every output exactly
    two = to_bf16_bits(np.full(H, 2.0))
    a1 = oracle.bf16_bits_to_f32(oracle.rmsnorm(to_bf16_bits(x), ones, 1e-6))
    a2 = oracle.bf16_bits_to_f32(oracle.rmsnorm(to_bf16_bits(x), two, 1e-6))
    assert np.array_equal(a2, 2 * a1)


def test_rmsnorm_rejects_bad_width():
    with pytest.raises(ValueError):
        oracle.rmsnorm(to_bf16_bits(np.ones((1, 384))), to_bf16_bits(np.ones(384)), 1e-6)
