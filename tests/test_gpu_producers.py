"""Fused producers on the GPU (RMSNorm -> FP8 and SwiGLU -> FP8) against the
oracle: the kernel's bf16 values y within one bf16 ulp of the operators'
fp64 values, and its codes and scales bit for bit equal to the oracle's
quantize_act of that bf16 y (and to jetfp8_quantize_act of it).

Domain (stated, not hidden): RMSNorm rows whose sum of squares overflows
fp32 are outside the contract; for SwiGLU gates g < -87 the exact result is
below 2^-119 |u| in magnitude and the kernel's fp32 sigmoid underflows, so
there the bar is an absolute 2^-119 |u| (plus one ulp).

Shapes: tiny and ragged row counts, the toy decoder (hidden 512, intermediate
1536), the 8B-class hidden 4096 / intermediate 14336 and the 32B-class
hidden 5120 at thousands of tokens; inputs with outlier channels, Student-t
tails, zero rows and extreme gate values (e^-g overflowing and vanishing).
"""
import numpy as np
import pytest
import torch

import oracle
import e4m3_group_quantise_gb300 as jf
from e4m3_group_quantise_gb300 import synthetic as syn
from gpu_util import ORACLE_THREADS, assert_bitexact, bits, require_gpu

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def u16(t):
    return bits(t)


def check_codes_of_own_y(q, s, y, what):
    """Codes and scales: the oracle's quantize_act of the kernel's own bf16 y,
    bit for bit, and the library's quantize_act of it."""
    oq, os_ = oracle.quantize_act(u16(y), threads=ORACLE_THREADS)
    assert_bitexact(q, oq, f"{what} q")
    assert_bitexact(s, os_, f"{what} s")
    q2, s2 = jf.quantize_act(y)
    assert torch.equal(q, q2) and torch.equal(s, s2)


def check_rmsnorm(x, gamma, eps, what):
    q, s, y = jf.rmsnorm_quantize_act(x, gamma, eps, want_y=True)
    assert jf.jetfp8_poll_device_error() == 0
    oy = oracle.rmsnorm(u16(x), u16(gamma), eps, threads=ORACLE_THREADS)
    ok, worst, idx = oracle.bf16_within_ulp(u16(y), oy)
    assert ok, f"{what} y: {worst:.3g} bf16 ulps from the fp64 RMSNorm at flat index {idx}"
    check_codes_of_own_y(q, s, y, what)
    return q, s, y


def check_swiglu(gu, what):
    q, s, y = jf.swiglu_quantize_act(gu, want_y=True)
    assert jf.jetfp8_poll_device_error() == 0
    oy = oracle.swiglu(u16(gu), threads=ORACLE_THREADS)
    I = oy.shape[1]
    g64 = oracle.bf16_bits_to_f32(u16(gu)).astype(np.float64)
    gate, up = g64[:, :I], g64[:, I:]
    got = oracle.bf16_bits_to_f32(u16(y)).astype(np.float64)
    err = np.abs(got - oy)
    bound = oracle.bf16_ulp(oy) + np.where(gate < -87.0, 2.0 ** -119 * np.abs(up), 0.0)
    assert np.all(err <= bound), f"{what} y: worst error / bound {np.max(err / bound):.3g}"
    check_codes_of_own_y(q, s, y, what)
    return q, s, y


@pytest.mark.parametrize("M,H", [(1, 256), (7, 512), (256, 512), (1000, 4096), (333, 5120),
                                 (37, 33024), (5, 65536)])
def test_rmsnorm_parity(M, H):
    """Includes rows wider than 32768 columns (one warp per row, eight values
    per lane, the row read twice)."""
    x = syn.activation(M, H, seed=M + H, outlier_scale=20.0, device=DEV)
    gamma = (syn.normal_bf16((H,), 0.1, seed=H, tensor="w", device=DEV) + 1.0).to(torch.bfloat16)
    check_rmsnorm(x, gamma, 1e-6, f"rmsnorm {M}x{H}")


def test_rmsnorm_special_rows():
    H = 512
    x = syn.activation(8, H, seed=3, student_t=True, outlier_scale=100.0, device=DEV)
    x[1] = 0                                   # zero row: y = 0 (eps > 0), s = 0
    x[2] = 4.0e17                              # huge values (sum of squares 8e37, still finite in fp32)
    x[3, :] = 0
    x[3, 5] = -1e-30                           # one tiny value
    gamma = torch.ones(H, dtype=torch.bfloat16, device=DEV)
    q, s, y = check_rmsnorm(x, gamma, 1e-5, "rmsnorm special")
    assert not y[1].any() and not s[:, 1].any()


def test_rmsnorm_modes_and_empty():
    x = syn.activation(64, 1024, seed=4, device=DEV)
    gamma = torch.ones(1024, dtype=torch.bfloat16, device=DEV)
    q1, s1, _ = jf.rmsnorm_quantize_act(x, gamma, 1e-6)                  # codes only
    _, _, y = jf.rmsnorm_quantize_act(x, gamma, 1e-6, quantize=False)    # y only
    q2, s2 = jf.quantize_act(y)
    assert torch.equal(q1, q2) and torch.equal(s1, s2)
    e = torch.empty(0, 1024, dtype=torch.bfloat16, device=DEV)
    q, s, _ = jf.rmsnorm_quantize_act(e, gamma, 1e-6)
    assert q.shape == (0, 1024)


def test_rmsnorm_8b_training_size():
    x = syn.activation(16384, 4096, seed=5, outlier_scale=20.0, device=DEV)
    gamma = (syn.normal_bf16((4096,), 0.1, seed=5, tensor="w", device=DEV) + 1.0).to(torch.bfloat16)
    check_rmsnorm(x, gamma, 1e-6, "rmsnorm 16384x4096")


def many_rows():
    """A row count of several rows per SM plus a ragged remainder."""
    return 8 * torch.cuda.get_device_properties(0).multi_processor_count + 37


@pytest.mark.parametrize("H", [256, 5120, 16384])
def test_rmsnorm_parity_many_rows(H):
    """One warp per row (H 256, eight rows per block), five warps of one quad
    per thread (5120, one row per block), eight warps of two quads (16384)."""
    M = many_rows()
    x = syn.activation(M, H, seed=H + 1, outlier_scale=20.0, device=DEV)
    gamma = (syn.normal_bf16((H,), 0.1, seed=H, tensor="w", device=DEV) + 1.0).to(torch.bfloat16)
    check_rmsnorm(x, gamma, 1e-6, f"rmsnorm {M}x{H}")


@pytest.mark.parametrize("H", [4096, 8192, 16384, 32768, 33024])
def test_rmsnorm_rows_batch_invariant(H):
    """A row's bits do not depend on the batch: rows of a large batch equal
    the same rows normalised alone or in small batches (one to sixteen warps
    per row, one or two quads per thread)."""
    M = many_rows()
    x = syn.activation(M, H, seed=H + 2, outlier_scale=20.0, device=DEV)
    gamma = (syn.normal_bf16((H,), 0.1, seed=H + 3, tensor="w", device=DEV) + 1.0).to(torch.bfloat16)
    q, s, y = jf.rmsnorm_quantize_act(x, gamma, 1e-6, want_y=True)
    assert jf.jetfp8_poll_device_error() == 0
    for a, b in [(0, 1), (5, 69), (M - 40, M)]:
        qa, sa, ya = jf.rmsnorm_quantize_act(x[a:b].contiguous(), gamma, 1e-6, want_y=True)
        assert torch.equal(ya, y[a:b]) and torch.equal(qa, q[a:b]) and torch.equal(sa, s[:, a:b])


@pytest.mark.parametrize("M,I", [(1, 256), (7, 512), (256, 1536), (300, 14336), (64, 27648)])
def test_swiglu_parity(M, I):
    gu = syn.activation(M, 2 * I, seed=M + I, outlier_scale=20.0, device=DEV)
    check_swiglu(gu, f"swiglu {M}x{I}")


def test_swiglu_extreme_gates():
    I = 256
    g = torch.linspace(-120.0, 120.0, I, device=DEV)
    gu = torch.cat([g.expand(4, I), torch.randn(4, I, device=DEV) * 3], dim=1).to(torch.bfloat16).contiguous()
    gu[1, :I] = 0                          # silu(0) = 0
    gu[2, I:] = 0                          # up = 0
    gu[3, :I] = 88.5                       # e^-g below fp32's normal range: 1 + e^-g rounds to 1
    check_swiglu(gu, "swiglu extremes")


def test_swiglu_8b_training_size():
    gu = syn.activation(4096, 2 * 14336, seed=6, device=DEV)
    check_swiglu(gu, "swiglu 4096x14336")


def test_producers_negative_zero_outputs():
    """bf16 outputs of -0 inside groups with nonzero values (the quantiser
    takes the correctly rounded division for a lane holding a -0): RMSNorm of
    zeros under negative gamma, SwiGLU of zero gates with negative up values."""
    H = 1024
    x = syn.activation(16, H, seed=7, device=DEV)
    x[:, ::7] = 0
    gamma = torch.ones(H, dtype=torch.bfloat16, device=DEV)
    gamma[::2] = -1.0
    q, s, y = check_rmsnorm(x, gamma, 1e-6, "rmsnorm -0")
    assert (u16(y) == 0x8000).any() and bool((s > 0).all())
    I = 512
    gu = syn.activation(16, 2 * I, seed=8, device=DEV)
    gu[:, :I:5] = 0                                  # gates of 0: silu(0) = +0
    gu[:, I::5] = -gu[:, I::5].abs() - 0.5           # negative up values there: y = -0
    q, s, y = check_swiglu(gu, "swiglu -0")
    assert (u16(y) == 0x8000).any() and bool((s > 0).all())
