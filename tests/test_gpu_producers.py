"""Fused producers on the GPU (RMSNorm -> FP8 and SwiGLU -> FP8) against the
oracle, bit for bit: the bf16 values y, the codes and the scales.  The codes
must also equal jetfp8_quantize_act applied to the kernel's own y.

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


def check_rmsnorm(x, gamma, eps, what):
    q, s, y = jf.rmsnorm_quantize_act(x, gamma, eps, want_y=True)
    assert jf.jetfp8_poll_device_error() == 0
    oy = oracle.rmsnorm(u16(x), u16(gamma), eps, threads=ORACLE_THREADS)
    assert_bitexact(y.view(torch.int16), oy.view(np.int16), f"{what} y")
    oq, os_ = oracle.quantize_act(oy, threads=ORACLE_THREADS)
    assert_bitexact(q, oq, f"{what} q")
    assert_bitexact(s, os_, f"{what} s")
    q2, s2 = jf.quantize_act(y)
    assert torch.equal(q, q2) and torch.equal(s, s2)
    return q, s, y


def check_swiglu(gu, what):
    q, s, y = jf.swiglu_quantize_act(gu, want_y=True)
    assert jf.jetfp8_poll_device_error() == 0
    oy = oracle.swiglu(u16(gu), threads=ORACLE_THREADS)
    assert_bitexact(y.view(torch.int16), oy.view(np.int16), f"{what} y")
    oq, os_ = oracle.quantize_act(oy, threads=ORACLE_THREADS)
    assert_bitexact(q, oq, f"{what} q")
    assert_bitexact(s, os_, f"{what} s")
    q2, s2 = jf.quantize_act(y)
    assert torch.equal(q, q2) and torch.equal(s, s2)
    return q, s, y


@pytest.mark.parametrize("M,H", [(1, 256), (7, 512), (256, 512), (1000, 4096), (333, 5120)])
def test_rmsnorm_bitexact(M, H):
    x = syn.activation(M, H, seed=M + H, outlier_scale=20.0, device=DEV)
    gamma = (syn.normal_bf16((H,), 0.1, seed=H, tensor="w", device=DEV) + 1.0).to(torch.bfloat16)
    check_rmsnorm(x, gamma, 1e-6, f"rmsnorm {M}x{H}")


def test_rmsnorm_special_rows():
    H = 512
    x = syn.activation(8, H, seed=3, student_t=True, outlier_scale=100.0, device=DEV)
    x[1] = 0                                   # zero row: y = 0 (eps > 0), s = 0
    x[2] = 3.0e38                              # huge values: the sum of squares overflows to inf
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


@pytest.mark.parametrize("M,I", [(1, 256), (7, 512), (256, 1536), (300, 14336), (64, 27648)])
def test_swiglu_bitexact(M, I):
    gu = syn.activation(M, 2 * I, seed=M + I, outlier_scale=20.0, device=DEV)
    check_swiglu(gu, f"swiglu {M}x{I}")


def test_swiglu_extreme_gates():
    I = 256
    g = torch.linspace(-120.0, 120.0, I, device=DEV)
    gu = torch.cat([g.expand(4, I), torch.randn(4, I, device=DEV) * 3], dim=1).to(torch.bfloat16).contiguous()
    gu[1, :I] = 0                          # silu(0) = 0
    gu[2, I:] = 0                          # up = 0
    gu[3, :I] = 88.5                       # e^-g small but normal; 1 + e^-g rounds to 1
    check_swiglu(gu, "swiglu extremes")


def test_swiglu_8b_training_size():
    gu = syn.activation(4096, 2 * 14336, seed=6, device=DEV)
    check_swiglu(gu, "swiglu 4096x14336")
