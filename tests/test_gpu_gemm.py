"""GPU FP8 GEMMs (Fprop, Dgrad, Wgrad) vs the oracle's fp64 sums.

Bar, per element: |gpu - ref| <= 1e-3 * sum|a*b| + 1 bf16 ulp(ref).
The oracle quantises the inputs itself (its codes are first checked
bit-exact against the GPU's), then sums the dequantised products in fp64.
Shapes: tiny (full compare), ragged token counts that leave partial tiles,
narrow N (the 128-wide tile path), the 8B decode shapes and the 8B
training-step shapes at full size (sampled elements: four corner tiles,
first and last rows, 4096 seeded random elements).
"""
import numpy as np
import pytest
import torch

import oracle
import e4m3_group_quantise_gb300 as jf
from e4m3_group_quantise_gb300 import synthetic as syn
from gpu_util import ORACLE_THREADS, assert_bitexact, assert_gemm_close, bits, require_gpu, sample_indices

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def run_fprop(M, N, K, seed, sample=None, outliers=20.0):
    x = syn.activation(M, K, seed=seed, outlier_scale=outliers, device=DEV)
    w = syn.weight(N, K, seed=seed, device=DEV)
    qx, sx = jf.quantize_act(x)
    qw, sw, _ = jf.quantize_weight(w, transposed=False)
    y = jf.gemm_fprop(qx, sx, qw, sw)
    assert jf.jetfp8_poll_device_error() == 0
    ox = oracle.quantize_act(bits(x), threads=ORACLE_THREADS)
    ow = oracle.quantize_weight(bits(w), threads=ORACLE_THREADS)
    assert_bitexact(qx, ox[0], "qx")
    assert_bitexact(qw, ow[0], "qw")
    if sample is None:
        ref, asum = oracle.gemm_fprop(ox[0], ox[1], ow[0], ow[1], threads=ORACLE_THREADS)
        return assert_gemm_close(y, ref, asum, f"fprop {M}x{N}x{K}")
    r, c = sample_indices(M, N, sample, seed)
    ref, asum = oracle.gemm_fprop(ox[0], ox[1], ow[0], ow[1], r, c, threads=ORACLE_THREADS)
    return assert_gemm_close(y, ref, asum, f"fprop {M}x{N}x{K}", r, c)


def run_dgrad(M, N, K, seed, sample=None, sigma=1e-2):
    dy = syn.grad_output(M, N, seed=seed, device=DEV, sigma=sigma)
    w = syn.weight(N, K, seed=seed, device=DEV)
    qdy, sdy = jf.quantize_act(dy)
    qw, sw, qwt = jf.quantize_weight(w)
    dx = jf.gemm_dgrad(qdy, sdy, qwt, sw)
    assert jf.jetfp8_poll_device_error() == 0
    ody = oracle.quantize_act(bits(dy), threads=ORACLE_THREADS)
    ow = oracle.quantize_weight(bits(w), threads=ORACLE_THREADS)
    assert_bitexact(qdy, ody[0], "qdy")
    assert_bitexact(qw, ow[0], "qw")
    if sample is None:
        ref, asum = oracle.gemm_dgrad(ody[0], ody[1], ow[0], ow[1], threads=ORACLE_THREADS)
        return assert_gemm_close(dx, ref, asum, f"dgrad {M}x{N}x{K}")
    r, c = sample_indices(M, K, sample, seed)
    ref, asum = oracle.gemm_dgrad(ody[0], ody[1], ow[0], ow[1], r, c, threads=ORACLE_THREADS)
    return assert_gemm_close(dx, ref, asum, f"dgrad {M}x{N}x{K}", r, c)


def run_wgrad(M, N, K, seed, sample=None, sigma=1e-2, outliers=20.0):
    x = syn.activation(M, K, seed=seed, outlier_scale=outliers, device=DEV)
    dy = syn.grad_output(M, N, seed=seed, device=DEV, sigma=sigma)
    qxt, sxt = jf.quantize_act_transposed(x)
    qdyt, sdyt = jf.quantize_act_transposed(dy)
    dw = jf.gemm_wgrad(qdyt, sdyt, qxt, sxt)
    assert jf.jetfp8_poll_device_error() == 0
    oxt = oracle.quantize_act_transposed(bits(x), threads=ORACLE_THREADS)
    odyt = oracle.quantize_act_transposed(bits(dy), threads=ORACLE_THREADS)
    assert_bitexact(qxt, oxt[0], "qxt")
    assert_bitexact(qdyt, odyt[0], "qdyt")
    if sample is None:
        ref, asum = oracle.gemm_wgrad(odyt[0], odyt[1], oxt[0], oxt[1], threads=ORACLE_THREADS)
        return assert_gemm_close(dw, ref, asum, f"wgrad {M}x{N}x{K}")
    r, c = sample_indices(N, K, sample, seed)
    ref, asum = oracle.gemm_wgrad(odyt[0], odyt[1], oxt[0], oxt[1], r, c, threads=ORACLE_THREADS)
    return assert_gemm_close(dw, ref, asum, f"wgrad {M}x{N}x{K}", r, c)


# ------------------------------------------------------------ tiny, full compare
def test_tiny_layer_all_three():
    run_fprop(256, 512, 512, 0, outliers=0.0)
    run_dgrad(256, 512, 512, 0)
    run_wgrad(256, 512, 512, 0, outliers=0.0)


@pytest.mark.parametrize("M", [1, 7, 64, 129, 255, 300])
def test_fprop_ragged_tokens(M):
    run_fprop(M, 384, 640, M)


@pytest.mark.parametrize("N", [128, 384, 1024])
def test_fprop_narrow_and_partial_n(N):
    run_fprop(200, N, 256, N)


@pytest.mark.parametrize("M,N,K", [(1, 256, 128), (130, 640, 384), (300, 128, 256)])
def test_dgrad_ragged(M, N, K):
    run_dgrad(M, N, K, M + N)


@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (384, 384, 640), (1024, 128, 256)])
def test_wgrad_shapes(M, N, K):
    run_wgrad(M, N, K, M + K)


@pytest.mark.parametrize("M,N,K", [(384, 1024, 1024), (256, 2048, 1024), (128, 128, 4096)])
def test_wgrad_tile_widths(M, N, K):
    """Wgrad problems whose tile count makes the launcher pick 64-, 128- and
    32-wide tiles (output 1024 x 1024: 64; 2048 x 1024: 128; 128 x 4096: 32),
    each a different slab layout of the per-column-scale read-back."""
    run_wgrad(M, N, K, M + N + K)


def test_many_tiles_persistent_loop():
    """More tiles than SMs on every variant (each CTA walks several tiles)."""
    run_fprop(2048, 4096, 512, 5, sample=2048)
    run_dgrad(2048, 512, 4096, 6, sample=2048)
    run_wgrad(1024, 2048, 4096, 7, sample=2048)


def test_odd_tile_counts_and_ragged_rows():
    """Many tiles with an odd number of 128- and 256-column tiles per row of
    tiles and a ragged last row tile (19207 = 150 x 128 + 7 rows): the
    persistent loop's last wave is partial and its last tiles are clipped on
    both axes."""
    run_fprop(19207, 384, 256, 41, sample=4096)
    run_dgrad(19207, 256, 384, 42, sample=4096)
    run_wgrad(256, 19200, 384, 43, sample=4096)


# ------------------------------------------------------------ decode shapes
@pytest.mark.parametrize("proj", list(syn.PROJ_8B))
@pytest.mark.parametrize("M", [64, 256])
def test_decode_shapes(proj, M):
    N, K = syn.PROJ_8B[proj]
    run_fprop(M, N, K, 21, sample=4096, outliers=0.0)


# ------------------------------------------------------------ training-step shapes, full size
@pytest.mark.parametrize("proj", list(syn.PROJ_8B))
def test_train_8b_full_size(proj):
    N, K = syn.PROJ_8B[proj]
    M = 16384
    run_fprop(M, N, K, 31, sample=4096)
    run_dgrad(M, N, K, 32, sample=4096)
    run_wgrad(M, N, K, 33, sample=4096)


def test_deterministic_repeat():
    M, N, K = 1024, 2048, 1024
    x = syn.activation(M, K, seed=1, device=DEV)
    w = syn.weight(N, K, seed=1, device=DEV)
    dy = syn.grad_output(M, N, seed=1, device=DEV)
    qx, sx = jf.quantize_act(x)
    qw, sw, qwt = jf.quantize_weight(w)
    qdy, sdy = jf.quantize_act(dy)
    qxt, sxt = jf.quantize_act_transposed(x)
    qdyt, sdyt = jf.quantize_act_transposed(dy)
    outs = []
    for _ in range(3):
        outs.append((jf.gemm_fprop(qx, sx, qw, sw), jf.gemm_dgrad(qdy, sdy, qwt, sw),
                     jf.gemm_wgrad(qdyt, sdyt, qxt, sxt)))
    for o in outs[1:]:
        assert all(torch.equal(a, b) for a, b in zip(outs[0], o))


def test_zero_scales_give_zero():
    """All-zero activations: scales 0, codes 0, output exactly 0."""
    x = torch.zeros(128, 256, dtype=torch.bfloat16, device=DEV)
    w = syn.weight(256, 256, seed=2, device=DEV)
    qx, sx = jf.quantize_act(x)
    qw, sw, _ = jf.quantize_weight(w)
    y = jf.gemm_fprop(qx, sx, qw, sw)
    assert torch.count_nonzero(y) == 0
