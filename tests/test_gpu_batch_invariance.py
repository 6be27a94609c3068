"""Batch invariance of the per-token path: a token's Fprop output row, and its
Dgrad row, are bit-identical whether the token is computed alone (decode,
M = 1), in a small decode batch, or inside a large prefill / training batch.
This is the strongest form of "the inference graph is a subgraph of the
training forward graph" (Jet-RL, "Architecture Centrale"): a KV-cached
rollout step and the full-sequence training forward see the same numbers in
every linear layer.

Why it holds: quantisation is per token (1x128 groups), and the GEMM reduces
every output element the same way for any M -- the four K = 32 steps of one
128-wide group summed by the tensor core in fp32, then the groups in order in
fp32 registers.  There is no split-K, and the tile width the launcher picks
(128 columns for small problems, 256 for large ones) does not enter an
element's reduction; the shapes below cross that switch.
"""
import pytest
import torch

import e4m3_group_quantise_gb300 as jf
from e4m3_group_quantise_gb300 import synthetic as syn
from gpu_util import require_gpu

pytestmark = pytest.mark.gpu
DEV = "cuda"
M_FULL = 4096
R0 = 37                                   # sub-batches start off any tile boundary
SUB_M = [1, 2, 63, 64, 65, 128, 200, 1000]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


@pytest.mark.parametrize("proj", ["qkv", "down", "gate_up"])
def test_fprop_rows_independent_of_batch(proj):
    N, K = syn.PROJ_8B[proj]
    x = syn.activation(M_FULL, K, seed=7, outlier_scale=20.0, device=DEV)
    qw, sw, _ = jf.quantize_weight(syn.weight(N, K, seed=7, device=DEV), transposed=False)
    qx, sx = jf.quantize_act(x)
    y_full = jf.gemm_fprop(qx, sx, qw, sw)
    for m in SUB_M:
        xs = x[R0:R0 + m].contiguous()
        qxs, sxs = jf.quantize_act(xs)
        assert torch.equal(qxs, qx[R0:R0 + m]), (proj, m, "codes")
        assert torch.equal(sxs, sx[:, R0:R0 + m]), (proj, m, "scales")
        ys = jf.gemm_fprop(qxs, sxs, qw, sw)
        assert torch.equal(ys, y_full[R0:R0 + m]), (proj, m)
    assert jf.jetfp8_poll_device_error() == 0


def test_fprop_prefill_vs_decode_16384():
    """The training-size batch (16384 tokens) against single-token decode on
    the gate_up projection."""
    N, K = syn.PROJ_8B["gate_up"]
    x = syn.activation(16384, K, seed=8, outlier_scale=20.0, device=DEV)
    qw, sw, _ = jf.quantize_weight(syn.weight(N, K, seed=8, device=DEV), transposed=False)
    qx, sx = jf.quantize_act(x)
    y_full = jf.gemm_fprop(qx, sx, qw, sw)
    for r in (0, 5, 8191, 16383):
        qxs, sxs = jf.quantize_act(x[r:r + 1].contiguous())
        assert torch.equal(jf.gemm_fprop(qxs, sxs, qw, sw), y_full[r:r + 1]), r


@pytest.mark.parametrize("proj", ["o", "down"])
def test_dgrad_rows_independent_of_batch(proj):
    N, K = syn.PROJ_8B[proj]
    dy = syn.grad_output(M_FULL, N, seed=9, device=DEV)
    _, sw, qwt = jf.quantize_weight(syn.weight(N, K, seed=9, device=DEV))
    qdy, sdy = jf.quantize_act(dy)
    dx_full = jf.gemm_dgrad(qdy, sdy, qwt, sw)
    for m in SUB_M:
        qs, ss = jf.quantize_act(dy[R0:R0 + m].contiguous())
        assert torch.equal(jf.gemm_dgrad(qs, ss, qwt, sw), dx_full[R0:R0 + m]), (proj, m)
    assert jf.jetfp8_poll_device_error() == 0
