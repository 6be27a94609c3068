"""32B-class long-rollout training shapes at full size (M = 32768 tokens):
X ~ Student-t(3) with 1% of input channels x100, W ~ N(0, 0.02),
dY ~ N(0, 1e-3); both activations quantised by the one-pass dual kernel (the
training path), then Fprop, Dgrad and Wgrad on the GPU.

The oracle checks samples, quantising only the slices they touch.  Every
1x128 token group, every 128x128 weight block and every 128-token column
group is quantised independently of the others, so the codes of a slice are
the codes of the whole tensor:
  * X and dY rows: 128 leading rows, 128 trailing rows, 64 seeded rows;
  * X and dY column blocks (for the transposed operands): first, last and a
    seeded 128-wide block;
  * W: the whole tensor.
Codes and scales are compared bit-exactly on the slices; GEMM outputs on
sampled elements with |gpu - ref| <= 1e-3 * sum|a*b| + 1 bf16 ulp(ref).
"""
import numpy as np
import pytest
import torch

import oracle
import e4m3_group_quantise_gb300 as jf
from e4m3_group_quantise_gb300 import synthetic as syn
from gpu_util import ORACLE_THREADS, assert_bitexact, assert_gemm_close, bits, require_gpu

pytestmark = pytest.mark.gpu
DEV = "cuda"
M = 32768


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def sample_rows(R: int, rng) -> np.ndarray:
    rows = np.concatenate([np.arange(128), np.arange(R - 128, R), rng.integers(128, R - 128, 64)])
    return np.unique(rows)


def sample_col_blocks(C: int, rng) -> np.ndarray:
    blocks = np.unique([0, C // 128 - 1, int(rng.integers(1, C // 128 - 1))])
    return np.concatenate([np.arange(b * 128, (b + 1) * 128) for b in blocks])


def pairs(n_rows: int, n_cols: int, n: int, rng):
    """Local (row, col) sample pairs: the full first 32x32 corner plus n seeded pairs."""
    rr, cc = np.meshgrid(np.arange(min(32, n_rows)), np.arange(min(32, n_cols)), indexing="ij")
    r = np.concatenate([rr.ravel(), rng.integers(0, n_rows, n)])
    c = np.concatenate([cc.ravel(), rng.integers(0, n_cols, n)])
    return r.astype(np.int64), c.astype(np.int64)


@pytest.mark.parametrize("proj", list(syn.PROJ_32B))
def test_train_32b_full_size(proj):
    N, K = syn.PROJ_32B[proj]
    seed = 40 + list(syn.PROJ_32B).index(proj)
    rng = np.random.default_rng(seed)
    x = syn.activation(M, K, seed=seed, outlier_scale=100.0, student_t=True, device=DEV)
    w = syn.weight(N, K, seed=seed, device=DEV)
    dy = syn.grad_output(M, N, seed=seed, device=DEV, sigma=1e-3)

    qx, sx, qxt, sxt = jf.quantize_act_dual(x)
    qdy, sdy, qdyt, sdyt = jf.quantize_act_dual(dy)
    qw, sw, qwt = jf.quantize_weight(w)
    y = jf.gemm_fprop(qx, sx, qw, sw)
    dx = jf.gemm_dgrad(qdy, sdy, qwt, sw)
    dw = jf.gemm_wgrad(qdyt, sdyt, qxt, sxt)
    torch.cuda.synchronize()
    assert jf.jetfp8_poll_device_error() == 0

    # ---- weight: whole tensor, bit-exact
    ow = oracle.quantize_weight(bits(w), threads=ORACLE_THREADS)
    assert_bitexact(qw, ow[0], "qw")
    assert_bitexact(sw, ow[1], "sw")
    assert_bitexact(qwt, np.ascontiguousarray(ow[0].T), "qwt")

    # ---- row slices of X and dY (1x128 groups along the row)
    R = sample_rows(M, rng)
    Rt = torch.from_numpy(R).to(DEV)
    ox = oracle.quantize_act(bits(x.index_select(0, Rt)), threads=ORACLE_THREADS)
    ody = oracle.quantize_act(bits(dy.index_select(0, Rt)), threads=ORACLE_THREADS)
    assert_bitexact(qx.index_select(0, Rt), ox[0], "qx rows")
    assert_bitexact(sx.index_select(1, Rt), ox[1], "sx rows")
    assert_bitexact(qdy.index_select(0, Rt), ody[0], "qdy rows")
    assert_bitexact(sdy.index_select(1, Rt), ody[1], "sdy rows")

    # fprop: sampled rows x sampled output columns
    r, c = pairs(R.size, N, 4096, rng)
    ref, asum = oracle.gemm_fprop(ox[0], ox[1], ow[0], ow[1], r, c, threads=ORACLE_THREADS)
    assert_gemm_close(y.index_select(0, Rt), ref, asum, f"32b fprop {proj}", r, c)
    # dgrad: sampled rows x sampled input columns
    r, c = pairs(R.size, K, 4096, rng)
    ref, asum = oracle.gemm_dgrad(ody[0], ody[1], ow[0], ow[1], r, c, threads=ORACLE_THREADS)
    assert_gemm_close(dx.index_select(0, Rt), ref, asum, f"32b dgrad {proj}", r, c)

    # ---- column blocks of X and dY (128-token groups down each column)
    Cx = sample_col_blocks(K, rng)
    Cdy = sample_col_blocks(N, rng)
    Cxt, Cdyt = torch.from_numpy(Cx).to(DEV), torch.from_numpy(Cdy).to(DEV)
    oxt = oracle.quantize_act_transposed(bits(x.index_select(1, Cxt)), threads=ORACLE_THREADS)
    odyt = oracle.quantize_act_transposed(bits(dy.index_select(1, Cdyt)), threads=ORACLE_THREADS)
    assert_bitexact(qxt.index_select(0, Cxt), oxt[0], "qxt columns")
    assert_bitexact(sxt.index_select(1, Cxt), oxt[1], "sxt columns")
    assert_bitexact(qdyt.index_select(0, Cdyt), odyt[0], "qdyt columns")
    assert_bitexact(sdyt.index_select(1, Cdyt), odyt[1], "sdyt columns")

    # wgrad: sampled output rows (dY columns) x sampled output columns (X columns)
    r, c = pairs(Cdy.size, Cx.size, 2048, rng)
    ref, asum = oracle.gemm_wgrad(odyt[0], odyt[1], oxt[0], oxt[1], r, c, threads=ORACLE_THREADS)
    got = dw.index_select(0, Cdyt).index_select(1, Cxt)
    assert_gemm_close(got, ref, asum, f"32b wgrad {proj}", r, c)
