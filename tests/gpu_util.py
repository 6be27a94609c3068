"""Helpers for the GPU parity tests (test infrastructure)."""
import numpy as np
import pytest
import torch

import oracle
from e4m3_group_quantise_gb300 import synthetic as syn

ORACLE_THREADS = 16


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def assert_bitexact(got: torch.Tensor, want: np.ndarray, what: str):
    g = to_np(got)
    assert g.shape == want.shape, (what, g.shape, want.shape)
    if g.dtype == np.float32:
        g, want = g.view(np.uint32), want.view(np.uint32)
    bad = np.argwhere(g != want)
    assert bad.size == 0, f"{what}: {len(bad)} mismatches, first at {bad[:5].tolist()}: " \
                          f"{[(int(g[tuple(i)]), int(want[tuple(i)])) for i in bad[:5]]}"


# (case, worst error/bound, elements compared) of every GEMM parity check in
# this session; printed at the end of the run (see conftest.py) so that a
# shrinking margin shows up before it turns into a failure
GEMM_MARGINS = []
# Margin guard, tighter than the bar: rounding the exact result to bf16 alone
# uses up to half of the bound (0.5 ulp of the bf16 ulp term), and the
# kernel's fp32 accumulation adds of the order of 1e-3 more (measured worst
# 0.39 over every case), so a case above 0.6 has lost accumulation accuracy
# even if it is still within the bar.
MARGIN_GUARD = 0.6


def assert_gemm_close(got: torch.Tensor, ref: np.ndarray, asum: np.ndarray, what: str, rows=None, cols=None):
    g = got.float().cpu().numpy()
    if rows is not None:
        g = g[rows, cols]
    ok, worst, idx = oracle.gemm_within_tolerance(g, ref, asum)
    GEMM_MARGINS.append((what, worst, int(np.asarray(ref).size)))
    assert ok, f"{what}: outside tolerance, worst error/bound {worst:.4g} at flat index {idx} " \
               f"(got {g.ravel()[idx]!r}, ref {np.asarray(ref).ravel()[idx]!r})"
    assert worst <= MARGIN_GUARD, f"{what}: within the bar but past the margin guard ({worst:.4g} > {MARGIN_GUARD})"
    return worst


def sample_indices(R: int, C: int, n: int, seed: int):
    """Four corner 128x128 tiles (clipped), row 0, last row, and n seeded random elements."""
    rng = np.random.default_rng(seed)
    rows, cols = [], []
    for r0 in (0, max(0, R - 128)):
        for c0 in (0, max(0, C - 128)):
            rr, cc = np.meshgrid(np.arange(r0, min(R, r0 + 128)), np.arange(c0, min(C, c0 + 128)), indexing="ij")
            rows.append(rr.ravel())
            cols.append(cc.ravel())
    for r in (0, R - 1):
        rows.append(np.full(C, r))
        cols.append(np.arange(C))
    rows.append(rng.integers(0, R, n))
    cols.append(rng.integers(0, C, n))
    rows = np.concatenate(rows).astype(np.int64)
    cols = np.concatenate(cols).astype(np.int64)
    key = np.unique(rows * C + cols)
    return key // C, key % C


def bits(t: torch.Tensor) -> np.ndarray:
    return syn.bf16_bits(t)
