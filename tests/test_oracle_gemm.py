"""Pins for the oracle's fp64 GEMMs (CPU only).

Independent checks:
  * brute force: dense dequantised matrices built here from a library
    decode (torch float8_e4m3fn) and multiplied with numpy's matmul;
  * closed forms: scale-1 small-integer codes give exact integers; a
    448*identity weight gives Y = 448 * deq(X) exactly;
  * K additivity: a 2-group GEMM equals the sum of its two 1-group GEMMs;
  * transpose identity: dgrad(dY, W) = fprop(dY, W^T) bit-for-bit;
  * sampled elements equal the same elements of the full GEMM.
"""
import numpy as np
import pytest
import torch

from e4m3_brute import TABLE


def bf16_from_normal(shape, sigma, seed):
    g = torch.Generator().manual_seed(seed)
    t = (torch.randn(*shape, generator=g) * sigma).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def lib_deq(q):
    """Library decode (torch) of a code tensor, as float64."""
    return torch.from_numpy(np.ascontiguousarray(q)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def dense_act(q, s):
    """q [R,C], s [C/128,R] -> deq [R,C] (1x128 groups along C)."""
    return lib_deq(q) * np.repeat(s.T.astype(np.float64), 128, axis=1)


def dense_weight(q, s):
    return lib_deq(q) * np.kron(s.astype(np.float64), np.ones((128, 128)))


@pytest.fixture(scope="module")
def tiny(oracle_mod):
    M, N, K = 256, 512, 512
    x = bf16_from_normal((M, K), 1.0, 100)
    w = bf16_from_normal((N, K), 0.02, 101)
    dy = bf16_from_normal((M, N), 1e-2, 102)
    qx, sx = oracle_mod.quantize_act(x)
    qw, sw, qwt = oracle_mod.quantize_weight(w, True)
    qdy, sdy = oracle_mod.quantize_act(dy)
    qxt, sxt = oracle_mod.quantize_act_transposed(x)
    qdyt, sdyt = oracle_mod.quantize_act_transposed(dy)
    return dict(M=M, N=N, K=K, qx=qx, sx=sx, qw=qw, sw=sw, qwt=qwt, qdy=qdy, sdy=sdy,
                qxt=qxt, sxt=sxt, qdyt=qdyt, sdyt=sdyt)


def test_fprop_vs_dense_matmul(oracle_mod, tiny):
    t = tiny
    y, asum = oracle_mod.gemm_fprop(t["qx"], t["sx"], t["qw"], t["sw"])
    ref = dense_act(t["qx"], t["sx"]) @ dense_weight(t["qw"], t["sw"]).T
    aref = np.abs(dense_act(t["qx"], t["sx"])) @ np.abs(dense_weight(t["qw"], t["sw"])).T
    assert np.allclose(y, ref, rtol=0, atol=1e-12 * aref.max())
    assert np.allclose(asum, aref, rtol=1e-12)


def test_dgrad_vs_dense_matmul(oracle_mod, tiny):
    t = tiny
    dx, asum = oracle_mod.gemm_dgrad(t["qdy"], t["sdy"], t["qw"], t["sw"])
    ref = dense_act(t["qdy"], t["sdy"]) @ dense_weight(t["qw"], t["sw"])
    aref = np.abs(dense_act(t["qdy"], t["sdy"])) @ np.abs(dense_weight(t["qw"], t["sw"]))
    assert dx.shape == (t["M"], t["K"])
    assert np.allclose(dx, ref, rtol=0, atol=1e-12 * aref.max())
    assert np.allclose(asum, aref, rtol=1e-12)


def test_wgrad_vs_dense_matmul(oracle_mod, tiny):
    t = tiny
    dw, asum = oracle_mod.gemm_wgrad(t["qdyt"], t["sdyt"], t["qxt"], t["sxt"])
    a = dense_act(t["qdyt"], t["sdyt"])        # [N, M], 128-token groups
    b = dense_act(t["qxt"], t["sxt"])          # [K, M]
    ref = a @ b.T
    aref = np.abs(a) @ np.abs(b).T
    assert dw.shape == (t["N"], t["K"])
    assert np.allclose(dw, ref, rtol=0, atol=1e-12 * aref.max())
    assert np.allclose(asum, aref, rtol=1e-12)


def test_dgrad_equals_fprop_on_transposed_weight(oracle_mod, tiny):
    t = tiny
    dx, a1 = oracle_mod.gemm_dgrad(t["qdy"], t["sdy"], t["qw"], t["sw"])
    y, a2 = oracle_mod.gemm_fprop(t["qdy"], t["sdy"], np.ascontiguousarray(t["qw"].T),
                                  np.ascontiguousarray(t["sw"].T))
    assert np.array_equal(dx, y) and np.array_equal(a1, a2)


def test_integer_closed_form(oracle_mod):
    """Scale 1 and small-integer codes: every product and sum is an exact
    integer, so the oracle must return exactly the integer matmul."""
    rng = np.random.default_rng(0)
    M, N, K = 64, 256, 256
    ints = rng.integers(-8, 9, size=(M, K))
    wint = rng.integers(-8, 9, size=(N, K))
    enc = {v: c for c, v in enumerate(TABLE) if np.isfinite(v) and c < 0x80}
    def codes(a):
        out = np.empty(a.shape, np.uint8)
        for v in np.unique(a):
            out[a == v] = enc[abs(float(v))] | (0x80 if v < 0 else 0)
        return out
    qx, qw = codes(ints), codes(wint)
    sx = np.ones((K // 128, M), np.float32)
    sw = np.ones((N // 128, K // 128), np.float32)
    y, _ = oracle_mod.gemm_fprop(qx, sx, qw, sw)
    assert np.array_equal(y, (ints @ wint.T).astype(np.float64))


def test_identity_weight(oracle_mod):
    """W = 448 * I: the diagonal blocks get s = 1 and code 0x7e, the other
    blocks are all zero, so Y = 448 * deq(X) exactly."""
    M, K = 32, 256
    x = bf16_from_normal((M, K), 1.0, 3)
    w = np.zeros((K, K), np.float32)
    np.fill_diagonal(w, 448.0)
    wb = torch.from_numpy(w).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    qx, sx = oracle_mod.quantize_act(x)
    qw, sw, _ = oracle_mod.quantize_weight(wb)
    assert np.all(np.diag(sw) == 1.0) and np.count_nonzero(sw) == 2
    y, _ = oracle_mod.gemm_fprop(qx, sx, qw, sw)
    assert np.array_equal(y, 448.0 * dense_act(qx, sx))


def test_k_additivity(oracle_mod):
    """Groups are independent along K: the GEMM over K = 2 groups equals the
    sum of the GEMMs over each group (quantised separately)."""
    M, N, K = 40, 128, 256
    x = bf16_from_normal((M, K), 1.0, 21)
    w = bf16_from_normal((N, K), 0.02, 22)
    qx, sx = oracle_mod.quantize_act(x)
    qw, sw, _ = oracle_mod.quantize_weight(w)
    y, asum = oracle_mod.gemm_fprop(qx, sx, qw, sw)
    parts = []
    for g in range(2):
        xg = np.ascontiguousarray(x[:, g * 128:(g + 1) * 128])
        wg = np.ascontiguousarray(w[:, g * 128:(g + 1) * 128])
        qxg, sxg = oracle_mod.quantize_act(xg)
        qwg, swg, _ = oracle_mod.quantize_weight(wg)
        assert np.array_equal(qxg, qx[:, g * 128:(g + 1) * 128])
        assert np.array_equal(sxg[0], sx[g]) and np.array_equal(swg[:, 0], sw[:, g])
        parts.append(oracle_mod.gemm_fprop(qxg, sxg, qwg, swg)[0])
    # equal up to fp64 summation order (relative to the sum of |terms|)
    assert np.all(np.abs(y - (parts[0] + parts[1])) <= 1e-13 * asum)


def test_sampled_elements_match_full(oracle_mod, tiny):
    t = tiny
    rng = np.random.default_rng(4)
    rows = rng.integers(0, t["M"], 200)
    cols = rng.integers(0, t["N"], 200)
    full, fa = oracle_mod.gemm_fprop(t["qx"], t["sx"], t["qw"], t["sw"])
    v, a = oracle_mod.gemm_fprop(t["qx"], t["sx"], t["qw"], t["sw"], rows, cols, threads=3)
    assert np.array_equal(v, full[rows, cols]) and np.array_equal(a, fa[rows, cols])
    full, fa = oracle_mod.gemm_wgrad(t["qdyt"], t["sdyt"], t["qxt"], t["sxt"])
    r2 = rng.integers(0, t["N"], 100)
    c2 = rng.integers(0, t["K"], 100)
    v, a = oracle_mod.gemm_wgrad(t["qdyt"], t["sdyt"], t["qxt"], t["sxt"], r2, c2, threads=2)
    assert np.array_equal(v, full[r2, c2])


def test_planted_index_mistake_is_caught(oracle_mod, tiny):
    """A plausible mistake -- using the weight block scale of the wrong
    block -- changes the result far beyond the GEMM tolerance, so the
    dense-matmul pin above would catch it."""
    t = tiny
    sw_bad = np.ascontiguousarray(t["sw"].T)   # transposed block scales
    y_bad, _ = oracle_mod.gemm_fprop(t["qx"], t["sx"], t["qw"], sw_bad)
    ref = dense_act(t["qx"], t["sx"]) @ dense_weight(t["qw"], t["sw"]).T
    aref = np.abs(dense_act(t["qx"], t["sx"])) @ np.abs(dense_weight(t["qw"], t["sw"])).T
    assert np.any(np.abs(y_bad - ref) > 1e-3 * aref)
