"""GPU quantisers vs the CPU oracle: codes and scales bit-exact.

Covers tiny and ragged shapes (tails of every tile), special values (zero
groups, bf16 subnormals, signed zeros, saturation, outlier channels), the
8B-class layer shapes at full size, values placed on and next to E4M3
rounding midpoints, and the conversion of every finite bf16 value |x| <= 448
(groups whose scale is exactly 1).
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


def special_values(M, K, seed):
    """N(0,1) rows mixed with zero groups, subnormal groups, signed zeros,
    large values and exact ties."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(M, K, generator=g)
    x[0, :128] = 0.0                                    # zero group
    if M > 1:
        x[1, :128] = -0.0                               # negative-zero group
        x[1, 5] = 3.0
        x[1, 6] = -0.0
    if M > 2:
        x[2, :128] = torch.randn(128, generator=g) * 1e-39   # bf16 subnormals -> subnormal scale
    if M > 3:
        x[3, :128] = torch.randn(128, generator=g) * 3e38    # near the top of the range
    if M > 4:
        x[4, :128] = 448.0 * 2.0 ** -3                   # all equal to the amax
    if M > 5 and K >= 256:
        x[5, 128:256] = torch.tensor([2.125, 2.375, 1.9375, 56.0] * 32)  # ties after scaling
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("M,K", [(256, 512), (1, 128), (3, 384), (31, 1152), (33, 1024),
                                 (64, 4096), (129, 256), (300, 2048), (1000, 128)])
def test_quantize_act_bitexact(M, K):
    x = syn.activation(M, K, seed=M * 7 + K, outlier_scale=20.0)
    q, s = jf.quantize_act(x.to(DEV))
    oq, os_ = oracle.quantize_act(bits(x))
    assert_bitexact(q, oq, "codes")
    assert_bitexact(s, os_, "scales")


def test_quantize_act_special_values():
    x = special_values(64, 512, 1)
    q, s = jf.quantize_act(x.to(DEV))
    oq, os_ = oracle.quantize_act(bits(x))
    assert_bitexact(q, oq, "codes")
    assert_bitexact(s, os_, "scales")
    assert os_[0, 2] > 0 and os_[0, 2] < np.finfo(np.float32).tiny   # a subnormal scale was exercised


@pytest.mark.parametrize("M,C", [(128, 128), (256, 512), (384, 640), (128, 4096), (1024, 384)])
def test_quantize_act_transposed_bitexact(M, C):
    x = syn.activation(M, C, seed=M + C, outlier_scale=20.0)
    qt, st = jf.quantize_act_transposed(x.to(DEV))
    oq, os_ = oracle.quantize_act_transposed(bits(x))
    assert_bitexact(qt, oq, "codes")
    assert_bitexact(st, os_, "scales")


def test_quantize_act_transposed_special_values():
    x = special_values(256, 256, 2).T.contiguous()     # groups along rows now hold the specials
    qt, st = jf.quantize_act_transposed(x.to(DEV))
    oq, os_ = oracle.quantize_act_transposed(bits(x))
    assert_bitexact(qt, oq, "codes")
    assert_bitexact(st, os_, "scales")


@pytest.mark.parametrize("N,K", [(128, 128), (512, 512), (384, 1152), (6144, 4096)])
@pytest.mark.parametrize("transposed", [True, False])
def test_quantize_weight_bitexact(N, K, transposed):
    w = syn.weight(N, K, seed=N + K)
    q, s, qt = jf.quantize_weight(w.to(DEV), transposed=transposed)
    oq, os_, oqt = oracle.quantize_weight(bits(w), transposed, threads=ORACLE_THREADS)
    assert_bitexact(q, oq, "codes")
    assert_bitexact(s, os_, "scales")
    if transposed:
        assert_bitexact(qt, oqt, "transposed codes")


def test_quantize_weight_special_values():
    w = special_values(256, 384, 3)
    q, s, qt = jf.quantize_weight(w.to(DEV))
    oq, os_, oqt = oracle.quantize_weight(bits(w), True)
    assert_bitexact(q, oq, "codes")
    assert_bitexact(s, os_, "scales")
    assert_bitexact(qt, oqt, "transposed codes")


def test_quantize_weight_group_matches_single_calls():
    """One grouped launch over the 8B-class projections (mixed with and
    without transposed codes) gives, bit for bit, what one call per weight
    gives; small entries are also checked against the oracle."""
    shapes = [(6144, 4096), (4096, 4096), (28672, 4096), (4096, 14336), (128, 128), (384, 1152)]
    ws = [syn.weight(n, k, seed=11 + i, index=i, device=DEV) for i, (n, k) in enumerate(shapes)]
    ws[4] = special_values(128, 128, 5).to(DEV)
    transposed = [True, True, True, True, False, True]
    qs = [torch.empty(w.shape, dtype=torch.uint8, device=DEV) for w in ws]
    ss = [torch.empty((w.shape[0] // 128, w.shape[1] // 128), dtype=torch.float32, device=DEV) for w in ws]
    qts = [torch.empty((w.shape[1], w.shape[0]), dtype=torch.uint8, device=DEV) if t else None
           for w, t in zip(ws, transposed)]
    jf.jetfp8_quantize_weight_group(ws, qs, ss, qts)
    assert jf.jetfp8_poll_device_error() == 0
    for i, (w, t) in enumerate(zip(ws, transposed)):
        q1, s1, qt1 = jf.quantize_weight(w, transposed=t)
        assert torch.equal(qs[i], q1) and torch.equal(ss[i], s1), f"entry {i}"
        if t:
            assert torch.equal(qts[i], qt1), f"entry {i} transposed"
    for i in (4, 5):
        oq, os_, oqt = oracle.quantize_weight(bits(ws[i].cpu()), transposed[i], threads=ORACLE_THREADS)
        assert_bitexact(qs[i], oq, f"entry {i} codes")
        assert_bitexact(ss[i], os_, f"entry {i} scales")
        if transposed[i]:
            assert_bitexact(qts[i], oqt, f"entry {i} transposed codes")


def test_quantize_weights_chunks_past_the_group_limit():
    """quantize_weights splits more than eight weights over several launches."""
    ws = [syn.weight(128 * (1 + i % 3), 256, seed=40 + i, device=DEV) for i in range(11)]
    got = jf.quantize_weights(ws)
    for w, (q, s, qt) in zip(ws, got):
        q1, s1, qt1 = jf.quantize_weight(w)
        assert torch.equal(q, q1) and torch.equal(s, s1) and torch.equal(qt, qt1)


def tie_groups(rows, seed):
    """Groups made to hit E4M3 rounding midpoints: amax = 448 * 2^e (an exact
    power-of-two scale), the other values exact midpoints between neighbouring
    E4M3 values times 2^e, and their bf16 neighbours -- every value lands on
    or next to a rounding boundary, exercising the exact-division fallback."""
    codes = torch.arange(0, 0x7F, dtype=torch.int32).to(torch.uint8)
    vals = codes.view(torch.float8_e4m3fn).float()
    mids = (vals[:-1] + vals[1:]) / 2
    g = torch.Generator().manual_seed(seed)
    out = torch.empty(rows, 128)
    for r in range(rows):
        e = int(torch.randint(-30, 10, (1,), generator=g))
        pick = mids[torch.randint(0, mids.numel(), (127,), generator=g)]
        sign = torch.where(torch.rand(127, generator=g) < 0.5, -1.0, 1.0)
        row = torch.cat([torch.tensor([448.0]), pick * sign]) * 2.0 ** e
        out[r] = row
    x = out.to(torch.bfloat16)
    # nudge a third of the entries to a bf16 neighbour of the midpoint
    bits = x.view(torch.int16)
    nudge = (torch.randint(0, 3, bits.shape, generator=g) - 1).to(torch.int16)
    nudge[:, 0] = 0
    return (bits + nudge).view(torch.bfloat16)


def test_rounding_midpoints_all_quantisers():
    x = tie_groups(256, 9)                                     # [256, 128]
    q, s = jf.quantize_act(x.to(DEV))
    oq, os_ = oracle.quantize_act(bits(x))
    assert_bitexact(q, oq, "act codes")
    assert_bitexact(s, os_, "act scales")
    xt = x.T.contiguous()                                      # [128, 256]: groups along rows
    qt, st = jf.quantize_act_transposed(xt.to(DEV))
    oqt, ost = oracle.quantize_act_transposed(bits(xt))
    assert_bitexact(qt, oqt, "transposed codes")
    w = x[:128].reshape(128, 128).contiguous()
    w[0, 0] = 448.0 * 2.0 ** 5                                  # one pow2 scale for the block
    qw, sw, qwt = jf.quantize_weight(w.to(DEV))
    oqw, osw, oqwt = oracle.quantize_weight(bits(w), True)
    assert_bitexact(qw, oqw, "weight codes")
    assert_bitexact(qwt, oqwt, "weight transposed codes")


def test_all_bf16_values_scale_one():
    """Every finite bf16 value with |x| <= 448 in groups whose amax is 448, so
    s = 1 and the code is the E4M3 rounding of x itself."""
    allb = torch.arange(-32768, 32768, dtype=torch.int32).to(torch.int16).view(torch.bfloat16).float()
    v = allb[torch.isfinite(allb) & (allb.abs() <= 448.0)]
    n = (v.numel() + 126) // 127 * 127
    pad = torch.zeros(n)
    pad[:v.numel()] = v
    x = torch.cat([torch.full((n // 127, 1), 448.0), pad.view(-1, 127)], dim=1).to(torch.bfloat16)
    q, s = jf.quantize_act(x.to(DEV))
    oq, os_ = oracle.quantize_act(bits(x))
    assert np.all(os_ == 1.0)
    assert_bitexact(q, oq, "codes")


@pytest.mark.parametrize("M,K", [(128, 128), (256, 512), (384, 1152), (1024, 384), (128, 4096)])
def test_dual_output_bitexact(M, K):
    """One pass, both layouts: identical to the oracle's 1x128 and 128x1
    quantisations and to the two single-output kernels."""
    x = syn.activation(M, K, seed=M * 3 + K, outlier_scale=20.0)
    xd = x.to(DEV)
    q, s, qt, st = jf.quantize_act_dual(xd)
    oq, os_ = oracle.quantize_act(bits(x))
    oqt, ost = oracle.quantize_act_transposed(bits(x))
    assert_bitexact(q, oq, "codes")
    assert_bitexact(s, os_, "scales")
    assert_bitexact(qt, oqt, "transposed codes")
    assert_bitexact(st, ost, "transposed scales")
    q1, s1 = jf.quantize_act(xd)
    q2, s2 = jf.quantize_act_transposed(xd)
    assert torch.equal(q, q1) and torch.equal(s, s1) and torch.equal(qt, q2) and torch.equal(st, s2)


def test_dual_output_special_values():
    x = torch.cat([special_values(128, 256, 4), tie_groups(128, 5).repeat(1, 2)], dim=0).contiguous()
    q, s, qt, st = jf.quantize_act_dual(x.to(DEV))
    oq, os_ = oracle.quantize_act(bits(x))
    oqt, ost = oracle.quantize_act_transposed(bits(x))
    assert_bitexact(q, oq, "codes")
    assert_bitexact(s, os_, "scales")
    assert_bitexact(qt, oqt, "transposed codes")
    assert_bitexact(st, ost, "transposed scales")


def test_dual_output_full_size_gradient():
    """dY of the 8B gate_up projection [16384, 28672] through the dual kernel,
    checked against the single-output kernels (themselves checked against the
    oracle at this size above) and against the oracle on slices."""
    M, N = 16384, 28672
    dy = syn.grad_output(M, N, seed=6, device=DEV)
    q, s, qt, st = jf.quantize_act_dual(dy)
    q1, s1 = jf.quantize_act(dy)
    assert torch.equal(q, q1) and torch.equal(s, s1)
    del q1, s1
    q2, s2 = jf.quantize_act_transposed(dy)
    assert torch.equal(qt, q2) and torch.equal(st, s2)
    del q2, s2
    rows = slice(4096, 4096 + 256)
    oq, os_ = oracle.quantize_act(bits(dy[rows]), threads=ORACLE_THREADS)
    assert_bitexact(q[rows], oq, "codes (row block)")
    sl = slice(N - 256, N)
    oqt, ost = oracle.quantize_act_transposed(bits(dy[:, sl]), threads=ORACLE_THREADS)
    assert_bitexact(qt[sl], oqt, "transposed codes (column block)")
    assert_bitexact(st[:, sl].contiguous(), ost, "transposed scales (column block)")


def test_empty_inputs():
    x = torch.empty(0, 256, dtype=torch.bfloat16, device=DEV)
    q, s = jf.quantize_act(x)
    assert q.shape == (0, 256) and s.shape == (2, 0)
    qt, st = jf.quantize_act_transposed(x)
    assert qt.shape == (256, 0)


@pytest.mark.parametrize("name,shape", [("x_8b_hidden", (16384, 4096)), ("x_8b_inter", (16384, 14336))])
def test_full_size_act_quantisers(name, shape):
    """The 8B-class training-step activations at full size, every code compared."""
    M, K = shape
    x = syn.activation(M, K, seed=11, outlier_scale=20.0, device=DEV)
    xb = bits(x)
    q, s = jf.quantize_act(x)
    oq, os_ = oracle.quantize_act(xb, threads=ORACLE_THREADS)
    assert_bitexact(q, oq, "codes")
    assert_bitexact(s, os_, "scales")
    del q, s, oq, os_
    qt, st = jf.quantize_act_transposed(x)
    oqt, ost = oracle.quantize_act_transposed(xb, threads=ORACLE_THREADS)
    assert_bitexact(qt, oqt, "transposed codes")
    assert_bitexact(st, ost, "transposed scales")


def test_full_size_gradient_slices():
    """dY of the 8B gate_up projection [16384, 28672]: full-tensor quantisers on
    the GPU, checked on column slices (the transposed quantiser's groups are
    per column, so a slice is an exact sub-problem) and full row-blocks."""
    M, N = 16384, 28672
    dy = syn.grad_output(M, N, seed=5, device=DEV)
    q, s = jf.quantize_act(dy)
    qt, st = jf.quantize_act_transposed(dy)
    rows = slice(8192, 8192 + 512)
    sub = bits(dy[rows])
    oq, os_ = oracle.quantize_act(sub, threads=ORACLE_THREADS)
    assert_bitexact(q[rows], oq, "codes (row block)")
    assert_bitexact(s[:, rows].contiguous(), os_, "scales (row block)")
    for c0 in (0, 12800, N - 128):
        sl = slice(c0, c0 + 128)
        oqt, ost = oracle.quantize_act_transposed(bits(dy[:, sl]), threads=ORACLE_THREADS)
        assert_bitexact(qt[sl], oqt, f"transposed codes cols {c0}")
        assert_bitexact(st[:, sl].contiguous(), ost, f"transposed scales cols {c0}")


def test_repeatable():
    x = syn.activation(512, 2048, seed=3, device=DEV)
    a = jf.quantize_act(x)
    b = jf.quantize_act(x)
    assert all(torch.equal(u, v) for u, v in zip(a, b))


def test_scale_for_every_bf16_amax():
    """The group scale s = amax / 448 for every non-negative finite bf16
    amax (the only values amax takes): row i holds the i-th pattern once and
    zeros elsewhere; every kernel's scale must equal the oracle's IEEE
    division, and the codes must match too."""
    pats = np.arange(0, 0x7F80, dtype=np.uint16)
    n = pats.size
    rows = -(-n // 128) * 128
    xb = np.zeros((rows, 128), dtype=np.uint16)
    xb[:n, 7] = pats
    xb[:n, 100] = pats >> 1                   # a second, smaller value in the group
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16)
    ox = oracle.quantize_act(xb, threads=ORACLE_THREADS)
    q, s = jf.quantize_act(x.to(DEV))
    assert_bitexact(q, ox[0], "codes")
    assert_bitexact(s, ox[1], "scales")
    # the same values down the columns, for the transposed and dual kernels
    xt = x.t().contiguous()                   # [128, rows]: each column one group of 128 tokens
    oxt = oracle.quantize_act_transposed(bits(xt), threads=ORACLE_THREADS)
    qt, st = jf.quantize_act_transposed(xt.to(DEV))
    assert_bitexact(qt, oxt[0], "transposed codes")
    assert_bitexact(st, oxt[1], "transposed scales")
    qd, sd, qdt, sdt = jf.quantize_act_dual(xt.to(DEV))
    assert_bitexact(qdt, oxt[0], "dual transposed codes")
    assert_bitexact(sdt, oxt[1], "dual transposed scales")
