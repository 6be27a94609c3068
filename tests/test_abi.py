"""The C-ABI library on the host (no GPU needed): it loads, exports every
function that include/jetfp8.h declares, and rejects bad arguments before
touching the device (status codes only; no compute call is made)."""
import ctypes
import subprocess

import pytest

import e4m3_group_quantise_gb300 as jf
from e4m3_group_quantise_gb300 import jetfp8 as J


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    return jf.load_library()


def test_exports_every_declared_symbol(lib):
    names = jf.declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    # and the dynamic symbol table exports exactly the C-ABI (hidden visibility elsewhere)
    out = subprocess.run(["nm", "-D", "--defined-only", J.LIB_PATH], capture_output=True, text=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    assert set(names) <= exported
    assert {e for e in exported if e.startswith("jetfp8_")} == set(names)


def test_status_strings(lib):
    for code, name in J.STATUS.items():
        assert jf.jetfp8_status_string(code).startswith(name)
    assert "unknown" in jf.jetfp8_status_string(99)


def test_act_scale_count(lib):
    assert jf.jetfp8_act_scale_count(16384, 4096) == 32 * 16384
    assert jf.jetfp8_act_scale_count(0, 128) == 0
    assert jf.jetfp8_act_scale_count(5, 100) == 0
    assert jf.jetfp8_act_scale_count(-1, 128) == 0


A16 = 0x10000          # fake, 16-byte aligned "device" addresses: never dereferenced,
B16 = 0x20000000       # every call below is rejected by the host checks first
C16 = 0x40000000
D16 = 0x60000000
E16 = 0x80000000


def test_e4m3_encode_range_validation(lib):
    f = lib.jetfp8_e4m3_encode_range
    assert f(0, -1, B16, None) == J.ERR_SHAPE
    assert f(0, (1 << 32) + 1, B16, None) == J.ERR_SHAPE         # past the last pattern
    assert f(0xFFFFFFFF, 2, B16, None) == J.ERR_SHAPE
    assert f(7, 0, None, None) == J.OK                            # empty: nothing to do
    assert f(0, 16, None, None) == J.ERR_INVALID_VALUE
    assert f(0, 16, B16 + 8, None) == J.ERR_ALIGNMENT


def test_quantize_act_validation(lib):
    f = lib.jetfp8_quantize_act
    assert f(A16, 4, 100, B16, C16, None) == J.ERR_SHAPE          # K % 128
    assert f(A16, -1, 128, B16, C16, None) == J.ERR_SHAPE
    assert f(A16, 4, 0, B16, C16, None) == J.ERR_SHAPE
    assert f(None, 0, 128, None, None, None) == J.OK              # empty: nothing to do
    assert f(None, 4, 128, B16, C16, None) == J.ERR_INVALID_VALUE
    assert f(A16 + 4, 4, 128, B16, C16, None) == J.ERR_ALIGNMENT
    assert f(A16, 4, 128, A16 + 64, C16, None) == J.ERR_INVALID_VALUE  # q overlaps x
    assert f(A16, 4, 128, B16, B16 + 256, None) == J.ERR_INVALID_VALUE  # s overlaps q
    assert f(A16, 1 << 31, 128, B16, C16, None) == J.ERR_SHAPE     # row count limit
    # the launch grid has ceil(K / 1024) blocks along y (at most 65535): the
    # first K past that limit is a shape error, not a failed launch
    assert f(A16, 1, 65535 * 1024 + 128, B16, C16, None) == J.ERR_SHAPE


def test_quantize_transposed_validation(lib):
    f = lib.jetfp8_quantize_act_transposed
    assert f(A16, 100, 128, B16, C16, None) == J.ERR_SHAPE        # M % 128
    assert f(A16, 128, 64, B16, C16, None) == J.ERR_SHAPE         # C % 128
    assert f(None, 0, 128, None, None, None) == J.OK
    assert f(A16, 128, 128, None, C16, None) == J.ERR_INVALID_VALUE
    assert f(A16, 128, 128, B16 + 8, C16, None) == J.ERR_ALIGNMENT
    assert f(A16, 128, 128, A16 + 16, C16, None) == J.ERR_INVALID_VALUE


def test_quantize_dual_validation(lib):
    f = lib.jetfp8_quantize_act_dual
    assert f(A16, 100, 128, B16, C16, D16, E16, None) == J.ERR_SHAPE      # M % 128
    assert f(A16, 128, 100, B16, C16, D16, E16, None) == J.ERR_SHAPE      # K % 128
    assert f(None, 0, 128, None, None, None, None, None) == J.OK
    assert f(A16, 128, 128, B16, C16, None, E16, None) == J.ERR_INVALID_VALUE
    assert f(A16, 128, 128, B16, C16, D16 + 4, E16, None) == J.ERR_ALIGNMENT
    assert f(A16, 128, 128, B16, C16, B16 + 64, E16, None) == J.ERR_INVALID_VALUE   # qt overlaps q


def test_quantize_weight_validation(lib):
    f = lib.jetfp8_quantize_weight
    assert f(A16, 100, 128, B16, C16, None, None) == J.ERR_SHAPE
    assert f(A16, 128, 0, B16, C16, None, None) == J.ERR_SHAPE
    assert f(A16, 128, 128, None, C16, None, None) == J.ERR_INVALID_VALUE
    assert f(A16, 128, 128, B16, C16, D16 + 4, None) == J.ERR_ALIGNMENT
    assert f(A16, 128, 128, B16, C16, B16 + 128, None) == J.ERR_INVALID_VALUE   # qt overlaps q


def _group_args(entries):
    """Host arrays for jetfp8_quantize_weight_group from (w, N, K, q, s, qt) tuples."""
    n = max(len(entries), 1)
    P, I = ctypes.c_void_p * n, ctypes.c_int64 * n
    cols = list(zip(*entries)) if entries else [()] * 6
    return (P(*cols[0]), I(*cols[1]), I(*cols[2]), P(*cols[3]), P(*cols[4]), P(*cols[5]))


def test_quantize_weight_group_validation(lib):
    f = lib.jetfp8_quantize_weight_group
    f.argtypes = [ctypes.c_int] + [ctypes.c_void_p] * 7
    good = (A16, 128, 256, B16, C16, None)                       # W 128x256: 64 KB, q 32 KB, s 8 B
    other = (D16, 256, 128, D16 + (1 << 20), D16 + (2 << 20), D16 + (3 << 20))
    assert f(0, None, None, None, None, None, None, None) == J.OK   # empty group: nothing to do
    assert f(-1, *_group_args([good]), None) == J.ERR_SHAPE
    assert f(J.WEIGHT_GROUP_MAX + 1, *_group_args([good] * 9), None) == J.ERR_SHAPE
    w, n, k, q, s, qt = _group_args([good])
    assert f(1, w, n, k, q, s, None, None) == J.ERR_INVALID_VALUE   # the qt array itself is required
    assert f(2, *_group_args([good, (A16, 100, 128, B16, C16, None)]), None) == J.ERR_SHAPE
    assert f(2, *_group_args([good, (D16, 128, 128, None, C16, None)]), None) == J.ERR_INVALID_VALUE
    assert f(2, *_group_args([good, (D16 + 4, 128, 128, E16, E16 + 65536, None)]), None) == J.ERR_ALIGNMENT
    # an output of one entry overlapping an input or output of another
    assert f(2, *_group_args([good, (D16, 128, 128, A16 + 4096, E16, None)]), None) == J.ERR_INVALID_VALUE
    assert f(2, *_group_args([good, (D16, 128, 128, E16, B16 + 16, None)]), None) == J.ERR_INVALID_VALUE
    assert f(2, *_group_args([good, (D16, 128, 128, E16, E16 + 65536, C16)]), None) == J.ERR_INVALID_VALUE
    # the same entries one by one are accepted by the single call's checks
    # (they reach the device check, which fails here without a GPU)
    import torch
    if not torch.cuda.is_available():
        assert f(2, *_group_args([good, other]), None) == J.ERR_UNSUPPORTED_DEVICE


def test_rmsnorm_quantize_validation(lib):
    f = lib.jetfp8_rmsnorm_quantize_act
    assert f(A16, B16, 1e-6, 4, 384, C16, D16, None, None) == J.ERR_SHAPE        # H % 256
    assert f(A16, B16, 1e-6, -1, 512, C16, D16, None, None) == J.ERR_SHAPE
    assert f(A16, B16, 1e-6, 4, 0, C16, D16, None, None) == J.ERR_SHAPE
    assert f(None, None, 1e-6, 0, 512, None, None, None, None) == J.OK             # empty
    assert f(A16, B16, -1.0, 4, 512, C16, D16, None, None) == J.ERR_INVALID_VALUE   # eps < 0
    assert f(A16, B16, float("nan"), 4, 512, C16, D16, None, None) == J.ERR_INVALID_VALUE
    assert f(A16, B16, float("inf"), 4, 512, C16, D16, None, None) == J.ERR_INVALID_VALUE
    assert f(A16, B16, 1e-6, 4, 512, C16, None, None, None) == J.ERR_INVALID_VALUE  # q without s
    assert f(A16, B16, 1e-6, 4, 512, None, None, None, None) == J.ERR_INVALID_VALUE  # nothing to write
    assert f(None, B16, 1e-6, 4, 512, C16, D16, None, None) == J.ERR_INVALID_VALUE
    assert f(A16, B16 + 2, 1e-6, 4, 512, C16, D16, None, None) == J.ERR_ALIGNMENT
    assert f(A16, B16, 1e-6, 4, 512, None, None, E16 + 8, None) == J.ERR_ALIGNMENT
    assert f(A16, B16, 1e-6, 4, 512, A16 + 16, D16, None, None) == J.ERR_INVALID_VALUE   # q overlaps x
    assert f(A16, B16, 1e-6, 4, 512, C16, D16, C16 + 16, None) == J.ERR_INVALID_VALUE    # y overlaps q


def test_swiglu_quantize_validation(lib):
    f = lib.jetfp8_swiglu_quantize_act
    assert f(A16, 4, 128, C16, D16, None, None) == J.ERR_SHAPE                  # I % 256
    assert f(A16, 4, 0, C16, D16, None, None) == J.ERR_SHAPE
    assert f(None, 0, 256, None, None, None, None) == J.OK
    assert f(A16, 4, 256, None, D16, None, None) == J.ERR_INVALID_VALUE         # s without q
    assert f(A16, 4, 256, None, None, None, None) == J.ERR_INVALID_VALUE
    assert f(A16 + 4, 4, 256, C16, D16, None, None) == J.ERR_ALIGNMENT
    assert f(A16, 4, 256, A16 + 1024, D16, None, None) == J.ERR_INVALID_VALUE    # q inside gu


@pytest.mark.parametrize("name", ["jetfp8_gemm_fprop", "jetfp8_gemm_dgrad", "jetfp8_gemm_wgrad"])
def test_gemm_validation(lib, name):
    f = getattr(lib, name)
    assert f(A16, B16, C16, D16, E16, 128, 100, 128, None) == J.ERR_SHAPE
    assert f(A16, B16, C16, D16, E16, 128, 128, 0, None) == J.ERR_SHAPE
    assert f(A16, B16, C16, D16, E16, -1, 128, 128, None) == J.ERR_SHAPE
    assert f(None, None, None, None, None, 0, 128, 128, None) == J.OK
    assert f(None, B16, C16, D16, E16, 128, 128, 128, None) == J.ERR_INVALID_VALUE
    assert f(A16, B16, C16, D16, E16 + 2, 128, 128, 128, None) == J.ERR_ALIGNMENT
    assert f(A16, B16, C16, D16, A16, 128, 128, 128, None) == J.ERR_INVALID_VALUE   # output aliases input
    if name == "jetfp8_gemm_wgrad":
        assert f(A16, B16, C16, D16, E16, 100, 128, 128, None) == J.ERR_SHAPE   # token groups


def test_no_device_reported_cleanly(lib):
    """Without a usable sm_103 device, valid arguments give UNSUPPORTED_DEVICE
    (never a crash, never a CPU fallback)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert lib.jetfp8_quantize_act(A16, 4, 128, B16, C16, None) == J.ERR_UNSUPPORTED_DEVICE
    assert lib.jetfp8_gemm_fprop(A16, B16, C16, D16, E16, 128, 128, 128, None) == J.ERR_UNSUPPORTED_DEVICE
    assert lib.jetfp8_poll_device_error(None) == J.ERR_UNSUPPORTED_DEVICE
    assert lib.jetfp8_watchdog_selftest(0, None) == J.ERR_SHAPE
    assert lib.jetfp8_rmsnorm_quantize_act(A16, B16, 1e-6, 4, 512, C16, D16, None, None) == J.ERR_UNSUPPORTED_DEVICE
    assert lib.jetfp8_swiglu_quantize_act(A16, 4, 256, None, None, E16, None) == J.ERR_UNSUPPORTED_DEVICE


def test_binding_refuses_cpu_tensors(lib):
    import torch
    x = torch.zeros(4, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        jf.quantize_act(x)
