"""The quantisers' per-element code, checked exhaustively on the host (no
GPU, no CUDA code).

The CUDA quantisers code x of a group with scale s = RN(amax / 448) through a
once-corrected quotient q0 = RN(x r), e = RN(x - q0 s), q = RN(q0 + e r)
(fused multiply-adds; r within an ulp of 1/s), where the definition
("Schéma de Quantification": per-group scale amax / 448, codes of x / s) is
the E4M3 code of the fp32 quotient RN(x / s).  q itself is not always the
correctly rounded quotient, so the claim that its code always is, is checked
here for every pair the kernels take this path for: every bf16 amax with
s >= 2^-100, every bf16 x with |x| <= amax other than -0, and r equal to
RN(1/s) or either fp32 neighbour.  The reference codes come from the
oracle's encoder.  A planted mistake (no correction step) must fail.
"""
import ctypes
import os
import subprocess

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "corrected_quotient_check.c")
BASE = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fno-fast-math", "-ffp-contract=off"]

AMAX_LO, AMAX_HI = 0x0001, 0x7F7F      # every positive finite bf16 amax


@pytest.fixture(scope="module")
def checker(tmp_path_factory):
    out = str(tmp_path_factory.mktemp("cq") / "libcq.so")
    try:   # threads when the compiler has OpenMP; the arithmetic is the same either way
        subprocess.check_call(BASE + ["-fopenmp", "-o", out, SRC, "-lm"], stderr=subprocess.DEVNULL)
    except subprocess.CalledProcessError:
        subprocess.check_call(BASE + ["-o", out, SRC, "-lm"])
    lib = ctypes.CDLL(out)
    lib.check_range.restype = ctypes.c_longlong
    lib.check_range.argtypes = [ctypes.c_uint32, ctypes.c_uint32, ctypes.c_int, ctypes.c_void_p,
                                ctypes.POINTER(ctypes.c_longlong), ctypes.POINTER(ctypes.c_longlong)]
    enc = ctypes.cast(oracle._load().jo_e4m3_encode, ctypes.c_void_p)

    def run(lo, hi, variant):
        pairs, qdiff = ctypes.c_longlong(0), ctypes.c_longlong(0)
        bad = lib.check_range(lo, hi, variant, enc, ctypes.byref(pairs), ctypes.byref(qdiff))
        return bad, pairs.value, qdiff.value

    return run


@pytest.mark.parametrize("variant", [0, 1, 2], ids=["rn", "below", "above"])
def test_corrected_quotient_codes_are_exact_for_every_bf16_pair(checker, variant):
    bad, pairs, qdiff = checker(AMAX_LO, AMAX_HI, variant)
    # every magnitude m <= amax with both signs (less -0), for the ~32k
    # amax values whose scale is at least 2^-100: over a billion pairs
    assert pairs > 1_000_000_000
    # the quotient itself differs from RN(x / s) on some pairs (so this is a
    # statement about codes, not about the quotient) ...
    assert qdiff > 0
    # ... but never its code
    assert bad == 0


def test_planted_mistake_uncorrected_quotient_fails(checker):
    # q = RN(x RN(1/s)) alone: codes differ from the definition somewhere
    # (on scales of one binade of amax, which is enough to show it)
    bad, pairs, _ = checker(0x3F80, 0x3FFF, 3)
    assert pairs > 0 and bad > 0
