"""Thin Python binding of the jetfp8 C-ABI (``include/jetfp8.h``).

Argument marshalling only: every step of the FP8 path runs in the CUDA
library ``libjetfp8.so``.  There is no fallback -- if the library is missing
or cannot be loaded, every call raises.

Two layers:
  * ``jetfp8_*`` functions with the C names take torch tensors for every
    buffer (inputs and preallocated outputs) and pass raw device pointers and
    the current CUDA stream;
  * allocating helpers (``quantize_act``, ``gemm_fprop`` ...) create the
    outputs with torch (device memory only) and call the ``jetfp8_*`` layer.
Codes are returned as ``torch.uint8`` tensors holding E4M3 bit patterns
(``.view(torch.float8_e4m3fn)`` reinterprets them without a copy).
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libjetfp8.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "jetfp8.h")

STATUS = {
    0: "JETFP8_OK",
    1: "JETFP8_ERR_INVALID_VALUE",
    2: "JETFP8_ERR_SHAPE",
    3: "JETFP8_ERR_ALIGNMENT",
    4: "JETFP8_ERR_UNSUPPORTED_DEVICE",
    5: "JETFP8_ERR_LAUNCH",
    6: "JETFP8_ERR_TIMEOUT",
}
OK, ERR_INVALID_VALUE, ERR_SHAPE, ERR_ALIGNMENT, ERR_UNSUPPORTED_DEVICE, ERR_LAUNCH, ERR_TIMEOUT = range(7)


class Jetfp8Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


_lib = None


def load_library():
    """Load ``libjetfp8.so`` (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"jetfp8 CUDA library not built ({LIB_PATH} missing); "
                           "run e4m3_group_quantise_gb300.build.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, S = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.jetfp8_quantize_act.argtypes = [P, I, I, P, P, P]
    lib.jetfp8_quantize_act_transposed.argtypes = [P, I, I, P, P, P]
    lib.jetfp8_quantize_weight.argtypes = [P, I, I, P, P, P, P]
    lib.jetfp8_quantize_weight_group.argtypes = [S, P, P, P, P, P, P, P]
    lib.jetfp8_quantize_act_dual.argtypes = [P, I, I, P, P, P, P, P]
    lib.jetfp8_rmsnorm_quantize_act.argtypes = [P, P, ctypes.c_float, I, I, P, P, P, P]
    lib.jetfp8_swiglu_quantize_act.argtypes = [P, I, I, P, P, P, P]
    for name in ("jetfp8_gemm_fprop", "jetfp8_gemm_dgrad", "jetfp8_gemm_wgrad"):
        getattr(lib, name).argtypes = [P, P, P, P, P, I, I, I, P]
    for name in ("jetfp8_quantize_act", "jetfp8_quantize_act_transposed", "jetfp8_quantize_weight",
                 "jetfp8_quantize_weight_group", "jetfp8_quantize_act_dual", "jetfp8_rmsnorm_quantize_act", "jetfp8_swiglu_quantize_act",
                 "jetfp8_gemm_fprop", "jetfp8_gemm_dgrad", "jetfp8_gemm_wgrad"):
        getattr(lib, name).restype = S
    lib.jetfp8_e4m3_encode_range.argtypes = [ctypes.c_uint32, I, P, P]
    lib.jetfp8_e4m3_encode_range.restype = S
    lib.jetfp8_act_scale_count.argtypes = [I, I]
    lib.jetfp8_act_scale_count.restype = ctypes.c_size_t
    lib.jetfp8_status_string.argtypes = [S]
    lib.jetfp8_status_string.restype = ctypes.c_char_p
    lib.jetfp8_poll_device_error.argtypes = [P]
    lib.jetfp8_poll_device_error.restype = S
    lib.jetfp8_watchdog_selftest.argtypes = [I, P]
    lib.jetfp8_watchdog_selftest.restype = S
    _lib = lib
    return lib


def declared_functions(header: str = HEADER_PATH):
    """Names of the functions ``include/jetfp8.h`` declares."""
    text = open(header).read()
    return sorted(set(re.findall(r"JETFP8_API\s+[\w\s\*]+?\b(jetfp8_\w+)\s*\(", text)))


# ------------------------------------------------------------------ helpers
def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t) -> int:
    if t is None:
        return 0
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _check(status: int, where: str):
    if status != OK:
        raise Jetfp8Error(status, where)


def _want(t: torch.Tensor, dtype, shape, name):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


# ------------------------------------------------- C-named, preallocated
def jetfp8_quantize_act(x, q, s, stream=None):
    M, K = x.shape
    _want(x, torch.bfloat16, (M, K), "x")
    _want(q, torch.uint8, (M, K), "q")
    _want(s, torch.float32, (K // 128, M), "s")
    _check(load_library().jetfp8_quantize_act(_ptr(x), M, K, _ptr(q), _ptr(s), _stream(stream)),
           "jetfp8_quantize_act")


def jetfp8_quantize_act_transposed(x, qt, st, stream=None):
    M, C = x.shape
    _want(x, torch.bfloat16, (M, C), "x")
    _want(qt, torch.uint8, (C, M), "qt")
    _want(st, torch.float32, (M // 128, C), "st")
    _check(load_library().jetfp8_quantize_act_transposed(_ptr(x), M, C, _ptr(qt), _ptr(st), _stream(stream)),
           "jetfp8_quantize_act_transposed")


def jetfp8_quantize_act_dual(x, q, s, qt, st, stream=None):
    M, K = x.shape
    _want(x, torch.bfloat16, (M, K), "x")
    _want(q, torch.uint8, (M, K), "q")
    _want(s, torch.float32, (K // 128, M), "s")
    _want(qt, torch.uint8, (K, M), "qt")
    _want(st, torch.float32, (M // 128, K), "st")
    _check(load_library().jetfp8_quantize_act_dual(_ptr(x), M, K, _ptr(q), _ptr(s), _ptr(qt), _ptr(st),
                                                   _stream(stream)), "jetfp8_quantize_act_dual")


def jetfp8_rmsnorm_quantize_act(x, gamma, eps, q, s, y=None, stream=None):
    M, H = x.shape
    _want(x, torch.bfloat16, (M, H), "x")
    _want(gamma, torch.bfloat16, (H,), "gamma")
    if q is not None or s is not None:
        _want(q, torch.uint8, (M, H), "q")
        _want(s, torch.float32, (H // 128, M), "s")
    if y is not None:
        _want(y, torch.bfloat16, (M, H), "y")
    _check(load_library().jetfp8_rmsnorm_quantize_act(_ptr(x), _ptr(gamma), float(eps), M, H, _ptr(q), _ptr(s),
                                                      _ptr(y), _stream(stream)), "jetfp8_rmsnorm_quantize_act")


def jetfp8_swiglu_quantize_act(gu, q, s, y=None, stream=None):
    M, I2 = gu.shape
    I = I2 // 2
    _want(gu, torch.bfloat16, (M, 2 * I), "gu")
    if q is not None or s is not None:
        _want(q, torch.uint8, (M, I), "q")
        _want(s, torch.float32, (I // 128, M), "s")
    if y is not None:
        _want(y, torch.bfloat16, (M, I), "y")
    _check(load_library().jetfp8_swiglu_quantize_act(_ptr(gu), M, I, _ptr(q), _ptr(s), _ptr(y), _stream(stream)),
           "jetfp8_swiglu_quantize_act")


def jetfp8_quantize_weight(w, q, s, qt=None, stream=None):
    N, K = w.shape
    _want(w, torch.bfloat16, (N, K), "w")
    _want(q, torch.uint8, (N, K), "q")
    _want(s, torch.float32, (N // 128, K // 128), "s")
    if qt is not None:
        _want(qt, torch.uint8, (K, N), "qt")
    _check(load_library().jetfp8_quantize_weight(_ptr(w), N, K, _ptr(q), _ptr(s), _ptr(qt), _stream(stream)),
           "jetfp8_quantize_weight")


WEIGHT_GROUP_MAX = 8


def jetfp8_quantize_weight_group(ws, qs, ss, qts=None, stream=None):
    """jetfp8_quantize_weight on each (w, q, s, qt) entry, in one launch."""
    n = len(ws)
    qts = [None] * n if qts is None else list(qts)
    if not (len(qs) == len(ss) == len(qts) == n):
        raise ValueError("jetfp8_quantize_weight_group: one q, s and qt per weight")
    if n > WEIGHT_GROUP_MAX:
        raise ValueError(f"jetfp8_quantize_weight_group: at most {WEIGHT_GROUP_MAX} weights per launch")
    for w, q, s, qt in zip(ws, qs, ss, qts):
        N, K = w.shape
        _want(w, torch.bfloat16, (N, K), "w")
        _want(q, torch.uint8, (N, K), "q")
        _want(s, torch.float32, (N // 128, K // 128), "s")
        if qt is not None:
            _want(qt, torch.uint8, (K, N), "qt")
    P = ctypes.c_void_p * max(n, 1)
    I = ctypes.c_int64 * max(n, 1)
    _check(load_library().jetfp8_quantize_weight_group(
        n, P(*[_ptr(w) for w in ws]), I(*[w.shape[0] for w in ws]), I(*[w.shape[1] for w in ws]),
        P(*[_ptr(q) for q in qs]), P(*[_ptr(s) for s in ss]), P(*[_ptr(qt) for qt in qts]), _stream(stream)),
        "jetfp8_quantize_weight_group")


def jetfp8_e4m3_encode_range(first, codes, stream=None):
    """codes[i] = the GPU's E4M3 code of the fp32 pattern first + i (a test hook
    for the conversion the quantisers end in)."""
    _want(codes, torch.uint8, (codes.numel(),), "codes")
    _check(load_library().jetfp8_e4m3_encode_range(int(first), codes.numel(), _ptr(codes), _stream(stream)),
           "jetfp8_e4m3_encode_range")


def jetfp8_gemm_fprop(qx, sx, qw, sw, y, stream=None):
    M, K = qx.shape
    N = qw.shape[0]
    _want(qx, torch.uint8, (M, K), "qx")
    _want(sx, torch.float32, (K // 128, M), "sx")
    _want(qw, torch.uint8, (N, K), "qw")
    _want(sw, torch.float32, (N // 128, K // 128), "sw")
    _want(y, torch.bfloat16, (M, N), "y")
    _check(load_library().jetfp8_gemm_fprop(_ptr(qx), _ptr(sx), _ptr(qw), _ptr(sw), _ptr(y), M, N, K,
                                             _stream(stream)), "jetfp8_gemm_fprop")


def jetfp8_gemm_dgrad(qdy, sdy, qwt, sw, dx, stream=None):
    M, N = qdy.shape
    K = qwt.shape[0]
    _want(qdy, torch.uint8, (M, N), "qdy")
    _want(sdy, torch.float32, (N // 128, M), "sdy")
    _want(qwt, torch.uint8, (K, N), "qwt")
    _want(sw, torch.float32, (N // 128, K // 128), "sw")
    _want(dx, torch.bfloat16, (M, K), "dx")
    _check(load_library().jetfp8_gemm_dgrad(_ptr(qdy), _ptr(sdy), _ptr(qwt), _ptr(sw), _ptr(dx), M, N, K,
                                            _stream(stream)), "jetfp8_gemm_dgrad")


def jetfp8_gemm_wgrad(qdyt, sdyt, qxt, sxt, dw, stream=None):
    N, M = qdyt.shape
    K = qxt.shape[0]
    _want(qdyt, torch.uint8, (N, M), "qdyt")
    _want(sdyt, torch.float32, (M // 128, N), "sdyt")
    _want(qxt, torch.uint8, (K, M), "qxt")
    _want(sxt, torch.float32, (M // 128, K), "sxt")
    _want(dw, torch.bfloat16, (N, K), "dw")
    _check(load_library().jetfp8_gemm_wgrad(_ptr(qdyt), _ptr(sdyt), _ptr(qxt), _ptr(sxt), _ptr(dw), M, N, K,
                                            _stream(stream)), "jetfp8_gemm_wgrad")


def jetfp8_poll_device_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error status."""
    return load_library().jetfp8_poll_device_error(_stream(stream))


def jetfp8_watchdog_selftest(timeout_us: int, stream=None) -> int:
    return load_library().jetfp8_watchdog_selftest(int(timeout_us), _stream(stream))


def jetfp8_act_scale_count(rows: int, cols: int) -> int:
    return load_library().jetfp8_act_scale_count(rows, cols)


def jetfp8_status_string(status: int) -> str:
    return load_library().jetfp8_status_string(status).decode()


# --------------------------------------------------------- allocating API
def quantize_act(x: torch.Tensor, stream=None):
    """bf16 [M,K] -> (codes uint8 [M,K], scales fp32 [K/128, M])."""
    M, K = x.shape
    q = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    s = torch.empty((K // 128, M), dtype=torch.float32, device=x.device)
    jetfp8_quantize_act(x, q, s, stream)
    return q, s


def quantize_act_transposed(x: torch.Tensor, stream=None):
    """bf16 [M,C] -> (codes uint8 [C,M], scales fp32 [M/128, C])."""
    M, C = x.shape
    qt = torch.empty((C, M), dtype=torch.uint8, device=x.device)
    st = torch.empty((M // 128, C), dtype=torch.float32, device=x.device)
    jetfp8_quantize_act_transposed(x, qt, st, stream)
    return qt, st


def quantize_act_dual(x: torch.Tensor, stream=None):
    """bf16 [M,K] -> (q [M,K], s [K/128,M], qt [K,M], st [M/128,K]) in one pass."""
    M, K = x.shape
    q = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    s = torch.empty((K // 128, M), dtype=torch.float32, device=x.device)
    qt = torch.empty((K, M), dtype=torch.uint8, device=x.device)
    st = torch.empty((M // 128, K), dtype=torch.float32, device=x.device)
    jetfp8_quantize_act_dual(x, q, s, qt, st, stream)
    return q, s, qt, st


def rmsnorm_quantize_act(x: torch.Tensor, gamma: torch.Tensor, eps: float, quantize: bool = True,
                         want_y: bool = False, stream=None):
    """RMSNorm fused with the 1x128 quantiser: (q, s, y) with y None unless
    ``want_y``; ``quantize=False`` gives only y (q and s None)."""
    M, H = x.shape
    q = torch.empty((M, H), dtype=torch.uint8, device=x.device) if quantize else None
    s = torch.empty((H // 128, M), dtype=torch.float32, device=x.device) if quantize else None
    y = torch.empty((M, H), dtype=torch.bfloat16, device=x.device) if want_y or not quantize else None
    jetfp8_rmsnorm_quantize_act(x, gamma, eps, q, s, y, stream)
    return q, s, y


def swiglu_quantize_act(gu: torch.Tensor, quantize: bool = True, want_y: bool = False, stream=None):
    """SwiGLU of a gate_up output [M, 2I] fused with the 1x128 quantiser:
    (q, s, y) as for ``rmsnorm_quantize_act``."""
    M, I = gu.shape[0], gu.shape[1] // 2
    q = torch.empty((M, I), dtype=torch.uint8, device=gu.device) if quantize else None
    s = torch.empty((I // 128, M), dtype=torch.float32, device=gu.device) if quantize else None
    y = torch.empty((M, I), dtype=torch.bfloat16, device=gu.device) if want_y or not quantize else None
    jetfp8_swiglu_quantize_act(gu, q, s, y, stream)
    return q, s, y


def quantize_weight(w: torch.Tensor, transposed: bool = True, stream=None):
    """bf16 [N,K] -> (codes [N,K], scales [N/128, K/128], codes^T [K,N] or None)."""
    N, K = w.shape
    q = torch.empty((N, K), dtype=torch.uint8, device=w.device)
    s = torch.empty((N // 128, K // 128), dtype=torch.float32, device=w.device)
    qt = torch.empty((K, N), dtype=torch.uint8, device=w.device) if transposed else None
    jetfp8_quantize_weight(w, q, s, qt, stream)
    return q, s, qt


def quantize_weights(ws, transposed: bool = True, stream=None):
    """quantize_weight of every tensor in ws, one launch per (up to) eight
    tensors: a list of (codes, scales, codes^T or None)."""
    out = []
    for i in range(0, len(ws), WEIGHT_GROUP_MAX):
        chunk = ws[i:i + WEIGHT_GROUP_MAX]
        qs = [torch.empty(w.shape, dtype=torch.uint8, device=w.device) for w in chunk]
        ss = [torch.empty((w.shape[0] // 128, w.shape[1] // 128), dtype=torch.float32, device=w.device)
              for w in chunk]
        qts = [torch.empty((w.shape[1], w.shape[0]), dtype=torch.uint8, device=w.device) if transposed else None
               for w in chunk]
        jetfp8_quantize_weight_group(chunk, qs, ss, qts, stream)
        out.extend(zip(qs, ss, qts))
    return out


def gemm_fprop(qx, sx, qw, sw, stream=None):
    y = torch.empty((qx.shape[0], qw.shape[0]), dtype=torch.bfloat16, device=qx.device)
    jetfp8_gemm_fprop(qx, sx, qw, sw, y, stream)
    return y


def gemm_dgrad(qdy, sdy, qwt, sw, stream=None):
    dx = torch.empty((qdy.shape[0], qwt.shape[0]), dtype=torch.bfloat16, device=qdy.device)
    jetfp8_gemm_dgrad(qdy, sdy, qwt, sw, dx, stream)
    return dx


def gemm_wgrad(qdyt, sdyt, qxt, sxt, stream=None):
    dw = torch.empty((qdyt.shape[0], qxt.shape[0]), dtype=torch.bfloat16, device=qdyt.device)
    jetfp8_gemm_wgrad(qdyt, sdyt, qxt, sxt, dw, stream)
    return dw
