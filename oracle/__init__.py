"""CPU oracle for the FP8 linear-layer path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The CUDA library never imports it, links it or
shares code with it; the product path fails loudly when its own extension is
missing instead of falling back here.

The arithmetic lives in ``jetfp8_oracle.c`` (plain C, single-threaded, one
output element at a time); this module only marshals numpy arrays through
ctypes.  Splitting independent rows over threads (``threads=``) changes no
arithmetic: every output element is still produced by the same C loop.

What it computes (Jet-RL technical summaries, gist.science fr/pt,
"Schéma de Quantification" / "Esquema de Quantização"):
  * ``quantize_act``            1x128 groups along each row (activations,
                                 gradients); scales group-major [K/128][M].
  * ``quantize_act_transposed`` 128x1 groups along the token axis, written
                                 transposed (the WGrad operand); scales
                                 [M/128][C].
  * ``quantize_weight``         128x128 blocks; scales [N/128][K/128];
                                 optional transposed codes.
  * ``gemm_fprop/dgrad/wgrad``  exact fp64 sums of dequantised products,
                                 plus the sum of |products| for tolerances.
  * ``rmsnorm``, ``swiglu``     the operators fused in front of the linear
                                 layers ("Implémentation": fused activation /
                                 RMSNorm kernels), their textbook definitions
                                 evaluated in fp64; a kernel's bf16 output is
                                 checked against them to within one bf16
                                 ulp and its FP8 form against
                                 ``quantize_act`` of that bf16 output.
Readings the pages leave open (format E4M3-FN, s = amax/448 in fp32, RNE,
saturating, zero group -> s = 0 and codes 0) are stated in the C file.

No test in this package's pins is "parity unpinned": every function is
pinned by the ``-m "not gpu"`` tests (format definition, brute force,
closed forms, invariants, an independent library decode/cast).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "jetfp8_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libjetfp8_oracle.so")

# gcc flags: IEEE semantics kept (no fast-math, no FMA contraction).
_CFLAGS = ["-O2", "-std=c99", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", "-fno-strict-aliasing"]

_lib = None


def _fingerprint() -> str:
    """SHA-256 of the C source, the flags, gcc's version and the machine type."""
    import hashlib
    import platform
    h = hashlib.sha256()
    with open(_SRC, "rb") as f:
        h.update(f.read())
    h.update(" ".join(_CFLAGS).encode())
    h.update(subprocess.run(["gcc", "--version"], capture_output=True, text=True).stdout.encode())
    h.update(platform.machine().encode())
    return h.hexdigest()


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/libjetfp8_oracle.so`` (gcc) unless
    the library on disk was built from exactly the current inputs."""
    fp = _fingerprint()
    stamp = _LIB_PATH + ".sha256"
    if not force and os.path.exists(_LIB_PATH) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == fp:
                return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB_PATH)
    with open(stamp, "w") as f:
        f.write(fp + "\n")
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB_PATH)
    P = ctypes.c_void_p
    I = ctypes.c_int64
    lib.jo_e4m3_decode.restype = ctypes.c_double
    lib.jo_e4m3_decode.argtypes = [ctypes.c_uint8]
    lib.jo_e4m3_encode.restype = ctypes.c_uint8
    lib.jo_e4m3_encode.argtypes = [ctypes.c_float]
    lib.jo_e4m3_encode_array.argtypes = [P, I, P]
    lib.jo_e4m3_decode_array.argtypes = [P, I, P]
    lib.jo_e4m3_encode_check_range.restype = ctypes.c_int64
    lib.jo_e4m3_encode_check_range.argtypes = [ctypes.c_uint32, ctypes.c_uint64, P,
                                               ctypes.POINTER(ctypes.c_int64)]
    lib.jo_quantize_act.argtypes = [P, I, I, P, P]
    lib.jo_quantize_act_transposed.argtypes = [P, I, I, P, P]
    lib.jo_quantize_weight.argtypes = [P, I, I, P, P, P]
    for name in ("jo_gemm_fprop", "jo_gemm_dgrad", "jo_gemm_wgrad"):
        getattr(lib, name).argtypes = [P, P, P, P, I, I, I, P, P, I, P, P]
    lib.jo_swiglu_f64.argtypes = [P, I, I, P]
    lib.jo_rmsnorm_f64.argtypes = [P, P, ctypes.c_double, I, I, P]
    _lib = lib
    return lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _as_bf16_bits(x) -> np.ndarray:
    """Accept uint16 bf16 bit patterns (numpy) or a CPU torch bfloat16 tensor."""
    if isinstance(x, np.ndarray):
        if x.dtype != np.uint16:
            raise TypeError("oracle expects bf16 bit patterns as uint16")
        return np.ascontiguousarray(x)
    # torch tensor (CPU, bfloat16): reinterpret the bits
    import torch
    if x.dtype != torch.bfloat16:
        raise TypeError("oracle expects a bfloat16 tensor")
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy()).view(np.uint16)


# ----------------------------------------------------------------- codec
def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    lib = _load()
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    lib.jo_e4m3_decode_array(_ptr(c), c.size, _ptr(out))
    return out


def e4m3_encode(values: np.ndarray) -> np.ndarray:
    lib = _load()
    v = np.ascontiguousarray(values, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    lib.jo_e4m3_encode_array(_ptr(v), v.size, _ptr(out))
    return out


def e4m3_encode_check_range(lo: int, codes: np.ndarray):
    """Count fp32 patterns lo..lo+len(codes)-1 whose oracle code differs
    from ``codes``.  Returns (mismatches, index of the first one or -1)."""
    lib = _load()
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    first = ctypes.c_int64(-1)
    bad = lib.jo_e4m3_encode_check_range(ctypes.c_uint32(lo), ctypes.c_uint64(c.size),
                                         _ptr(c), ctypes.byref(first))
    return int(bad), int(first.value)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ------------------------------------------------------------- quantise
def _row_chunks(n: int, threads: int):
    threads = max(1, min(threads, n))
    step = -(-n // threads)
    return [(a, min(n, a + step)) for a in range(0, n, step)]


def quantize_act(x, threads: int = 1):
    """X bf16 [M,K] -> (q uint8 [M,K], s float32 [K/128, M])."""
    lib = _load()
    xb = _as_bf16_bits(x)
    M, K = xb.shape
    if K % 128:
        raise ValueError("K must be a multiple of 128")
    G = K // 128
    q = np.empty((M, K), dtype=np.uint8)
    s = np.empty((G, M), dtype=np.float32)
    if threads <= 1 or M < 2:
        lib.jo_quantize_act(_ptr(xb), M, K, _ptr(q), _ptr(s))
        return q, s

    def work(r):
        a, b = r
        sub_x = np.ascontiguousarray(xb[a:b])
        sub_q = np.empty((b - a, K), dtype=np.uint8)
        sub_s = np.empty((G, b - a), dtype=np.float32)
        lib.jo_quantize_act(_ptr(sub_x), b - a, K, _ptr(sub_q), _ptr(sub_s))
        q[a:b] = sub_q
        s[:, a:b] = sub_s

    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(work, _row_chunks(M, threads)))
    return q, s


def quantize_act_transposed(x, threads: int = 1):
    """X bf16 [M,C] -> (qt uint8 [C,M], st float32 [M/128, C])."""
    lib = _load()
    xb = _as_bf16_bits(x)
    M, C = xb.shape
    if M % 128 or C % 128:
        raise ValueError("M and C must be multiples of 128")
    G = M // 128
    qt = np.empty((C, M), dtype=np.uint8)
    st = np.empty((G, C), dtype=np.float32)
    if threads <= 1:
        lib.jo_quantize_act_transposed(_ptr(xb), M, C, _ptr(qt), _ptr(st))
        return qt, st

    # independent column slices
    def work(r):
        a, b = r
        sub_x = np.ascontiguousarray(xb[:, a:b])
        sub_q = np.empty((b - a, M), dtype=np.uint8)
        sub_s = np.empty((G, b - a), dtype=np.float32)
        lib.jo_quantize_act_transposed(_ptr(sub_x), M, b - a, _ptr(sub_q), _ptr(sub_s))
        qt[a:b] = sub_q
        st[:, a:b] = sub_s

    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(work, _row_chunks(C, threads)))
    return qt, st


def quantize_weight(w, want_transposed: bool = False, threads: int = 1):
    """W bf16 [N,K] -> (q uint8 [N,K], s float32 [N/128, K/128], qt [K,N] or None)."""
    lib = _load()
    wb = _as_bf16_bits(w)
    N, K = wb.shape
    if N % 128 or K % 128:
        raise ValueError("N and K must be multiples of 128")
    q = np.empty((N, K), dtype=np.uint8)
    s = np.empty((N // 128, K // 128), dtype=np.float32)
    qt = np.empty((K, N), dtype=np.uint8) if want_transposed else None
    if threads <= 1:
        lib.jo_quantize_weight(_ptr(wb), N, K, _ptr(q), _ptr(s),
                               _ptr(qt) if qt is not None else None)
        return q, s, qt

    bands = [(a * 128, b * 128) for a, b in _row_chunks(N // 128, threads)]

    def work(r):
        a, b = r
        sub_w = np.ascontiguousarray(wb[a:b])
        sub_q = np.empty((b - a, K), dtype=np.uint8)
        sub_s = np.empty(((b - a) // 128, K // 128), dtype=np.float32)
        lib.jo_quantize_weight(_ptr(sub_w), b - a, K, _ptr(sub_q), _ptr(sub_s), None)
        q[a:b] = sub_q
        s[a // 128:b // 128] = sub_s

    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(work, bands))
    if qt is not None:
        qt[...] = q.T
    return q, s, qt


# ---------------------------------------------------------------- GEMMs
def _gemm(name, a_q, a_s, b_q, b_s, M, N, K, out_shape, rows, cols, threads):
    lib = _load()
    fn = getattr(lib, name)
    arrays = [np.ascontiguousarray(a_q, dtype=np.uint8), np.ascontiguousarray(a_s, dtype=np.float32),
              np.ascontiguousarray(b_q, dtype=np.uint8), np.ascontiguousarray(b_s, dtype=np.float32)]
    full = rows is None
    if full:
        R, C = out_shape
        rr, cc = np.meshgrid(np.arange(R, dtype=np.int64), np.arange(C, dtype=np.int64), indexing="ij")
        rows, cols = rr.ravel(), cc.ravel()
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    n = rows.size
    val = np.empty(n, dtype=np.float64)
    asum = np.empty(n, dtype=np.float64)

    def work(r):
        a, b = r
        fn(*[_ptr(x) for x in arrays], M, N, K,
           _ptr(rows[a:b]), _ptr(cols[a:b]), b - a,
           ctypes.c_void_p(val.ctypes.data + 8 * a), ctypes.c_void_p(asum.ctypes.data + 8 * a))

    chunks = _row_chunks(n, threads) if n else []
    if threads <= 1:
        for c in chunks:
            work(c)
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(work, chunks))
    if full:
        return val.reshape(out_shape), asum.reshape(out_shape)
    return val, asum


def gemm_fprop(qx, sx, qw, sw, rows=None, cols=None, threads: int = 1):
    """Y [M,N] = deq(X) deq(W)^T in fp64 (+ sum of |terms|).
    qx [M,K], sx [K/128,M], qw [N,K], sw [N/128,K/128]."""
    M, K = qx.shape
    N = qw.shape[0]
    return _gemm("jo_gemm_fprop", qx, sx, qw, sw, M, N, K, (M, N), rows, cols, threads)


def gemm_dgrad(qdy, sdy, qw, sw, rows=None, cols=None, threads: int = 1):
    """dX [M,K] = deq(dY) deq(W) in fp64 (+ sum of |terms|).
    qdy [M,N], sdy [N/128,M], qw [N,K] (natural layout), sw [N/128,K/128]."""
    M, N = qdy.shape
    K = qw.shape[1]
    return _gemm("jo_gemm_dgrad", qdy, sdy, qw, sw, M, N, K, (M, K), rows, cols, threads)


def gemm_wgrad(qdyt, sdyt, qxt, sxt, rows=None, cols=None, threads: int = 1):
    """dW [N,K] = deq(dY)^T deq(X) over tokens in fp64 (+ sum of |terms|).
    qdyt [N,M], sdyt [M/128,N], qxt [K,M], sxt [M/128,K]."""
    N, M = qdyt.shape
    K = qxt.shape[0]
    return _gemm("jo_gemm_wgrad", qdyt, sdyt, qxt, sxt, M, N, K, (N, K), rows, cols, threads)


# ------------------------------------------------------------ tolerance
def bf16_ulp(ref: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |ref| (8 significant bits); below the
    smallest normal (2^-126) the subnormal spacing 2^-133."""
    a = np.abs(np.asarray(ref, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    ulp = np.exp2(e - 7)
    return np.where(a >= 2.0 ** -126, ulp, 2.0 ** -133)


def gemm_within_tolerance(got, ref, abssum, rel: float = 1e-3):
    """The GEMM bar: |got - ref| <= rel * sum|a*b| + ulp_bf16(ref), per element.
    Returns (all_ok, worst ratio err/bound, flat index of the worst)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    bound = rel * np.asarray(abssum, dtype=np.float64) + bf16_ulp(ref)
    ratio = np.abs(got - ref) / bound
    if ratio.size == 0:
        return True, 0.0, -1
    worst = int(np.nanargmax(np.where(np.isnan(ratio), np.inf, ratio)))
    ok = bool(np.all(np.isfinite(got)) and np.all(ratio <= 1.0))
    return ok, float(ratio.ravel()[worst]), worst


def bf16_within_ulp(got_bits, ref, ulps: float = 1.0):
    """The producers' bar: a bf16 result (bit patterns) within ``ulps`` bf16
    ulps of the fp64 value, per element.  Returns (all_ok, worst error in
    ulps, flat index of the worst)."""
    got = bf16_bits_to_f32(got_bits).astype(np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref) / bf16_ulp(ref)
    if err.size == 0:
        return True, 0.0, -1
    worst = int(np.nanargmax(np.where(np.isnan(err), np.inf, err)))
    ok = bool(np.all(err <= ulps))
    return ok, float(err.ravel()[worst]), worst


# ------------------------------------------------------------ producers
def swiglu(gu, threads: int = 1) -> np.ndarray:
    """gate_up output bf16 [M, 2I] -> y float64 [M, I] = silu(gate) * up,
    evaluated in fp64 (the kernel's bf16 y is checked against it to within
    one bf16 ulp)."""
    lib = _load()
    g = _as_bf16_bits(gu)
    M, I2 = g.shape
    if I2 % 2:
        raise ValueError("gate_up width must be even")
    I = I2 // 2
    y = np.empty((M, I), dtype=np.float64)

    def work(r):
        a, b = r
        sub = np.ascontiguousarray(g[a:b])
        out = np.empty((b - a, I), dtype=np.float64)
        lib.jo_swiglu_f64(_ptr(sub), b - a, I, _ptr(out))
        y[a:b] = out

    chunks = _row_chunks(M, max(1, threads)) if M else []
    if threads <= 1:
        for c in chunks:
            work(c)
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(work, chunks))
    return y


def rmsnorm(x, gamma, eps: float, threads: int = 1) -> np.ndarray:
    """x bf16 [M, H], gamma bf16 [H] -> y float64 [M, H], RMSNorm in fp64.
    ``eps`` is taken at fp32 precision (the C-ABI passes it as a float)."""
    lib = _load()
    xb = _as_bf16_bits(x)
    gb = np.ascontiguousarray(_as_bf16_bits(gamma).reshape(-1))
    M, H = xb.shape
    if gb.size != H:
        raise ValueError("gamma must have H entries")
    eps64 = float(np.float32(eps))
    y = np.empty((M, H), dtype=np.float64)

    def work(r):
        a, b = r
        sub = np.ascontiguousarray(xb[a:b])
        out = np.empty((b - a, H), dtype=np.float64)
        lib.jo_rmsnorm_f64(_ptr(sub), _ptr(gb), ctypes.c_double(eps64), b - a, H, _ptr(out))
        y[a:b] = out

    chunks = _row_chunks(M, max(1, threads)) if M else []
    if threads <= 1:
        for c in chunks:
            work(c)
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(work, chunks))
    return y
