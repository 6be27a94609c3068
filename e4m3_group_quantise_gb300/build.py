"""Build the CUDA library ``libjetfp8.so`` in-tree with nvcc (sm_103a only),
and the native timing harness ``jetfp8_bench`` that drives it.

Four translation units (C-ABI, quantisers, GEMM, producers) compile in parallel and
link into one shared object with the CUDA runtime linked statically, so the
library needs nothing at load time but the driver (which it reaches through
the runtime only when a call is made).  The harness (host C++ only) links
against that library, found next to it at run time.
"""
from __future__ import annotations

import hashlib
import os
import platform
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(PKG, "libjetfp8.so")
HARNESS_PATH = os.path.join(PKG, "jetfp8_bench")
SOURCES = ["api.cu", "quantize.cu", "gemm.cu", "producers.cu"]
HARNESS_SOURCE = "harness.cpp"
HEADERS = ["ptx.cuh", "internal.cuh", "e4m3.cuh"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# IEEE division and denormals are part of the numerical contract: no
# fast-math, no flush-to-zero.
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr",
              "-Xcompiler", "-fPIC,-fvisibility=hidden", "-ftz=false", "-prec-div=true",
              "-prec-sqrt=true", "-fmad=true"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


STAMP_PATH = LIB_PATH + ".sha256"


def _fingerprint(cc: str) -> str:
    """SHA-256 of everything the library is built from: the sources and
    headers, this script (flags), the compiler's version and the host
    machine type (a library built on another architecture is never reused)."""
    h = hashlib.sha256()
    files = [os.path.join(CSRC, f) for f in SOURCES + HEADERS + [HARNESS_SOURCE]] + [
        os.path.join(INCLUDE, "jetfp8.h"), os.path.abspath(__file__)]
    for f in files:
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    ver = subprocess.run([cc, "--version"], capture_output=True, text=True).stdout
    h.update(ver.encode())
    h.update(platform.machine().encode())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile and link ``libjetfp8.so`` unless the library on disk was built
    from exactly the current inputs (same fingerprint); returns its path."""
    cc = nvcc()
    fp = _fingerprint(cc)
    if (not force and not ptxas_info and os.path.exists(LIB_PATH) and os.path.exists(HARNESS_PATH)
            and os.path.exists(STAMP_PATH)):
        with open(STAMP_PATH) as f:
            if f.read().strip() == fp:
                return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    extra = ["-Xptxas", "-v"] if ptxas_info else []

    def compile_one(src):
        obj = os.path.join(BUILD_DIR, os.path.splitext(src)[0] + ".o")
        if src == HARNESS_SOURCE:     # host code only
            cmd = [cc, "-O2", "-std=c++17", "-Xcompiler", "-pthread", "-I", INCLUDE, "-c",
                   os.path.join(CSRC, src), "-o", obj]
        else:
            cmd = [cc, *ARCH, *NVCC_FLAGS, *extra, "-I", INCLUDE, "-I", CSRC, "-c", os.path.join(CSRC, src), "-o",
                   obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{res.stdout}\n{res.stderr}")
        return obj, res.stderr

    with ThreadPoolExecutor(len(SOURCES) + 1) as ex:
        results = list(ex.map(compile_one, SOURCES + [HARNESS_SOURCE]))
    harness_obj = results.pop()[0]
    if verbose or ptxas_info:
        for _, log in results:
            sys.stderr.write(log)
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *[o for o, _ in results]]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, LIB_PATH)
    tmp = HARNESS_PATH + f".tmp{os.getpid()}"
    cmd = [cc, "-o", tmp, harness_obj, "-L", PKG, "-ljetfp8", "-Xcompiler", "-pthread", "-Xlinker",
           "-rpath,$ORIGIN"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"harness link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, HARNESS_PATH)
    with open(STAMP_PATH, "w") as f:
        f.write(fp + "\n")
    return LIB_PATH


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv)
    print(LIB_PATH)
