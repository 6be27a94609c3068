"""The product path (the package and bench's timed arm) never reaches the
oracle, and fails loudly instead of falling back when the CUDA library is
missing; the binding rejects host tensors before it calls the library."""
import ast
import os

import pytest
import torch

import e4m3_group_quantise_gb300 as jf
from e4m3_group_quantise_gb300 import jetfp8 as J

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "e4m3_group_quantise_gb300")


def _imports(path):
    tree = ast.parse(open(path).read())
    names = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            names.update(a.name.split(".")[0] for a in node.names)
        elif isinstance(node, ast.ImportFrom) and node.module:
            names.add(node.module.split(".")[0])
    return names


def test_package_never_imports_the_oracle():
    for name in os.listdir(PKG):
        if name.endswith(".py"):
            assert "oracle" not in _imports(os.path.join(PKG, name)), name


def test_missing_library_fails_loudly(monkeypatch):
    monkeypatch.setattr(J, "_lib", None)
    monkeypatch.setattr(J, "LIB_PATH", os.path.join(PKG, "no_such_libjetfp8.so"))
    with pytest.raises(RuntimeError, match="not built"):
        J.load_library()
    x = torch.zeros(128, 128, dtype=torch.bfloat16)
    with pytest.raises((RuntimeError, ValueError)):
        jf.quantize_act(x)


def test_binding_rejects_host_tensors_and_non_tensors():
    """Host memory never reaches the library (its pointers are device
    pointers); dtype and shape checks follow on device tensors."""
    x = torch.zeros(128, 256, dtype=torch.bfloat16)
    q = torch.zeros(128, 256, dtype=torch.uint8)
    s = torch.zeros(2, 128, dtype=torch.float32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        jf.jetfp8_quantize_act(x, q, s)
    with pytest.raises(ValueError, match="CUDA tensor"):
        jf.jetfp8_gemm_fprop(q, s, q, s, x)
    with pytest.raises(TypeError):
        J._want(x.float().numpy(), torch.bfloat16, (128, 256), "x")
