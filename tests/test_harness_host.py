"""The native timing harness (jetfp8_bench, C++ over the C-ABI) on the host:
it is built by build(), links against the in-tree library, and rejects bad
arguments with a message and exit status 1 before touching a GPU."""
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
EXE = os.path.join(ROOT, "e4m3_group_quantise_gb300", "jetfp8_bench")


@pytest.fixture(scope="module")
def exe():
    import __graft_entry__
    __graft_entry__.build()
    assert os.path.exists(EXE)
    return EXE


def test_links_the_in_tree_library(exe):
    out = subprocess.run(["ldd", exe], capture_output=True, text=True).stdout
    line = [l for l in out.splitlines() if "libjetfp8.so" in l]
    assert line and os.path.join(ROOT, "e4m3_group_quantise_gb300", "libjetfp8.so") in line[0]


@pytest.mark.parametrize("args,msg", [
    (["--workload", "train-70b"], "unknown workload"),
    (["--steps", "0"], "arguments"),
    (["--streams", "3"], "arguments"),
    (["--bogus"], "unknown argument"),
    (["--steps"], "missing value"),
])
def test_rejects_bad_arguments(exe, args, msg):
    out = subprocess.run([exe, *args], capture_output=True, text=True, timeout=60)
    assert out.returncode == 1
    assert msg in out.stderr
