"""The library from plain C: tests/c_abi_check.c includes only halo.h and
stencil.h, allocates with the CUDA runtime and calls the C ABI directly (no
Python, no PyTorch).  Compiled and linked on any machine; run on a GPU."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_abi_check.c")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def build_consumer(out):
    from domain_decomposition_halo_build_gb300 import _build
    lib = _build.build()
    libdir = os.path.dirname(lib)
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(CUDA, "include"), SRC, "-o", out, "-L", libdir, "-lhalo",
           "-L", os.path.join(CUDA, "lib64"), "-lcudart", "-lm", "-Wl,-rpath," + libdir]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    return out


def test_c_consumer_compiles_and_links(tmp_path):
    build_consumer(str(tmp_path / "c_abi_check"))


@pytest.mark.gpu
def test_c_consumer_runs(tmp_path):
    exe = build_consumer(str(tmp_path / "c_abi_check"))
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c abi ok" in r.stdout
