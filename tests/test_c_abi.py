"""The C ABI from plain C: tests/c_abi_smoke.c is compiled with gcc against
include/mp_layout.h and the built library (no Python, no torch on its path).
On the CPU the program is only compiled (the header must be valid C11); on a
GPU it runs a layout -> dispatch -> combine pass, the same dispatch in one call
(mp_layout_dispatch), a low-latency dispatch -> weighted combine pass and the
low-latency dispatch with MXFP8 quantisation in the row copy, and checks them."""
import os
import shutil
import subprocess

import pytest

from combine_mp_layout_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_abi_smoke.c")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _cc(out, extra):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    cmd = [cc, "-std=c11", "-O1", "-Wall", "-Wextra", "-Werror",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
           SRC, "-o", out] + extra
    subprocess.run(cmd, check=True, capture_output=True, text=True)


def _link(exe):
    lib = _build.build()
    libdir = os.path.dirname(lib)
    cudalib = os.path.join(CUDA, "lib64")
    _cc(exe, ["-L", libdir, "-l:" + os.path.basename(lib), "-Wl,-rpath," + libdir,
              "-L", cudalib, "-lcudart", "-Wl,-rpath," + cudalib])


def test_c_program_compiles_and_links(tmp_path):
    """Valid C11 against the header, and every call it makes resolves in the library."""
    _cc(str(tmp_path / "c_abi_smoke.o"), ["-c"])
    _link(str(tmp_path / "c_abi_smoke"))


@pytest.mark.gpu
def test_c_program_runs_a_pass(tmp_path):
    exe = str(tmp_path / "c_abi_smoke")
    _link(exe)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert "c abi smoke ok" in r.stdout
