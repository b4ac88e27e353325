"""The C ABI from plain C (no GPU): `include/dsa.h` compiles as C99 with
warnings as errors, a C program links against libdsa.so, and the host-only
entry points answer as the header documents (tests/c/abi_check.c)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_header_and_library_from_c(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    import __graft_entry__
    __graft_entry__.build()
    import dsa_sparse_attention_03_gb300 as dsa
    libdir = os.path.dirname(dsa.LIB_PATH)
    exe = str(tmp_path / "abi_check")
    cmd = [cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "c", "abi_check.c"), "-o", exe, "-L", libdir, "-ldsa",
           "-Wl,-rpath," + libdir]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    run = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, run.stdout + run.stderr
    assert run.stdout.strip().endswith("all ok"), run.stdout
