"""The grid-barrier protocol without a GPU: host threads run the same
arrive-and-spin template the top-k kernel's grid barriers use
(``csrc/barrier_protocol.h``) through ``tests/c/barrier_check.cc``.  With every
arrival they all pass; with one arrival dropped every waiter gives up at the
limit, records the timeout, and returns instead of waiting forever."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_dropped_arrival_times_out_on_host_threads(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    exe = str(tmp_path / "barrier_check")
    cmd = [cxx, "-std=c++17", "-O1", "-Wall", "-Wextra", "-Werror", "-pthread",
           "-I", os.path.join(ROOT, "dsa_sparse_attention_03_gb300", "csrc"),
           os.path.join(ROOT, "tests", "c", "barrier_check.cc"), "-o", exe]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    run = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, run.stdout + run.stderr
    assert run.stdout.strip().endswith("all ok"), run.stdout
