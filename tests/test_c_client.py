"""The C ABI from plain C: tests/c_client.c is compiled with gcc as C99
against include/fa.h, linked with libfa.so and run (no GPU needed)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c99_client_compiles_links_and_runs(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("no gcc")
    from exact_io_aware_35_gb300 import build as fa_build
    lib = fa_build.build()
    libdir = os.path.dirname(lib)
    exe = str(tmp_path / "c_client")
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic-errors",
           "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c_client.c"), "-o", exe,
           "-L", libdir, "-lfa", "-Wl,-rpath," + libdir]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().endswith("ok")
