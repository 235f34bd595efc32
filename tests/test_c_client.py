"""The C ABI from plain C: tests/c_client.c is compiled with gcc as C99
against include/fa.h, linked with libfa.so and run (no GPU needed); built
with the CUDA runtime, its GPU mode runs fa_fwd and fa_bwd with no PyTorch
and checks them against tests/golden/c_client_case.txt (oracle values)."""
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


CUDA_HOME = os.environ.get("CUDA_HOME", "/usr/local/cuda")


@pytest.mark.gpu
def test_c99_client_gpu_mode_matches_the_oracle(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("no gcc")
    from exact_io_aware_35_gb300 import build as fa_build
    lib = fa_build.build()
    libdir = os.path.dirname(lib)
    exe = str(tmp_path / "c_client_gpu")
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-DFA_CLIENT_GPU",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA_HOME, "include"),
           os.path.join(ROOT, "tests", "c_client.c"), "-o", exe,
           "-L", libdir, "-lfa", "-Wl,-rpath," + libdir,
           "-L", os.path.join(CUDA_HOME, "lib64"), "-lcudart", "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    case = os.path.join(ROOT, "tests", "golden", "c_client_case.txt")
    # a fresh process: no PyTorch, no CUDA context but the client's own
    r = subprocess.run([exe, "gpu", case], capture_output=True, text=True, timeout=300)
    print(r.stdout)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().endswith("ok")
