"""The C ABI used from plain C: tests/c/abi_check.c includes include/tkq.h as
strict C11, links libtkq.so and the CUDA runtime, and compares the library's
results with the C oracle.  On the CPU it is only compiled and linked; the GPU
test runs it."""
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c", "abi_check.c")


def _cuda_home():
    return os.environ.get("CUDA_HOME", "/usr/local/cuda")


def build_client(out_dir):
    from fp8_activation_quantization_gb300 import _build
    import oracle
    lib = _build.build()
    oracle.build()
    exe = os.path.join(out_dir, "abi_check")
    cuda = _cuda_home()
    cmd = ["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-O1", SRC,
           os.path.join(ROOT, "oracle", "tkq_oracle.c"), "-ffp-contract=off",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(ROOT, "oracle"),
           "-I", os.path.join(cuda, "include"),
           "-L", os.path.dirname(lib), "-ltkq",
           "-L", os.path.join(cuda, "lib64"), "-L", os.path.join(cuda, "lib"), "-lcudart", "-lm",
           "-Wl,-rpath," + os.path.dirname(lib), "-Wl,-rpath," + os.path.join(cuda, "lib64"),
           "-Wl,-rpath," + os.path.join(cuda, "lib"), "-o", exe]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return exe


def test_c_client_compiles_and_links(tmp_path):
    exe = build_client(str(tmp_path))
    assert os.path.exists(exe)


@pytest.mark.gpu
def test_c_client_runs_and_matches_the_oracle(tmp_path, cuda_device):
    exe = build_client(str(tmp_path))
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr + r.stdout
    assert "abi_check: OK" in r.stdout
