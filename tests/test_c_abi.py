"""libasyncpipe from a plain C program (tests/c/abi_check.c): the headers
compile as C99 and the library links and works without Python or torch."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA_HOME = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _build(tmp_path) -> str:
    from async_global_shared_gb300 import build

    lib = build.build()
    exe = str(tmp_path / "abi_check")
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-O1",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA_HOME, "include"),
           os.path.join(ROOT, "tests", "c", "abi_check.c"), "-o", exe,
           "-L", os.path.dirname(lib), "-lasyncpipe", "-Wl,-rpath," + os.path.dirname(lib),
           "-L", os.path.join(CUDA_HOME, "lib64"), "-lcudart", "-Wl,-rpath," + os.path.join(CUDA_HOME, "lib64")]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    # the library's soname is its file name
    return exe


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_c_program_argument_checks(tmp_path):
    exe = _build(tmp_path)
    r = subprocess.run([exe, "--no-gpu"], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert "c abi ok" in r.stdout


@pytest.mark.gpu
def test_c_program_on_gpu(tmp_path):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    exe = _build(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c abi ok" in r.stdout
