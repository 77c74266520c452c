"""The boundary from plain C: tests/c_abi_check.c compiled with gcc as C11
against include/lact.h and linked with liblact.so, run on the host (no GPU
needed for the calls it makes)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "chunk_test_step_b300")


@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc not installed")
def test_header_compiles_as_c_and_host_calls_answer(tmp_path):
    lib = os.path.join(PKG, "liblact.so")
    if not os.path.exists(lib):
        from chunk_test_step_b300 import build
        build.build()
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    exe = str(tmp_path / "c_abi_check")
    cmd = ["gcc", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
           os.path.join(ROOT, "tests", "c_abi_check.c"), "-o", exe, "-L", PKG, "-llact", f"-Wl,-rpath,{PKG}",
           "-L", os.path.join(cuda, "lib64"), "-lcudart", f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    out = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, (out.returncode, out.stderr)
    assert out.stdout.startswith("workspace_bytes ")
