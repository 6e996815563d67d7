"""The boundary is a C ABI: a plain C99 program (tests/c_abi_check.c) compiles
against include/ with -pedantic, links the built library and calls its
host-only entry points (no GPU needed)."""
import os
import shutil
import subprocess

import pytest

import skinny_bf16_gemm_residual_gb300 as sgr
from skinny_bf16_gemm_residual_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_plain_c_client(tmp_path):
    gcc = shutil.which("gcc")
    if not gcc:
        pytest.skip("gcc not available")
    sgr.load()  # builds the library if needed
    lib_dir = os.path.dirname(build.LIB_PATH)
    exe = str(tmp_path / "c_abi_check")
    cc = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                         f"-I{os.path.join(ROOT, 'include')}", os.path.join(ROOT, "tests", "c_abi_check.c"),
                         f"-L{lib_dir}", "-lskinny_gemm_residual", f"-Wl,-rpath,{lib_dir}", "-o", exe],
                        capture_output=True, text=True)
    assert cc.returncode == 0, cc.stderr
    run = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0 and run.stdout.strip() == "ok", run.stdout + run.stderr
