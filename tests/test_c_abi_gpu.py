"""A decode driven from a C program alone (CUDA runtime buffers, the public
header's entry point) and checked there against the C oracle."""
import os
import shutil
import subprocess
from pathlib import Path

import pytest

import paged_attention_decode_kv_gb300 as vt

ROOT = Path(__file__).resolve().parents[1]


@pytest.mark.gpu
def test_c_program_runs_a_decode(tmp_path):
    if shutil.which("gcc") is None:
        pytest.fail("gcc is needed to build the C test program")
    import oracle
    from paged_attention_decode_kv_gb300 import build_lib
    build_lib.build()
    oracle_lib = oracle.build()
    cuda = Path(os.environ.get("CUDA_HOME", "/usr/local/cuda"))
    libdirs = [d for d in (cuda / "lib64", cuda / "lib") if (d / "libcudart.so").exists()]
    assert libdirs, f"no libcudart.so under {cuda}"
    exe = tmp_path / "c_abi_gpu"
    cmd = ["gcc", "-std=c99", "-O2", "-Wall", "-Wextra", "-Werror", f"-I{ROOT / 'include'}", f"-I{cuda / 'include'}",
           str(ROOT / "tests" / "c_abi_gpu.c"), str(vt.LIBRARY_PATH), str(oracle_lib), f"-L{libdirs[0]}", "-lcudart",
           "-lm", f"-Wl,-rpath,{vt.LIBRARY_PATH.parent}", f"-Wl,-rpath,{Path(oracle_lib).parent}",
           f"-Wl,-rpath,{libdirs[0]}", "-o", str(exe)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert run.returncode == 0 and "c abi gpu: ok" in run.stdout, run.stdout + run.stderr
