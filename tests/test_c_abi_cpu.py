"""The boundary from plain C: a C99 program that includes only the public
header compiles with gcc (-Wall -Wextra -Werror -pedantic), links the built
library, and its host-side calls behave as documented (no GPU needed)."""
import shutil
import subprocess
from pathlib import Path

import pytest

import paged_attention_decode_kv_gb300 as vt

ROOT = Path(__file__).resolve().parents[1]


def test_c_program_against_the_header(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    from paged_attention_decode_kv_gb300 import build_lib
    build_lib.build()
    lib = vt.LIBRARY_PATH
    exe = tmp_path / "c_abi_host"
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", f"-I{ROOT / 'include'}",
           str(ROOT / "tests" / "c_abi_host.c"), str(lib), f"-Wl,-rpath,{lib.parent}", "-o", str(exe)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0 and "c abi: ok" in run.stdout, run.stdout + run.stderr
