"""Builds libvt_paged_attn.so in-tree with nvcc for sm_103a (GB300).

Each translation unit compiles in its own nvcc process, in parallel, then one
link step produces ``_build/libvt_paged_attn.so`` beside this file.  The CUDA
runtime is linked statically, so the library needs only the NVIDIA driver at
run time; nothing is installed outside the repository.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

HERE = Path(__file__).resolve().parent
CSRC = HERE / "csrc"
INCLUDE = HERE.parent / "include"
BUILD = HERE / "_build"
LIBRARY = BUILD / "libvt_paged_attn.so"
SOURCES = [
    "vt_paged_attn_api.cu",
    "decode_d64.cu",
    "decode_d128_bf16.cu",
    "decode_d256_bf16.cu",
    "decode_d512_bf16.cu",
    "decode_d128_f32.cu",
    "decode_d256_f32.cu",
    "decode_e4m3.cu",
]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr", f"-I{INCLUDE}"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and Path(cand).exists():
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def _inputs():
    return [CSRC / s for s in SOURCES] + sorted(CSRC.glob("*.cuh")) + [INCLUDE / "vt_paged_attn.h", Path(__file__)]


def up_to_date() -> bool:
    if not LIBRARY.exists():
        return False
    t = LIBRARY.stat().st_mtime
    return all(p.stat().st_mtime <= t for p in _inputs())


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> Path:
    if not force and up_to_date():
        return LIBRARY
    obj_dir = BUILD / "obj"
    obj_dir.mkdir(parents=True, exist_ok=True)
    exe = nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []

    def compile_one(src: str):
        obj = obj_dir / (Path(src).stem + ".o")
        cmd = [exe, *ARCH, *FLAGS, *extra, "-c", str(CSRC / src), "-o", str(obj)]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, obj, r

    with ThreadPoolExecutor(max_workers=min(len(SOURCES), os.cpu_count() or 4)) as pool:
        results = list(pool.map(compile_one, SOURCES))
    for src, _, r in results:
        if verbose or ptxas_info:
            sys.stderr.write(r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    tmp = LIBRARY.with_suffix(f".{os.getpid()}.tmp")
    cmd = [exe, *ARCH, "-shared", "-cudart", "static", "-o", str(tmp),
           *[str(obj) for _, obj, _ in results], "-lpthread", "-ldl", "-lrt"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIBRARY)
    return LIBRARY


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))
