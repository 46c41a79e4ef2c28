"""Builds synth/libsynth.so, the GPU cache-fill generator (test and benchmark
input generation only)."""
from __future__ import annotations

import os
import shutil
import subprocess
from pathlib import Path

HERE = Path(__file__).resolve().parent
LIB = HERE / "libsynth.so"


def build(force: bool = False) -> Path:
    src = HERE / "fill.cu"
    if not force and LIB.exists() and LIB.stat().st_mtime >= src.stat().st_mtime:
        return LIB
    tmp = LIB.with_suffix(f".{os.getpid()}.tmp")
    nvcc = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo",
                    "-std=c++17", "-Xcompiler", "-fPIC", "-shared", "-cudart", "static",
                    str(src), "-o", str(tmp)], check=True)
    os.replace(tmp, LIB)
    return LIB
