"""The C ABI used from plain C programs (no Python, no torch): compiled with
gcc against include/dv.h and linked with libdv.so."""
import os
import subprocess
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent
PKG = ROOT / "kv_cache_streaming_gb300"
CUDA = Path(os.environ.get("CUDA_HOME", "/usr/local/cuda"))


def _build(src, out, cflags=(), libs=()):
    cmd = ["gcc", "-std=c11", "-O1", "-Wall", "-I", str(ROOT / "include"), *cflags, str(src),
           "-L", str(PKG), "-ldv", f"-Wl,-rpath,{PKG}", *libs, "-o", str(out)]
    subprocess.run(cmd, check=True)


def test_host_side_abi_from_c(tmp_path):
    exe = tmp_path / "abi_host"
    _build(ROOT / "tests" / "c" / "abi_host.c", exe)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr


@pytest.mark.gpu
def test_gpu_round_trip_from_c(tmp_path):
    exe = tmp_path / "gpu_roundtrip"
    cuda_lib = next(p for p in (CUDA / "lib64", CUDA / "lib") if p.exists())
    _build(ROOT / "tests" / "c" / "gpu_roundtrip.c", exe, cflags=["-I", str(CUDA / "include")],
           libs=["-L", str(cuda_lib), f"-Wl,-rpath,{cuda_lib}", "-lcudart"])
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
