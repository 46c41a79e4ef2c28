"""Builds libdv.so (the copy library) in-tree with nvcc for sm_103a.

    python kv_cache_streaming_gb300/build.py

(run it as a script, or load it by path: importing the package itself loads
the library this file builds).

Translation units compile in parallel; the result is
``kv_cache_streaming_gb300/libdv.so``.  The CUDA runtime is linked
statically; the driver is reached through the runtime, so the library also
loads (for symbol checks) on a machine without a GPU driver.  A linker
version script (``csrc/libdv.map``) exports the C ABI alone.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
OBJ = PKG / "_build"
LIB = PKG / "libdv.so"
LIB_CHECKED = PKG / "libdv_checked.so"  # device-side bounds checks (debugging)
SOURCES = ["dv_api.cu", "dv_replica.cu", "dv_sched.cu", "dv_hostmem.cu", "dv_kernels.cu",
           "dv_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and Path(cand).exists():
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libdv")


def _compile(src: str, checked: bool) -> Path:
    out_dir = OBJ / ("checked" if checked else "release")
    out = out_dir / (Path(src).stem + ".o")
    defs = ["-DDV_CHECKED=1"] if checked else []
    cmd = [nvcc(), *ARCH, "-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC",
           "-Xcompiler", "-Wall", *defs, "-I", str(ROOT / "include"), "-c", str(CSRC / src),
           "-o", str(out)]
    subprocess.run(cmd, check=True)
    return out


def _stale(target: Path, deps) -> bool:
    if not target.exists():
        return True
    t = target.stat().st_mtime
    return any(Path(d).stat().st_mtime > t for d in deps)


def build(force: bool = False, checked: bool = False) -> Path:
    """Builds libdv.so, or with `checked` the bounds-checked libdv_checked.so."""
    lib = LIB_CHECKED if checked else LIB
    deps = [CSRC / s for s in SOURCES] + [CSRC / "dv_plan.h", CSRC / "dv_host.h",
                                          CSRC / "libdv.map", ROOT / "include" / "dv.h",
                                          Path(__file__)]
    if not force and not _stale(lib, deps):
        return lib
    (OBJ / ("checked" if checked else "release")).mkdir(parents=True, exist_ok=True)
    with ThreadPoolExecutor(len(SOURCES)) as ex:
        objs = list(ex.map(lambda src: _compile(src, checked), SOURCES))
    tmp = lib.with_suffix(f".{os.getpid()}.tmp")
    subprocess.run([nvcc(), *ARCH, "-shared", "-cudart", "static",
                    "-Xlinker", f"--version-script={CSRC / 'libdv.map'}", "-o", str(tmp),
                    *map(str, objs)], check=True)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, checked="--checked" in sys.argv))
