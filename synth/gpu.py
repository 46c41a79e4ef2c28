"""GPU side of the seeded cache fill (``synth/fill.cu``): fills a device
tensor with the same bytes ``synth.fill_bytes`` produces on the host."""
from __future__ import annotations

import ctypes

import synth
from synth import build as _build

_KIND = {"raw": 0, "fp16": 1, "bf16": 2, "fp32": 3}
_lib = None


def _load():
    global _lib
    if _lib is None:
        if not _build.LIB.exists():
            raise RuntimeError(f"{_build.LIB} is missing: run synth.build.build()")
        lib = ctypes.CDLL(str(_build.LIB))
        lib.synth_fill.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int,
                                   ctypes.c_void_p]
        lib.synth_fill.restype = ctypes.c_int
        _lib = lib
    return _lib


def fill_tensor(t, seed: int, kv: int, kind: str, stream=None) -> None:
    """Fill device tensor ``t`` (whole allocation view) as tensor ``kv`` of a
    cache with seed ``seed``."""
    import torch
    nbytes = t.numel() * t.element_size()
    s = (stream or torch.cuda.current_stream()).cuda_stream
    rc = _load().synth_fill(t.data_ptr(), nbytes, synth.stream_base(seed, kv), _KIND[kind], s)
    if rc != 0:
        raise RuntimeError(f"synth_fill failed with code {rc}")


def fill_cache(geom, k, v, seed: int, stream=None) -> None:
    fill_tensor(k, seed, 0, geom.kind, stream)
    fill_tensor(v, seed, 1, geom.kind, stream)
