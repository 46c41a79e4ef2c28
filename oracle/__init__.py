"""Oracle of the KV-cache buffered copy: a plain CPU loop nest in C
(``oracle/dv_oracle.c``) behind a ctypes wrapper.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference leg may import this package.  The copy
library never imports, links or calls it, and shares no code with it.

What it follows ("DejaVu: KV-Cache Streaming for Fast, Fault-Tolerant
Generative LLM Serving"):

* pack = gather of the non-contiguous K/V slices into one contiguous buffer
  (§3 DejaVuLib implementation, "Buffered copies", Fig 6, Fig 7a; Table 1
  gather);
* unpack = the scatter of such a buffer back into the same slices (Table 1
  scatter / stream_in);
* swap-out, layer streaming, decode-delta replication and restore are
  compositions of pack/unpack with plain byte copies (§3 microbatch swapping,
  Fig 9; layer-by-layer prompt streaming, Fig 7b; state replication and
  recovery, Fig 10); their oracle results are the same byte strings;
* the staging size is 2*B*S*H*D*P*N bytes for a full cache (KV-cache capacity
  page, "KV Cache 的容量计算").

parity: pinned for every function here (see ``tests/test_oracle_pins.py``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "dv_oracle.c"
_BUILD = _HERE / "_build"
_LIB_PATH = _BUILD / "liboracle.so"
_lib = None

_i32p = ctypes.POINTER(ctypes.c_int32)
_i64p = ctypes.POINTER(ctypes.c_int64)
_u8p = ctypes.POINTER(ctypes.c_uint8)


def build(src: Path = _SRC, out: Path = _LIB_PATH, extra_flags=()) -> Path:
    """Compile the oracle with gcc into a shared library."""
    out.parent.mkdir(parents=True, exist_ok=True)
    tmp = out.with_suffix(f".{os.getpid()}.tmp.so")
    cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-shared", "-fPIC", *extra_flags,
           str(src), "-o", str(tmp)]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _bind(lib):
    geo = [ctypes.c_int32] * 6 + [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, _i32p, _i32p]
    lib.oracle_check.argtypes = geo
    lib.oracle_check.restype = ctypes.c_int
    lib.oracle_staging_elems.argtypes = [ctypes.c_int32] * 5 + [_i32p, _i32p]
    lib.oracle_staging_elems.restype = ctypes.c_int64
    lib.oracle_pack.argtypes = [_u8p, _u8p] + geo + [_u8p]
    lib.oracle_pack.restype = ctypes.c_int64
    lib.oracle_unpack.argtypes = [_u8p, _u8p] + geo + [_u8p]
    lib.oracle_unpack.restype = ctypes.c_int64
    lib.oracle_source_of.argtypes = geo + [_i64p, ctypes.c_int64, _i64p, _i32p]
    lib.oracle_source_of.restype = ctypes.c_int64
    return lib


def load(path: Path | None = None):
    """Load (building first if needed) the oracle library."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(str(path)))
    if _lib is None:
        if not _LIB_PATH.exists() or _LIB_PATH.stat().st_mtime < _SRC.stat().st_mtime:
            build()
        _lib = _bind(ctypes.CDLL(str(_LIB_PATH)))
    return _lib


class Oracle:
    """Oracle bound to one compiled copy of ``dv_oracle.c`` (the default build,
    or a variant compiled by a test)."""

    def __init__(self, lib=None):
        self.lib = lib if lib is not None else load()

    # -- helpers ----------------------------------------------------------
    @staticmethod
    def _ranges(seq_start, seq_end):
        s = np.ascontiguousarray(seq_start, dtype=np.int32)
        e = np.ascontiguousarray(seq_end, dtype=np.int32)
        return s, e, s.ctypes.data_as(_i32p), e.ctypes.data_as(_i32p)

    @staticmethod
    def _geo(g):
        return (g.num_layers, g.batch, g.num_heads, g.head_dim, g.max_seq, g.elem_bytes,
                g.layer_elems)

    # -- API ----------------------------------------------------------------
    def check(self, g, l0, l1, seq_start, seq_end) -> int:
        s, e, sp, ep = self._ranges(seq_start, seq_end)
        return self.lib.oracle_check(*self._geo(g), l0, l1, sp, ep)

    def staging_bytes(self, g, l0, l1, seq_start, seq_end) -> int:
        s, e, sp, ep = self._ranges(seq_start, seq_end)
        return self.lib.oracle_staging_elems(g.batch, g.num_heads, g.head_dim, l0, l1, sp,
                                             ep) * g.elem_bytes

    def pack(self, g, k: np.ndarray, v: np.ndarray, l0, l1, seq_start, seq_end) -> np.ndarray:
        """Staging bytes gathered from cache byte arrays ``k`` and ``v``."""
        s, e, sp, ep = self._ranges(seq_start, seq_end)
        if self.check(g, l0, l1, s, e):
            raise ValueError("oracle: bad geometry or ranges")
        k = np.ascontiguousarray(k).view(np.uint8).reshape(-1)
        v = np.ascontiguousarray(v).view(np.uint8).reshape(-1)
        assert k.size >= g.tensor_bytes and v.size >= g.tensor_bytes
        out = np.empty(self.staging_bytes(g, l0, l1, s, e), dtype=np.uint8)
        n = self.lib.oracle_pack(k.ctypes.data_as(_u8p), v.ctypes.data_as(_u8p), *self._geo(g),
                                 l0, l1, sp, ep, out.ctypes.data_as(_u8p))
        assert n * g.elem_bytes == out.size
        return out

    def unpack(self, g, k: np.ndarray, v: np.ndarray, l0, l1, seq_start, seq_end,
               staging: np.ndarray) -> None:
        """Scatter ``staging`` into cache byte arrays ``k`` and ``v`` in place."""
        s, e, sp, ep = self._ranges(seq_start, seq_end)
        if self.check(g, l0, l1, s, e):
            raise ValueError("oracle: bad geometry or ranges")
        assert k.dtype == np.uint8 and v.dtype == np.uint8
        assert k.flags.c_contiguous and v.flags.c_contiguous
        assert k.size >= g.tensor_bytes and v.size >= g.tensor_bytes
        st = np.ascontiguousarray(staging).view(np.uint8).reshape(-1)
        if st.size < self.staging_bytes(g, l0, l1, s, e):
            raise ValueError("oracle: staging too small")
        self.lib.oracle_unpack(k.ctypes.data_as(_u8p), v.ctypes.data_as(_u8p), *self._geo(g),
                               l0, l1, sp, ep, st.ctypes.data_as(_u8p))

    def source_of(self, g, l0, l1, seq_start, seq_end, offsets):
        """For ascending staging element offsets: (kv, element index) of the
        cache element held there."""
        s, e, sp, ep = self._ranges(seq_start, seq_end)
        offs = np.ascontiguousarray(offsets, dtype=np.int64)
        idx = np.empty(offs.size, np.int64)
        kv = np.empty(offs.size, np.int32)
        n = self.lib.oracle_source_of(*self._geo(g), l0, l1, sp, ep,
                                      offs.ctypes.data_as(_i64p), offs.size,
                                      idx.ctypes.data_as(_i64p), kv.ctypes.data_as(_i32p))
        if n != offs.size:
            raise ValueError("oracle: offsets out of range or not ascending")
        return kv, idx

    # -- compositions (pages: swap, layer streaming, replication) ------------
    def swap_out(self, g, k, v, l0, l1, seq_start, seq_end) -> np.ndarray:
        """Bytes a swap-out leaves in host memory: the pack of the ranges."""
        return self.pack(g, k, v, l0, l1, seq_start, seq_end)

    def stream_layers(self, g, k, v, l0, l1, seq_start, seq_end) -> np.ndarray:
        """Host buffer after streaming layers l0..l1 one at a time: per-layer
        packs laid end to end."""
        parts = [self.pack(g, k, v, l, l + 1, seq_start, seq_end) for l in range(l0, l1)]
        return np.concatenate(parts) if parts else np.empty(0, np.uint8)

    def restore(self, g, records) -> tuple[np.ndarray, np.ndarray]:
        """A zeroed cache after unpacking replica records ``(l0, l1, s, e,
        bytes)`` in order (snapshot first, then deltas)."""
        k = np.zeros(g.tensor_bytes, np.uint8)
        v = np.zeros(g.tensor_bytes, np.uint8)
        for (l0, l1, s, e, data) in records:
            self.unpack(g, k, v, l0, l1, s, e, data)
        return k, v


_default = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default
