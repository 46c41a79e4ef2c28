"""ctypes binding of libdv (``include/dv.h``): argument marshalling only.

Every function here has the name of the C entry point it calls and does no
copy work of its own.  Buffers may be given as torch tensors (device or
pinned host; their ``data_ptr()`` and byte size are used) or as
``(address, nbytes)`` pairs.  Streams may be ``torch.cuda.Stream`` objects,
raw ``cudaStream_t`` integers, or ``None`` for torch's current stream.
A status other than DV_OK raises ``DvError`` with the library's message.
"""
from __future__ import annotations

import ctypes
import os
from pathlib import Path

import numpy as np

PKG = Path(__file__).resolve().parent
# DV_LIBRARY=checked loads the bounds-checked debugging build instead.
library_path = PKG / ("libdv_checked.so" if os.environ.get("DV_LIBRARY") == "checked"
                      else "libdv.so")

DV_MAX_BATCH = 1024
(DV_OK, DV_ERR_INVALID_ARG, DV_ERR_RANGE, DV_ERR_BUFFER_TOO_SMALL, DV_ERR_MISALIGNED,
 DV_ERR_CUDA, DV_ERR_TIMEOUT, DV_ERR_UNSUPPORTED) = range(8)
DV_VARIANT_AUTO, DV_VARIANT_FLAT, DV_VARIANT_TILE, DV_VARIANT_TOKEN = 0, 1, 2, 3

if not library_path.exists():
    raise ImportError(f"{library_path} is missing: build it with "
                      "`python kv_cache_streaming_gb300/build.py` (needs nvcc)")
lib = ctypes.CDLL(str(library_path))


class dv_cache(ctypes.Structure):
    _fields_ = [("num_layers", ctypes.c_int32), ("batch", ctypes.c_int32),
                ("num_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("max_seq", ctypes.c_int32), ("elem_bytes", ctypes.c_int32),
                ("layer_stride_elems", ctypes.c_int64),
                ("k_base", ctypes.c_void_p), ("v_base", ctypes.c_void_p)]


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_I32P = _P  # int32 host arrays, passed by address
_CP = ctypes.POINTER(dv_cache)
_RANGE = [_CP, _I32, _I32, _I32P, _I32P]


def _sig(name, args, res=ctypes.c_int):
    fn = getattr(lib, name)
    fn.argtypes = args
    fn.restype = res
    return fn


_abi = _sig("dv_abi_version", [], _I32)
_status_string = _sig("dv_status_string", [ctypes.c_int], ctypes.c_char_p)
_last_error = _sig("dv_last_error", [], ctypes.c_char_p)
_staging_bytes = _sig("dv_staging_bytes", _RANGE + [ctypes.POINTER(_SZ)])
_extent = _sig("dv_allocation_extent", [_P, ctypes.POINTER(_SZ)])
_debug_fault = _sig("dv_debug_fault", [ctypes.POINTER(ctypes.c_uint64)])
_host_alloc = _sig("dv_host_alloc", [_SZ, ctypes.POINTER(_P)])
_host_free = _sig("dv_host_free", [_P])
_pack = _sig("dv_kv_pack_variant", _RANGE + [_P, _SZ, _P, _I32])
_unpack = _sig("dv_kv_unpack_variant", _RANGE + [_P, _SZ, _P, _I32])
_swap_out = _sig("dv_swap_out", _RANGE + [_P, _SZ, _P, _SZ, _P])
_swap_in = _sig("dv_swap_in", _RANGE + [_P, _SZ, _P, _SZ, _P])
_swap_out_noalloc = _sig("dv_swap_out_noalloc", _RANGE + [_P, _SZ, _P])
_naive_gather = _sig("dv_naive_gather", _RANGE + [_P, _SZ, _P, ctypes.POINTER(_I64)])
_unpack_records = _sig("dv_kv_unpack_records", [_CP, _I32, _I32P, _I32P, _P, _SZ, _P])
DV_NOALLOC_STAGING_BYTES = 64 << 20
_streamer_create = _sig("dv_streamer_create", [ctypes.POINTER(_P), _P, _P, _SZ, _P, _P])
_stream_layer = _sig("dv_stream_layer", [_P, _CP, _I32, _I32P, _I32P, _P, _SZ, _I32])
_streamer_wait = _sig("dv_streamer_wait", [_P])
_streamer_destroy = _sig("dv_streamer_destroy", [_P], None)
_fetcher_create = _sig("dv_fetcher_create", [ctypes.POINTER(_P), _P, _P, _SZ, _P, _P])
_fetch_layer = _sig("dv_fetch_layer", [_P, _CP, _I32, _I32P, _I32P, _P, _SZ, _I32])
_fetcher_wait = _sig("dv_fetcher_wait", [_P])
_fetcher_destroy = _sig("dv_fetcher_destroy", [_P], None)
_replica_create = _sig("dv_replica_create", [ctypes.POINTER(_P), _P, _SZ, _I32])
_replica_append = _sig("dv_replica_append", [_P] + _RANGE + [_I64, _P, _SZ, _P])
_replica_append_streamed = _sig("dv_replica_append_streamed", [_P, _P] + _RANGE + [_I64])
_replica_restore = _sig("dv_replica_restore", [_P, _CP, _I64, _P, _SZ, _P])
_replica_restore_batched = _sig("dv_replica_restore_batched", [_P, _CP, _I64, _P, _SZ, _P])
_replica_restore_fetched = _sig("dv_replica_restore_fetched", [_P, _CP, _I64, _P])
_replica_restore_fetched_steps = _sig("dv_replica_restore_fetched_steps",
                                      [_P, _CP, _I64, _I64, _P])
_replica_truncate = _sig("dv_replica_truncate", [_P, _I64])
_replica_info = _sig("dv_replica_info", [_P, ctypes.POINTER(_I64), ctypes.POINTER(_SZ)])
_replica_destroy = _sig("dv_replica_destroy", [_P], None)
_swapper_create = _sig("dv_swapper_create", [ctypes.POINTER(_P), _CP, _CP, _P, _P, _P])
_swapper_acquire = _sig("dv_swapper_acquire", [_P, _P, ctypes.POINTER(_I32)])
_swapper_prefetch = _sig("dv_swapper_prefetch", [_P, _P])
_swapper_release = _sig("dv_swapper_release", [_P, _P, _I32, _I32, _I32P, _I32P, _I64])
_swapper_wait = _sig("dv_swapper_wait", [_P])
_swapper_destroy = _sig("dv_swapper_destroy", [_P], None)
_delta_streamer_create = _sig("dv_delta_streamer_create",
                              [ctypes.POINTER(_P), _P, _P, _P, _P, _SZ])
_delta_stream = _sig("dv_delta_stream", [_P, _CP, _I32, _I32, _I32P, _I32P, _I64])
_delta_streamer_join = _sig("dv_delta_streamer_join", [_P])
_delta_streamer_wait = _sig("dv_delta_streamer_wait", [_P])
_delta_streamer_destroy = _sig("dv_delta_streamer_destroy", [_P], None)


class DvError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_status_string(status).decode()}: {message}")
        self.status = status


def _check(status: int) -> None:
    if status != DV_OK:
        raise DvError(status, _last_error().decode(errors="replace"))


def dv_abi_version() -> int:
    return _abi()


# ---- marshalling helpers -------------------------------------------------------

def _buf(x, nbytes=None):
    """(address, nbytes) of a tensor, a pair, or None."""
    if x is None:
        return None, 0
    if isinstance(x, tuple):
        return int(x[0]), int(x[1] if nbytes is None else nbytes)
    if isinstance(x, HostBuffer):
        return x.ptr, int(x.nbytes if nbytes is None else nbytes)
    if hasattr(x, "data_ptr"):
        if hasattr(x, "is_contiguous") and not x.is_contiguous():
            raise TypeError("a tensor buffer must be contiguous (its bytes are one range)")
        n = x.numel() * x.element_size()
        return x.data_ptr(), int(n if nbytes is None else nbytes)
    raise TypeError(f"cannot use {type(x).__name__} as a buffer")


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _addr(a):
    """Address of a contiguous int32 numpy array's data (the cheapest route
    through ctypes; read-only arrays are copied first)."""
    try:
        return ctypes.addressof(ctypes.c_int32.from_buffer(a)), a
    except (TypeError, ValueError):
        a = a.copy()
        return ctypes.addressof(ctypes.c_int32.from_buffer(a)), a


def _ranges(seq_start, seq_end, batch):
    """int32 copies (or views) of the ranges and their addresses; the library
    reads exactly `batch` entries of each, so shorter arrays are refused."""
    s = np.ascontiguousarray(seq_start, dtype=np.int32).reshape(-1)
    e = np.ascontiguousarray(seq_end, dtype=np.int32).reshape(-1)
    if s.size != batch or e.size != batch:
        raise ValueError(f"seq_start / seq_end need {batch} entries (got {s.size}, {e.size})")
    sp, s = _addr(s)
    ep, e = _addr(e)
    return s, e, sp, ep


class Cache:
    """Geometry plus K/V base addresses of one cache (layout in ``dv.h``).

    ``k`` and ``v`` are device tensors (any dtype; only their addresses are
    used) or raw addresses.  ``layer_stride_elems`` 0 means layers are packed
    densely."""

    def __init__(self, num_layers, batch, num_heads, head_dim, max_seq, elem_bytes, k, v,
                 layer_stride_elems=0):
        for t in (k, v):
            if hasattr(t, "is_contiguous") and not t.is_contiguous():
                raise TypeError("K and V tensors must be contiguous (the layout is by address)")
        self.k, self.v = k, v  # keep the tensors alive
        kp = k.data_ptr() if hasattr(k, "data_ptr") else int(k)
        vp = v.data_ptr() if hasattr(v, "data_ptr") else int(v)
        self.c = dv_cache(num_layers, batch, num_heads, head_dim, max_seq, elem_bytes,
                          layer_stride_elems, kp, vp)
        self.ref = ctypes.byref(self.c)

    @classmethod
    def from_geometry(cls, g, k, v):
        return cls(g.num_layers, g.batch, g.num_heads, g.head_dim, g.max_seq, g.elem_bytes,
                   k, v, g.layer_stride_elems)

    @property
    def num_layers(self):
        return self.c.num_layers

    @property
    def batch(self):
        return self.c.batch


# ---- entry points --------------------------------------------------------------

def dv_debug_fault():
    """The first out-of-bounds access the checked build recorded (0: none), or
    None for the regular build.  Waits for the device and clears the record."""
    out = ctypes.c_uint64(0)
    st = _debug_fault(ctypes.byref(out))
    if st == DV_ERR_UNSUPPORTED:
        return None
    _check(st)
    return out.value


class HostBuffer:
    """Pinned, mapped host memory from ``dv_host_alloc`` (huge pages where the
    kernel gives them).  Pass it wherever a call takes pinned host memory, or
    view it as a uint8 CPU tensor with ``tensor()``; the memory is freed by
    ``close()`` or once neither the buffer nor a tensor over it is referenced."""

    def __init__(self, nbytes):
        p = _P()
        _check(_host_alloc(int(nbytes), ctypes.byref(p)))
        self.ptr, self.nbytes = p.value, int(nbytes)

    def tensor(self):
        import torch
        if not self.ptr:
            raise ValueError("the buffer is closed")
        arr = (ctypes.c_uint8 * self.nbytes).from_address(self.ptr)
        arr._owner = self  # the tensor keeps the buffer alive
        return torch.frombuffer(arr, dtype=torch.uint8)

    def close(self):
        if self.ptr:
            ptr, self.ptr = self.ptr, None
            _check(_host_free(ptr))

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def dv_host_alloc(nbytes) -> HostBuffer:
    return HostBuffer(nbytes)


def dv_host_free(buf: HostBuffer) -> None:
    buf.close()


def host_empty(nbytes):
    """A uint8 CPU tensor of ``nbytes`` over pinned, mapped host memory from
    ``dv_host_alloc`` (zeroed)."""
    return HostBuffer(nbytes).tensor()


def dv_allocation_extent(ptr):
    """Bytes from ``ptr`` (tensor or address) to the end of its CUDA
    allocation, or None when the driver cannot tell."""
    addr = ptr.data_ptr() if hasattr(ptr, "data_ptr") else int(ptr)
    out = _SZ(0)
    st = _extent(addr, ctypes.byref(out))
    if st == DV_ERR_UNSUPPORTED:
        return None
    _check(st)
    return out.value


def dv_staging_bytes(cache: Cache, l0, l1, seq_start, seq_end) -> int:
    s, e, sp, ep = _ranges(seq_start, seq_end, cache.c.batch)
    out = _SZ(0)
    _check(_staging_bytes(cache.ref, l0, l1, sp, ep, ctypes.byref(out)))
    return out.value


def dv_kv_pack(cache: Cache, l0, l1, seq_start, seq_end, dst, stream=None,
               variant=DV_VARIANT_AUTO, dst_bytes=None) -> None:
    s, e, sp, ep = _ranges(seq_start, seq_end, cache.c.batch)
    d, n = _buf(dst, dst_bytes)
    _check(_pack(cache.ref, l0, l1, sp, ep, d, n, _stream(stream), variant))


def dv_kv_unpack(cache: Cache, l0, l1, seq_start, seq_end, src, stream=None,
                 variant=DV_VARIANT_AUTO, src_bytes=None) -> None:
    s, e, sp, ep = _ranges(seq_start, seq_end, cache.c.batch)
    d, n = _buf(src, src_bytes)
    _check(_unpack(cache.ref, l0, l1, sp, ep, d, n, _stream(stream), variant))


def _record_tables(records, batch):
    """int32 arrays of a record list [(l0, l1, seq_start, seq_end), ...]: the
    layer pairs, and per record the starts then the ends."""
    n = len(records)
    layers = np.empty(2 * n, np.int32)
    ranges = np.empty(2 * batch * n, np.int32)
    for i, (l0, l1, s, e) in enumerate(records):
        s = np.asarray(s, dtype=np.int32).reshape(-1)
        e = np.asarray(e, dtype=np.int32).reshape(-1)
        if s.size != batch or e.size != batch:
            raise ValueError(f"record {i}: seq_start / seq_end need {batch} entries")
        layers[2 * i:2 * i + 2] = (l0, l1)
        ranges[2 * batch * i:2 * batch * i + batch] = s
        ranges[2 * batch * i + batch:2 * batch * (i + 1)] = e
    return layers, ranges


def dv_kv_unpack_records(cache: Cache, records, src, stream=None, src_bytes=None) -> None:
    """Unpacks log records [(l0, l1, seq_start, seq_end), ...] lying back to
    back in ``src`` (device or pinned host memory), as dv_kv_unpack of each in
    order."""
    d, n = _buf(src, src_bytes)
    if not records:
        _check(_unpack_records(cache.ref, 0, None, None, d, n, _stream(stream)))
        return
    layers, ranges = _record_tables(records, cache.c.batch)
    lp, layers = _addr(layers)
    rp, ranges = _addr(ranges)
    _check(_unpack_records(cache.ref, len(records), lp, rp, d, n, _stream(stream)))


def dv_naive_gather(cache: Cache, l0, l1, seq_start, seq_end, dst, stream=None,
                    dst_bytes=None) -> int:
    """The per-region copy baseline; returns the number of copies enqueued."""
    s, e, sp, ep = _ranges(seq_start, seq_end, cache.c.batch)
    d, n = _buf(dst, dst_bytes)
    calls = _I64(0)
    _check(_naive_gather(cache.ref, l0, l1, sp, ep, d, n, _stream(stream), ctypes.byref(calls)))
    return calls.value


def dv_swap_out(cache: Cache, l0, l1, seq_start, seq_end, host_dst, staging=None,
                stream=None) -> None:
    s, e, sp, ep = _ranges(seq_start, seq_end, cache.c.batch)
    h, hn = _buf(host_dst)
    st, sn = _buf(staging)
    _check(_swap_out(cache.ref, l0, l1, sp, ep, h, hn, st, sn, _stream(stream)))


def dv_swap_in(cache: Cache, l0, l1, seq_start, seq_end, host_src, staging=None,
               stream=None) -> None:
    s, e, sp, ep = _ranges(seq_start, seq_end, cache.c.batch)
    h, hn = _buf(host_src)
    st, sn = _buf(staging)
    _check(_swap_in(cache.ref, l0, l1, sp, ep, h, hn, st, sn, _stream(stream)))


def dv_swap_out_noalloc(cache: Cache, l0, l1, seq_start, seq_end, host_dst,
                        stream=None) -> None:
    """dv_swap_out through libdv's built-in 64 MiB staging buffer (no
    allocation by the caller); see dv.h for the limits."""
    s, e, sp, ep = _ranges(seq_start, seq_end, cache.c.batch)
    h, hn = _buf(host_dst)
    _check(_swap_out_noalloc(cache.ref, l0, l1, sp, ep, h, hn, _stream(stream)))


class Streamer:
    """Handle of ``dv_streamer`` (two slots, pack and copy streams)."""

    def __init__(self, slot0, slot1, pack_stream=None, copy_stream=None):
        a0, n0 = _buf(slot0)
        a1, n1 = _buf(slot1)
        self._keep = (slot0, slot1, pack_stream, copy_stream)
        h = _P()
        _check(_streamer_create(ctypes.byref(h), a0, a1, min(n0, n1), _stream(pack_stream),
                                _stream(copy_stream)))
        self.h = h

    def stream_layer(self, cache: Cache, layer, seq_start, seq_end, host_dst, l0=0):
        s, e, sp, ep = _ranges(seq_start, seq_end, cache.c.batch)
        d, n = _buf(host_dst)
        _check(_stream_layer(self.h, cache.ref, layer, sp, ep, d, n, l0))

    def wait(self):
        _check(_streamer_wait(self.h))

    def close(self):
        if self.h:
            _streamer_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def dv_streamer_create(slot0, slot1, pack_stream=None, copy_stream=None) -> Streamer:
    return Streamer(slot0, slot1, pack_stream, copy_stream)


def dv_stream_layer(streamer: Streamer, cache: Cache, layer, seq_start, seq_end, host_dst,
                    l0=0) -> None:
    streamer.stream_layer(cache, layer, seq_start, seq_end, host_dst, l0)


def dv_streamer_wait(streamer: Streamer) -> None:
    streamer.wait()


def dv_streamer_destroy(streamer: Streamer) -> None:
    streamer.close()


class Fetcher:
    """Handle of ``dv_fetcher`` (two slots, copy and unpack streams)."""

    def __init__(self, slot0, slot1, copy_stream=None, unpack_stream=None):
        a0, n0 = _buf(slot0)
        a1, n1 = _buf(slot1)
        self._keep = (slot0, slot1, copy_stream, unpack_stream)
        h = _P()
        _check(_fetcher_create(ctypes.byref(h), a0, a1, min(n0, n1), _stream(copy_stream),
                               _stream(unpack_stream)))
        self.h = h

    def fetch_layer(self, cache: Cache, layer, seq_start, seq_end, host_src, l0=0):
        s, e, sp, ep = _ranges(seq_start, seq_end, cache.c.batch)
        d, n = _buf(host_src)
        _check(_fetch_layer(self.h, cache.ref, layer, sp, ep, d, n, l0))

    def wait(self):
        _check(_fetcher_wait(self.h))

    def close(self):
        if self.h:
            _fetcher_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def dv_fetcher_create(slot0, slot1, copy_stream=None, unpack_stream=None) -> Fetcher:
    return Fetcher(slot0, slot1, copy_stream, unpack_stream)


def dv_fetch_layer(fetcher: Fetcher, cache: Cache, layer, seq_start, seq_end, host_src,
                   l0=0) -> None:
    fetcher.fetch_layer(cache, layer, seq_start, seq_end, host_src, l0)


def dv_fetcher_wait(fetcher: Fetcher) -> None:
    fetcher.wait()


def dv_fetcher_destroy(fetcher: Fetcher) -> None:
    fetcher.close()


class Replica:
    """Handle of ``dv_replica``: a record log in a pinned host arena."""

    def __init__(self, host_arena, batch):
        a, n = _buf(host_arena)
        self._keep = host_arena
        h = _P()
        _check(_replica_create(ctypes.byref(h), a, n, batch))
        self.h = h

    def append(self, cache: Cache, l0, l1, seq_start, seq_end, step, staging=None, stream=None):
        s, e, sp, ep = _ranges(seq_start, seq_end, cache.c.batch)
        st, sn = _buf(staging)
        _check(_replica_append(self.h, cache.ref, l0, l1, sp, ep, step, st, sn, _stream(stream)))

    def append_streamed(self, streamer: "Streamer", cache: Cache, l0, l1, seq_start, seq_end,
                        step):
        s, e, sp, ep = _ranges(seq_start, seq_end, cache.c.batch)
        _check(_replica_append_streamed(self.h, streamer.h, cache.ref, l0, l1, sp, ep, step))

    def restore(self, cache: Cache, upto_step=-1, staging=None, stream=None):
        st, sn = _buf(staging)
        _check(_replica_restore(self.h, cache.ref, upto_step, st, sn, _stream(stream)))

    def restore_batched(self, cache: Cache, upto_step=-1, staging=None, stream=None):
        st, sn = _buf(staging)
        _check(_replica_restore_batched(self.h, cache.ref, upto_step, st, sn, _stream(stream)))

    def restore_fetched(self, cache: Cache, fetcher: "Fetcher", upto_step=-1, from_step=None):
        if from_step is None:
            _check(_replica_restore_fetched(self.h, cache.ref, upto_step, fetcher.h))
        else:
            _check(_replica_restore_fetched_steps(self.h, cache.ref, from_step, upto_step,
                                                  fetcher.h))

    def truncate(self, step):
        _check(_replica_truncate(self.h, step))

    def info(self):
        n = _I64(0)
        b = _SZ(0)
        _check(_replica_info(self.h, ctypes.byref(n), ctypes.byref(b)))
        return n.value, b.value

    def close(self):
        if self.h:
            _replica_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def dv_replica_create(host_arena, batch) -> Replica:
    return Replica(host_arena, batch)


def dv_replica_append(replica: Replica, cache: Cache, l0, l1, seq_start, seq_end, step,
                      staging=None, stream=None) -> None:
    replica.append(cache, l0, l1, seq_start, seq_end, step, staging, stream)


def dv_replica_append_streamed(replica: Replica, streamer: Streamer, cache: Cache, l0, l1,
                               seq_start, seq_end, step) -> None:
    replica.append_streamed(streamer, cache, l0, l1, seq_start, seq_end, step)


def dv_replica_restore(replica: Replica, cache: Cache, upto_step=-1, staging=None,
                       stream=None) -> None:
    replica.restore(cache, upto_step, staging, stream)


def dv_replica_restore_batched(replica: Replica, cache: Cache, upto_step=-1, staging=None,
                               stream=None) -> None:
    replica.restore_batched(cache, upto_step, staging, stream)


def dv_replica_restore_fetched(replica: Replica, cache: Cache, fetcher: Fetcher,
                               upto_step=-1) -> None:
    replica.restore_fetched(cache, fetcher, upto_step)


def dv_replica_restore_fetched_steps(replica: Replica, cache: Cache, from_step, upto_step,
                                     fetcher: Fetcher) -> None:
    replica.restore_fetched(cache, fetcher, upto_step, from_step)


def dv_replica_truncate(replica: Replica, step) -> None:
    replica.truncate(step)


def dv_replica_info(replica: Replica):
    return replica.info()


def dv_replica_destroy(replica: Replica) -> None:
    replica.close()


class Swapper:
    """Handle of ``dv_swapper``: microbatches through two device caches."""

    def __init__(self, slot0: Cache, slot1: Cache, fetcher: Fetcher, compute_stream=None,
                 swap_stream=None):
        self._keep = (slot0, slot1, fetcher, compute_stream, swap_stream)
        self.slots = (slot0, slot1)
        h = _P()
        _check(_swapper_create(ctypes.byref(h), slot0.ref, slot1.ref, fetcher.h,
                               _stream(compute_stream), _stream(swap_stream)))
        self.h = h

    def acquire(self, mb: Replica) -> int:
        """The cache (0 or 1) that holds microbatch ``mb`` for its next step."""
        slot = _I32(-1)
        _check(_swapper_acquire(self.h, mb.h, ctypes.byref(slot)))
        return slot.value

    def prefetch(self, mb: Replica) -> None:
        _check(_swapper_prefetch(self.h, mb.h))

    def release(self, mb: Replica, l0, l1, seq_start, seq_end, step) -> None:
        s, e, sp, ep = _ranges(seq_start, seq_end, self.slots[0].c.batch)
        _check(_swapper_release(self.h, mb.h, l0, l1, sp, ep, step))

    def wait(self):
        _check(_swapper_wait(self.h))

    def close(self):
        if self.h:
            _swapper_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def dv_swapper_create(slot0, slot1, fetcher, compute_stream=None, swap_stream=None) -> Swapper:
    return Swapper(slot0, slot1, fetcher, compute_stream, swap_stream)


def dv_swapper_acquire(sw: Swapper, mb: Replica) -> int:
    return sw.acquire(mb)


def dv_swapper_prefetch(sw: Swapper, mb: Replica) -> None:
    sw.prefetch(mb)


def dv_swapper_release(sw: Swapper, mb: Replica, l0, l1, seq_start, seq_end, step) -> None:
    sw.release(mb, l0, l1, seq_start, seq_end, step)


def dv_swapper_wait(sw: Swapper) -> None:
    sw.wait()


def dv_swapper_destroy(sw: Swapper) -> None:
    sw.close()


class DeltaStreamer:
    """Handle of ``dv_delta_streamer``: decode deltas streamed to a replica on
    a side stream."""

    def __init__(self, replica: Replica, compute_stream=None, side_stream=None, staging=None):
        st, sn = _buf(staging)
        self._keep = (replica, compute_stream, side_stream, staging)
        h = _P()
        _check(_delta_streamer_create(ctypes.byref(h), replica.h, _stream(compute_stream),
                                      _stream(side_stream), st, sn))
        self.h = h

    def stream(self, cache: Cache, l0, l1, seq_start, seq_end, step) -> None:
        s, e, sp, ep = _ranges(seq_start, seq_end, cache.c.batch)
        _check(_delta_stream(self.h, cache.ref, l0, l1, sp, ep, step))

    def join(self):
        _check(_delta_streamer_join(self.h))

    def wait(self):
        _check(_delta_streamer_wait(self.h))

    def close(self):
        if self.h:
            _delta_streamer_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def dv_delta_streamer_create(replica, compute_stream=None, side_stream=None,
                             staging=None) -> DeltaStreamer:
    return DeltaStreamer(replica, compute_stream, side_stream, staging)


def dv_delta_stream(ds: DeltaStreamer, cache: Cache, l0, l1, seq_start, seq_end, step) -> None:
    ds.stream(cache, l0, l1, seq_start, seq_end, step)


def dv_delta_streamer_join(ds: DeltaStreamer) -> None:
    ds.join()


def dv_delta_streamer_wait(ds: DeltaStreamer) -> None:
    ds.wait()


def dv_delta_streamer_destroy(ds: DeltaStreamer) -> None:
    ds.close()
