"""The C ABI without a GPU: the library loads, exports what dv.h declares,
and its host-side planning and validation behave (CPU)."""
import re
from pathlib import Path

import numpy as np
import pytest

import kv_cache_streaming_gb300 as dv  # noqa: E402
import oracle  # noqa: E402
from synth.configs import Geometry, GEOMETRIES  # noqa: E402
from tests import oracle_pins as P  # noqa: E402

HEADER = Path(__file__).resolve().parent.parent / "include" / "dv.h"


def declared_functions():
    text = HEADER.read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dv_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported():
    names = declared_functions()
    assert len(names) >= 20
    for name in names:
        assert hasattr(dv.lib, name), name


def test_only_the_c_abi_is_exported():
    """The library's dynamic symbol table holds the functions of dv.h and nothing
    else (no C++ internals, no statically linked CUDA runtime)."""
    import shutil
    import subprocess
    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("nm not available")
    out = subprocess.run([nm, "-D", "--defined-only", str(dv.library_path)],
                         capture_output=True, text=True, check=True).stdout
    exported = sorted({line.split()[-1] for line in out.splitlines()
                       if len(line.split()) >= 3 and line.split()[1] in "TtWwDdBbRrVv"})
    assert exported == declared_functions(), set(exported) ^ set(declared_functions())


def test_abi_version():
    assert dv.dv_abi_version() == 1


def _cache(g):
    # addresses are never dereferenced by the host-only calls below
    return dv.Cache.from_geometry(g, 0x1000, 0x2000)


def test_staging_bytes_matches_oracle():
    orc = oracle.default()
    rng = np.random.default_rng(4)
    for g in GEOMETRIES + P.READING_GEOMS:
        for _ in range(5):
            s, e = P.random_ranges(g, rng)
            l0 = int(rng.integers(0, g.num_layers + 1))
            l1 = int(rng.integers(l0, g.num_layers + 1))
            assert dv.dv_staging_bytes(_cache(g), l0, l1, s, e) == orc.staging_bytes(g, l0, l1, s, e)


def test_full_cache_size_is_the_capacity_formula():
    for g in GEOMETRIES:
        s = np.zeros(g.batch, np.int32)
        e = np.full(g.batch, g.max_seq, np.int32)
        want = 2 * g.batch * g.max_seq * g.num_heads * g.head_dim * g.elem_bytes * g.num_layers
        assert dv.dv_staging_bytes(_cache(g), 0, g.num_layers, s, e) == want


def _status(fn):
    with pytest.raises(dv.DvError) as ei:
        fn()
    return ei.value.status


def test_validation_errors():
    g = Geometry("v", 2, 2, 2, 64, 16, 2, "raw")
    c = _cache(g)
    ok_s, ok_e = np.zeros(2, np.int32), np.full(2, 4, np.int32)
    st = lambda f: _status(f)  # noqa: E731
    assert st(lambda: dv.dv_staging_bytes(c, 0, 3, ok_s, ok_e)) == dv.DV_ERR_RANGE
    assert st(lambda: dv.dv_staging_bytes(c, 2, 1, ok_s, ok_e)) == dv.DV_ERR_RANGE
    assert st(lambda: dv.dv_staging_bytes(c, 0, 2, [5, 0], [4, 4])) == dv.DV_ERR_RANGE
    assert st(lambda: dv.dv_staging_bytes(c, 0, 2, [0, 0], [17, 4])) == dv.DV_ERR_RANGE
    assert st(lambda: dv.dv_staging_bytes(c, 0, 2, [-1, 0], [3, 4])) == dv.DV_ERR_RANGE
    bad = dv.Cache(2, 2, 2, 60, 16, 2, 0x1000, 0x2000)  # head_dim not a multiple of 8
    assert st(lambda: dv.dv_staging_bytes(bad, 0, 2, ok_s, ok_e)) == dv.DV_ERR_UNSUPPORTED
    bad = dv.Cache(2, 2, 2, 64, 16, 3, 0x1000, 0x2000)
    assert st(lambda: dv.dv_staging_bytes(bad, 0, 2, ok_s, ok_e)) == dv.DV_ERR_INVALID_ARG
    bad = dv.Cache(2, 2, 2, 64, 16, 2, 0x1000, 0x2000, layer_stride_elems=100)
    assert st(lambda: dv.dv_staging_bytes(bad, 0, 2, ok_s, ok_e)) == dv.DV_ERR_INVALID_ARG
    bad = dv.Cache(2, 2, 2, 64, 16, 2, 0x1000, 0x2000, layer_stride_elems=2 * 2 * 64 * 16 + 4)
    assert st(lambda: dv.dv_staging_bytes(bad, 0, 2, ok_s, ok_e)) == dv.DV_ERR_MISALIGNED
    big = dv.Cache(1, dv.DV_MAX_BATCH + 1, 1, 8, 4, 2, 0x1000, 0x2000)
    n = dv.DV_MAX_BATCH + 1
    assert st(lambda: dv.dv_staging_bytes(big, 0, 1, np.zeros(n), np.ones(n))) == \
        dv.DV_ERR_UNSUPPORTED
    need = dv.dv_staging_bytes(c, 0, 2, ok_s, ok_e)
    # too-small destination / source is caught before any pointer is touched
    assert st(lambda: dv.dv_kv_pack(c, 0, 2, ok_s, ok_e, (0x3000, need - 16), stream=0)) == \
        dv.DV_ERR_BUFFER_TOO_SMALL
    assert st(lambda: dv.dv_kv_unpack(c, 0, 2, ok_s, ok_e, (0x3000, need - 16), stream=0)) == \
        dv.DV_ERR_BUFFER_TOO_SMALL
    assert st(lambda: dv.dv_kv_pack(c, 0, 2, ok_s, ok_e, (0x3000, need), stream=0,
                                    variant=7)) == dv.DV_ERR_INVALID_ARG
    # an empty pack enqueues nothing and needs no buffer
    dv.dv_kv_pack(c, 1, 1, ok_s, ok_e, None, stream=0)
    dv.dv_kv_pack(c, 0, 2, ok_s, ok_s, None, stream=0)


def test_slab_beyond_32_bit_chunk_indexing_is_refused():
    """One (layer, K|V) slab must stay under 2^31 16-byte chunks (32 GiB):
    larger ranges are refused on the host, before any launch."""
    g = Geometry("huge", 1, 1024, 128, 128, 1 << 17, 2, "fp16")
    c = dv.Cache.from_geometry(g, 0x1000, 0x2000)
    s = np.zeros(g.batch, np.int32)
    e = np.full(g.batch, g.max_seq, np.int32)  # H * T * C = 128 * 2^27 * 16 = 2^38 chunks
    assert _status(lambda: dv.dv_staging_bytes(c, 0, 1, s, e)) == dv.DV_ERR_UNSUPPORTED
    e[:] = 1  # a one-token slab is fine
    assert dv.dv_staging_bytes(c, 0, 1, s, e) == 2 * 1024 * 128 * 128 * 2


def test_binding_refuses_ranges_of_the_wrong_length():
    """The library reads `batch` entries of each range array: the binding
    refuses shorter or longer arrays before calling it."""
    g = Geometry("v", 2, 4, 2, 64, 16, 2, "raw")
    c = _cache(g)
    with pytest.raises(ValueError):
        dv.dv_staging_bytes(c, 0, 2, [0, 0], [1, 1])
    with pytest.raises(ValueError):
        dv.dv_kv_pack(c, 0, 2, np.zeros(5), np.ones(5), (0x3000, 1 << 20), stream=0)
    ro = np.zeros(4, np.int32)
    ro.setflags(write=False)  # read-only arrays are accepted (copied)
    assert dv.dv_staging_bytes(c, 0, 2, ro, ro + 3) == 2 * 2 * 2 * 64 * 2 * 12


def test_binding_refuses_a_non_contiguous_tensor_buffer():
    """A buffer is one byte range: a strided view is refused before the
    library sees its address."""
    import torch
    g = Geometry("v", 2, 4, 2, 64, 16, 2, "raw")
    c = _cache(g)
    s = np.zeros(4, np.int32)
    strided = torch.zeros(64, 64, dtype=torch.uint8).t()
    with pytest.raises(TypeError):
        dv.dv_kv_pack(c, 0, 2, s, s + 1, strided, stream=0)
    with pytest.raises(TypeError):
        dv.Cache.from_geometry(g, strided, torch.zeros(16))


def test_last_error_is_per_thread():
    """Threads that fail validation at the same time each read their own
    message (the library's only mutable global state is that thread-local
    string)."""
    import threading
    g = Geometry("thr", 2, 2, 2, 64, 32, 2, "fp16")
    c = _cache(g)
    ok = np.zeros(2, np.int32), np.full(2, 32, np.int32)
    barrier = threading.Barrier(8)
    seen = {}

    def worker(i):
        barrier.wait()
        for _ in range(200):
            if i % 2:  # a layer range past the cache
                with pytest.raises(dv.DvError) as ei:
                    dv.dv_staging_bytes(c, 0, 3 + i, *ok)
                want = f"layer range [0,{3 + i})"
            else:       # a token range past max_seq
                e = np.array([32, 40 + i], np.int32)
                with pytest.raises(dv.DvError) as ei:
                    dv.dv_staging_bytes(c, 0, 2, ok[0], e)
                want = f"[0,{40 + i})"
            if want not in str(ei.value):
                seen[i] = str(ei.value)
                return
        seen[i] = None

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(8)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert all(v is None for v in seen.values()) and len(seen) == 8, seen


def test_package_without_the_library_refuses_to_import(tmp_path):
    """No CPU fallback: a copy of the package without libdv.so fails at import
    with a message that names the missing library and the build step."""
    import shutil
    import subprocess
    import sys
    pkg = Path(dv.__file__).resolve().parent
    dst = tmp_path / pkg.name
    dst.mkdir()
    for name in ("__init__.py", "dv.py"):
        shutil.copy(pkg / name, dst / name)
    r = subprocess.run([sys.executable, "-c", f"import {pkg.name}"], cwd=str(tmp_path),
                       capture_output=True, text=True, timeout=120,
                       env={k: v for k, v in __import__("os").environ.items()
                            if k not in ("PYTHONPATH", "DV_LIBRARY")})
    assert r.returncode != 0
    assert "ImportError" in r.stderr and "libdv.so is missing" in r.stderr
    assert "build.py" in r.stderr
