"""Pinned host memory from dv_host_alloc: the host side of a swap, fused and
staged, against the oracle; a replica arena; alignment, zero fill, sizes
around the huge-page size, and the errors of dv_host_free."""
import numpy as np
import pytest
import torch

import kv_cache_streaming_gb300 as dv
import oracle
from synth.configs import Geometry
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu
ORC = oracle.default()


def huge_page_bytes():
    try:
        with open("/sys/kernel/mm/transparent_hugepage/hpage_pmd_size") as f:
            return int(f.read())
    except (OSError, ValueError):
        return 2 << 20


@pytest.mark.parametrize("size", ["1", "hp-1", "hp+1", "hp+12345"])
def test_alloc_alignment_zero_fill_and_free(size):
    hp = huge_page_bytes()
    n = {"1": 1, "hp-1": hp - 1, "hp+1": hp + 1, "hp+12345": hp + 12345}[size]
    buf = dv.HostBuffer(n)
    assert buf.ptr % hp == 0
    t = buf.tensor()
    assert t.numel() == n and t.data_ptr() == buf.ptr
    assert not t[:min(n, 1 << 20)].any() and not t[-min(n, 1 << 20):].any()
    t[-1] = 7                                          # the last byte is writable
    assert int(t[-1]) == 7
    ptr = buf.ptr
    del t
    buf.close()
    buf.close()                                        # a second close does nothing
    with pytest.raises(dv.DvError) as ei:              # the library no longer knows it
        dv.dv._check(dv.dv._host_free(ptr))
    assert ei.value.status == dv.DV_ERR_INVALID_ARG


def test_alloc_refuses_zero_bytes():
    with pytest.raises(dv.DvError) as ei:
        dv.HostBuffer(0)
    assert ei.value.status == dv.DV_ERR_INVALID_ARG


@pytest.mark.parametrize("staged", [False, True])
def test_swap_through_host_alloc_memory(staged):
    g = Geometry("hswap", 4, 3, 3, 128, 200, 2, "bf16")
    rng = np.random.default_rng(21)
    kh, vh = H.host_cache(g, 22)
    cache = H.device_cache(g, fill=(kh, vh))
    s = np.zeros(g.batch, np.int32)
    e = rng.integers(1, g.max_seq + 1, size=g.batch).astype(np.int32)
    n = ORC.staging_bytes(g, 0, g.num_layers, s, e)
    staging = H.device_bytes(2 * (n // g.num_layers) + 16) if staged else None
    host = dv.HostBuffer(n)
    dv.dv_swap_out(cache, 0, g.num_layers, s, e, host, staging=staging)
    torch.cuda.synchronize()
    want = ORC.swap_out(g, kh, vh, 0, g.num_layers, s, e)
    assert np.array_equal(host.tensor().numpy(), want)
    fresh = H.device_cache(g, fill="zero")
    dv.dv_swap_in(fresh, 0, g.num_layers, s, e, host, staging=staging)
    kw, vw = np.zeros_like(kh), np.zeros_like(vh)
    ORC.unpack(g, kw, vw, 0, g.num_layers, s, e, want)
    assert np.array_equal(H.to_np(fresh.k), kw) and np.array_equal(H.to_np(fresh.v), vw)
    host.close()


def test_replica_in_host_alloc_memory():
    g = Geometry("hrep", 3, 4, 2, 128, 64, 2, "fp16")
    kh, vh = H.host_cache(g, 23)
    cache = H.device_cache(g, fill=(kh, vh))
    zero = np.zeros(g.batch, np.int32)
    len0 = np.array([9, 64, 0, 31], np.int32)
    e1 = np.minimum(len0 + 1, g.max_seq).astype(np.int32)
    records = [(0, g.num_layers, zero, len0), (0, g.num_layers, len0, e1)]
    arena = dv.HostBuffer(sum(ORC.staging_bytes(g, *r) for r in records))
    rep = dv.Replica(arena, g.batch)                   # the buffer itself, no tensor
    for k, r in enumerate(records):
        rep.append(cache, *r, step=k)
    z = H.device_cache(g, fill="zero")
    rep.restore_batched(z)
    kw, vw = ORC.restore(g, [(*r, ORC.pack(g, kh, vh, *r)) for r in records])
    assert np.array_equal(H.to_np(z.k), kw) and np.array_equal(H.to_np(z.v), vw)
    rep.close()
    arena.close()


def test_alloc_and_free_from_many_threads():
    """Eight threads allocate, write, check and free buffers of their own at
    once: every call succeeds and no two live buffers overlap."""
    import threading
    torch.cuda.synchronize()
    errors, spans, lock = [], [], threading.Lock()

    def work(i):
        try:
            for r in range(6):
                n = (i + 1) * 4096 + r * 16
                buf = dv.HostBuffer(n)
                with lock:
                    spans.append((buf.ptr, buf.ptr + n, True))
                t = buf.tensor()
                t.fill_(i)
                assert int(t.sum()) == i * n
                with lock:
                    spans.remove((buf.ptr, buf.ptr + n, True))
                del t
                buf.close()
        except Exception as e:  # noqa: BLE001 - reported below
            errors.append(repr(e))

    def check_overlap():
        with lock:
            live = sorted(spans)
        for (a0, a1, _), (b0, b1, _) in zip(live, live[1:]):
            assert a1 <= b0

    threads = [threading.Thread(target=work, args=(i,)) for i in range(8)]
    for th in threads:
        th.start()
    for _ in range(20):
        check_overlap()
    for th in threads:
        th.join()
    assert not errors, errors
