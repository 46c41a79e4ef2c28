"""Parity of the CUDA path with the oracle, byte for byte, on seeded inputs
small enough for the oracle (several tiles, ragged tails, empty ranges)."""
import zlib

import numpy as np
import pytest
import torch

import kv_cache_streaming_gb300 as dv
import oracle
import synth
from synth.configs import Geometry, TINY, seed_of, tiny_ranges
from tests import gpu_helpers as H
from tests import oracle_pins as P

pytestmark = pytest.mark.gpu
ORC = oracle.default()
VARIANTS = [dv.DV_VARIANT_AUTO, dv.DV_VARIANT_FLAT, dv.DV_VARIANT_TILE]

GEOMS = [
    Geometry("c16", 3, 5, 3, 128, 300, 2, "fp16"),      # C = 16, 32-token tiles
    Geometry("c8", 2, 4, 5, 64, 200, 2, "bf16"),        # C = 8, 64-token tiles
    Geometry("c12", 2, 3, 2, 96, 100, 2, "fp16"),       # C = 12, generic kernels
    Geometry("p1", 2, 3, 2, 128, 64, 1, "raw"),         # 1-byte elements, x = 16
    Geometry("p4", 2, 3, 2, 64, 64, 4, "fp32"),         # 4-byte elements, x = 4
    Geometry("pad", 3, 2, 2, 128, 50, 2, "fp16", layer_stride_elems=2 * 2 * 128 * 50 + 64),
    Geometry("b40", 1, 40, 2, 64, 32, 2, "fp16"),       # batch > 32: 1024-entry tables
    Geometry("b1024", 2, 1024, 1, 64, 24, 2, "fp16"),   # the largest batch the ABI takes
    Geometry("c1", 2, 3, 2, 8, 70, 2, "fp16"),          # C = 1: one chunk per token
    Geometry("c5", 2, 3, 2, 40, 90, 2, "fp16"),         # odd C
    Geometry("c64", 2, 2, 2, 512, 40, 2, "fp16"),       # the largest C the tile kernel takes
    Geometry("c128", 1, 2, 2, 1024, 20, 2, "fp16"),     # beyond it: flat kernel only
    Geometry("s1", 2, 3, 2, 64, 1, 2, "fp16"),          # max_seq 1: a K token is contiguous
    Geometry("b1", 2, 1, 3, 128, 64, 2, "bf16"),        # batch 1
]


def range_sets(g, rng):
    B, S = g.batch, g.max_seq
    out = [("full", np.zeros(B, np.int32), np.full(B, S, np.int32)),
           ("empty", np.zeros(B, np.int32), np.zeros(B, np.int32))]
    pos = rng.integers(0, S, size=B).astype(np.int32)
    e = pos + 1
    e[::3] = pos[::3]  # some finished sequences
    out.append(("decode", pos, e.astype(np.int32)))
    n = min(3, S)  # a few equal-length ranges (multi-token deltas)
    pos = rng.integers(0, S - n + 1, size=B).astype(np.int32)
    e = pos + n
    e[1::3] = pos[1::3]
    out.append(("multi", pos, e.astype(np.int32)))
    for i in range(3):
        s, e = P.random_ranges(g, rng)
        out.append((f"rand{i}", s, e))
    return out


def variants_for(s, e, g=None):
    lens = (np.asarray(e) - np.asarray(s))
    one_token = lens.max() > 0 and len(set(lens[lens > 0].tolist())) == 1  # equal lengths
    base = VARIANTS
    if g is not None and g.head_dim * g.elem_bytes // 16 > 64:  # no tile kernel for C > 64
        base = [dv.DV_VARIANT_AUTO, dv.DV_VARIANT_FLAT]
    return base + ([dv.DV_VARIANT_TOKEN] if one_token else [])


def check_pack_unpack(g, cache, kh, vh, l0, l1, s, e, variant):
    n = ORC.staging_bytes(g, l0, l1, s, e)
    dst = H.device_bytes(n + 64, fill=0xEE)
    dv.dv_kv_pack(cache, l0, l1, s, e, dst, variant=variant)
    got = H.to_np(dst)
    want = ORC.pack(g, kh, vh, l0, l1, s, e)
    assert np.array_equal(got[:n], want), (g.name, l0, l1, s, e, variant)
    assert (got[n:] == 0xEE).all()  # nothing written past the staging bytes
    # unpack into a sentinel cache: exactly the selected slices change
    back = H.device_cache(g, fill=0x5A)
    dv.dv_kv_unpack(back, l0, l1, s, e, dst, variant=variant, src_bytes=n)
    kw = np.full(g.tensor_bytes, 0x5A, np.uint8)
    vw = np.full(g.tensor_bytes, 0x5A, np.uint8)
    ORC.unpack(g, kw, vw, l0, l1, s, e, want)
    assert np.array_equal(H.to_np(back.k), kw)
    assert np.array_equal(H.to_np(back.v), vw)


def test_gpu_fill_matches_host_generator():
    for g in (TINY, GEOMS[1], GEOMS[4]):
        c = H.device_cache(g, fill="synth", seed=99)
        kh, vh = H.host_cache(g, 99)
        assert np.array_equal(H.to_np(c.k), kh) and np.array_equal(H.to_np(c.v), vh)


@pytest.mark.parametrize("variant", VARIANTS + [dv.DV_VARIANT_TOKEN])
def test_tiny_workload(variant):
    """Tiny cache: prompt [0,37), then the decode token at 37; unpack into a
    zeroed cache."""
    g, seed = TINY, seed_of(1)
    kh, vh = H.host_cache(g, seed)
    cache = H.device_cache(g, fill=(kh, vh))
    (ps, pe), (ds, de) = tiny_ranges()
    for s, e in ((ps, pe), (ds, de)):
        n = ORC.staging_bytes(g, 0, g.num_layers, s, e)
        dst = H.device_bytes(n)
        dv.dv_kv_pack(cache, 0, g.num_layers, s, e, dst, variant=variant)
        want = ORC.pack(g, kh, vh, 0, g.num_layers, s, e)
        assert np.array_equal(H.to_np(dst)[:n], want)
        z = H.device_cache(g, fill="zero")
        dv.dv_kv_unpack(z, 0, g.num_layers, s, e, dst, variant=variant, src_bytes=n)
        kw, vw = np.zeros_like(kh), np.zeros_like(vh)
        ORC.unpack(g, kw, vw, 0, g.num_layers, s, e, want)
        assert np.array_equal(H.to_np(z.k), kw) and np.array_equal(H.to_np(z.v), vw)


@pytest.mark.parametrize("g", GEOMS, ids=lambda g: g.name)
def test_pack_unpack_geometries(g):
    rng = np.random.default_rng(zlib.crc32(g.name.encode()))  # stable across processes
    kh, vh = H.host_cache(g, 1234)
    cache = H.device_cache(g, fill=(kh, vh))
    for name, s, e in range_sets(g, rng):
        for l0, l1 in ((0, g.num_layers), (g.num_layers - 1, g.num_layers)):
            for variant in variants_for(s, e, g):
                check_pack_unpack(g, cache, kh, vh, l0, l1, s, e, variant)


@pytest.mark.parametrize("g, lens", [
    (Geometry("grp16", 2, 12, 37, 128, 160, 2, "fp16"),      # C = 16: 64-token block
     [1, 2, 3, 31, 32, 33, 63, 64, 65, 0, 17, 129]),
    (Geometry("grp8", 2, 10, 37, 64, 300, 2, "bf16"),        # C = 8: 128-token block
     [1, 5, 63, 64, 65, 127, 128, 129, 0, 257]),
], ids=["c16", "c8"])
def test_grouped_tiles_at_the_block_edges(g, lens):
    """The tile variant with ranges around half the token block (grouped tiles up
    to it, the tile kernel's one-head tiles beyond, both in one call) and 37
    heads (no group size divides it: every sequence's last group is partial)."""
    kh, vh = H.host_cache(g, 4321)
    cache = H.device_cache(g, fill=(kh, vh))
    rng = np.random.default_rng(55)
    ln = np.array(lens, np.int32)
    s = np.array([rng.integers(0, g.max_seq - n + 1) for n in ln], np.int32)
    e = (s + ln).astype(np.int32)
    for l0, l1 in ((0, g.num_layers), (1, 2)):
        check_pack_unpack(g, cache, kh, vh, l0, l1, s, e, dv.DV_VARIANT_TILE)
        check_pack_unpack(g, cache, kh, vh, l0, l1, s, e, dv.DV_VARIANT_AUTO)
    # every range short: a launch of grouped tiles alone
    short = np.minimum(ln, 16).astype(np.int32)
    check_pack_unpack(g, cache, kh, vh, 0, g.num_layers, s, (s + short).astype(np.int32),
                      dv.DV_VARIANT_TILE)


@pytest.mark.parametrize("variant", VARIANTS)
def test_pack_to_and_unpack_from_pinned_host(variant):
    g = GEOMS[0]
    rng = np.random.default_rng(8)
    kh, vh = H.host_cache(g, 77)
    cache = H.device_cache(g, fill=(kh, vh))
    s, e = P.random_ranges(g, rng)
    n = ORC.staging_bytes(g, 0, g.num_layers, s, e)
    host = H.pinned(n)
    dv.dv_kv_pack(cache, 0, g.num_layers, s, e, host, variant=variant)
    torch.cuda.synchronize()
    want = ORC.pack(g, kh, vh, 0, g.num_layers, s, e)
    assert np.array_equal(host.numpy()[:n], want)
    back = H.device_cache(g, fill=0x11)
    dv.dv_kv_unpack(back, 0, g.num_layers, s, e, host, variant=variant)
    kw = np.full_like(kh, 0x11)
    vw = np.full_like(vh, 0x11)
    ORC.unpack(g, kw, vw, 0, g.num_layers, s, e, want)
    assert np.array_equal(H.to_np(back.k), kw) and np.array_equal(H.to_np(back.v), vw)


@pytest.mark.parametrize("staged", [False, True])
def test_swap_out_and_in(staged):
    g = Geometry("swap", 5, 4, 3, 128, 256, 2, "fp16")
    rng = np.random.default_rng(9)
    kh, vh = H.host_cache(g, 5)
    cache = H.device_cache(g, fill=(kh, vh))
    s = np.zeros(g.batch, np.int32)
    e = rng.integers(1, g.max_seq + 1, size=g.batch).astype(np.int32)
    n = ORC.staging_bytes(g, 0, g.num_layers, s, e)
    slab = n // g.num_layers
    staging = H.device_bytes(2 * slab + 16) if staged else None  # 2 layers per group
    host = H.pinned(n)
    dv.dv_swap_out(cache, 0, g.num_layers, s, e, host, staging=staging)
    torch.cuda.synchronize()
    want = ORC.swap_out(g, kh, vh, 0, g.num_layers, s, e)
    assert np.array_equal(host.numpy()[:n], want)
    fresh = H.device_cache(g, fill="zero")
    dv.dv_swap_in(fresh, 0, g.num_layers, s, e, host, staging=staging)
    kw, vw = np.zeros_like(kh), np.zeros_like(vh)
    ORC.unpack(g, kw, vw, 0, g.num_layers, s, e, want)
    assert np.array_equal(H.to_np(fresh.k), kw) and np.array_equal(H.to_np(fresh.v), vw)


def test_stream_layers_matches_oracle_and_swap_out():
    g = Geometry("stream", 6, 3, 4, 64, 128, 2, "fp16")
    kh, vh = H.host_cache(g, 6)
    cache = H.device_cache(g, fill=(kh, vh))
    s = np.zeros(g.batch, np.int32)
    e = np.array([100, 128, 7], np.int32)
    n = ORC.staging_bytes(g, 0, g.num_layers, s, e)
    slab = n // g.num_layers
    slots = (H.device_bytes(slab), H.device_bytes(slab))
    pack_stream, copy_stream = torch.cuda.Stream(), torch.cuda.Stream()
    host = H.pinned(n, fill=0)
    st = dv.Streamer(slots[0], slots[1], pack_stream, copy_stream)
    torch.cuda.synchronize()
    for layer in range(g.num_layers):
        st.stream_layer(cache, layer, s, e, host, l0=0)
    st.wait()
    want = ORC.stream_layers(g, kh, vh, 0, g.num_layers, s, e)
    assert np.array_equal(host.numpy()[:n], want)
    assert np.array_equal(want, ORC.swap_out(g, kh, vh, 0, g.num_layers, s, e))
    st.close()


@pytest.mark.parametrize("one_stream", [False, True])
def test_fetch_layers_matches_oracle(one_stream):
    """The receiving side of layer streaming: the slabs of [l0, l1) in host
    memory (the bytes one pack over that range gives) come into a sentinel
    cache one layer at a time, in order and out of order; the cache then
    equals the oracle's unpack, and a streamer-fetcher round trip restores
    the source slices."""
    g = Geometry("fetch", 6, 3, 4, 64, 128, 2, "fp16")
    kh, vh = H.host_cache(g, 16)
    s = np.array([0, 5, 100], np.int32)
    e = np.array([100, 128, 101], np.int32)
    l0, l1 = 1, 6
    n = ORC.staging_bytes(g, l0, l1, s, e)
    slab = n // (l1 - l0)
    data = ORC.pack(g, kh, vh, l0, l1, s, e)
    host = H.pinned(n + 64, fill=0)
    host.numpy()[:n] = data
    slots = (H.device_bytes(slab), H.device_bytes(slab))
    cs = torch.cuda.Stream()
    us = cs if one_stream else torch.cuda.Stream()
    kw = np.full(g.tensor_bytes, 0x5A, np.uint8)
    vw = np.full(g.tensor_bytes, 0x5A, np.uint8)
    ORC.unpack(g, kw, vw, l0, l1, s, e, data)
    for order in (range(l0, l1), [5, 2, 4, 1, 3]):
        back = H.device_cache(g, fill=0x5A)
        f = dv.Fetcher(slots[0], slots[1], cs, us)
        torch.cuda.synchronize()
        for layer in order:
            f.fetch_layer(back, layer, s, e, host, l0=l0)
        f.wait()
        assert np.array_equal(H.to_np(back.k), kw) and np.array_equal(H.to_np(back.v), vw)
        f.close()
    # round trip: stream out of one cache, fetch into another, layer by layer
    cache = H.device_cache(g, fill=(kh, vh))
    back = H.device_cache(g, fill=0x5A)
    out = H.pinned(n)
    ps, pc = torch.cuda.Stream(), torch.cuda.Stream()
    st = dv.Streamer(H.device_bytes(slab), H.device_bytes(slab), ps, pc)
    f = dv.Fetcher(slots[0], slots[1], cs, us)
    torch.cuda.synchronize()
    for layer in range(l0, l1):
        st.stream_layer(cache, layer, s, e, out, l0=l0)
        cs.wait_stream(pc)  # the layer's bytes are in host memory before they are fetched
        f.fetch_layer(back, layer, s, e, out, l0=l0)
    f.wait()
    st.wait()
    assert np.array_equal(H.to_np(back.k), kw) and np.array_equal(H.to_np(back.v), vw)
    st.close()
    f.close()


def test_fetcher_errors_enqueue_nothing():
    g = Geometry("fetcherr", 3, 2, 2, 64, 64, 2, "fp16")
    s, e = np.zeros(2, np.int32), np.full(2, 64, np.int32)
    n = ORC.staging_bytes(g, 0, 3, s, e)
    slab = n // 3
    back = H.device_cache(g, fill=0x11)
    host = H.pinned(n, fill=0x22)
    big = (H.device_bytes(slab), H.device_bytes(slab))
    small = (H.device_bytes(slab // 2), H.device_bytes(slab // 2))
    assert _status(lambda: dv.Fetcher(big[0], big[0])) == dv.DV_ERR_INVALID_ARG
    f = dv.Fetcher(small[0], small[1])
    assert _status(lambda: f.fetch_layer(back, 0, s, e, host)) == dv.DV_ERR_BUFFER_TOO_SMALL
    f.close()
    f = dv.Fetcher(big[0], big[1])
    assert _status(lambda: f.fetch_layer(back, 2, s, e, (host.data_ptr(), 2 * slab))) == \
        dv.DV_ERR_BUFFER_TOO_SMALL                        # layer 2 lies past the buffer
    assert _status(lambda: f.fetch_layer(back, 0, s, e, host, l0=1)) == dv.DV_ERR_RANGE
    pageable = np.zeros(n, np.uint8)
    assert _status(lambda: f.fetch_layer(back, 0, s, e, (pageable.ctypes.data, n))) == \
        dv.DV_ERR_INVALID_ARG
    f.wait()
    f.close()
    torch.cuda.synchronize()
    assert (H.to_np(back.k) == 0x11).all() and (H.to_np(back.v) == 0x11).all()


@pytest.mark.parametrize("mode", ["fused", "staged", "streamed"])
def test_replica_snapshot_deltas_restore_truncate(mode):
    """streamed: the appends go through a layer streamer whose slots hold two
    of the snapshot's layers, so the snapshot goes in two groups (layers 0-1,
    then 2) and each delta in one."""
    g = Geometry("rep", 3, 4, 2, 128, 64, 2, "bf16")
    kh, vh = H.host_cache(g, 12)
    cache = H.device_cache(g, fill=(kh, vh))
    len0 = np.array([5, 20, 1, 33], np.int32)
    zero = np.zeros(g.batch, np.int32)
    steps = 6
    total = ORC.staging_bytes(g, 0, g.num_layers, zero, len0 + steps)
    arena = H.pinned(total + 4096)
    staging = H.device_bytes(total) if mode == "staged" else None
    streamer = None
    if mode == "streamed":
        slot = 2 * ORC.staging_bytes(g, 0, 1, zero, len0)
        torch.cuda.synchronize()
        streamer = dv.Streamer(H.device_bytes(slot), H.device_bytes(slot), torch.cuda.Stream(),
                               torch.cuda.Stream())
    rep = dv.Replica(arena, g.batch)

    def append(l0, l1, s, e, step):
        if streamer:
            rep.append_streamed(streamer, cache, l0, l1, s, e, step=step)
        else:
            rep.append(cache, l0, l1, s, e, step=step, staging=staging)

    append(0, g.num_layers, zero, len0, 0)
    pos = len0.copy()
    records = [(0, g.num_layers, zero, len0.copy())]
    for k in range(1, steps + 1):
        act = np.array([1, 1, 1 if k < 3 else 0, 1], np.int32)  # sequence 2 finishes
        append(0, g.num_layers, pos, pos + act, k)
        records.append((0, g.num_layers, pos.copy(), (pos + act).copy()))
        pos = pos + act
    if streamer:
        streamer.wait()
    torch.cuda.synchronize()
    nrec, used = rep.info()
    assert nrec == steps + 1
    assert used == sum(ORC.staging_bytes(g, a, b, s, e) for a, b, s, e in records)
    # the arena holds the records end to end
    want_arena = np.concatenate([ORC.pack(g, kh, vh, a, b, s, e) for a, b, s, e in records])
    assert np.array_equal(arena.numpy()[:used], want_arena)
    # restore everything into a zeroed cache = the live cache on [0, pos)
    z = H.device_cache(g, fill="zero")
    rep.restore(z, staging=staging)
    kw, vw = ORC.restore(g, [(a, b, s, e, ORC.pack(g, kh, vh, a, b, s, e))
                             for a, b, s, e in records])
    assert np.array_equal(H.to_np(z.k), kw) and np.array_equal(H.to_np(z.v), vw)
    # acknowledged prefix: truncate at step 4 keeps steps 0..3 only
    rep.truncate(4)
    assert rep.info()[0] == 4
    z2 = H.device_cache(g, fill="zero")
    rep.restore(z2, staging=staging)
    kw, vw = ORC.restore(g, [(a, b, s, e, ORC.pack(g, kh, vh, a, b, s, e))
                             for a, b, s, e in records[:4]])
    assert np.array_equal(H.to_np(z2.k), kw) and np.array_equal(H.to_np(z2.v), vw)
    rep.close()
    if streamer:
        streamer.close()


def test_replica_append_streamed_errors():
    g = Geometry("reperr", 3, 4, 2, 128, 64, 2, "bf16")
    cache = H.device_cache(g, fill=0x21)
    zero = np.zeros(g.batch, np.int32)
    len0 = np.array([5, 20, 1, 33], np.int32)
    slab = ORC.staging_bytes(g, 0, 1, zero, len0)
    arena = H.pinned(ORC.staging_bytes(g, 0, g.num_layers, zero, len0) + 64)
    rep = dv.Replica(arena, g.batch)
    small = dv.Streamer(H.device_bytes(slab - 16), H.device_bytes(slab - 16))
    # one layer of the record is larger than a slot: refused before anything is enqueued
    assert _status(lambda: rep.append_streamed(small, cache, 0, 3, zero, len0, step=0)) == \
        dv.DV_ERR_BUFFER_TOO_SMALL
    assert rep.info() == (0, 0)
    ok = dv.Streamer(H.device_bytes(slab), H.device_bytes(slab))
    rep.append_streamed(ok, cache, 0, 3, zero, len0, step=1)       # three groups of one layer
    assert _status(lambda: rep.append_streamed(ok, cache, 0, 3, zero, len0, step=2)) == \
        dv.DV_ERR_BUFFER_TOO_SMALL                                  # the arena is full
    assert _status(lambda: rep.append_streamed(ok, cache, 0, 1, zero, zero + 1, step=0)) == \
        dv.DV_ERR_INVALID_ARG                                       # step before the last record's
    assert _status(lambda: rep.append_streamed(ok, cache, 0, 1, zero, zero + 65, step=3)) == \
        dv.DV_ERR_RANGE
    ok.wait()
    torch.cuda.synchronize()
    assert rep.info() == (1, 3 * slab)
    assert (arena.numpy()[:3 * slab] == 0x21).all()               # every byte of the cache is 0x21
    small.close()
    ok.close()
    rep.close()


def _status(fn):
    with pytest.raises(dv.DvError) as ei:
        fn()
    return ei.value.status


def test_errors_with_real_buffers_enqueue_nothing():
    g = Geometry("err", 2, 2, 2, 64, 32, 2, "fp16")
    cache = H.device_cache(g, fill=0x33)
    s, e = np.zeros(2, np.int32), np.full(2, 32, np.int32)
    n = ORC.staging_bytes(g, 0, 2, s, e)
    dst = H.device_bytes(n + 64, fill=0x44)
    # misaligned destination
    assert _status(lambda: dv.dv_kv_pack(cache, 0, 2, s, e, (dst.data_ptr() + 8, n))) == \
        dv.DV_ERR_MISALIGNED
    # pageable host memory is refused
    pageable = np.zeros(n + 64, np.uint8)
    assert _status(lambda: dv.dv_kv_pack(cache, 0, 2, s, e, (pageable.ctypes.data, n))) == \
        dv.DV_ERR_INVALID_ARG
    # A claimed size past the end of the allocation is refused by the driver
    # range check.  Exercised only when the library itself reports, before the
    # call, an extent shorter than the claim: the call that follows is then
    # refused on the host and no kernel can run out of bounds.
    gb = Geometry("err2", 2, 2, 2, 128, 2048, 2, "fp16")
    cb = H.device_cache(gb, fill=0x33)
    sb, eb = np.zeros(2, np.int32), np.full(2, 2048, np.int32)
    nb = ORC.staging_bytes(gb, 0, 2, sb, eb)
    small = H.device_bytes(1 << 20)
    ext = dv.dv_allocation_extent(small)
    if ext is not None and ext < nb:
        assert _status(lambda: dv.dv_kv_pack(cb, 0, 2, sb, eb, (small.data_ptr(), nb))) == \
            dv.DV_ERR_BUFFER_TOO_SMALL
    huge_layers = 1 << 20
    ext_k = dv.dv_allocation_extent(cb.k)
    lay = gb.tensor_bytes // gb.num_layers
    if ext_k is not None and ext_k < huge_layers * lay:
        big = dv.Cache(huge_layers, 2, 2, 128, 2048, 2, cb.k, cb.v)
        assert _status(lambda: dv.dv_kv_pack(big, huge_layers - 1, huge_layers, sb, eb,
                                             (dst.data_ptr(), nb // 2))) == \
            dv.DV_ERR_BUFFER_TOO_SMALL
    # the tile kernel refuses more than 64 chunks per token
    wide = Geometry("wide", 1, 2, 1, 1024, 8, 2, "fp16")
    cw = H.device_cache(wide, fill=0x33)
    sw, ew = np.zeros(2, np.int32), np.full(2, 8, np.int32)
    nw = ORC.staging_bytes(wide, 0, 1, sw, ew)
    dw = H.device_bytes(nw)
    assert _status(lambda: dv.dv_kv_pack(cw, 0, 1, sw, ew, dw, variant=dv.DV_VARIANT_TILE)) == \
        dv.DV_ERR_UNSUPPORTED
    # the token kernel refuses ranges of different lengths
    assert _status(lambda: dv.dv_kv_pack(cache, 0, 2, s, np.array([32, 16], np.int32), dst,
                                         variant=dv.DV_VARIANT_TOKEN)) == dv.DV_ERR_UNSUPPORTED
    # staging smaller than one layer slab
    host = H.pinned(n)
    tiny_stg = H.device_bytes(n // 4)
    assert _status(lambda: dv.dv_swap_out(cache, 0, 2, s, e, host, staging=tiny_stg)) == \
        dv.DV_ERR_BUFFER_TOO_SMALL
    # swap to device memory instead of pinned host memory is refused
    assert _status(lambda: dv.dv_swap_out(cache, 0, 2, s, e, dst)) == dv.DV_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert (H.to_np(dst) == 0x44).all()  # no failed call wrote anything


def test_naive_gather_matches_the_pack():
    """The per-region copy baseline writes the staging bytes of the pack, for
    ranges shorter than C (per-token copies) and longer (per-row copies), to
    device memory and to pinned host memory."""
    g = Geometry("naive", 3, 3, 2, 128, 64, 2, "fp16")  # C = 16
    kh, vh = H.host_cache(g, 41)
    cache = H.device_cache(g, fill=(kh, vh))
    cases = [(np.array([5, 0, 9], np.int32), np.array([6, 0, 12], np.int32)),   # < C tokens
             (np.array([0, 3, 10], np.int32), np.array([40, 64, 30], np.int32))]  # >= C tokens
    for s, e in cases:
        n = ORC.staging_bytes(g, 0, g.num_layers, s, e)
        want = ORC.pack(g, kh, vh, 0, g.num_layers, s, e)
        dst = H.device_bytes(n)
        calls = dv.dv_naive_gather(cache, 0, g.num_layers, s, e, dst)
        assert calls > 0
        assert np.array_equal(H.to_np(dst)[:n], want)
        host = H.pinned(n)
        dv.dv_naive_gather(cache, 0, g.num_layers, s, e, host)
        torch.cuda.synchronize()
        assert np.array_equal(host.numpy()[:n], want)


def test_replica_compaction():
    """Compaction: the snapshot + deltas of a replica replaced by one snapshot of
    the used prefix (truncate to nothing, append the prefix); the compacted
    replica restores the same cache and takes only the prefix's bytes."""
    g = Geometry("compact", 2, 3, 2, 64, 40, 2, "fp16")
    kh, vh = H.host_cache(g, 57)
    cache = H.device_cache(g, fill=(kh, vh))
    zero = np.zeros(g.batch, np.int32)
    pos = np.array([4, 9, 2], np.int32)
    arena = H.pinned(ORC.staging_bytes(g, 0, g.num_layers, zero, pos + 5) + 4096)
    rep = dv.Replica(arena, g.batch)
    rep.append(cache, 0, g.num_layers, zero, pos, step=0)
    for k in range(1, 6):
        rep.append(cache, 0, g.num_layers, pos, pos + 1, step=k)
        pos = pos + 1
    before = H.device_cache(g, fill="zero")
    rep.restore(before)
    rep.truncate(0)  # compaction: the whole log is replaced ...
    assert rep.info() == (0, 0)
    rep.append(before, 0, g.num_layers, zero, pos, step=5)  # ... by one snapshot of the prefix
    after = H.device_cache(g, fill="zero")
    rep.restore(after)
    torch.cuda.synchronize()
    assert rep.info() == (1, ORC.staging_bytes(g, 0, g.num_layers, zero, pos))
    assert torch.equal(before.k, after.k) and torch.equal(before.v, after.v)
    mk, mv = P.selected_mask(g, 0, g.num_layers, zero, pos)
    kw = np.where(np.repeat(mk, 2), kh, 0).astype(np.uint8)
    vw = np.where(np.repeat(mv, 2), vh, 0).astype(np.uint8)
    assert np.array_equal(H.to_np(after.k), kw) and np.array_equal(H.to_np(after.v), vw)
    rep.close()


def test_concurrent_calls_from_threads():
    """Eight host threads, each on its own stream, pack different ranges of
    one cache and unpack them into caches of their own at the same time (the
    library holds no per-call global state): every result equals the
    oracle's."""
    import threading
    g = Geometry("thr", 3, 4, 4, 128, 256, 2, "fp16")
    kh, vh = H.host_cache(g, 77)
    cache = H.device_cache(g, fill=(kh, vh))
    rng = np.random.default_rng(77)
    jobs = [P.random_ranges(g, rng) for _ in range(8)]
    outs = [H.device_bytes(ORC.staging_bytes(g, 0, g.num_layers, s, e)) for s, e in jobs]
    backs = [H.device_cache(g, fill=0x5A) for _ in jobs]
    torch.cuda.synchronize()
    barrier = threading.Barrier(len(jobs))
    errors = []

    def worker(i):
        try:
            s, e = jobs[i]
            st = torch.cuda.Stream()
            barrier.wait()
            for _ in range(20):
                dv.dv_kv_pack(cache, 0, g.num_layers, s, e, outs[i], stream=st)
                dv.dv_kv_unpack(backs[i], 0, g.num_layers, s, e, outs[i], stream=st)
            st.synchronize()
        except Exception as ex:  # reported below, from the main thread
            errors.append(repr(ex))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(jobs))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for (s, e), out, back in zip(jobs, outs, backs):
        n = ORC.staging_bytes(g, 0, g.num_layers, s, e)
        want = ORC.pack(g, kh, vh, 0, g.num_layers, s, e)
        assert np.array_equal(H.to_np(out)[:n], want)
        kw = np.full(g.tensor_bytes, 0x5A, np.uint8)
        vw = np.full(g.tensor_bytes, 0x5A, np.uint8)
        ORC.unpack(g, kw, vw, 0, g.num_layers, s, e, want)
        assert np.array_equal(H.to_np(back.k), kw) and np.array_equal(H.to_np(back.v), vw)


def test_concurrent_staged_swaps_from_threads():
    """Six host threads, each on its own stream with its own staging buffer,
    swap different ranges of one cache out to pinned host memory and back in
    to caches of their own, staged (two halves per buffer: the copies of every
    thread share the library's copy stream, ordered by each call's events),
    20 times each: every host buffer and cache equals the oracle's."""
    import threading
    g = Geometry("thrswap", 6, 4, 4, 128, 256, 2, "bf16")
    kh, vh = H.host_cache(g, 78)
    cache = H.device_cache(g, fill=(kh, vh))
    rng = np.random.default_rng(78)
    jobs = [P.random_ranges(g, rng) for _ in range(6)]
    hosts = [H.pinned(ORC.staging_bytes(g, 0, g.num_layers, s, e), fill=0) for s, e in jobs]
    stgs = [H.device_bytes(2 * max(16, ORC.staging_bytes(g, 0, 1, s, e))) for s, e in jobs]
    backs = [H.device_cache(g, fill=0x3C) for _ in jobs]
    torch.cuda.synchronize()
    barrier = threading.Barrier(len(jobs))
    errors = []

    def worker(i):
        try:
            s, e = jobs[i]
            st = torch.cuda.Stream()
            barrier.wait()
            for _ in range(20):
                dv.dv_swap_out(cache, 0, g.num_layers, s, e, hosts[i], staging=stgs[i], stream=st)
                dv.dv_swap_in(backs[i], 0, g.num_layers, s, e, hosts[i], staging=stgs[i],
                              stream=st)
            st.synchronize()
        except Exception as ex:  # reported below, from the main thread
            errors.append(repr(ex))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(jobs))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    assert not errors, errors
    for (s, e), host, back in zip(jobs, hosts, backs):
        n = ORC.staging_bytes(g, 0, g.num_layers, s, e)
        want = ORC.pack(g, kh, vh, 0, g.num_layers, s, e)
        assert np.array_equal(host[:n].numpy(), want)
        kw = np.full(g.tensor_bytes, 0x3C, np.uint8)
        vw = np.full(g.tensor_bytes, 0x3C, np.uint8)
        ORC.unpack(g, kw, vw, 0, g.num_layers, s, e, want)
        assert np.array_equal(H.to_np(back.k), kw) and np.array_equal(H.to_np(back.v), vw)
