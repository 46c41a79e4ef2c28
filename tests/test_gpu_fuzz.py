"""Seeded random cases of pack and unpack against the oracle, byte for byte.

Each case draws a cache geometry (element size 1, 2 or 4 bytes; 1 to 80
chunks per token; batch up to 200; max_seq 1 to 260; sometimes padded
layers), a layer range, a range pattern (ragged, equal-length multi-token,
one-token decode with finished sequences, full, prefixes, all empty), a
kernel (the automatic choice or one forced, where it applies) and where the
staging bytes live (device or pinned host memory).  The pack must give the
oracle's bytes and write nothing past them; the unpack into a sentinel cache
must give the oracle's cache, every byte outside the selected slices
untouched."""
import numpy as np
import pytest

import kv_cache_streaming_gb300 as dv
import oracle
from synth.configs import Geometry
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu
ORC = oracle.default()
CASES = 160
MAX_TENSOR_BYTES = 6 << 20


def _geometry(rng, i, max_bytes=MAX_TENSOR_BYTES):
    """A random geometry whose K and V tensors hold at most max_bytes each."""
    while True:
        P = int(rng.choice([1, 2, 2, 2, 4]))
        x = 16 // P
        C = int(rng.choice([1, 2, 3, 4, 5, 8, 8, 12, 16, 16, 24, 32, 64, 80]))
        B = int(rng.choice([1, 2, 3, 5, 8, 13, 32, 33, 40, 200]))
        H = int(rng.integers(1, 7))
        S = int(rng.choice([1, 2, 7, 8, 9, 31, 64, 100, 129, 260]))
        L = int(rng.integers(1, 5))
        D = C * x
        dense = B * H * D * S
        pad = int(rng.choice([0, 0, 0, x, 5 * x, 64 * x]))
        stride = dense + pad if pad else 0
        g = Geometry(f"fz{i}", L, B, H, D, S, P, {1: "raw", 2: "fp16", 4: "fp32"}[P],
                     layer_stride_elems=stride)
        if g.tensor_bytes <= max_bytes:
            return g


def _ranges(g, rng):
    B, S = g.batch, g.max_seq
    kind = rng.choice(["ragged", "equal", "decode", "full", "prefix", "empty"])
    if kind == "ragged":
        a = rng.integers(0, S + 1, size=B)
        c = rng.integers(0, S + 1, size=B)
        s, e = np.minimum(a, c), np.maximum(a, c)
    elif kind == "equal":
        n = int(rng.integers(1, S + 1))
        s = rng.integers(0, S - n + 1, size=B)
        e = s + n
        e = np.where(rng.random(B) < 0.25, s, e)  # some finished sequences
    elif kind == "decode":
        s = rng.integers(0, S, size=B)
        e = np.where(rng.random(B) < 0.3, s, s + 1)
    elif kind == "full":
        s, e = np.zeros(B), np.full(B, S)
    elif kind == "prefix":
        s, e = np.zeros(B), rng.integers(0, S + 1, size=B)
    else:
        s = rng.integers(0, S + 1, size=B)
        e = s
    return str(kind), s.astype(np.int32), e.astype(np.int32)


def _variant(g, s, e, rng):
    lens = e - s
    active = lens[lens > 0]
    choices = [dv.DV_VARIANT_AUTO, dv.DV_VARIANT_FLAT]
    if g.head_dim * g.elem_bytes // 16 <= 64:
        choices.append(dv.DV_VARIANT_TILE)
    if active.size and (active == active[0]).all():
        choices.append(dv.DV_VARIANT_TOKEN)
    return int(rng.choice(choices))


def _buffer(nbytes, host, fill):
    return H.pinned(nbytes, fill=fill) if host else H.device_bytes(nbytes, fill=fill)


@pytest.mark.parametrize("block", range(4))
def test_random_pack_unpack_matches_oracle(block):
    rng = np.random.default_rng(0xF022 + block)
    for i in range(block * CASES // 4, (block + 1) * CASES // 4):
        g = _geometry(rng, i)
        seed = 9000 + i
        kh, vh = H.host_cache(g, seed)
        cache = H.device_cache(g, fill=(kh, vh))
        l0 = int(rng.integers(0, g.num_layers + 1))
        l1 = int(rng.integers(l0, g.num_layers + 1))
        kind, s, e = _ranges(g, rng)
        variant = _variant(g, s, e, rng)
        host = bool(rng.random() < 0.25)
        where = (g, l0, l1, kind, s.tolist(), e.tolist(), variant, host)
        n = ORC.staging_bytes(g, l0, l1, s, e)
        assert dv.dv_staging_bytes(cache, l0, l1, s, e) == n, where
        want = ORC.pack(g, kh, vh, l0, l1, s, e)
        dst = _buffer(n + 48, host, 0xEE)
        dv.dv_kv_pack(cache, l0, l1, s, e, dst, variant=variant)
        got = H.to_np(dst)
        assert np.array_equal(got[:n], want), where
        assert (got[n:] == 0xEE).all(), where
        src = _buffer(n + 48, not host, 0x00)  # the unpack reads from the other memory kind
        src.copy_(dst)
        back = H.device_cache(g, fill=0x5A)
        dv.dv_kv_unpack(back, l0, l1, s, e, src, variant=variant, src_bytes=n)
        kw = np.full(g.tensor_bytes, 0x5A, np.uint8)
        vw = np.full(g.tensor_bytes, 0x5A, np.uint8)
        ORC.unpack(g, kw, vw, l0, l1, s, e, want)
        assert np.array_equal(H.to_np(back.k), kw), where
        assert np.array_equal(H.to_np(back.v), vw), where
        del cache, back, dst, src


def test_random_grouped_tiles_match_oracle():
    """Grouped tiles (C = 8 or 16): random head counts (1..80, so the last group of
    a sequence is often partial), ranges mostly shorter than half the token block
    mixed with longer ones, through the tile variant and the automatic choice,
    to and from device or pinned host memory."""
    rng = np.random.default_rng(0x6A0)
    for i in range(40):
        C = int(rng.choice([8, 16]))
        tb = 1024 // C
        nh = int(rng.integers(1, 81))
        B = int(rng.choice([1, 3, 8, 33]))
        S = int(rng.choice([tb // 2, tb, 2 * tb + 5]))
        L = int(rng.integers(1, 4))
        g = Geometry(f"gz{i}", L, B, nh, C * 8, S, 2, "fp16")
        if g.tensor_bytes > (24 << 20):
            continue
        kh, vh = H.host_cache(g, 7700 + i)
        cache = H.device_cache(g, fill=(kh, vh))
        short = rng.random(B) < 0.75
        lens = np.where(short, rng.integers(0, tb // 2 + 1, size=B),
                        rng.integers(0, S + 1, size=B))
        lens = np.minimum(lens, S)
        s = np.array([rng.integers(0, S - n + 1) for n in lens], np.int32)
        e = (s + lens).astype(np.int32)
        l0 = int(rng.integers(0, L))
        l1 = int(rng.integers(l0 + 1, L + 1))
        variant = int(rng.choice([dv.DV_VARIANT_TILE, dv.DV_VARIANT_AUTO]))
        host = bool(rng.random() < 0.25)
        where = (g, l0, l1, s.tolist(), e.tolist(), variant, host)
        n = ORC.staging_bytes(g, l0, l1, s, e)
        want = ORC.pack(g, kh, vh, l0, l1, s, e)
        dst = _buffer(n + 48, host, 0xEE)
        dv.dv_kv_pack(cache, l0, l1, s, e, dst, variant=variant)
        got = H.to_np(dst)
        assert np.array_equal(got[:n], want), where
        assert (got[n:] == 0xEE).all(), where
        back = H.device_cache(g, fill=0x5A)
        dv.dv_kv_unpack(back, l0, l1, s, e, dst, variant=variant, src_bytes=n)
        kw = np.full(g.tensor_bytes, 0x5A, np.uint8)
        vw = np.full(g.tensor_bytes, 0x5A, np.uint8)
        ORC.unpack(g, kw, vw, l0, l1, s, e, want)
        assert np.array_equal(H.to_np(back.k), kw), where
        assert np.array_equal(H.to_np(back.v), vw), where
        del cache, back, dst


def _restore_into_zero(g, rep, how, slab, total, rng):
    """A zeroed cache after restoring the replica: record-batched fused or
    staged (a staging buffer between the largest layer slab and the whole
    log), or pipelined through a fetcher with slots of that size."""
    import torch
    z = H.device_cache(g, fill="zero")
    size = int(rng.integers(slab, max(slab, total) + 1)) // 16 * 16 + 16
    # the zero fill runs on torch's stream; a fetcher's streams are ordered
    # after earlier work on the cache by the caller (here: all of it ends)
    torch.cuda.synchronize()
    if how == "fused":
        rep.restore_batched(z)
    elif how == "staged":
        rep.restore_batched(z, staging=H.device_bytes(size))
    else:
        cs = torch.cuda.Stream()
        f = dv.Fetcher(H.device_bytes(size), H.device_bytes(size), cs, torch.cuda.Stream())
        rep.restore_fetched(z, f)
        f.wait()
        f.close()
    return z


@pytest.mark.parametrize("block", range(2))
def test_random_replica_logs_restore_like_the_oracle(block):
    """Random logs (1 to 40 records, each over its own layer range and range
    pattern, the live cache rewritten now and then so that later records
    carry new bytes for slices earlier records wrote) restore to the cache
    the oracle's in-order restore gives; the arena holds the oracle's records
    end to end, whichever way they were appended."""
    import torch
    rng = np.random.default_rng(0x5E57 + block)
    for i in range(20):
        g = _geometry(rng, 1000 + 100 * block + i, max_bytes=1 << 20)
        seed = 7000 + 100 * block + i
        kh, vh = H.host_cache(g, seed)
        cache = H.device_cache(g, fill=(kh, vh))
        nrec = int(rng.integers(1, 41))
        logs = []
        for r in range(nrec):
            if rng.random() < 0.15:  # new live content
                kh, vh = H.host_cache(g, seed * 31 + r)
                cache = H.device_cache(g, fill=(kh, vh))
            l0 = int(rng.integers(0, g.num_layers))
            l1 = int(rng.integers(l0 + 1, g.num_layers + 1))
            _, s, e = _ranges(g, rng)
            logs.append((l0, l1, s, e, ORC.pack(g, kh, vh, l0, l1, s, e), cache))
        total = sum(d.size for *_, d, _ in logs)
        arena = H.pinned(total + 64)
        rep = dv.Replica(arena, g.batch)
        slabs = [d.size // (l1 - l0) for l0, l1, _, _, d, _ in logs if d.size]
        slab = max(slabs) if slabs else 16
        # appended fused, staged, or through a layer streamer whose slots hold
        # between one layer slab and the whole log (records split into groups)
        mode = str(rng.choice(["fused", "staged", "streamed"]))
        streamer = staging = None
        if mode == "streamed":
            slot = (int(rng.integers(slab, max(slab, total) + 1)) + 15) // 16 * 16
            streamer = dv.Streamer(H.device_bytes(slot), H.device_bytes(slot),
                                   torch.cuda.current_stream(), torch.cuda.Stream())
        elif mode == "staged":
            staging = H.device_bytes(max(total, 16))
        for step, (l0, l1, s, e, _, c) in enumerate(logs):
            if streamer:
                rep.append_streamed(streamer, c, l0, l1, s, e, step=step)
            else:
                rep.append(c, l0, l1, s, e, step=step, staging=staging)
        if streamer:
            streamer.wait()
            streamer.close()
        torch.cuda.synchronize()
        assert np.array_equal(arena.numpy()[:total],
                              np.concatenate([d for *_, d, _ in logs]) if total else
                              np.empty(0, np.uint8)), (g, nrec, mode)
        how = str(rng.choice(["fused", "staged", "fetched"]))
        z = _restore_into_zero(g, rep, how, slab, total, rng)
        kw, vw = ORC.restore(g, [(l0, l1, s, e, d) for l0, l1, s, e, d, _ in logs])
        where = (g, nrec, mode, how)
        assert np.array_equal(H.to_np(z.k), kw), where
        assert np.array_equal(H.to_np(z.v), vw), where
        rep.close()
        del z, cache, arena, logs


@pytest.mark.parametrize("block", range(2))
def test_random_decode_logs_restore_like_the_oracle(block):
    """Random decode logs, the run kernel's domain: a snapshot, then stretches
    of one-token records (each one token further on for the live sequences),
    broken at random by a change of the live set, a change of layer range, a
    ragged or multi-token record, a repeated position (a record over the
    previous one's slices, with new bytes) or new live content.  Restored
    fused, staged or through a fetcher, and by dv_kv_unpack_records from
    device memory, each against the oracle's in-order restore."""
    import torch
    rng = np.random.default_rng(0xD0C + block)
    for i in range(16):
        g = _geometry(rng, 2000 + 100 * block + i, max_bytes=2 << 20)
        if g.max_seq < 4:
            continue
        seed = 9000 + 100 * block + i
        kh, vh = H.host_cache(g, seed)
        cache = H.device_cache(g, fill=(kh, vh))
        B, S, L = g.batch, g.max_seq, g.num_layers
        zs = np.zeros(B, np.int32)
        pos = rng.integers(0, max(1, S // 3), size=B).astype(np.int32)
        logs = [(0, L, zs, pos.copy(), ORC.pack(g, kh, vh, 0, L, zs, pos), cache)]
        live = rng.random(B) < 0.8
        l0, l1 = 0, L
        for r in range(int(rng.integers(2, 90))):
            u = rng.random()
            if u < 0.05:
                live = rng.random(B) < 0.7
            elif u < 0.08:
                l0 = int(rng.integers(0, L))
                l1 = int(rng.integers(l0 + 1, L + 1))
            elif u < 0.1:
                kh, vh = H.host_cache(g, seed * 31 + r)
                cache = H.device_cache(g, fill=(kh, vh))
            elif u < 0.12:
                pos = np.maximum(pos - 1, 0).astype(np.int32)   # the last token again
            act = (live & (pos < S)).astype(np.int32)
            if rng.random() < 0.05:                              # a multi-token record
                act = np.minimum(rng.integers(0, 3, size=B), S - pos).astype(np.int32)
            s, e = pos.copy(), (pos + act).astype(np.int32)
            logs.append((l0, l1, s, e, ORC.pack(g, kh, vh, l0, l1, s, e), cache))
            pos = e
        total = sum(d.size for *_, d, _ in logs)
        arena = H.pinned(total + 64)
        rep = dv.Replica(arena, g.batch)
        for step, (a0, a1, s, e, _, c) in enumerate(logs):
            rep.append(c, a0, a1, s, e, step=step)
        slabs = [d.size // (a1 - a0) for a0, a1, _, _, d, _ in logs if d.size]
        slab = max(slabs) if slabs else 16
        kw, vw = ORC.restore(g, [(a0, a1, s, e, d) for a0, a1, s, e, d, _ in logs])
        for how in ("fused", "staged", "fetched"):
            z = _restore_into_zero(g, rep, how, slab, total, rng)
            where = (g, len(logs), how)
            assert np.array_equal(H.to_np(z.k), kw), where
            assert np.array_equal(H.to_np(z.v), vw), where
        z = H.device_cache(g, fill="zero")
        src = torch.from_numpy(np.concatenate([d for *_, d, _ in logs]) if total
                               else np.zeros(16, np.uint8)).cuda()
        torch.cuda.synchronize()
        dv.dv_kv_unpack_records(z, [(a0, a1, s, e) for a0, a1, s, e, _, _ in logs], src)
        assert np.array_equal(H.to_np(z.k), kw), (g, "unpack_records")
        assert np.array_equal(H.to_np(z.v), vw), (g, "unpack_records")
        rep.close()
        del z, cache, arena, logs
