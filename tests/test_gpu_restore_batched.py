"""Parity of the record-batched restore (dv_replica_restore_batched) with the
oracle's in-order restore of the same log: a snapshot and many decode deltas
in few launches, records with their own layer ranges, records that rewrite
what earlier records wrote (later wins), empty records, more records than one
launch takes, batch 1024, fused, staged and pipelined through a fetcher,
upto_step, and the errors."""
import numpy as np
import pytest
import torch

import kv_cache_streaming_gb300 as dv
import oracle
from synth.configs import Geometry
from tests import gpu_helpers as H
from tests import oracle_pins as P

pytestmark = pytest.mark.gpu
ORC = oracle.default()

GEOMS = [
    Geometry("c16", 3, 5, 3, 128, 300, 2, "fp16"),
    Geometry("c8", 2, 4, 5, 64, 200, 2, "bf16"),
    Geometry("c5", 2, 3, 2, 40, 90, 2, "fp16"),      # odd C: generic kernel
    Geometry("p1", 2, 3, 2, 128, 64, 1, "raw"),
    Geometry("p4", 2, 3, 2, 64, 64, 4, "fp32"),
    Geometry("pad", 3, 2, 2, 128, 50, 2, "fp16", layer_stride_elems=2 * 2 * 128 * 50 + 64),
    Geometry("b40", 1, 40, 2, 64, 32, 2, "fp16"),    # batch > 32
]


class Log:
    """A live cache and a replica of it; `records` mirrors the log for the
    oracle: (l0, l1, s, e, the bytes the oracle packs from the live cache as
    it was at the append)."""

    def __init__(self, g, seed, capacity):
        self.g = g
        self.seed = seed
        self.kh, self.vh = H.host_cache(g, seed)
        self.cache = H.device_cache(g, fill=(self.kh, self.vh))
        self.arena = H.pinned(capacity + 4096)
        self.rep = dv.Replica(self.arena, g.batch)
        self.records = []

    def rewrite(self, salt):
        """New content for the whole live cache (a later record over the same
        slices then carries different bytes)."""
        self.kh, self.vh = H.host_cache(self.g, self.seed * 7919 + salt)
        self.cache.k.copy_(torch.from_numpy(self.kh))
        self.cache.v.copy_(torch.from_numpy(self.vh))

    def append(self, l0, l1, s, e):
        s = np.asarray(s, np.int32)
        e = np.asarray(e, np.int32)
        step = len(self.records)
        self.rep.append(self.cache, l0, l1, s, e, step=step)
        self.records.append((l0, l1, s.copy(), e.copy(),
                             ORC.pack(self.g, self.kh, self.vh, l0, l1, s, e)))

    def check(self, staging_bytes=None, upto=-1, batched=True, slot_bytes=None,
              one_stream=False):
        """Restores into a zeroed cache and compares with the oracle: record by
        record, record-batched (fused, or staged through staging_bytes), or
        pipelined through a fetcher with slots of slot_bytes."""
        g = self.g
        z = H.device_cache(g, fill="zero")
        staging = H.device_bytes(staging_bytes) if staging_bytes else None
        # the zero fill (on torch's stream) ends before the fetcher's streams
        # touch the cache
        torch.cuda.synchronize()
        if slot_bytes:
            cs = torch.cuda.Stream()
            f = dv.Fetcher(H.device_bytes(slot_bytes), H.device_bytes(slot_bytes), cs,
                           cs if one_stream else torch.cuda.Stream())
            self.rep.restore_fetched(z, f, upto_step=upto)
            f.wait()
            f.close()
        elif batched:
            self.rep.restore_batched(z, upto_step=upto, staging=staging)
        else:
            self.rep.restore(z, upto_step=upto, staging=staging)
        recs = self.records if upto < 0 else self.records[:upto]
        kw, vw = ORC.restore(g, recs)
        assert np.array_equal(H.to_np(z.k), kw), (g.name, staging_bytes, upto)
        assert np.array_equal(H.to_np(z.v), vw), (g.name, staging_bytes, upto)


def min_staging(log):
    """The smallest staging buffer a staged restore of the log accepts: the
    largest layer slab of any record."""
    slab = max(d.size // (l1 - l0) for l0, l1, _, _, d in log.records if d.size)
    return (slab + 15) // 16 * 16


def standard_log(g, seed):
    """Snapshot of ragged prefixes, then decode deltas (some sequences
    finish), a ragged multi-token record, an empty record, records over part
    of the layers, and records that rewrite earlier slices."""
    rng = np.random.default_rng(seed)
    B, S, L = g.batch, g.max_seq, g.num_layers
    zero = np.zeros(B, np.int32)
    pos = rng.integers(S // 4, S // 2, size=B).astype(np.int32)
    full = ORC.staging_bytes(g, 0, L, zero, np.full(B, S, np.int32))
    log = Log(g, seed, 4 * full)
    log.append(0, L, zero, pos)                               # snapshot
    live = np.ones(B, bool)
    for k in range(12):                                       # one-token deltas
        if k == 5:
            live[::3] = False
        act = np.where(live & (pos < S), 1, 0).astype(np.int32)
        log.append(0, L, pos, pos + act)
        pos = pos + act
    n = np.minimum(rng.integers(0, 4, size=B), S - pos).astype(np.int32)
    log.append(0, L, pos, pos + n)                            # ragged multi-token
    pos = pos + n
    log.append(0, L, pos, pos)                                # empty record
    a = np.maximum(pos - 3, 0).astype(np.int32)
    log.append(0, 1, a, pos)                                  # first layer only ...
    if L > 1:
        log.append(1, L, a, pos)                              # ... the others: disjoint
    log.rewrite(1)
    b = np.maximum(pos - 2, 0).astype(np.int32)
    log.append(0, L, b, pos)                                  # overwrites the last two
    log.rewrite(2)
    s, e = P.random_ranges(g, rng)
    log.append(0, L, s, e)                                    # random ranges over all
    log.rewrite(3)
    log.append(L - 1, L, zero, np.minimum(pos, S).astype(np.int32))  # last layer again
    return log


@pytest.mark.parametrize("g", GEOMS, ids=lambda g: g.name)
def test_batched_restore_matches_oracle(g):
    log = standard_log(g, 101)
    log.check()                                   # fused
    log.check(staging_bytes=log.rep.info()[1])    # staged, everything fits
    log.check(upto=7)                             # snapshot + first deltas only
    log.check(batched=False)                      # the per-record restore agrees
    log.check(slot_bytes=log.rep.info()[1])       # pipelined through a fetcher
    log.check(slot_bytes=min_staging(log), upto=9)


def test_staging_smaller_than_the_log():
    """Staged: launches cut where the staging buffer is full; a record larger
    than the staging buffer (the snapshot here) is restored by itself in layer
    groups."""
    g = GEOMS[0]
    log = standard_log(g, 202)
    snap = log.records[0][4].size
    slab = min_staging(log)
    assert slab < snap
    for stg in (slab, slab + 16, 3 * slab // 2 // 16 * 16, max(snap, slab), 2 * snap):
        log.check(staging_bytes=stg)
        log.check(slot_bytes=stg)
    log.check(slot_bytes=slab, one_stream=True)


def test_many_records_several_launches():
    """More one-token records than one launch takes (128 at batch 2), the
    staged form with a buffer that holds 50 of them."""
    g = Geometry("many", 2, 2, 2, 64, 400, 2, "fp16")
    zero = np.zeros(2, np.int32)
    log = Log(g, 303, ORC.staging_bytes(g, 0, 2, zero, np.full(2, 400, np.int32)))
    pos = np.array([3, 0], np.int32)
    log.append(0, 2, zero, pos)
    for k in range(300):
        act = np.array([1, 1 if k % 5 else 0], np.int32)
        log.append(0, 2, pos, pos + act)
        pos = pos + act
    one = ORC.staging_bytes(g, 0, 2, pos, pos + 1)
    log.check()
    log.check(staging_bytes=50 * one)
    log.check(staging_bytes=log.rep.info()[1])
    log.check(slot_bytes=50 * one)


def test_batch_1024_two_records_per_launch():
    g = Geometry("b1024", 2, 1024, 1, 64, 24, 2, "fp16")
    rng = np.random.default_rng(404)
    zero = np.zeros(g.batch, np.int32)
    log = Log(g, 404, 3 * ORC.staging_bytes(g, 0, 2, zero, np.full(g.batch, 24, np.int32)))
    pos = rng.integers(0, 12, size=g.batch).astype(np.int32)
    log.append(0, 2, zero, pos)
    for k in range(7):
        act = (rng.random(g.batch) < 0.8).astype(np.int32)
        log.append(0, 2, pos, pos + act)
        pos = pos + act
    log.rewrite(5)
    log.append(0, 2, np.maximum(pos - 1, 0).astype(np.int32), pos)
    log.check()
    log.check(staging_bytes=max(min_staging(log), log.rep.info()[1] // 3 // 16 * 16))


def test_overlapping_deltas_later_wins():
    """Every record rewrites the same token of every sequence with new bytes:
    no two records can share a launch, and the last one must win."""
    g = Geometry("same", 2, 3, 2, 128, 16, 2, "bf16")
    pos = np.array([4, 9, 15], np.int32)
    log = Log(g, 505, 16 * ORC.staging_bytes(g, 0, 2, pos, pos + 1))
    for k in range(10):
        log.rewrite(10 + k)
        log.append(0, 2, pos, pos + 1)
    log.check()
    log.check(staging_bytes=ORC.staging_bytes(g, 0, 2, pos, pos + 1))
    log.check(slot_bytes=ORC.staging_bytes(g, 0, 2, pos, pos + 1))


def test_errors_enqueue_nothing():
    g = GEOMS[0]
    log = standard_log(g, 606)
    torch.cuda.synchronize()
    z = H.device_cache(g, fill="zero")
    with pytest.raises(dv.DvError) as ei:       # a record larger than staging needs a slab
        log.rep.restore_batched(z, staging=H.device_bytes(min_staging(log) - 16))
    assert ei.value.status == dv.DV_ERR_BUFFER_TOO_SMALL
    small = min_staging(log) - 16                # ... and so does a fetcher's slot
    f = dv.Fetcher(H.device_bytes(small), H.device_bytes(small))
    with pytest.raises(dv.DvError) as ei:
        log.rep.restore_fetched(z, f)
    assert ei.value.status == dv.DV_ERR_BUFFER_TOO_SMALL
    f.close()
    other = Geometry("other", 3, 5, 2, 128, 300, 2, "fp16")  # records do not fit this cache
    zo = H.device_cache(other, fill="zero")
    with pytest.raises(dv.DvError) as ei:
        log.rep.restore_batched(zo)
    assert ei.value.status == dv.DV_ERR_INVALID_ARG
    assert not H.to_np(z.k).any() and not H.to_np(z.v).any()
    assert not H.to_np(zo.k).any() and not H.to_np(zo.v).any()


def decode_run_log(g, seed, steps, finish_at=None, rng=None):
    """Snapshot, then `steps` one-token deltas of every live sequence (a run of
    one-token records for the run kernel); at step `finish_at` every third
    sequence finishes (the run breaks and a new one starts with fewer
    sequences)."""
    rng = rng or np.random.default_rng(seed)
    B, S, L = g.batch, g.max_seq, g.num_layers
    zero = np.zeros(B, np.int32)
    pos = rng.integers(0, S - steps, size=B).astype(np.int32)
    full = ORC.staging_bytes(g, 0, L, zero, np.full(B, S, np.int32))
    log = Log(g, seed, 2 * full)
    log.append(0, L, zero, pos)
    live = np.ones(B, bool)
    for k in range(steps):
        if finish_at is not None and k == finish_at:
            live[::3] = False
            if not live.any():
                live[-1] = True
        act = live.astype(np.int32)
        log.append(0, L, pos, pos + act)
        pos = pos + act
    return log


RUN_GEOMS = GEOMS + [
    Geometry("c16-long", 2, 3, 2, 128, 400, 2, "bf16"),   # TB = 64: runs over several blocks
    Geometry("c8-long", 2, 2, 3, 64, 400, 2, "fp16"),     # TB = 128
]


@pytest.mark.parametrize("g", RUN_GEOMS, ids=lambda g: g.name)
def test_runs_of_one_token_records(g):
    """Runs of one-token decode deltas (the run kernel): long runs crossing
    token blocks, a run broken where sequences finish, fused, staged with a
    buffer that cuts the runs into pieces of 37 records, and through a
    fetcher whose slots hold 37 or 1 records."""
    steps = min(g.max_seq - 2, 150)
    log = decode_run_log(g, 707, steps, finish_at=steps // 3)
    one = log.records[1][4].size
    log.check()
    log.check(staging_bytes=log.rep.info()[1])
    log.check(staging_bytes=max(min_staging(log), 37 * one))
    log.check(slot_bytes=max(min_staging(log), 37 * one))
    log.check(slot_bytes=max(min_staging(log), one), upto=20)
    log.check(upto=steps // 3 + 5)


@pytest.mark.parametrize("g", [Geometry("runlen16", 2, 4, 2, 128, 720, 2, "fp16"),
                               Geometry("runlen8", 2, 4, 3, 64, 720, 2, "bf16")],
                         ids=["C16", "C8"])
def test_run_lengths_around_the_token_block(g):
    """Runs of every length near the tile's token block (64 tokens at head_dim
    128, 128 at 64, in 2-byte elements) and near half of it (the longest run
    in grouped tiles), each followed by a record that breaks the run."""
    B = g.batch
    zero = np.zeros(B, np.int32)
    log = Log(g, 808, 2 * ORC.staging_bytes(g, 0, 2, zero, np.full(B, g.max_seq, np.int32)))
    pos = np.array([0, 5, 63, 64], np.int32)
    for n in (1, 2, 3, 5, 17, 32, 33, 63, 64, 65, 127, 129):
        for k in range(n):
            log.append(0, 2, pos, pos + 1)
            pos = pos + 1
        log.append(0, 2, pos, pos + np.array([1, 0, 1, 0], np.int32))   # breaks the run
        pos = pos + np.array([1, 0, 1, 0], np.int32)
    assert pos.max() <= g.max_seq
    log.check()
    log.check(staging_bytes=log.rep.info()[1])


@pytest.mark.parametrize("where", ["device", "host"])
def test_unpack_records_matches_oracle(where):
    """dv_kv_unpack_records of a log held in device memory or pinned host
    memory: the standard log (snapshot, deltas, ragged, empty and overlapping
    records) and a decode run, against the oracle's in-order unpack."""
    for g, log in ((GEOMS[0], standard_log(GEOMS[0], 909)),
                   (GEOMS[1], decode_run_log(GEOMS[1], 910, 90, finish_at=40))):
        records = [(l0, l1, s, e) for l0, l1, s, e, _ in log.records]
        data = np.concatenate([d for *_, d in log.records])
        src = torch.from_numpy(data)
        src = src.cuda() if where == "device" else src.pin_memory()
        z = H.device_cache(g, fill="zero")
        torch.cuda.synchronize()
        dv.dv_kv_unpack_records(z, records, src)
        kw, vw = ORC.restore(g, log.records)
        assert np.array_equal(H.to_np(z.k), kw), g.name
        assert np.array_equal(H.to_np(z.v), vw), g.name


def test_unpack_records_errors_enqueue_nothing():
    g = GEOMS[0]
    log = decode_run_log(g, 911, 20)
    records = [(l0, l1, s, e) for l0, l1, s, e, _ in log.records]
    data = torch.from_numpy(np.concatenate([d for *_, d in log.records])).cuda()
    z = H.device_cache(g, fill="zero")
    torch.cuda.synchronize()
    with pytest.raises(dv.DvError) as ei:          # one byte short
        dv.dv_kv_unpack_records(z, records, data, src_bytes=data.numel() - 16)
    assert ei.value.status == dv.DV_ERR_BUFFER_TOO_SMALL
    bad = list(records)
    l0, l1, s, e = bad[5]
    bad[5] = (l0, l1, s, e + g.max_seq)            # a range past the cache
    with pytest.raises(dv.DvError) as ei:
        dv.dv_kv_unpack_records(z, bad, data)
    assert ei.value.status == dv.DV_ERR_RANGE
    assert not H.to_np(z.k).any() and not H.to_np(z.v).any()
    dv.dv_kv_unpack_records(z, [], None)           # nothing to do


def test_fetched_restore_in_parts_matches_the_whole():
    """dv_replica_restore_fetched_steps: the log restored in consecutive step
    ranges into the same cache (the snapshot, the first deltas, the rest)
    equals the oracle's in-order restore of the whole log, and a range that
    stops short leaves the later records out."""
    for g, log in ((GEOMS[0], standard_log(GEOMS[0], 111)),
                   (RUN_GEOMS[-2], decode_run_log(RUN_GEOMS[-2], 112, 120, finish_at=50))):
        n = len(log.records)
        slot = max(min_staging(log), 64 << 10)
        cs = torch.cuda.Stream()
        f = dv.Fetcher(H.device_bytes(slot), H.device_bytes(slot), cs, torch.cuda.Stream())
        for cuts in ((1, n // 2), (3, 4, n - 1), (n,)):
            z = H.device_cache(g, fill="zero")
            torch.cuda.synchronize()
            lo = 0
            for hi in cuts + (n,):
                log.rep.restore_fetched(z, f, upto_step=hi, from_step=lo)
                lo = hi
            f.wait()
            kw, vw = ORC.restore(g, log.records)
            assert np.array_equal(H.to_np(z.k), kw), (g.name, cuts)
            assert np.array_equal(H.to_np(z.v), vw), (g.name, cuts)
        z = H.device_cache(g, fill="zero")
        torch.cuda.synchronize()
        log.rep.restore_fetched(z, f, upto_step=n // 2, from_step=2)
        f.wait()
        kw, vw = ORC.restore(g, log.records[2:n // 2])
        assert np.array_equal(H.to_np(z.k), kw) and np.array_equal(H.to_np(z.v), vw)
        f.close()
