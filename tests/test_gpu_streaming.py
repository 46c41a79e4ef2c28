"""Decode deltas streamed beside the compute (dv_delta_streamer; §3 "Token
computation and streaming parallelization", Fig 7c) against the oracle.  A
decode step is a stand-in compute (a read of the whole cache) and the write of
one seeded token per live sequence; the step's delta goes to the replica on a
side stream that waits only for that step's write.  The host model is the
seeded cache with every write applied by the oracle's unpack: each streamed
record must be the oracle's pack of the model's token, and the replica must
restore to the oracle's in-order restore.  Fused and staged appends, eager and
captured in a CUDA graph."""
import numpy as np
import pytest
import torch

import kv_cache_streaming_gb300 as dv
import oracle
import synth
from synth import gpu as synth_gpu
from synth.configs import Geometry
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu
ORC = oracle.default()

G = Geometry("tokstream", 4, 5, 3, 128, 96, 2, "bf16")


def decode_steps(cache, ds, kh, vh, pos, steps, compute, salt):
    """Enqueues `steps` decode steps on `compute`, each streamed through `ds`;
    applies the same writes to the host model; returns the steps' ranges."""
    g, L = G, G.num_layers
    ranges = []
    for i in range(steps):
        act = (np.arange(g.batch) + i) % 4 != 0          # a different sequence rests each step
        e = (pos + act).astype(np.int32)
        nt = ORC.staging_bytes(g, 0, L, pos, e)
        with torch.cuda.stream(compute):
            tok = H.device_bytes(nt)   # allocated on the stream that uses it
            _ = cache.k.view(torch.int32).sum() + cache.v.view(torch.int32).sum()
            synth_gpu.fill_tensor(tok[:nt], salt + i, 0, g.kind, compute)
            dv.dv_kv_unpack(cache, 0, L, pos, e, tok, stream=compute, src_bytes=nt)
        ORC.unpack(g, kh, vh, 0, L, pos, e, synth.fill_bytes(salt + i, 0, nt, g.kind))
        ds.stream(cache, 0, L, pos, e, step=i)
        ranges.append((pos.copy(), e))
        pos = e
    return ranges


def check_replica(rep, arena, kh, vh, ranges, snapshot):
    g, L = G, G.num_layers
    off = snapshot[4].size
    assert np.array_equal(arena[:off].numpy(), snapshot[4])
    recs = [snapshot]
    for s, e in ranges:
        want = ORC.pack(g, kh, vh, 0, L, s, e)
        assert np.array_equal(arena[off:off + want.size].numpy(), want)
        recs.append((0, L, s, e, want))
        off += want.size
    assert rep.info() == (1 + len(ranges), off)
    z = H.device_cache(g, fill="zero")
    rep.restore_batched(z)
    kw, vw = ORC.restore(g, recs)
    assert np.array_equal(H.to_np(z.k), kw) and np.array_equal(H.to_np(z.v), vw)


def setup(seed):
    g = G
    kh, vh = H.host_cache(g, seed)
    cache = H.device_cache(g, fill=(kh.copy(), vh.copy()))
    zs = np.zeros(g.batch, np.int32)
    pos = np.array([10, 3, 40, 0, 25], np.int32)
    snap = ORC.pack(g, kh, vh, 0, g.num_layers, zs, pos)
    arena = H.pinned(ORC.staging_bytes(g, 0, g.num_layers, zs, np.full(g.batch, g.max_seq,
                                                                       np.int32)))
    rep = dv.Replica(arena, g.batch)
    rep.append(cache, 0, g.num_layers, zs, pos, step=-1)
    torch.cuda.synchronize()
    return kh, vh, cache, pos, arena, rep, (0, g.num_layers, zs, pos.copy(), snap)


@pytest.mark.parametrize("staged", [False, True], ids=["fused", "staged"])
def test_streamed_deltas_match_the_oracle(staged):
    kh, vh, cache, pos, arena, rep, snap = setup(801)
    compute, side = torch.cuda.Stream(), torch.cuda.Stream()
    staging = H.device_bytes(1 << 20) if staged else None
    ds = dv.DeltaStreamer(rep, compute, side, staging)
    ranges = decode_steps(cache, ds, kh, vh, pos, 20, compute, 9100)
    ds.join()
    ds.wait()
    torch.cuda.synchronize()
    check_replica(rep, arena, kh, vh, ranges, snap)
    ds.close()


def test_streamed_deltas_in_a_cuda_graph():
    """The decode loop with its streaming captured in one CUDA graph on the
    compute stream and replayed: the replica holds the oracle's deltas."""
    kh, vh, cache, pos, arena, rep, snap = setup(802)
    compute, side = torch.cuda.Stream(), torch.cuda.Stream()
    ds = dv.DeltaStreamer(rep, compute, side)
    # an eager round first (occupancy queries, lazy loading), then back to the snapshot
    kh0, vh0 = kh.copy(), vh.copy()
    decode_steps(cache, ds, kh, vh, pos, 2, compute, 9200)
    ds.join()
    torch.cuda.synchronize()
    rep.truncate(0)
    cache.k.copy_(torch.from_numpy(kh0))
    cache.v.copy_(torch.from_numpy(vh0))
    kh, vh = kh0, vh0
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=compute, capture_error_mode="relaxed"):
        ranges = decode_steps(cache, ds, kh, vh, pos, 12, compute, 9300)
        ds.join()
    graph.replay()
    torch.cuda.synchronize()
    check_replica(rep, arena, kh, vh, ranges, snap)
    ds.close()


def test_delta_streamer_errors():
    kh, vh, cache, pos, arena, rep, snap = setup(803)
    s = torch.cuda.Stream()
    with pytest.raises(dv.DvError) as ei:              # the side stream is the compute stream
        dv.DeltaStreamer(rep, s, s)
    assert ei.value.status == dv.DV_ERR_INVALID_ARG
    ds = dv.DeltaStreamer(rep, s, torch.cuda.Stream(), H.device_bytes(256))
    with pytest.raises(dv.DvError) as ei:              # staging smaller than a layer slab
        ds.stream(cache, 0, G.num_layers, pos, pos + 1, step=0)
    assert ei.value.status == dv.DV_ERR_BUFFER_TOO_SMALL
    ds.close()
    ds = dv.DeltaStreamer(rep, s, torch.cuda.Stream())
    with pytest.raises(dv.DvError) as ei:              # steps must not go back
        ds.stream(cache, 0, G.num_layers, pos, pos + 1, step=-5)
    assert ei.value.status == dv.DV_ERR_INVALID_ARG
    assert rep.info()[0] == 1
    ds.join()
    ds.wait()
    ds.close()
