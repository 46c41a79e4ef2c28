"""The pack and unpack calls inside a CUDA graph captured in torch's default
(global) capture mode, as a serving engine captures its decode step: the
replayed graph moves the same bytes as the eager calls."""
import numpy as np
import pytest
import torch

import kv_cache_streaming_gb300 as dv
import oracle
from synth.configs import Geometry
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu
ORC = oracle.default()


def test_pack_unpack_in_a_globally_captured_graph():
    g = Geometry("cap", 4, 4, 8, 128, 256, 2, "fp16")
    kh, vh = H.host_cache(g, 91)
    cache = H.device_cache(g, fill=(kh, vh))
    back = H.device_cache(g, fill="zero")
    pos = np.array([10, 200, 0, 77], np.int32)
    e1 = pos + np.array([1, 1, 0, 1], np.int32)          # a decode delta (token kernel)
    s2 = np.zeros(g.batch, np.int32)
    e2 = np.array([100, 256, 3, 64], np.int32)           # ragged prefixes (tile / flat)
    n1 = ORC.staging_bytes(g, 0, g.num_layers, pos, e1)
    n2 = ORC.staging_bytes(g, 0, g.num_layers, s2, e2)
    b1, b2 = H.device_bytes(n1), H.device_bytes(n2)
    host = H.pinned(n1)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):  # eager once (first-use set-up happens here)
        dv.dv_kv_pack(cache, 0, g.num_layers, pos, e1, b1, stream=s)
        dv.dv_kv_pack(cache, 0, g.num_layers, s2, e2, b2, stream=s)
    torch.cuda.synchronize()
    b1.zero_()
    b2.zero_()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):  # default capture_error_mode="global"
        dv.dv_kv_pack(cache, 0, g.num_layers, pos, e1, b1, stream=s)
        dv.dv_kv_pack(cache, 0, g.num_layers, s2, e2, b2, stream=s)
        dv.dv_kv_pack(cache, 0, g.num_layers, pos, e1, host, stream=s)  # zero copy to host
        dv.dv_kv_unpack(back, 0, g.num_layers, s2, e2, b2, stream=s)
        dv.dv_kv_unpack(back, 0, g.num_layers, pos, e1, b1, stream=s)
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    assert np.array_equal(H.to_np(b1)[:n1], ORC.pack(g, kh, vh, 0, g.num_layers, pos, e1))
    assert np.array_equal(H.to_np(b2)[:n2], ORC.pack(g, kh, vh, 0, g.num_layers, s2, e2))
    assert np.array_equal(host.numpy()[:n1], H.to_np(b1)[:n1])
    kw, vw = np.zeros_like(kh), np.zeros_like(vh)
    ORC.unpack(g, kw, vw, 0, g.num_layers, s2, e2, ORC.pack(g, kh, vh, 0, g.num_layers, s2, e2))
    ORC.unpack(g, kw, vw, 0, g.num_layers, pos, e1, ORC.pack(g, kh, vh, 0, g.num_layers, pos, e1))
    assert np.array_equal(H.to_np(back.k), kw) and np.array_equal(H.to_np(back.v), vw)


def test_batched_restore_in_a_globally_captured_graph():
    """dv_replica_restore_batched, fused and staged, captured in global mode:
    each replay restores the snapshot + deltas the oracle's in-order restore
    gives."""
    g = Geometry("caprep", 3, 5, 4, 128, 128, 2, "bf16")
    kh, vh = H.host_cache(g, 93)
    cache = H.device_cache(g, fill=(kh, vh))
    zero = np.zeros(g.batch, np.int32)
    pos = np.array([70, 5, 33, 100, 64], np.int32)
    full = ORC.staging_bytes(g, 0, g.num_layers, zero, np.full(g.batch, g.max_seq, np.int32))
    arena = H.pinned(full)
    rep = dv.Replica(arena, g.batch)
    records = [(0, g.num_layers, zero, pos.copy())]
    rep.append(cache, 0, g.num_layers, zero, pos, step=0)
    for k in range(1, 9):
        act = np.array([1, 1, 0 if k > 4 else 1, 1, 1], np.int32)
        rep.append(cache, 0, g.num_layers, pos, pos + act, step=k)
        records.append((0, g.num_layers, pos.copy(), (pos + act).copy()))
        pos = pos + act
    torch.cuda.synchronize()
    kw, vw = ORC.restore(g, [(a, b, s_, e_, ORC.pack(g, kh, vh, a, b, s_, e_))
                             for a, b, s_, e_ in records])
    fused = H.device_cache(g, fill="zero")
    staged = H.device_cache(g, fill="zero")
    stg = H.device_bytes(rep.info()[1])
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):  # eager once
        rep.restore_batched(fused, stream=s)
        rep.restore_batched(staged, staging=stg, stream=s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        rep.restore_batched(fused, stream=s)
        rep.restore_batched(staged, staging=stg, stream=s)
    for _ in range(2):
        for c in (fused, staged):
            c.k.zero_()
            c.v.zero_()
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        for c in (fused, staged):
            assert np.array_equal(H.to_np(c.k), kw) and np.array_equal(H.to_np(c.v), vw)
    rep.close()


def test_unpack_records_in_a_globally_captured_graph():
    """dv_kv_unpack_records of a device-resident log (a snapshot, a run of
    one-token deltas, a ragged record) captured in global mode: each replay
    gives the oracle's in-order restore."""
    g = Geometry("caplog", 2, 4, 3, 128, 200, 2, "fp16")
    kh, vh = H.host_cache(g, 95)
    zero = np.zeros(g.batch, np.int32)
    pos = np.array([50, 7, 120, 90], np.int32)
    records = [(0, g.num_layers, zero, pos.copy())]
    for k in range(40):
        records.append((0, g.num_layers, pos.copy(), (pos + 1).astype(np.int32)))
        pos = pos + 1
    records.append((0, g.num_layers, pos.copy(), (pos + np.array([2, 0, 3, 1])).astype(np.int32)))
    data = [ORC.pack(g, kh, vh, a, b, s_, e_) for a, b, s_, e_ in records]
    kw, vw = ORC.restore(g, [(a, b, s_, e_, d) for (a, b, s_, e_), d in zip(records, data)])
    log = torch.from_numpy(np.concatenate(data)).cuda()
    z = H.device_cache(g, fill="zero")
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):  # eager once
        dv.dv_kv_unpack_records(z, records, log, stream=s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        dv.dv_kv_unpack_records(z, records, log, stream=s)
    for _ in range(2):
        z.k.zero_()
        z.v.zero_()
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        assert np.array_equal(H.to_np(z.k), kw) and np.array_equal(H.to_np(z.v), vw)
