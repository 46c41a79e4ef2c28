"""Splitting a cache at the source and merging blocks at the target through
the ABI's layer and per-sequence ranges ("DejaVu: KV-Cache Streaming...",
§3 DejaVuLib primitives, Table 1 stream_out / stream_in: the cache is split
by the pipeline setting at the source, or blocks are merged at the target).

Two cases, each compared with the oracle byte for byte:
- a prompt worker's cache split by layer range (pipeline stages) and by
  sequence subset (microbatches), each piece one pack; the pieces unpacked
  into one target cache give back the source's slices and touch nothing else;
- two prompt workers of batch 3 merged into one token worker of batch 6: a
  source's staging bytes are the bytes the target's ranges ask for when the
  target's ranges select that source's sequences and leave the rest empty."""
import numpy as np
import pytest

import kv_cache_streaming_gb300 as dv
import oracle
from synth.configs import Geometry
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu
ORC = oracle.default()


def _pack(g, cache, kh, vh, l0, l1, s, e):
    n = ORC.staging_bytes(g, l0, l1, s, e)
    buf = H.device_bytes(n)
    dv.dv_kv_pack(cache, l0, l1, s, e, buf)
    got = H.to_np(buf)[:n]
    assert np.array_equal(got, ORC.pack(g, kh, vh, l0, l1, s, e))
    return buf, n


def test_split_by_stage_and_microbatch_then_merge():
    g = Geometry("split", 4, 6, 3, 64, 96, 2, "fp16")
    kh, vh = H.host_cache(g, 41)
    src = H.device_cache(g, fill=(kh, vh))
    s = np.array([0, 3, 0, 10, 0, 7], np.int32)
    e = np.array([80, 50, 96, 11, 1, 60], np.int32)
    even = np.arange(g.batch) % 2 == 0
    pieces = []  # (l0, l1, starts, ends): stage x microbatch
    for l0, l1 in ((0, 2), (2, 4)):
        for mask in (even, ~even):
            pieces.append((l0, l1, np.where(mask, s, 0).astype(np.int32),
                           np.where(mask, e, 0).astype(np.int32)))
    dst = H.device_cache(g, fill=0x5A)
    kw = np.full(g.tensor_bytes, 0x5A, np.uint8)
    vw = np.full(g.tensor_bytes, 0x5A, np.uint8)
    total = 0
    for l0, l1, ps, pe in pieces:
        buf, n = _pack(g, src, kh, vh, l0, l1, ps, pe)
        dv.dv_kv_unpack(dst, l0, l1, ps, pe, buf, src_bytes=n)
        ORC.unpack(g, kw, vw, l0, l1, ps, pe, ORC.pack(g, kh, vh, l0, l1, ps, pe))
        total += n
    # the pieces together are the whole selection, once
    assert total == ORC.staging_bytes(g, 0, g.num_layers, s, e)
    assert np.array_equal(H.to_np(dst.k), kw) and np.array_equal(H.to_np(dst.v), vw)
    # merged, the target holds the source's selected slices
    back = H.device_bytes(total)
    dv.dv_kv_pack(dst, 0, g.num_layers, s, e, back)
    assert np.array_equal(H.to_np(back)[:total], ORC.pack(g, kh, vh, 0, g.num_layers, s, e))


def test_two_prompt_workers_merge_into_a_larger_batch():
    small = Geometry("prompt", 3, 3, 4, 128, 64, 2, "bf16")
    big = Geometry("token", 3, 6, 4, 128, 64, 2, "bf16")
    srcs = [H.host_cache(small, 51), H.host_cache(small, 52)]
    ranges = [(np.array([0, 0, 5], np.int32), np.array([40, 64, 9], np.int32)),
              (np.array([0, 2, 0], np.int32), np.array([1, 30, 64], np.int32))]
    dst = H.device_cache(big, fill=0x00)
    kw = np.zeros(big.tensor_bytes, np.uint8)
    vw = np.zeros(big.tensor_bytes, np.uint8)
    for w, ((kh, vh), (s, e)) in enumerate(zip(srcs, ranges)):
        cache = H.device_cache(small, fill=(kh, vh))
        buf, n = _pack(small, cache, kh, vh, 0, small.num_layers, s, e)
        # the target's ranges: this worker's sequences at batch slots 3w..3w+2
        ts = np.zeros(big.batch, np.int32)
        te = np.zeros(big.batch, np.int32)
        ts[3 * w:3 * w + 3] = s
        te[3 * w:3 * w + 3] = e
        assert dv.dv_staging_bytes(dst, 0, big.num_layers, ts, te) == n
        dv.dv_kv_unpack(dst, 0, big.num_layers, ts, te, buf, src_bytes=n)
        ORC.unpack(big, kw, vw, 0, big.num_layers, ts, te,
                   ORC.pack(small, kh, vh, 0, small.num_layers, s, e))
    assert np.array_equal(H.to_np(dst.k), kw) and np.array_equal(H.to_np(dst.v), vw)
