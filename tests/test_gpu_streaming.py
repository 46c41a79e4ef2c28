"""Decode-delta streaming overlapped with the next step's compute: the host
replica must hold exactly the tokens the decode steps wrote, in every
scheduling mode (inline on the compute stream, or on a side stream that
waits only for its own step's write)."""
import sys
from pathlib import Path

import pytest
import torch

import kv_cache_streaming_gb300 as dv

sys.path.insert(0, str(Path(__file__).resolve().parent.parent))
import bench  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode", ["inline", "overlapped"])
def test_streamed_deltas_equal_written_tokens(mode):
    ds = bench.DecodeStreaming(torch, dv, steps=6)
    ds.host.fill_(0)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        ds.run(mode, s)
    torch.cuda.synchronize()
    assert torch.equal(ds.host.cuda(), ds.tokens)
    # and the cache holds the written tokens: pack them back
    back = torch.empty_like(ds.tokens)
    for i, (a, b) in enumerate(ds.deltas[:6]):
        dv.dv_kv_pack(ds.cache, 0, ds.g.num_layers, a, b, back[i * ds.dsz:(i + 1) * ds.dsz])
    torch.cuda.synchronize()
    assert torch.equal(back, ds.tokens)
