"""dv_swap_out_noalloc: the swap-out for callers that cannot allocate device
memory (a host embedding the library without a device allocator of its own,
or a process whose device memory another allocator owns entirely).  Its
staging is libdv's built-in 64 MiB device buffer; its output must be the
bytes dv_swap_out leaves, exactly, call after call.

This file is collected last on purpose, so that a run stopping at its first
failure has already run every other test; it also passes when run alone."""
import numpy as np
import pytest
import torch

import kv_cache_streaming_gb300 as dv
from synth.configs import Geometry
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu

# Layer slabs of about 50 MB: one layer per group of the 64 MiB buffer, so a
# swap of 10 layers goes through the buffer 10 times.
G = Geometry("noalloc", 10, 8, 16, 128, 1024, 2, "fp16")


def _ranges(rng):
    s = rng.integers(0, 100, size=G.batch).astype(np.int32)
    e = rng.integers(600, G.max_seq + 1, size=G.batch).astype(np.int32)
    return s, e


def test_noalloc_swap_out_matches_swap_out_on_two_calls():
    rng = np.random.default_rng(2024)
    cache = H.device_cache(G, fill="synth", seed=31)
    stream = torch.cuda.current_stream()
    calls = [_ranges(rng), _ranges(rng)]
    outs = []
    for s, e in calls:
        n = dv.dv_staging_bytes(cache, 0, G.num_layers, s, e)
        slab = n // G.num_layers
        assert 32 << 20 < slab <= dv.DV_NOALLOC_STAGING_BYTES  # one layer per group
        host = H.pinned(n, fill=0xCD)
        dv.dv_swap_out_noalloc(cache, 0, G.num_layers, s, e, host, stream=stream)
        outs.append((s, e, n, host))
    torch.cuda.synchronize()
    for s, e, n, host in outs:
        want = H.pinned(n, fill=0x00)
        dv.dv_swap_out(cache, 0, G.num_layers, s, e, want, staging=None, stream=stream)
        torch.cuda.synchronize()
        assert torch.equal(host[:n], want[:n])


def test_noalloc_refuses_a_layer_larger_than_its_buffer():
    big = Geometry("noalloc-big", 2, 8, 20, 128, 8192, 2, "fp16")
    cache = dv.Cache.from_geometry(big, 0x1000, 0x2000)  # refused before any pointer is used
    s = np.zeros(big.batch, np.int32)
    e = np.full(big.batch, big.max_seq, np.int32)
    assert dv.dv_staging_bytes(cache, 0, 1, s, e) > dv.DV_NOALLOC_STAGING_BYTES
    with pytest.raises(dv.DvError) as ei:
        dv.dv_swap_out_noalloc(cache, 0, 2, s, e, (0x3000, 1 << 40), stream=0)
    assert ei.value.status == dv.DV_ERR_BUFFER_TOO_SMALL
    assert "built-in" in str(ei.value)
