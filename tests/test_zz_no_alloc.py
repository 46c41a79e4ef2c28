"""dv_swap_out_noalloc: the swap-out for callers that cannot allocate device
memory (a host embedding the library without a device allocator of its own,
or a process whose device memory another allocator owns entirely).  Its
staging is libdv's built-in 64 MiB device buffer.  Its output must be the
bytes dv_swap_out leaves, exactly, call after call, and the oracle's; a call
must not change the device's free memory.

This file is collected last on purpose, so that a run stopping at its first
failure has already run every other test; it also passes when run alone."""
import numpy as np
import pytest
import torch

import kv_cache_streaming_gb300 as dv
import oracle
from synth.configs import Geometry
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu
ORC = oracle.default()

# Layer slabs of about 50 MB: one layer per group of the 64 MiB buffer, so a
# swap of 10 layers goes through the buffer 10 times, in order.
G = Geometry("noalloc", 10, 8, 16, 128, 1024, 2, "fp16")
# Layer slabs of a few MB: several layers per group, in two halves.
SMALL = Geometry("noalloc-small", 12, 4, 16, 128, 512, 2, "bf16")


def _ranges(g, rng, lo, hi):
    s = rng.integers(0, lo, size=g.batch).astype(np.int32)
    e = rng.integers(hi, g.max_seq + 1, size=g.batch).astype(np.int32)
    return s, e


@pytest.mark.parametrize("g, l0, l1, seed", [(G, 0, 10, 31), (SMALL, 3, 11, 32)],
                         ids=["one-layer-groups", "multi-layer-groups"])
def test_noalloc_swap_out_matches_swap_out_and_the_oracle_on_two_calls(g, l0, l1, seed):
    rng = np.random.default_rng(2024 + seed)
    kh, vh = H.host_cache(g, seed)
    cache = H.device_cache(g, fill=(kh, vh))
    stream = torch.cuda.current_stream()
    lo, hi = (100, 600) if g is G else (50, 200)
    calls = [_ranges(g, rng, lo, hi), _ranges(g, rng, lo, hi)]
    outs = []
    for s, e in calls:
        n = dv.dv_staging_bytes(cache, l0, l1, s, e)
        slab = n // (l1 - l0)
        if g is G:
            assert 32 << 20 < slab <= dv.DV_NOALLOC_STAGING_BYTES  # one layer per group
        else:
            assert 2 * slab <= dv.DV_NOALLOC_STAGING_BYTES // 2     # layers share each half
        host = H.pinned(n, fill=0xCD)
        dv.dv_swap_out_noalloc(cache, l0, l1, s, e, host, stream=stream)
        outs.append((s, e, n, host))
    torch.cuda.synchronize()
    for s, e, n, host in outs:
        want = H.pinned(n, fill=0x00)
        dv.dv_swap_out(cache, l0, l1, s, e, want, staging=None, stream=stream)
        torch.cuda.synchronize()
        assert torch.equal(host[:n], want[:n])
        assert np.array_equal(host[:n].numpy(), ORC.pack(g, kh, vh, l0, l1, s, e))


def test_noalloc_call_leaves_free_device_memory_unchanged():
    """After a first call (which looks up the buffer's address and may set up
    the copy stream), a call changes neither the device's free memory nor
    torch's reserved memory: nothing is allocated for it."""
    rng = np.random.default_rng(77)
    cache = H.device_cache(SMALL, fill="synth", seed=33)
    s, e = _ranges(SMALL, rng, 50, 200)
    n = dv.dv_staging_bytes(cache, 0, SMALL.num_layers, s, e)
    host = H.pinned(n)
    dv.dv_swap_out_noalloc(cache, 0, SMALL.num_layers, s, e, host)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    reserved0 = torch.cuda.memory_reserved()
    for _ in range(3):
        dv.dv_swap_out_noalloc(cache, 0, SMALL.num_layers, s, e, host)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert torch.cuda.memory_reserved() == reserved0


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
