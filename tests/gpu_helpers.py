"""Shared helpers of the GPU tests: cache allocation, seeded fills, and
host copies for comparison with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import kv_cache_streaming_gb300 as dv
import synth
from synth import gpu as synth_gpu


def device_cache(g, fill=None, seed=0, device="cuda"):
    """A cache of geometry ``g`` on the GPU.  fill: None (uninitialised),
    'zero', a byte value (int), 'synth' (seeded generator on the GPU), or a
    (k_bytes, v_bytes) pair of host numpy arrays to upload."""
    k = torch.empty(g.tensor_bytes, dtype=torch.uint8, device=device)
    v = torch.empty(g.tensor_bytes, dtype=torch.uint8, device=device)
    if fill == "zero":
        k.zero_()
        v.zero_()
    elif isinstance(fill, int):
        k.fill_(fill)
        v.fill_(fill)
    elif fill == "synth":
        synth_gpu.fill_cache(g, k, v, seed)
    elif isinstance(fill, tuple):
        k.copy_(torch.from_numpy(fill[0]))
        v.copy_(torch.from_numpy(fill[1]))
    return dv.Cache.from_geometry(g, k, v)


def host_cache(g, seed):
    """The seeded cache bytes computed on the host (numpy generator)."""
    return (synth.fill_bytes(seed, 0, g.tensor_bytes, g.kind),
            synth.fill_bytes(seed, 1, g.tensor_bytes, g.kind))


def to_np(t):
    torch.cuda.synchronize()
    return t.detach().cpu().numpy().reshape(-1).view(np.uint8)


def pinned(nbytes, fill=None):
    t = torch.empty(max(nbytes, 16), dtype=torch.uint8, pin_memory=True)
    if fill is not None:
        t.fill_(fill)
    return t


def device_bytes(nbytes, fill=None):
    t = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda")
    if fill is not None:
        t.fill_(fill)
    return t

