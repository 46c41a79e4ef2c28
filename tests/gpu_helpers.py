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



_TORCH_VIEW = {1: torch.uint8, 2: torch.int16, 4: torch.int32}
_NP_VIEW = {1: np.uint8, 2: np.uint16, 4: np.uint32}


def sampled_check(orc, g, seed, staging, l0, l1, s, e, rng, nsamples=200_000):
    """Compares sampled elements of a staging buffer (device or pinned host
    tensor) with the values the oracle's nest and the seeded generator give
    for the cache element held at each offset."""
    n_bytes = orc.staging_bytes(g, l0, l1, s, e)
    n = n_bytes // g.elem_bytes
    if n == 0:
        return 0
    offs = np.unique(np.concatenate([rng.integers(0, n, size=min(nsamples, n)),
                                     np.array([0, n - 1])]))
    kv, idx = orc.source_of(g, l0, l1, s, e, offs)
    want_k = synth.fill_elements(seed, 0, idx, g.elem_bytes, g.kind)
    want_v = synth.fill_elements(seed, 1, idx, g.elem_bytes, g.kind)
    want = np.where(kv == 0, want_k, want_v)
    flat = staging[:n_bytes].view(_TORCH_VIEW[g.elem_bytes])
    got = flat[torch.from_numpy(offs).to(flat.device)].cpu().numpy().view(_NP_VIEW[g.elem_bytes])
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, f"{bad.size} of {offs.size} sampled elements differ (first offset " \
                          f"{offs[bad[0]] if bad.size else -1})"
    return offs.size


def cache_views(g, cache):
    """K as [L, B, H, D/x, S, x] and V as [L, B, H, S, D] views (element
    dtype of the cache's width) of a dense-layered cache."""
    x = 16 // g.elem_bytes
    dt = _TORCH_VIEW[g.elem_bytes]
    L, B, H, D, S = g.num_layers, g.batch, g.num_heads, g.head_dim, g.max_seq
    k = cache.k.view(dt).view(L, g.layer_elems)[:, :B * H * D * S].view(L, B, H, D // x, S, x)
    v = cache.v.view(dt).view(L, g.layer_elems)[:, :B * H * D * S].view(L, B, H, S, D)
    return k, v


def assert_prefix_equal_rest_zero(g, got, want, lengths):
    """got == want on tokens [0, len_b) of every sequence, zero beyond."""
    gk, gv = cache_views(g, got)
    wk, wv = cache_views(g, want)
    for b, n in enumerate(lengths):
        n = int(n)
        assert torch.equal(gk[:, b, :, :, :n, :], wk[:, b, :, :, :n, :]), f"K of sequence {b}"
        assert torch.equal(gv[:, b, :, :n, :], wv[:, b, :, :n, :]), f"V of sequence {b}"
        assert not gk[:, b, :, :, n:, :].any(), f"K of sequence {b} written past {n}"
        assert not gv[:, b, :, n:, :].any(), f"V of sequence {b} written past {n}"
