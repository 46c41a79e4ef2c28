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


def layer_geometry(g):
    """The one-layer geometry of g's layers (the oracle's unit of work for
    full-size comparisons, layer by layer)."""
    from dataclasses import replace
    return replace(g, name=g.name + "-layer", num_layers=1)


def host_layer(g, seed, l, threads=4):
    """Bytes of layer l of the seeded cache of geometry g (K, V), computed on
    the host: the generator's fill of the tensor from layer l's first byte."""
    lb = g.layer_elems * g.elem_bytes
    g1 = layer_geometry(g)
    return (synth.fill_bytes(seed, 0, g1.tensor_bytes, g.kind, offset=l * lb, threads=threads),
            synth.fill_bytes(seed, 1, g1.tensor_bytes, g.kind, offset=l * lb, threads=threads))


def layer_workers(per_worker_bytes, most=4):
    """How many layers to compare at once: up to `most`, as host memory
    allows (MemAvailable, with a quarter kept free)."""
    avail = 0
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    avail = int(line.split()[1]) * 1024
    except OSError:
        pass
    return max(1, min(most, int(0.75 * avail) // max(per_worker_bytes, 1)))


def for_each_layer(fn, layers, per_worker_bytes):
    """Runs fn(l) for every layer in `layers`, several at once on threads (the
    oracle's C calls and numpy release the interpreter lock); re-raises the
    first failure."""
    from concurrent.futures import ThreadPoolExecutor
    workers = layer_workers(per_worker_bytes)
    if workers == 1:
        for l in layers:
            fn(l)
        return
    with ThreadPoolExecutor(workers) as ex:
        for r in [ex.submit(fn, l) for l in layers]:
            r.result()


def device_layer(g, cache, l):
    """Layer l of a device cache (K, V bytes) copied to host numpy arrays."""
    lb = g.layer_elems * g.elem_bytes
    return (cache.k[l * lb:(l + 1) * lb].cpu().numpy(),
            cache.v[l * lb:(l + 1) * lb].cpu().numpy())
