"""Microbatch swapping through two device caches (dv_swapper; §3 "Microbatch
swapping", Fig 9) against the oracle.  Each microbatch has a host model: the
seeded cache computed on the host, with every decode write applied by the
oracle's unpack, and the list of records its replica should hold (the
oracle's pack of its prompt, then each step's written token).  After every
acquire the cache the swapper hands out must hold the model's bytes on the
microbatch's used prefix, and at the end each replica must restore to the
oracle's in-order restore of the model's records.  Also: the pipelined form
(no host wait between steps), one and two microbatches (no swap after the
first), and the errors."""
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

G = Geometry("mbswap", 3, 6, 4, 128, 160, 2, "fp16")


class Microbatch:
    def __init__(self, g, seed, p, o, rounds):
        self.g, self.p, self.o = g, p, o
        zs = np.zeros(g.batch, np.int32)
        self.kh, self.vh = H.host_cache(g, seed)
        self.lens = p.copy()
        snap = ORC.pack(g, self.kh, self.vh, 0, g.num_layers, zs, p)
        self.records = [(0, g.num_layers, zs, p.copy(), snap)]
        cap = ORC.staging_bytes(g, 0, g.num_layers, zs, p + rounds) + 4096
        self.arena = H.pinned(cap)
        self.rep = dv.Replica(self.arena, g.batch)
        src = H.device_cache(g, fill=(self.kh, self.vh))
        self.rep.append(src, 0, g.num_layers, zs, p, step=0)
        torch.cuda.synchronize()
        del src

    def used_bytes_match(self, cache):
        """The device cache holds the model's bytes on [0, lens) of every
        sequence (compared as the oracle's pack of the model against the
        GPU's pack of the cache)."""
        g = self.g
        zs = np.zeros(g.batch, np.int32)
        n = ORC.staging_bytes(g, 0, g.num_layers, zs, self.lens)
        got = H.device_bytes(n)
        dv.dv_kv_pack(cache, 0, g.num_layers, zs, self.lens, got)
        want = ORC.pack(g, self.kh, self.vh, 0, g.num_layers, zs, self.lens)
        return np.array_equal(H.to_np(got)[:n], want)


def make_microbatches(n, rounds, seed=500):
    rng = np.random.default_rng(seed)
    out = []
    for m in range(n):
        p = rng.integers(8, G.max_seq - rounds - 8, size=G.batch).astype(np.int32)
        o = rng.integers(0, rounds + 2, size=G.batch).astype(np.int32)  # some finish early
        out.append(Microbatch(G, seed + m, p, o, rounds))
    return out


def run_rounds(mbs, rounds, check_each_step, compute, swap, fetch_streams, prefetch=True):
    """rounds x N steps through a swapper; returns the swapper's two caches."""
    g, L = G, G.num_layers
    caches = [H.device_cache(g, fill="zero") for _ in range(2)]
    slot_bytes = max(ORC.staging_bytes(g, 0, 1, np.zeros(g.batch, np.int32), mb.p + rounds)
                     for mb in mbs)
    slot_bytes = (slot_bytes + 15) // 16 * 16
    f = dv.Fetcher(H.device_bytes(slot_bytes), H.device_bytes(slot_bytes), *fetch_streams)
    torch.cuda.synchronize()
    sw = dv.Swapper(caches[0], caches[1], f, compute, swap)
    order = [m for _ in range(rounds) for m in range(len(mbs))]
    for i, m in enumerate(order):
        mb = mbs[m]
        slot = sw.acquire(mb.rep)
        if prefetch and i + 1 < len(order):
            sw.prefetch(mbs[order[i + 1]].rep)
        cache = caches[slot]
        if check_each_step:
            torch.cuda.synchronize()
            assert mb.used_bytes_match(cache), f"step {i}: microbatch {m} swapped in wrong"
        # the step: a stand-in compute (a read of the cache) and the decode write
        ln = mb.lens
        act = ((ln - mb.p) < mb.o).astype(np.int32)
        nt = ORC.staging_bytes(g, 0, L, ln, ln + act)
        with torch.cuda.stream(compute):
            _ = cache.k.view(torch.int32).sum() + cache.v.view(torch.int32).sum()
            if nt:
                tok = H.device_bytes(nt)
                synth_gpu.fill_tensor(tok[:nt], 7000 + 10 * i + m, 0, g.kind, compute)
                dv.dv_kv_unpack(cache, 0, L, ln, ln + act, tok, stream=compute, src_bytes=nt)
        tok_h = synth.fill_bytes(7000 + 10 * i + m, 0, nt, g.kind) if nt else np.empty(0, np.uint8)
        if nt:
            ORC.unpack(g, mb.kh, mb.vh, 0, L, ln, ln + act, tok_h)
        mb.records.append((0, L, ln.copy(), (ln + act).astype(np.int32), tok_h))
        sw.release(mb.rep, 0, L, ln, ln + act, step=i + 1)
        mb.lens = (ln + act).astype(np.int32)
    sw.wait()
    torch.cuda.synchronize()
    last = order[-1]
    sw.close()
    f.close()
    return caches, sw, last


@pytest.mark.parametrize("check_each_step, prefetch",
                         [(True, True), (False, True), (True, False)],
                         ids=["checked", "pipelined", "no-prefetch"])
def test_swapper_matches_the_oracle(check_each_step, prefetch):
    """no-prefetch: every acquire finds its microbatch out of the caches and
    swaps it in itself, into the cache the previous step did not use."""
    rounds = 3
    mbs = make_microbatches(4, rounds)
    compute = torch.cuda.Stream()
    swap = torch.cuda.Stream(priority=-1)
    fetch = (torch.cuda.Stream(priority=-1), torch.cuda.Stream(priority=-1))
    caches, _, last = run_rounds(mbs, rounds, check_each_step, compute, swap, fetch, prefetch)
    for m, mb in enumerate(mbs):
        assert mb.rep.info()[0] == 1 + rounds
        z = H.device_cache(G, fill="zero")
        mb.rep.restore_batched(z)
        kw, vw = ORC.restore(G, mb.records)
        assert np.array_equal(H.to_np(z.k), kw), f"microbatch {m}"
        assert np.array_equal(H.to_np(z.v), vw), f"microbatch {m}"
    # the cache the last step ran in holds the last microbatch's current state
    assert any(mbs[last].used_bytes_match(c) for c in caches)


@pytest.mark.parametrize("n", [1, 2])
def test_swapper_with_one_or_two_microbatches(n):
    """With no more microbatches than caches, each stays resident after its
    first swap-in; the deltas still go to the replicas."""
    rounds = 3
    mbs = make_microbatches(n, rounds, seed=600 + n)
    s = torch.cuda.Stream()
    caches, _, _ = run_rounds(mbs, rounds, True, s, torch.cuda.Stream(), (s, s))
    for mb in mbs:
        z = H.device_cache(G, fill="zero")
        mb.rep.restore(z)
        kw, vw = ORC.restore(G, mb.records)
        assert np.array_equal(H.to_np(z.k), kw) and np.array_equal(H.to_np(z.v), vw)


def test_swapper_errors():
    mbs = make_microbatches(2, 1, seed=700)
    c0 = H.device_cache(G, fill="zero")
    c1 = H.device_cache(G, fill="zero")
    f = dv.Fetcher(H.device_bytes(4 << 20), H.device_bytes(4 << 20))
    other = Geometry("other", 3, 6, 4, 128, 150, 2, "fp16")
    with pytest.raises(dv.DvError) as ei:
        dv.Swapper(c0, H.device_cache(other, fill="zero"), f)
    assert ei.value.status == dv.DV_ERR_INVALID_ARG
    with pytest.raises(dv.DvError):
        dv.Swapper(c0, c0, f)
    sw = dv.Swapper(c0, c1, f)
    sw.acquire(mbs[0].rep)
    with pytest.raises(dv.DvError) as ei:             # the first is not released yet
        sw.acquire(mbs[1].rep)
    assert ei.value.status == dv.DV_ERR_INVALID_ARG
    zs = np.zeros(G.batch, np.int32)
    with pytest.raises(dv.DvError):                   # not the acquired one
        sw.release(mbs[1].rep, 0, G.num_layers, zs, zs, step=1)
    with pytest.raises(dv.DvError) as ei:             # a range past the cache
        sw.release(mbs[0].rep, 0, G.num_layers, zs, zs + G.max_seq + 1, step=1)
    assert ei.value.status == dv.DV_ERR_RANGE
    sw.release(mbs[0].rep, 0, G.num_layers, zs, zs, step=1)   # an empty update is fine
    sw.wait()
    sw.close()
    f.close()
