"""Parity at the workloads' full sizes, in the launch configuration the
benchmark uses.  Every byte the GPU path writes is compared with the oracle,
layer by layer: the oracle packs (and restores) each layer of a host copy of
the seeded cache, made by the generator for that layer alone, and the GPU's
staging bytes and restored caches must equal them exactly.  Properties that
hold at any size are checked too: round trips, bytes outside the ranges
untouched, streamed bytes equal to one pack."""
import gc

import numpy as np
import pytest
import torch

import kv_cache_streaming_gb300 as dv
import oracle
import synth
from synth import configs as C
from synth import gpu as synth_gpu
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu
ORC = oracle.default()


@pytest.fixture(autouse=True)
def _release_memory():
    yield
    gc.collect()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def test_gpt2_layer_stream_deltas_and_unpack():
    """Workload 2: prompt [0,1000) streamed layer by layer to pinned host, 24
    one-token deltas, and everything unpacked into a zeroed cache, which then
    equals the live cache on every token (prompt + deltas cover [0,1024))."""
    g, seed = C.GPT2, C.seed_of(2)
    cache = H.device_cache(g, fill="synth", seed=seed)
    (ps, pe), deltas = C.gpt2_ranges()
    n = dv.dv_staging_bytes(cache, 0, g.num_layers, ps, pe)
    slab = n // g.num_layers
    host = H.pinned(n, fill=0)
    pack_s, copy_s = torch.cuda.Stream(), torch.cuda.Stream()
    st = dv.Streamer(H.device_bytes(slab), H.device_bytes(slab), pack_s, copy_s)
    torch.cuda.synchronize()
    for l in range(g.num_layers):
        st.stream_layer(cache, l, ps, pe, host, l0=0)
    st.wait()
    kh, vh = H.host_cache(g, seed)
    want = ORC.stream_layers(g, kh, vh, 0, g.num_layers, ps, pe)
    assert np.array_equal(host[:n].numpy(), want), "streamed prompt bytes differ from the oracle"
    # the streamed bytes equal one pack of all layers
    whole = H.device_bytes(n)
    dv.dv_kv_pack(cache, 0, g.num_layers, ps, pe, whole)
    torch.cuda.synchronize()
    assert torch.equal(whole[:n].cpu(), host[:n])
    # 24 decode deltas, every element checked
    dsz = dv.dv_staging_bytes(cache, 0, g.num_layers, *deltas[0])
    dbuf = H.device_bytes(len(deltas) * dsz)
    for k, (s, e) in enumerate(deltas):
        dv.dv_kv_pack(cache, 0, g.num_layers, s, e, dbuf[k * dsz:(k + 1) * dsz])
    got = dbuf[:len(deltas) * dsz].cpu().numpy()
    for k, (s, e) in enumerate(deltas):
        assert np.array_equal(got[k * dsz:(k + 1) * dsz], ORC.pack(g, kh, vh, 0, g.num_layers, s, e))
    # unpack everything into a zeroed cache
    back = H.device_cache(g, fill="zero")
    for l in range(g.num_layers):
        dv.dv_kv_unpack(back, l, l + 1, ps, pe, whole[l * slab:(l + 1) * slab])
    for k, (s, e) in enumerate(deltas):
        dv.dv_kv_unpack(back, 0, g.num_layers, s, e, dbuf[k * dsz:(k + 1) * dsz])
    torch.cuda.synchronize()
    assert torch.equal(back.k, cache.k) and torch.equal(back.v, cache.v)
    st.close()


def test_opt13b_swap_out_and_in():
    """Workload 3: swap-out of the lognormal used prefixes to pinned host
    (fused and staged give the same bytes), swap-in into a fresh zeroed
    cache."""
    g, seed = C.OPT13B, C.seed_of(3)
    lens = C.opt13b_lengths()
    zs = np.zeros(g.batch, np.int32)
    cache = H.device_cache(g, fill="synth", seed=seed)
    n = dv.dv_staging_bytes(cache, 0, g.num_layers, zs, lens)
    host_f = H.pinned(n, fill=0)
    host_s = H.pinned(n, fill=0)
    staging = H.device_bytes(4 * (n // g.num_layers))
    dv.dv_swap_out(cache, 0, g.num_layers, zs, lens, host_f)
    dv.dv_swap_out(cache, 0, g.num_layers, zs, lens, host_s, staging=staging)
    torch.cuda.synchronize()
    assert torch.equal(host_f[:n], host_s[:n])
    g1 = H.layer_geometry(g)
    slab = n // g.num_layers
    hf = host_f.numpy()

    def layer(l):
        kh, vh = H.host_layer(g, seed, l)
        want = ORC.pack(g1, kh, vh, 0, 1, zs, lens)
        assert np.array_equal(hf[l * slab:(l + 1) * slab], want), f"layer {l}"

    H.for_each_layer(layer, range(g.num_layers), 4 * g1.tensor_bytes)
    for stg in (None, staging):
        fresh = H.device_cache(g, fill="zero")
        dv.dv_swap_in(fresh, 0, g.num_layers, zs, lens, host_f, staging=stg)
        torch.cuda.synchronize()
        H.assert_prefix_equal_rest_zero(g, fresh, cache, lens)
        del fresh
        torch.cuda.empty_cache()


def test_opt66b_microbatch_rotation():
    """Workload 4: four microbatches rotated through one device cache: swap-in
    of the used prefix, a one-token decode write, the delta packed to the
    microbatch's host replica, swap-out of the grown prefix.  Each
    microbatch's host bytes must equal, layer by layer, the oracle's pack of
    the host copy of its cache after the same writes (the seeded fill, then
    every written token unpacked by the oracle); the replica's deltas must
    equal the written tokens."""
    g = C.OPT66B_STAGE
    rounds = 4
    mbs = C.opt66b_microbatches()
    L = g.num_layers
    zs = np.zeros(g.batch, np.int32)
    seeds = [C.seed_of(4) * 10 + m for m in range(len(mbs))]
    dev = H.device_cache(g, fill="zero")  # the one rotated device buffer
    hosts, reps, lens, arenas = [], [], [], []
    for m, (p, o) in enumerate(mbs):
        src = H.device_cache(g, fill="synth", seed=seeds[m])
        final = p + np.minimum(o, rounds)
        cap = dv.dv_staging_bytes(src, 0, L, zs, final)
        host = H.pinned(cap, fill=0)
        dv.dv_swap_out(src, 0, L, zs, p, host)  # the microbatch's prompt cache
        torch.cuda.synchronize()
        del src
        tok = dv.dv_staging_bytes(dev, 0, L, zs, np.ones(g.batch, np.int32))
        arena = H.pinned(rounds * tok)
        hosts.append(host)
        arenas.append(arena)
        reps.append(dv.Replica(arena, g.batch))
        lens.append(p.copy())
    torch.cuda.empty_cache()
    written = [[] for _ in mbs]   # per microbatch: (start, end, token seed, bytes)
    for r in range(rounds):
        for m, (p, o) in enumerate(mbs):
            ln = lens[m]
            act = ((ln - p) < o).astype(np.int32)
            dv.dv_swap_in(dev, 0, L, zs, ln, hosts[m])
            # the decode write: one seeded token per active sequence
            nt = dv.dv_staging_bytes(dev, 0, L, ln, ln + act)
            token = H.device_bytes(nt)
            synth_gpu.fill_tensor(token[:nt], 1000 * m + r, 0, g.kind)
            dv.dv_kv_unpack(dev, 0, L, ln, ln + act, token, src_bytes=nt)
            reps[m].append(dev, 0, L, ln, ln + act, step=r)
            dv.dv_swap_out(dev, 0, L, zs, ln + act, hosts[m])
            written[m].append((ln.copy(), (ln + act).astype(np.int32), 1000 * m + r, nt))
            lens[m] = ln + act
    torch.cuda.synchronize()
    g1 = H.layer_geometry(g)
    for m in range(len(mbs)):
        off = 0
        for s_, e_, tseed, nt in written[m]:
            want = synth.fill_bytes(tseed, 0, nt, g.kind)
            assert np.array_equal(arenas[m][off:off + nt].numpy(), want), f"microbatch {m}"
            off += nt
        assert reps[m].info() == (rounds, off)
        n = dv.dv_staging_bytes(dev, 0, L, zs, lens[m])
        slab = n // L
        hm = hosts[m].numpy()

        def layer(l, m=m, slab=slab, hm=hm):
            kh, vh = H.host_layer(g, seeds[m], l)
            for s_, e_, tseed, nt in written[m]:
                tl = nt // L
                tok = synth.fill_bytes(tseed, 0, nt, g.kind)[l * tl:(l + 1) * tl]
                ORC.unpack(g1, kh, vh, 0, 1, s_, e_, tok)
            want = ORC.pack(g1, kh, vh, 0, 1, zs, lens[m])
            assert np.array_equal(hm[l * slab:(l + 1) * slab], want), f"microbatch {m} layer {l}"

        H.for_each_layer(layer, range(L), 4 * g1.tensor_bytes)
    for rep in reps:
        rep.close()


def test_bloom_replica_256_steps_and_restore():
    """Workload 5: snapshot of [0,len0) plus 256 one-token deltas to a host
    replica, restored into a zeroed cache record by record, record-batched
    and through a fetcher: equal to the live cache on [0, len0+256) of every
    sequence, zero beyond.  Then, layer by layer, every byte of the replica
    (the snapshot's and each delta's share of that layer) equals the oracle's
    pack of the host copy of the layer, and the batched restore's layer equals
    the oracle's restore of the same records."""
    g, seed = C.BLOOM_STAGE, C.seed_of(5)
    len0 = C.bloom_lengths()
    steps = C.BLOOM_DECODE_STEPS
    L = g.num_layers
    zs = np.zeros(g.batch, np.int32)
    cache = H.device_cache(g, fill="synth", seed=seed)
    total = dv.dv_staging_bytes(cache, 0, L, zs, len0 + steps)
    arena = H.pinned(total)
    rep = dv.Replica(arena, g.batch)
    rep.append(cache, 0, L, zs, len0, step=0)
    pos = len0.copy()
    for k in range(1, steps + 1):
        rep.append(cache, 0, L, pos, pos + 1, step=k)
        pos = pos + 1
    torch.cuda.synchronize()
    nrec, used = rep.info()
    assert nrec == steps + 1 and used == total
    back = H.device_cache(g, fill="zero")
    rep.restore(back)
    torch.cuda.synchronize()
    H.assert_prefix_equal_rest_zero(g, back, cache, pos)
    snap = dv.dv_staging_bytes(cache, 0, L, zs, len0)
    slot = snap // L
    back.k.zero_()
    back.v.zero_()
    torch.cuda.synchronize()
    cs = torch.cuda.Stream()
    f = dv.Fetcher(H.device_bytes(slot), H.device_bytes(slot), cs, torch.cuda.Stream())
    rep.restore_fetched(back, f)
    f.wait()
    f.close()
    H.assert_prefix_equal_rest_zero(g, back, cache, pos)
    # the record-batched restore: the snapshot alone, the 256 deltas as one run
    back.k.zero_()
    back.v.zero_()
    rep.restore_batched(back)
    torch.cuda.synchronize()
    H.assert_prefix_equal_rest_zero(g, back, cache, pos)
    del cache
    torch.cuda.empty_cache()
    dsz = dv.dv_staging_bytes(back, 0, L, len0, len0 + 1)
    g1 = H.layer_geometry(g)
    snap_l, d_l = snap // L, dsz // L
    an = arena.numpy()

    def layer(l):
        kh, vh = H.host_layer(g, seed, l)
        want = ORC.pack(g1, kh, vh, 0, 1, zs, len0)
        assert np.array_equal(an[l * snap_l:(l + 1) * snap_l], want), f"snapshot, layer {l}"
        recs = [(0, 1, zs, len0, want)]
        for k in range(steps):
            a = (len0 + k).astype(np.int32)
            d = ORC.pack(g1, kh, vh, 0, 1, a, a + 1)
            off = snap + k * dsz + l * d_l
            assert np.array_equal(an[off:off + d_l], d), f"delta {k}, layer {l}"
            recs.append((0, 1, a, a + 1, d))
        del kh, vh
        kw, vw = ORC.restore(g1, recs)
        gk, gv = H.device_layer(g, back, l)
        assert np.array_equal(gk, kw) and np.array_equal(gv, vw), f"restored layer {l}"

    H.for_each_layer(layer, range(L), 6 * g1.tensor_bytes)
    rep.close()


def test_largest_launch_beyond_2_31_chunks():
    """The whole BLOOM-stage cache ([0, 2048) of every sequence, all 14 layers:
    52.6 GB of staging, 3.3e9 16-byte chunks, more than 2^31) in one pack
    launch per kernel variant, and one unpack back into the zeroed cache:
    sampled staging elements equal the oracle's over the whole launch, and the
    first and last layers' staging bytes and unpacked layers equal the
    oracle's and the generator's byte for byte."""
    g, seed = C.BLOOM_STAGE, C.seed_of(5)
    rng = np.random.default_rng(55)
    zs = np.zeros(g.batch, np.int32)
    full = np.full(g.batch, g.max_seq, np.int32)
    L = g.num_layers
    cache = H.device_cache(g, fill="synth", seed=seed)
    n = dv.dv_staging_bytes(cache, 0, L, zs, full)
    assert n == 2 * g.tensor_bytes and n // 16 > 2 ** 31
    slab = n // L
    g1 = H.layer_geometry(g)
    stg = torch.empty(n, dtype=torch.uint8, device="cuda")
    for variant in (dv.DV_VARIANT_AUTO, dv.DV_VARIANT_FLAT):
        stg[-(1 << 20):].zero_()
        dv.dv_kv_pack(cache, 0, L, zs, full, stg, variant=variant)
        torch.cuda.synchronize()
        H.sampled_check(ORC, g, seed, stg, 0, L, zs, full, rng)
        for l in (0, L - 1):
            kh, vh = H.host_layer(g, seed, l)
            want = ORC.pack(g1, kh, vh, 0, 1, zs, full)
            got = stg[l * slab:(l + 1) * slab].cpu().numpy()
            assert np.array_equal(got, want), f"variant {variant}, layer {l}"
            del kh, vh, want, got
    cache.k.zero_()
    cache.v.zero_()
    dv.dv_kv_unpack(cache, 0, L, zs, full, stg)
    torch.cuda.synchronize()
    del stg
    torch.cuda.empty_cache()
    for l in (0, L - 1):
        kh, vh = H.host_layer(g, seed, l)
        gk, gv = H.device_layer(g, cache, l)
        assert np.array_equal(gk, kh) and np.array_equal(gv, vh), f"unpacked layer {l}"
