"""Parity at the workloads' full sizes, in the launch configuration the
benchmark uses.  Outputs are checked on sampled elements the oracle computes
one by one (its nest gives the cache element held at a staging offset, the
seeded generator its value) and by properties that hold at any size: round
trips, bytes outside the ranges untouched, streamed bytes equal to one pack."""
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
    rng = np.random.default_rng(1)
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
    H.sampled_check(ORC, g, seed, host, 0, g.num_layers, ps, pe, rng)
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
    for k, (s, e) in enumerate(deltas):
        H.sampled_check(ORC, g, seed, dbuf[k * dsz:(k + 1) * dsz], 0, g.num_layers, s, e, rng,
                        nsamples=dsz // g.elem_bytes)
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
    rng = np.random.default_rng(3)
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
    H.sampled_check(ORC, g, seed, host_f, 0, g.num_layers, zs, lens, rng)
    assert torch.equal(host_f[:n], host_s[:n])
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
    microbatch's host bytes must equal the pack of a reference cache that
    received the same writes; the deltas must equal the written tokens; the
    prompt bytes are sampled against the oracle."""
    g = C.OPT66B_STAGE
    rounds = 4
    mbs = C.opt66b_microbatches()
    L = g.num_layers
    zs = np.zeros(g.batch, np.int32)
    rng = np.random.default_rng(4)
    seeds = [C.seed_of(4) * 10 + m for m in range(len(mbs))]
    dev = H.device_cache(g, fill="zero")  # the one rotated device buffer
    refs, hosts, reps, lens, arenas = [], [], [], [], []
    for m, (p, o) in enumerate(mbs):
        ref = H.device_cache(g, fill="synth", seed=seeds[m])
        final = p + np.minimum(o, rounds)
        cap = dv.dv_staging_bytes(ref, 0, L, zs, final)
        host = H.pinned(cap, fill=0)
        dv.dv_swap_out(ref, 0, L, zs, p, host)  # the microbatch's prompt cache
        torch.cuda.synchronize()
        H.sampled_check(ORC, g, seeds[m], host, 0, L, zs, p, rng, nsamples=50_000)
        tok = dv.dv_staging_bytes(ref, 0, L, zs, np.ones(g.batch, np.int32))
        arena = H.pinned(rounds * tok)
        refs.append(ref)
        hosts.append(host)
        arenas.append(arena)
        reps.append(dv.Replica(arena, g.batch))
        lens.append(p.copy())
    written = [[] for _ in mbs]
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
            dv.dv_kv_unpack(refs[m], 0, L, ln, ln + act, token, src_bytes=nt)
            reps[m].append(dev, 0, L, ln, ln + act, step=r)
            dv.dv_swap_out(dev, 0, L, zs, ln + act, hosts[m])
            written[m].append((token, nt))
            lens[m] = ln + act
    torch.cuda.synchronize()
    for m in range(len(mbs)):
        n = dv.dv_staging_bytes(refs[m], 0, L, zs, lens[m])
        want = H.device_bytes(n)
        dv.dv_kv_pack(refs[m], 0, L, zs, lens[m], want)
        torch.cuda.synchronize()
        assert torch.equal(hosts[m][:n], want[:n].cpu()), f"microbatch {m}"
        off = 0
        for token, nt in written[m]:
            assert torch.equal(arenas[m][off:off + nt], token[:nt].cpu())
            off += nt
        assert reps[m].info() == (rounds, off)
    for rep in reps:
        rep.close()


def test_bloom_replica_256_steps_and_restore():
    """Workload 5: snapshot of [0,len0) plus 256 one-token deltas to a host
    replica, restored into a zeroed cache: equal to the live cache on
    [0, len0+256) of every sequence, zero beyond."""
    g, seed = C.BLOOM_STAGE, C.seed_of(5)
    rng = np.random.default_rng(5)
    len0 = C.bloom_lengths()
    steps = C.BLOOM_DECODE_STEPS
    zs = np.zeros(g.batch, np.int32)
    cache = H.device_cache(g, fill="synth", seed=seed)
    total = dv.dv_staging_bytes(cache, 0, g.num_layers, zs, len0 + steps)
    arena = H.pinned(total)
    rep = dv.Replica(arena, g.batch)
    rep.append(cache, 0, g.num_layers, zs, len0, step=0)
    pos = len0.copy()
    for k in range(1, steps + 1):
        rep.append(cache, 0, g.num_layers, pos, pos + 1, step=k)
        pos = pos + 1
    torch.cuda.synchronize()
    nrec, used = rep.info()
    assert nrec == steps + 1 and used == total
    snap = dv.dv_staging_bytes(cache, 0, g.num_layers, zs, len0)
    H.sampled_check(ORC, g, seed, arena, 0, g.num_layers, zs, len0, rng)
    d1 = dv.dv_staging_bytes(cache, 0, g.num_layers, len0, len0 + 1)
    H.sampled_check(ORC, g, seed, arena[snap:snap + d1], 0, g.num_layers, len0, len0 + 1, rng)
    back = H.device_cache(g, fill="zero")
    rep.restore(back)
    torch.cuda.synchronize()
    H.assert_prefix_equal_rest_zero(g, back, cache, pos)
    # the record-batched restore: the snapshot alone, the 256 deltas in 4
    # launches of the record kernel (72 records per launch at batch 32)
    back.k.zero_()
    back.v.zero_()
    rep.restore_batched(back)
    torch.cuda.synchronize()
    H.assert_prefix_equal_rest_zero(g, back, cache, pos)
    rep.close()


def test_largest_launch_beyond_2_31_chunks():
    """The whole BLOOM-stage cache ([0, 2048) of every sequence, all 14 layers:
    52.6 GB of staging, 3.3e9 16-byte chunks, more than 2^31) in one pack
    launch per kernel variant, and one unpack back into the zeroed cache:
    sampled staging elements equal the oracle's, sampled cache elements the
    generator's."""
    g, seed = C.BLOOM_STAGE, C.seed_of(5)
    rng = np.random.default_rng(55)
    zs = np.zeros(g.batch, np.int32)
    full = np.full(g.batch, g.max_seq, np.int32)
    cache = H.device_cache(g, fill="synth", seed=seed)
    n = dv.dv_staging_bytes(cache, 0, g.num_layers, zs, full)
    assert n == 2 * g.tensor_bytes and n // 16 > 2 ** 31
    stg = torch.empty(n, dtype=torch.uint8, device="cuda")
    for variant in (dv.DV_VARIANT_AUTO, dv.DV_VARIANT_FLAT):
        stg[-(1 << 20):].zero_()
        dv.dv_kv_pack(cache, 0, g.num_layers, zs, full, stg, variant=variant)
        torch.cuda.synchronize()
        H.sampled_check(ORC, g, seed, stg, 0, g.num_layers, zs, full, rng)
    cache.k.zero_()
    cache.v.zero_()
    dv.dv_kv_unpack(cache, 0, g.num_layers, zs, full, stg)
    torch.cuda.synchronize()
    del stg
    view = {2: torch.int16}[g.elem_bytes]
    for kv, t in ((0, cache.k), (1, cache.v)):
        idx = np.unique(np.concatenate([rng.integers(0, g.tensor_elems, size=200_000),
                                        np.array([0, g.tensor_elems - 1])]))
        got = t.view(view)[torch.from_numpy(idx).cuda()].cpu().numpy().view(np.uint16)
        want = synth.fill_elements(seed, kv, idx, g.elem_bytes, g.kind)
        assert np.array_equal(got, want), f"{'KV'[kv]}: sampled elements differ after unpack"
