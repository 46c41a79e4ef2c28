"""Using the KV-cache buffered copy from Python, end to end, on one GPU.

    python examples/usage.py

Packs and unpacks a GPT2-1.5B-shaped fp16 cache, swaps it to pinned host
memory and back, streams it out and back layer by layer, keeps a host
replica of a snapshot and decode deltas and restores from it (record by
record, batched, pipelined through a fetcher), streams deltas beside the
compute, and runs two microbatches through two device caches.
"""
import numpy as np
import torch

import kv_cache_streaming_gb300 as dv


def main():
    L, B, H, D, S = 48, 8, 25, 64, 1024                    # fp16 cache, x = 8
    k = torch.randint(0, 255, (L * B * H * D * S * 2,), dtype=torch.uint8, device="cuda")
    v = torch.randint(0, 255, (L * B * H * D * S * 2,), dtype=torch.uint8, device="cuda")
    cache = dv.Cache(L, B, H, D, S, 2, k, v)                # K [L][B][H][D/8][S][8], V [L][B][H][S][D]

    s = np.zeros(B, np.int32)
    e = np.full(B, 1000, np.int32)                          # token range per sequence
    n = dv.dv_staging_bytes(cache, 0, L, s, e)
    stg = torch.empty(n, dtype=torch.uint8, device="cuda")
    dv.dv_kv_pack(cache, 0, L, s, e, stg)                   # gather
    dv.dv_kv_unpack(cache, 0, L, s, e, stg)                 # scatter back

    host = torch.empty(n, dtype=torch.uint8, pin_memory=True)
    dv.dv_swap_out(cache, 0, L, s, e, host)                 # zero-copy pack into host memory
    dv.dv_swap_in(cache, 0, L, s, e, host)

    slab = n // L                                           # one layer of the ranges
    slots = [torch.empty(slab, dtype=torch.uint8, device="cuda") for _ in range(4)]
    out, cp, up = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    streamer = dv.Streamer(slots[0], slots[1], torch.cuda.current_stream(), out)
    fetcher = dv.Fetcher(slots[2], slots[3], cp, up)        # copy and unpack streams
    for l in range(L):                                      # layer by layer, both ways
        streamer.stream_layer(cache, l, s, e, host)         # pack, then copy to host
        cp.wait_stream(out)                                 # layer l is in host memory
        fetcher.fetch_layer(cache, l, s, e, host)           # copy back, then unpack
    fetcher.wait()

    delta = dv.dv_staging_bytes(cache, 0, L, e, e + 1)      # one decode token
    arena = dv.host_empty(n + 8 * delta)                   # pinned host memory on huge pages
    rep = dv.Replica(arena, B)
    rep.append(cache, 0, L, s, e, step=0)                   # snapshot
    ds = dv.DeltaStreamer(rep, torch.cuda.current_stream(), torch.cuda.Stream())
    for t in range(4):                                      # decode steps: deltas on a side stream
        ds.stream(cache, 0, L, e + t, e + t + 1, step=1 + t)
    ds.join()
    rep.restore(cache)                                      # replay into a cache
    rep.restore_batched(cache)                              # the same: one run-kernel launch for the deltas
    for st in (cp, up):                                     # order the fetcher's streams
        st.wait_stream(torch.cuda.current_stream())         # after the calls above
    rep.restore_fetched(cache, fetcher)                     # the same, copies pipelined
    fetcher.wait()
    rep.truncate(0)                                         # the same log, appended through
    rep.append_streamed(streamer, cache, 0, 1, s, e, step=0)   # the streamer's slots (a layer
    for t in range(4):                                         # of the snapshot: one slot)
        rep.append_streamed(streamer, cache, 0, 1, e + t, e + t + 1, step=1 + t)
    streamer.wait()

    # two microbatches through two device caches (each kept as a replica)
    caches = [dv.Cache(L, B, H, D, S, 2, torch.zeros_like(k), torch.zeros_like(v))
              for _ in range(2)]
    mbs = []
    for m in range(2):
        a = torch.empty(n + 8 * delta, dtype=torch.uint8, pin_memory=True)
        r = dv.Replica(a, B)
        r.append(cache, 0, L, s, e, step=0)                 # both start from this prompt cache
        mbs.append((r, a))
    torch.cuda.synchronize()
    sw = dv.Swapper(caches[0], caches[1], fetcher, torch.cuda.current_stream(),
                    torch.cuda.Stream())
    for step in range(1, 3):
        for m in range(2):
            slot = sw.acquire(mbs[m][0])                    # swapped in (or prefetched)
            sw.prefetch(mbs[1 - m][0])                      # the other one, meanwhile
            # ... the step's compute on caches[slot], writing token e + 3 + step ...
            sw.release(mbs[m][0], 0, L, e + 3 + step, e + 4 + step, step=step)
    sw.wait()
    torch.cuda.synchronize()
    return {"dv": dv, "cache": cache, "k": k, "v": v, "stg": stg, "host": host, "L": L,
            "s": s, "e": e, "caches": caches, "mbs": mbs}


if __name__ == "__main__":
    main()
    print("usage example: done")
