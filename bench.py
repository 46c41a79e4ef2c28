#!/usr/bin/env python
"""Benchmark of the KV-cache buffered copy on GB300.

Headline workload (one step): the BLOOM-176B pipeline-stage-shaped cache
(14 resident layers, batch 32, 112 heads, head_dim 128, max_seq 2048, bf16
bit patterns from the seeded generator; used lengths len0 uniform in
[64, 1536]), as the replica of §3 "Fault detection and recovery" (Fig 10)
builds and uses it:
  1. the snapshot: the used prefixes [0, len0) of all 14 layers packed into a
     device log buffer (19.1 GB, one launch);
  2. 256 decode steps' one-token deltas (one token of every sequence at all
     layers, 25.7 MB each) packed into the log after it, in an order where no
     two consecutive packs share a K line (as between real decode steps,
     whose compute evicts L2);
  3. the restore: the whole log (snapshot + 256 deltas) unpacked into a second
     cache with one dv_kv_unpack_records call.
`value` is the pack/unpack throughput of that step with every buffer in HBM:
bytes read plus bytes written by all its launches, divided by the step time
(the step runs as one CUDA graph replay on one stream; every buffer is read at
least 19 GB of traffic after it was written, so L2 serves none of it).  `e2e`
is the same byte count through the public API with pinned host buffers: the
snapshot and the deltas appended to a host replica through a layer streamer
(dv_replica_append_streamed: packs into two device slots, copy engines to the
host), each part restored into the second cache through a fetcher
(dv_replica_restore_fetched_steps) while the next goes out.  Side sections: the
GPT2-1.5B step (layer-by-layer prompt packs + 24 deltas), swap against the
measured host-link peak, the other workloads, microbatch swapping and decode
streaming.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time
from pathlib import Path

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

import numpy as np  # noqa: E402

from synth.configs import (GPT2, GPT2_PROMPT, GPT2_DECODE_STEPS, BLOOM_STAGE,  # noqa: E402
                           BLOOM_DECODE_STEPS, Geometry, seed_of, gpt2_ranges, bloom_lengths)

METRIC = "KV pack/unpack GB/s (bytes read + written, HBM-resident step)"
UNIT = "GB/s"
WORKLOAD = ("bloom-176b-stage-shaped KV cache L14 B32 H112 D128 S2048 bf16: replica snapshot "
            "[0, len0) (len0 uniform [64, 1536]) + 256 one-token decode deltas packed, then the "
            "whole log restored into a second cache")
HBM_NOMINAL_GBS = 7900.0  # GB300 HBM3e, nominal (the measured copy peak is the roofline)
CPU_SAMPLE_SECONDS = 12.0  # CPU work of each oracle baseline sample (all its threads)
L2_NOTE = ("inputs larger than L2: 102.9 GB read + written per step; every buffer read at "
           "least 19 GB of traffic after it was written; consecutive delta packs share no K line")


def workload_config(world):
    """The `config` of both arms' JSON lines (the same workload either way)."""
    g = BLOOM_STAGE
    return {"workload": WORKLOAD, "layers": g.num_layers, "batch": g.batch,
            "heads": g.num_heads, "head_dim": g.head_dim, "max_seq": g.max_seq,
            "elem": "bf16", "decode_steps": BLOOM_DECODE_STEPS, "l2": L2_NOTE,
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def delta_order(n, stride=8):
    """0, 8, 16, ..., 1, 9, ...: no two consecutive entries are within 8 of
    each other, so consecutive one-token packs never read the same K line."""
    return [k for r in range(stride) for k in range(r, n, stride)]


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="mine", choices=["mine", "reference"])
    ap.add_argument("--no-swap", action="store_true", help="skip the swap / link section")
    ap.add_argument("--kernel-case", default=None,
                    choices=["tile-pack", "tile-unpack", "delta-pack", "delta-unpack",
                             "flat-pack", "flat-unpack", "record-restore", "swap-out",
                             "swap-in", "ragged-pack", "ragged-unpack", "delta-graph-pack",
                             "delta-graph-unpack", "bloom-snapshot-pack",
                             "bloom-snapshot-unpack", "bloom-delta-pack", "bloom-run-restore",
                             "short-ragged-pack", "short-ragged-unpack", "group-pack",
                             "group-unpack", "gpt2-step"],
                    help="run one kernel of the step on an 8-layer cache of the workload's "
                         "shape, 5 launches, and exit (a small case for profilers); "
                         "flat-*: ragged 16..64-token ranges of the OPT-13B-shaped cache, "
                         "flat kernel; record-restore: 5 staged batched restores of 96 "
                         "one-token deltas (even and odd sequences in turn: no runs) of the "
                         "whole cache, one record-kernel launch each; "
                         "swap-*: fused swap of the 8-layer prompt to / from pinned host "
                         "memory (the tile kernel on the host link); ragged-*: the OPT-13B "
                         "workload's lognormal used prefixes, 4 layers, tile kernel; "
                         "delta-graph-*: a CUDA graph of 32 one-token deltas 8 tokens apart "
                         "on a BLOOM-stage-shaped cache cut to 4 layers and max_seq 512, "
                         "5 replays (for graph-level counters); bloom-*: the headline "
                         "step's kernels on its workload cut to 2 layers and batch 16 "
                         "(snapshot pack / unpack: 3 launches; delta pack: 8 launches, 8 "
                         "tokens apart; run restore: 3 launches of 256 one-token records); "
                         "short-ragged-*: the flat-* ranges under the automatic kernel choice; "
                         "group-*: ragged 2..32-token ranges of 32 sequences, 40 layers, "
                         "head_dim 128, all in grouped tiles; "
                         "gpt2-step: the GPT2-1.5B side-section step (one stream), 3 graph "
                         "replays after one eager step")
    return ap.parse_args()


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per launch of the
# headline step's kernels, from one ncu capture of a smaller case of the same
# kernel (`--kernel-case ...`), scaled to one launch of the step by the units
# it moves (traffic grows in proportion).  None until captured, and set back to
# None whenever the kernel changes.
TRAFFIC_PER_LAUNCH = {
    # bloom-snapshot-pack: 2.870 GB per launch of the cut x 19.137 / 1.463 GB
    "pack snapshot (tile kernel)": 2.8696e9 * 19136724992 / 1463074816,
    # bloom-delta-pack: 4.594 MB of reads per launch of the cut (its 1.8 MB of
    # staging writes are still in L2 when it ends) x 14
    "pack one-token delta (token kernel)": 4.594e6 * 14,
    # bloom-snapshot-unpack: 2.866 GB per launch of the cut
    "unpack snapshot (tile kernel)": 2.8659e9 * 19136724992 / 1463074816,
    # bloom-run-restore: 0.885 GB per launch of the cut (256 records) x 14
    "unpack 256 one-token deltas (run kernel)": 0.8851e9 * 14,
}


def peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# ---- distributed plumbing (one process per GPU; no data-path collective) ------

def dist_init(backend=None):
    """(rank, world, local_rank) from the torchrun environment; joins the
    process group (NCCL on GPUs, gloo when asked) when world > 1."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world <= 1:
        return 0, 1, 0
    import torch
    import torch.distributed as td
    rank = int(os.environ["RANK"])
    local = int(os.environ.get("LOCAL_RANK", rank))
    backend = backend or "nccl"
    if backend == "nccl":
        torch.cuda.set_device(local)
        td.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        td.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as td
        td.barrier()


def max_over_ranks(x, world):
    """The largest `x` over all ranks (the slowest rank's time)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as td
    dev = "cuda" if td.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    td.all_reduce(t, op=td.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(bytes_per_step, steps, max_secs, world):
    """GB/s of all ranks together: every rank moves the same bytes per step
    (weak scaling), timed by the slowest rank."""
    return world * bytes_per_step * steps / max_secs / 1e9


# ---- clocks ------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,"
              "temperature.gpu,temperature.memory,clocks.mem")

    def __init__(self, local_rank):
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        self.index = vis.split(",")[local_rank] if vis else str(local_rank)
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", self.index], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.2)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, mx, reasons, power = [], [], set(), []
        extra = {"gpu_temp_c": [], "mem_temp_c": [], "mem_mhz": []}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
            for key, val in zip(extra, parts[9:12]):
                try:
                    extra[key].append(float(val))
                except ValueError:  # "N/A" where the GPU does not report it
                    pass
        out = {"sm_mhz": statistics.median(sm) if sm else None,
               "sm_max_mhz": max(mx) if mx else None,
               "power_w_max": max(power) if power else None,
               "samples": len(sm), "reasons": sorted(reasons)}
        out.update({k: (max(v) if "temp" in k else statistics.median(v)) if v else None
                    for k, v in extra.items()})
        return out


def gpu_identity(local_rank):
    """Name, VBIOS, ECC mode, power limit and memory size of the GPU the bench
    runs on (read once; None when nvidia-smi cannot tell)."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    index = vis.split(",")[local_rank] if vis else str(local_rank)
    fields = ["name", "vbios_version", "ecc.mode.current", "power.limit", "memory.total"]
    try:
        out = subprocess.run(["nvidia-smi", f"--query-gpu={','.join(fields)}",
                              "--format=csv,noheader", "-i", index], capture_output=True,
                             text=True, timeout=20).stdout.strip()
    except (OSError, subprocess.SubprocessError):
        return None
    vals = [v.strip() for v in out.split(",")]
    return dict(zip(fields, vals)) if len(vals) == len(fields) else None


# ---- the reference arm: the CPU oracle on a bounded sample --------------------

def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


class OracleSample:
    """The oracle on a bounded sample of the headline workload.  A unit is one
    layer and two sequences of the BLOOM-stage cache (a cache of that shape:
    1 layer, batch 2, 112 heads, head_dim 128, max_seq 2048): the snapshot pack
    of the two sequences' [0, len0), their 256 one-token deltas, and the unpack
    of the snapshot and every delta into a zeroed cache, in log order.  The 224
    units of the workload are dealt round-robin to `threads` threads, each with
    its own seeded cache; the oracle's C functions run without the interpreter
    lock, so each thread has a core.  A step runs `units` units."""

    UNIT_G = Geometry("bloom-unit", 1, 2, 112, 128, 2048, 2, "bf16")

    def __init__(self, units, threads=1):
        from concurrent.futures import ThreadPoolExecutor
        import oracle
        import synth
        g = self.UNIT_G
        self.threads = max(1, min(threads, units))
        len0 = bloom_lengths()
        pairs = [len0[2 * j:2 * j + 2].astype(np.int32) for j in range(BLOOM_STAGE.batch // 2)]
        every = [(l, pairs[j]) for l in range(BLOOM_STAGE.num_layers) for j in range(len(pairs))]
        self.units = every[:units]
        self.orc = oracle.default()
        seed = seed_of(5)
        self.caches = []
        for t in range(self.threads):
            kh = synth.fill_bytes(seed * 100 + t, 0, g.tensor_bytes, g.kind)
            vh = synth.fill_bytes(seed * 100 + t, 1, g.tensor_bytes, g.kind)
            self.caches.append((kh, vh, np.zeros_like(kh), np.zeros_like(vh)))
        self.pool = ThreadPoolExecutor(self.threads) if self.threads > 1 else None
        how = ("single-thread C loop nest" if self.threads == 1 else
               f"C loop nest, units dealt to {self.threads} threads")
        self.desc = (f"{len(self.units)} of the workload's 224 units (one layer x two sequences: "
                     f"snapshot pack, 256 one-token delta packs, all unpacked), {how}")

    def _units(self, t, units):
        g, orc = self.UNIT_G, self.orc
        kh, vh, kz, vz = self.caches[t]
        zs = np.zeros(2, np.int32)
        moved = 0
        for _, l0 in units:
            snap = orc.pack(g, kh, vh, 0, 1, zs, l0)
            dels = [orc.pack(g, kh, vh, 0, 1, l0 + k, l0 + k + 1)
                    for k in range(BLOOM_DECODE_STEPS)]
            orc.unpack(g, kz, vz, 0, 1, zs, l0, snap)
            for k, d in enumerate(dels):
                orc.unpack(g, kz, vz, 0, 1, l0 + k, l0 + k + 1, d)
            moved += 2 * 2 * (snap.size + sum(d.size for d in dels))
        return moved

    def step(self):
        """Returns (bytes read + written, seconds)."""
        parts = [self.units[t::self.threads] for t in range(self.threads)]
        t0 = time.perf_counter()
        if self.pool is None:
            moved = self._units(0, parts[0])
        else:
            moved = sum(self.pool.map(lambda t: self._units(t, parts[t]), range(self.threads)))
        return moved, time.perf_counter() - t0

    def run(self, cpu_seconds):
        """Repeats step() until the threads together have worked about
        `cpu_seconds`; returns (bytes read + written, seconds, passes)."""
        moved = secs = 0.0
        passes = 0
        while passes == 0 or secs * self.threads < cpu_seconds:
            m, dt = self.step()
            moved += m
            secs += dt
            passes += 1
        return moved, secs, passes

    def close(self):
        if self.pool is not None:
            self.pool.shutdown()


def run_reference(args):
    """The reference arm: the oracle, as it stands, on the machine's host cores.
    Each step is a bounded sample of the headline workload (one unit per
    core), sized so that the whole run stays near two minutes."""
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    cores = host_cores()
    # about 0.5 s of oracle work per unit and core
    per_core = int(max(1, min(4, 100.0 / (0.5 * (args.steps + args.warmup)))))
    smp = OracleSample(cores * per_core, threads=cores)
    for _ in range(args.warmup):
        smp.step()
    moved = secs = 0.0
    for _ in range(args.steps):
        m, dt = smp.step()
        moved += m
        secs += dt
    value = moved / secs / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * secs / max(args.steps, 1), 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "u16", "data": "synthetic",
            "config": workload_config(world),
            "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": smp.threads,
                             "kind": "oracle", "sample": smp.desc + " per step"},
            "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    smp.close()
    print(json.dumps(line), flush=True)


# ---- the GPU arm ---------------------------------------------------------------

class Bloom:
    """The headline step on the BLOOM-176B-stage-shaped cache (see the module
    docstring): snapshot + 256 one-token deltas packed into a device log, the
    whole log restored into a second cache."""

    def __init__(self):
        import torch
        import kv_cache_streaming_gb300 as dv
        from synth import gpu as synth_gpu
        self.torch, self.dv = torch, dv
        g = self.g = BLOOM_STAGE
        L = g.num_layers
        self.k = torch.empty(g.tensor_bytes, dtype=torch.uint8, device="cuda")
        self.v = torch.empty(g.tensor_bytes, dtype=torch.uint8, device="cuda")
        synth_gpu.fill_cache(g, self.k, self.v, seed_of(5))
        self.kb = torch.zeros_like(self.k)
        self.vb = torch.zeros_like(self.v)
        self.cache = dv.Cache.from_geometry(g, self.k, self.v)
        self.cache_b = dv.Cache.from_geometry(g, self.kb, self.vb)
        self.zs = np.zeros(g.batch, np.int32)
        self.len0 = bloom_lengths()
        self.nd = BLOOM_DECODE_STEPS
        self.deltas = [(self.len0 + k, self.len0 + k + 1) for k in range(self.nd)]
        self.order = delta_order(self.nd)
        self.snap = dv.dv_staging_bytes(self.cache, 0, L, self.zs, self.len0)
        self.dsz = dv.dv_staging_bytes(self.cache, 0, L, *self.deltas[0])
        self.total = self.snap + self.nd * self.dsz
        self.log = torch.empty(self.total, dtype=torch.uint8, device="cuda")
        self.records = [(0, L, self.zs, self.len0)] + [(0, L, s, e) for s, e in self.deltas]
        self.bytes_per_step = 2 * 2 * self.total
        self.stream = torch.cuda.Stream()

    def delta_at(self, k):
        """(address, bytes) of delta k's record in the device log."""
        return (self.log.data_ptr() + self.snap + k * self.dsz, self.dsz)

    def device_step(self, s):
        """Snapshot pack, the 256 delta packs (in `order`), the restore."""
        dv, L = self.dv, self.g.num_layers
        dv.dv_kv_pack(self.cache, 0, L, self.zs, self.len0, (self.log.data_ptr(), self.snap), s)
        for k in self.order:
            a, b = self.deltas[k]
            dv.dv_kv_pack(self.cache, 0, L, a, b, self.delta_at(k), s)
        dv.dv_kv_unpack_records(self.cache_b, self.records, self.log, s)

    def launches_per_step(self):
        # snapshot pack, one pack per delta, the restore: the snapshot by the
        # tile kernel, the 256-record run by one run-kernel launch
        return 1 + self.nd + 2

    def capture(self):
        torch = self.torch
        with torch.cuda.stream(self.stream):
            self.device_step(self.stream)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=self.stream, capture_error_mode="relaxed"):
            self.device_step(self.stream)
        torch.cuda.synchronize()

    def timed_value(self, steps, warmup, world):
        torch = self.torch
        for _ in range(warmup):
            self.graph.replay()
        torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(self.stream):
            e0.record(self.stream)
            for _ in range(steps):
                self.graph.replay()
            e1.record(self.stream)
        torch.cuda.synchronize()
        barrier(world)
        return e0.elapsed_time(e1) / 1e3

    def clear_b(self):
        self.kb.zero_()
        self.vb.zero_()
        self.torch.cuda.synchronize()

    def verify(self):
        """The second cache equals the first on [0, len0 + 256) of every
        sequence and is zero beyond (it started zeroed)."""
        torch, g = self.torch, self.g
        torch.cuda.synchronize()
        L, B, H, D, S = g.num_layers, g.batch, g.num_heads, g.head_dim, g.max_seq
        x = 16 // g.elem_bytes
        views = []
        for t in (self.k, self.v, self.kb, self.vb):
            views.append(t.view(torch.int16))
        ka, va, kb, vb = views
        ka, kb = (t.view(L, B, H, D // x, S, x) for t in (ka, kb))
        va, vb = (t.view(L, B, H, S, D) for t in (va, vb))
        for b_ in range(B):
            n = int(self.len0[b_]) + self.nd
            if not (torch.equal(kb[:, b_, :, :, :n], ka[:, b_, :, :, :n]) and
                    torch.equal(vb[:, b_, :, :n], va[:, b_, :, :n])):
                return False
            if kb[:, b_, :, :, n:].any() or vb[:, b_, :, n:].any():
                return False
        return True

    def kernel_times(self, reps=5):
        """Average launch time of each launch kind as it runs in the step: the
        step's launches of one kind captured in their own CUDA graph, replayed
        `reps` times (L2 flushed before each replay), CUDA events on the
        launching stream around each replay.  Returns (kind, seconds per
        launch, algorithmic bytes per launch, launches per step)."""
        torch, dv, g = self.torch, self.dv, self.g
        L = g.num_layers
        s = self.stream
        lp = self.log.data_ptr()
        kinds = {
            "pack snapshot (tile kernel)": (
                [lambda: dv.dv_kv_pack(self.cache, 0, L, self.zs, self.len0, (lp, self.snap), s)],
                2 * self.snap),
            "pack one-token delta (token kernel)": (
                [lambda k=k: dv.dv_kv_pack(self.cache, 0, L, *self.deltas[k], self.delta_at(k), s)
                 for k in self.order], 2 * self.dsz),
            "unpack snapshot (tile kernel)": (
                [lambda: dv.dv_kv_unpack(self.cache_b, 0, L, self.zs, self.len0,
                                         (lp, self.snap), s)], 2 * self.snap),
            "unpack 256 one-token deltas (run kernel)": (
                [lambda: dv.dv_kv_unpack_records(self.cache_b, self.records[1:],
                                                 (lp + self.snap, self.nd * self.dsz), s)],
                2 * self.nd * self.dsz),
        }
        flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        out = []
        for name, (calls, nbytes) in kinds.items():
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=s, capture_error_mode="relaxed"):
                for fn in calls:
                    fn()
            ms = []
            with torch.cuda.stream(s):
                for r in range(reps + 1):
                    flush.fill_(r)
                    a = torch.cuda.Event(enable_timing=True)
                    b = torch.cuda.Event(enable_timing=True)
                    a.record(s)
                    graph.replay()
                    b.record(s)
                    torch.cuda.synchronize()
                    if r:
                        ms.append(a.elapsed_time(b))
            n = len(calls)
            out.append((name, statistics.median(ms) / 1e3 / n, nbytes, n))
            del graph
        del flush
        return out

    # one step through the public API with pinned host buffers
    def setup_e2e(self):
        torch, dv, g = self.torch, self.dv, self.g
        # the replica's arena in pinned host memory backed by huge pages
        # (dv_host_alloc): every pass over it runs at the link rate
        self.arena = dv.host_empty(self.total)
        self.replica = dv.Replica(self.arena, g.batch)
        slot = dv.dv_staging_bytes(self.cache, 0, 1, self.zs, self.len0)  # one snapshot layer
        self.slots = (torch.empty(slot, dtype=torch.uint8, device="cuda"),
                      torch.empty(slot, dtype=torch.uint8, device="cuda"))
        self.in_copy = torch.cuda.Stream()
        self.in_unpack = torch.cuda.Stream()
        self.fetcher = dv.Fetcher(self.slots[0], self.slots[1], self.in_copy, self.in_unpack)
        # the appends go through a layer streamer: packs into its two device
        # slots, copy engines take them to the host, so both directions of
        # the link run on copy engines and each pack overlaps the previous copy
        self.out_slots = (torch.empty(slot, dtype=torch.uint8, device="cuda"),
                          torch.empty(slot, dtype=torch.uint8, device="cuda"))
        self.out_pack = torch.cuda.Stream()
        self.out_copy = torch.cuda.Stream()
        self.streamer = dv.Streamer(self.out_slots[0], self.out_slots[1], self.out_pack,
                                    self.out_copy)

    E2E_DELTA_CHUNK = 16  # deltas restored as they accumulate, this many at a time

    def e2e_step(self):
        """The log through the host replica and back: the snapshot appended
        layer by layer through the streamer (each layer packed into a device
        slot while the previous one is copied to pinned memory by a copy
        engine), each layer restored into the second cache through the fetcher
        as soon as it is in host memory (the host-to-device copy of layer l
        overlaps the device-to-host copy of layer l+1: copy engines both
        ways), then the 256 deltas appended the same way in decode order, each
        16 restored (one run of records) while the next 16 go out."""
        g, s = self.g, self.stream
        L = g.num_layers
        rep, st = self.replica, self.streamer
        rep.truncate(0)
        self.in_unpack.wait_stream(s)    # the second cache is free
        self.out_pack.wait_stream(s)     # the first cache is written
        for l in range(L):
            rep.append_streamed(st, self.cache, l, l + 1, self.zs, self.len0, step=l)
            self.in_copy.wait_stream(self.out_copy)  # layer l is in host memory
            rep.restore_fetched(self.cache_b, self.fetcher, upto_step=l + 1, from_step=l)
        chunk = self.E2E_DELTA_CHUNK
        for k0 in range(0, self.nd, chunk):
            for k in range(k0, min(self.nd, k0 + chunk)):
                a, b = self.deltas[k]
                rep.append_streamed(st, self.cache, 0, L, a, b, step=L + k)
            self.in_copy.wait_stream(self.out_copy)  # these deltas are in host memory
            rep.restore_fetched(self.cache_b, self.fetcher, upto_step=L + k0 + chunk,
                                from_step=L + k0)
        s.wait_stream(self.out_copy)
        s.wait_stream(self.in_unpack)

    def timed_e2e(self, steps, warmup, world):
        """Seconds of each of `steps` end-to-end steps, each timed from an idle
        GPU to its last unpack (the host link is shared with other tenants of
        the machine: the median step is the robust figure)."""
        torch = self.torch
        for _ in range(warmup):
            self.e2e_step()
        torch.cuda.synchronize()
        barrier(world)
        ts = []
        for _ in range(steps):
            t0 = time.perf_counter()
            self.e2e_step()
            torch.cuda.synchronize()
            ts.append(time.perf_counter() - t0)
        barrier(world)
        return ts

    def close_e2e(self):
        self.fetcher.close()
        self.streamer.close()
        self.replica.close()
        del self.arena, self.slots, self.out_slots


def link_peaks(torch, nbytes=2 << 30, reps=5):
    """The host link measured in this run: large pinned cudaMemcpyAsync each
    way alone and both ways at once (GB/s, median of `reps`).  The host
    buffers come from dv_host_alloc (huge pages), whose passes run at the link
    rate every time (torch's pinned buffers showed slow passes on some boxes,
    which once put the both-ways figure at 231 GB/s)."""
    import kv_cache_streaming_gb300 as dv
    s = torch.cuda.Stream()
    host = dv.host_empty(nbytes)
    dev = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    host2 = dv.host_empty(nbytes)
    dev2 = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    s2 = torch.cuda.Stream()

    def timed(fn):
        ts = []
        for _ in range(reps):
            torch.cuda.synchronize()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(s):
                a.record(s)
                fn()
                b.record(s)
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b) / 1e3)
        return statistics.median(ts)

    def both():
        s2.wait_stream(s)
        host.copy_(dev, non_blocking=True)
        with torch.cuda.stream(s2):
            dev2.copy_(host2, non_blocking=True)
        s.wait_stream(s2)

    out = {"d2h_gbs": nbytes / timed(lambda: host.copy_(dev, non_blocking=True)) / 1e9,
           "h2d_gbs": nbytes / timed(lambda: dev.copy_(host, non_blocking=True)) / 1e9,
           "bidir_gbs": 2 * nbytes / timed(both) / 1e9}
    del host, dev, host2, dev2
    torch.cuda.empty_cache()
    return {k: round(v, 2) for k, v in out.items()}


def host_memory_passes(torch, dv, dev, passes=6):
    """Device-to-host copy passes over all of `dev` (in 1 GiB copies) into
    pinned memory of each kind: torch's pinned allocator (cudaHostAlloc, base
    pages) and dv_host_alloc (huge pages where the kernel gives them).  GB/s
    of each pass."""
    n = dev.numel()
    s = torch.cuda.Stream()
    out = {}
    for kind in ("torch_pinned", "dv_host_alloc"):
        host = (torch.empty(n, dtype=torch.uint8, pin_memory=True) if kind == "torch_pinned"
                else dv.host_empty(n))
        rates = []
        for r in range(passes + 1):
            torch.cuda.synchronize()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(s):
                a.record(s)
                for o in range(0, n, 1 << 30):
                    host[o:o + (1 << 30)].copy_(dev[o:o + (1 << 30)], non_blocking=True)
                b.record(s)
            torch.cuda.synchronize()
            if r:
                rates.append(round(n / (a.elapsed_time(b) / 1e3) / 1e9, 1))
        out[kind] = {"passes_gbs": rates, "median_gbs": statistics.median(rates),
                     "min_gbs": min(rates)}
        del host
    out["bytes_per_pass"] = n
    return out


class Bench:
    def __init__(self):
        import torch
        import kv_cache_streaming_gb300 as dv
        from synth import gpu as synth_gpu
        self.torch, self.dv = torch, dv
        g = GPT2
        self.g = g
        self.k = torch.empty(g.tensor_bytes, dtype=torch.uint8, device="cuda")
        self.v = torch.empty(g.tensor_bytes, dtype=torch.uint8, device="cuda")
        synth_gpu.fill_cache(g, self.k, self.v, seed_of(2))
        self.kb = torch.zeros_like(self.k)
        self.vb = torch.zeros_like(self.v)
        self.cache = dv.Cache.from_geometry(g, self.k, self.v)
        self.cache_b = dv.Cache.from_geometry(g, self.kb, self.vb)
        (self.ps, self.pe), self.deltas = gpt2_ranges()
        self.slab = dv.dv_staging_bytes(self.cache, 0, 1, self.ps, self.pe)
        self.dsz = dv.dv_staging_bytes(self.cache, 0, g.num_layers, *self.deltas[0])
        L = g.num_layers
        self.stg = torch.empty(L * self.slab, dtype=torch.uint8, device="cuda")
        self.dstg = torch.empty(GPT2_DECODE_STEPS * self.dsz, dtype=torch.uint8, device="cuda")
        self.bytes_per_step = 2 * 2 * (L * self.slab + GPT2_DECODE_STEPS * self.dsz)
        self.launches_per_step = 2 * (L + GPT2_DECODE_STEPS)
        self.stream = torch.cuda.Stream()
        self.stream_b = torch.cuda.Stream()
        self.events = [torch.cuda.Event() for _ in range(L + GPT2_DECODE_STEPS)]

    # one step, all buffers in HBM
    def device_step(self, stream, two_streams=True):
        """Packs on `stream`; each unpack waits for its own pack only (an event),
        on a second stream when `two_streams`, so that the two sides of the
        transfer overlap the way a sender and a receiver do."""
        dv, g = self.dv, self.g
        sp, dp = self.stg.data_ptr(), self.dstg.data_ptr()
        sb = self.stream_b if two_streams else stream
        L = g.num_layers
        for l in range(L):
            dv.dv_kv_pack(self.cache, l, l + 1, self.ps, self.pe, (sp + l * self.slab, self.slab),
                          stream)
            self.events[l].record(stream)
        for k, (s, e) in enumerate(self.deltas):
            dv.dv_kv_pack(self.cache, 0, L, s, e, (dp + k * self.dsz, self.dsz), stream)
            self.events[L + k].record(stream)
        for l in range(L):
            sb.wait_event(self.events[l])
            dv.dv_kv_unpack(self.cache_b, l, l + 1, self.ps, self.pe,
                            (sp + l * self.slab, self.slab), sb)
        for k, (s, e) in enumerate(self.deltas):
            sb.wait_event(self.events[L + k])
            dv.dv_kv_unpack(self.cache_b, 0, L, s, e, (dp + k * self.dsz, self.dsz), sb)
        stream.wait_stream(sb)

    def verify(self):
        """After the step (prompt [0,1000) + deltas 1000..1023 = every token of
        every sequence), the second cache equals the first, byte for byte."""
        torch = self.torch
        torch.cuda.synchronize()
        return bool(torch.equal(self.kb, self.k) and torch.equal(self.vb, self.v))

    def clear_b(self):
        self.kb.zero_()
        self.vb.zero_()
        self.torch.cuda.synchronize()

    def capture(self):
        torch = self.torch
        with torch.cuda.stream(self.stream):
            self.device_step(self.stream)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=self.stream, capture_error_mode="relaxed"):
            self.device_step(self.stream)
        self.graph_serial = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph_serial, stream=self.stream, capture_error_mode="relaxed"):
            self.device_step(self.stream, two_streams=False)
        torch.cuda.synchronize()

    def timed_serial(self, steps=50):
        """The same step with every launch on one stream, for reference."""
        torch = self.torch
        for _ in range(3):
            self.graph_serial.replay()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(self.stream):
            e0.record(self.stream)
            for _ in range(steps):
                self.graph_serial.replay()
            e1.record(self.stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / 1e3 / steps

    def timed_value(self, steps, warmup, world):
        torch = self.torch
        for _ in range(warmup):
            self.graph.replay()
        torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(self.stream):
            e0.record(self.stream)
            for _ in range(steps):
                self.graph.replay()
            e1.record(self.stream)
        torch.cuda.synchronize()
        barrier(world)
        return e0.elapsed_time(e1) / 1e3

    def kernel_times(self, reps=5):
        """Average launch time of each launch kind as it runs in the step: the
        step's launches of one kind captured in their own CUDA graph, replayed
        `reps` times (L2 flushed before each replay), CUDA events on the
        launching stream around each replay.  Returns (kind, seconds per
        launch, algorithmic bytes per launch, launches per step)."""
        torch, dv, g = self.torch, self.dv, self.g
        s = self.stream
        sp, dp = self.stg.data_ptr(), self.dstg.data_ptr()
        kinds = {
            "pack prompt layer (tile kernel)": (
                lambda l: dv.dv_kv_pack(self.cache, l, l + 1, self.ps, self.pe,
                                        (sp + l * self.slab, self.slab), s),
                g.num_layers, 2 * self.slab),
            "unpack prompt layer (tile kernel)": (
                lambda l: dv.dv_kv_unpack(self.cache_b, l, l + 1, self.ps, self.pe,
                                          (sp + l * self.slab, self.slab), s),
                g.num_layers, 2 * self.slab),
            "pack decode delta (token kernel)": (
                lambda k: dv.dv_kv_pack(self.cache, 0, g.num_layers, *self.deltas[k],
                                        (dp + k * self.dsz, self.dsz), s),
                GPT2_DECODE_STEPS, 2 * self.dsz),
            "unpack decode delta (token kernel)": (
                lambda k: dv.dv_kv_unpack(self.cache_b, 0, g.num_layers, *self.deltas[k],
                                          (dp + k * self.dsz, self.dsz), s),
                GPT2_DECODE_STEPS, 2 * self.dsz),
        }
        flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        out = []
        for name, (fn, n, nbytes) in kinds.items():
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=s, capture_error_mode="relaxed"):
                for i in range(n):
                    fn(i)
            ms = []
            with torch.cuda.stream(s):
                for r in range(reps + 1):
                    flush.fill_(r)
                    a = torch.cuda.Event(enable_timing=True)
                    b = torch.cuda.Event(enable_timing=True)
                    a.record(s)
                    graph.replay()
                    b.record(s)
                    torch.cuda.synchronize()
                    if r:
                        ms.append(a.elapsed_time(b))
            out.append((name, statistics.median(ms) / 1e3 / n, nbytes, n))
            del graph
        del flush
        return out

    # one step through the public API with pinned host buffers
    def setup_e2e(self):
        torch, dv, g = self.torch, self.dv, self.g
        self.host_prompt = torch.empty(g.num_layers * self.slab, dtype=torch.uint8,
                                       pin_memory=True)
        self.arena = torch.empty(GPT2_DECODE_STEPS * self.dsz, dtype=torch.uint8, pin_memory=True)
        self.slots = (torch.empty(self.slab, dtype=torch.uint8, device="cuda"),
                      torch.empty(self.slab, dtype=torch.uint8, device="cuda"))
        self.copy_stream = torch.cuda.Stream()
        self.in_copy = torch.cuda.Stream()
        self.in_unpack = torch.cuda.Stream()
        self.in_slots = (torch.empty(self.slab, dtype=torch.uint8, device="cuda"),
                         torch.empty(self.slab, dtype=torch.uint8, device="cuda"))
        self.streamer = dv.Streamer(self.slots[0], self.slots[1], self.stream, self.copy_stream)
        self.fetcher = dv.Fetcher(self.in_slots[0], self.in_slots[1], self.in_copy,
                                  self.in_unpack)
        self.restore_staging = torch.empty(GPT2_DECODE_STEPS * self.dsz, dtype=torch.uint8,
                                           device="cuda")
        self.replica = dv.Replica(self.arena, g.batch)

    def e2e_step(self):
        """Layer by layer: the streamer packs layer l and copies it to pinned
        host memory (copy engine); as soon as that copy is done, the fetcher
        copies layer l back into one of its device slots (copy engine) and
        unpacks it into the second cache on its own stream: host-to-device
        traffic of layer l overlaps device-to-host traffic of layer l+1 on the
        full-duplex link, and the unpack of layer l the copy of layer l+1.
        Then the 24 deltas go to the host replica (fused pack into host
        memory) and are restored from it (record-batched, staged)."""
        g = self.g
        s = self.stream
        for l in range(g.num_layers):
            self.streamer.stream_layer(self.cache, l, self.ps, self.pe, self.host_prompt, l0=0)
            self.in_copy.wait_stream(self.copy_stream)  # layer l is in host memory
            self.fetcher.fetch_layer(self.cache_b, l, self.ps, self.pe, self.host_prompt, l0=0)
        self.replica.truncate(0)
        for k, (a, b) in enumerate(self.deltas):
            self.replica.append(self.cache, 0, g.num_layers, a, b, step=k, stream=s)
        si = self.in_unpack
        si.wait_stream(s)
        self.replica.restore_batched(self.cache_b, staging=self.restore_staging, stream=si)
        s.wait_stream(si)

    def timed_e2e(self, steps, warmup, world):
        """Seconds of each of `steps` end-to-end steps, every step timed from an
        idle GPU to its last copy (the host link is shared with other tenants
        of the machine: the median step is the robust figure)."""
        torch = self.torch
        for _ in range(warmup):
            self.e2e_step()
        torch.cuda.synchronize()
        barrier(world)
        ts = []
        for _ in range(steps):
            t0 = time.perf_counter()
            self.e2e_step()
            torch.cuda.synchronize()
            ts.append(time.perf_counter() - t0)
        barrier(world)
        return ts

    # swap section: used cache to pinned host and back, against the link peak
    def swap_section(self, reps=3):
        torch, dv, g = self.torch, self.dv, self.g
        s = self.stream
        zs = np.zeros(g.batch, np.int32)
        full = np.full(g.batch, g.max_seq, np.int32)
        n = dv.dv_staging_bytes(self.cache, 0, g.num_layers, zs, full)
        host = dv.host_empty(n)  # huge-page pinned memory: every pass at the link rate
        dev = torch.empty(n, dtype=torch.uint8, device="cuda")
        staging = torch.empty(4 * (n // g.num_layers), dtype=torch.uint8, device="cuda")

        def timed(fn):
            ts = []
            for _ in range(reps):
                torch.cuda.synchronize()
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                with torch.cuda.stream(s):
                    a.record(s)
                    fn()
                    b.record(s)
                torch.cuda.synchronize()
                ts.append(a.elapsed_time(b) / 1e3)
            return statistics.median(ts)

        res = {"payload_bytes": n}
        res["link_d2h_gbs"] = n / timed(lambda: host.copy_(dev, non_blocking=True)) / 1e9
        res["link_h2d_gbs"] = n / timed(lambda: dev.copy_(host, non_blocking=True)) / 1e9
        host2 = dv.host_empty(n)
        dev2 = torch.empty(n, dtype=torch.uint8, device="cuda")
        s2 = torch.cuda.Stream()

        def both():
            s2.wait_stream(s)
            host.copy_(dev, non_blocking=True)
            with torch.cuda.stream(s2):
                dev2.copy_(host2, non_blocking=True)
            s.wait_stream(s2)

        res["link_bidir_gbs"] = 2 * n / timed(both) / 1e9
        del host2, dev2
        for name, stg in (("fused", None), ("staged", staging)):
            t_out = timed(lambda: dv.dv_swap_out(self.cache, 0, g.num_layers, zs, full, host,
                                                 staging=stg, stream=s))
            t_in = timed(lambda: dv.dv_swap_in(self.cache_b, 0, g.num_layers, zs, full, host,
                                               staging=stg, stream=s))
            res[f"out_{name}_gbs"] = n / t_out / 1e9
            res[f"in_{name}_gbs"] = n / t_in / 1e9
        # the layer-pipelined forms: dv_stream_layer out, dv_fetch_layer in, one
        # layer slab per slot, copies on their own stream
        slab = n // g.num_layers
        slots = [torch.empty(slab, dtype=torch.uint8, device="cuda") for _ in range(4)]
        cp = torch.cuda.Stream()
        st = dv.Streamer(slots[0], slots[1], s, cp)
        ft = dv.Fetcher(slots[2], slots[3], cp, s)

        def stream_out():
            for l in range(g.num_layers):
                st.stream_layer(self.cache, l, zs, full, host)
            s.wait_stream(cp)

        def fetch_in():
            cp.wait_stream(s)
            for l in range(g.num_layers):
                ft.fetch_layer(self.cache_b, l, zs, full, host)

        res["stream_out_gbs"] = n / timed(stream_out) / 1e9
        res["fetch_in_gbs"] = n / timed(fetch_in) / 1e9
        st.close()
        ft.close()
        del slots
        best_out = max(res["out_fused_gbs"], res["out_staged_gbs"])
        best_in = max(res["in_fused_gbs"], res["in_staged_gbs"])
        res["out_frac_of_link"] = best_out / res["link_d2h_gbs"]
        res["in_frac_of_link"] = best_in / res["link_h2d_gbs"]
        del host, dev, staging
        return {k: (round(v, 3) if isinstance(v, float) else v) for k, v in res.items()}


def naive_vs_buffered(torch, dv, reps=3):
    """The pages' one microbenchmark claim (buffered copy vs many small copies,
    §5.1, Fig 11) on GB300: one decode step's delta moved to pinned host memory
    (a) with one copy call per contiguous region (dv_naive_gather) and (b) as
    one pack into device staging plus one copy (the buffered copy), for the
    GPT2-1.5B-shaped cache and one OPT-66B-stage microbatch.  Wall time of the
    calls plus the stream, median of `reps`."""
    from synth.configs import OPT66B_STAGE, opt66b_microbatches
    from synth import gpu as synth_gpu
    out = {}
    s = torch.cuda.Stream()
    for name, g, pos in (("gpt2-1.5b delta", GPT2, np.full(GPT2.batch, GPT2_PROMPT, np.int32)),
                         ("opt-66b-stage delta", OPT66B_STAGE, opt66b_microbatches()[0][0])):
        k = torch.empty(g.tensor_bytes, dtype=torch.uint8, device="cuda")
        v = torch.empty(g.tensor_bytes, dtype=torch.uint8, device="cuda")
        synth_gpu.fill_cache(g, k, v, seed_of(4))
        cache = dv.Cache.from_geometry(g, k, v)
        e = pos + 1
        n = dv.dv_staging_bytes(cache, 0, g.num_layers, pos, e)
        host_a = torch.empty(n, dtype=torch.uint8, pin_memory=True)
        host_b = torch.empty(n, dtype=torch.uint8, pin_memory=True)
        stg = torch.empty(n, dtype=torch.uint8, device="cuda")
        torch.cuda.synchronize()

        def naive():
            return dv.dv_naive_gather(cache, 0, g.num_layers, pos, e, host_a, stream=s)

        def buffered():
            dv.dv_kv_pack(cache, 0, g.num_layers, pos, e, stg, stream=s)
            with torch.cuda.stream(s):
                host_b.copy_(stg, non_blocking=True)

        def wall(fn):
            ts = []
            for _ in range(reps + 1):
                torch.cuda.synchronize()
                t0 = time.perf_counter()
                fn()
                s.synchronize()
                ts.append(time.perf_counter() - t0)
            return statistics.median(ts[1:])

        calls = naive()
        t_naive, t_buf = wall(naive), wall(buffered)
        same = bool(torch.equal(host_a, host_b))
        out[name] = {"bytes": n, "naive_copies": calls, "naive_ms": round(t_naive * 1e3, 3),
                     "buffered_ms": round(t_buf * 1e3, 4),
                     "speedup": round(t_naive / t_buf, 1), "same_bytes": same}
        del k, v, cache, host_a, host_b, stg
        torch.cuda.empty_cache()
    return out


class DecodeStreaming:
    """Decode steps with each step's delta streamed to a host replica (§3
    "Token computation and streaming parallelization", Fig 7c), on the
    GPT2-1.5B-shaped cache.  A decode step is a stand-in compute (a full read
    of the cache's K and V, as attention reads them, reduced on the device)
    followed by the decode write of the new token (an unpack of a seeded
    one-token buffer).  Modes: "compute_only"; "inline", each delta appended
    (dv_replica_append, the pack storing straight into pinned memory) on the
    compute stream after its step; "overlapped", each delta streamed by the
    library's dv_delta_streamer on a side stream that waits only for its own
    step's write, so that it runs while the next step computes.  Each mode's
    `steps` decode steps are one CUDA graph."""

    def __init__(self, torch, dv, steps=GPT2_DECODE_STEPS):
        from synth import gpu as synth_gpu
        self.torch, self.dv, self.steps = torch, dv, steps
        g = self.g = GPT2
        self.k = torch.empty(g.tensor_bytes, dtype=torch.uint8, device="cuda")
        self.v = torch.empty(g.tensor_bytes, dtype=torch.uint8, device="cuda")
        synth_gpu.fill_cache(g, self.k, self.v, seed_of(2))
        self.cache = dv.Cache.from_geometry(g, self.k, self.v)
        (_, _), self.deltas = gpt2_ranges()
        self.dsz = dv.dv_staging_bytes(self.cache, 0, g.num_layers, *self.deltas[0])
        self.tokens = torch.empty(steps * self.dsz, dtype=torch.uint8, device="cuda")
        synth_gpu.fill_tensor(self.tokens, 777, 0, g.kind)
        self.arena = torch.empty(steps * self.dsz, dtype=torch.uint8, pin_memory=True)
        self.replica = dv.Replica(self.arena, g.batch)
        self.acc = torch.zeros(1, dtype=torch.int64, device="cuda")
        self.kv32 = (self.k.view(torch.int32), self.v.view(torch.int32))
        self.s_side = torch.cuda.Stream()

    def _compute_and_write(self, i, s):
        torch, dv, g = self.torch, self.dv, self.g
        self.acc += self.kv32[0].sum(dtype=torch.int64) + self.kv32[1].sum(dtype=torch.int64)
        a, b = self.deltas[i]
        tok = self.tokens[i * self.dsz:(i + 1) * self.dsz]
        dv.dv_kv_unpack(self.cache, 0, g.num_layers, a, b, tok, stream=s)

    def run(self, mode, s, ds=None):
        """Enqueues `steps` decode steps on stream `s` (inside a capture or
        not); `ds` is the delta streamer of the overlapped mode."""
        g = self.g
        for i in range(self.steps):
            self._compute_and_write(i, s)
            a, b = self.deltas[i]
            if mode == "inline":
                self.replica.append(self.cache, 0, g.num_layers, a, b, step=i, stream=s)
            elif mode == "overlapped":
                ds.stream(self.cache, 0, g.num_layers, a, b, step=i)
        if mode == "overlapped":
            ds.join()

    def measure(self, reps=5):
        torch = self.torch
        s = torch.cuda.Stream()
        ds = self.dv.DeltaStreamer(self.replica, s, self.s_side)
        out = {}
        for mode in ("compute_only", "inline", "overlapped"):
            self.replica.truncate(0)
            with torch.cuda.stream(s):
                self.run(mode, s, ds)
            torch.cuda.synchronize()
            self.replica.truncate(0)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=s, capture_error_mode="relaxed"):
                self.run(mode, s, ds)
            ts = []
            with torch.cuda.stream(s):
                for r in range(reps + 1):
                    a = torch.cuda.Event(enable_timing=True)
                    b = torch.cuda.Event(enable_timing=True)
                    a.record(s)
                    graph.replay()
                    b.record(s)
                    torch.cuda.synchronize()
                    if r:
                        ts.append(a.elapsed_time(b))
            out[mode] = statistics.median(ts) / self.steps
            del graph
        same = bool(torch.equal(self.arena.cuda(), self.tokens))
        ds.close()
        base = out["compute_only"]
        return {"steps": self.steps, "delta_bytes": self.dsz,
                "step_ms": {k: round(v, 4) for k, v in out.items()},
                "overhead_inline": round(out["inline"] / base - 1, 4),
                "overhead_overlapped": round(out["overlapped"] / base - 1, 4),
                "replica_equals_written_tokens": same,
                "path": "dv_delta_streamer (side stream) against dv_replica_append on the "
                        "compute stream"}


class MicrobatchSwapping:
    """Microbatch swapping on the OPT-66B-stage workload (§3 "Microbatch
    swapping", Fig 9): N = 4 microbatches share the GPU; each microbatch's
    cache lives in a host replica (a snapshot of its prompt cache plus one
    record per decode step: the swap-out is delta-only).  A round processes
    the microbatches in turn: swap-in (restore snapshot + deltas into a device
    cache, copy engine + unpack), a stand-in compute (a read of the used bytes
    of the cache, as attention reads them) and the decode write of one token
    per active sequence, then the swap-out of that token (a one-token pack
    straight into the replica).
      serial: one device cache, everything in order on one stream (swap-ins
              through a fetcher whose unpacks run on that stream).
      double: the library's dv_swapper over two caches (the pages' 2*M):
              while microbatch x computes in one cache, x+1 is swapped in to
              the other on high-priority streams, and x's update is swapped
              out after its compute."""

    def __init__(self, torch, dv, rounds=8):
        from synth import gpu as synth_gpu
        from synth.configs import OPT66B_STAGE, opt66b_microbatches
        self.torch, self.dv, self.rounds = torch, dv, rounds
        g = self.g = OPT66B_STAGE
        self.synth_gpu = synth_gpu
        self.mbs = opt66b_microbatches()
        self.N = len(self.mbs)
        L = g.num_layers
        self.zs = np.zeros(g.batch, np.int32)
        self.slots = [dv.Cache.from_geometry(
            g, torch.empty(g.tensor_bytes, dtype=torch.uint8, device="cuda"),
            torch.empty(g.tensor_bytes, dtype=torch.uint8, device="cuda")) for _ in range(2)]
        self.per_token = dv.dv_staging_bytes(self.slots[0], 0, L, self.zs,
                                             np.ones(g.batch, np.int32)) // g.batch
        self.fslots = (torch.empty(256 << 20, dtype=torch.uint8, device="cuda"),
                       torch.empty(256 << 20, dtype=torch.uint8, device="cuda"))
        self.replicas, self.arenas, self.lens = [], [], []
        for m, (p, o) in enumerate(self.mbs):
            seed = seed_of(4) * 10 + m
            cap = int((p.sum() + g.batch * (rounds + 1)) * self.per_token)  # + per_op's
            arena = dv.host_empty(cap)
            rep = dv.Replica(arena, g.batch)
            slot = self.slots[0]
            synth_gpu.fill_cache(g, slot.k, slot.v, seed)
            rep.append(slot, 0, L, self.zs, p, step=0)  # the prompt cache arrives
            torch.cuda.synchronize()
            self.arenas.append(arena)
            self.replicas.append(rep)
            self.lens.append(p.copy())
        self.step_no = [1] * self.N
        self.tok = torch.empty(g.batch * self.per_token, dtype=torch.uint8, device="cuda")
        self.acc = torch.zeros(1, dtype=torch.int64, device="cuda")

    def _compute_and_write(self, m, slot, s):
        """Stand-in compute on stream s, then the decode write of microbatch m's
        next token into `slot`; returns the active sequences."""
        torch, dv, g = self.torch, self.dv, self.g
        p, o = self.mbs[m]
        ln = self.lens[m]
        used = int(ln.sum()) * self.per_token  # bytes a decode step would read
        with torch.cuda.stream(s):
            self.acc += slot.k[:used // 2].view(torch.int32).sum(dtype=torch.int64)
            self.acc += slot.v[:used // 2].view(torch.int32).sum(dtype=torch.int64)
        act = ((ln - p) < o).astype(np.int32)
        nt = dv.dv_staging_bytes(slot, 0, g.num_layers, ln, ln + act)
        if nt:
            tok = self.tok[:nt]
            with torch.cuda.stream(s):
                self.synth_gpu.fill_tensor(tok, 1000 * m + self.step_no[m], 0, g.kind, s)
            dv.dv_kv_unpack(slot, 0, g.num_layers, ln, ln + act, tok, stream=s)
        return act

    def run(self, mode, s, s2=None, s3=None):
        """`rounds` rounds over the N microbatches; returns the seconds taken."""
        torch, dv, g = self.torch, self.dv, self.g
        L = g.num_layers
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        if mode == "serial":
            slot = self.slots[0]
            fc = torch.cuda.Stream()
            fetcher = dv.Fetcher(self.fslots[0], self.fslots[1], fc, s)
            for _ in range(self.rounds):
                for m in range(self.N):
                    fc.wait_stream(s)  # after the previous append and compute
                    self.replicas[m].restore_fetched(slot, fetcher)
                    act = self._compute_and_write(m, slot, s)
                    ln = self.lens[m]
                    self.replicas[m].append(slot, 0, L, ln, ln + act, step=self.step_no[m],
                                            stream=s)
                    self.lens[m] = ln + act
                    self.step_no[m] += 1
            torch.cuda.synchronize()
            fetcher.close()
        else:
            fetcher = dv.Fetcher(self.fslots[0], self.fslots[1], s2, s3)
            sw = dv.Swapper(self.slots[0], self.slots[1], fetcher, s, s2)
            order = [m for _ in range(self.rounds) for m in range(self.N)]
            for i, m in enumerate(order):
                sl = sw.acquire(self.replicas[m])
                if i + 1 < len(order):  # the next microbatch comes in to the other cache
                    sw.prefetch(self.replicas[order[i + 1]])
                act = self._compute_and_write(m, self.slots[sl], s)
                ln = self.lens[m]
                sw.release(self.replicas[m], 0, L, ln, ln + act, step=self.step_no[m])
                self.lens[m] = ln + act
                self.step_no[m] += 1
            sw.wait()
            torch.cuda.synchronize()
            sw.close()
            fetcher.close()
        return time.perf_counter() - t0

    def reset(self):
        """Back to the prompt caches: every replica keeps its snapshot only."""
        for m, (p, o) in enumerate(self.mbs):
            self.replicas[m].truncate(1)
            self.lens[m] = p.copy()
            self.step_no[m] = 1

    def measure(self):
        torch = self.torch
        # the swap stream runs at high priority: its short unpack kernels then
        # get SMs ahead of the compute, so its copy-engine pipeline never stalls
        s = torch.cuda.Stream()
        s2, s3 = torch.cuda.Stream(priority=-1), torch.cuda.Stream(priority=-1)
        t_serial = self.run("serial", s)
        self.reset()
        t_double = self.run("double", s, s2, s3)
        steps = self.rounds * self.N
        # the parts on their own: a swap-in (restore) and a compute + write
        slot = self.slots[0]
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        fc = torch.cuda.Stream()
        fetcher = self.dv.Fetcher(self.fslots[0], self.fslots[1], fc, s)
        for m in range(self.N):
            fc.wait_stream(s)
            self.replicas[m].restore_fetched(slot, fetcher)
        s.synchronize()
        t_in = (time.perf_counter() - t0) / self.N
        fetcher.close()
        in_bytes = sum(r.info()[1] for r in self.replicas) / self.N
        t0 = time.perf_counter()
        for m in range(self.N):
            used = int(self.lens[m].sum()) * self.per_token
            with torch.cuda.stream(s):
                self.acc += slot.k[:used // 2].view(torch.int32).sum(dtype=torch.int64)
                self.acc += slot.v[:used // 2].view(torch.int32).sum(dtype=torch.int64)
        s.synchronize()
        t_comp = (time.perf_counter() - t0) / self.N
        ops = self.per_op(s)
        return {"microbatches": self.N, "rounds": self.rounds,
                "ms_per_microbatch_step": {"serial": round(1e3 * t_serial / steps, 3),
                                           "double": round(1e3 * t_double / steps, 3)},
                "speedup_double": round(t_serial / t_double, 3),
                "swap_in_ms": round(1e3 * t_in, 3), "swap_in_bytes": int(in_bytes),
                "swap_in_gbs": round(in_bytes / t_in / 1e9, 1),
                "compute_ms": round(1e3 * t_comp, 3), "per_op": ops,
                "note": "the double schedule can hide at most min(swap-in, compute) per step"}

    def per_op(self, s):
        """Each operation of a microbatch step on its own, payload GB/s (CUDA
        events on `s`, median over the microbatches): the delta append (the
        swap-out of delta-only swapping, fused into the pinned replica), and
        the swap-out / swap-in of a microbatch's whole used prefix (fused, the
        full-prefix reading of a swap)."""
        torch, dv, g = self.torch, self.dv, self.g
        L = g.num_layers
        slot = self.slots[0]
        big = max(dv.dv_staging_bytes(slot, 0, L, self.zs, ln) for ln in self.lens)
        host = dv.host_empty(big)

        def ev_time(fn):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            a.record(s)
            fn()
            b.record(s)
            torch.cuda.synchronize()
            return a.elapsed_time(b) / 1e3

        app, out, inn = [], [], []
        for m in range(self.N):
            ln = self.lens[m]
            rep = self.replicas[m]
            nt = dv.dv_staging_bytes(slot, 0, L, ln, ln + 1)
            for _ in range(2):  # the first of each is a warm-up
                t = ev_time(lambda: rep.append(slot, 0, L, ln, ln + 1, step=self.step_no[m],
                                               stream=s))
                rep.truncate(self.step_no[m])
            app.append((nt, t))
            n = dv.dv_staging_bytes(slot, 0, L, self.zs, ln)
            for _ in range(2):
                to = ev_time(lambda: dv.dv_swap_out(slot, 0, L, self.zs, ln, host, stream=s))
                ti = ev_time(lambda: dv.dv_swap_in(slot, 0, L, self.zs, ln, host, stream=s))
            out.append((n, to))
            inn.append((n, ti))
        del host
        med = lambda xs: statistics.median(b / t / 1e9 for b, t in xs)  # noqa: E731
        return {"delta_append_gbs": round(med(app), 1),
                "delta_append_us": round(1e6 * statistics.median(t for _, t in app), 1),
                "delta_bytes": int(statistics.median(b for b, _ in app)),
                "prefix_swap_out_gbs": round(med(out), 1),
                "prefix_swap_in_gbs": round(med(inn), 1),
                "prefix_bytes": int(statistics.median(b for b, _ in out))}


def workload_section(torch, dv):
    """The other workloads' operations on their full sizes (seeded caches, the
    same calls the parity tests check), as payload GB/s; one timed run each
    after a warm-up of the same call."""
    from synth.configs import TINY, GPT2, OPT13B, BLOOM_STAGE, tiny_ranges, opt13b_lengths, \
        bloom_lengths, BLOOM_DECODE_STEPS
    from synth import gpu as synth_gpu
    s = torch.cuda.Stream()
    out = {}

    def cache_of(g, seed):
        k = torch.empty(g.tensor_bytes, dtype=torch.uint8, device="cuda")
        v = torch.empty(g.tensor_bytes, dtype=torch.uint8, device="cuda")
        synth_gpu.fill_cache(g, k, v, seed)
        return dv.Cache.from_geometry(g, k, v)

    def timed(fn, reps=3):
        ts = []
        for _ in range(reps + 1):
            torch.cuda.synchronize()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(s):
                a.record(s)
                fn()
                b.record(s)
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b) / 1e3)
        return statistics.median(ts[1:])

    # workload 1: tiny cache, prompt [0,37) and the decode token (latency)
    c = cache_of(TINY, seed_of(1))
    (ps, pe), (ds, de) = tiny_ranges()
    buf = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    L = TINY.num_layers
    def graph_us(fn, n=20):
        """GPU time per call: n calls captured in one graph, replayed."""
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s, capture_error_mode="relaxed"):
            for _ in range(n):
                fn()
        t = timed(graph.replay)
        del graph
        return round(1e6 * t / n, 2)

    def host_us(fn, n=200):
        """Host time per call (argument checks and the launch), eager."""
        with torch.cuda.stream(s):
            fn()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            for _ in range(n):
                fn()
            t1 = time.perf_counter()
        torch.cuda.synchronize()
        return round(1e6 * (t1 - t0) / n, 2)

    pp = lambda: dv.dv_kv_pack(c, 0, L, ps, pe, buf, s)  # noqa: E731
    pt = lambda: dv.dv_kv_pack(c, 0, L, ds, de, buf, s)  # noqa: E731
    up = lambda: dv.dv_kv_unpack(c, 0, L, ps, pe, buf, s)  # noqa: E731
    out["tiny"] = {"pack_prompt_gpu_us": graph_us(pp), "pack_token_gpu_us": graph_us(pt),
                   "unpack_prompt_gpu_us": graph_us(up), "host_us_per_call": host_us(pt)}

    def restore_pair(g, c, rep, staging=None, reps=3):
        """One replica restored record by record and record-batched into two
        caches of the same initial content: times (CUDA events on the stream,
        host submission included) and whether the results agree."""
        a = cache_of(g, 0)
        b = cache_of(g, 0)
        t_rec = timed(lambda: rep.restore(a, staging=staging, stream=s), reps)
        t_bat = timed(lambda: rep.restore_batched(b, staging=staging, stream=s), reps)
        torch.cuda.synchronize()
        same = bool(torch.equal(a.k, b.k) and torch.equal(a.v, b.v))
        del a, b
        return t_rec, t_bat, same

    # restore of a snapshot + decode deltas, record by record vs batched
    rb = {}
    nd = 64
    zs = np.zeros(TINY.batch, np.int32)
    arena = torch.empty(dv.dv_staging_bytes(c, 0, L, zs, pe + nd) + 4096, dtype=torch.uint8,
                        pin_memory=True)
    rep = dv.Replica(arena, TINY.batch)
    rep.append(c, 0, L, ps, pe, step=0, stream=s)
    for k in range(nd):
        rep.append(c, 0, L, pe + k, pe + k + 1, step=k + 1, stream=s)
    t_rec, t_bat, same = restore_pair(TINY, c, rep)
    rb["tiny: [0,37) + 64 one-token deltas, fused"] = {
        "records": nd + 1, "per_record_us": round(1e6 * t_rec, 1),
        "batched_us": round(1e6 * t_bat, 1), "speedup": round(t_rec / t_bat, 2),
        "same_result": same}
    rep.close()
    del c, buf, arena
    g = GPT2
    c = cache_of(g, seed_of(2))
    zs = np.zeros(g.batch, np.int32)
    p0 = np.full(g.batch, 1000, np.int32)
    nd = 24
    arena = torch.empty(dv.dv_staging_bytes(c, 0, g.num_layers, zs, p0 + nd), dtype=torch.uint8,
                        pin_memory=True)
    rep = dv.Replica(arena, g.batch)
    rep.append(c, 0, g.num_layers, zs, p0, step=0, stream=s)
    for k in range(nd):
        rep.append(c, 0, g.num_layers, p0 + k, p0 + k + 1, step=k + 1, stream=s)
    stg = torch.empty(dv.dv_staging_bytes(c, 0, 1, zs, p0), dtype=torch.uint8, device="cuda")
    for name, st in (("fused", None), ("staged (one-layer staging buffer)", stg)):
        t_rec, t_bat, same = restore_pair(g, c, rep, staging=st)
        rb[f"gpt2-1.5b: [0,1000) + 24 one-token deltas, {name}"] = {
            "records": nd + 1, "bytes": rep.info()[1], "per_record_ms": round(1e3 * t_rec, 3),
            "batched_ms": round(1e3 * t_bat, 3), "speedup": round(t_rec / t_bat, 3),
            "same_result": same}
    # the deltas alone (the swap-in of delta-only swapping, snapshot elsewhere)
    rep.truncate(0)
    for k in range(nd):
        rep.append(c, 0, g.num_layers, p0 + k, p0 + k + 1, step=k + 1, stream=s)
    for name, st in (("fused", None), ("staged (one-layer staging buffer)", stg)):
        t_rec, t_bat, same = restore_pair(g, c, rep, staging=st)
        rb[f"gpt2-1.5b: 24 one-token deltas only, {name}"] = {
            "records": nd, "bytes": rep.info()[1], "per_record_us": round(1e6 * t_rec, 1),
            "batched_us": round(1e6 * t_bat, 1), "speedup": round(t_rec / t_bat, 3),
            "same_result": same}
    out["restore_batched"] = rb
    rep.close()
    del c, arena, stg
    torch.cuda.empty_cache()
    # workload 3: OPT-13B swap-out / swap-in of the used prefixes
    g = OPT13B
    c = cache_of(g, seed_of(3))
    lens = opt13b_lengths()
    zs = np.zeros(g.batch, np.int32)
    n = dv.dv_staging_bytes(c, 0, g.num_layers, zs, lens)
    host = dv.host_empty(n)
    stg = torch.empty(4 * (n // g.num_layers), dtype=torch.uint8, device="cuda")
    res = {"payload_bytes": n}
    for name, st in (("fused", None), ("staged", stg)):
        res[f"out_{name}_gbs"] = round(n / timed(lambda: dv.dv_swap_out(
            c, 0, g.num_layers, zs, lens, host, staging=st, stream=s)) / 1e9, 1)
        res[f"in_{name}_gbs"] = round(n / timed(lambda: dv.dv_swap_in(
            c, 0, g.num_layers, zs, lens, host, staging=st, stream=s)) / 1e9, 1)
    out["opt-13b swap"] = res
    del c, host, stg
    torch.cuda.empty_cache()
    # workload 5: BLOOM stage, snapshot + 256 one-token deltas to a replica, restore
    g = BLOOM_STAGE
    c = cache_of(g, seed_of(5))
    len0 = bloom_lengths()
    zs = np.zeros(g.batch, np.int32)
    total = dv.dv_staging_bytes(c, 0, g.num_layers, zs, len0 + BLOOM_DECODE_STEPS)
    arena = dv.host_empty(total)
    rep = dv.Replica(arena, g.batch)
    snap = dv.dv_staging_bytes(c, 0, g.num_layers, zs, len0)

    def append_all():
        rep.truncate(0)
        rep.append(c, 0, g.num_layers, zs, len0, step=0, stream=s)
        pos = len0.copy()
        for k in range(1, BLOOM_DECODE_STEPS + 1):
            rep.append(c, 0, g.num_layers, pos, pos + 1, step=k, stream=s)
            pos = pos + 1

    t_app = timed(append_all, reps=1)
    back = cache_of(g, 0)
    t_res = timed(lambda: rep.restore(back, stream=s), reps=1)
    t_bat = timed(lambda: rep.restore_batched(back, stream=s), reps=1)
    out["bloom-176b-stage replica"] = {
        "records": BLOOM_DECODE_STEPS + 1, "bytes": total, "snapshot_bytes": snap,
        "append_gbs": round(total / t_app / 1e9, 1), "restore_gbs": round(total / t_res / 1e9, 1),
        "restore_batched_gbs": round(total / t_bat / 1e9, 1), "delta_append_us": None}
    # one delta on its own (the per-step replication cost)
    pos = len0 + BLOOM_DECODE_STEPS - 1
    rep.truncate(BLOOM_DECODE_STEPS)
    t_one = timed(lambda: (rep.truncate(BLOOM_DECODE_STEPS),
                           rep.append(c, 0, g.num_layers, pos, pos + 1, step=BLOOM_DECODE_STEPS,
                                      stream=s)))
    out["bloom-176b-stage replica"]["delta_append_us"] = round(1e6 * t_one, 1)
    rep.close()
    del c, back, arena
    torch.cuda.empty_cache()
    return out


def hbm_section(torch, dv, peak):
    """Device-resident pack and unpack of each larger workload's own ranges
    (staging buffer in device memory, inputs larger than L2, L2 flushed before
    every timed launch or graph replay), as GB/s read + written and as a
    fraction of the HBM copy peak.  Per workload: every resident layer in one
    launch, the same layers one launch per layer (a CUDA graph of the layer
    launches, as layer streaming issues them), and one-token decode deltas
    (a CUDA graph of 8 deltas at positions 8 tokens apart, so that no two
    share a cache line).  Prefix ranges go to the tile kernel and deltas to
    the token kernel, which is also what the automatic choice takes for
    them; each is forced here so that the label names the kernel timed.
    After the timed unpacks, the second cache is packed again and must give
    the staging bytes back."""
    from synth.configs import OPT13B, OPT66B_STAGE, BLOOM_STAGE, opt13b_lengths, \
        opt66b_microbatches, bloom_lengths
    from synth import gpu as synth_gpu
    s = torch.cuda.Stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    tile, token = dv.DV_VARIANT_TILE, dv.DV_VARIANT_TOKEN

    def timed(fn, per=1, reps=5):
        ms = []
        with torch.cuda.stream(s):
            for r in range(reps + 1):
                flush.fill_(r)
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(s)
                fn()
                b.record(s)
                torch.cuda.synchronize()
                if r:
                    ms.append(a.elapsed_time(b))
        return statistics.median(ms) / 1e3 / per

    def graphed(calls):
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s, capture_error_mode="relaxed"):
            for fn in calls:
                fn()
        return graph

    def figure(payload, secs, kernel, launches):
        gbs = 2 * payload / secs / 1e9
        return {"kernel": kernel, "launches": launches, "payload_bytes_per_launch": payload,
                "us_per_launch": round(secs * 1e6, 2), "gbs": round(gbs, 1),
                "frac_of_peak": round(gbs / peak, 4),
                "frac_of_nominal": round(gbs / HBM_NOMINAL_GBS, 4)}

    cases = [
        ("opt-13b: used prefixes [0, len), lognormal(400)", OPT13B, 3,
         np.zeros(OPT13B.batch, np.int32), opt13b_lengths()),
        ("opt-66b-stage: microbatch 0 at the end of generation [0, p + o)", OPT66B_STAGE, 4,
         np.zeros(OPT66B_STAGE.batch, np.int32),
         (lambda p, o: (p + o).astype(np.int32))(*opt66b_microbatches()[0])),
        ("bloom-176b-stage: replica snapshot [0, len0), uniform [64, 1536]", BLOOM_STAGE, 5,
         np.zeros(BLOOM_STAGE.batch, np.int32), bloom_lengths()),
    ]
    out = {}
    for name, g, idx, st, en in cases:
        L = g.num_layers
        ka = torch.empty(g.tensor_bytes, dtype=torch.uint8, device="cuda")
        va = torch.empty(g.tensor_bytes, dtype=torch.uint8, device="cuda")
        synth_gpu.fill_cache(g, ka, va, seed_of(idx))
        ca = dv.Cache.from_geometry(g, ka, va)
        kb = torch.zeros(g.tensor_bytes, dtype=torch.uint8, device="cuda")
        vb = torch.zeros(g.tensor_bytes, dtype=torch.uint8, device="cuda")
        cb = dv.Cache.from_geometry(g, kb, vb)
        n = dv.dv_staging_bytes(ca, 0, L, st, en)
        slab = n // L
        stg = torch.empty(n, dtype=torch.uint8, device="cuda")
        sp = stg.data_ptr()
        res = {"layers": L, "payload_bytes": n}
        res["pack_all_layers"] = figure(n, timed(
            lambda: dv.dv_kv_pack(ca, 0, L, st, en, stg, s, variant=tile)), "tile", 1)
        res["unpack_all_layers"] = figure(n, timed(
            lambda: dv.dv_kv_unpack(cb, 0, L, st, en, stg, s, variant=tile)), "tile", 1)
        gp = graphed([lambda l=l: dv.dv_kv_pack(ca, l, l + 1, st, en, (sp + l * slab, slab), s,
                                                 variant=tile) for l in range(L)])
        res["pack_per_layer"] = figure(slab, timed(gp.replay, per=L), "tile", L)
        gu = graphed([lambda l=l: dv.dv_kv_unpack(cb, l, l + 1, st, en, (sp + l * slab, slab),
                                                   s, variant=tile) for l in range(L)])
        res["unpack_per_layer"] = figure(slab, timed(gu.replay, per=L), "tile", L)
        del gp, gu
        back = torch.empty_like(stg)
        dv.dv_kv_pack(cb, 0, L, st, en, back, s)
        torch.cuda.synchronize()
        res["verified"] = bool(torch.equal(back, stg))
        del back
        # one-token deltas at 8 positions 8 tokens apart, inside the cache
        pos = [((en - 1 + 8 * k) % g.max_seq).astype(np.int32) for k in range(8)]
        dsz = dv.dv_staging_bytes(ca, 0, L, pos[0], pos[0] + 1)
        gp = graphed([lambda k=k: dv.dv_kv_pack(ca, 0, L, pos[k], pos[k] + 1,
                                                 (sp + k * dsz, dsz), s, variant=token)
                      for k in range(8)])
        res["delta_pack"] = figure(dsz, timed(gp.replay, per=8), "token", 8)
        gu = graphed([lambda k=k: dv.dv_kv_unpack(cb, 0, L, pos[k], pos[k] + 1,
                                                   (sp + k * dsz, dsz), s, variant=token)
                      for k in range(8)])
        res["delta_unpack"] = figure(dsz, timed(gu.replay, per=8), "token", 8)
        del gp, gu
        out[name] = res
        del ca, cb, ka, va, kb, vb, stg
        torch.cuda.empty_cache()
    del flush
    return out


def gpt2_section(torch, steps=100):
    """The GPT2-1.5B step (48 per-layer prompt packs, 24 one-token deltas, all
    unpacked into a second cache) as a side section: its value with every
    launch on one stream (packs, then unpacks: each slab read ~5 GB of traffic
    after it was written), the same step with each unpack on a second stream
    right after its pack (sender and receiver overlapped; part of each slab
    can still be in L2 then), per-kernel times, the swap / link figures and
    the end-to-end step through the API (layer streamer out, fetcher in,
    deltas to a replica and back)."""
    b = Bench()
    b.capture()
    serial = b.timed_serial(steps)
    two = b.timed_value(steps, 3, 1) / steps
    b.clear_b()
    b.graph_serial.replay()
    ok = b.verify()
    kt = b.kernel_times()
    swap = b.swap_section()
    b.setup_e2e()
    b.clear_b()
    ts = b.timed_e2e(10, 2, 1)
    e2e_ok = b.verify()
    hbm_peak = peaks()[0]
    out = {"workload": ("gpt2-1.5b-shaped KV cache L48 B8 H25 D64 S1024 fp16: prompt [0,1000) "
                        "packed layer by layer + 24 one-token decode deltas, all unpacked into a "
                        "second cache"),
           "bytes_per_step": b.bytes_per_step,
           "value": round(b.bytes_per_step / serial / 1e9, 2),
           "frac_of_measured_peak": round(b.bytes_per_step / serial / 1e9 / hbm_peak, 4),
           "timing": "one stream: every pack, then every unpack; CUDA graph; mean over "
                     f"{steps} replays",
           "two_stream_value": round(b.bytes_per_step / two / 1e9, 2),
           "two_stream_note": "each unpack right after its pack on a second stream: part of "
                              "the slab may still be in L2",
           "verified": ok,
           "kernels": [{"kernel": n_, "avg_launch_us": round(t * 1e6, 2),
                        "gbs": round(nb / t / 1e9, 1),
                        "frac_of_peak": round(nb / t / 1e9 / hbm_peak, 4),
                        "launches_per_step": c} for n_, t, nb, c in kt],
           "e2e_gbs": round(b.bytes_per_step / statistics.median(ts) / 1e9, 2),
           "e2e_verified": e2e_ok,
           "e2e_path": "per layer: dv_stream_layer (pack + D2H copy) then dv_fetch_layer (H2D "
                       "copy + unpack on the fetcher's two streams); dv_replica_append x24 "
                       "(fused) + dv_replica_restore_batched (staged)"}
    del b
    torch.cuda.empty_cache()
    return out, swap


def run_mine(args):
    import torch
    rank, world, local = dist_init()
    if world == 1:
        torch.cuda.set_device(0)
    import __graft_entry__
    if rank == 0:
        __graft_entry__.build()
    barrier(world)
    __graft_entry__.build()  # no-op when up to date; every rank imports the package
    b = Bloom()
    b.capture()
    clocks = ClockSampler(local)
    clocks.start()
    secs = b.timed_value(args.steps, max(args.warmup, 3), world)
    clk = clocks.stop()
    secs = max_over_ranks(secs, world)
    value = whole_job_rate(b.bytes_per_step, args.steps, secs, world)
    b.clear_b()
    b.graph.replay()
    step_ok = b.verify()
    # kernel roofline, live: the launch kind with the most time per step
    kt = b.kernel_times()
    hbm_peak, peak_kind = peaks()
    name, t_launch, nbytes, _ = max(kt, key=lambda r: r[1] * r[3])
    achieved = nbytes / t_launch / 1e9
    # e2e through the public API with host buffers
    link = link_peaks(torch)
    b.setup_e2e()
    e2e_steps = max(3, min(args.steps, 20))
    b.clear_b()
    e2e_ts = b.timed_e2e(e2e_steps, 2, world)
    e2e_ok = b.verify()
    e2e_med = max_over_ranks(statistics.median(e2e_ts), world)
    e2e_value = whole_job_rate(b.bytes_per_step, 1, e2e_med, world)
    e2e_all = whole_job_rate(b.bytes_per_step, e2e_steps, max_over_ranks(sum(e2e_ts), world),
                             world)
    link_bytes = 2 * b.total  # every log byte crosses once each way
    serial_link_s = b.total / (link["d2h_gbs"] * 1e9) + b.total / (link["h2d_gbs"] * 1e9)
    b.close_e2e()
    hostmem = host_memory_passes(torch, b.dv, b.log) if rank == 0 and not args.no_swap else None
    per_step = {"bytes_per_step": b.bytes_per_step, "log_bytes": b.total,
                "snapshot_bytes": b.snap, "delta_bytes": b.dsz,
                "launches_per_step": b.launches_per_step()}
    del b
    torch.cuda.empty_cache()
    # The sections below describe one GPU and only rank 0 prints them: the other
    # ranks skip them (they would pin about 20 GB of host memory each).
    extra = rank == 0 and not args.no_swap
    gpt2, swap = gpt2_section(torch) if extra else (None, None)
    naive = naive_vs_buffered(torch, __import__("kv_cache_streaming_gb300")) if extra else None
    import kv_cache_streaming_gb300 as dv
    streaming = DecodeStreaming(torch, dv).measure() if extra else None
    mb_swap = MicrobatchSwapping(torch, dv).measure() if extra else None
    torch.cuda.empty_cache()
    workloads = workload_section(torch, dv) if extra else None
    torch.cuda.empty_cache()
    hbm = hbm_section(torch, dv, hbm_peak) if extra else None
    cpu = None
    if rank == 0 and world == 1:  # the CPU baseline is an N = 1 figure
        cores = host_cores()
        smp = OracleSample(2 * cores, threads=cores)
        moved, dt, passes = smp.run(cpu_seconds=CPU_SAMPLE_SECONDS)
        smp.close()
        one = OracleSample(2)
        moved1, dt1, passes1 = one.run(cpu_seconds=CPU_SAMPLE_SECONDS)
        cpu = {"value": round(moved / dt / 1e9, 3), "unit": UNIT, "cores": smp.threads,
               "kind": "oracle",
               "sample": smp.desc + f", {passes} passes, {dt:.1f} s on {smp.threads} threads",
               "single_thread": {"value": round(moved1 / dt1 / 1e9, 3), "cores": 1,
                                 "sample": one.desc + f", {passes1} passes, {dt1:.1f} s"}}
        del smp, one
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3),
        "ms_per_step": round(1e3 * secs / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u16", "data": "synthetic",
        "config": workload_config(world),
        "timing": "CUDA-graph replay of the step on one stream, CUDA events on that stream; "
                  "per-kernel figures: each launch kind of one step in its own CUDA graph, L2 "
                  "flushed before each replay, median of 5",
        "step_verified": step_ok,
        "frac_of_measured_peak": round(value / hbm_peak, 4),
        "frac_of_nominal_peak": round(value / HBM_NOMINAL_GBS, 4),
        "step": per_step,
        "roofline": {"bound": "hbm", "kernel": name, "achieved": round(achieved, 1),
                     "peak": hbm_peak, "unit": "GB/s", "frac": round(achieved / hbm_peak, 4),
                     "peak_kind": peak_kind, "nominal_peak": HBM_NOMINAL_GBS,
                     "frac_of_nominal": round(achieved / HBM_NOMINAL_GBS, 4),
                     "traffic": TRAFFIC_PER_LAUNCH.get(name),
                     "algorithmic_bytes_per_launch": nbytes,
                     "avg_launch_us": round(t_launch * 1e6, 2)},
        "kernels": [{"kernel": n_, "avg_launch_us": round(t * 1e6, 2),
                     "gbs": round(nb / t / 1e9, 1), "frac_of_peak": round(nb / t / 1e9 / hbm_peak, 4),
                     "launches_per_step": c, "ms_per_step": round(t * c * 1e3, 3),
                     "traffic": TRAFFIC_PER_LAUNCH.get(n_)}
                    for n_, t, nb, c in kt],
        "cpu_baseline": cpu,
        "e2e": {"value": round(e2e_value, 2), "unit": UNIT, "h2d_bytes_per_step": per_step["log_bytes"],
                "d2h_bytes_per_step": per_step["log_bytes"], "steps": e2e_steps, "verified": e2e_ok,
                "link_gbs": round(world * link_bytes / e2e_med / 1e9, 2),
                "link_peaks_gbs": link,
                "link_frac_of_serial_peak": round(serial_link_s / e2e_med, 4),
                "link_frac_of_bidir_peak": round(link_bytes / e2e_med / 1e9 / link["bidir_gbs"], 4),
                "timing": "median step (each step synchronised); over all steps: "
                          f"{e2e_all:.1f} GB/s, slowest step {max(e2e_ts) * 1e3:.1f} ms, "
                          f"fastest {min(e2e_ts) * 1e3:.1f} ms",
                "step_ms": [round(x * 1e3, 1) for x in e2e_ts],
                "path": "dv_replica_append_streamed of the snapshot one layer at a time "
                        "(a layer streamer: each pack into one of two device slots while "
                        "the other is copied to the host by a copy engine), each layer "
                        "restored through a fetcher (dv_replica_restore_fetched_steps) while "
                        "the next goes out; then the 256 deltas appended the same way, each "
                        f"{Bloom.E2E_DELTA_CHUNK} restored as a run of records while the next "
                        f"{Bloom.E2E_DELTA_CHUNK} go out (one-layer slots)"},
        "host_memory": hostmem,
        "gpt2_step": gpt2,
        "swap": swap,
        "naive_vs_buffered": naive,
        "decode_streaming": streaming,
        "microbatch_swapping": mb_swap,
        "workloads": workloads,
        "hbm_by_workload": hbm,
        "gpu_launches": per_step["launches_per_step"] * args.steps,
        "clocks": clk,
        "gpu": gpu_identity(local),
    }
    print(json.dumps(line), flush=True)


def run_kernel_case(case):
    """One kernel of the step on the first 8 layers of the workload's cache
    (inputs larger than L2, under 1 GB on the device), launched 5 times."""
    from dataclasses import replace
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import kv_cache_streaming_gb300 as dv
    from synth import gpu as synth_gpu
    torch.cuda.set_device(0)
    if case == "record-restore":
        run_record_case(torch, dv, synth_gpu)
        return
    if case.startswith("flat") or case.startswith("short-ragged"):
        run_flat_case(case, torch, dv, synth_gpu)
        return
    if case.startswith("group"):
        run_group_case(case, torch, dv, synth_gpu)
        return
    if case.startswith("ragged"):
        run_ragged_case(case, torch, dv, synth_gpu)
        return
    if case.startswith("delta-graph"):
        run_delta_graph_case(case, torch, dv, synth_gpu)
        return
    if case.startswith("bloom"):
        run_bloom_case(case, torch, dv, synth_gpu)
        return
    if case == "gpt2-step":
        b = Bench()
        with torch.cuda.stream(b.stream):
            b.device_step(b.stream, two_streams=False)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=b.stream, capture_error_mode="relaxed"):
            b.device_step(b.stream, two_streams=False)
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
        print(f"gpt2-step: 3 replays of {b.launches_per_step} launches, verified {b.verify()}")
        return
    g = replace(GPT2, num_layers=8)
    k = torch.empty(g.tensor_bytes, dtype=torch.uint8, device="cuda")
    v = torch.empty(g.tensor_bytes, dtype=torch.uint8, device="cuda")
    synth_gpu.fill_cache(g, k, v, seed_of(2))
    cache = dv.Cache.from_geometry(g, k, v)
    (ps, pe), deltas = gpt2_ranges()
    s, e = deltas[0] if case.startswith("delta") else (ps, pe)
    n = dv.dv_staging_bytes(cache, 0, g.num_layers, s, e)
    if case.startswith("swap"):
        host = torch.empty(n, dtype=torch.uint8, pin_memory=True)
        dv.dv_swap_out(cache, 0, g.num_layers, s, e, host)
        for _ in range(5):
            if case == "swap-out":
                dv.dv_swap_out(cache, 0, g.num_layers, s, e, host)
            else:
                dv.dv_swap_in(cache, 0, g.num_layers, s, e, host)
        torch.cuda.synchronize()
        print(f"{case}: 5 fused launches of {n} payload bytes each over the host link")
        return
    stg = torch.empty(n, dtype=torch.uint8, device="cuda")
    dv.dv_kv_pack(cache, 0, g.num_layers, s, e, stg)
    for _ in range(5):
        if case.endswith("-pack"):
            dv.dv_kv_pack(cache, 0, g.num_layers, s, e, stg)
        else:
            dv.dv_kv_unpack(cache, 0, g.num_layers, s, e, stg)
    torch.cuda.synchronize()
    print(f"{case}: 5 launches of {2 * n} algorithmic bytes each")


def run_flat_case(case, torch, dv, synth_gpu):
    """Ragged short ranges: 16..64 tokens at seeded positions of each of the 8
    sequences of the OPT-13B-shaped cache, all 40 layers (about 260 MB of
    staging, more than L2), 5 launches; flat-*: the flat kernel forced,
    short-ragged-*: the automatic choice (the tile kernel for the ranges of
    more than 32 tokens, grouped tiles in a second launch for the others)."""
    from synth.configs import OPT13B
    g = OPT13B
    k = torch.empty(g.tensor_bytes, dtype=torch.uint8, device="cuda")
    v = torch.empty(g.tensor_bytes, dtype=torch.uint8, device="cuda")
    synth_gpu.fill_cache(g, k, v, seed_of(3))
    cache = dv.Cache.from_geometry(g, k, v)
    rng = np.random.default_rng(seed_of(3))
    s = rng.integers(0, g.max_seq - 64, size=g.batch).astype(np.int32)
    e = (s + rng.integers(16, 65, size=g.batch)).astype(np.int32)
    n = dv.dv_staging_bytes(cache, 0, g.num_layers, s, e)
    stg = torch.empty(n, dtype=torch.uint8, device="cuda")
    var = dv.DV_VARIANT_FLAT if case.startswith("flat") else dv.DV_VARIANT_AUTO
    dv.dv_kv_pack(cache, 0, g.num_layers, s, e, stg, variant=var)
    for _ in range(5):
        if case.endswith("-pack"):
            dv.dv_kv_pack(cache, 0, g.num_layers, s, e, stg, variant=var)
        else:
            dv.dv_kv_unpack(cache, 0, g.num_layers, s, e, stg, variant=var)
    torch.cuda.synchronize()
    print(f"{case}: 5 launches of {2 * n} algorithmic bytes each "
          f"(ranges of {int((e - s).min())}..{int((e - s).max())} tokens)")


def run_group_case(case, torch, dv, synth_gpu):
    """Ragged short ranges in grouped tiles: 2..32 tokens at seeded positions of
    each of 32 sequences, a cache of 40 layers, 40 heads, head_dim 128 (fp16)
    and 128 token slots (3.4 GB; about 450 MB of staging, more than L2), every
    range at most half the tile kernel's token block, so the tile kernel's
    launch is all grouped tiles (group_kernel); 5 launches."""
    from synth.configs import Geometry
    g = Geometry("group-c16", 40, 32, 40, 128, 128, 2, "fp16")
    k = torch.empty(g.tensor_bytes, dtype=torch.uint8, device="cuda")
    v = torch.empty(g.tensor_bytes, dtype=torch.uint8, device="cuda")
    synth_gpu.fill_cache(g, k, v, seed_of(3))
    cache = dv.Cache.from_geometry(g, k, v)
    rng = np.random.default_rng(seed_of(3))
    s = rng.integers(0, g.max_seq - 32, size=g.batch).astype(np.int32)
    e = (s + rng.integers(2, 33, size=g.batch)).astype(np.int32)
    n = dv.dv_staging_bytes(cache, 0, g.num_layers, s, e)
    stg = torch.empty(n, dtype=torch.uint8, device="cuda")
    tile = dv.DV_VARIANT_TILE
    dv.dv_kv_pack(cache, 0, g.num_layers, s, e, stg, variant=tile)
    for _ in range(5):
        if case.endswith("-pack"):
            dv.dv_kv_pack(cache, 0, g.num_layers, s, e, stg, variant=tile)
        else:
            dv.dv_kv_unpack(cache, 0, g.num_layers, s, e, stg, variant=tile)
    torch.cuda.synchronize()
    print(f"{case}: 5 launches of {2 * n} algorithmic bytes each "
          f"(ranges of {int((e - s).min())}..{int((e - s).max())} tokens)")


def run_ragged_case(case, torch, dv, synth_gpu):
    """Ragged long ranges, the tile kernel on the OPT-13B workload's used
    prefixes (lognormal, median 400): 4 of the 40 layers (about 590 MB of
    staging, more than L2; under 2 GB on the device), 5 launches."""
    from dataclasses import replace
    from synth.configs import OPT13B, opt13b_lengths
    g = replace(OPT13B, num_layers=4)
    k = torch.empty(g.tensor_bytes, dtype=torch.uint8, device="cuda")
    v = torch.empty(g.tensor_bytes, dtype=torch.uint8, device="cuda")
    synth_gpu.fill_cache(g, k, v, seed_of(3))
    cache = dv.Cache.from_geometry(g, k, v)
    s = np.zeros(g.batch, np.int32)
    e = opt13b_lengths()
    n = dv.dv_staging_bytes(cache, 0, g.num_layers, s, e)
    stg = torch.empty(n, dtype=torch.uint8, device="cuda")
    tile = dv.DV_VARIANT_TILE
    dv.dv_kv_pack(cache, 0, g.num_layers, s, e, stg, variant=tile)
    for _ in range(5):
        if case.endswith("-pack"):
            dv.dv_kv_pack(cache, 0, g.num_layers, s, e, stg, variant=tile)
        else:
            dv.dv_kv_unpack(cache, 0, g.num_layers, s, e, stg, variant=tile)
    torch.cuda.synchronize()
    print(f"{case}: 5 launches of {2 * n} algorithmic bytes each "
          f"(prefixes of {int(e.min())}..{int(e.max())} tokens)")


def run_delta_graph_case(case, torch, dv, synth_gpu):
    """One-token deltas of every sequence at all layers of a BLOOM-stage-shaped
    cache (batch 32, 112 heads, head_dim 128, bf16) cut to 4 layers and
    max_seq 512 (3.8 GB): 32 deltas at positions 8 tokens apart (no two share
    a K line), captured in one CUDA graph and replayed 5 times.  The graph
    writes 235 MB of deltas, more than L2, so graph-level DRAM counters include
    the write-back of the partly written K lines."""
    from dataclasses import replace
    from synth.configs import BLOOM_STAGE
    g = replace(BLOOM_STAGE, num_layers=4, max_seq=512)
    k = torch.empty(g.tensor_bytes, dtype=torch.uint8, device="cuda")
    v = torch.empty(g.tensor_bytes, dtype=torch.uint8, device="cuda")
    synth_gpu.fill_cache(g, k, v, seed_of(5))
    cache = dv.Cache.from_geometry(g, k, v)
    nd = 32
    pos = [np.full(g.batch, 8 * i + 3, np.int32) for i in range(nd)]
    one = dv.dv_staging_bytes(cache, 0, g.num_layers, pos[0], pos[0] + 1)
    stg = torch.empty(nd * one, dtype=torch.uint8, device="cuda")
    sp = stg.data_ptr()
    s = torch.cuda.Stream()
    fn = dv.dv_kv_pack if case.endswith("-pack") else dv.dv_kv_unpack
    for i in range(nd):  # eager first calls (occupancy queries) and the staging contents
        dv.dv_kv_pack(cache, 0, g.num_layers, pos[i], pos[i] + 1, (sp + i * one, one), s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s, capture_error_mode="relaxed"):
        for i in range(nd):
            fn(cache, 0, g.num_layers, pos[i], pos[i] + 1, (sp + i * one, one), s)
    for _ in range(5):
        graph.replay()
    torch.cuda.synchronize()
    print(f"{case}: 5 replays of a graph of {nd} deltas of {one} bytes each")


def run_bloom_case(case, torch, dv, synth_gpu):
    """The headline step's kernels on its workload (BLOOM-176B stage, bf16,
    112 heads, head_dim 128, max_seq 2048, len0 uniform in [64, 1536]) cut to
    2 of the 14 layers and the first 16 of the 32 sequences: 3.8 GB of cache,
    1.4 GB of snapshot staging (inputs larger than L2, a few GB on the device).
    Traffic per launch scales to the full step's launch by the bytes moved."""
    from dataclasses import replace
    g = replace(BLOOM_STAGE, num_layers=2, batch=16)
    L = g.num_layers
    k = torch.empty(g.tensor_bytes, dtype=torch.uint8, device="cuda")
    v = torch.empty(g.tensor_bytes, dtype=torch.uint8, device="cuda")
    synth_gpu.fill_cache(g, k, v, seed_of(5))
    cache = dv.Cache.from_geometry(g, k, v)
    len0 = bloom_lengths()[:g.batch]
    zs = np.zeros(g.batch, np.int32)
    if case in ("bloom-snapshot-pack", "bloom-snapshot-unpack"):
        n = dv.dv_staging_bytes(cache, 0, L, zs, len0)
        stg = torch.empty(n, dtype=torch.uint8, device="cuda")
        dv.dv_kv_pack(cache, 0, L, zs, len0, stg)
        for _ in range(3):
            if case.endswith("-pack"):
                dv.dv_kv_pack(cache, 0, L, zs, len0, stg)
            else:
                dv.dv_kv_unpack(cache, 0, L, zs, len0, stg)
        torch.cuda.synchronize()
        print(f"{case}: 3 launches of {2 * n} algorithmic bytes each")
        return
    nd = BLOOM_DECODE_STEPS
    one = dv.dv_staging_bytes(cache, 0, L, len0, len0 + 1)
    log = torch.empty(nd * one, dtype=torch.uint8, device="cuda")
    lp = log.data_ptr()
    for j in range(nd):
        dv.dv_kv_pack(cache, 0, L, len0 + j, len0 + j + 1, (lp + j * one, one))
    if case == "bloom-delta-pack":
        for j in range(0, 64, 8):
            dv.dv_kv_pack(cache, 0, L, len0 + j, len0 + j + 1, (lp + j * one, one))
        torch.cuda.synchronize()
        print(f"{case}: 8 launches of {2 * one} algorithmic bytes each")
        return
    back = dv.Cache.from_geometry(g, torch.zeros_like(k), torch.zeros_like(v))
    records = [(0, L, len0 + j, len0 + j + 1) for j in range(nd)]
    for _ in range(3):
        dv.dv_kv_unpack_records(back, records, log)
    torch.cuda.synchronize()
    print(f"{case}: 3 launches of {2 * nd * one} algorithmic bytes each ({nd} records)")


def run_record_case(torch, dv, synth_gpu):
    """A replica of 96 one-token decode deltas (positions 928..1023) of the
    workload's cache, the even and the odd sequences taking turns (so no two
    consecutive records share their live sequences and no run forms: the record
    kernel's case), 118 MB, restored 5 times through a device staging buffer:
    each restore is one host-to-device copy and one launch of the record kernel
    (96 records of batch 8 fit one launch)."""
    g = GPT2
    k = torch.empty(g.tensor_bytes, dtype=torch.uint8, device="cuda")
    v = torch.empty(g.tensor_bytes, dtype=torch.uint8, device="cuda")
    synth_gpu.fill_cache(g, k, v, seed_of(2))
    cache = dv.Cache.from_geometry(g, k, v)
    back = dv.Cache.from_geometry(g, torch.zeros_like(k), torch.zeros_like(v))
    p0, nd = 928, 96
    pos = np.full(g.batch, p0, np.int32)
    parity = np.arange(g.batch) % 2
    recs = [(pos + i, pos + i + (parity == i % 2)) for i in range(nd)]
    total = sum(dv.dv_staging_bytes(cache, 0, g.num_layers, a, b) for a, b in recs)
    arena = torch.empty(total, dtype=torch.uint8, pin_memory=True)
    rep = dv.Replica(arena, g.batch)
    for i, (a, b) in enumerate(recs):
        rep.append(cache, 0, g.num_layers, a, b, step=i)
    stg = torch.empty(total, dtype=torch.uint8, device="cuda")
    for _ in range(5):
        rep.restore_batched(back, staging=stg)
    torch.cuda.synchronize()
    for s_, e_ in recs:  # every restored slice equals the source cache's
        n = dv.dv_staging_bytes(cache, 0, g.num_layers, s_, e_)
        a = torch.empty(n, dtype=torch.uint8, device="cuda")
        b = torch.empty(n, dtype=torch.uint8, device="cuda")
        dv.dv_kv_pack(cache, 0, g.num_layers, s_, e_, a)
        dv.dv_kv_pack(back, 0, g.num_layers, s_, e_, b)
        torch.cuda.synchronize()
        assert torch.equal(a, b), "restored slices differ from the source cache"
    rep.close()
    print(f"record-restore: 5 launches of {2 * total} algorithmic bytes each "
          f"({nd} records, {total} bytes)")


def main():
    args = parse_args()
    if args.kernel_case:
        run_kernel_case(args.kernel_case)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_mine(args)


if __name__ == "__main__":
    main()
