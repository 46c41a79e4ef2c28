"""The five synthetic workloads: cache geometries, seeds and range draws.

Shapes follow the DejaVu paper's evaluated models (GPT2-1.5B, OPT-13B,
OPT-66B and BLOOM-176B; fp16, BLOOM in bf16 here), with the KV cache
preallocated at the maximum sequence length as in FasterTransformer
("DejaVu: KV-Cache Streaming...", §3 DejaVuLib implementation, Fig 6).
The request lengths of the paper come from LMSys conversations, which are not
used: seeded draws stand in for them (lognormal with sigma 1.0, or uniform).

Nothing here addresses a cache or orders a staging buffer.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

SEED_BASE = 20240301


@dataclass(frozen=True)
class Geometry:
    """A max-length-preallocated KV cache: ``num_layers`` resident layers,
    ``batch`` sequences, ``num_heads`` heads of ``head_dim`` elements,
    ``max_seq`` token slots, ``elem_bytes`` bytes per element."""
    name: str
    num_layers: int
    batch: int
    num_heads: int
    head_dim: int
    max_seq: int
    elem_bytes: int = 2
    kind: str = "fp16"          # fp16 | bf16 | fp32 | raw (fill rule only)
    layer_stride_elems: int = 0  # 0: B*H*D*S (layers stacked densely)

    @property
    def layer_elems(self) -> int:
        return self.layer_stride_elems or (
            self.batch * self.num_heads * self.head_dim * self.max_seq)

    @property
    def tensor_elems(self) -> int:
        """Elements in one of the K or V allocations (all layers)."""
        return self.num_layers * self.layer_elems

    @property
    def tensor_bytes(self) -> int:
        return self.tensor_elems * self.elem_bytes


@dataclass
class Workload:
    index: int                  # 1..5, in the order the workloads are listed
    geom: Geometry
    seed: int
    description: str
    extra: dict = field(default_factory=dict)


TINY = Geometry("tiny", 2, 2, 4, 64, 128, 2, "fp16")
GPT2 = Geometry("gpt2-1.5b", 48, 8, 25, 64, 1024, 2, "fp16")
OPT13B = Geometry("opt-13b", 40, 8, 40, 128, 2048, 2, "fp16")
OPT66B_STAGE = Geometry("opt-66b-stage", 16, 16, 72, 128, 2048, 2, "fp16")
BLOOM_STAGE = Geometry("bloom-176b-stage", 14, 32, 112, 128, 2048, 2, "bf16")

GEOMETRIES = [TINY, GPT2, OPT13B, OPT66B_STAGE, BLOOM_STAGE]


def seed_of(index: int) -> int:
    return SEED_BASE + index


# ---- range draws ---------------------------------------------------------

def tiny_ranges():
    """Prompt [0,37) on both sequences, then the decode token at 37."""
    b = TINY.batch
    prompt = (np.zeros(b, np.int32), np.full(b, 37, np.int32))
    decode = (np.full(b, 37, np.int32), np.full(b, 38, np.int32))
    return prompt, decode


GPT2_PROMPT = 1000
GPT2_DECODE_STEPS = 24


def gpt2_ranges():
    """Prompt [0,1000) on all 8 sequences, then 24 one-token decode ranges."""
    b = GPT2.batch
    prompt = (np.zeros(b, np.int32), np.full(b, GPT2_PROMPT, np.int32))
    decode = [(np.full(b, GPT2_PROMPT + k, np.int32), np.full(b, GPT2_PROMPT + k + 1, np.int32))
              for k in range(GPT2_DECODE_STEPS)]
    return prompt, decode


def _lognormal_int(rng, median, size, lo, hi):
    v = np.rint(rng.lognormal(math.log(median), 1.0, size=size))
    return np.clip(v, lo, hi).astype(np.int32)


def opt13b_lengths(seed: int | None = None) -> np.ndarray:
    """Used lengths of the 8 sequences: lognormal, median 400, sigma 1.0,
    rounded, clipped to [16, 2048]."""
    rng = np.random.default_rng(seed_of(3) if seed is None else seed)
    return _lognormal_int(rng, 400.0, OPT13B.batch, 16, OPT13B.max_seq)


def opt66b_microbatches(seed: int | None = None, n_micro: int = 4):
    """Per microbatch: prompt lengths p (lognormal median 250, clipped to
    [16,1024]) and output budgets o (lognormal median 200, clipped to
    [1, 2048-p-1]), 16 sequences each."""
    rng = np.random.default_rng(seed_of(4) if seed is None else seed)
    out = []
    for _ in range(n_micro):
        p = _lognormal_int(rng, 250.0, OPT66B_STAGE.batch, 16, 1024)
        o_raw = np.rint(rng.lognormal(math.log(200.0), 1.0, size=OPT66B_STAGE.batch))
        o = np.clip(o_raw, 1, OPT66B_STAGE.max_seq - p - 1).astype(np.int32)
        out.append((p, o))
    return out


BLOOM_DECODE_STEPS = 256


def bloom_lengths(seed: int | None = None) -> np.ndarray:
    """Initial lengths of the 32 sequences, uniform on [64, 1536]."""
    rng = np.random.default_rng(seed_of(5) if seed is None else seed)
    return rng.integers(64, 1537, size=BLOOM_STAGE.batch).astype(np.int32)


def workloads():
    return [
        Workload(1, TINY, seed_of(1), "tiny: prompt [0,37) then decode token 37"),
        Workload(2, GPT2, seed_of(2), "gpt2-1.5b: prompt 1000 layer-streamed, 24 decode deltas"),
        Workload(3, OPT13B, seed_of(3), "opt-13b: swap-out/in of lognormal used prefixes"),
        Workload(4, OPT66B_STAGE, seed_of(4), "opt-66b stage: 4 microbatches swap-in/delta/swap-out"),
        Workload(5, BLOOM_STAGE, seed_of(5), "bloom-176b stage: 256 deltas to a replica, restore"),
    ]
