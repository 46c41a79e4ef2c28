"""Microbatch swapping with delta-only swap-outs and two device slots: after
several rounds, each microbatch's host replica restores to a cache equal to a
reference that received the same decode writes, whether the rounds ran on one
slot in order or on two slots with swaps overlapping compute."""
import gc
import sys
from pathlib import Path

import pytest
import torch

import kv_cache_streaming_gb300 as dv

sys.path.insert(0, str(Path(__file__).resolve().parent.parent))
import bench  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode", ["serial", "double"])
def test_microbatch_swapping_restores_the_reference(mode):
    mb = bench.MicrobatchSwapping(torch, dv, rounds=2, keep_refs=True)
    s, s2, s3 = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    mb.run(mode, s, s2, s3)
    assert all(rep.info()[0] == 1 + 2 for rep in mb.replicas)  # snapshot + 2 deltas
    assert mb.check()
    del mb
    gc.collect()
    torch.cuda.empty_cache()
