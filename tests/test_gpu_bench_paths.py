"""The benchmark's own step and end-to-end step, in the launch configuration
it times (two streams, one CUDA graph; the layer-pipelined host round trip),
leave the second cache equal to the first on every token, and the streamed
host bytes are the oracle's, on sampled elements."""
import gc
import sys
from pathlib import Path

import numpy as np
import pytest
import torch

sys.path.insert(0, str(Path(__file__).resolve().parent.parent))
import bench  # noqa: E402
import oracle  # noqa: E402
from synth.configs import seed_of  # noqa: E402
from tests import gpu_helpers as H  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def b():
    bb = bench.Bench()
    yield bb
    del bb
    gc.collect()
    torch.cuda.empty_cache()


def test_graph_step_restores_every_token(b):
    b.clear_b()
    b.capture()
    b.graph.replay()
    assert b.verify()
    # the packed prompt slabs are the oracle's, on sampled elements
    H.sampled_check(oracle.default(), b.g, seed_of(2), b.stg, 0, b.g.num_layers, b.ps, b.pe,
                    np.random.default_rng(6))


def test_serial_graph_step_restores_every_token(b):
    b.clear_b()
    b.graph_serial.replay()
    assert b.verify()


def test_e2e_step_restores_every_token(b):
    b.setup_e2e()
    b.clear_b()
    b.e2e_step()
    assert b.verify()
    H.sampled_check(oracle.default(), b.g, seed_of(2), b.host_prompt, 0, b.g.num_layers, b.ps,
                    b.pe, np.random.default_rng(7))


@pytest.fixture(scope="module")
def bloom():
    gc.collect()
    torch.cuda.empty_cache()
    bb = bench.Bloom()
    yield bb
    del bb
    gc.collect()
    torch.cuda.empty_cache()


def test_headline_step_restores_every_token(bloom):
    """The headline step as the bench times it (one CUDA graph): the second
    cache equals the live one on [0, len0 + 256) of every sequence and is
    zero beyond; the snapshot and sampled deltas of the log are the oracle's,
    on sampled elements."""
    b = bloom
    b.clear_b()
    b.capture()
    b.graph.replay()
    assert b.verify()
    g, L = b.g, b.g.num_layers
    rng = np.random.default_rng(8)
    orc = oracle.default()
    H.sampled_check(orc, g, seed_of(5), b.log[:b.snap], 0, L, b.zs, b.len0, rng)
    for k in (0, 1, 7, 8, 255):
        a, e = b.deltas[k]
        off = b.snap + k * b.dsz
        H.sampled_check(orc, g, seed_of(5), b.log[off:off + b.dsz], 0, L, a, e, rng,
                        nsamples=50_000)


def test_headline_e2e_step_restores_every_token(bloom):
    """The end-to-end step (appends to the host replica, restore through the
    fetcher) restores every token, and the host log holds the bytes of the
    device log the graph step packs."""
    b = bloom
    with torch.cuda.stream(b.stream):
        b.device_step(b.stream)
    b.setup_e2e()
    b.clear_b()
    b.e2e_step()
    assert b.verify()
    step = 1 << 30
    for off in range(0, b.total, step):
        n = min(step, b.total - off)
        assert torch.equal(b.arena[off:off + n].cuda(), b.log[off:off + n]), off
    b.close_e2e()
