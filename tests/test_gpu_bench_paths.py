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
