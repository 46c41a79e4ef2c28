"""Host-memory transfers under extreme grid caps (the DV_HOST_CTAS override,
read once per process): 1 (one tile-kernel CTA, two flat / record CTAs, four
token CTAs walk the whole transfer) and 0 (no cap).  Fused swaps through every
kernel and a fused batched restore still produce the oracle's bytes."""
import os
import subprocess
import sys
from pathlib import Path

import pytest

pytestmark = pytest.mark.gpu
ROOT = Path(__file__).resolve().parent.parent

CHILD = r'''
import numpy as np, torch
import kv_cache_streaming_gb300 as dv
import oracle
from synth.configs import Geometry
from tests import gpu_helpers as H
ORC = oracle.default()
g = Geometry("cap", 2, 3, 4, 128, 96, 2, "fp16")
kh, vh = H.host_cache(g, 88)
cache = H.device_cache(g, fill=(kh, vh))
zero = np.zeros(3, np.int32)
cases = [(zero, np.array([90, 96, 40], np.int32)),             # long: tile kernel
         (np.array([3, 50, 7], np.int32), np.array([9, 53, 30], np.int32)),  # ragged: flat
         (np.array([5, 60, 9], np.int32), np.array([6, 61, 10], np.int32))]  # one token: token
for s, e in cases:
    n = ORC.staging_bytes(g, 0, 2, s, e)
    want = ORC.pack(g, kh, vh, 0, 2, s, e)
    host = H.pinned(n)
    dv.dv_swap_out(cache, 0, 2, s, e, host)
    torch.cuda.synchronize()
    assert np.array_equal(host.numpy()[:n], want)
    back = H.device_cache(g, fill=0x5A)
    dv.dv_swap_in(back, 0, 2, s, e, host)
    kw = np.full(g.tensor_bytes, 0x5A, np.uint8); vw = np.full(g.tensor_bytes, 0x5A, np.uint8)
    ORC.unpack(g, kw, vw, 0, 2, s, e, want)
    assert np.array_equal(H.to_np(back.k), kw) and np.array_equal(H.to_np(back.v), vw)
# a fused batched restore: the record kernel on host memory
arena = H.pinned(ORC.staging_bytes(g, 0, 2, zero, np.full(3, 96, np.int32)))
rep = dv.Replica(arena, 3)
pos = np.array([10, 4, 20], np.int32)
rep.append(cache, 0, 2, zero, pos, step=0)
recs = [(0, 2, zero, pos.copy())]
for k in range(1, 6):
    rep.append(cache, 0, 2, pos, pos + 1, step=k)
    recs.append((0, 2, pos.copy(), pos + 1))
    pos = pos + 1
z = H.device_cache(g, fill="zero")
rep.restore_batched(z)
kw, vw = ORC.restore(g, [(a, b, s_, e_, ORC.pack(g, kh, vh, a, b, s_, e_)) for a, b, s_, e_ in recs])
assert np.array_equal(H.to_np(z.k), kw) and np.array_equal(H.to_np(z.v), vw)
print("ok")
'''


@pytest.mark.parametrize("ctas", ["1", "0"])
def test_fused_transfers_under_grid_caps(ctas):
    env = dict(os.environ, DV_HOST_CTAS=ctas, PYTHONPATH=str(ROOT))
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=str(ROOT), env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:] + r.stderr[-2000:]
