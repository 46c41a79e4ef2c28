"""The usage example (examples/usage.py, which the README points to) runs as
written, and its pack / unpack / swap / stream / replica calls round-trip the
cache."""
import importlib.util
from pathlib import Path

import pytest
import torch

pytestmark = pytest.mark.gpu
ROOT = Path(__file__).resolve().parent.parent


def test_usage_example_runs():
    spec = importlib.util.spec_from_file_location("usage", ROOT / "examples" / "usage.py")
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    ns = mod.main()
    torch.cuda.synchronize()
    dv, cache, stg, host = ns["dv"], ns["cache"], ns["stg"], ns["host"]
    assert torch.equal(host.cuda(), stg)  # the swap-out and the streamer wrote the pack's bytes
    back = torch.empty_like(stg)
    L, s, e = ns["L"], ns["s"], ns["e"]
    dv.dv_kv_pack(cache, 0, L, s, e, back)
    torch.cuda.synchronize()
    assert torch.equal(back, stg)  # the fetches and restores put the same bytes back
    # each swapped cache holds its microbatch's prompt and tokens
    for c in ns["caches"]:
        got = torch.empty_like(stg)
        dv.dv_kv_pack(c, 0, L, s, e, got)
        torch.cuda.synchronize()
        assert torch.equal(got, stg)
    for r, _ in ns["mbs"]:
        assert r.info()[0] == 3
    del ns
    torch.cuda.empty_cache()
