"""The usage example in README.md runs as written, and its pack / unpack /
swap / replica calls round-trip the cache."""
import re
from pathlib import Path

import pytest
import torch

pytestmark = pytest.mark.gpu
ROOT = Path(__file__).resolve().parent.parent


def test_readme_example_runs():
    text = (ROOT / "README.md").read_text()
    code = re.search(r"```python\n(.*?)```", text, re.S).group(1)
    ns = {}
    exec(compile(code, "README.md", "exec"), ns)
    torch.cuda.synchronize()
    k, v, stg, host = ns["k"], ns["v"], ns["stg"], ns["host"]
    assert torch.equal(host.cuda(), stg)  # the swap-out and the streamer wrote the pack's bytes
    back = torch.empty_like(stg)
    cache = ns["cache"]
    ns["dv"].dv_kv_pack(cache, 0, ns["L"], ns["s"], ns["e"], back)
    torch.cuda.synchronize()
    assert torch.equal(back, stg)  # the fetches and restores put the same bytes back
    del ns
    torch.cuda.empty_cache()
