"""The parity suites again, under the bounds-checked build of the library:
every global access of every kernel is checked against the extents the host
validated, and no test may leave a recorded out-of-bounds access (checked in
tests/conftest.py)."""
import importlib.util
import os
import subprocess
import sys
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent
pytestmark = pytest.mark.gpu


def test_parity_suites_under_the_checked_build():
    spec = importlib.util.spec_from_file_location(
        "_dv_build", ROOT / "kv_cache_streaming_gb300" / "build.py")
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    b.build(checked=True)
    env = dict(os.environ, DV_LIBRARY="checked")
    cmd = [sys.executable, "-m", "pytest", "-x", "-q", "-m", "gpu", "-p", "no:cacheprovider",
           "tests/test_gpu_parity.py", "tests/test_gpu_streaming.py",
           "tests/test_gpu_restore_batched.py", "tests/test_gpu_fuzz.py",
           "tests/test_gpu_microbatch.py"]
    r = subprocess.run(cmd, cwd=str(ROOT), env=env, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]


def test_regular_build_reports_no_checks():
    import kv_cache_streaming_gb300 as dv
    if os.environ.get("DV_LIBRARY") != "checked":
        assert dv.dv_debug_fault() is None
