import sys
from pathlib import Path

ROOT = Path(__file__).resolve().parent.parent
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))


import os

import pytest


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a)")
    # Build (when missing or stale) the copy library, the GPU input generator
    # and the oracle before any test module imports them.
    import importlib.util
    from synth import build as synth_build
    import oracle
    # load the build script by path: importing the package loads libdv.so
    spec = importlib.util.spec_from_file_location(
        "_dv_build", ROOT / "kv_cache_streaming_gb300" / "build.py")
    dv_build = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(dv_build)
    dv_build.build()
    synth_build.build()
    oracle.load()


if os.environ.get("DV_LIBRARY") == "checked":
    @pytest.fixture(autouse=True)
    def _no_out_of_bounds_access(request):
        """Under the bounds-checked library, every GPU test must leave no
        recorded out-of-bounds access."""
        yield
        if request.node.get_closest_marker("gpu"):
            import kv_cache_streaming_gb300 as dv
            fault = dv.dv_debug_fault()
            assert fault == 0, f"out-of-bounds access recorded: {fault:#x}"
