"""The checking build (GDR_DEBUG: device-side index checks on the forward pass's global
accesses, a failed one recorded as GDR_ERR_BOUNDS and its access skipped) on small
parity cases, dense and packed, both gates, both paths, with many segments, and the
per-channel decay forward with warm-up segments and packed sequences: results
equal the oracle's within the usual tolerances and no check fails (GPU).  It runs in a
child process, since this one has the regular build loaded."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_checking_build_passes_parity_with_clean_status():
    sys.path.insert(0, ROOT)
    from chunked_gated_delta_07_gb300 import _build
    lib = _build.build(variant="debug")
    env = dict(os.environ, GDR_LIB=lib)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "debug_build_checks.py")], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "checking build: ok" in r.stdout
