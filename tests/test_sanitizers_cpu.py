"""The oracle's C code and the CUDA library's host code under AddressSanitizer and
UndefinedBehaviorSanitizer (CPU only; compute-sanitizer is not available for the
device side, whose checking build is GDR_DEBUG, tested on the GPU).

Both are built with -fsanitize=address,undefined and exercised in a child process
that preloads the sanitizer runtimes: every oracle entry point on small dense and
packed cases (results equal to the regular build's), and the library's argument
refusals.  A sanitizer report makes the child exit non-zero."""
import os
import re
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _runtime(name):
    path = subprocess.run(["gcc", f"-print-file-name={name}"], capture_output=True, text=True).stdout.strip()
    return path if os.path.isabs(path) and os.path.exists(path) else None


def _env(**kw):
    asan, ubsan = _runtime("libasan.so"), _runtime("libubsan.so")
    if not asan or not ubsan:
        pytest.skip("sanitizer runtimes not installed")
    return dict(os.environ, LD_PRELOAD=f"{asan}:{ubsan}",
                ASAN_OPTIONS="detect_leaks=0:abort_on_error=0:halt_on_error=1",
                UBSAN_OPTIONS="halt_on_error=1:print_stacktrace=1", OMP_NUM_THREADS="2", **kw)


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_oracle_and_host_code_under_asan_and_ubsan(tmp_path):
    sys.path.insert(0, ROOT)
    import oracle
    from chunked_gated_delta_07_gb300 import _build
    oracle.build()
    lib, rlib = oracle.build_sanitized(str(tmp_path))
    gdr_lib = _build.build(variant="asan")
    env = _env(GDR_LIB=gdr_lib)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "sanitized_checks.py"), lib, rlib],
                       env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-6000:]
    assert "sanitized checks: ok" in r.stdout
    assert "runtime error" not in r.stderr and "AddressSanitizer" not in r.stderr, r.stderr[-6000:]


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_a_planted_overflow_in_the_oracle_is_reported(tmp_path):
    """The harness itself: the oracle's key loop made to write one element past its
    buffer is caught (the child fails with a sanitizer report: UndefinedBehaviorSanitizer's
    object-size check or AddressSanitizer, whichever sees it first)."""
    sys.path.insert(0, ROOT)
    import oracle
    src = open(os.path.join(ROOT, "oracle", "gdr_oracle.c")).read()
    mutated, n = re.subn(r"for \(int i = 0; i < dk; i\+\+\) \{\n(\s+)kt\[i\] = widen",
                         r"for (int i = 0; i <= dk; i++) {\n\1kt[i] = widen", src, count=1)
    assert n == 1
    bad = tmp_path / "gdr_oracle_bad.c"
    bad.write_text(mutated)
    lib, rlib = oracle.build_sanitized(str(tmp_path / "bad"), gdr_src=str(bad))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "sanitized_checks.py"), lib, rlib,
                        "--forward-only"], env=_env(), capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, r.stdout[-2000:]
    assert "AddressSanitizer" in r.stderr or "runtime error" in r.stderr, r.stderr[-2000:]
