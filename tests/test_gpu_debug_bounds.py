"""The GPU suite once more on the bounds-checked build of the library (SD_DEBUG_BOUNDS).

Every index the matmul kernels compute for a global access or a weight, activation or partial-sum
copy (per call and inside the one-launch pass, the per-operation CUDA graph of the 64-layer stack
included) is checked against the extent the call's shapes imply; a failed check records its site in
the status word and skips the access.  The suite runs in a child process with SDV_DEBUG_BOUNDS=1,
and the conftest's fixture asserts after every test that no check failed.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.gpu


def test_gpu_suite_with_bounds_checks():
    if os.environ.get("SDV_DEBUG_BOUNDS") == "1":
        pytest.skip("this suite already runs on the bounds-checked build")
    env = dict(os.environ, SDV_DEBUG_BOUNDS="1")
    r = subprocess.run([sys.executable, "-c",
                        "from speculative_decoding_verify_gb300 import build as b; b.build(debug_bounds=True)"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    r = subprocess.run([sys.executable, "-m", "pytest", "tests", "-m", "gpu", "-x", "-q", "-p", "no:cacheprovider",
                        "--ignore=tests/test_gpu_debug_bounds.py"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=2400)
    assert r.returncode == 0, (r.stdout + r.stderr)[-4000:]
