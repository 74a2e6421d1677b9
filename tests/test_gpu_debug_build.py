"""The range-checking build (-DSPEC_DEBUG) on the GPU.

A child process loads libspecverify_debug.so (SPEC_VERIFY_DEBUG=1), calls
every entry point against the oracle (tests/debug_build_run.py) and checks
that no device-side range check failed: the kernels' own indexing stays
inside every buffer on these inputs, and the checks change no result.
"""

import os
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_every_entry_point_passes_its_range_checks():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ, SPEC_VERIFY_DEBUG="1")
    r = subprocess.run([sys.executable, os.path.join(HERE, "debug_build_run.py")], env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "range checks failed: 0" in r.stdout and "debug build ok" in r.stdout, r.stdout[-2000:]
