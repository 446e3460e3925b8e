"""The bounds-checking build of the library (build(debug=True): every global
access checked against its buffer's extent, a miss skipped and flagged
GDN_DEV_BOUNDS instead of read or written) runs the workloads, the edge
shapes and every entry point with no flag and the oracle's results. It runs
in a child process, since a process loads one build of the library."""
import os
import subprocess
import sys

import pytest
import torch

from speculative_decode_hybrid_gb300 import build as B

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_debug_bounds_build_runs_clean():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    lib = B.build(debug=True)
    env = dict(os.environ, GDNSPEC_LIB=lib)
    r = subprocess.run([sys.executable, os.path.join(HERE, "debug_bounds_cases.py")], env=env,
                       capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "debug-bounds ok" in r.stdout
