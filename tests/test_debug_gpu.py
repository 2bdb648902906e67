"""The index-checking debug build (-DTPAR_DEBUG) stands in for a memory
checker: every kernel form runs with each computed index checked against its
buffer (a failed check is reported through the device error word and the
access skipped, never a trap), and the checks are shown to fire."""
import os
import subprocess
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.gpu
def test_every_kernel_form_under_index_checks():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ, TPAR_DEBUG="1")
    r = subprocess.run([sys.executable, os.path.join(HERE, "debug_checks.py")], env=env, capture_output=True,
                       text=True, timeout=1200)
    assert r.returncode == 0, (r.stdout[-3000:], r.stderr[-3000:])
    assert "debug checks passed" in r.stdout
