"""The MP_CHECKS build on the GPU (the stand-in for a memory checker): tests/checks_child.py runs
in a child process with MAGICPIG_CHECKS=1, so that it loads libmagicpig_checks.so rather than
the product library this process has loaded. Clean inputs pass every index check and match the
oracle; a corrupted bucket table raises MP_ERR_BOUNDS with a bucket site, and nothing faults."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_checks_build_is_clean_on_valid_inputs_and_reports_a_corrupted_bucket_table():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from lsh_sampled_sparse_gb300.build import build
    build(checks=True)
    env = dict(os.environ, MAGICPIG_CHECKS="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "checks_child.py")],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "checks ok" in r.stdout
