"""The CUDA-core route for bf16 head dim 256 (LS_FORCE_SIMT=1), checked with
the same small-shape parity cases as the tensor-core kernels.  The library
reads the switch once per process, so the tensor-core small-shape tests of
test_gpu_parity.py run in a child pytest process with the switch set."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_simt_route_small_shapes(cuda_device):
    env = dict(os.environ, LS_FORCE_SIMT="1")
    cmd = [sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_gpu_parity.py"), "-m", "gpu",
           "-k", "test_small_shapes and tc_", "-q", "-x", "-p", "no:cacheprovider"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, f"LS_FORCE_SIMT=1:\n{r.stdout[-3000:]}\n{r.stderr[-2000:]}"
