"""The alternative kernels behind the environment switches, checked with the
same small-shape parity cases as the default ones.

LS_TC_FWD_VARIANT / LS_TC_BWD_VARIANT select the staged tensor-core kernels
(kept for comparison with the defaults) and LS_FORCE_SIMT routes bf16 head
dim 256 through the SIMT kernels.  The library reads each switch once per
process, so every setting runs the tensor-core small-shape tests of
test_gpu_parity.py in a child pytest process with the switch set.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SETTINGS = [
    {"LS_TC_FWD_VARIANT": "1", "LS_TC_BWD_VARIANT": "1"},
    {"LS_TC_FWD_VARIANT": "2", "LS_TC_BWD_VARIANT": "2"},
    {"LS_TC_FWD_VARIANT": "3"},
    {"LS_FORCE_SIMT": "1"},
]


@pytest.mark.parametrize("env", SETTINGS, ids=["+".join(f"{k}={v}" for k, v in s.items()) for s in SETTINGS])
def test_variant_small_shapes(cuda_device, env):
    full_env = dict(os.environ)
    full_env.update(env)
    cmd = [sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_gpu_parity.py"), "-m", "gpu",
           "-k", "test_small_shapes and tc_", "-q", "-x", "-p", "no:cacheprovider"]
    r = subprocess.run(cmd, cwd=ROOT, env=full_env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, f"{env}:\n{r.stdout[-3000:]}\n{r.stderr[-2000:]}"
