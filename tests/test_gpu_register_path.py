"""The parity tests with every world on the register kernels (GPU).

ZR_FUSED_KERNEL=1 sends every world to the plain-load kernels: the register
reduce-scatter and all-reduce (otherwise for worlds up to 4) and k_direct_reg
for the direct step and its norm pass (otherwise for gradients in pinned host
memory). The parity tests are run in a child process with it set, so the
register path is held to the oracle at the worlds and layouts (1 to 32
replicas; irregular, ragged, backward and random arrival) that the copy
pipeline takes in an ordinary run.
"""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

FILES = ["tests/test_gpu_parity.py", "tests/test_gpu_range.py", "tests/test_gpu_order.py",
         "tests/test_gpu_gradcheck.py", "tests/test_gpu_graph.py", "tests/test_gpu_e2e.py"]


def test_parity_tests_pass_on_the_register_kernels():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from zero_partition_aware_gb300 import build
    build.build()
    env = dict(os.environ, ZR_FUSED_KERNEL="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider", *FILES],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout and " error" not in r.stdout, r.stdout[-2000:]
