"""The parity tests on the bounds-checked build (GPU).

libzr_checked.so is the same library compiled with ZR_CHECKED: before every
vector access, each kernel checks the range its launch's plan gave it (a tile
inside its run, a replica's tile inside its param's gradient, a packing
super-tile inside its segment, a listed element's param inside the bucket),
counts a failure on the device and skips the access. The parity tests are run
against it in a child process (ZR_LIB), and must pass with no failed check:
the planning keeps every kernel inside its buffers on these layouts, and the
checks themselves change no result.
"""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

FILES = ["tests/test_gpu_parity.py", "tests/test_gpu_range.py", "tests/test_gpu_grouped.py",
         "tests/test_gpu_order.py", "tests/test_gpu_scaling.py", "tests/test_gpu_microstep.py",
         "tests/test_gpu_gradcheck.py", "tests/test_gpu_e2e.py"]


def test_parity_tests_pass_on_the_bounds_checked_build():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from zero_partition_aware_gb300 import build
    build.build()
    env = dict(os.environ, ZR_LIB=build.LIB_CHECKED, ZR_CHECKED_RUN="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider", *FILES],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout and " error" not in r.stdout, r.stdout[-2000:]
