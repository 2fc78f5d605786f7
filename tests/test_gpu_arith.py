"""The AdamW kernels' square root and divisions round as IEEE-754 does (GPU).

The kernels compute sqrt(v') and the two quotients of the AdamW update from
the hardware's approximate reciprocal (square root) and exact fma residuals
(Markstein's method), falling back to the IEEE operations outside the ranges
where that is exact. zr_arith_check runs the comparison on the device
against CUDA's sqrt.rn / rcp.rn / div.rn: every float for the square root,
every divisor of the range for the reciprocal, random and near-exact pairs
for the quotient, and random AdamW elements under several hyperparameter
sets. Any mismatch would break the bit-exact parity with the oracle, whose
arithmetic is IEEE float.
"""
import pytest
import torch

from zero_partition_aware_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def zr():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from zero_partition_aware_gb300 import build
    build.build()
    from zero_partition_aware_gb300 import zr as mod
    return mod


def test_sqrt_every_float(zr):
    n, bad = zr.zr_arith_check(0, 0, 1 << 32)
    assert n == 0, [hex(b) for b in bad]


def test_reciprocal_every_divisor_in_range(zr):
    n, bad = zr.zr_arith_check(1, 0, 1 << 32)
    assert n == 0, [hex(b) for b in bad]


@pytest.mark.parametrize("begin", [0, 1 << 40])
def test_quotients_random_and_near_exact(zr, begin):
    n, bad = zr.zr_arith_check(2, begin, 1 << 28)
    assert n == 0, bad


@pytest.mark.parametrize("hp", [
    W.AdamW(step=1),
    W.AdamW(step=10),
    W.AdamW(lr=3e-4, beta1=0.95, beta2=0.98, eps=1e-6, weight_decay=0.1, step=1000),
    W.AdamW(lr=1.0, beta1=0.0, beta2=0.0, eps=1e-30, weight_decay=0.0, step=1),
    W.AdamW(lr=1e-3, beta1=0.9, beta2=0.9999, eps=1e-12, weight_decay=0.01, step=3),
])
def test_adamw_elements(zr, hp):
    n, bad = zr.zr_arith_check(3, 7, 1 << 26, hp)
    assert n == 0, bad
