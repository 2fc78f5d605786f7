"""Failure injection through the C ABI (CPU).

With ZR_FAIL_AT_LAUNCH=n set, every kernel launch the library attempts once it
has launched n - 1 kernels fails with ZR_ERR_CUDA before anything is
enqueued. On a machine without a GPU a well-formed call otherwise fails later,
with ZR_ERR_STATE (no device); here the injected status and message must come
first, reach the caller through the C ABI and the Python binding unchanged,
and stop the call. Unset, the variable changes nothing.
"""
import ctypes
import os

import pytest


@pytest.fixture(scope="module")
def zr():
    from zero_partition_aware_gb300 import build
    build.build()
    from zero_partition_aware_gb300 import zr as mod
    return mod


@pytest.fixture
def inject(monkeypatch):
    def at(n):
        monkeypatch.setenv("ZR_FAIL_AT_LAUNCH", str(n))
    yield at
    monkeypatch.delenv("ZR_FAIL_AT_LAUNCH", raising=False)


def _no_gpu():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present: this check only runs on a machine without one")


def test_injected_failure_comes_before_any_device_call(zr, inject):
    _no_gpu()
    lay = zr.Layout([100, 200], 2, 1000)
    two = (ctypes.c_void_p * 2)(0x1000, 0x2000)
    L = zr._lib
    assert L.zr_reduce_scatter_avg(lay.handle, 0, two, zr.ZR_BF16, 0.5, two, None) == zr.ZR_ERR_STATE
    inject(zr.zr_launch_count() + 1)
    assert L.zr_reduce_scatter_avg(lay.handle, 0, two, zr.ZR_BF16, 0.5, two, None) == zr.ZR_ERR_CUDA
    assert "injected failure" in zr.last_error()
    hp = zr.zr_adamw(1e-3, 0.9, 0.999, 1e-8, 0.01, 1)
    assert L.zr_rs_adam_fused(lay.handle, 0, two, zr.ZR_BF16, 0.5, two, two, two, ctypes.byref(hp), None, None,
                              None) == zr.ZR_ERR_CUDA
    assert L.zr_gather_cast_bf16(lay.handle, two, ctypes.c_void_p(0x3000), None) == zr.ZR_ERR_CUDA
    assert L.zr_grad_accumulate(ctypes.c_void_p(0x1000), ctypes.c_void_p(0x2000), zr.ZR_BF16, 10,
                                None) == zr.ZR_ERR_CUDA
    assert L.zr_reduce_scatter_avg_range(lay.handle, 0, lay.n_buckets, two, zr.ZR_BF16, 0.5, two,
                                         None) == zr.ZR_ERR_CUDA
    # argument errors are still found first
    assert L.zr_reduce_scatter_avg(lay.handle, 9, two, zr.ZR_BF16, 0.5, two, None) == zr.ZR_ERR_INVALID_ARG


def test_injected_failure_reaches_python(zr, inject):
    _no_gpu()
    lay = zr.Layout([100, 200], 2, 1000)
    inject(1)
    with pytest.raises(zr.ZrError) as e:
        zr.zr_reduce_scatter_avg(lay, 0, [0x1000, 0x2000], 0.5, [0x3000, 0x4000], dtype=zr.ZR_BF16, stream=0)
    assert e.value.status == zr.ZR_ERR_CUDA and "injected failure" in str(e.value)


def test_a_later_launch_index_or_zero_changes_nothing(zr, inject):
    _no_gpu()
    lay = zr.Layout([100, 200], 2, 1000)
    two = (ctypes.c_void_p * 2)(0x1000, 0x2000)
    for n in (zr.zr_launch_count() + 5, 0):
        inject(n)
        assert zr._lib.zr_reduce_scatter_avg(lay.handle, 0, two, zr.ZR_BF16, 0.5, two, None) == zr.ZR_ERR_STATE
    assert "ZR_FAIL_AT_LAUNCH" not in os.environ or os.environ["ZR_FAIL_AT_LAUNCH"] == "0"
