"""Partition-aware ZeRO stage-1/2 gradient averaging + sharded AdamW for one GB300.

The compute lives in ``libzr.so`` (hand-written sm_103a CUDA behind a C ABI,
declared in ``include/zr.h``); ``zero_partition_aware_gb300.zr`` is the thin
ctypes binding with the same names. Importing the binding loads the library and
raises if it has not been built: there is no CPU fallback.
"""
import importlib

__all__ = ["zr", "workloads"]


def __getattr__(name):
    if name in ("zr", "workloads"):
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
