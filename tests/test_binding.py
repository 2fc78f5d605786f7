"""The ctypes binding hands libzr the pointer tables it was given (CPU only).

Each entry point is called against a fake library that reads every host
pointer table at call time, after the binding has had the chance to free
temporaries; the tables must still hold the caller's device addresses, each
argument its own.
"""
import ctypes
import gc

import numpy as np
import pytest


class FakeTensor:
    def __init__(self, addr, dtype="float32"):
        import torch
        self._addr = addr
        self.is_cuda = True
        self.dtype = {"float32": torch.float32, "bfloat16": torch.bfloat16}[dtype]

    def data_ptr(self):
        return self._addr

    def is_contiguous(self):
        return True

    def numel(self):
        return 10


def _table(addr, n):
    gc.collect()
    junk = [np.full(n, 0xDEAD, dtype=np.uint64) for _ in range(8)]  # reuse any freed buffer
    out = list(ctypes.cast(ctypes.c_void_p(addr), ctypes.POINTER(ctypes.c_uint64))[:n])
    del junk
    return out


class FakeLib:
    def __init__(self, world):
        self.world = world
        self.calls = {}

    def _rec(self, name, **tables):
        self.calls[name] = {k: _table(v, n) for k, (v, n) in tables.items()}
        return 0

    def zr_reduce_scatter_avg(self, h, b, x, d, s, g, st):
        return self._rec("rs", x=(x, self.world), g=(g, self.world))

    def zr_rs_adam_fused(self, h, b, x, d, s, p, m, v, hp, param, go, st):
        return self._rec("fused", x=(x, self.world), p=(p, self.world), m=(m, self.world), v=(v, self.world),
                         go=(go, self.world))

    def zr_adam_shard_step(self, h, r, p, m, v, g, hp, st):
        return self._rec("adam", p=(p, self.world), m=(m, self.world), v=(v, self.world), g=(g, self.world))

    def zr_gather_cast_bf16(self, h, p, param, st):
        return self._rec("cast", p=(p, self.world))

    def zr_allreduce_avg(self, h, b, x, d, s, post, out, st):
        return self._rec("ar", x=(x, self.world), out=(out, self.world))

    def zr_bucket_pack(self, h, b, grads, d, out, st):
        return self._rec("pack", grads=(grads, self.world * 2), out=(out, self.world))


def test_pointer_tables_survive_until_the_call(monkeypatch):
    from zero_partition_aware_gb300 import build
    build.build()
    from zero_partition_aware_gb300 import zr
    world = 4
    lay = zr.Layout([7, 9], world, 100)
    fake = FakeLib(world)
    monkeypatch.setattr(zr, "_lib", fake)
    base = {name: [0x10000 * (i + 1) + 0x1000000 * j for i in range(world)]
            for j, name in enumerate(["x", "p", "m", "v", "g", "out"])}
    T = {k: [FakeTensor(a, "bfloat16" if k == "x" else "float32") for a in v] for k, v in base.items()}
    hp = zr.zr_adamw(1e-3, 0.9, 0.999, 1e-8, 0.01, 1)
    s = 1

    zr.zr_rs_adam_fused(lay, 0, T["x"], 0.25, T["p"], T["m"], T["v"], hp, None, T["g"], stream=s)
    c = fake.calls["fused"]
    assert c["x"] == base["x"] and c["p"] == base["p"] and c["m"] == base["m"] and c["v"] == base["v"]
    assert c["go"] == base["g"]
    zr.zr_reduce_scatter_avg(lay, 0, T["x"], 0.25, T["g"], stream=s)
    assert fake.calls["rs"] == {"x": base["x"], "g": base["g"]}
    zr.zr_adam_shard_step(lay, -1, T["p"], T["m"], T["v"], T["g"], hp, stream=s)
    assert fake.calls["adam"] == {"p": base["p"], "m": base["m"], "v": base["v"], "g": base["g"]}
    zr.zr_gather_cast_bf16(lay, T["p"], 0x5000, stream=s)
    assert fake.calls["cast"] == {"p": base["p"]}
    zr.zr_allreduce_avg(lay, 0, T["x"], 0.25, T["out"], stream=s)
    assert fake.calls["ar"] == {"x": base["x"], "out": base["out"]}
    grads = [[FakeTensor(0x7000000 + 0x100 * (2 * k + i), "bfloat16") for i in range(2)] for k in range(world)]
    zr.zr_bucket_pack(lay, 0, grads, T["x"], stream=s)
    assert fake.calls["pack"]["grads"] == [0x7000000 + 0x100 * j for j in range(2 * world)]
    assert fake.calls["pack"]["out"] == base["x"]


def test_pointer_array_from_a_generator_keeps_every_tensor():
    """A PtrArray built from a generator addresses and keeps the same objects:
    tensors made inside the generator stay alive as long as the array."""
    import weakref
    from zero_partition_aware_gb300 import build
    build.build()
    from zero_partition_aware_gb300 import zr
    made = []

    def gen():
        for i in range(5):
            t = FakeTensor(0x9000000 + 0x100 * i)
            made.append(weakref.ref(t))
            yield t

    arr = zr.PtrArray(gen())
    gc.collect()
    assert [int(a) for a in arr.array] == [0x9000000 + 0x100 * i for i in range(5)]
    assert all(r() is not None for r in made)
    del arr
    gc.collect()
    assert all(r() is None for r in made)


class FakeHostTensor(FakeTensor):
    def __init__(self, addr, pinned):
        super().__init__(addr)
        self.is_cuda = False
        self._pinned = pinned

    def is_pinned(self):
        return self._pinned


def test_pinned_host_tensors_pass_and_pageable_ones_are_refused():
    """Pinned host memory that the runtime has mapped into the device's address
    space passes the binding as a device tensor does; the binding asks the
    library once per 2 MB page (zr_host_mapped) and refuses an unmapped page, or
    a pageable CPU tensor, before any call. With no GPU here the library's
    answer is 'not mapped', so the mapped case is seeded in the binding's cache."""
    from zero_partition_aware_gb300 import build
    build.build()
    from zero_partition_aware_gb300 import zr
    zr._MAPPED[0x6000000 >> 21] = True
    try:
        arr = zr.PtrArray([FakeTensor(0x5000000), FakeHostTensor(0x6000000, pinned=True)])
        assert [int(a) for a in arr.array] == [0x5000000, 0x6000000]
    finally:
        zr._MAPPED.pop(0x6000000 >> 21, None)
    with pytest.raises(ValueError, match="pageable"):
        zr.PtrArray([FakeHostTensor(0x6000000, pinned=False)])
    with pytest.raises(ValueError, match="not mapped"):
        zr.PtrArray([FakeHostTensor(0x7200000, pinned=True)])
    zr._MAPPED.pop(0x7200000 >> 21, None)
