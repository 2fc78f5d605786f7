"""zr_bucket_pack_noalloc against zr_bucket_pack, through the C ABI (GPU).

The allocation-free entry point serves callers that cannot call cudaMalloc --
for instance a framework that hands out all device memory from its own pool
under a fixed budget. It keeps the bucket's segment table in a fixed table
inside the library instead of allocating one, so consecutive calls reuse the
same table: this test makes two calls in a row (different buckets, different
sizes, so a stale table would show) and compares each result with the
ordinary entry point's, bit for bit (packing copies bits). It also checks that
a bucket too big for the table is refused. The file is named so that pytest
collects it last.
"""
import ctypes

import numpy as np
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


def _bits(t):
    return t.detach().cpu().view(torch.int16).numpy()


def _ptrs(addrs):
    return (ctypes.c_void_p * len(addrs))(*addrs)


@pytest.mark.parametrize("scattered", [True, False])
def test_noalloc_pack_equals_pack_on_two_calls(zr, scattered):
    rng = np.random.default_rng(11 if scattered else 12)
    world = 8
    numel = W.random_numels(rng, 60, 1, 40_000)
    B = 150_000
    lay = zr.Layout(numel, world, B)
    assert lay.n_buckets >= 2
    # gradients: each param its own tensor at a random 2-byte phase, or one flat tensor per rank
    keep, grads = [], []
    for k in range(world):
        if scattered:
            for n in numel:
                base = torch.randn(n + 8, device="cuda").to(torch.bfloat16)
                ph = int(rng.integers(0, 8))
                keep.append(base)
                grads.append(base[ph:ph + n].data_ptr())
        else:
            flat = torch.randn(sum(numel), device="cuda").to(torch.bfloat16)
            keep.append(flat)
            off = 0
            for n in numel:
                grads.append(flat[off:off + n].data_ptr())
                off += n
    g = _ptrs(grads)
    big = max(lay.bucket(b)[1] for b in range(lay.n_buckets))
    stream = torch.cuda.current_stream().cuda_stream
    # two calls in a row: the largest bucket, then the last (padding) bucket
    order = [int(np.argmax([lay.bucket(b)[1] for b in range(lay.n_buckets)])), lay.n_buckets - 1]
    for b in order:
        nb = lay.bucket(b)[1]
        ref = [torch.full((big + 16,), -1, dtype=torch.int16, device="cuda") for _ in range(world)]
        new = [torch.full((big + 16,), -1, dtype=torch.int16, device="cuda") for _ in range(world)]
        rc = zr._lib.zr_bucket_pack(lay.handle, b, g, zr.ZR_BF16, _ptrs([t.data_ptr() + 2 for t in ref]), stream)
        assert rc == zr.ZR_OK, zr.last_error()
        rc = zr._lib.zr_bucket_pack_noalloc(lay.handle, b, g, zr.ZR_BF16, _ptrs([t.data_ptr() + 2 for t in new]),
                                            stream)
        assert rc == zr.ZR_OK, zr.last_error()
        torch.cuda.synchronize()
        for k in range(world):
            a, c = _bits(ref[k]), _bits(new[k])
            assert np.array_equal(a[1:1 + nb], c[1:1 + nb]), (b, k)
            assert c[0] == -1 and np.all(c[1 + nb:] == -1), "wrote outside the bucket"


def test_noalloc_pack_refuses_a_bucket_beyond_its_table(zr):
    world = 32
    numel = [3] * 300  # 32 replicas x 300 unmergeable params = 9600 segments > 8192
    lay = zr.Layout(numel, world, 10 ** 9)
    bases = [torch.zeros(8, dtype=torch.bfloat16, device="cuda") for _ in range(world * 300)]
    g = _ptrs([t.data_ptr() for t in bases])
    out = [torch.zeros(lay.bucket(0)[1], dtype=torch.bfloat16, device="cuda") for _ in range(world)]
    rc = zr._lib.zr_bucket_pack_noalloc(lay.handle, 0, g, zr.ZR_BF16, _ptrs([t.data_ptr() for t in out]),
                                        torch.cuda.current_stream().cuda_stream)
    assert rc == zr.ZR_ERR_UNSUPPORTED
    assert "8192" in zr.last_error()
