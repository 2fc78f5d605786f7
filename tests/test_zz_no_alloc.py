"""zr_bucket_pack_noalloc against the oracle's packing and zr_bucket_pack (GPU).

The allocation-free entry point serves callers that cannot call cudaMalloc --
for instance a framework that hands out all device memory from its own pool
under a fixed budget. It keeps the bucket's segment table in a fixed table
inside the library instead of allocating one, so consecutive calls reuse the
same table: this test makes two calls in a row on different buckets with
different segment counts (a stale entry would show), the second through the
Python binding, and compares each result bit for bit (packing copies bits)
with the oracle's packing of the same gradients ("DeepSpeed ZeRO 通信优化深度
解析" §四: each param's gradient copied into the contiguous IPG bucket) and
with the ordinary entry point's. It also checks that a bucket too big for the
table is refused. The file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
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


def _host(t):
    """Raw bits of a device tensor: uint16 for 16-bit elements, uint32 for fp32."""
    t = t.detach().cpu().contiguous()
    return t.view(torch.int16).numpy().view(np.uint16) if t.element_size() == 2 else \
        t.view(torch.int32).numpy().view(np.uint32)


def _ptrs(addrs):
    return (ctypes.c_void_p * len(addrs))(*addrs)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("scattered", [True, False])
def test_noalloc_pack_equals_the_oracle_on_two_calls(zr, scattered, dtype):
    rng = np.random.default_rng((11 if scattered else 12) + (0 if dtype == "bf16" else 100))
    world = 8
    numel = W.random_numels(rng, 60, 1, 40_000)
    B = 60_000
    lay = zr.Layout(numel, world, B)
    olay = oracle.layout(numel, world, B)
    assert lay.n_buckets >= 2
    tdt, code, es = (torch.bfloat16, zr.ZR_BF16, 2) if dtype == "bf16" else (torch.float32, zr.ZR_FP32, 4)
    # gradients: each param its own tensor at a random element phase, or one flat tensor per rank
    keep, grads, host = [], [], []
    for k in range(world):
        row = []
        if scattered:
            for n in numel:
                base = torch.randn(n + 8, device="cuda").to(tdt)
                ph = int(rng.integers(0, 8))
                keep.append(base)
                grads.append(base[ph:ph + n].data_ptr())
                row.append(_host(base[ph:ph + n]))
        else:
            flat = torch.randn(sum(numel), device="cuda").to(tdt)
            keep.append(flat)
            off = 0
            for n in numel:
                grads.append(flat[off:off + n].data_ptr())
                row.append(_host(flat[off:off + n]))
                off += n
        host.append([np.ascontiguousarray(a) for a in row] if dtype == "bf16" else
                    [np.ascontiguousarray(a).view(np.float32) for a in row])
    g = _ptrs(grads)
    big = max(lay.bucket(b)[1] for b in range(lay.n_buckets))
    stream = torch.cuda.current_stream().cuda_stream
    # two calls in a row on buckets of different segment counts: the one holding
    # the most params, then the one holding the fewest (or the padding bucket)
    params_in = np.bincount([lay.param(i)[1] for i in range(len(numel))], minlength=lay.n_buckets)
    b1 = int(np.argmax(params_in))
    b2 = int(np.argmin(params_in)) if params_in.min() != params_in.max() else lay.n_buckets - 1
    assert b1 != b2 and params_in[b1] != params_in[b2]
    fill = -1 if es == 2 else 0x7FC0DEAD
    ftype = torch.int16 if es == 2 else torch.int32
    for call, b in enumerate((b1, b2)):
        nb = lay.bucket(b)[1]
        ref = [torch.full((big + 16,), fill, dtype=ftype, device="cuda").view(tdt) for _ in range(world)]
        new = [torch.full((big + 16,), fill, dtype=ftype, device="cuda").view(tdt) for _ in range(world)]
        rc = zr._lib.zr_bucket_pack(lay.handle, b, g, code, _ptrs([t.data_ptr() + es for t in ref]), stream)
        assert rc == zr.ZR_OK, zr.last_error()
        outs = [t[1:1 + nb] for t in new]
        if call == 0:  # through the C ABI
            rc = zr._lib.zr_bucket_pack_noalloc(lay.handle, b, g, code, _ptrs([t.data_ptr() for t in outs]), stream)
            assert rc == zr.ZR_OK, zr.last_error()
        else:          # through the Python binding
            zr.zr_bucket_pack_noalloc(lay, b, zr.PtrArray(grads), outs, dtype=code)
        torch.cuda.synchronize()
        want = oracle.bucket_pack(olay, b, host)
        for k in range(world):
            a, c = _host(ref[k]), _host(new[k])
            got = c[1:1 + nb]
            assert np.array_equal(got, want[k].view(got.dtype)), (b, k, "against the oracle")
            assert np.array_equal(a[1:1 + nb], got), (b, k, "against zr_bucket_pack")
            canary = np.array(fill, dtype=np.int64).astype(c.dtype)
            assert c[0] == canary and np.all(c[1 + nb:] == canary), "wrote outside the bucket"


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
