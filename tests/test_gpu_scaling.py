"""fp16 gradients through every device step, and the all-reduce path's postscale (GPU).

fp16 (IEEE binary16) gradients, as in the fp16 training the pages' all-reduce
path scales for ("DeepSpeed ZeRO 通信优化深度解析" §三.2, §六): packing, the
reduce-scatter, the all-reduce with a predivide factor's post-scaling, the
fused step, the direct step and the fp32 main-grad accumulation, against the
oracle bit for bit. Values span the fp16 range including subnormals.
"""
import numpy as np
import pytest
import torch

import oracle
from zero_partition_aware_gb300 import workloads as W

pytestmark = pytest.mark.gpu

CASES = [(4, 0, 9, 6000, 9000), (8, 1, 30, 5000, 20000), (16, 2, 40, 8000, 100_000), (3, 3, 15, 3000, 1),
         (40, 4, 12, 3000, 10_000)]


@pytest.fixture(scope="module")
def zr():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from zero_partition_aware_gb300 import build
    build.build()
    from zero_partition_aware_gb300 import zr as mod
    return mod


def _bits(t):
    t = t.detach().cpu().contiguous()
    return t.view(torch.int16).numpy().view(np.uint16) if t.element_size() == 2 else \
        t.view(torch.int32).numpy().view(np.uint32)


def _dev(a: np.ndarray, phase: int):
    dt = {np.dtype(np.float16): torch.float16, np.dtype(np.uint16): torch.bfloat16,
          np.dtype(np.float32): torch.float32}[a.dtype]
    base = torch.zeros(a.size + phase + 8, dtype=dt, device="cuda")
    v = base[phase:phase + a.size]
    src = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if a.dtype == np.uint16 else torch.from_numpy(a)
    v.copy_(src.cuda())
    return base, v


def _f16(rng, n):
    """fp16 values over the format's range: mostly normal gradients, some subnormal and large."""
    x = rng.standard_normal(n) * 1e-2
    x[rng.random(n) < 0.05] *= 1e-5          # subnormal territory (fp16 normals start at 6.1e-5)
    x[rng.random(n) < 0.02] *= 1e4
    return x.astype(np.float16)


def _grads(rng, numel, world, keep):
    host = [[_f16(rng, k) for k in numel] for _ in range(world)]
    dev = []
    for k in range(world):
        row = []
        for g in host[k]:
            base, v = _dev(g, int(rng.integers(0, 8)))
            keep.append(base)
            row.append(v)
        dev.append(row)
    return host, dev


@pytest.mark.parametrize("world,seed,n,hi,B", CASES)
def test_fp16_pack_rs_ar(zr, world, seed, n, hi, B):
    rng = np.random.default_rng(700 + seed)
    numel = W.random_numels(rng, n, 1, hi)
    lay = oracle.layout(numel, world, B)
    zl = zr.Layout(numel, world, B)
    keep = []
    host, dev = _grads(rng, numel, world, keep)
    scale = float(np.float32(1.0 / world))
    f = [1, 2, world][seed % 3]
    pre, post = float(np.float32(1.0 / f)), float(np.float32(f / world))
    for b in range(lay.n_buckets):
        _, nb = lay.bucket(b)
        ref = oracle.bucket_pack(lay, b, host)
        out = [torch.full((nb,), float("nan"), dtype=torch.float16, device="cuda") for _ in range(world)]
        zr.zr_bucket_pack(zl, b, dev, out)
        shards = [torch.full((lay.S,), float("nan"), device="cuda") for _ in range(world)]
        zr.zr_reduce_scatter_avg(zl, b, out, scale, shards)
        ar = [torch.full((nb,), float("nan"), device="cuda") for _ in range(world)]
        zr.zr_allreduce_avg(zl, b, out, pre, ar, postscale=post)
        torch.cuda.synchronize()
        for k in range(world):
            assert np.array_equal(_bits(out[k]), ref[k].view(np.uint16)), (b, k)
        ref_sh = [np.full(lay.S, np.nan, np.float32) for _ in range(world)]
        oracle.reduce_scatter_avg(lay, b, ref, scale, ref_sh)
        s, _ = lay.bucket(b)
        got = np.concatenate([_bits(t) for t in shards])[s:s + nb]
        assert np.array_equal(got, np.concatenate(ref_sh).view(np.uint32)[s:s + nb]), b
        ref_ar = oracle.allreduce_avg(world, ref, pre, post)[0].view(np.uint32)
        for k in range(world):
            assert np.array_equal(_bits(ar[k]), ref_ar), (b, k)


@pytest.mark.parametrize("world,seed,n,hi,B", CASES)
@pytest.mark.parametrize("path", ["fused", "direct"])
def test_fp16_step(zr, world, seed, n, hi, B, path):
    if path == "direct" and world > 32:
        pytest.skip("the direct step takes world <= 32")
    rng = np.random.default_rng(800 + seed)
    numel = W.random_numels(rng, n, 1, hi)
    lay = oracle.layout(numel, world, B)
    zl = zr.Layout(numel, world, B)
    keep = []
    host, dev = _grads(rng, numel, world, keep)
    hp = W.AdamW(step=int(rng.integers(1, 20)))
    scale = float(np.float32(1.0 / world))
    flat = lambda std: np.concatenate([(rng.standard_normal(lay.T) * std).astype(np.float32),
                                       np.zeros(lay.P - lay.T, np.float32)])
    p_np, m_np, v_np = np.split(flat(0.02), world), np.split(np.abs(flat(1e-4)), world), \
        np.split(np.abs(flat(1e-4)), world)

    def dev_list(arrs):
        out = []
        for a in arrs:
            base, v = _dev(np.ascontiguousarray(a), int(rng.integers(0, 4)))
            keep.append(base)
            out.append(v)
        return out

    P_, M_, V_ = dev_list(p_np), dev_list(m_np), dev_list(v_np)
    param = torch.full((lay.P,), float("nan"), dtype=torch.bfloat16, device="cuda")
    if path == "direct":
        plan = zr.DirectPlan(zl, dev)
        for b in range(lay.n_buckets):
            zr.zr_step_direct(plan, b, scale, P_, M_, V_, hp, param)
    else:
        for b in range(lay.n_buckets):
            _, nb = lay.bucket(b)
            out = [torch.empty((nb,), dtype=torch.float16, device="cuda") for _ in range(world)]
            zr.zr_bucket_pack(zl, b, dev, out)
            zr.zr_rs_adam_fused(zl, b, out, scale, P_, M_, V_, hp, param)
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    rp, rm, rv = [a.copy() for a in p_np], [a.copy() for a in m_np], [a.copy() for a in v_np]
    rparam = np.zeros(lay.P, np.uint16)
    for b in range(lay.n_buckets):
        oracle.rs_adam_fused(lay, b, oracle.bucket_pack(lay, b, host), scale, rp, rm, rv, hp, rparam)
    assert np.array_equal(_bits(param), rparam)
    for r in range(world):
        assert np.array_equal(_bits(P_[r]), rp[r].view(np.uint32)), r
        assert np.array_equal(_bits(M_[r]), rm[r].view(np.uint32)), r
        assert np.array_equal(_bits(V_[r]), rv[r].view(np.uint32)), r


@pytest.mark.parametrize("n", [1, 255, 4097, 100_003])
def test_fp16_grad_accumulate(zr, n):
    rng = np.random.default_rng(n)
    main = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    g = _f16(rng, n)
    keep = []
    mb, md = _dev(main.copy(), int(rng.integers(0, 4)))
    gb, gd = _dev(g, int(rng.integers(0, 8)))
    zr.zr_grad_accumulate(md, gd)
    torch.cuda.synchronize()
    ref = main.copy()
    oracle.grad_accumulate(ref, g)
    assert np.array_equal(_bits(md), ref.view(np.uint32))


@pytest.mark.parametrize("dt", ["bf16", "fp32"])
@pytest.mark.parametrize("world,f", [(8, 2), (16, 4), (6, 3)])
def test_allreduce_postscale(zr, dt, world, f):
    rng = np.random.default_rng(world + f)
    numel = W.random_numels(rng, 20, 1, 4000)
    lay = oracle.layout(numel, world, 8000)
    zl = zr.Layout(numel, world, 8000)
    pre, post = float(np.float32(1.0 / f)), float(np.float32(f / world))
    for b in range(lay.n_buckets):
        _, nb = lay.bucket(b)
        x = [(rng.standard_normal(nb) * 1e-2).astype(np.float32) for _ in range(world)]
        if dt == "bf16":
            x = [oracle.f32_to_bf16(a) for a in x]
        keep, xd = [], []
        for a in x:
            base, v = _dev(a, int(rng.integers(0, 4)))
            keep.append(base)
            xd.append(v)
        ar = [torch.full((nb,), float("nan"), device="cuda") for _ in range(world)]
        zr.zr_allreduce_avg(zl, b, xd, pre, ar, postscale=post)
        torch.cuda.synchronize()
        ref = oracle.allreduce_avg(world, x, pre, post)[0].view(np.uint32)
        for k in range(world):
            assert np.array_equal(_bits(ar[k]), ref)
