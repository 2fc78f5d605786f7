"""Every device step under a gradient arrival order other than the flat one (GPU).

Layouts built with zr_layout_create_ordered (buckets filled in backward
order, or a random order) against the oracle's ordered layout: packing, the
reduce-scatter, the all-reduce reference, the fused step and the direct step,
element by element and bit for bit. Gradients are per-parameter tensors at
random element phases; the master/m/v shards at random phases too.
"""
import numpy as np
import pytest
import torch

import oracle
from zero_partition_aware_gb300 import workloads as W

pytestmark = pytest.mark.gpu

CASES = [(4, 0, 9, 6000, 9000), (8, 1, 30, 5000, 20000), (16, 2, 60, 8000, 100_000), (3, 3, 15, 3000, 1),
         (32, 4, 25, 3000, 40_000)]


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
    return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else \
        t.view(torch.int32).numpy().view(np.uint32)


def _order(kind, rng, n):
    return list(range(n - 1, -1, -1)) if kind == "reverse" else [int(x) for x in rng.permutation(n)]


def _dev(a: np.ndarray, phase: int):
    """A device copy of a (bf16 bits or fp32) at an element phase inside a larger buffer."""
    dt = torch.bfloat16 if a.dtype == np.uint16 else torch.float32
    base = torch.zeros(a.size + phase + 8, dtype=dt, device="cuda")
    v = base[phase:phase + a.size]
    t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if a.dtype == np.uint16 else torch.from_numpy(a)
    v.copy_(t.cuda())
    return base, v


def _setup(world, seed, n, hi, B, kind):
    rng = np.random.default_rng(500 + seed)
    numel = W.random_numels(rng, n, 1, hi)
    order = _order(kind, rng, n)
    lay = oracle.layout(numel, world, B, order=order)
    grads = [[(rng.integers(-8, 9, k).astype(np.float32) * np.float32(0.25)).astype(np.float32) for k in numel]
             for _ in range(world)]
    grads = [[W.bf16_bits(torch.from_numpy(g).to(torch.bfloat16)) for g in row] for row in grads]
    return rng, numel, order, lay, grads


@pytest.mark.parametrize("world,seed,n,hi,B", CASES)
@pytest.mark.parametrize("kind", ["reverse", "random"])
def test_pack_rs_ar_under_order(zr, world, seed, n, hi, B, kind):
    rng, numel, order, lay, grads = _setup(world, seed, n, hi, B, kind)
    zl = zr.Layout(numel, world, B, arrival=order)
    keep, gdev = [], []
    for k in range(world):
        row = []
        for g in grads[k]:
            base, v = _dev(g, int(rng.integers(0, 8)))
            keep.append(base)
            row.append(v)
        gdev.append(row)
    scale = float(np.float32(1.0 / world))
    for b in range(lay.n_buckets):
        _, nb = lay.bucket(b)
        ref = oracle.bucket_pack(lay, b, grads)
        out = [torch.full((nb,), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(world)]
        zr.zr_bucket_pack(zl, b, gdev, out)
        shards = [torch.full((lay.S,), float("nan"), device="cuda") for _ in range(world)]
        zr.zr_reduce_scatter_avg(zl, b, out, scale, shards)
        ar = [torch.full((nb,), float("nan"), device="cuda") for _ in range(world)]
        zr.zr_allreduce_avg(zl, b, out, scale, ar)
        torch.cuda.synchronize()
        for k in range(world):
            assert np.array_equal(_bits(out[k]), ref[k]), (b, k)
        ref_sh = [np.full(lay.S, np.nan, np.float32) for _ in range(world)]
        oracle.reduce_scatter_avg(lay, b, ref, scale, ref_sh)
        fm = lay.flat_map(b)
        got_full = np.concatenate([_bits(s) for s in shards])
        ref_full = np.concatenate(ref_sh).view(np.uint32)
        assert np.array_equal(got_full[fm], ref_full[fm]), b
        ref_ar = oracle.allreduce_avg(world, ref, scale)[0].view(np.uint32)
        for k in range(world):
            assert np.array_equal(_bits(ar[k]), ref_ar), (b, k)


@pytest.mark.parametrize("world,seed,n,hi,B", CASES)
@pytest.mark.parametrize("kind", ["reverse", "random"])
@pytest.mark.parametrize("path", ["fused", "direct"])
def test_step_under_order(zr, world, seed, n, hi, B, kind, path):
    rng, numel, order, lay, grads = _setup(world, seed, n, hi, B, kind)
    if path == "direct" and world > 32:
        pytest.skip("the direct step takes world <= 32")
    zl = zr.Layout(numel, world, B, arrival=order)
    hp = W.AdamW(step=int(rng.integers(1, 20)))
    scale = float(np.float32(1.0 / world))
    flat = lambda std: np.concatenate([(rng.standard_normal(lay.T) * std).astype(np.float32),
                                       np.zeros(lay.P - lay.T, np.float32)])
    p_np, m_np, v_np = np.split(flat(0.02), world), np.split(np.abs(flat(1e-4)), world), \
        np.split(np.abs(flat(1e-4)), world)
    keep = []

    def dev_list(arrs):
        out = []
        for a in arrs:
            base, v = _dev(np.ascontiguousarray(a), int(rng.integers(0, 4)))
            keep.append(base)
            out.append(v)
        return out

    P_, M_, V_ = dev_list(p_np), dev_list(m_np), dev_list(v_np)
    param = torch.full((lay.P,), float("nan"), dtype=torch.bfloat16, device="cuda")
    gdev = []
    for k in range(world):
        row = []
        for g in grads[k]:
            base, v = _dev(g, int(rng.integers(0, 8)))
            keep.append(base)
            row.append(v)
        gdev.append(row)
    if path == "direct":
        plan = zr.DirectPlan(zl, gdev)
        for b in range(lay.n_buckets):
            zr.zr_step_direct(plan, b, scale, P_, M_, V_, hp, param)
    else:
        for b in range(lay.n_buckets):
            _, nb = lay.bucket(b)
            out = [torch.empty((nb,), dtype=torch.bfloat16, device="cuda") for _ in range(world)]
            zr.zr_bucket_pack(zl, b, gdev, out)
            zr.zr_rs_adam_fused(zl, b, out, scale, P_, M_, V_, hp, param)
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    rp, rm, rv = [a.copy() for a in p_np], [a.copy() for a in m_np], [a.copy() for a in v_np]
    rparam = np.zeros(lay.P, np.uint16)
    for b in range(lay.n_buckets):
        oracle.rs_adam_fused(lay, b, oracle.bucket_pack(lay, b, grads), scale, rp, rm, rv, hp, rparam)
    assert np.array_equal(_bits(param), rparam)
    for r in range(world):
        assert np.array_equal(_bits(P_[r]), rp[r].view(np.uint32)), r
        assert np.array_equal(_bits(M_[r]), rm[r].view(np.uint32)), r
        assert np.array_equal(_bits(V_[r]), rv[r].view(np.uint32)), r


@pytest.mark.parametrize("kind", ["reverse", "random", "flat"])
@pytest.mark.parametrize("world,seed,n,hi,B", [(8, 11, 40, 6000, 20000), (16, 12, 80, 9000, 100_000),
                                               (3, 13, 12, 3000, 1)])
def test_packed_buckets_reduced_in_flat_order(zr, kind, world, seed, n, hi, B):
    """DPGroup.step_packed: each bucket packed in arrival order, then reduced by
    the direct step over the bucket buffers' param slices (flat order); equal
    to the oracle's pack + fused step bit for bit."""
    from zero_partition_aware_gb300.engine import DPGroup
    rng = np.random.default_rng(900 + seed)
    numel = W.random_numels(rng, n, 1, hi)
    order = None if kind == "flat" else _order(kind, rng, n)
    lay = oracle.layout(numel, world, B, order=order)
    grads = [[W.bf16_bits(torch.from_numpy((rng.standard_normal(k) * 1e-2).astype(np.float32)).to(torch.bfloat16))
              for k in numel] for _ in range(world)]
    keep, rows = [], []
    for row in grads:
        r_ = []
        for g in row:
            base, v = _dev(g, int(rng.integers(0, 8)))
            keep.append(base)
            r_.append(v)
        rows.append(r_)
    flat = lambda std: (rng.standard_normal(lay.T) * std).astype(np.float32)
    master, m, v = flat(0.02), np.abs(flat(1e-4)), np.abs(flat(1e-4))
    hp = W.AdamW(step=3)
    grp = DPGroup(numel, world, B, arrival=order)
    grp.load_flat(*(torch.from_numpy(x).cuda() for x in (master, m, v)))
    grp.param.fill_(float("nan"))
    plan = grp.pack_plan(grp.grad_table(rows))
    grp.step_packed(plan, hp)
    torch.cuda.synchronize()
    pad = lambda x: np.concatenate([x, np.zeros(lay.P - lay.T, np.float32)])
    rp, rm, rv = ([a.copy() for a in np.split(pad(x), world)] for x in (master, m, v))
    rparam = np.zeros(lay.P, np.uint16)
    for b in range(lay.n_buckets):
        oracle.rs_adam_fused(lay, b, oracle.bucket_pack(lay, b, grads), grp.scale, rp, rm, rv, hp, rparam)
    assert np.array_equal(_bits(grp.param[: lay.P]), rparam)
    for r in range(world):
        for a, b_ in ((grp.master[r], rp[r]), (grp.m[r], rm[r]), (grp.v[r], rv[r])):
            assert np.array_equal(_bits(a), b_.view(np.uint32)), r
