"""Grouped reduce-scatter and all-reduce over a contiguous gradient buffer, and
the fused step on buckets of many runs (GPU), against the oracle.

zr_reduce_scatter_avg_range and zr_allreduce_avg_range read every rank's
buckets back to back from one buffer ("DeepSpeed ZeRO 通信优化深度解析" §五
contiguous_gradients; "Megatron-LM 分布式训练（四）" §"梯度缓冲区+分桶+overlap"),
consecutive buckets sharing launches. Here each rank's buffer is the oracle's
packing of every bucket, concatenated in bucket order; the results must equal
the oracle's per-bucket reduce-scatter and all-reduce bit for bit, and a range
must write nothing outside its buckets. zr_rs_adam_fused on buckets filled in
backward order has one run per param: hundreds of runs per bucket, and their
edge tiles go to the kernel's end phase.
"""
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


def _bits(t):
    t = t.detach().cpu().contiguous()
    return t.view(torch.int16).numpy().view(np.uint16) if t.element_size() == 2 else \
        t.view(torch.int32).numpy().view(np.uint32)


def _dev(a: np.ndarray, phase: int, keep: list):
    dt = {np.dtype(np.uint16): torch.bfloat16, np.dtype(np.float16): torch.float16}.get(a.dtype, torch.float32)
    base = torch.zeros(a.size + phase + 8, dtype=dt, device="cuda")
    v = base[phase:phase + a.size]
    src = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if a.dtype == np.uint16 else torch.from_numpy(a)
    v.copy_(src.cuda())
    keep.append(base)
    return v


CASES = {
    # name: (world, n params, max numel, bucket, arrival)
    "flat16": (16, 300, 50_000, 400_000, None),
    "reverse8": (8, 400, 20_000, 300_000, "reverse"),
    "random32": (32, 200, 30_000, 250_000, "random"),
    "world40": (40, 80, 5000, 60_000, None),         # above the copy pipeline's 32: per-bucket register kernel
    "one_per_bucket": (4, 60, 3000, 1, None),        # every param its own bucket: many buckets per launch
    "world3": (3, 120, 20_000, 150_000, None),        # the register kernels' side of the routing
    "world5": (5, 120, 20_000, 150_000, "reverse"),   # the pipeline's side, with a one-replica last unit
}


def _setup(name, dtype):
    world, n, hi, B, arrival = CASES[name]
    rng = np.random.default_rng(sum(map(ord, name)) + (7 if dtype == "fp32" else 0))
    numel = W.random_numels(rng, n, 1, hi)
    order = None
    if arrival == "reverse":
        order = list(range(n - 1, -1, -1))
    elif arrival == "random":
        order = [int(x) for x in rng.permutation(n)]
    lay = oracle.layout(numel, world, B, order=order)
    raw = [[(rng.standard_normal(k) * 1e-2).astype(np.float32) for k in numel] for _ in range(world)]
    if dtype == "bf16":
        grads = [[oracle.f32_to_bf16(x) for x in row] for row in raw]
    elif dtype == "fp16":  # numpy's conversion rounds to nearest even
        grads = [[x.astype(np.float16) for x in row] for row in raw]
    else:
        grads = raw
    packs = [oracle.bucket_pack(lay, b, grads) for b in range(lay.n_buckets)]
    bufs = [np.concatenate([packs[b][k] for b in range(lay.n_buckets)]) for k in range(world)]
    return rng, numel, order, lay, packs, bufs


@pytest.mark.parametrize("dtype", ["bf16", "fp32", "fp16"])
@pytest.mark.parametrize("name", list(CASES))
def test_grouped_reduce_scatter_and_allreduce_equal_the_oracle(zr, name, dtype):
    rng, numel, order, lay, packs, bufs = _setup(name, dtype)
    world, nb = lay.world, lay.n_buckets
    zl = zr.Layout(numel, world, CASES[name][3], arrival=order)
    keep = []
    x = [_dev(a, int(rng.integers(0, 8)), keep) for a in bufs]
    scale = float(np.float32(1.0 / world))
    starts = np.concatenate([[0], np.cumsum([lay.bucket(b)[1] for b in range(nb)])]).astype(np.int64)
    lo, hi = (0, nb) if nb < 3 else (1, nb - 1)
    for first, count in ((0, nb), (lo, hi - lo)):
        # the reduce-scatter into NaN-filled partitions
        g = [_dev(np.full(lay.S, np.nan, np.float32), int(rng.integers(0, 4)), keep) for _ in range(world)]
        zr.zr_reduce_scatter_avg_range(zl, first, count, x, scale, g)
        g_ref = [np.full(lay.S, np.nan, np.float32) for _ in range(world)]
        for b in range(first, first + count):
            oracle.reduce_scatter_avg(lay, b, packs[b], scale, g_ref)
        # the all-reduce with a post-scale, into NaN-filled outputs of the buffers' layout:
        # at random phases for the whole range, at one shared phase for the inner one
        post = 2.0
        shared = int(rng.integers(0, 4))
        out = [_dev(np.full(int(starts[-1]), np.nan, np.float32), int(rng.integers(0, 4)) if first == 0 else shared, keep)
               for _ in range(world)]
        zr.zr_allreduce_avg_range(zl, first, count, x, scale, out, postscale=post)
        torch.cuda.synchronize()
        for r in range(world):
            assert np.array_equal(_bits(g[r]), g_ref[r].view(np.uint32)), ("rs", first, count, r)
        want = np.full(int(starts[-1]), np.nan, np.float32)
        for b in range(first, first + count):
            want[starts[b]:starts[b + 1]] = oracle.allreduce_avg(world, packs[b], scale, post)[0]
        for k in range(world):
            assert np.array_equal(_bits(out[k]), want.view(np.uint32)), ("ar", first, count, k)


def test_grouped_calls_share_launches(zr):
    """One-param buckets (world 4, the register kernels' range): the grouped calls
    take far fewer launches than buckets."""
    rng, numel, order, lay, packs, bufs = _setup("one_per_bucket", "bf16")
    zl = zr.Layout(numel, lay.world, 1)
    keep = []
    x = [_dev(a, 0, keep) for a in bufs]
    g = [torch.zeros(lay.S, device="cuda") for _ in range(lay.world)]
    n0 = zr.zr_launch_count()
    zr.zr_reduce_scatter_avg_range(zl, 0, lay.n_buckets, x, 0.25, g)
    n1 = zr.zr_launch_count()
    out = [torch.zeros(bufs[0].size, device="cuda") for _ in range(lay.world)]
    zr.zr_allreduce_avg_range(zl, 0, lay.n_buckets, x, 0.25, out)
    n2 = zr.zr_launch_count()
    torch.cuda.synchronize()
    assert lay.n_buckets == 60 and n1 - n0 <= 2 and n2 - n1 <= 2
    with pytest.raises(zr.ZrError):
        zr.zr_reduce_scatter_avg_range(zl, 59, 2, x, 0.25, g)
    with pytest.raises(zr.ZrError):
        zr.zr_allreduce_avg_range(zl, 0, 1, x, 0.25, out, postscale=float("inf"))


@pytest.mark.parametrize("world,n,hi,dt", [(4, 2000, 300, "bf16"), (16, 900, 3000, "bf16"), (8, 700, 1000, "fp32")])
def test_fused_on_buckets_of_many_runs(zr, world, n, hi, dt):
    """Backward arrival into one large bucket: every param is its own run, more
    runs than one launch carries (256) and most tiles at a run's edge. The
    fused step from the packed bucket == the oracle's, with the averaged
    gradient and every state element bit for bit."""
    rng = np.random.default_rng(world * 1000 + n)
    numel = W.random_numels(rng, n, 1, hi)
    order = list(range(n - 1, -1, -1))
    lay = oracle.layout(numel, world, 1 << 24, order=order)
    zl = zr.Layout(numel, world, 1 << 24, arrival=order)
    assert lay.n_buckets == 1 and len(lay.runs_of(0)) > 256
    raw = [[(rng.standard_normal(k) * 1e-2).astype(np.float32) for k in numel] for _ in range(world)]
    grads = [[oracle.f32_to_bf16(x) for x in row] for row in raw] if dt == "bf16" else raw
    pack = oracle.bucket_pack(lay, 0, grads)
    keep = []
    x = [_dev(a, int(rng.integers(0, 8)), keep) for a in pack]
    flat = lambda std: np.concatenate([(rng.standard_normal(lay.T) * std).astype(np.float32),
                                       np.zeros(lay.P - lay.T, np.float32)])
    p, m, v = ([np.ascontiguousarray(a) for a in np.split(s_, world)]
               for s_ in (flat(0.02), np.abs(flat(1e-4)), np.abs(flat(1e-4))))
    P_ = [_dev(a, int(rng.integers(0, 4)), keep) for a in p]
    M_ = [_dev(a, int(rng.integers(0, 4)), keep) for a in m]
    V_ = [_dev(a, int(rng.integers(0, 4)), keep) for a in v]
    G_ = [_dev(np.full(lay.S, np.nan, np.float32), int(rng.integers(0, 4)), keep) for _ in range(world)]
    param = torch.full((lay.P,), float("nan"), dtype=torch.bfloat16, device="cuda")
    hp = W.AdamW(step=5)
    scale = float(np.float32(1.0 / world))
    n0 = zr.zr_launch_count()
    zr.zr_rs_adam_fused(zl, 0, x, scale, P_, M_, V_, hp, param, G_)
    torch.cuda.synchronize()
    assert zr.zr_launch_count() - n0 >= 2
    rparam = np.zeros(lay.P, np.uint16)
    g_ref = [np.full(lay.S, np.nan, np.float32) for _ in range(world)]
    oracle.rs_adam_fused(lay, 0, pack, scale, p, m, v, hp, rparam, g_ref)
    assert np.array_equal(_bits(param), rparam)
    for r in range(world):
        for a, b_ in ((P_[r], p[r]), (M_[r], m[r]), (V_[r], v[r]), (G_[r], g_ref[r])):
            assert np.array_equal(_bits(a), b_.view(np.uint32)), r


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("name", ["flat16", "reverse8", "world3", "world5", "world40", "one_per_bucket"])
def test_grouped_fused_step_equals_the_oracle(zr, name, dtype):
    """zr_rs_adam_fused_range over a contiguous buffer per rank, on the whole
    range and on an inner one, equals the oracle's fused step per bucket:
    master, m, v, the averaged gradient and the bf16 params, bit for bit, and
    nothing outside the range's partition slices changes."""
    rng, numel, order, lay, packs, bufs = _setup(name, dtype)
    world, nb = lay.world, lay.n_buckets
    zl = zr.Layout(numel, world, CASES[name][3], arrival=order)
    keep = []
    x = [_dev(a, int(rng.integers(0, 8)), keep) for a in bufs]
    scale = float(np.float32(1.0 / world))
    hp = W.AdamW(step=3)
    lo, hi = (0, nb) if nb < 3 else (1, nb - 1)
    for first, count in ((0, nb), (lo, hi - lo)):
        flat = lambda std: np.concatenate([(rng.standard_normal(lay.T) * std).astype(np.float32),
                                           np.zeros(lay.P - lay.T, np.float32)])
        p, m, v = ([np.ascontiguousarray(a) for a in np.split(s_, world)]
                   for s_ in (flat(0.02), np.abs(flat(1e-4)), np.abs(flat(1e-4))))
        P_ = [_dev(a, int(rng.integers(0, 4)), keep) for a in p]
        M_ = [_dev(a, int(rng.integers(0, 4)), keep) for a in m]
        V_ = [_dev(a, int(rng.integers(0, 4)), keep) for a in v]
        G_ = [_dev(np.full(lay.S, np.nan, np.float32), int(rng.integers(0, 4)), keep) for _ in range(world)]
        param = torch.full((lay.P,), -1, dtype=torch.int16, device="cuda").view(torch.bfloat16)
        zr.zr_rs_adam_fused_range(zl, first, count, x, scale, P_, M_, V_, hp, param, G_)
        torch.cuda.synchronize()
        rparam = np.full(lay.P, 0xFFFF, np.uint16)
        g_ref = [np.full(lay.S, np.nan, np.float32) for _ in range(world)]
        for b in range(first, first + count):
            oracle.rs_adam_fused(lay, b, packs[b], scale, p, m, v, hp, rparam, g_ref)
        assert np.array_equal(_bits(param), rparam), ("params", first, count)
        for r in range(world):
            for a, b_ in ((P_[r], p[r]), (M_[r], m[r]), (V_[r], v[r]), (G_[r], g_ref[r])):
                assert np.array_equal(_bits(a), b_.view(np.uint32)), (first, count, r)
