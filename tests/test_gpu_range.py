"""The direct step over a range of buckets in shared launches (GPU).

zr_step_direct_range groups consecutive buckets into one launch while the
launch's argument block holds their runs (256), bucket tables (16) and listed
boundary tiles (1,024). The cases below force each of those splits, and the
overflow of listed tiles into the per-tile kernel; the results must equal the
oracle's per-bucket step bit for bit. zr_rs_direct_norm_range must give the
oracle's averages bit for bit and its sums within the check's bound (exactly,
on integer gradients).
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
    dt = torch.bfloat16 if a.dtype == np.uint16 else torch.float32
    base = torch.zeros(a.size + phase + 8, dtype=dt, device="cuda")
    v = base[phase:phase + a.size]
    src = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if a.dtype == np.uint16 else torch.from_numpy(a)
    v.copy_(src.cuda())
    keep.append(base)
    return v


CASES = {
    # name: (world, n params, max numel, bucket, arrival)
    "many_runs": (16, 700, 3000, 150_000, "reverse"),
    "many_buckets": (8, 40, 5000, 1, "flat"),
    "many_boundaries": (2, 6000, 300, 1 << 22, "flat"),   # two runs of ~615 listed tiles: split between them
    "overflow_tiles": (1, 6000, 300, 1 << 22, "flat"),    # one run of ~1,229: the rest to the per-tile kernel
    "mixed": (32, 300, 20_000, 200_000, "random"),
}


def _setup(name, integer=False):
    world, n, hi, B, arrival = CASES[name]
    rng = np.random.default_rng(sum(map(ord, name)))
    numel = W.random_numels(rng, n, 1, hi)
    order = None
    if arrival == "reverse":
        order = list(range(n - 1, -1, -1))
    elif arrival == "random":
        order = [int(x) for x in rng.permutation(n)]
    lay = oracle.layout(numel, world, B, order=order)
    if integer:
        raw = [[rng.integers(-8, 9, k).astype(np.float32) for k in numel] for _ in range(world)]
    else:
        raw = [[(rng.standard_normal(k) * 1e-2).astype(np.float32) for k in numel] for _ in range(world)]
    grads = [[oracle.f32_to_bf16(x) for x in row] for row in raw]
    return rng, numel, order, lay, grads


@pytest.mark.parametrize("name", list(CASES))
def test_range_step_equals_oracle(zr, name):
    rng, numel, order, lay, grads = _setup(name)
    world = lay.world
    zl = zr.Layout(numel, world, CASES[name][3], arrival=order)
    keep = []
    rows = [[_dev(g, int(rng.integers(0, 8)), keep) for g in row] for row in grads]
    plan = zr.DirectPlan(zl, rows)
    flat = lambda std: np.concatenate([(rng.standard_normal(lay.T) * std).astype(np.float32),
                                       np.zeros(lay.P - lay.T, np.float32)])
    p, m, v = ([np.ascontiguousarray(a) for a in np.split(x, world)]
               for x in (flat(0.02), np.abs(flat(1e-4)), np.abs(flat(1e-4))))
    P_ = [_dev(a, int(rng.integers(0, 4)), keep) for a in p]
    M_ = [_dev(a, int(rng.integers(0, 4)), keep) for a in m]
    V_ = [_dev(a, int(rng.integers(0, 4)), keep) for a in v]
    param = torch.full((lay.P,), float("nan"), dtype=torch.bfloat16, device="cuda")
    hp = W.AdamW(step=3)
    scale = float(np.float32(1.0 / world))
    n0 = zr.zr_launch_count()
    zr.zr_step_direct_range(plan, 0, lay.n_buckets, scale, P_, M_, V_, hp, param)
    torch.cuda.synchronize()
    launches = zr.zr_launch_count() - n0
    rparam = np.zeros(lay.P, np.uint16)
    for b in range(lay.n_buckets):
        oracle.rs_adam_fused(lay, b, oracle.bucket_pack(lay, b, grads), scale, p, m, v, hp, rparam)
    assert np.array_equal(_bits(param), rparam)
    for r in range(world):
        for a, b_ in ((P_[r], p[r]), (M_[r], m[r]), (V_[r], v[r])):
            assert np.array_equal(_bits(a), b_.view(np.uint32)), r
    if name == "many_buckets":
        assert lay.n_buckets > 16 and launches < lay.n_buckets


@pytest.mark.parametrize("name", ["many_runs", "many_buckets", "many_boundaries", "overflow_tiles"])
def test_range_norm_pass_equals_oracle(zr, name):
    rng, numel, order, lay, grads = _setup(name, integer=True)
    world = lay.world
    zl = zr.Layout(numel, world, CASES[name][3], arrival=order)
    keep = []
    plan = zr.DirectPlan(zl, [[_dev(g, int(rng.integers(0, 8)), keep) for g in row] for row in grads])
    g_out = [_dev(np.full(lay.S, np.nan, np.float32), int(rng.integers(0, 4)), keep) for _ in range(world)]
    chk = zr.GradCheck()
    scale = float(np.float32(1.0 / world))
    zr.zr_rs_direct_norm_range(plan, 0, lay.n_buckets, scale, g_out, chk)
    zr.zr_grad_check_finalize(chk, 1.0)
    got = zr.zr_gradcheck_read(chk)
    g_ref = [np.full(lay.S, np.nan, np.float32) for _ in range(world)]
    for b in range(lay.n_buckets):
        oracle.reduce_scatter_avg(lay, b, oracle.bucket_pack(lay, b, grads), scale, g_ref)
    for r in range(world):
        assert np.array_equal(_bits(g_out[r]), g_ref[r].view(np.uint32)), r
    ref = oracle.grad_check(g_ref, 1.0)
    assert got["nonfinite"] == ref.nonfinite and got["skip"] == ref.skip
    assert got["sumsq"] == ref.sumsq and got["coef"] == ref.coef  # integer grads, power-of-two world: exact


def test_range_norm_pass_repeats_bit_for_bit(zr):
    """The norm pass over several launches of one call, on non-integer gradients
    (whose sum depends on the order of the adds): three passes give the same
    outcome bit for bit, as the launches add to the check's slots in launch
    order even when a launch starts before the one before it has completed."""
    rng, numel, order, lay, grads = _setup("many_buckets")
    world = lay.world
    zl = zr.Layout(numel, world, CASES["many_buckets"][3], arrival=order)
    keep = []
    plan = zr.DirectPlan(zl, [[_dev(g, int(rng.integers(0, 8)), keep) for g in row] for row in grads])
    g_out = [_dev(np.zeros(lay.S, np.float32), 0, keep) for _ in range(world)]
    chk = zr.GradCheck()
    scale = float(np.float32(1.0 / world))
    outs = []
    for _ in range(3):
        n0 = zr.zr_launch_count()
        zr.zr_rs_direct_norm_range(plan, 0, lay.n_buckets, scale, g_out, chk)
        launches = zr.zr_launch_count() - n0
        zr.zr_grad_check_finalize(chk, 1.0)
        outs.append(zr.zr_gradcheck_read(chk))
    assert launches > 2
    assert outs[0] == outs[1] == outs[2]
    g_ref = [np.zeros(lay.S, np.float32) for _ in range(world)]
    for b in range(lay.n_buckets):
        oracle.reduce_scatter_avg(lay, b, oracle.bucket_pack(lay, b, grads), scale, g_ref)
    for r in range(world):
        assert np.array_equal(_bits(g_out[r]), g_ref[r].view(np.uint32)), r
    ref = oracle.grad_check(g_ref, 1.0)
    assert abs(outs[0]["sumsq"] - ref.sumsq) <= 1e-6 * ref.sumsq


def test_range_step_completes_before_later_work(zr):
    """A large first launch and small later ones in one range call: work queued
    on the stream right after the call (device copies, no host wait between)
    must see every launch's results. A later launch of the call may start while
    the one before drains, but completes only after it."""
    world = 8
    rng = np.random.default_rng(11)
    numel = [3_000_000] + [int(x) for x in rng.integers(1, 4000, 40)]
    lay = oracle.layout(numel, world, 1)  # one bucket per param: the big one opens the first launch
    zl = zr.Layout(numel, world, 1)
    keep = []
    raw = [[(rng.standard_normal(k) * 1e-2).astype(np.float32) for k in numel] for _ in range(world)]
    grads = [[oracle.f32_to_bf16(x) for x in row] for row in raw]
    plan = zr.DirectPlan(zl, [[_dev(g, 0, keep) for g in row] for row in grads])
    flat = lambda std: np.concatenate([(rng.standard_normal(lay.T) * std).astype(np.float32),
                                       np.zeros(lay.P - lay.T, np.float32)])
    p, m, v = ([np.ascontiguousarray(a) for a in np.split(x, world)]
               for x in (flat(0.02), np.abs(flat(1e-4)), np.abs(flat(1e-4))))
    P_ = [_dev(a, 0, keep) for a in p]
    M_ = [_dev(a, 0, keep) for a in m]
    V_ = [_dev(a, 0, keep) for a in v]
    param = torch.zeros(lay.P, dtype=torch.bfloat16, device="cuda")
    hp = W.AdamW(step=4)
    scale = float(np.float32(1.0 / world))
    torch.cuda.synchronize()
    n0 = zr.zr_launch_count()
    zr.zr_step_direct_range(plan, 0, lay.n_buckets, scale, P_, M_, V_, hp, param)
    launches = zr.zr_launch_count() - n0
    copies = [t.clone() for t in [param] + P_ + M_ + V_]  # queued behind the call
    torch.cuda.synchronize()
    assert launches >= 3
    rparam = np.zeros(lay.P, np.uint16)
    for b in range(lay.n_buckets):
        oracle.rs_adam_fused(lay, b, oracle.bucket_pack(lay, b, grads), scale, p, m, v, hp, rparam)
    assert np.array_equal(_bits(copies[0]), rparam)
    for r in range(world):
        for a, b_ in ((copies[1 + r], p[r]), (copies[1 + world + r], m[r]), (copies[1 + 2 * world + r], v[r])):
            assert np.array_equal(_bits(a), b_.view(np.uint32)), r


def test_range_subsets_and_bad_ranges(zr):
    """Two half ranges equal one full range; out-of-range buckets are refused."""
    rng, numel, order, lay, grads = _setup("many_buckets")
    world = lay.world
    zl = zr.Layout(numel, world, 1)
    keep = []
    rows = [[_dev(g, 1, keep) for g in row] for row in grads]
    plan = zr.DirectPlan(zl, rows)
    hp = W.AdamW(step=2)
    states = []
    for split in (None, lay.n_buckets // 2):
        P_ = [torch.full((lay.S,), 0.01, device="cuda") for _ in range(world)]
        M_ = [torch.zeros(lay.S, device="cuda") for _ in range(world)]
        V_ = [torch.zeros(lay.S, device="cuda") for _ in range(world)]
        param = torch.zeros(lay.P, dtype=torch.bfloat16, device="cuda")
        if split is None:
            zr.zr_step_direct_range(plan, 0, lay.n_buckets, 0.125, P_, M_, V_, hp, param)
        else:
            zr.zr_step_direct_range(plan, 0, split, 0.125, P_, M_, V_, hp, param)
            zr.zr_step_direct_range(plan, split, lay.n_buckets - split, 0.125, P_, M_, V_, hp, param)
        torch.cuda.synchronize()
        states.append([_bits(t) for t in P_ + M_ + V_] + [_bits(param)])
    for a, b in zip(*states):
        assert np.array_equal(a, b)
    for first, count in ((-1, 2), (0, lay.n_buckets + 1), (3, -1)):
        with pytest.raises(zr.ZrError):
            zr.zr_step_direct_range(plan, first, count, 0.125, P_, M_, V_, hp, param)
    zr.zr_step_direct_range(plan, 2, 0, 0.125, P_, M_, V_, hp, param)  # empty range: nothing to do


@pytest.mark.parametrize("world,s_phase,q_phase", [(8, 0, 0), (8, 1, 3), (16, 2, 6), (16, 3, 5), (40, 1, 2)])
def test_flat_view_shards_anchor_on_the_params(zr, world, s_phase, q_phase):
    """Master, m and v as views of one flat buffer each (partition r at rS, the
    buffer s_phase fp32 elements past a 16-byte boundary), the bf16 params
    q_phase elements past one, S odd: tiles are anchored on the params where
    the phases agree modulo 4 elements. The direct range step (world <= 32) and
    the per-bucket fused step from packed buckets must equal the oracle bit for
    bit."""
    rng = np.random.default_rng(world * 100 + s_phase * 10 + q_phase)
    numel = W.random_numels(rng, 60, 1, 40_000)
    lay = oracle.layout(numel, world, 200_000)
    if lay.S % 2 == 0:  # an odd S puts the partitions at every phase; world more elements add one to S
        numel[-1] += world
        lay = oracle.layout(numel, world, 200_000)
    assert lay.S % 2 == 1
    zl = zr.Layout(numel, world, 200_000)
    raw = [[(rng.standard_normal(k) * 1e-2).astype(np.float32) for k in numel] for _ in range(world)]
    grads = [[oracle.f32_to_bf16(x) for x in row] for row in raw]
    keep = []
    rows = [[_dev(g, int(rng.integers(0, 8)), keep) for g in row] for row in grads]
    flat = lambda std: np.concatenate([(rng.standard_normal(lay.T) * std).astype(np.float32),
                                       np.zeros(lay.P - lay.T, np.float32)])
    state = [flat(0.02), np.abs(flat(1e-4)), np.abs(flat(1e-4))]
    hp = W.AdamW(step=4)
    scale = float(np.float32(1.0 / world))
    rp, rm, rv = ([a.copy() for a in np.split(x, world)] for x in state)
    rparam = np.zeros(lay.P, np.uint16)
    for b in range(lay.n_buckets):
        oracle.rs_adam_fused(lay, b, oracle.bucket_pack(lay, b, grads), scale, rp, rm, rv, hp, rparam)
    for packed in ((False, True) if world <= 32 else (True,)):  # the direct step takes world <= 32
        views = []
        for x in state:
            buf = _dev(x, s_phase, keep)
            views.append([buf[r * lay.S:(r + 1) * lay.S] for r in range(world)])
        P_, M_, V_ = views
        qbuf = torch.zeros(lay.P + 8, dtype=torch.bfloat16, device="cuda")
        param = qbuf[q_phase:q_phase + lay.P]
        param.fill_(float("nan"))
        if packed:
            for b in range(lay.n_buckets):
                _, nb = lay.bucket(b)
                bk = [torch.empty(nb, dtype=torch.bfloat16, device="cuda") for _ in range(world)]
                zr.zr_bucket_pack(zl, b, rows, bk)
                zr.zr_rs_adam_fused(zl, b, bk, scale, P_, M_, V_, hp, param)
        else:
            zr.zr_step_direct_range(zr.DirectPlan(zl, rows), 0, lay.n_buckets, scale, P_, M_, V_, hp, param)
        torch.cuda.synchronize()
        assert np.array_equal(_bits(param), rparam), packed
        for r in range(world):
            for a, b_ in ((P_[r], rp[r]), (M_[r], rm[r]), (V_[r], rv[r])):
                assert np.array_equal(_bits(a), b_.view(np.uint32)), (packed, r)
