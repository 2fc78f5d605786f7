"""The global gradient check and the clipped step (GPU) against the oracle.

Between the DP sync of every bucket and optimizer.step() ("Megatron-LM
分布式训练（四）" §"跨 model-parallel 的梯度收尾"; "DeepSpeed ZeRO 通信优化深度解析"
§六): the averaging of every bucket into the fp32 gradient partitions with the
sums of squares (packed buckets or the direct plan), the check (norm,
overflow count, clip coefficient), then the clipped AdamW + bf16 cast.

Comparisons:
- the averaged gradients bit for bit;
- the overflow count and skip exactly;
- with integer-valued gradients every square and partial sum is exact on both
  sides, so sumsq, norm and coef must be equal bit for bit; with other values
  sumsq is within 1e-6 relative (the kernels add 8 fp32 squares in fp32) and
  coef within 2e-6 relative;
- the updated master, m, v and bf16 params bit for bit against the oracle's
  step run with the device's coefficient (the coefficient is fixed by the
  pages only up to the rounding of the norm; given it, the step is exact);
- max_norm <= 0 reproduces the one-pass direct step bit for bit, and an
  overflowed step leaves every state and the parameter buffer untouched.
"""
import numpy as np
import pytest
import torch

import oracle
from zero_partition_aware_gb300 import workloads as W

pytestmark = pytest.mark.gpu

RTOL_SUMSQ = 1e-6
RTOL_COEF = 2e-6


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
    dt = {np.dtype(np.float16): torch.float16, np.dtype(np.uint16): torch.bfloat16,
          np.dtype(np.float32): torch.float32}[a.dtype]
    base = torch.zeros(a.size + phase + 8, dtype=dt, device="cuda")
    v = base[phase:phase + a.size]
    src = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if a.dtype == np.uint16 else torch.from_numpy(a)
    v.copy_(src.cuda())
    keep.append(base)
    return v


def _grad_values(rng, n, dtype, kind):
    if kind == "int":
        x = rng.integers(-8, 9, n).astype(np.float32)
    else:
        x = (rng.standard_normal(n) * 1e-2).astype(np.float32)
    if dtype == "bf16":
        return oracle.f32_to_bf16(x)
    if dtype == "fp16":
        return x.astype(np.float16)
    return x


def _setup(world, seed, n, hi, B, dtype, kind, arrival=None):
    rng = np.random.default_rng(900 + seed)
    numel = W.random_numels(rng, n, 1, hi)
    order = None
    if arrival == "reverse":
        order = list(range(n - 1, -1, -1))
    lay = oracle.layout(numel, world, B, order=order)
    grads = [[_grad_values(rng, k, dtype, kind) for k in numel] for _ in range(world)]
    return rng, numel, order, lay, grads


def _state(rng, lay, keep):
    flat = lambda std: np.concatenate([(rng.standard_normal(lay.T) * std).astype(np.float32),
                                       np.zeros(lay.P - lay.T, np.float32)])
    p, m, v = (np.split(flat(0.02), lay.world), np.split(np.abs(flat(1e-4)), lay.world),
               np.split(np.abs(flat(1e-4)), lay.world))
    host = [[np.ascontiguousarray(a) for a in arrs] for arrs in (p, m, v)]
    dev = [[_dev(a, int(rng.integers(0, 4)), keep) for a in arrs] for arrs in host]
    return host, dev


def _check_stats(got, ref, exact):
    assert got["nonfinite"] == ref.nonfinite
    assert got["skip"] == ref.skip
    if ref.skip:
        return
    if exact:
        assert got["sumsq"] == ref.sumsq and got["norm"] == ref.norm and got["coef"] == ref.coef
    else:
        assert abs(got["sumsq"] - ref.sumsq) <= RTOL_SUMSQ * ref.sumsq
        assert abs(got["coef"] - ref.coef) <= RTOL_COEF * ref.coef


CASES = [(4, 0, 9, 6000, 9000), (8, 1, 30, 5000, 20000), (16, 2, 40, 8000, 100_000), (3, 3, 15, 3000, 1),
         (32, 4, 25, 3000, 40_000)]


def _run_case(zr, world, seed, n, hi, B, dtype, kind, path, max_norm_frac, arrival=None):
    rng, numel, order, lay, grads = _setup(world, seed, n, hi, B, dtype, kind, arrival)
    zl = zr.Layout(numel, world, B, arrival=order)
    keep = []
    scale = float(np.float32(1.0 / world))
    g_out = [_dev(np.full(lay.S, np.nan, np.float32), int(rng.integers(0, 4)), keep) for _ in range(world)]
    chk = zr.GradCheck()
    if path == "direct":
        rows = [[_dev(g, int(rng.integers(0, 8)), keep) for g in row] for row in grads]
        plan = zr.DirectPlan(zl, rows)
        for b in range(lay.n_buckets):
            zr.zr_rs_direct_norm(plan, b, scale, g_out, chk)
    else:
        for b in range(lay.n_buckets):
            packed = oracle.bucket_pack(lay, b, grads)
            bdev = [_dev(x, int(rng.integers(0, 8)), keep) for x in packed]
            zr.zr_reduce_scatter_avg_norm(zl, b, bdev, scale, g_out, chk)
    # the oracle's averages and check
    g_ref = [np.full(lay.S, np.nan, np.float32) for _ in range(world)]
    for b in range(lay.n_buckets):
        oracle.reduce_scatter_avg(lay, b, oracle.bucket_pack(lay, b, grads), scale, g_ref)
    for r in range(world):
        assert np.array_equal(_bits(g_out[r]), g_ref[r].view(np.uint32)), r
    ref0 = oracle.grad_check(g_ref, 0.0)
    max_norm = float(np.float32(ref0.norm * max_norm_frac)) if max_norm_frac > 0 else 0.0
    ref = oracle.grad_check(g_ref, max_norm)
    zr.zr_grad_check_finalize(chk, max_norm)
    got = zr.zr_gradcheck_read(chk)
    _check_stats(got, ref, exact=kind == "int" and world & (world - 1) == 0)
    # the clipped step
    (p, m, v), (P_, M_, V_) = _state(rng, lay, keep)
    param = torch.full((lay.P,), float("nan"), dtype=torch.bfloat16, device="cuda")
    hp = W.AdamW(step=int(rng.integers(1, 20)))
    zr.zr_adam_clip_step(zl, P_, M_, V_, g_out, hp, chk, param)
    torch.cuda.synchronize()
    rparam = np.zeros(lay.P, np.uint16)
    oracle.adam_clip_step(lay, p, m, v, g_ref, hp, got["coef"], got["skip"], rparam)
    assert np.array_equal(_bits(param), rparam)
    for r in range(world):
        for a, b_ in ((P_[r], p[r]), (M_[r], m[r]), (V_[r], v[r])):
            assert np.array_equal(_bits(a), b_.view(np.uint32)), r
    return got, ref


@pytest.mark.parametrize("world,seed,n,hi,B", CASES)
@pytest.mark.parametrize("path", ["direct", "packed"])
@pytest.mark.parametrize("kind,frac", [("int", 0.5), ("normal", 0.3), ("normal", 0.0), ("int", 2.0)])
def test_check_and_clipped_step_bf16(zr, world, seed, n, hi, B, path, kind, frac):
    got, ref = _run_case(zr, world, seed, n, hi, B, "bf16", kind, path, frac)
    if frac == 0.5:
        assert got["coef"] < 1.0


@pytest.mark.parametrize("world,seed,n,hi,B", CASES[:3])
@pytest.mark.parametrize("path", ["direct", "packed"])
@pytest.mark.parametrize("dtype", ["fp16", "fp32"])
def test_check_and_clipped_step_other_dtypes(zr, world, seed, n, hi, B, path, dtype):
    _run_case(zr, world, seed, n, hi, B, dtype, "normal", path, 0.4)


@pytest.mark.parametrize("world,seed,n,hi,B", CASES[:3])
def test_check_under_reverse_arrival(zr, world, seed, n, hi, B):
    _run_case(zr, world, seed, n, hi, B, "bf16", "int", "direct", 0.5, arrival="reverse")


@pytest.mark.parametrize("world", [4, 16])
def test_without_clipping_equals_the_one_pass_step(zr, world):
    from zero_partition_aware_gb300.engine import DPGroup
    rng = np.random.default_rng(world)
    numel = W.random_numels(rng, 60, 1, 40_000)
    wl = W.Workload("c", tuple(numel), world, 1 << 19, ("normal", 1e-2), 0.02, ("absnormal", 1e-4), W.AdamW(step=3))
    inp = W.draw_inputs(wl, "cuda", seed=world)
    hp = W.AdamW(step=3)
    groups = []
    for _ in range(2):
        g = DPGroup(numel, world, wl.bucket)
        g.load_flat(inp["master"], inp["m"], inp["v"])
        groups.append(g)
    L = groups[0].layout
    rows = [[inp["grads"][k][0][L.param(i)[0]: L.param(i)[0] + numel[i]] for i in range(len(numel))]
            for k in range(world)]
    a, b = groups
    a.step_direct(a.direct_plan(a.grad_table(rows)), hp)
    b.step_direct_clipped(b.direct_plan(b.grad_table(rows)), hp, 0.0)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(a.param[: L.P]), _bits(b.param[: L.P]))
    for r in range(world):
        for x, y in ((a.master[r], b.master[r]), (a.m[r], b.m[r]), (a.v[r], b.v[r])):
            assert np.array_equal(_bits(x), _bits(y)), r
    st = zr.zr_gradcheck_read(b.check)
    assert st["coef"] == 1.0 and not st["skip"]


@pytest.mark.parametrize("plant", ["inf", "-inf", "nan", "huge"])
@pytest.mark.parametrize("path", ["direct", "packed"])
def test_overflow_skips_the_step(zr, plant, path):
    world, n = 8, 20
    rng = np.random.default_rng(77)
    numel = W.random_numels(rng, n, 1, 5000)
    lay = oracle.layout(numel, world, 9000)
    zl = zr.Layout(numel, world, 9000)
    grads = [[_grad_values(rng, k, "bf16", "normal") for k in numel] for _ in range(world)]
    val = {"inf": np.float32(np.inf), "-inf": np.float32(-np.inf), "nan": np.float32(np.nan),
           "huge": np.float32(2.0 ** 70)}[plant]
    i = int(rng.integers(0, n))
    grads[3][i][int(rng.integers(0, numel[i]))] = oracle.f32_to_bf16(np.array([val], np.float32))[0]
    keep = []
    scale = float(np.float32(1.0 / world))
    g_out = [_dev(np.zeros(lay.S, np.float32), 1, keep) for _ in range(world)]
    chk = zr.GradCheck()
    if path == "direct":
        plan = zr.DirectPlan(zl, [[_dev(g, 3, keep) for g in row] for row in grads])
        for b in range(lay.n_buckets):
            zr.zr_rs_direct_norm(plan, b, scale, g_out, chk)
    else:
        for b in range(lay.n_buckets):
            zr.zr_reduce_scatter_avg_norm(zl, b, [_dev(x, 5, keep) for x in oracle.bucket_pack(lay, b, grads)],
                                          scale, g_out, chk)
    g_ref = [np.zeros(lay.S, np.float32) for _ in range(world)]
    for b in range(lay.n_buckets):
        oracle.reduce_scatter_avg(lay, b, oracle.bucket_pack(lay, b, grads), scale, g_ref)
    ref = oracle.grad_check(g_ref, 1.0)
    assert ref.skip and ref.nonfinite == 1
    zr.zr_grad_check_finalize(chk, 1.0)
    (p, m, v), (P_, M_, V_) = _state(rng, lay, keep)
    param = torch.full((lay.P,), 1.5, dtype=torch.bfloat16, device="cuda")
    zr.zr_adam_clip_step(zl, P_, M_, V_, g_out, W.AdamW(step=2), chk, param)
    got = zr.zr_gradcheck_read(chk)
    assert got["skip"] and got["nonfinite"] == 1 and got["coef"] == 1.0
    assert (_bits(param) == oracle.f32_to_bf16(np.array([1.5], np.float32))[0]).all()
    for r in range(world):
        for a, b_ in ((P_[r], p[r]), (M_[r], m[r]), (V_[r], v[r])):
            assert np.array_equal(_bits(a), b_.view(np.uint32)), r


@pytest.mark.parametrize("scale_to", [1e-35, 1e-20, 1e17, 3e18])
def test_norm_across_magnitudes(zr, scale_to):
    """Squares outside [2^-100, 2^100] take the exact double route; the norm stays within 1e-6."""
    world = 4
    rng = np.random.default_rng(5)
    numel = W.random_numels(rng, 12, 1, 3000)
    lay = oracle.layout(numel, world, 4000)
    zl = zr.Layout(numel, world, 4000)
    grads = [[(rng.standard_normal(k) * scale_to).astype(np.float32) for k in numel] for _ in range(world)]
    keep = []
    g_out = [_dev(np.zeros(lay.S, np.float32), 0, keep) for _ in range(world)]
    chk = zr.GradCheck()
    plan = zr.DirectPlan(zl, [[_dev(g, 1, keep) for g in row] for row in grads])
    for b in range(lay.n_buckets):
        zr.zr_rs_direct_norm(plan, b, 0.25, g_out, chk)
    zr.zr_grad_check_finalize(chk, 0.0)
    got = zr.zr_gradcheck_read(chk)
    g_ref = [np.zeros(lay.S, np.float32) for _ in range(world)]
    for b in range(lay.n_buckets):
        oracle.reduce_scatter_avg(lay, b, oracle.bucket_pack(lay, b, grads), 0.25, g_ref)
    ref = oracle.grad_check(g_ref, 0.0)
    assert got["nonfinite"] == ref.nonfinite == 0
    assert ref.sumsq > 0 and abs(got["sumsq"] - ref.sumsq) <= RTOL_SUMSQ * ref.sumsq


def test_outcome_repeats_and_sums_are_cleared(zr):
    """Two identical steps give bit-identical outcomes: the blocks' sums are added
    in a fixed order and finalize clears them."""
    world = 16
    rng = np.random.default_rng(6)
    numel = W.random_numels(rng, 200, 1, 200_000)
    lay = oracle.layout(numel, world, 1 << 21)
    zl = zr.Layout(numel, world, 1 << 21)
    keep = []
    grads = [[torch.randn(k, device="cuda").mul_(1e-2).to(torch.bfloat16) for k in numel] for _ in range(world)]
    g_out = [torch.zeros(lay.S, device="cuda") for _ in range(world)]
    plan = zr.DirectPlan(zl, grads)
    chk = zr.GradCheck()
    outs = []
    for _ in range(3):
        for b in range(lay.n_buckets):
            zr.zr_rs_direct_norm(plan, b, 1.0 / 16, g_out, chk)
        zr.zr_grad_check_finalize(chk, 1.0)
        outs.append(zr.zr_gradcheck_read(chk))
    assert outs[0] == outs[1] == outs[2]
    ref = oracle.grad_check([t.cpu().numpy() for t in g_out], 1.0)
    assert abs(outs[0]["sumsq"] - ref.sumsq) <= RTOL_SUMSQ * ref.sumsq
    # a reset drops sums of an abandoned pass
    zr.zr_rs_direct_norm(plan, 0, 1.0 / 16, g_out, chk)
    zr.zr_gradcheck_reset(chk)
    for b in range(lay.n_buckets):
        zr.zr_rs_direct_norm(plan, b, 1.0 / 16, g_out, chk)
    zr.zr_grad_check_finalize(chk, 1.0)
    assert zr.zr_gradcheck_read(chk) == outs[0]
