"""The step captured in a CUDA graph and replayed (GPU).

Every libzr kernel takes its tables as launch parameters (copied into the
graph when it is captured) or from memory a plan or a check object owns, and no
entry point allocates device memory or synchronises, so a whole step can be
captured once and replayed. Replays must equal eager steps bit for bit: the
direct step over every bucket, the step with the global gradient check (whose
outcome stays on the device between its kernels), and the micro-step path.
"""
import numpy as np
import pytest
import torch

from zero_partition_aware_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mods():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from zero_partition_aware_gb300 import build
    build.build()
    from zero_partition_aware_gb300 import engine, zr
    return engine, zr


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16 if t.element_size() == 2 else torch.int32).numpy()


def _groups(engine, numel, world, B, inp):
    out = []
    for _ in range(2):
        g = engine.DPGroup(numel, world, B)
        g.load_flat(inp["master"], inp["m"], inp["v"])
        out.append(g)
    return out


def _same(a, b, L, world):
    assert np.array_equal(_bits(a.param[: L.P]), _bits(b.param[: L.P]))
    for r in range(world):
        for x, y in ((a.master[r], b.master[r]), (a.m[r], b.m[r]), (a.v[r], b.v[r])):
            assert np.array_equal(_bits(x), _bits(y)), r


def _capture(fn):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # eager warm-up: per-device launch caches filled outside capture
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


@pytest.mark.parametrize("world,n,hi,B", [(16, 200, 200_000, 1 << 21), (4, 30, 20_000, 40_000)])
def test_direct_step_graph_replays_eager_steps(mods, world, n, hi, B):
    engine, zr = mods
    rng = np.random.default_rng(world)
    numel = W.random_numels(rng, n, 1, hi)
    wl = W.Workload("g", tuple(numel), world, B, ("normal", 1e-2), 0.02, ("absnormal", 1e-4), W.AdamW(step=2))
    inp = W.draw_inputs(wl, "cuda", seed=world)
    hp = W.AdamW(step=2)
    a, b = _groups(engine, numel, world, B, inp)
    L = a.layout
    rows = [[inp["grads"][k][0][L.param(i)[0]: L.param(i)[0] + numel[i]] for i in range(n)] for k in range(world)]
    pa, pb = a.direct_plan(a.grad_table(rows)), b.direct_plan(b.grad_table(rows))
    for _ in range(4):  # eager: the warm-up step of b is matched by one more eager step of a
        a.step_direct(pa, hp)
    g = _capture(lambda: b.step_direct(pb, hp))
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    _same(a, b, L, world)


def test_clipped_step_graph_replays_eager_steps(mods):
    engine, zr = mods
    world, n, B = 8, 120, 1 << 20
    rng = np.random.default_rng(3)
    numel = W.random_numels(rng, n, 1, 100_000)
    wl = W.Workload("gc", tuple(numel), world, B, ("normal", 1e-2), 0.02, ("absnormal", 1e-4), W.AdamW(step=2))
    inp = W.draw_inputs(wl, "cuda", seed=3)
    hp = W.AdamW(step=2)
    a, b = _groups(engine, numel, world, B, inp)
    L = a.layout
    rows = [[inp["grads"][k][0][L.param(i)[0]: L.param(i)[0] + numel[i]] for i in range(n)] for k in range(world)]
    pa, pb = a.direct_plan(a.grad_table(rows)), b.direct_plan(b.grad_table(rows))
    b.grad_shards()
    for _ in range(3):
        a.step_direct_clipped(pa, hp, 0.5)
    g = _capture(lambda: b.step_direct_clipped(pb, hp, 0.5))
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    _same(a, b, L, world)
    sa, sb = zr.zr_gradcheck_read(a.check), zr.zr_gradcheck_read(b.check)
    assert sa == sb and sa["coef"] < 1.0


def test_micro_step_path_graph_replays_eager_steps(mods):
    """First micro-step, a middle one and the last folded into the fused step."""
    engine, zr = mods
    world, n, B = 8, 40, 300_000
    rng = np.random.default_rng(4)
    numel = W.random_numels(rng, n, 1, 50_000)
    wl = W.Workload("gm", tuple(numel), world, B, ("normal", 1e-3), 0.02, ("absnormal", 1e-4), W.AdamW(step=2),
                    micro_steps=3)
    inp = W.draw_inputs(wl, "cuda", seed=4)
    hp = W.AdamW(step=2)
    groups = []
    for _ in range(2):
        g = engine.DPGroup(numel, world, B, grad_dtype=torch.float32, allocate_buckets=False)
        g.load_flat(inp["master"], inp["m"], inp["v"])
        groups.append(g)
    a, b = groups
    L = a.layout
    mbs = [[torch.zeros(L.P, dtype=torch.bfloat16, device="cuda") for _ in range(3)] for _ in range(world)]
    for k in range(world):
        for s_ in range(3):
            mbs[k][s_][: L.T].copy_(inp["grads"][k][s_])

    def step(grp):
        main = grp._main
        for k in range(world):
            zr.zr_grad_accumulate_first(main[k], mbs[k][0])
            zr.zr_grad_accumulate(main[k], mbs[k][1])
        grp.step_in_place_acc(grp._views, grp._last, hp)

    for grp in (a, b):
        grp._main = [torch.zeros(L.P, dtype=torch.float32, device="cuda") for _ in range(world)]
        grp._views = grp.main_grad_views(grp._main)
        grp._last = grp.main_grad_views([row[2] for row in mbs])
    for _ in range(3):
        step(a)
    g = _capture(lambda: step(b))
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    _same(a, b, L, world)
