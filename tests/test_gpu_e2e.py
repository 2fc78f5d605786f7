"""The pipelined and overlapped steps (GPU) against the oracle.

DPGroup.step_direct_from_host copies each bucket's gradients in on one
stream, runs zr_step_direct on another and copies the bucket's bf16 params out
on a third. DPGroup.step_overlapped packs bucket b+1 on a second stream while
bucket b is reduced ("DeepSpeed ZeRO 通信优化深度解析" §四, §五 overlap_comm;
"Megatron-LM 分布式训练（四）" §"梯度缓冲区+分桶+overlap"). A stream-ordering
mistake would corrupt the overlapped path and the sequential one alike, so
both are held to the oracle's bucket path (bucket_pack, then rs_adam_fused
per bucket, in bucket order), bit for bit, over two consecutive steps where
the pipeline reuses its buffers.
"""
import numpy as np
import pytest
import torch

import oracle
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


def _oracle_steps(numel, world, B, grads_flat, master, m, v, hp, steps, arrival=None):
    """`steps` oracle steps from the flat [T] state and each rank's flat [T] bf16
    gradients: per bucket, in bucket order, the pack and the fused step.
    Returns the partitions (master, m, v as [world][S] fp32) and the bf16 params."""
    lay = oracle.layout(numel, world, B, order=arrival)
    g = [oracle.params_from_flat(lay, W.bf16_bits(t.cpu())) for t in grads_flat]
    p, mm, vv = (oracle.shards_from_flat(lay, t.cpu().numpy()) for t in (master, m, v))
    param = np.zeros(lay.P, np.uint16)
    scale = float(np.float32(1.0 / world))
    for _ in range(steps):
        for b in range(lay.n_buckets):
            oracle.rs_adam_fused(lay, b, oracle.bucket_pack(lay, b, g), scale, p, mm, vv, hp, param)
    return lay, p, mm, vv, param


def _assert_oracle(grp, lay, p, m, v, param, what):
    assert np.array_equal(_bits(grp.param[: lay.P]).view(np.uint16), param), f"{what}: params"
    for r in range(lay.world):
        for dev, ref, nm in ((grp.master[r], p[r], "master"), (grp.m[r], m[r], "m"), (grp.v[r], v[r], "v")):
            assert np.array_equal(_bits(dev).view(np.uint32), ref.view(np.uint32)), f"{what}: {nm} of rank {r}"


@pytest.mark.parametrize("grouped", [False, True], ids=["per_bucket", "groups_of_3"])
@pytest.mark.parametrize("world,n,hi,B", [(4, 40, 30_000, 60_000), (16, 120, 200_000, 1 << 21)])
def test_from_host_equals_device_resident(mods, world, n, hi, B, grouped):
    engine, zr = mods
    rng = np.random.default_rng(world)
    numel = W.random_numels(rng, n, 1, hi)
    wl = W.Workload("e2e", tuple(numel), world, B, ("int", -8, 8), 0.02, ("absnormal", 1e-4), W.AdamW(step=3))
    offs = W.arena_offsets(numel, 256)
    arena_n = offs[-1] + numel[-1]
    gen = W.generator("cuda", 5)
    master = torch.randn(wl.total, generator=gen, device="cuda").mul_(0.02)
    m = W.draw_state(wl, wl.total, gen, "cuda")
    v = W.draw_state(wl, wl.total, gen, "cuda")
    arenas = [W.draw_grad(wl, arena_n, gen, "cuda") for _ in range(world)]
    hp = W.AdamW(step=3)

    def group(dev_arenas):
        g = engine.DPGroup(numel, world, B, device="cuda")
        g.load_flat(master, m, v)
        views = [[a[o:o + k] for o, k in zip(offs, numel)] for a in dev_arenas]
        return g, g.direct_plan(g.grad_table(views))

    # reference: gradients resident on the device
    ref, ref_plan = group(arenas)
    for _ in range(2):
        ref.step_direct(ref_plan, hp)
    # the pipelined step: device arenas start as garbage, the host holds the gradients
    dev = [torch.full_like(a, float("nan")) for a in arenas]
    host = [a.cpu().pin_memory() for a in arenas]
    got, got_plan = group(dev)
    L = got.layout
    lo, hiw = [None] * L.n_buckets, [0] * L.n_buckets
    for i, k in enumerate(numel):
        b = L.param(i)[1]
        lo[b] = offs[i] if lo[b] is None else lo[b]
        hiw[b] = offs[i] + k
    # per bucket, or groups of three consecutive buckets copied as one range per rank
    groups = [(b, min(b + 3, L.n_buckets)) for b in range(0, L.n_buckets, 3)] if grouped else None
    spans = groups or [(b, b + 1) for b in range(L.n_buckets)]
    pairs = [[(h[lo[b0]:hiw[b1 - 1]], d[lo[b0]:hiw[b1 - 1]]) for h, d in zip(host, dev)] for b0, b1 in spans]
    param_host = torch.full((L.P,), -1, dtype=torch.int16).pin_memory().view(torch.bfloat16)
    for step in range(2):  # the second step reuses the device arenas and the host buffer
        if step:
            for d in dev:
                d.fill_(float("nan"))
            param_host.view(torch.int16).fill_(-1)
        got.step_direct_from_host(got_plan, hp, pairs, param_host, groups=groups)
    torch.cuda.synchronize()
    flat = [torch.cat([a[o:o + k] for o, k in zip(offs, numel)]) for a in arenas]
    lay, p, m_, v_, param = _oracle_steps(numel, world, B, flat, master, m, v, hp, 2)
    _assert_oracle(got, lay, p, m_, v_, param, "host-pipelined step")
    assert np.array_equal(_bits(param_host).view(np.uint16), param), "the host copy of the params"
    assert np.array_equal(_bits(got.param[: L.P]), _bits(ref.param[: L.P]))
    assert np.array_equal(_bits(param_host), _bits(ref.param[: L.P]))
    for r in range(world):
        for a, b in ((got.master[r], ref.master[r]), (got.m[r], ref.m[r]), (got.v[r], ref.v[r])):
            assert np.array_equal(_bits(a), _bits(b)), r


@pytest.mark.parametrize("flat_order", [False, True], ids=["fused", "flat_order_reverse_arrival"])
@pytest.mark.parametrize("world,n,hi,B", [(4, 40, 30_000, 60_000), (16, 120, 200_000, 1 << 21), (8, 5, 1000, 1)])
def test_overlapped_pack_and_fused_equal_the_oracle(mods, world, n, hi, B, flat_order):
    """Packing bucket b+1 on a second stream while bucket b is reduced (two
    bucket buffer sets), two steps in a row, equals the oracle's two steps bit
    for bit, and so does the sequential step; with flat_order, under backward
    arrival, each bucket is reduced by the direct kernel over the buffer set's
    param slices."""
    engine, zr = mods
    rng = np.random.default_rng(100 + world)
    numel = W.random_numels(rng, n, 1, hi)
    wl = W.Workload("ov", tuple(numel), world, B, ("normal", 1e-2), 0.02, ("absnormal", 1e-4), W.AdamW(step=2))
    inp = W.draw_inputs(wl, "cuda", seed=world)
    hp = W.AdamW(step=2)
    arrival = list(range(n - 1, -1, -1)) if flat_order else None
    groups = []
    for _ in range(2):
        g = engine.DPGroup(numel, world, B, device="cuda", arrival=arrival)
        g.load_flat(inp["master"], inp["m"], inp["v"])
        groups.append(g)
    L = groups[0].layout
    rows = [[inp["grads"][k][0][L.param(i)[0]: L.param(i)[0] + numel[i]] for i in range(len(numel))]
            for k in range(world)]
    a, b = groups
    ta, tb = a.grad_table(rows), b.grad_table(rows)
    a.step(ta, hp, plan=a.pack_plan(ta))
    plans = b.overlap_plans(tb)
    for _ in range(2):  # twice: the second step reuses both buffer sets
        b.step_overlapped(plans, hp, flat_order=flat_order)
    a.step(ta, hp, plan=a.pack_plan(ta))
    torch.cuda.synchronize()
    lay, p, m_, v_, param = _oracle_steps(numel, world, B, [inp["grads"][k][0] for k in range(world)],
                                          inp["master"], inp["m"], inp["v"], hp, 2, arrival=arrival)
    _assert_oracle(b, lay, p, m_, v_, param, "overlapped step")
    _assert_oracle(a, lay, p, m_, v_, param, "sequential step")
    assert np.array_equal(_bits(a.param[: L.P]), _bits(b.param[: L.P]))
    for r in range(world):
        for x, y in ((a.master[r], b.master[r]), (a.m[r], b.m[r]), (a.v[r], b.v[r])):
            assert np.array_equal(_bits(x), _bits(y)), r


@pytest.mark.parametrize("world,n,hi,B", [(4, 40, 30_000, 60_000), (16, 120, 200_000, 1 << 21)])
def test_host_resident_gradients_equal_the_oracle(mods, world, n, hi, B):
    """The direct step reading every rank's gradients in place from pinned host
    memory (a plan over pinned host tensors at random element phases) and
    writing the bf16 params into a pinned host buffer, two steps in a row, equals
    the oracle's two steps bit for bit; the device parameter buffer is left
    alone."""
    engine, zr = mods
    rng = np.random.default_rng(300 + world)
    numel = W.random_numels(rng, n, 1, hi)
    wl = W.Workload("zc", tuple(numel), world, B, ("normal", 1e-2), 0.02, ("absnormal", 1e-4), W.AdamW(step=4))
    inp = W.draw_inputs(wl, "cuda", seed=world + 1)
    hp = W.AdamW(step=4)
    g = engine.DPGroup(numel, world, B, device="cuda")
    g.load_flat(inp["master"], inp["m"], inp["v"])
    L = g.layout
    keep, rows = [], []
    for k in range(world):
        flat = inp["grads"][k][0].cpu()
        row = []
        for i, c in enumerate(numel):
            ph = int(rng.integers(0, 8))
            t = torch.empty(c + 8, dtype=torch.bfloat16).pin_memory()
            s0 = L.param(i)[0]
            t[ph:ph + c].copy_(flat[s0:s0 + c])
            keep.append(t)
            row.append(t[ph:ph + c])
        rows.append(row)
    plan = g.direct_plan(g.grad_table(rows))
    param_host = torch.full((L.P + 8,), -1, dtype=torch.int16).pin_memory().view(torch.bfloat16)
    g.param.view(torch.int16).fill_(7)
    for _ in range(2):
        g.step_direct(plan, hp, param_out=param_host)
    torch.cuda.synchronize()
    lay, p, m_, v_, param = _oracle_steps(numel, world, B, [inp["grads"][k][0] for k in range(world)],
                                          inp["master"], inp["m"], inp["v"], hp, 2)
    assert np.array_equal(_bits(param_host[: L.P]).view(np.uint16), param), "params in host memory"
    assert np.all(_bits(param_host[L.P:]) == -1), "wrote past the parameter buffer"
    assert np.all(_bits(g.param[: L.P]) == 7), "the device parameter buffer was written"
    for r in range(world):
        for dev, ref, nm in ((g.master[r], p[r], "master"), (g.m[r], m_[r], "m"), (g.v[r], v_[r], "v")):
            assert np.array_equal(_bits(dev).view(np.uint32), ref.view(np.uint32)), f"{nm} of rank {r}"


def test_host_mapped_answers_and_leaves_no_error(mods):
    """zr_host_mapped answers 1 for pinned host memory (mapped at the same
    address). For a pageable numpy buffer the answer depends on the system (a
    device that uses the host's page tables reaches any host memory at the same
    address); either way the call succeeds and leaves no pending CUDA error
    behind: the next library launch succeeds. The binding itself refuses
    pageable tensors whatever the system allows."""
    import ctypes
    engine, zr = mods
    pinned = torch.zeros(1 << 20, dtype=torch.float32).pin_memory()
    pageable = np.zeros(1 << 20, np.float32)
    m = ctypes.c_int32(-1)
    assert zr._lib.zr_host_mapped(pinned.data_ptr(), ctypes.byref(m)) == zr.ZR_OK and m.value == 1
    assert zr._lib.zr_host_mapped(pageable.ctypes.data, ctypes.byref(m)) == zr.ZR_OK and m.value in (0, 1)
    assert zr._lib.zr_host_mapped(pageable.ctypes.data, None) == zr.ZR_ERR_INVALID_ARG
    acc = torch.zeros(1 << 20, device="cuda")
    zr.zr_grad_accumulate(acc, torch.ones(1 << 20, dtype=torch.bfloat16, device="cuda"))
    torch.cuda.synchronize()
    assert float(acc.sum()) == float(1 << 20)
    with pytest.raises(ValueError, match="pageable"):
        zr.zr_grad_accumulate(acc, torch.ones(1 << 20, dtype=torch.bfloat16))
