"""A launch that fails in the middle of a step (GPU): the error reaches the
caller and no later bucket runs.

The library's failure injection (ZR_FAIL_AT_LAUNCH, see zr_launch_count in
include/zr.h) makes one launch of a step fail on the host, before it is
enqueued. DPGroup.step_direct must raise the library's status and message;
the buckets whose launches ran must equal the oracle's step, and every bucket
after the failing launch must be untouched (state and parameters as before).
Once the variable is cleared the same group steps normally again.
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
    t = t.detach().cpu().contiguous()
    return t.view(torch.int16).numpy().view(np.uint16) if t.element_size() == 2 else \
        t.view(torch.int32).numpy().view(np.uint32)


@pytest.mark.parametrize("per_bucket", [True, False], ids=["per_bucket", "grouped"])
def test_failure_mid_step_stops_the_step(mods, monkeypatch, per_bucket):
    engine, zr = mods
    rng = np.random.default_rng(3)
    world, B = 8, 4000
    numel = W.random_numels(rng, 120, 200, 3000)
    wl = W.Workload("fail", tuple(numel), world, B, ("normal", 1e-2), 0.02, ("absnormal", 1e-4), W.AdamW(step=2))
    inp = W.draw_inputs(wl, "cuda", seed=3)
    grp = engine.DPGroup(numel, world, B)
    grp.load_flat(inp["master"], inp["m"], inp["v"])
    L = grp.layout
    assert L.n_buckets > 20  # more than one grouped launch (16 buckets each) and more than 5 buckets
    rows = [[inp["grads"][k][0][L.param(i)[0]: L.param(i)[0] + numel[i]] for i in range(len(numel))]
            for k in range(world)]
    plan = grp.direct_plan(grp.grad_table(rows))
    before = [_bits(t[: L.P]) for t in grp.flat_state()] + [_bits(grp.param[: L.P])]
    torch.cuda.synchronize()
    fail_at = 5 if per_bucket else 2  # the 5th bucket's launch, or the grouped call's second launch
    monkeypatch.setenv("ZR_FAIL_AT_LAUNCH", str(zr.zr_launch_count() + fail_at))
    n0 = zr.zr_launch_count()
    with pytest.raises(zr.ZrError) as e:
        grp.step_direct(plan, wl.adam, per_bucket=per_bucket)
    assert e.value.status == zr.ZR_ERR_CUDA and "injected failure" in str(e.value)
    assert zr.zr_launch_count() - n0 == fail_at - 1
    torch.cuda.synchronize()
    after = [_bits(t[: L.P]) for t in grp.flat_state()] + [_bits(grp.param[: L.P])]
    # the oracle's step, bucket by bucket
    lay = oracle.layout(numel, world, B)
    g = [oracle.params_from_flat(lay, W.bf16_bits(inp["grads"][k][0].cpu())) for k in range(world)]
    p, m, v = (oracle.shards_from_flat(lay, t.cpu().numpy()) for t in (inp["master"], inp["m"], inp["v"]))
    param = np.zeros(lay.P, np.uint16)
    for b in range(lay.n_buckets):
        oracle.rs_adam_fused(lay, b, oracle.bucket_pack(lay, b, g), grp.scale, p, m, v, wl.adam, param)
    want = [np.concatenate(a).view(np.uint32) for a in (p, m, v)] + [param]
    # the buckets that ran form a prefix: each equals the oracle, every later one is untouched
    done = 0
    for b in range(L.n_buckets):
        s, n = L.bucket(b)
        sl = slice(s, s + n)
        if all(np.array_equal(x[sl], y[sl]) for x, y in zip(after, want)):
            assert done == b, f"bucket {b} ran after an untouched bucket"
            done += 1
        else:
            assert all(np.array_equal(x[sl], y[sl]) for x, y in zip(after, before)), f"bucket {b} half-written"
    assert 1 <= done < L.n_buckets
    if per_bucket:
        assert done == fail_at - 1
    # cleared: the library is usable again; the step from the same inputs equals the oracle everywhere
    monkeypatch.delenv("ZR_FAIL_AT_LAUNCH")
    grp2 = engine.DPGroup(numel, world, B)
    grp2.load_flat(inp["master"], inp["m"], inp["v"])
    grp2.step_direct(grp2.direct_plan(grp2.grad_table(rows)), wl.adam, per_bucket=per_bucket)
    torch.cuda.synchronize()
    got = [_bits(t[: L.P]) for t in grp2.flat_state()] + [_bits(grp2.param[: L.P])]
    for x, y in zip(got, want):
        assert np.array_equal(x, y)
