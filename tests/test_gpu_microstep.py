"""fp32 main-grad accumulation over micro-steps, with the last micro-step
folded into the fused step (GPU), against the oracle.

"Megatron-LM 分布式训练（四）" §"四步接力": every micro-step's bf16 grad is added
into the fp32 contiguous main_grad buffer, which is then reduced bucket by
bucket. zr_grad_accumulate_first starts the sum (0 + g, no read of the buffer);
zr_rs_adam_fused_acc adds the last micro-step's grads while it averages, so
the accumulated main_grad is never stored. Both must equal the oracle's
accumulation followed by its fused step, bit for bit, and the fused-acc call
must leave main_in untouched.
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
    dt = {np.dtype(np.float16): torch.float16, np.dtype(np.uint16): torch.bfloat16,
          np.dtype(np.float32): torch.float32}[a.dtype]
    base = torch.zeros(a.size + phase + 8, dtype=dt, device="cuda")
    v = base[phase:phase + a.size]
    src = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if a.dtype == np.uint16 else torch.from_numpy(a)
    v.copy_(src.cuda())
    keep.append(base)
    return v


def _half(rng, n, dt, std=1e-3):
    x = (rng.standard_normal(n) * std).astype(np.float32)
    x[rng.random(n) < 0.01] = -0.0
    return oracle.f32_to_bf16(x) if dt == "bf16" else x.astype(np.float16)


@pytest.mark.parametrize("n", [1, 7, 255, 4097, 100_003])
@pytest.mark.parametrize("dt", ["bf16", "fp16", "fp32"])
def test_accumulate_first(zr, n, dt):
    rng = np.random.default_rng(n)
    g = (rng.standard_normal(n) * 1e-3).astype(np.float32) if dt == "fp32" else _half(rng, n, dt)
    if dt == "fp32":
        g[rng.random(n) < 0.01] = -0.0
    keep = []
    main = _dev(np.full(n, np.nan, np.float32), int(rng.integers(0, 4)), keep)
    gd = _dev(g, int(rng.integers(0, 8)), keep)
    zr.zr_grad_accumulate_first(main, gd)
    torch.cuda.synchronize()
    ref = np.zeros(n, np.float32)
    oracle.grad_accumulate(ref, g)
    assert np.array_equal(_bits(main), ref.view(np.uint32))
    assert not (_bits(main) == 0x80000000).any()  # 0 + -0 = +0


CASES = [(2, 0, 9, 6000, 9000), (4, 1, 20, 5000, 12000), (8, 2, 40, 8000, 100_000), (3, 3, 15, 3000, 1),
         (16, 4, 25, 3000, 40_000), (32, 5, 12, 2000, 30_000)]


@pytest.mark.parametrize("world,seed,n,hi,B", CASES)
@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_fused_acc_equals_accumulate_then_fused(zr, world, seed, n, hi, B, dt):
    rng = np.random.default_rng(1100 + seed)
    numel = W.random_numels(rng, n, 1, hi)
    lay = oracle.layout(numel, world, B)
    zl = zr.Layout(numel, world, B)
    keep = []
    hp = W.AdamW(step=int(rng.integers(1, 20)))
    scale = float(np.float32(1.0 / world))
    flat = lambda std: np.concatenate([(rng.standard_normal(lay.T) * std).astype(np.float32),
                                       np.zeros(lay.P - lay.T, np.float32)])
    p, m, v = (np.split(flat(0.02), world), np.split(np.abs(flat(1e-4)), world), np.split(np.abs(flat(1e-4)), world))
    p, m, v = ([np.ascontiguousarray(a) for a in arrs] for arrs in (p, m, v))
    P_ = [_dev(a, int(rng.integers(0, 4)), keep) for a in p]
    M_ = [_dev(a, int(rng.integers(0, 4)), keep) for a in m]
    V_ = [_dev(a, int(rng.integers(0, 4)), keep) for a in v]
    param = torch.full((lay.P,), float("nan"), dtype=torch.bfloat16, device="cuda")
    gout = [_dev(np.full(lay.S, np.nan, np.float32), int(rng.integers(0, 4)), keep) for _ in range(world)]
    rparam = np.zeros(lay.P, np.uint16)
    rg = [np.full(lay.S, np.nan, np.float32) for _ in range(world)]
    for b in range(lay.n_buckets):
        _, nb = lay.bucket(b)
        main = [(rng.standard_normal(nb) * 3e-3).astype(np.float32) for _ in range(world)]
        last = [_half(rng, nb, dt) for _ in range(world)]
        main_d = [_dev(a, int(rng.integers(0, 4)), keep) for a in main]
        last_d = [_dev(a, int(rng.integers(0, 8)), keep) for a in last]
        before = [_bits(t).copy() for t in main_d]
        zr.zr_rs_adam_fused_acc(zl, b, main_d, last_d, scale, P_, M_, V_, hp, param, shard_grad_out=gout)
        torch.cuda.synchronize()
        for k in range(world):
            assert np.array_equal(_bits(main_d[k]), before[k]), "main_in was written"
        acc = [a.copy() for a in main]
        for k in range(world):
            oracle.grad_accumulate(acc[k], last[k])
        oracle.rs_adam_fused(lay, b, acc, scale, p, m, v, hp, rparam, rg)
    assert np.array_equal(_bits(param), rparam)
    for r in range(world):
        for a, b_ in ((P_[r], p[r]), (M_[r], m[r]), (V_[r], v[r]), (gout[r], rg[r])):
            assert np.array_equal(_bits(a), b_.view(np.uint32)), r


def test_fused_acc_rejects(zr):
    lay = zr.Layout([100, 200], 40, 1000)
    two = [torch.zeros(8, device="cuda") for _ in range(40)]
    with pytest.raises(zr.ZrError) as e:
        zr.zr_rs_adam_fused_acc(lay, 0, two, [t.to(torch.bfloat16) for t in two], 0.5, two, two, two, W.AdamW())
    assert e.value.status == zr.ZR_ERR_UNSUPPORTED
