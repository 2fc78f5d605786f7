"""GPU parity: libzr's sm_103a kernels against the CPU oracle, element by element.

Small cases span many warp-tiles with ragged tails, every 16-byte phase of
every stream and several world sizes (including the >64 launch-parameter
layout); outputs are compared bit-exactly, which is stricter than the
required 1e-6 relative (fp32) and 2^-8 relative (bf16). Guard zones around
every output check that nothing outside it is written. The full-size
workloads are compared at every element in tests/test_gpu_whole.py.
"""
import numpy as np
import pytest
import torch

import oracle
from zero_partition_aware_gb300 import workloads as W

pytestmark = pytest.mark.gpu

RTOL_F32 = 1e-6          # fp32 outputs: |gpu - ref| <= 1e-6 |ref| (we also demand bit equality)
RTOL_BF16 = 2.0 ** -8    # bf16 outputs
CANARY16 = 0x7FA5        # a NaN pattern no kernel writes
CANARY32 = 0x7FC0DEAD


@pytest.fixture(scope="module")
def zr():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from zero_partition_aware_gb300 import build
    build.build()
    from zero_partition_aware_gb300 import zr as mod
    return mod


# ----------------------------------------------------------------------------
# helpers
# ----------------------------------------------------------------------------

def _bits(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.view(torch.int32).numpy().view(np.uint32)


class Guarded:
    """A device view of n elements at a chosen element phase, with canary zones."""

    def __init__(self, n, dtype, phase, pad=40):
        self.n, self.phase = n, phase
        self.base = torch.empty(phase + n + pad, dtype=dtype, device="cuda")
        if dtype == torch.bfloat16:
            self.base.view(torch.int16).fill_(CANARY16)
            self.canary = np.uint16(CANARY16)
        else:
            self.base.view(torch.int32).fill_(CANARY32)
            self.canary = np.uint32(CANARY32)
        self.view = self.base[phase:phase + n]

    def set(self, values: np.ndarray):
        values = np.ascontiguousarray(values)
        if values.dtype == np.uint16:
            t = torch.from_numpy(values.view(np.int16)).view(torch.bfloat16)
        else:
            t = torch.from_numpy(values.astype(np.float32))
        self.view.copy_(t.to(self.base.dtype).cuda())

    def bits(self) -> np.ndarray:
        return _bits(self.view)

    def check_guards(self):
        b = _bits(self.base)
        assert np.all(b[: self.phase] == self.canary), "write before the buffer"
        assert np.all(b[self.phase + self.n:] == self.canary), "write past the buffer"


def _bf16_np(rng, n, std=1e-2):
    x = torch.from_numpy(rng.standard_normal(n).astype(np.float32) * np.float32(std))
    return W.bf16_bits(x.to(torch.bfloat16))


def _f32_np(rng, n, std=1.0):
    return (rng.standard_normal(n) * std).astype(np.float32)


def _assert_same(got_bits, ref, what, dtype="f32"):
    ref_bits = ref.view(np.uint32) if dtype == "f32" else ref
    if np.array_equal(got_bits, ref_bits):
        return
    bad = np.nonzero(got_bits != ref_bits)[0]
    if dtype == "f32":
        g = got_bits.view(np.float32)
        r = ref_bits.view(np.float32)
        rel = np.max(np.abs(g[bad] - r[bad]) / np.maximum(np.abs(r[bad]), 1e-30))
        tol_ok = rel <= RTOL_F32
    else:
        g = oracle.bf16_to_f32(got_bits)
        r = oracle.bf16_to_f32(ref_bits)
        rel = np.max(np.abs(g[bad] - r[bad]) / np.maximum(np.abs(r[bad]), 1e-30))
        tol_ok = rel <= RTOL_BF16
    raise AssertionError(f"{what}: {bad.size} elements differ (first at {bad[:5]}), max rel {rel:.3g}, "
                         f"within tolerance: {tol_ok}")


def _rand_phases(rng, k, es):
    return [int(x) for x in rng.integers(0, 16 // es, k)]


CASES = [  # (world, numel list generator seed, n params, max numel, bucket)
    (1, 0, 5, 3000, 2500),
    (2, 1, 9, 6000, 7000),
    (3, 2, 12, 5000, 9000),
    (4, 3, 7, 9000, 8192),
    (8, 4, 20, 4000, 15000),
    (16, 5, 40, 3000, 30000),
    (32, 6, 30, 4000, 50000),
    (100, 7, 10, 2000, 6000),
]


def _case(world, seed, n, hi, B):
    rng = np.random.default_rng(100 + seed)
    numel = W.random_numels(rng, n, 1, hi)
    return rng, numel, oracle.layout(numel, world, B)


# ----------------------------------------------------------------------------
# per-kernel parity
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("world,seed,n,hi,B", CASES)
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_pack(zr, world, seed, n, hi, B, dtype):
    rng, numel, lay = _case(world, seed, n, hi, B)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    es = 2 if dtype == "bf16" else 4
    zl = zr.Layout(numel, world, B)
    grads_np = [[(_bf16_np(rng, m) if dtype == "bf16" else _f32_np(rng, m)) for m in numel] for _ in range(world)]
    # half the replicas hold their params contiguously (merged segments), half scattered at random phases
    grads_dev, keep = [], []
    for k in range(world):
        row = []
        if k % 2 == 0:
            flat = np.concatenate(grads_np[k])
            g = Guarded(len(flat), tdt, int(rng.integers(0, 16 // es)))
            g.set(flat)
            keep.append(g)
            pos = 0
            for m in numel:
                row.append(g.view[pos:pos + m])
                pos += m
        else:
            for i, m in enumerate(numel):
                g = Guarded(m, tdt, int(rng.integers(0, 16 // es)))
                g.set(grads_np[k][i])
                keep.append(g)
                row.append(g.view)
        grads_dev.append(row)
    table = zr.PtrArray([t for row in grads_dev for t in row])
    for b in range(lay.n_buckets):
        _, nb = lay.bucket(b)
        outs = [Guarded(nb, tdt, ph) for ph in _rand_phases(rng, world, es)]
        zr.zr_bucket_pack(zl, b, table, [o.view for o in outs])
        torch.cuda.synchronize()
        want = oracle.bucket_pack(lay, b, grads_np)
        for k in range(world):
            outs[k].check_guards()
            assert np.array_equal(outs[k].bits(), want[k].view(outs[k].bits().dtype)), (b, k)
    # the planned path: one launch per bucket from device-resident descriptors
    mx = max(lay.bucket(b)[1] for b in range(lay.n_buckets))
    outs = [Guarded(mx, tdt, ph) for ph in _rand_phases(rng, world, es)]
    plan = zr.PackPlan(zl, table, [o.view for o in outs])
    for b in range(lay.n_buckets):
        _, nb = lay.bucket(b)
        for o in outs:
            o.view.view(torch.int16 if es == 2 else torch.int32).fill_(CANARY16 if es == 2 else CANARY32)
        zr.zr_bucket_pack_planned(plan, b)
        torch.cuda.synchronize()
        want = oracle.bucket_pack(lay, b, grads_np)
        for k in range(world):
            outs[k].check_guards()
            got = outs[k].bits()
            assert np.array_equal(got[:nb], want[k].view(got.dtype)), (b, k)
            assert np.all(got[nb:] == outs[k].canary), "planned pack wrote past the bucket"
    plan.close()
    for g in keep:
        g.check_guards()


def _buckets_on_device(rng, lay, b, world, tdt, es):
    _, nb = lay.bucket(b)
    vals = [(_bf16_np(rng, nb) if tdt == torch.bfloat16 else _f32_np(rng, nb, 1e-2)) for _ in range(world)]
    dev = []
    for k in range(world):
        g = Guarded(nb, tdt, int(rng.integers(0, 16 // es)))
        g.set(vals[k])
        dev.append(g)
    return vals, dev


@pytest.mark.parametrize("world,seed,n,hi,B", CASES)
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_reduce_scatter_avg(zr, world, seed, n, hi, B, dtype):
    rng, numel, lay = _case(world, seed, n, hi, B)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    es = 2 if dtype == "bf16" else 4
    zl = zr.Layout(numel, world, B)
    scale = float(np.float32(1.0 / world))
    for b in range(lay.n_buckets):
        vals, dev = _buckets_on_device(rng, lay, b, world, tdt, es)
        init = [np.full(lay.S, np.float32(np.nan), np.float32) for _ in range(world)]
        shards = [Guarded(lay.S, torch.float32, ph) for ph in _rand_phases(rng, world, 4)]
        for s, i0 in zip(shards, init):
            s.set(i0)
        zr.zr_reduce_scatter_avg(zl, b, [d.view for d in dev], scale, [s.view for s in shards])
        torch.cuda.synchronize()
        want = [i0.copy() for i0 in init]
        oracle.reduce_scatter_avg(lay, b, vals, scale, want)
        for r in range(world):
            shards[r].check_guards()
            # positions outside the bucket keep their NaN fill (same bits on both sides)
            _assert_same(shards[r].bits(), want[r], f"RS bucket {b} rank {r}")
        for d in dev:
            d.check_guards()


@pytest.mark.parametrize("world,seed,n,hi,B", CASES)
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("phases", ["same", "mixed"])
def test_rs_adam_fused(zr, world, seed, n, hi, B, dtype, phases):
    rng, numel, lay = _case(world, seed, n, hi, B)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    es = 2 if dtype == "bf16" else 4
    zl = zr.Layout(numel, world, B)
    scale = float(np.float32(1.0 / world))
    hp = W.AdamW(step=int(rng.integers(1, 20)))
    p_np = [_f32_np(rng, lay.S, 0.02) for _ in range(world)]
    m_np = [np.abs(_f32_np(rng, lay.S, 1e-4)) for _ in range(world)]
    v_np = [np.abs(_f32_np(rng, lay.S, 1e-4)) for _ in range(world)]
    for arrs in (p_np, m_np, v_np):  # the padding is zero, as the caller initialises it
        flat = np.concatenate(arrs)
        flat[lay.T:] = 0
        for r in range(world):
            arrs[r][:] = flat[r * lay.S:(r + 1) * lay.S]

    def mk(arrs):
        out = []
        for r in range(world):
            ph = 0 if phases == "same" else int(rng.integers(0, 4))
            g = Guarded(lay.S, torch.float32, ph)
            g.set(arrs[r])
            out.append(g)
        return out

    P_, M_, V_ = mk(p_np), mk(m_np), mk(v_np)
    G_ = mk([np.full(lay.S, np.float32(np.nan), np.float32) for _ in range(world)])
    param = Guarded(lay.P, torch.bfloat16, int(rng.integers(0, 8)))
    param.set(np.full(lay.P, 0x7FA5, np.uint16))
    want_p = [a.copy() for a in p_np]
    want_m = [a.copy() for a in m_np]
    want_v = [a.copy() for a in v_np]
    want_g = [np.full(lay.S, np.float32(np.nan), np.float32) for _ in range(world)]
    want_param = np.full(lay.P, 0x7FA5, np.uint16)
    for b in range(lay.n_buckets):
        vals, dev = _buckets_on_device(rng, lay, b, world, tdt, es)
        zr.zr_rs_adam_fused(zl, b, [d.view for d in dev], scale, [x.view for x in P_], [x.view for x in M_],
                            [x.view for x in V_], hp, param.view, [x.view for x in G_])
        oracle.rs_adam_fused(lay, b, vals, scale, want_p, want_m, want_v, hp, want_param, want_g)
    torch.cuda.synchronize()
    for r in range(world):
        for got, want, nm in ((P_, want_p, "p"), (M_, want_m, "m"), (V_, want_v, "v"), (G_, want_g, "g")):
            got[r].check_guards()
            _assert_same(got[r].bits(), want[r], f"fused {nm} rank {r}")
    param.check_guards()
    _assert_same(param.bits(), want_param, "fused param", dtype="bf16")


@pytest.mark.parametrize("world,seed,n,hi,B", CASES[:7])
def test_fused_without_optional_outputs_and_unfused_agree(zr, world, seed, n, hi, B):
    """Fused (no param, no grad out) == RS + AdamW + gather on the GPU, bit for bit."""
    rng, numel, lay = _case(world, seed, n, hi, B)
    zl = zr.Layout(numel, world, B)
    scale = float(np.float32(1.0 / world))
    hp = W.AdamW(step=3)
    dev = lambda a: torch.from_numpy(a).cuda()
    p0 = [_f32_np(rng, lay.S, 0.02) for _ in range(world)]
    flat = np.concatenate(p0)
    flat[lay.T:] = 0
    p0 = [flat[r * lay.S:(r + 1) * lay.S].copy() for r in range(world)]
    pa, pb = [dev(a) for a in p0], [dev(a) for a in p0]
    ma, mb = [torch.zeros(lay.S, device="cuda") for _ in range(world)], [torch.zeros(lay.S, device="cuda") for _ in range(world)]
    va, vb = [torch.zeros(lay.S, device="cuda") for _ in range(world)], [torch.zeros(lay.S, device="cuda") for _ in range(world)]
    g = [torch.zeros(lay.S, device="cuda") for _ in range(world)]
    for b in range(lay.n_buckets):
        _, nb = lay.bucket(b)
        x = [dev(_bf16_np(rng, nb).view(np.int16)).view(torch.bfloat16) for _ in range(world)]
        zr.zr_rs_adam_fused(zl, b, x, scale, pa, ma, va, hp)
        zr.zr_reduce_scatter_avg(zl, b, x, scale, g)
    zr.zr_adam_shard_step(zl, -1, pb, mb, vb, g, hp)
    param_a = torch.zeros(lay.P, dtype=torch.bfloat16, device="cuda")
    zr.zr_gather_cast_bf16(zl, pa, param_a)
    param_b = torch.zeros(lay.P, dtype=torch.bfloat16, device="cuda")
    zr.zr_gather_cast_bf16(zl, pb, param_b)
    torch.cuda.synchronize()
    for r in range(world):
        assert torch.equal(pa[r].view(torch.int32), pb[r].view(torch.int32))
        assert torch.equal(ma[r].view(torch.int32), mb[r].view(torch.int32))
        assert torch.equal(va[r].view(torch.int32), vb[r].view(torch.int32))
    assert torch.equal(param_a.view(torch.int16), param_b.view(torch.int16))


@pytest.mark.parametrize("world,seed,n,hi,B", CASES)
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("outputs", ["random_phases", "one_phase"])
def test_allreduce_avg(zr, world, seed, n, hi, B, dtype, outputs):
    """Outputs at random 16-byte phases and at one shared phase (then every
    output's stores are aligned like replica 0's)."""
    rng, numel, lay = _case(world, seed, n, hi, B)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    es = 2 if dtype == "bf16" else 4
    zl = zr.Layout(numel, world, B)
    scale = float(np.float32(1.0 / world))
    for b in range(min(lay.n_buckets, 3)):
        _, nb = lay.bucket(b)
        vals, dev = _buckets_on_device(rng, lay, b, world, tdt, es)
        phases = _rand_phases(rng, world, 4) if outputs == "random_phases" else [int(rng.integers(0, 4))] * world
        outs = [Guarded(nb, torch.float32, ph) for ph in phases]
        zr.zr_allreduce_avg(zl, b, [d.view for d in dev], scale, [o.view for o in outs])
        torch.cuda.synchronize()
        want = oracle.allreduce_avg(world, vals, scale)
        for k in range(world):
            outs[k].check_guards()
            _assert_same(outs[k].bits(), want[k], f"AR bucket {b} replica {k}")


@pytest.mark.parametrize("world,seed,n,hi,B", CASES)
@pytest.mark.parametrize("rank", [-1, 0])
def test_adam_shard_step(zr, world, seed, n, hi, B, rank):
    rng, numel, lay = _case(world, seed, n, hi, B)
    zl = zr.Layout(numel, world, B)
    hp = W.AdamW(step=int(rng.integers(1, 50)))
    arrs = {k: [(_f32_np(rng, lay.S, s) if k != "v" else np.abs(_f32_np(rng, lay.S, s))) for _ in range(world)]
            for k, s in (("p", 0.02), ("m", 1e-4), ("v", 1e-4), ("g", 1e-3))}
    dev = {k: [Guarded(lay.S, torch.float32, int(rng.integers(0, 4))) for _ in range(world)] for k in arrs}
    for k in arrs:
        for r in range(world):
            dev[k][r].set(arrs[k][r])
    zr.zr_adam_shard_step(zl, rank, *[[d.view for d in dev[k]] for k in ("p", "m", "v", "g")], hp)
    torch.cuda.synchronize()
    for r in range(world):
        p, m, v = arrs["p"][r].copy(), arrs["m"][r].copy(), arrs["v"][r].copy()
        if rank in (-1, r):
            oracle.adamw(p, m, v, arrs["g"][r], hp)
        for k, want in (("p", p), ("m", m), ("v", v), ("g", arrs["g"][r])):
            dev[k][r].check_guards()
            _assert_same(dev[k][r].bits(), want, f"adam {k} rank {r}")


@pytest.mark.parametrize("world,seed,n,hi,B", CASES)
def test_gather_cast_bf16(zr, world, seed, n, hi, B):
    rng, numel, lay = _case(world, seed, n, hi, B)
    zl = zr.Layout(numel, world, B)
    shards = [_f32_np(rng, lay.S, 0.05) for _ in range(world)]
    shards[0][0] = np.float32(3.0e38)  # near the top of the bf16 range
    dev = [Guarded(lay.S, torch.float32, int(rng.integers(0, 4))) for _ in range(world)]
    for d, s in zip(dev, shards):
        d.set(s)
    out = Guarded(lay.P, torch.bfloat16, int(rng.integers(0, 8)))
    zr.zr_gather_cast_bf16(zl, [d.view for d in dev], out.view)
    torch.cuda.synchronize()
    out.check_guards()
    _assert_same(out.bits(), oracle.gather_cast_bf16(lay, shards), "gather-cast", dtype="bf16")


@pytest.mark.parametrize("n", [1, 7, 255, 256, 257, 4099, 100_003])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_grad_accumulate(zr, n, dtype):
    rng = np.random.default_rng(n)
    es = 2 if dtype == "bf16" else 4
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    acc = _f32_np(rng, n, 1e-3)
    g = _bf16_np(rng, n, 1e-3) if dtype == "bf16" else _f32_np(rng, n, 1e-3)
    for pa in range(4):
        A = Guarded(n, torch.float32, pa)
        A.set(acc)
        G = Guarded(n, tdt, int(rng.integers(0, 16 // es)))
        G.set(g)
        zr.zr_grad_accumulate(A.view, G.view)
        torch.cuda.synchronize()
        want = acc.copy()
        oracle.grad_accumulate(want, g)
        A.check_guards()
        _assert_same(A.bits(), want, "accumulate")


def test_empty_and_degenerate_calls(zr):
    zr.zr_grad_accumulate(torch.zeros(0, device="cuda"), torch.zeros(0, device="cuda"))
    lay = zr.Layout([], 4, 10)
    zr.zr_gather_cast_bf16(lay, [torch.zeros(1, device="cuda")] * 4, torch.zeros(1, dtype=torch.bfloat16, device="cuda"))
    with pytest.raises(zr.ZrError):  # no bucket 0 in an empty layout
        zr.zr_reduce_scatter_avg(lay, 0, [torch.zeros(1, device="cuda")] * 4, 0.25, [torch.zeros(1, device="cuda")] * 4)
    # world = 1 with one element: identity average, one padding-free partition
    one = zr.Layout([1], 1, 1)
    x = torch.tensor([1.5], dtype=torch.bfloat16, device="cuda")
    g = torch.zeros(1, device="cuda")
    zr.zr_reduce_scatter_avg(one, 0, [x], 1.0, [g])
    torch.cuda.synchronize()
    assert g.item() == 1.5


@pytest.mark.parametrize("world,dtype,phases", [(16, "bf16", "same"), (16, "bf16", "mixed"), (8, "fp32", "same"),
                                                 (4, "bf16", "mixed"), (3, "bf16", "same")])
def test_fused_medium_many_pipeline_tiles(zr, world, dtype, phases):
    """A few million elements: most tiles go through the shared-memory pipeline; every element compared."""
    rng = np.random.default_rng(world * 7 + len(phases))
    numel = [int(x) for x in rng.integers(50_000, 400_000, 12)] + [1, 7, 1000]
    B = 1_000_000
    lay = oracle.layout(numel, world, B)
    zl = zr.Layout(numel, world, B)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    es = 2 if dtype == "bf16" else 4
    scale = float(np.float32(1.0 / world))
    hp = W.AdamW(step=5)

    def mk(arrs):
        out = []
        for r in range(world):
            g = Guarded(lay.S, torch.float32, 0 if phases == "same" else int(rng.integers(0, 4)))
            g.set(arrs[r])
            out.append(g)
        return out

    flat = lambda std, absval=False: np.concatenate([_f32_np(rng, lay.T, std), np.zeros(lay.P - lay.T, np.float32)])
    p_np = np.split(flat(0.02), world)
    m_np = np.split(np.abs(flat(1e-4)), world)
    v_np = np.split(np.abs(flat(1e-4)), world)
    P_, M_, V_ = mk(p_np), mk(m_np), mk(v_np)
    param = Guarded(lay.P, torch.bfloat16, int(rng.integers(0, 8)))
    want = [[a.copy() for a in p_np], [a.copy() for a in m_np], [a.copy() for a in v_np]]
    want_param = np.full(lay.P, CANARY16, np.uint16)
    for b in range(lay.n_buckets):
        vals, dev = _buckets_on_device(rng, lay, b, world, tdt, es)
        zr.zr_rs_adam_fused(zl, b, [d.view for d in dev], scale, [x.view for x in P_], [x.view for x in M_],
                            [x.view for x in V_], hp, param.view)
        oracle.rs_adam_fused(lay, b, vals, scale, want[0], want[1], want[2], hp, want_param)
        torch.cuda.synchronize()
    for r in range(world):
        for got, w, nm in ((P_, want[0], "p"), (M_, want[1], "m"), (V_, want[2], "v")):
            got[r].check_guards()
            _assert_same(got[r].bits(), w[r], f"{nm} rank {r}")
    param.check_guards()
    _assert_same(param.bits(), want_param, "param", dtype="bf16")


@pytest.mark.parametrize("world,seed,n,hi,B", [c for c in CASES if c[0] <= 32] + [(16, 9, 30, 300_000, 2_000_000)])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("phases", ["same", "mixed"])
def test_step_direct(zr, world, seed, n, hi, B, dtype, phases):
    """Steps 1-4 from per-parameter tensors without a bucket buffer == oracle pack + fused step."""
    rng, numel, lay = _case(world, seed, n, hi, B)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    es = 2 if dtype == "bf16" else 4
    zl = zr.Layout(numel, world, B)
    scale = float(np.float32(1.0 / world))
    hp = W.AdamW(step=int(rng.integers(1, 20)))
    grads_np = [[(_bf16_np(rng, m) if dtype == "bf16" else _f32_np(rng, m, 1e-2)) for m in numel]
                for _ in range(world)]
    grads_dev, keep = [], []
    for k in range(world):
        row = []
        if k % 2 == 0:
            flat = np.concatenate(grads_np[k])
            g = Guarded(len(flat), tdt, int(rng.integers(0, 16 // es)))
            g.set(flat)
            keep.append(g)
            pos = 0
            for m in numel:
                row.append(g.view[pos:pos + m])
                pos += m
        else:
            for i, m in enumerate(numel):
                g = Guarded(m, tdt, int(rng.integers(0, 16 // es)))
                g.set(grads_np[k][i])
                keep.append(g)
                row.append(g.view)
        grads_dev.append(row)
    plan = zr.DirectPlan(zl, grads_dev)

    def mk(arrs):
        out = []
        for r in range(world):
            gg = Guarded(lay.S, torch.float32, 0 if phases == "same" else int(rng.integers(0, 4)))
            gg.set(arrs[r])
            out.append(gg)
        return out

    flat = lambda std: np.concatenate([_f32_np(rng, lay.T, std), np.zeros(lay.P - lay.T, np.float32)])
    p_np = np.split(flat(0.02), world)
    m_np = np.split(np.abs(flat(1e-4)), world)
    v_np = np.split(np.abs(flat(1e-4)), world)
    P_, M_, V_ = mk(p_np), mk(m_np), mk(v_np)
    G_ = mk([np.full(lay.S, np.float32(np.nan), np.float32) for _ in range(world)])
    param = Guarded(lay.P, torch.bfloat16, int(rng.integers(0, 8)))
    want = [[a.copy() for a in p_np], [a.copy() for a in m_np], [a.copy() for a in v_np],
            [np.full(lay.S, np.float32(np.nan), np.float32) for _ in range(world)]]
    want_param = np.full(lay.P, CANARY16, np.uint16)
    for b in range(lay.n_buckets):
        zr.zr_step_direct(plan, b, scale, [x.view for x in P_], [x.view for x in M_], [x.view for x in V_], hp,
                          param.view, [x.view for x in G_])
        bucket = oracle.bucket_pack(lay, b, grads_np)
        oracle.rs_adam_fused(lay, b, bucket, scale, want[0], want[1], want[2], hp, want_param, want[3])
    torch.cuda.synchronize()
    for r in range(world):
        for got, w, nm in ((P_, want[0], "p"), (M_, want[1], "m"), (V_, want[2], "v"), (G_, want[3], "g")):
            got[r].check_guards()
            _assert_same(got[r].bits(), w[r], f"direct {nm} rank {r}")
    param.check_guards()
    _assert_same(param.bits(), want_param, "direct param", dtype="bf16")
    for g in keep:
        g.check_guards()
    plan.close()


def test_determinism(zr):
    rng, numel, lay = _case(16, 5, 40, 3000, 30000)
    zl = zr.Layout(numel, 16, 30000)
    outs = []
    for _ in range(2):
        p = [torch.full((lay.S,), 0.01, device="cuda") for _ in range(16)]
        m = [torch.zeros(lay.S, device="cuda") for _ in range(16)]
        v = [torch.zeros(lay.S, device="cuda") for _ in range(16)]
        param = torch.zeros(lay.P, dtype=torch.bfloat16, device="cuda")
        gen = torch.Generator(device="cuda").manual_seed(7)
        for b in range(lay.n_buckets):
            _, nb = lay.bucket(b)
            x = [torch.randn(nb, generator=gen, device="cuda").to(torch.bfloat16) for _ in range(16)]
            zr.zr_rs_adam_fused(zl, b, x, 1 / 16, p, m, v, W.AdamW(), param)
        torch.cuda.synchronize()
        outs.append((torch.cat(p).clone(), param.clone()))
    assert torch.equal(outs[0][0].view(torch.int32), outs[1][0].view(torch.int32))
    assert torch.equal(outs[0][1].view(torch.int16), outs[1][1].view(torch.int16))


# ----------------------------------------------------------------------------
# Whole workloads
# ----------------------------------------------------------------------------

def test_tiny_workload_end_to_end(zr):
    """The 7-parameter workload through the engine (pack + fused per bucket) == the oracle, every element."""
    from zero_partition_aware_gb300.engine import DPGroup
    wl = W.WORKLOADS["tiny"]
    lay = oracle.layout(list(wl.numel), wl.world, wl.bucket)
    inp = W.draw_inputs(wl, "cpu", seed=0)
    grp = DPGroup(list(wl.numel), wl.world, wl.bucket)
    grp.load_flat(inp["master"].cuda(), inp["m"].cuda(), inp["v"].cuda())
    grads_dev = [[t for t in torch.split(inp["grads"][k][0].cuda(), list(wl.numel))] for k in range(wl.world)]
    grp.step(grp.grad_table(grads_dev), wl.adam)
    torch.cuda.synchronize()
    grads = [oracle.params_from_flat(lay, W.bf16_bits(inp["grads"][k][0])) for k in range(wl.world)]
    p = oracle.shards_from_flat(lay, inp["master"].numpy())
    m = oracle.shards_from_flat(lay, inp["m"].numpy())
    v = oracle.shards_from_flat(lay, inp["v"].numpy())
    param = np.zeros(lay.P, np.uint16)
    for b in range(lay.n_buckets):
        oracle.rs_adam_fused(lay, b, oracle.bucket_pack(lay, b, grads), grp.scale, p, m, v, wl.adam, param)
    for r in range(wl.world):
        _assert_same(_bits(grp.master[r]), p[r], f"master {r}")
        _assert_same(_bits(grp.m[r]), m[r], f"m {r}")
        _assert_same(_bits(grp.v[r]), v[r], f"v {r}")
    _assert_same(_bits(grp.param[: lay.P]), param, "param", dtype="bf16")
