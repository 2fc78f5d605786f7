"""Pins of the oracle's arithmetic (CPU only).

Each oracle function is tied to something other than itself: exact rational
sums within the fp32 error bound, closed forms, identities the pages state
(all-reduce = reduce-scatter + all-gather), special cases that reduce to a
library routine (torch's bf16 cast, numpy's fp32 add, torch.optim.AdamW), and
cases whose result is known exactly (integer gradients, rank-order tie).
Sources: "DeepSpeed ZeRO 通信优化深度解析" §二, §三.2, §六; "Megatron-LM 分布式训练
（四）" §"通信模式", §"四步接力"; "07. 大规模训练时通信瓶颈在哪里？" §"三种原语",
§"Ring=RS+AG".
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import brute
from zero_partition_aware_gb300 import workloads as W

U = 2.0 ** -24  # unit roundoff of binary32


def _bits(t):
    return W.bf16_bits(t)


def _rand_bf16(rng, shape, std=1e-2):
    x = torch.from_numpy(rng.standard_normal(shape).astype(np.float32) * np.float32(std))
    return _bits(x.to(torch.bfloat16))


# ----------------------------------------------------------------------------
# bf16 conversions: the library routine is torch's CPU cast (round to nearest even)
# ----------------------------------------------------------------------------

def test_cast_matches_torch_round_to_nearest_even():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(100_000).astype(np.float32) * 0.02,
        (rng.standard_normal(20_000) * 1e30).astype(np.float32),
        np.array([0.0, -0.0, 1.0, -1.0, np.inf, -np.inf, 3.4e38, -3.4e38,
                  1e-40, -1e-40, 1.0000001, 1.00390625, 1.01171875, 65504.0], np.float32),
    ])
    # exact ties: bf16 midpoints (low 16 bits = 0x8000), odd and even kept bit
    ties = (rng.integers(0, 1 << 15, 5000, dtype=np.uint32) << 16 | 0x8000).astype(np.uint32)
    x = np.concatenate([x, ties.view(np.float32)])
    x = x[np.isfinite(x) | np.isinf(x)]
    got = oracle.f32_to_bf16(x)
    want = _bits(torch.from_numpy(x).to(torch.bfloat16))
    assert np.array_equal(got, want)


def test_cast_nan_is_quiet_nan():
    x = np.array([np.nan, -np.nan], np.float32)
    got = oracle.f32_to_bf16(x)
    assert all(((g >> 7) & 0xFF) == 0xFF and (g & 0x7F) != 0 for g in got)


def test_widening_matches_torch():
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    t = W.from_bf16_bits(bits).float().numpy()
    got = oracle.bf16_to_f32(bits)
    fin = np.isfinite(t)
    assert np.array_equal(got[fin].view(np.uint32), t[fin].view(np.uint32))
    assert np.all(np.isnan(got[~fin]) == np.isnan(t[~fin]))


# ----------------------------------------------------------------------------
# Averaging (reduce-scatter / all-reduce with predivide)
# ----------------------------------------------------------------------------

def _tiny_case(seed, world, numel, B, dtype=np.uint16):
    rng = np.random.default_rng(seed)
    lay = oracle.layout(numel, world, B)
    grads = []
    for k in range(world):
        if dtype == np.uint16:
            grads.append([_rand_bf16(rng, n) for n in numel])
        else:
            grads.append([rng.standard_normal(n).astype(np.float32) * np.float32(1e-2)
                          for n in numel])
    return lay, grads


def _rs_all(lay, grads, scale):
    shards = [np.full(lay.S, np.nan, np.float32) for _ in range(lay.world)]
    for b in range(lay.n_buckets):
        bucket = oracle.bucket_pack(lay, b, grads)
        oracle.reduce_scatter_avg(lay, b, bucket, scale, shards)
    return shards


@pytest.mark.parametrize("world", [1, 2, 3, 4, 8, 16])
def test_rs_equals_exact_mean_within_error_bound(world):
    numel = [37, 1, 300, 129, 64]
    lay, grads = _tiny_case(world, world, numel, 200)
    scale = np.float32(1.0 / world)
    shards = _rs_all(lay, grads, float(scale))
    flat = np.concatenate(shards)
    for f in range(lay.P):
        if f < lay.T:
            i = int(np.searchsorted(lay.offset, f, side="right") - 1)
            e = f - int(lay.offset[i])
            vals = [brute.bf16_value(int(grads[k][i][e])) for k in range(world)]
        else:
            vals = [Fraction(0)] * world
        exact = sum(vals, Fraction(0)) * Fraction(float(scale))
        # bound for fl(x_k*s) summed left to right: gamma_N * sum |x_k s|
        mag = float(sum(abs(v) for v in vals) * Fraction(float(scale)))
        gamma = world * U / (1 - world * U)
        assert abs(float(flat[f]) - float(exact)) <= gamma * mag + 1e-45


def test_rs_rank_order_is_observable_and_fixed():
    """N=4, s=1/4 exact. Replica values 2^26, 4, -2^26, 0 give terms 2^24, 1, -2^24, 0.
    In rank order: (0 + 2^24) + 1 = 2^24 + 1 rounds (tie, to even) to 2^24; then - 2^24
    gives 0; + 0 = 0. Any other order that adds 1 to -2^24 first would give 1."""
    vals = np.array([2.0 ** 26, 4.0, -(2.0 ** 26), 0.0], np.float32)
    bucket = [_bits(torch.tensor([v]).to(torch.bfloat16)) for v in vals]
    out = oracle.allreduce_avg(4, bucket, 0.25)
    assert out[0][0] == 0.0
    rev = oracle.allreduce_avg(4, bucket[::-1], 0.25)
    assert rev[0][0] == 1.0


def test_rs_concat_equals_allreduce_bitwise():
    """all-reduce = reduce-scatter + all-gather ("Ring=RS+AG"; "通信模式")."""
    numel = [1000, 5661, 4096, 8385, 10, 6144, 777]
    lay, grads = _tiny_case(7, 4, numel, 8192)
    shards = _rs_all(lay, grads, 0.25)
    flat_rs = np.concatenate(shards)
    for b in range(lay.n_buckets):
        start, nb = lay.bucket(b)
        bucket = oracle.bucket_pack(lay, b, grads)
        ar = oracle.allreduce_avg(4, bucket, 0.25)
        for k in range(4):
            assert np.array_equal(ar[k].view(np.uint32), flat_rs[start:start + nb].view(np.uint32))


def test_rs_independent_of_bucket_size():
    numel = [513, 77, 2000, 1, 1024, 9, 300]
    base = None
    for B in [1, 100, 777, 2048, 10 ** 6]:
        lay, grads = _tiny_case(11, 8, numel, B)
        flat = np.concatenate(_rs_all(lay, grads, 0.125)).view(np.uint32)
        if base is None:
            base = flat
        assert np.array_equal(flat, base)


def test_integer_grads_average_exactly():
    """Integer grads in [-8, 8], N=16: every partial sum is an exact multiple of 1/16."""
    wl = W.replace(W.WORKLOADS["irregular_10k"], numel=(1000, 333, 4097, 1, 2500))
    lay = oracle.layout(list(wl.numel), 16, 3000)
    inp = W.draw_inputs(wl, "cpu", seed=3)
    grads = [oracle.params_from_flat(lay, _bits(inp["grads"][k][0])) for k in range(16)]
    flat = np.concatenate(_rs_all(lay, grads, 1.0 / 16))
    ints = np.stack([inp["grads"][k][0].float().numpy() for k in range(16)]).astype(np.int64)
    exact = ints.sum(axis=0) / 16.0
    assert np.array_equal(flat[: lay.T], exact.astype(np.float32))
    assert np.all(flat[lay.T:] == 0)


def test_world_one_is_identity():
    lay, grads = _tiny_case(5, 1, [100, 200, 3], 64)
    flat = np.concatenate(_rs_all(lay, grads, 1.0))
    want = oracle.bf16_to_f32(np.concatenate(grads[0]))
    assert np.array_equal(flat[: lay.T].view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("world", [2, 4, 8, 16, 32])
def test_equal_replicas_average_to_the_replica(world):
    rng = np.random.default_rng(world)
    numel = [123, 456]
    g = [_rand_bf16(rng, n) for n in numel]
    lay = oracle.layout(numel, world, 10 ** 6)
    flat = np.concatenate(_rs_all(lay, [g] * world, 1.0 / world))
    want = oracle.bf16_to_f32(np.concatenate(g))
    assert np.array_equal(flat[: lay.T].view(np.uint32), want.view(np.uint32))


def test_fp32_replicas_average():
    lay, grads = _tiny_case(9, 4, [50, 60, 70], 64, dtype=np.float32)
    flat = np.concatenate(_rs_all(lay, grads, 0.25))
    x = np.stack([np.concatenate(g) for g in grads]).astype(np.float64)
    exact = x.sum(axis=0) * 0.25
    mag = np.abs(x).sum(axis=0) * 0.25
    gamma = 4 * U / (1 - 4 * U)
    assert np.all(np.abs(flat[: lay.T] - exact) <= gamma * mag + 1e-45)


# ----------------------------------------------------------------------------
# Packing and accumulation
# ----------------------------------------------------------------------------

def test_pack_places_params_by_flat_offset():
    numel = [1000, 5661, 4096, 8385, 10, 6144, 777]
    lay, grads = _tiny_case(2, 4, numel, 8192)
    for k in range(4):
        flat = np.concatenate(grads[k] + [np.zeros(lay.P - lay.T, np.uint16)])
        for b in range(lay.n_buckets):
            start, nb = lay.bucket(b)
            got = oracle.bucket_pack(lay, b, grads)[k]
            assert np.array_equal(got, flat[start:start + nb])


def test_grad_accumulate_matches_numpy_fp32_add():
    rng = np.random.default_rng(4)
    acc = rng.standard_normal(5000).astype(np.float32)
    mb = _rand_bf16(rng, 5000, 1e-3)
    want = acc + W.from_bf16_bits(mb).float().numpy()
    oracle.grad_accumulate(acc, mb)
    assert np.array_equal(acc.view(np.uint32), want.view(np.uint32))
    g32 = rng.standard_normal(5000).astype(np.float32)
    want2 = acc + g32
    oracle.grad_accumulate(acc, g32)
    assert np.array_equal(acc.view(np.uint32), want2.view(np.uint32))


# ----------------------------------------------------------------------------
# AdamW
# ----------------------------------------------------------------------------

def _f32(x):
    return float(np.float32(x))


HP = W.AdamW(lr=_f32(1e-3), beta1=_f32(0.9), beta2=_f32(0.999), eps=_f32(1e-8),
             weight_decay=_f32(0.01), step=1)


def test_adamw_closed_form_at_step_one():
    """t=1, m=v=0: m_hat = g and sqrt(v_hat) = |g|, so p1 = p0 (1 - lr wd) - lr g / (|g| + eps)."""
    rng = np.random.default_rng(0)
    n = 20000
    p = (rng.standard_normal(n) * 0.02).astype(np.float32)
    g = (rng.standard_normal(n) * 1e-2).astype(np.float32)
    g[:10] = np.float32(1e-9)  # |g| comparable to eps
    p0 = p.copy().astype(np.float64)
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    oracle.adamw(p, m, v, g, HP)
    lr, wd, eps = HP.lr, HP.weight_decay, HP.eps
    gd = g.astype(np.float64)
    want = p0 * (1 - lr * wd) - lr * gd / (np.abs(gd) + eps)
    assert np.all(np.abs(p - want) <= 1e-6 * (np.abs(p0) + lr))
    assert np.allclose(m, (1 - 0.9) * gd, rtol=1e-6)
    assert np.allclose(v, (1 - 0.999) * gd * gd, rtol=1e-4)


def test_adamw_zero_grad_is_pure_decay():
    n = 1000
    p = np.linspace(-1, 1, n, dtype=np.float32)
    p0 = p.copy()
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    oracle.adamw(p, m, v, np.zeros(n, np.float32), HP)
    decay = np.float32(1 - np.float64(HP.lr) * np.float64(HP.weight_decay))
    assert np.array_equal(p.view(np.uint32), (p0 * decay).view(np.uint32))
    assert np.all(m == 0) and np.all(v == 0)


@pytest.mark.parametrize("step", [1, 2, 10, 1000])
def test_adamw_matches_torch_optim(step):
    rng = np.random.default_rng(step)
    n = 4096
    p = (rng.standard_normal(n) * 0.02).astype(np.float32)
    g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    m = np.abs(rng.standard_normal(n) * 1e-4).astype(np.float32) if step > 1 else np.zeros(n, np.float32)
    v = np.abs(rng.standard_normal(n) * 1e-4).astype(np.float32) if step > 1 else np.zeros(n, np.float32)
    hp = W.AdamW(HP.lr, HP.beta1, HP.beta2, HP.eps, HP.weight_decay, step)
    tp = torch.nn.Parameter(torch.from_numpy(p.copy()))
    opt = torch.optim.AdamW([tp], lr=hp.lr, betas=(hp.beta1, hp.beta2), eps=hp.eps,
                            weight_decay=hp.weight_decay, foreach=False, fused=False)
    tp.grad = torch.from_numpy(g.copy())
    if step > 1:
        opt.state[tp] = {"step": torch.tensor(float(step - 1)),
                         "exp_avg": torch.from_numpy(m.copy()),
                         "exp_avg_sq": torch.from_numpy(v.copy())}
    opt.step()
    p_before, m_before, v_before = p.copy(), m.copy(), v.copy()
    oracle.adamw(p, m, v, g, hp)
    st = opt.state[tp]
    # relative to the operands' magnitude: p' = p*decay - update may cancel
    for mine, ref, before in ((p, tp.detach().numpy(), p_before),
                              (m, st["exp_avg"].numpy(), m_before),
                              (v, st["exp_avg_sq"].numpy(), v_before)):
        scale = np.maximum(np.abs(ref), np.abs(before))
        assert np.all(np.abs(mine - ref) <= 1e-6 * scale + 1e-12), np.max(np.abs(mine - ref))


def test_adamw_scalars():
    c = oracle.adamw_scalars(W.AdamW(HP.lr, HP.beta1, HP.beta2, HP.eps, HP.weight_decay, 10))
    b1, b2 = np.float64(HP.beta1), np.float64(HP.beta2)
    assert c[0] == np.float32(HP.beta1) and c[2] == np.float32(HP.beta2)
    assert c[1] == np.float32(1 - b1) and c[3] == np.float32(1 - b2)
    assert c[4] == np.float32(np.float64(HP.lr) / (1 - b1 ** 10))
    assert c[5] == np.float32(np.sqrt(1 - b2 ** 10))
    assert c[6] == np.float32(1 - np.float64(HP.lr) * np.float64(HP.weight_decay))
    assert c[7] == np.float32(HP.eps)


# ----------------------------------------------------------------------------
# Gather-cast and the fused step
# ----------------------------------------------------------------------------

def test_gather_cast_is_concatenation_then_cast():
    lay = oracle.layout([1000, 5661, 4096, 8385, 10, 6144, 777], 4, 8192)
    rng = np.random.default_rng(1)
    flat = (rng.standard_normal(lay.T) * 0.02).astype(np.float32)
    shards = oracle.shards_from_flat(lay, flat)
    out = oracle.gather_cast_bf16(lay, shards)
    want = _bits(torch.from_numpy(flat).to(torch.bfloat16))
    assert np.array_equal(out[: lay.T], want)
    assert np.all(out[lay.T:] == 0)


@pytest.mark.parametrize("name", ["tiny"])
def test_fused_equals_rs_then_adamw_then_gather(name):
    wl = W.WORKLOADS[name]
    lay = oracle.layout(list(wl.numel), wl.world, wl.bucket)
    inp = W.draw_inputs(wl, "cpu", seed=0)
    grads = [oracle.params_from_flat(lay, _bits(inp["grads"][k][0])) for k in range(wl.world)]
    scale = 1.0 / wl.world
    # unfused: RS over all buckets, AdamW per shard, then gather-cast
    p_a = oracle.shards_from_flat(lay, inp["master"].numpy())
    m_a = oracle.shards_from_flat(lay, inp["m"].numpy())
    v_a = oracle.shards_from_flat(lay, inp["v"].numpy())
    g_a = _rs_all(lay, grads, scale)
    for r in range(wl.world):
        oracle.adamw(p_a[r], m_a[r], v_a[r], g_a[r], wl.adam)
    param_a = oracle.gather_cast_bf16(lay, p_a)
    # fused, bucket by bucket
    p_b = oracle.shards_from_flat(lay, inp["master"].numpy())
    m_b = oracle.shards_from_flat(lay, inp["m"].numpy())
    v_b = oracle.shards_from_flat(lay, inp["v"].numpy())
    g_b = [np.full(lay.S, np.nan, np.float32) for _ in range(wl.world)]
    param_b = np.full(lay.P, 0xFFFF, np.uint16)
    for b in range(lay.n_buckets):
        bucket = oracle.bucket_pack(lay, b, grads)
        oracle.rs_adam_fused(lay, b, bucket, scale, p_b, m_b, v_b, wl.adam, param_b, g_b)
    for r in range(wl.world):
        for a, bb in ((p_a, p_b), (m_a, m_b), (v_a, v_b), (g_a, g_b)):
            assert np.array_equal(a[r].view(np.uint32), bb[r].view(np.uint32))
    assert np.array_equal(param_a, param_b)
    # padding master stays zero
    assert np.all(np.concatenate(p_b)[lay.T:] == 0)
