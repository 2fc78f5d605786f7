"""Pins of the oracle's global gradient check and the step it steers.

After every bucket has been averaged into the partitions and before
optimizer.step() ("Megatron-LM 分布式训练（四）" §"跨 model-parallel 的梯度收尾": DP
sync, then the gradient fix-ups, then the step; "DeepSpeed ZeRO 通信优化深度解析"
§六: fp16 safety), the check takes the global L2 norm of the averaged
gradient over every rank's partition, counts the elements whose fp32 square
is not finite (an overflowed step is skipped) and forms the clip
coefficient min(1, max_norm / (norm + 1e-6)). Pinned here:
- the sum of squares against the exact rational sum, within the bound of
  n double roundings, and equal to it where every partial sum is exact;
- the norm against numpy's norm of the concatenated gradient;
- the coefficient against torch.nn.utils.clip_grad_norm_ on the same
  gradient (a small norm, so that the 1e-6 term shows);
- the overflow count at the edge of the fp32 square's range;
- the clipped step: skip leaves everything unchanged; coef = 1 is the plain
  AdamW followed by the bf16 cast; coef = 1/2 on even integer gradients is
  AdamW on the halved gradients; the whole two-pass step with max_norm = 0
  equals the fused per-bucket step bit for bit.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from zero_partition_aware_gb300 import workloads as W


def _shards(rng, world, S, scale=1e-3):
    return [(rng.standard_normal(S) * scale).astype(np.float32) for _ in range(world)]


@pytest.mark.parametrize("world,S,seed", [(1, 1, 0), (2, 7, 1), (4, 1000, 2), (8, 333, 3)])
def test_sumsq_within_double_rounding_of_the_exact_sum(world, S, seed):
    rng = np.random.default_rng(seed)
    g = _shards(rng, world, S)
    # a spread of magnitudes: fp32 subnormals, large and exact zeros
    g[0][::5] *= np.float32(1e-36)
    g[-1][::7] = np.float32(3e18)
    g[-1][1::9] = 0
    st = oracle.grad_check(g, 0.0)
    exact = sum(Fraction(float(x)) ** 2 for a in g for x in a)
    n = world * S
    assert abs(Fraction(st.sumsq) - exact) <= exact * Fraction(n, 2 ** 53)
    assert st.nonfinite == 0 and not st.skip and st.coef == 1.0


def test_sumsq_exact_on_integers():
    rng = np.random.default_rng(5)
    g = [rng.integers(-1000, 1001, 4000).astype(np.float32) for _ in range(4)]
    st = oracle.grad_check(g, 0.0)
    assert st.sumsq == float(sum(int(x) ** 2 for a in g for x in a))
    # 3-4-5: a norm that is exact in every format
    st = oracle.grad_check([np.array([3.0], np.float32), np.array([4.0], np.float32)], 0.0)
    assert st.norm == 5.0


@pytest.mark.parametrize("world,S", [(3, 50), (16, 2048)])
def test_norm_matches_numpy(world, S):
    rng = np.random.default_rng(world)
    g = _shards(rng, world, S, 1e-2)
    st = oracle.grad_check(g, 0.0)
    ref = np.linalg.norm(np.concatenate(g).astype(np.float64))
    assert abs(st.norm - ref) <= 1e-13 * ref


@pytest.mark.parametrize("max_norm_frac", [0.001, 0.3, 0.999, 1.0, 1.5])
def test_coef_matches_torch_clip_grad_norm(max_norm_frac):
    rng = np.random.default_rng(11)
    g = _shards(rng, 4, 300, 1e-5)  # norm about 3.5e-4: the 1e-6 term moves the coefficient by ~3e-3
    flat = np.concatenate(g).astype(np.float64)
    norm = float(np.linalg.norm(flat))
    max_norm = float(np.float32(norm * max_norm_frac))
    st = oracle.grad_check(g, max_norm)
    t = torch.nn.Parameter(torch.ones(flat.size, dtype=torch.float64))
    t.grad = torch.from_numpy(flat.copy())
    total = float(torch.nn.utils.clip_grad_norm_([t], max_norm))
    assert abs(total - st.norm) <= 1e-12 * st.norm
    i = int(np.argmax(np.abs(flat)))
    coef_t = float(t.grad[i]) / flat[i]
    assert abs(st.coef - coef_t) <= 2.0 ** -23 * coef_t
    if max_norm >= norm + 1e-6:
        assert st.coef == 1.0


def test_clipped_norm_is_max_norm():
    rng = np.random.default_rng(12)
    g = _shards(rng, 8, 1000, 1e-2)
    st = oracle.grad_check(g, 0.05)
    assert st.coef < 1.0
    clipped = np.concatenate([a * np.float32(st.coef) for a in g]).astype(np.float64)
    target = 0.05 * st.norm / (st.norm + 1e-6)
    assert abs(np.linalg.norm(clipped) - target) <= 1e-6 * target


def test_no_clipping_when_max_norm_not_positive():
    rng = np.random.default_rng(13)
    g = _shards(rng, 2, 100, 10.0)
    for mn in (0.0, -1.0):
        assert oracle.grad_check(g, mn).coef == 1.0


def test_overflow_count_at_the_edge_of_the_fp32_square():
    g = [np.zeros(16, np.float32) for _ in range(3)]
    g[0][1] = np.inf
    g[1][2] = -np.inf
    g[2][3] = np.nan
    g[2][4] = np.float32(2.0 ** 64)          # square 2^128 overflows fp32
    g[1][5] = np.float32(-(2.0 ** 64))
    g[0][6] = np.float32(2.0 ** 63)          # square 2^126 is finite
    g[0][7] = np.float32(1.8446743e19)       # just below 2^64: square rounds to FLT_MAX or below
    big = np.float32(1.8446743e19)
    sq_finite = np.isfinite(np.float32(big) * np.float32(big))
    st = oracle.grad_check(g, 1.0)
    assert st.nonfinite == 5 + (0 if sq_finite else 1)
    assert st.skip and st.coef == 1.0
    g = [np.zeros(16, np.float32) for _ in range(3)]
    g[0][6] = np.float32(2.0 ** 63)
    st = oracle.grad_check(g, 0.0)
    assert st.nonfinite == 0 and not st.skip and st.sumsq == 2.0 ** 126


def _state(rng, lay):
    def flat(std, absval=False):
        a = np.concatenate([(rng.standard_normal(lay.T) * std).astype(np.float32), np.zeros(lay.P - lay.T, np.float32)])
        return np.abs(a) if absval else a
    return (oracle.shards_from_flat(lay, flat(0.02)), oracle.shards_from_flat(lay, flat(1e-4, True)),
            oracle.shards_from_flat(lay, flat(1e-4, True)))


def _copy(arrs):
    return [a.copy() for a in arrs]


@pytest.mark.parametrize("world,numel", [(4, [1000, 5661, 4096, 8385, 10, 6144, 777]), (3, [5, 7, 1])])
def test_skip_changes_nothing(world, numel):
    rng = np.random.default_rng(21)
    lay = oracle.layout(numel, world, 8192)
    p, m, v = _state(rng, lay)
    g = _shards(rng, world, lay.S)
    g[0][0] = np.nan
    param = np.full(lay.P, 0x1234, np.uint16)
    p0, m0, v0 = _copy(p), _copy(m), _copy(v)
    st = oracle.grad_check(g, 1.0)
    oracle.adam_clip_step(lay, p, m, v, g, W.AdamW(step=3), st.coef, st.skip, param)
    assert (param == 0x1234).all()
    for a, b in zip(p + m + v, p0 + m0 + v0):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("world,numel", [(4, [1000, 5661, 4096, 8385, 10, 6144, 777]), (5, [3, 9, 11])])
def test_coef_one_is_adamw_then_cast(world, numel):
    rng = np.random.default_rng(22)
    lay = oracle.layout(numel, world, 8192)
    p, m, v = _state(rng, lay)
    g = _shards(rng, world, lay.S)
    hp = W.AdamW(step=4)
    rp, rm, rv = _copy(p), _copy(m), _copy(v)
    for r in range(world):
        oracle.adamw(rp[r], rm[r], rv[r], g[r], hp)
    param = np.zeros(lay.P, np.uint16)
    oracle.adam_clip_step(lay, p, m, v, g, hp, 1.0, False, param)
    assert np.array_equal(param, oracle.gather_cast_bf16(lay, rp))
    for a, b in zip(p + m + v, rp + rm + rv):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_half_coef_on_even_integers_is_adamw_on_halved_grads():
    rng = np.random.default_rng(23)
    lay = oracle.layout([300, 200, 501], 4, 600)
    p, m, v = _state(rng, lay)
    g = [(rng.integers(-50, 51, lay.S) * 2).astype(np.float32) for _ in range(lay.world)]
    hp = W.AdamW(step=2)
    rp, rm, rv = _copy(p), _copy(m), _copy(v)
    for r in range(lay.world):
        oracle.adamw(rp[r], rm[r], rv[r], (g[r] // 2).astype(np.float32), hp)
    oracle.adam_clip_step(lay, p, m, v, g, hp, 0.5, False, None)
    for a, b in zip(p + m + v, rp + rm + rv):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("world,seed,n,hi,B", [(4, 0, 9, 3000, 5000), (8, 1, 30, 2000, 9000), (3, 2, 5, 100, 1)])
def test_two_pass_step_without_clipping_equals_the_fused_step(world, seed, n, hi, B):
    rng = np.random.default_rng(seed)
    numel = W.random_numels(rng, n, 1, hi)
    lay = oracle.layout(numel, world, B)
    grads = [[W.bf16_bits(torch.from_numpy((rng.standard_normal(k) * 1e-2).astype(np.float32)).to(torch.bfloat16))
              for k in numel] for _ in range(world)]
    hp = W.AdamW(step=5)
    scale = float(np.float32(1.0 / world))
    p, m, v = _state(rng, lay)
    fp, fm, fv = _copy(p), _copy(m), _copy(v)
    fparam = np.zeros(lay.P, np.uint16)
    g = [np.zeros(lay.S, np.float32) for _ in range(world)]
    for b in range(lay.n_buckets):
        bucket = oracle.bucket_pack(lay, b, grads)
        oracle.rs_adam_fused(lay, b, bucket, scale, fp, fm, fv, hp, fparam)
        oracle.reduce_scatter_avg(lay, b, bucket, scale, g)
    st = oracle.grad_check(g, 0.0)
    assert st.coef == 1.0 and not st.skip
    param = np.zeros(lay.P, np.uint16)
    oracle.adam_clip_step(lay, p, m, v, g, hp, st.coef, st.skip, param)
    assert np.array_equal(param, fparam)
    for a, b in zip(p + m + v, fp + fm + fv):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
