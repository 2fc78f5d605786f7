"""Pins of the oracle's fp16 gradients and the all-reduce path's pre/post scaling.

The all-reduce path that runs when reduce_scatter is off keeps fp16 training's
pre- and post-scaling: gradient_predivide_factor f divides before the
reduction and postscale_gradients multiplies by f/N after it
("DeepSpeed ZeRO 通信优化深度解析" §三.2 and §六). Pinned here:
- the binary16 decode against numpy's float16 -> float32 widening, for all 65,536
  bit patterns;
- fp16 gradients average exactly as the same values given as fp32 (widening is
  exact, so the sums cannot differ);
- postscale 1 (f = N) is the plain all-reduce average, equal to the
  reduce-scatter's result;
- with integer-valued gradients every partial sum is exact, so any power-of-two
  split of 1/N between the predivide and the postscale gives the exact mean.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from zero_partition_aware_gb300 import workloads as W


def test_f16_decode_every_bit_pattern():
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16).view(np.float16)
    got = oracle.f16_to_f32(h)
    ref = h.astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


@pytest.mark.parametrize("world,seed", [(2, 0), (4, 1), (8, 2), (5, 3)])
def test_fp16_averages_as_its_fp32_widening(world, seed):
    rng = np.random.default_rng(seed)
    numel = W.random_numels(rng, 12, 1, 3000)
    lay = oracle.layout(numel, world, 4000)
    g16 = [[(rng.standard_normal(k) * 3e-3).astype(np.float16) for k in numel] for _ in range(world)]
    g32 = [[a.astype(np.float32) for a in row] for row in g16]
    s = float(np.float32(1.0 / world))
    for b in range(lay.n_buckets):
        x16, x32 = oracle.bucket_pack(lay, b, g16), oracle.bucket_pack(lay, b, g32)
        a16 = [np.full(lay.S, np.nan, np.float32) for _ in range(world)]
        a32 = [np.full(lay.S, np.nan, np.float32) for _ in range(world)]
        oracle.reduce_scatter_avg(lay, b, x16, s, a16)
        oracle.reduce_scatter_avg(lay, b, x32, s, a32)
        for r in range(world):
            assert np.array_equal(a16[r].view(np.uint32), a32[r].view(np.uint32))
        ar16 = oracle.allreduce_avg(world, x16, s)
        ar32 = oracle.allreduce_avg(world, x32, s)
        assert np.array_equal(ar16[0].view(np.uint32), ar32[0].view(np.uint32))


@pytest.mark.parametrize("dt", [np.uint16, np.float16, np.float32])
def test_postscale_one_is_the_reduce_scatter_average(dt):
    rng = np.random.default_rng(7)
    world = 6
    numel = W.random_numels(rng, 10, 1, 2000)
    lay = oracle.layout(numel, world, 3000)
    raw = [[(rng.standard_normal(k) * 1e-2).astype(np.float32) for k in numel] for _ in range(world)]
    if dt == np.uint16:
        g = [[oracle.f32_to_bf16(a) for a in row] for row in raw]
    else:
        g = [[a.astype(dt) for a in row] for row in raw]
    s = float(np.float32(1.0 / world))
    for b in range(lay.n_buckets):
        x = oracle.bucket_pack(lay, b, g)
        sh = [np.full(lay.S, np.nan, np.float32) for _ in range(world)]
        oracle.reduce_scatter_avg(lay, b, x, s, sh)
        full = np.concatenate(sh)[lay.flat_map(b)]
        for out in oracle.allreduce_avg(world, x, s, 1.0):
            assert np.array_equal(out.view(np.uint32), full.view(np.uint32))


@pytest.mark.parametrize("world,f", [(8, 1), (8, 2), (8, 8), (16, 4), (4, 2)])
@pytest.mark.parametrize("dt", [np.float16, np.uint16])
def test_predivide_split_gives_the_exact_mean_on_integer_grads(world, f, dt):
    rng = np.random.default_rng(world * 10 + f)
    nb = 3000
    ints = [rng.integers(-64, 65, nb) for _ in range(world)]
    if dt == np.float16:
        x = [a.astype(np.float16) for a in ints]
    else:
        x = [oracle.f32_to_bf16(a.astype(np.float32)) for a in ints]
    out = oracle.allreduce_avg(world, x, float(np.float32(1.0 / f)), float(np.float32(f / world)))[0]
    exact = [Fraction(int(sum(int(a[e]) for a in ints)), world) for e in range(nb)]
    assert all(Fraction(float(out[e])) == exact[e] for e in range(nb))
