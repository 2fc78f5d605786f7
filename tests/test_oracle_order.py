"""Pins of the oracle's layout under an arrival order other than the flat one.

Backward produces grads from the last layers to the first, and each grad is
copied into the IPG bucket as soon as it is produced ("DeepSpeed ZeRO 通信优化深度解析"
§四). The flat layout and the partitions stay those of the flat order; only the
bucket walk follows the arrival order. Pinned here:
- the flat order gives exactly the layout of zro_layout (pinned elsewhere);
- the bucket walk's defining properties under any order;
- the runs' defining properties: together they cover every bucket position once,
  each maps bucket positions to flat positions as the bucket's content does,
  and no two consecutive runs could have been merged;
- the averaged gradient and the optimizer step of an element do not depend on
  which bucket, or where in it, the element travelled: the final master, m, v
  and bf16 params equal those of the flat order bit for bit.
"""
import numpy as np
import pytest

import oracle
from zero_partition_aware_gb300 import workloads as W


def _orders(rng, n):
    yield "reverse", list(range(n - 1, -1, -1))
    yield "random", [int(x) for x in rng.permutation(n)]
    # interleaved layers: pairs swapped (weights and biases arriving bias first)
    o = list(range(n))
    for i in range(0, n - 1, 2):
        o[i], o[i + 1] = o[i + 1], o[i]
    yield "pairs", o


CASES = [(4, 0, 7, 3000, 8192), (8, 1, 40, 5000, 12_000), (16, 2, 120, 20_000, 60_000), (3, 3, 25, 900, 1),
         (5, 4, 60, 4000, 10 ** 9), (2, 5, 1, 100, 50)]


@pytest.mark.parametrize("world,seed,n,hi,B", CASES)
def test_flat_order_is_the_flat_layout(world, seed, n, hi, B):
    rng = np.random.default_rng(seed)
    numel = W.random_numels(rng, n, 1, hi)
    a = oracle.layout(numel, world, B)
    b = oracle.layout(numel, world, B, order=list(range(n)))
    for f in ("offset", "bucket_of", "bucket_range", "slices", "runs"):
        assert np.array_equal(getattr(a, f), getattr(b, f)), f
    for k in range(a.n_buckets):
        s, nb = a.bucket(k)
        assert np.array_equal(b.flat_map(k), np.arange(s, s + nb))


@pytest.mark.parametrize("world,seed,n,hi,B", CASES)
def test_bucket_walk_follows_arrival(world, seed, n, hi, B):
    rng = np.random.default_rng(seed + 100)
    numel = W.random_numels(rng, n, 1, hi)
    for name, order in _orders(rng, n):
        lay = oracle.layout(numel, world, B, order=order)
        # buckets are consecutive stretches of the arrival order, in order
        bs = [int(lay.bucket_of[i]) for i in order]
        assert bs[0] == 0 and all(y - x in (0, 1) for x, y in zip(bs, bs[1:])), name
        fill = {}
        for i in order:
            b = int(lay.bucket_of[i])
            assert int(lay.bucket_pos[i]) == fill.get(b, 0), name
            fill[b] = fill.get(b, 0) + int(numel[i])
        # the closing rule: a bucket closes only before a param that would overflow it
        for k in range(1, n):
            i, j = order[k - 1], order[k]
            if lay.bucket_of[j] != lay.bucket_of[i]:
                assert fill[int(lay.bucket_of[i])] + numel[j] > B
        # sizes, padding with the bucket of the last flat param
        pb = int(lay.bucket_of[n - 1])
        for b in range(lay.n_buckets):
            size, pad, _ = (int(x) for x in lay.bucket_info[b])
            extra = lay.P - lay.T if b == pb else 0
            assert size == fill[b] + extra
            assert pad == (fill[b] if b == pb else -1)
        # slices: bucket position = the param's position + the slice's offset in the param
        for p, b, dst, po, bo, pao, num in lay.slices:
            assert bo == lay.bucket_pos[p] + po and b == lay.bucket_of[p]
            assert lay.offset[p] + po == dst * lay.S + pao


@pytest.mark.parametrize("world,seed,n,hi,B", CASES)
def test_runs_cover_map_and_are_maximal(world, seed, n, hi, B):
    rng = np.random.default_rng(seed + 200)
    numel = W.random_numels(rng, n, 1, hi)
    for name, order in _orders(rng, n):
        lay = oracle.layout(numel, world, B, order=order)
        for b in range(lay.n_buckets):
            _, nb = lay.bucket(b)
            fm = lay.flat_map(b)
            assert sorted(fm.tolist()) == sorted(set(fm.tolist())) and (fm >= 0).all()
            seen = np.zeros(nb, dtype=np.int64)
            rs = lay.runs_of(b)
            for _, dst, bo, pao, num in rs:
                seen[bo:bo + num] += 1
                assert np.array_equal(fm[bo:bo + num], dst * lay.S + pao + np.arange(num)), name
            assert (seen == 1).all(), name
            rs = rs[np.argsort(rs[:, 2])]
            for (_, d0, x0, p0, n0), (_, d1, x1, p1, _) in zip(rs, rs[1:]):
                assert not (d0 == d1 and x0 + n0 == x1 and p0 + n0 == p1), "mergeable runs left apart"


def _step(lay, grads, p, m, v, hp, scale):
    param = np.zeros(lay.P, np.uint16)
    for b in range(lay.n_buckets):
        bucket = oracle.bucket_pack(lay, b, grads)
        oracle.rs_adam_fused(lay, b, bucket, scale, p, m, v, hp, param)
    return param


@pytest.mark.parametrize("world,seed,n,hi,B", CASES[:4])
def test_results_do_not_depend_on_arrival_order(world, seed, n, hi, B):
    rng = np.random.default_rng(seed + 300)
    numel = W.random_numels(rng, n, 1, hi)
    wl = W.Workload("o", tuple(numel), world, B, ("normal", 1e-2), 0.02, ("absnormal", 1e-4), W.AdamW(step=4))
    inp = W.draw_inputs(wl, "cpu", seed=seed)
    hp = W.AdamW(step=4)
    scale = float(np.float32(1.0 / world))
    base = oracle.layout(numel, world, B)
    grads = [oracle.params_from_flat(base, W.bf16_bits(inp["grads"][k][0])) for k in range(world)]

    def run(lay):
        p = oracle.shards_from_flat(lay, inp["master"].numpy())
        m = oracle.shards_from_flat(lay, inp["m"].numpy())
        v = oracle.shards_from_flat(lay, inp["v"].numpy())
        return _step(lay, grads, p, m, v, hp, scale), p, m, v

    ref = run(base)
    for name, order in _orders(rng, n):
        got = run(oracle.layout(numel, world, B, order=order))
        assert np.array_equal(got[0], ref[0]), name
        for r in range(world):
            for a, c in zip(got[1:], ref[1:]):
                assert np.array_equal(a[r].view(np.uint32), c[r].view(np.uint32)), name


def test_reduce_scatter_then_concat_equals_allreduce_under_order():
    rng = np.random.default_rng(9)
    numel = W.random_numels(rng, 30, 1, 3000)
    world = 4
    lay = oracle.layout(numel, world, 9000, order=list(range(29, -1, -1)))
    grads = [[rng.integers(0, 1 << 16, size=k, dtype=np.uint16) & np.uint16(0x7f7f) for k in numel]
             for _ in range(world)]
    for b in range(lay.n_buckets):
        bucket = oracle.bucket_pack(lay, b, grads)
        shards = [np.full(lay.S, np.nan, np.float32) for _ in range(world)]
        oracle.reduce_scatter_avg(lay, b, bucket, 0.25, shards)
        ar = oracle.allreduce_avg(world, bucket, 0.25)[0]
        full = np.concatenate(shards)
        assert np.array_equal(full[lay.flat_map(b)].view(np.uint32), ar.view(np.uint32))


def test_order_must_be_a_permutation():
    with pytest.raises(oracle.OracleError):
        oracle.layout([3, 4, 5], 2, 10, order=[0, 0, 2])
    with pytest.raises(oracle.OracleError):
        oracle.layout([3, 4, 5], 2, 10, order=[0, 1, 3])
