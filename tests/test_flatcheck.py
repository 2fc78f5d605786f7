"""The whole-array checker (tests/flatcheck.py) on the CPU, before it judges a GPU.

The checker recomputes each flat element from its replicas' gradients through
the oracle's elementwise averaging, AdamW and cast, chunk by chunk. Here it is
held against the oracle's own bucket path (bucket_pack, then rs_adam_fused per
bucket over whole partitions, "DeepSpeed ZeRO 通信优化深度解析" §三.2, §四) on
small layouts, with chunks that cut params, buckets and partitions at odd
places: it must report no mismatch, and exactly the planted ones when single
elements of the outputs or inputs are altered.
"""
import numpy as np
import pytest
import torch

import oracle
from zero_partition_aware_gb300 import workloads as W

import flatcheck


def _case(seed, world, n, hi, bucket, grad=("normal", 1e-2), state=("absnormal", 1e-4), step=3):
    rng = np.random.default_rng(seed)
    numel = W.random_numels(rng, n, 1, hi)
    wl = W.Workload("chk", tuple(numel), world, bucket, grad, 0.02, state, W.AdamW(step=step))
    lay = oracle.layout(numel, world, bucket)
    inp = W.draw_inputs(wl, "cpu", seed=seed)
    offs = W.arena_offsets(numel, 8)
    size = offs[-1] + numel[-1]
    arenas = []
    for k in range(world):
        a = torch.zeros(size, dtype=torch.bfloat16)
        for i, o in enumerate(offs):
            a[o:o + numel[i]] = inp["grads"][k][0][int(lay.offset[i]): int(lay.offset[i]) + numel[i]]
        arenas.append(a)
    before = []
    for name in ("master", "m", "v"):
        t = torch.zeros(lay.P, dtype=torch.float32)
        t[: lay.T] = inp[name]
        before.append(t)
    return wl, lay, inp, arenas, offs, before


def _oracle_bucket_path(wl, lay, inp, before, coef=None):
    """after (flat master, m, v) and the bf16 params by the oracle's bucket path."""
    grads = [oracle.params_from_flat(lay, W.bf16_bits(inp["grads"][k][0])) for k in range(wl.world)]
    p, m, v = ([t.numpy()[r * lay.S:(r + 1) * lay.S].copy() for r in range(lay.world)]
               for t in before)
    param = np.zeros(lay.P, np.uint16)
    scale = float(np.float32(1.0 / wl.world))
    if coef is None:
        for b in range(lay.n_buckets):
            oracle.rs_adam_fused(lay, b, oracle.bucket_pack(lay, b, grads), scale, p, m, v, wl.adam, param)
        g = None
    else:
        g = [np.zeros(lay.S, np.float32) for _ in range(lay.world)]
        for b in range(lay.n_buckets):
            oracle.reduce_scatter_avg(lay, b, oracle.bucket_pack(lay, b, grads), scale, g)
        oracle.adam_clip_step(lay, p, m, v, g, wl.adam, coef, False, param)
        g = torch.from_numpy(np.concatenate(g))
    after = [torch.from_numpy(np.concatenate(a)) for a in (p, m, v)]
    return after, torch.from_numpy(param.view(np.int16)).view(torch.bfloat16), g, scale


@pytest.mark.parametrize("seed,world,n,hi,bucket,chunk", [(1, 4, 30, 3000, 5000, 777),
                                                          (2, 16, 60, 20_000, 40_000, 4099),
                                                          (3, 3, 12, 500, 1, 100)])
def test_checker_agrees_with_the_bucket_path(seed, world, n, hi, bucket, chunk):
    wl, lay, inp, arenas, offs, before = _case(seed, world, n, hi, bucket)
    after, param, _, scale = _oracle_bucket_path(wl, lay, inp, before)
    res = flatcheck.check_whole(lay, scale, wl.adam, flatcheck.ArenaGrads(arenas, lay, offs), before, after,
                                param, chunk=chunk)
    assert res["elements"] == lay.P
    assert all(res[k] == 0 for k in ("master", "m", "v", "param")), res


def test_checker_finds_planted_mistakes():
    wl, lay, inp, arenas, offs, before = _case(4, 8, 40, 5000, 9000)
    after, param, _, scale = _oracle_bucket_path(wl, lay, inp, before)
    src = flatcheck.ArenaGrads(arenas, lay, offs)
    j = lay.T // 3
    after[1][j] = torch.nextafter(after[1][j], torch.tensor(1.0))  # one ulp on m
    q = param.view(torch.int16)
    q[lay.T - 1] ^= 1                                                # the last real param's low bit
    res = flatcheck.check_whole(lay, scale, wl.adam, src, before, after, param, chunk=1000)
    assert (res["master"], res["m"], res["v"], res["param"]) == (0, 1, 0, 1)
    assert res["m_first"] == j and res["param_first"] == lay.T - 1
    # an input the step did not see: replica 5's gradient of one element changed
    after[1][j] = torch.nextafter(after[1][j], torch.tensor(-1.0))
    q[lay.T - 1] ^= 1
    i = 7
    arenas[5][offs[i]] = arenas[5][offs[i]] + 1.0
    res = flatcheck.check_whole(lay, scale, wl.adam, src, before, after, param, chunk=1000)
    f = int(lay.offset[i])
    assert res["master_first"] == f and res["m"] == 1 and res["v"] == 1 and res["master"] == 1


def test_checker_micro_steps_and_integer_average():
    """FlatGrads of several micro-steps (the accumulated main_grad checked too),
    and the exact-integer check on integer gradients."""
    world, S_ = 4, 3
    wl, lay, inp, arenas, offs, before = _case(5, world, 20, 2000, 4000, grad=("int", -8, 8))
    scale = float(np.float32(1.0 / world))
    rng = np.random.default_rng(5)
    mb = [[torch.from_numpy(rng.integers(-8, 9, lay.P).astype(np.float32)).to(torch.bfloat16) for _ in range(S_)]
          for _ in range(world)]
    for row in mb:
        for t in row:
            t[lay.T:] = 0
    # the oracle's micro-step path: accumulate into fp32, then the bucket path over the sums
    mains = []
    for row in mb:
        acc = np.zeros(lay.P, np.float32)
        for t in row[:-1]:
            oracle.grad_accumulate(acc, W.bf16_bits(t))
        mains.append(torch.from_numpy(acc.copy()))
        oracle.grad_accumulate(acc, W.bf16_bits(row[-1]))
        row.append(acc)
    p, m, v = ([t.numpy()[r * lay.S:(r + 1) * lay.S].copy() for r in range(world)] for t in before)
    param = np.zeros(lay.P, np.uint16)
    for b in range(lay.n_buckets):
        s0, nb = lay.bucket(b)
        oracle.rs_adam_fused(lay, b, [np.ascontiguousarray(row[-1][s0:s0 + nb]) for row in mb], scale, p, m, v,
                             wl.adam, param)
    for row in mb:
        row.pop()
    after = [torch.from_numpy(np.concatenate(a)) for a in (p, m, v)]
    qt = torch.from_numpy(param.view(np.int16)).view(torch.bfloat16)
    res = flatcheck.check_whole(lay, scale, wl.adam, flatcheck.FlatGrads(mb), before, after, qt,
                                main_after=mains, chunk=333)
    assert all(res[k] == 0 for k in ("master", "m", "v", "param", "main_grad")), res
    mains[2][100] += 1.0
    res = flatcheck.check_whole(lay, scale, wl.adam, flatcheck.FlatGrads(mb), before, after, qt,
                                main_after=mains, chunk=333)
    assert res["main_grad"] == 1 and res["main_grad_first"] == 100
    # integer gradients: the average is the exact sum / N everywhere
    after2, param2, _, _ = _oracle_bucket_path(wl, lay, inp, before)
    res = flatcheck.check_whole(lay, scale, wl.adam, flatcheck.ArenaGrads(arenas, lay, offs), before, after2,
                                param2, integer_avg=True, chunk=500)
    assert all(res[k] == 0 for k in ("master", "m", "v", "param", "integer_avg")), res


def test_checker_clipped_step():
    wl, lay, inp, arenas, offs, before = _case(6, 8, 50, 8000, 20_000)
    coef = 0.37
    after, param, g, scale = _oracle_bucket_path(wl, lay, inp, before, coef=coef)
    res = flatcheck.check_whole(lay, scale, wl.adam, flatcheck.ArenaGrads(arenas, lay, offs), before, after,
                                param, grad_after=[g], coef=coef, chunk=2048)
    assert all(res[k] == 0 for k in ("grad", "master", "m", "v", "param")), res
    g[17] = 0.5
    res = flatcheck.check_whole(lay, scale, wl.adam, flatcheck.ArenaGrads(arenas, lay, offs), before, after,
                                param, grad_after=[g], coef=coef, chunk=2048)
    assert res["grad"] == 1 and res["grad_first"] == 17 and res["master"] == 0
