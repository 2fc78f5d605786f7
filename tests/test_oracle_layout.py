"""Pins of the oracle's flat layout, buckets, slices and runs (CPU only).

The oracle is checked against a per-element brute force (``oracle/brute.py``),
against the defining properties of the bucket walk, and against a worked
example done by hand for the 7-parameter workload.
Sources: "DeepSpeed ZeRO 通信优化深度解析" §二 (equal partitions per rank),
§三.2 (param_to_partition_ids, grad_start_offset, (dst_rank, bucket_offset,
numel) slices, merging of same-destination fragments), §四 (IPG bucket of
reduce_bucket_size elements).
"""
import numpy as np
import pytest

import oracle
from oracle import brute
from zero_partition_aware_gb300 import workloads as W


def _check_buckets(lay, numel, B):
    """A bucket is a contiguous run of params, at most B elements unless it holds a
    single oversized param, and it was closed only because the next param would overflow."""
    nb = lay.n_buckets
    assert nb >= 1
    groups = [[i for i in range(len(numel)) if lay.bucket_of[i] == b] for b in range(nb)]
    flat = [i for g in groups for i in g]
    assert flat == list(range(len(numel)))
    for b, g in enumerate(groups):
        assert g, "empty bucket"
        assert g == list(range(g[0], g[-1] + 1))
        tot = sum(numel[i] for i in g)
        assert tot <= B or len(g) == 1
        if b + 1 < nb:
            assert tot + numel[groups[b + 1][0]] > B
        s, e = (int(x) for x in lay.bucket_range[b])
        assert s == int(lay.offset[g[0]])
        assert e == (int(lay.offset[groups[b + 1][0]]) if b + 1 < nb else lay.P)


def _check_layout(numel, world, B):
    lay = oracle.layout(numel, world, B)
    T = sum(numel)
    assert lay.T == T
    assert lay.P % world == 0 and 0 <= lay.P - T < world
    assert lay.S * world == lay.P
    assert list(lay.offset) == list(np.cumsum([0] + list(numel))[:-1])
    _check_buckets(lay, numel, B)
    # slices against the per-element labelling
    starts = [int(x) for x in lay.bucket_range[:, 0]]
    want = brute.brute_slices(numel, world, list(lay.bucket_of), starts)
    got = [tuple(int(x) for x in row) for row in lay.slices]
    assert got == want
    # runs against maximal (bucket, rank) stretches over [0, P)
    ranges = [tuple(int(x) for x in r) for r in lay.bucket_range]
    want_runs = brute.brute_runs(numel, world, ranges)
    got_runs = [tuple(int(x) for x in row) for row in lay.runs]
    assert got_runs == want_runs
    # invariants
    per_param = np.zeros(len(numel), dtype=np.int64)
    for row in lay.slices:
        per_param[row[0]] += row[6]
    assert list(per_param) == list(numel)
    covered = sorted((int(r[0]), int(r[2]), int(r[2] + r[4])) for r in lay.runs)
    for b in range(lay.n_buckets):
        segs = [(s, e) for bb, s, e in covered if bb == b]
        s0, n0 = lay.bucket(b)
        pos = 0
        for s, e in segs:
            assert s == pos
            pos = e
        assert pos == n0
    for i in range(len(numel)):
        ids, gso = lay.param_partitions(i)
        assert ids == list(range(ids[0], ids[-1] + 1))
        assert gso[0] == 0 and all(g > 0 for g in gso[1:])
    return lay


def test_worked_example_tiny():
    """Hand derivation for numel [1000, 5661, 4096, 8385, 10, 6144, 777], N=4, B=8192.

    T = 26073, P = ceil(26073/4)*4 = 26076, S = 6519. Offsets are prefix sums.
    p1 = [1000, 6661) crosses 6519: partitions {0, 1}, grad_start_offset {0, 5519}.
    p3 = [10757, 19142) crosses 13038: {1, 2}, {0, 2281}.
    p5 = [19152, 25296) crosses 19557: {2, 3}, {0, 405}.
    Buckets: 1000+5661 = 6661 fits; +4096 overflows -> b0 = [0, 6661);
    b1 = p2 alone (4096 + 8385 > 8192); p3 = 8385 > 8192 sits alone;
    b3 = p4..p6 (10+6144+777 = 6931) plus the 3 padding elements.
    """
    lay = _check_layout([1000, 5661, 4096, 8385, 10, 6144, 777], 4, 8192)
    assert (lay.T, lay.P, lay.S) == (26073, 26076, 6519)
    assert list(lay.offset) == [0, 1000, 6661, 10757, 19142, 19152, 25296]
    assert lay.param_partitions(1) == ([0, 1], [0, 5519])
    assert lay.param_partitions(3) == ([1, 2], [0, 2281])
    assert lay.param_partitions(5) == ([2, 3], [0, 405])
    for i in (0, 2, 4, 6):
        assert len(lay.param_partitions(i)[0]) == 1
    assert [tuple(r) for r in lay.bucket_range.tolist()] == [
        (0, 6661), (6661, 10757), (10757, 19142), (19142, 26076)]
    runs = {b: [tuple(r[1:]) for r in lay.runs_of(b).tolist()] for b in range(4)}
    assert runs[0] == [(0, 0, 0, 6519), (1, 6519, 0, 142)]
    assert runs[1] == [(1, 0, 142, 4096)]
    assert runs[2] == [(1, 0, 4238, 2281), (2, 2281, 0, 6104)]
    assert runs[3] == [(2, 0, 6104, 415), (3, 415, 0, 6519)]


def test_tiny_workload_shapes_match_the_worked_example():
    assert list(W.WORKLOADS["tiny"].numel) == [1000, 5661, 4096, 8385, 10, 6144, 777]


@pytest.mark.parametrize("seed", range(40))
def test_random_tiny_layouts_against_brute_force(seed):
    rng = np.random.default_rng(1000 + seed)
    n = int(rng.integers(1, 12))
    world = int(rng.choice([1, 2, 3, 4, 5, 7, 8, 13, 16, 32]))
    numel = W.random_numels(rng, n, 1, 700)
    B = int(rng.integers(1, 2000))
    _check_layout(numel, world, B)


def test_edge_layouts():
    _check_layout([1], 1, 1)                 # one element, one rank
    _check_layout([1], 32, 1)                # P = 32, S = 1: 31 padding elements over ranks
    _check_layout([5, 1, 1, 1], 8, 2)        # params straddling many 1-element partitions
    _check_layout([3, 3, 3], 3, 3)           # exact fit, no padding, full buckets
    _check_layout([10] * 7, 4, 1)            # every param oversized -> singleton buckets
    _check_layout([7], 4, 1000)              # one bucket with padding
    lay = oracle.layout([], 4, 10)           # empty model
    assert (lay.T, lay.P, lay.S, lay.n_buckets) == (0, 0, 0, 0)
    assert lay.slices.shape[0] == 0 and lay.runs.shape[0] == 0


@pytest.mark.parametrize("bad", [([0], 2, 4), ([1, -3], 2, 4), ([4], 0, 4), ([4], 2, 0)])
def test_invalid_layout_arguments(bad):
    with pytest.raises(oracle.OracleError):
        oracle.layout(*bad)


@pytest.mark.parametrize("name,T,P,S", [
    ("tiny", 26073, 26076, 6519),
    ("gpt2_124m", 124438272, 124438272, 15554784),
    ("llama_1p1b", 1100048384, 1100048384, 137506048),
    ("irregular_10k", 718175492, 718175504, 44885969),
    ("llama3_3b", 3212749824, 3212749824, 401593728),
])
def test_workload_sizes(name, T, P, S):
    wl = W.WORKLOADS[name]
    lay = oracle.layout(list(wl.numel), wl.world, wl.bucket)
    assert (lay.T, lay.P, lay.S) == (T, P, S)
    # runs tile [0, P) and each run lies in one bucket and one partition
    assert int(lay.runs[:, 4].sum()) == lay.P
    for b, dst, bo, po, n in lay.runs.tolist():
        s, nb = lay.bucket(b)
        assert 0 <= bo and bo + n <= nb
        assert 0 <= po and po + n <= lay.S
        assert s + bo == dst * lay.S + po
    assert int(lay.slices[:, 6].sum()) == lay.T


def test_bucket_counts_of_workloads():
    counts = {name: oracle.layout(list(wl.numel), wl.world, wl.bucket).n_buckets
              for name, wl in W.WORKLOADS.items()}
    assert counts["tiny"] == 4
    assert counts["irregular_10k"] >= 718175492 // (1 << 24)
