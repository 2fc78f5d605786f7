"""Pins of the oracle's byte accounting against the pages' own tables (CPU only).

Fixtures under tests/golden/ hold the numbers the pages print, each with its
page title and section.
"""
import json
import os

import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_memory_ledger_is_16_bytes():
    g = _golden("memory_ledger.json")
    assert sum(g["bytes_per_param"].values()) == g["total"] == 16
    # plain DP holds all 16 bytes for every param
    assert oracle.layout_bytes(0, 1000, 125) == g["total"] * 1000


@pytest.mark.parametrize("world", [1, 2, 4, 8, 16, 32])
@pytest.mark.parametrize("stage", ["0", "1", "15", "3"])
def test_stage_memory_matches_table(stage, world):
    row = _golden("zero_stages.json")["stages"][stage]
    S = 1000
    T = S * world  # no padding: the table's per-param coefficients apply exactly
    want = row["full"] * T + row["sharded"] * T / world
    assert oracle.layout_bytes(int(stage), T, S) == want


@pytest.mark.parametrize("world", [2, 4, 8, 16, 32, 64])
def test_comm_ratios(world):
    g = _golden("comm_volume.json")
    S, e = 12345, 2
    dp = oracle.comm_bytes(0, world, S, e)
    assert oracle.comm_bytes(1, world, S, e) / dp == g["initial_zero1_over_dp"]
    assert oracle.comm_bytes(2, world, S, e) / dp == g["partition_aware_over_dp"]
    assert oracle.comm_bytes(3, world, S, e) / dp == g["rs_over_allreduce"]
    # ring all-reduce: 2(N-1)/N of the P*e message
    P = S * world
    assert dp == pytest.approx(2 * (world - 1) / world * P * e, rel=0, abs=1e-6)
    ex = g["ring_allreduce_factor_examples"].get(str(world))
    if ex is not None:
        assert dp / (P * e) == ex


def test_single_rank_communicates_nothing():
    for scheme in range(4):
        assert oracle.comm_bytes(scheme, 1, 999, 2) == 0.0
